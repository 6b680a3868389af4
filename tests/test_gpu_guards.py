"""Device index checks (needs a GB300).

Every kernel that indexes the cache through caller data checks the index and,
when it is out of range, skips the access and sets a bit of the handle's
device status word (include/mla_draft.h, MLA_DEV_*): a slot outside the
cache (the append's slot scatter), a position outside the RoPE table, a
page id outside [0, num_pages) (the attention's key walk: the copy reads
zeros instead), a kv_len beyond the block's page table (clamped) and a
negative window (the block sees no key).  Each case below plants one such
index in otherwise valid inputs; the status reports it as MLA_ERR_DEVICE_CHECK
with the matching bit, the valid rows are computed as usual, and the word is
clear on the next call.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _status(dev):
    from head_latent_attention_qkv_gb300 import _lib
    import ctypes as C
    bits = C.c_int32(0)
    st = _lib.lib.mla_get_device_status(dev.handle.h, None, C.byref(bits))
    return st, bits.value


@pytest.mark.parametrize("name", ["qwen3_4b_prefill", "tiny_fp32"])
def test_append_with_a_slot_outside_the_cache(name):
    from head_latent_attention_qkv_gb300 import _lib, api, workloads
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload
    wl = workloads.make_workload(name, "small")
    dev = DeviceWorkload(wl)
    hid, pos, slots = dev.ctx
    num_slots = dev.cache.shape[0] * dev.cache.shape[1]
    bad = slots.clone()
    bad[3] = num_slots                 # one past the last slot
    dev.cache.fill_(float("nan"))
    api.mla_latent_cache_append(dev.handle, hid, pos, bad, dev.cache)
    torch.cuda.synchronize()
    st, bits = _status(dev)
    assert st == _lib.MLA_ERR_DEVICE_CHECK and bits & _lib.MLA_DEV_BAD_SLOT
    flat = dev.cache.float().view(num_slots, -1)
    good = torch.ones(len(slots), dtype=torch.bool, device="cuda")
    good[3] = False
    assert torch.isfinite(flat[slots[good]]).all()       # every valid token written
    assert torch.isnan(flat[slots[3]]).all()              # the skipped token's own slot untouched
    assert _status(dev) == (_lib.MLA_OK, 0)               # read once, then cleared
    dev.handle.close()


def test_append_with_a_position_outside_the_rope_table():
    from head_latent_attention_qkv_gb300 import _lib, api, workloads
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload
    wl = workloads.make_workload("qwen3_4b_prefill", "small")
    dev = DeviceWorkload(wl)
    hid, pos, slots = dev.ctx
    bad = pos.clone()
    bad[5] = wl.dims.max_position
    api.mla_latent_cache_append(dev.handle, hid, bad, slots, dev.cache)
    torch.cuda.synchronize()
    st, bits = _status(dev)
    assert st == _lib.MLA_ERR_DEVICE_CHECK and bits & _lib.MLA_DEV_BAD_POSITION
    dev.handle.close()


@pytest.mark.parametrize("name", ["qwen3_4b_prefill", "fp32_three_blocks"])
def test_attention_with_an_invalid_page_and_an_overlong_kv_len(name):
    from head_latent_attention_qkv_gb300 import _lib, api, workloads
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload
    if name == "fp32_three_blocks":
        wl = workloads.prefill_workload(name, workloads.TINY_FP32_MLA, 0, [64, 40, 30], 8,
                                        page_size=16)
    else:
        wl = workloads.make_workload(name, "small")
    dev = DeviceWorkload(wl)
    dev.run_all()
    torch.cuda.synchronize()
    assert _status(dev) == (_lib.MLA_OK, 0)
    s = dev.steps[0]
    ref = s["out"].clone()
    # block 1: its first page id out of range; block 2: kv_len past its table
    s["block_table"][1, 0] = -1
    s["kv_len"][2] = s["block_table"].shape[1] * wl.page_size + 5
    dev.reset_cache()
    dev.append_context()
    out = dev.run_step(0)
    torch.cuda.synchronize()
    st, bits = _status(dev)
    assert st == _lib.MLA_ERR_DEVICE_CHECK
    assert bits & _lib.MLA_DEV_BAD_PAGE and bits & _lib.MLA_DEV_BAD_LENGTH
    assert torch.isfinite(out.float()).all()
    T = wl.block_len
    # block 0 is untouched by either planted index
    assert torch.equal(out[:T], ref[:T])
    dev.handle.close()
