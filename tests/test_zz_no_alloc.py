"""The allocation-free latent append against the regular one (needs a GB300).

``mla_latent_cache_append_noalloc`` is for callers that cannot allocate
device memory where they append (host callbacks, allocator hooks, runtimes
whose memory pool is fixed in advance): it takes no workspace and stages its
projection in a fixed array inside the library.  Two calls in a row, each on
different tokens, must leave the same cache contents as the regular append,
within the parity tolerance; a request larger than the fixed array must be
refused.  This file is collected last so that a stop at its first failure
has already run every other test.
"""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _tol_check(a, b, dims):
    from tests.parity import compare
    written = np.isfinite(b).all(axis=1)
    assert np.array_equal(np.isfinite(a).all(axis=1), written), "different slots written"
    compare(a[written], b[written], dims, "noalloc append vs append")


@pytest.mark.parametrize("name", ["qwen3_4b_prefill", "tiny_fp32"])
def test_noalloc_append_matches_regular_append_on_two_calls(name):
    """bf16 (tolerance 2e-2 / 2e-3 of the rms) and fp32 (1e-4) layers."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_latent_attention_qkv_gb300 import _lib, api, workloads
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload

    wl = workloads.make_workload(name, "small")
    dev = DeviceWorkload(wl)
    h = dev.handle
    hid, pos, slots = dev.ctx
    cache_ref = torch.full_like(dev.cache, float("nan"))
    cache_new = torch.full_like(dev.cache, float("nan"))
    L = wl.dims.cache_dim
    halves = [slice(0, len(slots) // 2), slice(len(slots) // 2, len(slots))]
    stream = torch.cuda.current_stream()
    for part in halves:                       # two calls in a row, different tokens
        n = part.stop - part.start
        api.mla_latent_cache_append(h, hid[part], pos[part], slots[part], cache_ref)
        st = _lib.lib.mla_latent_cache_append_noalloc(
            h.h, C.c_void_p(hid[part].data_ptr()), C.c_void_p(pos[part].data_ptr()),
            C.c_void_p(slots[part].data_ptr()), n, C.c_void_p(cache_new.data_ptr()),
            cache_new.shape[0], C.c_void_p(stream.cuda_stream))
        _lib.check(st, "mla_latent_cache_append_noalloc")
        torch.cuda.synchronize()
        _tol_check(cache_new.float().cpu().numpy().reshape(-1, L),
                   cache_ref.float().cpu().numpy().reshape(-1, L), wl.dims)
    assert api.mla_get_device_status(h) == 0


def test_noalloc_append_refuses_more_tokens_than_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_latent_attention_qkv_gb300 import _lib, workloads
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload

    wl = workloads.make_workload("qwen3_4b_prefill", "small")
    dev = DeviceWorkload(wl)
    cap = _lib.lib.mla_append_noalloc_max_tokens(dev.handle.h)
    assert cap == (1 << 20) // wl.dims.cache_dim
    hid, pos, slots = dev.ctx
    st = _lib.lib.mla_latent_cache_append_noalloc(
        dev.handle.h, C.c_void_p(hid.data_ptr()), C.c_void_p(pos.data_ptr()),
        C.c_void_p(slots.data_ptr()), int(cap) + 1, C.c_void_p(dev.cache.data_ptr()),
        dev.cache.shape[0], None)
    assert st == _lib.MLA_ERR_INVALID_ARG
    assert b"exceeds the fixed scratch" in _lib.lib.mla_last_error()
