"""Forward overlapped with the cache append (needs a GB300).

``mla_draft_forward_after`` lets the forward's projections run while the
cache append runs on a second stream; only the attention waits for the
append.  The kernels are the same as in the serial order and deterministic,
so the overlapped step must reproduce the serial step bit for bit: outputs,
the cache and the visibility statistics.  The serial path itself is checked
against the oracle in test_gpu_parity.py.  The cache starts as NaN, so an
attention that ran before the append finished would show up as NaN rows.
"""
import numpy as np
import pytest

from head_latent_attention_qkv_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _state(dev):
    return ([s["out"].clone() for s in dev.steps], dev.cache.clone(),
            [s["vis_stats"].clone() for s in dev.steps])


def _overlapped(dev, side):
    for k in range(len(dev.steps)):
        dev.run_step_after(k, side, with_context=(k == 0))


def _assert_same(a, b, what):
    for x, y in zip(a[0], b[0]):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y), f"{what}: outputs"
    ca, cb = a[1], b[1]
    assert torch.equal(torch.isnan(ca), torch.isnan(cb)), f"{what}: written slots"
    assert torch.equal(torch.nan_to_num(ca), torch.nan_to_num(cb)), f"{what}: cache"
    for x, y in zip(a[2], b[2]):
        assert torch.equal(x, y), f"{what}: visibility statistics"


@pytest.mark.parametrize("size,name", [("small", n) for n in workloads.WORKLOADS]
                         + [("full", "qwen3_4b_prefill"), ("full", "qwen3_4b_cached_decode")])
def test_overlapped_step_equals_serial(size, name):
    from head_latent_attention_qkv_gb300 import api
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload
    wl = workloads.make_workload(name, size)
    dev = DeviceWorkload(wl)
    dev.run_all()
    torch.cuda.synchronize()
    serial = _state(dev)
    assert all(torch.isfinite(o.float()).all() for o in serial[0])

    side = torch.cuda.Stream()
    dev.reset_cache()
    for s in dev.steps:
        s["out"].fill_(float("nan"))
        s["vis_stats"].fill_(-7)
    _overlapped(dev, side)
    torch.cuda.synchronize()
    assert api.mla_get_device_status(dev.handle) == 0
    _assert_same(_state(dev), serial, f"{name} ({size}) eager")

    # the same step captured in one CUDA graph (the event forks and joins)
    g = torch.cuda.CUDAGraph()
    dev.reset_cache()
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        _overlapped(dev, side)
    for _ in range(2):
        dev.reset_cache()
        for s in dev.steps:
            s["out"].fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        _assert_same(_state(dev), serial, f"{name} ({size}) graph")
    assert api.mla_get_device_status(dev.handle) == 0
    dev.handle.close()


def test_forward_after_without_event_is_forward():
    from head_latent_attention_qkv_gb300 import api
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload
    wl = workloads.make_workload("qwen3_4b_prefill", "small")
    dev = DeviceWorkload(wl)
    outs = dev.run_all()
    s = dev.steps[0]
    again = api.mla_draft_forward_after(dev.handle, s["hidden"], s["positions"], s["slots"],
                                        dev.cache, s["desc"], cache_ready=None)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), outs[0].view(torch.int16))
    dev.handle.close()
