"""Failure path of the bounded device waits (needs a GB300).

Every wait in the library's kernels gives up after a budget of try_wait
rounds, sets MLA_DEV_TIMEOUT in the device status word and returns.  The
self-check entry point runs that wait on a barrier nothing arrives on (a flag
that nothing sets); the host then reads MLA_ERR_TIMEOUT, the word is cleared,
and the same handle still computes a parity-clean forward.  No GPU fault, trap
or hang is involved: the waiting kernel has one thread, issues no copies and
holds no tensor memory.
"""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_reports_timeout_and_handle_stays_usable():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_latent_attention_qkv_gb300 import _lib, api, workloads
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload
    from tests.parity import check_workload

    wl = workloads.make_workload("qwen3_4b_prefill", "small")
    dev = DeviceWorkload(wl)
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.mla_check_wait_timeout(dev.handle, 1000, gave_up)
    torch.cuda.synchronize()
    assert int(gave_up.item()) == 1
    bits = api.mla_get_device_status(dev.handle)
    assert bits & _lib.MLA_DEV_TIMEOUT, bits
    st = _lib.lib.mla_get_device_status(dev.handle.h, None, None)
    assert st == _lib.MLA_OK                  # read once, then cleared
    # the same handle still runs the forward, and matches the oracle
    check_workload(wl, dev=dev)


def test_wait_budget_argument_is_validated():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from head_latent_attention_qkv_gb300 import _lib, workloads
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload

    dev = DeviceWorkload(workloads.make_workload("tiny_fp32", "small"))
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0, (1 << 24) + 1):
        st = _lib.lib.mla_check_wait_timeout(dev.handle.h, bad, gave_up.data_ptr(), None)
        assert st == _lib.MLA_ERR_INVALID_ARG
    dev.handle.close()
