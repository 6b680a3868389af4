"""The latent attention entry point alone against the fp64 oracle (needs a GB300).

``mla_latent_attention`` takes absorbed query rows and the paged latent cache
and returns the latent output and each row's log-sum-exp ("MLA (Multi-Head
Latent Attention)" blog, forward_mqa / decode_attention_fwd).  Inputs are
seeded synthetic query rows and cache entries; the oracle
(``oracle.mla_grad.latent_attention`` and ``latent_lse``) reads key j of a
block at ``block_table[j // P] * P + j % P`` and applies the visibility of the
workload (windows, masked rows).  Bars, from the kernel's arithmetic: for
bf16 layers the probabilities multiply the values as bf16 (relative rounding
at most 2^-9 each) and the output is stored in fp16 (2^-11), so an element
may differ from the fp64 value by 2^-8 * sum_j p_j |v_j| + 2^-10 |o| (the
first term bounds the bf16 rounding of every weight at twice its size, the
second the fp16 store and fp32 accumulation), and the mean error stays within
2e-3 of the output's rms; fp32 layers: 1e-4 of the rms for both.  The lse
within 2e-3 absolute (1e-5 for fp32), rows without keys exactly +0 with
lse = -inf; the forward's own attention gives the same output bit for bit.
"""
import numpy as np
import pytest

from head_latent_attention_qkv_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(wl, step_index=-1, blocks=None, seed=101):
    from head_latent_attention_qkv_gb300 import api
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload
    from oracle import mla, mla_grad

    dev = DeviceWorkload(wl)
    step, s = wl.steps[step_index], dev.steps[step_index]
    d, P, T, H = wl.dims, wl.page_size, wl.block_len, wl.dims.num_heads
    q, cache_vals = W.attention_inputs(wl, step, seed)
    dt = api.torch_dtype(d)
    q_dev = torch.from_numpy(q).to(dt).cuda()
    dev.cache.copy_(torch.from_numpy(cache_vals).to(dt).view(dev.cache.shape))
    rows = q.shape[0]
    lse = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    o = api.mla_latent_attention(dev.handle, q_dev, s["positions"], dev.cache, s["desc"], lse=lse)
    torch.cuda.synchronize()
    assert api.mla_get_device_status(dev.handle) == 0
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    scale = mla.softmax_scale(d)
    tol_o, tol_m = (1e-4, 1e-4) if d.dtype == "fp32" else (2e-2, 2e-3)
    tol_lse = 1e-5 if d.dtype == "fp32" else 2e-3
    blocks = range(len(step.kv_len)) if blocks is None else blocks
    got, ref, live = [], [], []
    for b in blocks:
        n = int(step.kv_len[b])
        slots = [int(step.block_table[b][j // P]) * P + j % P for j in range(n)]
        tok = slice(b * T, (b + 1) * T)
        vis = mla.visibility(step.block_positions[tok], n, int(step.window[b]),
                             step.q_visible[tok], n)
        vis_rows = np.repeat(vis, H, axis=0)
        r = slice(b * T * H, (b + 1) * T * H)
        o_ref, p_ref = mla_grad.latent_attention(q[r], cache_vals[slots], vis_rows, scale,
                                                 d.kv_lora_rank)
        mag = p_ref @ np.abs(cache_vals[slots][:, :d.kv_lora_rank])
        l_ref = mla_grad.latent_lse(q[r], cache_vals[slots], vis_rows, scale)
        has = vis_rows.any(axis=1)
        assert np.all(o[r][~has] == 0.0) and not np.signbit(o[r][~has]).any(), "masked rows not +0"
        assert np.all(np.isneginf(lse[r][~has])), "masked rows' lse not -inf"
        assert np.all(np.abs(lse[r][has] - l_ref[has]) <= tol_lse * np.maximum(1.0, np.abs(l_ref[has]))), (
            f"lse: max err {np.max(np.abs(lse[r][has] - l_ref[has])):.3e}")
        got.append(o[r][has]); ref.append(o_ref[has]); live.append(mag[has])
    got, ref, mag = np.concatenate(got), np.concatenate(ref), np.concatenate(live)
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    if d.dtype == "fp32":
        bound = np.full(err.shape, tol_o * rms)
    else:
        bound = 2.0 ** -8 * mag + 2.0 ** -10 * np.abs(ref) + 1e-6
    assert np.all(err <= bound) and err.mean() <= tol_m * rms, (
        f"o_lat: max {err.max() / rms:.3e} of rms, mean {err.mean() / rms:.3e}, "
        f"{int(np.count_nonzero(err > bound))} elements beyond the arithmetic bound")
    dev.handle.close()
    return err.max() / rms


@pytest.mark.parametrize("name", W.WORKLOADS)
def test_attention_entry_matches_oracle_small(name):
    _run(W.make_workload(name, "small"))


@pytest.mark.parametrize("name", ["qwen3_4b_prefill", "qwen3_4b_cached_decode",
                                  "qwen3_4b_decode_t1"])
def test_attention_entry_matches_oracle_full_size_sampled(name):
    wl = W.make_workload(name, "full")
    nb = len(wl.steps[-1].kv_len)
    rng = np.random.default_rng(0)
    _run(wl, blocks=sorted(rng.choice(nb, size=min(6, nb), replace=False).tolist()))


def test_attention_entry_equals_the_forwards_own_attention():
    """The forward leaves Q_abs and O_lat in its workspace: the attention entry
    on that Q_abs reproduces that O_lat bit for bit."""
    from head_latent_attention_qkv_gb300 import _lib, api
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload

    wl = W.make_workload("qwen3_4b_sliding_gate", "small")
    dev = DeviceWorkload(wl)
    dev.run_all()
    s = dev.steps[-1]
    M = s["hidden"].shape[0]
    H, L, r = wl.dims.num_heads, wl.dims.cache_dim, wl.dims.kv_lora_rank
    ws = dev.handle._ws
    qo = api.mla_forward_workspace_offset(dev.handle, M, _lib.MLA_WS_Q_ABS)
    oo = api.mla_forward_workspace_offset(dev.handle, M, _lib.MLA_WS_O_LAT)
    torch.cuda.synchronize()
    q_abs = ws[qo:qo + M * H * L * 2].view(torch.bfloat16).view(M * H, L).clone()
    o_fwd = ws[oo:oo + M * H * r * 2].view(torch.float16).view(M * H, r).clone()
    o = api.mla_latent_attention(dev.handle, q_abs, s["positions"], dev.cache, s["desc"])
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_fwd.view(torch.int16))
    dev.handle.close()


def test_negative_window_is_rejected_on_the_device():
    from head_latent_attention_qkv_gb300 import _lib, api
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload

    wl = W.make_workload("qwen3_4b_sliding_gate", "small")
    dev = DeviceWorkload(wl)
    s = dev.steps[-1]
    s["window"][1] = -5
    q, cache_vals = W.attention_inputs(wl, wl.steps[-1], 5)
    q_dev = torch.from_numpy(q).to(torch.bfloat16).cuda()
    dev.cache.copy_(torch.from_numpy(cache_vals).to(torch.bfloat16).view(dev.cache.shape))
    lse = torch.zeros(q.shape[0], dtype=torch.float32, device="cuda")
    o = api.mla_latent_attention(dev.handle, q_dev, s["positions"], dev.cache, s["desc"], lse=lse)
    torch.cuda.synchronize()
    bits = api.mla_get_device_status(dev.handle)
    assert bits & _lib.MLA_DEV_BAD_WINDOW
    rows = wl.block_len * wl.dims.num_heads
    assert torch.all(o[rows:2 * rows] == 0) and torch.all(torch.isneginf(lse[rows:2 * rows]))
    dev.handle.close()


@pytest.mark.parametrize("case", ["t1_ragged", "t1_window_masked", "t3_h8"])
def test_attention_entry_few_row_blocks_match_oracle(case):
    """The few-row kernel through the entry point: o_lat and LSE against the
    oracle, split merge included."""
    from tests.test_gpu_parity import _few_row_case
    _run(_few_row_case(case))
