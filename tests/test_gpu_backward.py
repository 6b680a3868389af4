"""Backward of the latent attention step against the fp64 gradient oracle
(needs a GB300).

``mla_latent_attention_backward`` returns dQ_abs and adds the gradient of
the cache entries (keys and values at once) into an fp32 buffer, from the
forward's output and per-row log-sum-exp ("Add config-selectable MLA draft
attention" (SpecForge PR #758), Validation: gradient parity of the draft's
attention; the forward is the MLA blog's forward_mqa).  Inputs are seeded
synthetic query rows, cache entries and upstream gradients; the oracle is
``oracle.mla_grad.latent_attention_backward`` (explicit formulas pinned by
finite differences and autograd), run per block and summed over blocks that
share cache slots.  Bars: the mean error of both gradients within 2e-3 of
their rms (1e-4 for the fp32 layer); per element, for bf16 layers, the
forward's output o_lat is an fp16 tensor, so D_i = <dO_i, O_i> carries an
error of at most 2^-11 sum_d |dO_id O_id| that every dS_ij of the row
inherits times P_ij: an element may differ by scale |dD_i| sum_j P_ij |e_jd|
(dQ) or scale sum_i P_ij |dD_i| |q_id| (dE) plus 2e-2 of the rms (the fp32
layer: 1e-4 of the rms).  Rows without a visible key get exactly zero.
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


def _check(got, ref, tol_max, tol_mean, what, extra=0.0):
    rms = np.sqrt(np.mean(ref ** 2))
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), what
    over = err > tol_max * rms + extra
    assert not over.any() and err.mean() <= tol_mean * rms, (
        f"{what}: max {err.max() / rms:.3e} mean {err.mean() / rms:.3e} of rms {rms:.3e}, "
        f"{int(over.sum())} elements beyond the bound")


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_4b_prefill", "qwen3_4b_sliding_gate",
                                  "qwen3_4b_cached_decode", "qwen3_4b_decode_t1",
                                  "deepseek_v3_block_parallel"])
def test_attention_backward_matches_gradient_oracle(name):
    from head_latent_attention_qkv_gb300 import api
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload
    from oracle import mla, mla_grad

    wl = W.make_workload(name, "small")
    dev = DeviceWorkload(wl)
    step, s = wl.steps[-1], dev.steps[-1]
    d, P, T, H = wl.dims, wl.page_size, wl.block_len, wl.dims.num_heads
    q, cache_vals = W.attention_inputs(wl, step, 301)
    d_o = W.attention_grad_inputs(wl, step, 302)
    dt = api.torch_dtype(d)
    q_dev = torch.from_numpy(q).to(dt).cuda()
    dev.cache.copy_(torch.from_numpy(cache_vals).to(dt).view(dev.cache.shape))
    rows = q.shape[0]
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    o = api.mla_latent_attention(dev.handle, q_dev, s["positions"], dev.cache, s["desc"], lse=lse)
    d_o_dev = torch.from_numpy(d_o).cuda()
    d_q = torch.full((rows, d.cache_dim), float("nan"), dtype=torch.float32, device="cuda")
    d_cache = torch.zeros(cache_vals.shape, dtype=torch.float32, device="cuda")
    api.mla_latent_attention_backward(dev.handle, q_dev, s["positions"], dev.cache, s["desc"], o,
                                      lse, d_o_dev, d_q, d_cache)
    torch.cuda.synchronize()
    assert api.mla_get_device_status(dev.handle) == 0
    d_q, d_cache = d_q.cpu().numpy(), d_cache.cpu().numpy()

    scale = mla.softmax_scale(d)
    ref_q = np.zeros_like(q, dtype=np.float64)
    ref_c = np.zeros(cache_vals.shape)
    fp16_o = d.dtype == "bf16"
    bnd_q = np.zeros_like(ref_q)
    bnd_c = np.zeros_like(ref_c)
    for b in range(len(step.kv_len)):
        n = int(step.kv_len[b])
        slots = np.array([int(step.block_table[b][j // P]) * P + j % P for j in range(n)])
        tok = slice(b * T, (b + 1) * T)
        vis = mla.visibility(step.block_positions[tok], n, int(step.window[b]),
                             step.q_visible[tok], n)
        vis_rows = np.repeat(vis, H, axis=0)
        r = slice(b * T * H, (b + 1) * T * H)
        dq, de = mla_grad.latent_attention_backward(q[r], cache_vals[slots], vis_rows, scale,
                                                    d.kv_lora_rank, d_o[r])
        ref_q[r] = dq
        np.add.at(ref_c, slots, de)
        if fp16_o:
            o_ref, p_ref = mla_grad.latent_attention(q[r], cache_vals[slots], vis_rows, scale,
                                                     d.kv_lora_rank)
            dD = 2.0 ** -11 * np.sum(np.abs(d_o[r] * o_ref), axis=1)          # [rows]
            bnd_q[r] = scale * dD[:, None] * (p_ref @ np.abs(cache_vals[slots]))
            np.add.at(bnd_c, slots, scale * (p_ref * dD[:, None]).T @ np.abs(q[r]))
        dead = ~vis_rows.any(axis=1)
        assert np.all(d_q[r][dead] == 0.0), "rows without keys must pass nothing back"
    tm, tn = (1e-4, 1e-4) if d.dtype == "fp32" else (2e-2, 2e-3)
    _check(d_q, ref_q, tm, tn, f"{name} dQ_abs", bnd_q)
    touched = np.abs(ref_c).sum(axis=1) > 0
    assert np.all(d_cache[~touched] == 0.0), "a slot no visible key uses received a gradient"
    _check(d_cache[touched], ref_c[touched], tm, tn, f"{name} dEntries", bnd_c[touched])
    dev.handle.close()
