"""Pins of the gradient oracle (oracle/mla_grad.py) on CPU.

The gradient oracle restates the block forward in torch float64 and lets
autograd differentiate it.  It is pinned to the numpy forward oracle, not to
itself: the two forwards must agree to rounding, and every gradient must match
central finite differences of the numpy oracle's forward along random
directions.  Special cases: a fully masked query row passes nothing back (its
upstream gradient is irrelevant), and a context key no query sees gets a zero
gradient.
"""
import zlib

import numpy as np
import pytest

pytest.importorskip("torch")

from head_latent_attention_qkv_gb300.workloads import MLADims, WEIGHT_FIELDS, weight_shapes
from oracle import mla, mla_grad

CASES = {
    "lowrank_interleaved_gate": dict(q_lora_rank=8, rope_style="interleaved", use_output_gate=True),
    "lowrank_neox": dict(q_lora_rank=8, rope_style="neox", use_output_gate=False),
    "noqlora_interleaved": dict(q_lora_rank=0, rope_style="interleaved", use_output_gate=False),
    "noqlora_neox_gate": dict(q_lora_rank=0, rope_style="neox", use_output_gate=True),
}


def _dims(**kw):
    return MLADims(hidden_size=24, num_heads=2, kv_lora_rank=8, qk_nope_head_dim=4,
                   qk_rope_head_dim=4, v_head_dim=4, rope_theta=1e4, dtype="fp32", **kw)


def _weights(d, rng):
    w = {}
    for name, shp in weight_shapes(d).items():
        if shp is None:
            w[name] = None
        elif name.endswith("layernorm"):
            w[name] = 1.0 + 0.1 * rng.standard_normal(shp)
        else:   # large enough that the softmax is far from uniform
            w[name] = 0.3 * rng.standard_normal(shp)
    return w


def _problem(case, window=0, masked=()):
    rng = np.random.default_rng(zlib.crc32(case.encode()))
    d = _dims(**CASES[case])
    w = _weights(d, rng)
    C, T = 5, 3
    ctx = rng.standard_normal((C, d.hidden_size))
    x = rng.standard_normal((T, d.hidden_size))
    ctx_pos = np.arange(C)
    pos = np.arange(C, C + T)
    qv = np.ones(T, dtype=np.uint8)
    qv[list(masked)] = 0
    vis = mla.visibility(pos, C + T, window, qv, C + T)
    g = rng.standard_normal((T, d.hidden_size))
    return d, w, x, pos, ctx, ctx_pos, vis, g, rng


def _np_forward(d, w, x, pos, ctx, ctx_pos, vis):
    hid = np.concatenate([ctx, x])
    entries = mla.latent_cache_entries(d, w, hid, np.concatenate([ctx_pos, pos]))
    return mla.block_forward(d, w, x, pos, [mla.expand_keys(d, w, entries)], vis)


@pytest.mark.parametrize("case", list(CASES))
def test_forward_restatement_matches_numpy_oracle(case):
    d, w, x, pos, ctx, ctx_pos, vis, g, _ = _problem(case, window=4, masked=(1,))
    out, _ = mla_grad.block_gradients(d, w, x, pos, ctx, ctx_pos, vis, g)
    ref = _np_forward(d, w, x, pos, ctx, ctx_pos, vis)
    assert np.max(np.abs(out - ref)) <= 1e-12 * np.max(np.abs(ref))


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("window,masked", [(0, ()), (4, (1,))])
def test_gradients_match_finite_differences_of_numpy_oracle(case, window, masked):
    d, w, x, pos, ctx, ctx_pos, vis, g, rng = _problem(case, window, masked)
    _, grads = mla_grad.block_gradients(d, w, x, pos, ctx, ctx_pos, vis, g)
    params = dict(w, x=x, ctx=ctx)
    eps = 1e-5
    for name in ["x", "ctx"] + [k for k in WEIGHT_FIELDS if w[k] is not None]:
        delta = rng.standard_normal(np.shape(params[name]))

        def loss(sign):
            p = dict(params)
            p[name] = params[name] + sign * eps * delta
            wp = {k: p[k] for k in WEIGHT_FIELDS}
            return np.sum(_np_forward(d, wp, p["x"], pos, p["ctx"], ctx_pos, vis) * g)

        fd = (loss(+1) - loss(-1)) / (2 * eps)
        an = float(np.sum(grads[name] * delta))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_a_masked_row_passes_nothing_back():
    d, w, x, pos, ctx, ctx_pos, vis, g, rng = _problem("lowrank_interleaved_gate", masked=(1,))
    _, g1 = mla_grad.block_gradients(d, w, x, pos, ctx, ctx_pos, vis, g)
    g2_out = g.copy()
    g2_out[1] = 100.0 * rng.standard_normal(d.hidden_size)     # the masked row's upstream gradient
    _, g2 = mla_grad.block_gradients(d, w, x, pos, ctx, ctx_pos, vis, g2_out)
    for k in g1:
        np.testing.assert_array_equal(g1[k], g2[k], err_msg=k)


def test_a_key_no_query_sees_gets_no_gradient():
    # window 3: the queries at positions 5..7 see keys 3..7 only; context keys 0..2 are unseen
    d, w, x, pos, ctx, ctx_pos, vis, g, _ = _problem("lowrank_neox", window=3)
    assert not vis[:, :3].any() and vis[:, 3:].any()
    _, grads = mla_grad.block_gradients(d, w, x, pos, ctx, ctx_pos, vis, g)
    assert np.all(grads["ctx"][:3] == 0.0)
    assert np.all(np.abs(grads["ctx"][3:]).sum(axis=1) > 0)


def _pins_pass(case="lowrank_interleaved_gate"):
    """True when the forward agrees with the numpy oracle and every gradient
    agrees with its finite differences (the two pins above, one problem)."""
    d, w, x, pos, ctx, ctx_pos, vis, g, rng = _problem(case, window=4, masked=(1,))
    out, grads = mla_grad.block_gradients(d, w, x, pos, ctx, ctx_pos, vis, g)
    ref = _np_forward(d, w, x, pos, ctx, ctx_pos, vis)
    if np.max(np.abs(out - ref)) > 1e-12 * np.max(np.abs(ref)):
        return False
    params = dict(w, x=x, ctx=ctx)
    for name in ["x", "ctx"] + [k for k in WEIGHT_FIELDS if w[k] is not None]:
        delta = rng.standard_normal(np.shape(params[name]))
        vals = []
        for sign in (1, -1):
            p = dict(params)
            p[name] = params[name] + sign * 1e-5 * delta
            vals.append(np.sum(_np_forward(d, {k: p[k] for k in WEIGHT_FIELDS}, p["x"], pos,
                                           p["ctx"], ctx_pos, vis) * g))
        fd = (vals[0] - vals[1]) / 2e-5
        an = float(np.sum(grads[name] * delta))
        if abs(fd - an) > 1e-6 * max(1.0, abs(an)):
            return False
    return True


def test_unmutated_gradient_oracle_passes_its_pins():
    assert _pins_pass()


@pytest.mark.parametrize("mutation", ["rope_sign", "gamma_dropped", "scale_nope_only",
                                      "latent_norm_detached", "gate_detached"])
def test_planted_mistakes_fail_the_pins(monkeypatch, mutation):
    import torch
    if mutation == "rope_sign":
        orig = mla_grad._rope
        monkeypatch.setattr(mla_grad, "_rope", lambda x, p, th, st: orig(x, -p, th, st))
    elif mutation == "gamma_dropped":
        monkeypatch.setattr(mla_grad, "_rms", lambda y, gm, eps: y * torch.rsqrt((y * y).mean(-1, keepdim=True) + eps))
    elif mutation == "scale_nope_only":
        monkeypatch.setattr(mla_grad, "_scale", lambda d: 1.0 / float(np.sqrt(d.qk_nope_head_dim)))
    elif mutation == "latent_norm_detached":      # same values, a gradient path cut
        orig = mla_grad._rms
        monkeypatch.setattr(mla_grad, "_rms", lambda y, gm, eps: orig(y, gm, eps).detach() + 0 * y.sum())
    elif mutation == "gate_detached":
        orig = torch.sigmoid
        monkeypatch.setattr(mla_grad.torch, "sigmoid", lambda t: orig(t).detach())
    assert not _pins_pass()


def _latent_problem(seed=3, R=6, J=9, rkv=8, dr=4):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((R, rkv + dr))
    e = rng.standard_normal((J, rkv + dr))
    vis = rng.random((R, J)) < 0.7
    vis[2] = False                       # a row that sees nothing
    vis[0] = True
    do = rng.standard_normal((R, rkv))
    return q, e, vis, 0.4, rkv, do, rng


def test_latent_attention_backward_matches_finite_differences():
    q, e, vis, scale, rkv, do, rng = _latent_problem()
    dq, de = mla_grad.latent_attention_backward(q, e, vis, scale, rkv, do)
    f = lambda qq, ee: np.sum(mla_grad.latent_attention(qq, ee, vis, scale, rkv)[0] * do)
    eps = 1e-6
    for which, grad in (("q", dq), ("e", de)):
        for _ in range(3):
            d = rng.standard_normal(q.shape if which == "q" else e.shape)
            if which == "q":
                fd = (f(q + eps * d, e) - f(q - eps * d, e)) / (2 * eps)
            else:
                fd = (f(q, e + eps * d) - f(q, e - eps * d)) / (2 * eps)
            an = float(np.sum(grad * d))
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (which, fd, an)


def test_latent_attention_forward_matches_a_per_row_softmax():
    # scores, softmax over the visible keys and latent average, row by row
    q, e, vis, scale, rkv, do, _ = _latent_problem()
    o, p = mla_grad.latent_attention(q, e, vis, scale, rkv)
    s = np.where(vis, (q @ e.T) * scale, -np.inf)
    for r in range(q.shape[0]):
        if not vis[r].any():
            assert np.all(o[r] == 0.0)
            continue
        w = np.exp(s[r] - s[r][vis[r]].max())
        w[~vis[r]] = 0.0
        np.testing.assert_allclose(o[r], (w / w.sum()) @ e[:, :rkv], rtol=1e-13, atol=1e-15)


def test_latent_attention_backward_agrees_with_autograd():
    import torch
    q, e, vis, scale, rkv, do, _ = _latent_problem(seed=5)
    dq, de = mla_grad.latent_attention_backward(q, e, vis, scale, rkv, do)
    qt = torch.tensor(q, requires_grad=True)
    et = torch.tensor(e, requires_grad=True)
    vt = torch.tensor(vis)
    s = torch.where(vt, (qt @ et.T) * scale, torch.full((q.shape[0], e.shape[0]), -torch.inf,
                                                        dtype=torch.float64))
    anyk = vt.any(dim=1, keepdim=True)
    p = torch.softmax(torch.where(anyk, s, torch.zeros_like(s)), dim=1) * anyk
    (gq, ge) = torch.autograd.grad(((p @ et[:, :rkv]) * torch.tensor(do)).sum(), [qt, et])
    np.testing.assert_allclose(dq, gq.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(de, ge.numpy(), rtol=1e-12, atol=1e-14)


def test_latent_attention_backward_ignores_rows_without_keys():
    q, e, vis, scale, rkv, do, rng = _latent_problem()
    dq1, de1 = mla_grad.latent_attention_backward(q, e, vis, scale, rkv, do)
    do2 = do.copy()
    do2[2] = 50 * rng.standard_normal(rkv)
    dq2, de2 = mla_grad.latent_attention_backward(q, e, vis, scale, rkv, do2)
    np.testing.assert_array_equal(dq1, dq2)
    np.testing.assert_array_equal(de1, de2)
    assert np.all(dq1[2] == 0.0)


def test_latent_lse_matches_library_logsumexp_and_closed_forms():
    from scipy.special import logsumexp
    q, e, vis, scale, rkv, do, _ = _latent_problem(seed=7)
    lse = mla_grad.latent_lse(q, e, vis, scale)
    s = (q @ e.T) * scale
    for r in range(q.shape[0]):
        if not vis[r].any():
            assert lse[r] == -np.inf
        else:
            assert abs(lse[r] - logsumexp(s[r][vis[r]])) <= 1e-12 * max(1.0, abs(lse[r]))
    # one visible key: the scaled score itself; n equal scores: score + log n
    one = np.zeros_like(vis)
    one[:, 4] = True
    np.testing.assert_allclose(mla_grad.latent_lse(q, e, one, scale), s[:, 4], rtol=1e-14)
    e_eq = np.repeat(e[:1], e.shape[0], axis=0)
    full = np.ones_like(vis)
    np.testing.assert_allclose(mla_grad.latent_lse(q, e_eq, full, scale),
                               (q @ e[0]) * scale + np.log(e.shape[0]), rtol=1e-13)
    # the output and the lse together: exp(s - lse) are the probabilities
    o, p = mla_grad.latent_attention(q, e, vis, scale, rkv)
    rows = vis.any(axis=1)
    np.testing.assert_allclose(np.where(vis[rows], np.exp(s[rows] - lse[rows, None]), 0.0),
                               p[rows], rtol=1e-12, atol=1e-15)


def test_latent_lse_mutation_is_caught():
    # natural log against log2 (a plausible slip in an exp2-domain kernel)
    from scipy.special import logsumexp
    q, e, vis, scale, rkv, do, _ = _latent_problem(seed=8)
    lse = mla_grad.latent_lse(q, e, vis, scale)
    wrong = lse / np.log(2.0)
    r = int(np.nonzero(vis.any(axis=1))[0][0])
    good = logsumexp(((q @ e.T) * scale)[r][vis[r]])
    assert abs(lse[r] - good) < 1e-12 and abs(wrong[r] - good) > 1e-6
