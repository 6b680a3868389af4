"""fp64 CPU oracle of the gradients of the MLA draft-layer forward.

TEST INFRASTRUCTURE (the layer's backward is the next step of the hot path;
this module only states what it must compute).  Only tests import it.

What it computes: for one query block of ``T`` tokens attending its context
(the tokens before it, whose latents come from their own hidden states) and
its own latents, the gradients of ``L = sum(out * grad_out)`` with respect to
the block's hidden states, the context hidden states and every weight of the
layer, where ``out`` is the layer's output for the block.  The forward is the
same expanded form as ``oracle.mla`` (MLA blog, wrapper forward and
``forward_mha``; SpecForge PR #758 masks, gate and zeroing), restated here in
torch float64 so that autograd differentiates it; storage in the layer dtype
(the bf16 cache and output) is not part of this function: its derivative is
taken as the identity, the usual reading when training through a rounded
tensor.

A fully masked query row outputs exactly zero, so nothing flows back through
it; a key no query sees receives no gradient.  The tests pin this module to
``oracle.mla`` by value (forward) and by central finite differences of
``oracle.mla``'s forward (gradients), not to itself.

``latent_attention_backward`` states the attention part alone in the latent
space (what a backward kernel over the latent cache computes: dQ_abs and the
gradient of the cache entries, which are keys and values at once), written as
explicit formulas and pinned by finite differences and by autograd.
"""
from __future__ import annotations

import numpy as np
import torch

WEIGHTS = ("fused_qkv_a_proj", "q_a_layernorm", "q_b_proj", "q_proj", "kv_a_proj_with_mqa",
           "kv_a_layernorm", "kv_b_proj", "gate_proj", "o_proj")


def _t(a):
    return torch.as_tensor(np.asarray(a, dtype=np.float64))


def _rms(y, gamma, eps):
    return y * torch.rsqrt((y * y).mean(dim=-1, keepdim=True) + eps) * gamma


def _rope(x, positions, theta, style):
    """Pairs rotated by pos * theta^(-2k/rope_dim): NeoX (k, k + half), or
    interleaved (2k, 2k + 1) written back in place."""
    rd = x.shape[-1]
    half = rd // 2
    k = torch.arange(half, dtype=torch.float64)
    ang = positions.to(torch.float64)[:, None] * (float(theta) ** (-2.0 * k / rd))[None, :]
    shape = (x.shape[0],) + (1,) * (x.dim() - 2) + (half,)
    cos, sin = torch.cos(ang).reshape(shape), torch.sin(ang).reshape(shape)
    if style == "neox":
        a, b = x[..., :half], x[..., half:]
        return torch.cat([a * cos - b * sin, b * cos + a * sin], dim=-1)
    a, b = x[..., 0::2], x[..., 1::2]
    return torch.stack([a * cos - b * sin, b * cos + a * sin], dim=-1).reshape(x.shape)


def _scale(d):
    if getattr(d, "softmax_scale", 0.0):
        return float(d.softmax_scale)
    return 1.0 / float(np.sqrt(d.qk_nope_head_dim + d.qk_rope_head_dim))


def block_forward(d, w, x, positions, ctx, ctx_positions, vis):
    """The layer output [T, D] for one block (torch float64, differentiable).

    x [T, D] block hidden, positions [T]; ctx [C, D] context hidden,
    ctx_positions [C]; the block's keys are the C context latents followed by
    its own T latents (logical positions 0 .. C + T - 1); vis [T, C + T] bool."""
    H, dn, dr, dv, r = (d.num_heads, d.qk_nope_head_dim, d.qk_rope_head_dim, d.v_head_dim,
                        d.kv_lora_rank)
    # latents of every key: [RMSNorm(kv_c) | RoPE(k_pe)]
    hid = torch.cat([ctx, x], dim=0)
    pos = torch.cat([ctx_positions, positions])
    w_kva = w["fused_qkv_a_proj"][d.q_lora_rank:] if d.q_lora_rank > 0 else w["kv_a_proj_with_mqa"]
    kv = hid @ w_kva.T
    c = _rms(kv[:, :r], w["kv_a_layernorm"], d.rms_norm_eps)
    k_pe = _rope(kv[:, r:], pos, d.rope_theta, d.rope_style)
    # expanded keys and values
    J = hid.shape[0]
    kvb = (c @ w["kv_b_proj"].T).reshape(J, H, dn + dv)
    K = torch.cat([kvb[..., :dn], k_pe[:, None, :].expand(J, H, dr)], dim=-1)   # [J, H, dqk]
    V = kvb[..., dn:]                                                          # [J, H, dv]
    # rotated queries
    if d.q_lora_rank > 0:
        q_c = _rms(x @ w["fused_qkv_a_proj"][:d.q_lora_rank].T, w["q_a_layernorm"], d.rms_norm_eps)
        q = q_c @ w["q_b_proj"].T
    else:
        q = x @ w["q_proj"].T
    q = q.reshape(x.shape[0], H, dn + dr)
    q = torch.cat([q[..., :dn], _rope(q[..., dn:], positions, d.rope_theta, d.rope_style)], dim=-1)
    # masked softmax; rows with no visible key are exactly zero
    s = torch.einsum("thd,jhd->htj", q, K) * _scale(d)
    vis_t = torch.as_tensor(vis, dtype=torch.bool)
    s = torch.where(vis_t[None], s, torch.full_like(s, -torch.inf))
    any_key = vis_t.any(dim=1)
    s = torch.where(any_key[None, :, None], s, torch.zeros_like(s))   # avoid 0/0 on empty rows
    p = torch.softmax(s, dim=2) * any_key[None, :, None]
    o = torch.einsum("htj,jhv->thv", p, V).reshape(x.shape[0], H * dv)
    if d.use_output_gate:
        o = o * torch.sigmoid(x @ w["gate_proj"].T)
    return o @ w["o_proj"].T


def block_gradients(d, weights, x, positions, ctx, ctx_positions, vis, grad_out):
    """Gradients of sum(out * grad_out) for one block.

    Inputs are numpy arrays (any float dtype, promoted to fp64); weights is a
    dict in ``torch.nn.Linear`` layout with None for unused fields.  Returns
    (out, grads) with numpy fp64 arrays: grads['x'], grads['ctx'] and one
    entry per weight that the configuration uses."""
    w = {k: _t(v).requires_grad_() for k, v in weights.items() if v is not None}
    xt, ct = _t(x).requires_grad_(), _t(ctx).requires_grad_()
    out = block_forward(d, w, xt, torch.as_tensor(np.asarray(positions, np.int64)), ct,
                        torch.as_tensor(np.asarray(ctx_positions, np.int64)), vis)
    names = ["x", "ctx"] + list(w)
    g = torch.autograd.grad((out * _t(grad_out)).sum(), [xt, ct] + list(w.values()),
                            allow_unused=True)
    grads = {n: (np.zeros(tuple(t.shape)) if gi is None else gi.detach().numpy())
             for n, t, gi in zip(names, [xt, ct] + list(w.values()), g)}
    return out.detach().numpy(), grads


# ---------------------------------------------------------------------------
# The latent-space attention and its backward (what an attention-backward
# kernel over the latent cache computes)
# ---------------------------------------------------------------------------
def latent_attention(q_abs, entries, vis, scale, rkv):
    """Absorbed attention over the latent cache (MLA blog, forward_mqa): rows
    of Q_abs [R, L] score every cache entry [J, L] (L = rkv + rope), softmax
    over the visible ones (vis [R, J]), output the probability-weighted latent
    c = entries[:, :rkv]; a row with no visible key is exactly zero.
    Returns (o_lat [R, rkv], p [R, J])."""
    q = np.asarray(q_abs, np.float64)
    e = np.asarray(entries, np.float64)
    s = np.where(vis, (q @ e.T) * scale, -np.inf)
    any_key = vis.any(axis=1)
    m = np.where(any_key, s.max(axis=1), 0.0)
    with np.errstate(invalid="ignore"):
        p = np.where(vis, np.exp(s - m[:, None]), 0.0)
    l = p.sum(axis=1)
    p = np.where(any_key[:, None], p / np.where(any_key, l, 1.0)[:, None], 0.0)
    return p @ e[:, :rkv], p


def latent_lse(q_abs, entries, vis, scale):
    """Per row, the natural log of the sum over visible keys of exp(scale *
    score): what the decode attention returns beside its output (MLA blog,
    forward_mqa: decode_attention_fwd fills ``lse``), the statistic that
    merges attention over disjoint key ranges (forward_mha,
    merge_attn_states).  Computed as max + log(sum(exp(s - max))); -inf for a
    row with no visible key.  Returns lse [R]."""
    q = np.asarray(q_abs, np.float64)
    e = np.asarray(entries, np.float64)
    s = np.where(vis, (q @ e.T) * scale, -np.inf)
    any_key = vis.any(axis=1)
    m = np.where(any_key, s.max(axis=1), 0.0)
    with np.errstate(invalid="ignore"):
        l = np.where(vis, np.exp(s - m[:, None]), 0.0).sum(axis=1)
    with np.errstate(divide="ignore"):
        return np.where(any_key, m + np.log(np.where(any_key, l, 1.0)), -np.inf)


def latent_attention_backward(q_abs, entries, vis, scale, rkv, d_o_lat):
    """Gradients of sum(o_lat * d_o_lat) for ``latent_attention``.

    With P the probabilities, V = entries[:, :rkv] and dO = d_o_lat:
      dP = dO V^T;  dS = P * (dP - rowsum(dP * P))   (softmax derivative,
      rowsum(dP * P) = rowsum(dO * o_lat));
      dQ_abs = scale * dS E;  dE = scale * dS^T Q_abs, plus P^T dO on the
      first rkv columns (the entries are both keys and values).
    Rows with no visible key have P = 0 and pass nothing back.
    Returns (dQ_abs [R, L], dE [J, L])."""
    q = np.asarray(q_abs, np.float64)
    e = np.asarray(entries, np.float64)
    do = np.asarray(d_o_lat, np.float64)
    o, p = latent_attention(q, e, vis, scale, rkv)
    dp = do @ e[:, :rkv].T
    ds = p * (dp - np.sum(do * o, axis=1, keepdims=True))
    dq = scale * (ds @ e)
    de = scale * (ds.T @ q)
    de[:, :rkv] += p.T @ do
    return dq, de
