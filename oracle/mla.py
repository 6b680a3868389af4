"""fp64 CPU oracle of the MLA draft-layer forward (expanded, non-absorbed form).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` import this
module.  The library's product path never calls it and shares no code with
it.

What it computes, in the order the sources give it:

* "MLA (Multi-Head Latent Attention)" blog, ``DeepseekV2MLAAttention.__init__``
  and ``MultiHeadLatentAttentionWrapper.forward``: the low-rank query
  (``fused_qkv_a_proj`` split into ``[q_lora_rank | kv_lora_rank +
  qk_rope_head_dim]``, ``q_a_layernorm``, ``q_b_proj``) or, without
  ``q_lora_rank``, ``q_proj`` plus ``kv_a_proj_with_mqa``; the latent split
  ``kv_c | k_pe``; ``kv_a_layernorm`` on ``kv_c`` only; RoPE on the query's
  rope slice and on the single shared ``k_pe`` head; ``o_proj`` at the end.
* Same blog, ``do_kv_cache_update`` / ``concat_and_cache_mla``: a cache entry
  is ``[kv_c_normed | k_pe]`` (512 + 64 = 576 wide for DeepSeek dims).
* Same blog, ``forward_mha``: ``kv_b_proj`` expands the latent into
  ``[H, qk_nope + v_head]`` per token, split into ``k_nope`` and ``v``; the
  full key is ``[k_nope | k_pe]`` with ``k_pe`` shared by all heads.
* Same blog, ``forward_impl`` (MQA branch) and ``forward_mqa``: the absorbed
  form (``q_nope @ W_UK``, attention over the latent, ``W_UV`` up-projection).
  Kept here only as a second form for the absorbed == expanded invariant.
* "Add config-selectable MLA draft attention" (SpecForge PR #758), Summary and
  Structure: full / sliding masks, zeroing of fully-masked queries, optional
  output gate, NeoX or interleaved rotation.
* "extract GQA/MLA attention into reusable layers" (SpecForge PR #1026),
  Modifications: masks applied by logical position; empty queries zeroed
  before ``o_proj``.

Readings where the pages are silent (each also listed in the design notes):
the softmax scale is ``1/sqrt(qk_nope + qk_rope)``; a key at logical position
``j`` is visible to a query at position ``p`` iff ``j < kv_len`` and (full mask
or ``p - j < window``) and the query row is not masked; the gate is
``o * sigmoid(x @ gate_proj.T)`` on the ``[H * v_head]`` attention output
before ``o_proj``; interleaved RoPE rotates pairs ``(2i, 2i+1)`` in place.

Every array is promoted to float64.  Dims are read from any object with the
attributes of ``MLADims`` (hidden_size, num_heads, q_lora_rank, ...); weights
are a dict of arrays in ``torch.nn.Linear`` layout ``[out, in]``.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(a):
    return np.asarray(a, dtype=F64)


def softmax_scale(d) -> float:
    """Reading: 1/sqrt(qk_nope_head_dim + qk_rope_head_dim) unless given."""
    if getattr(d, "softmax_scale", 0.0):
        return float(d.softmax_scale)
    return 1.0 / np.sqrt(d.qk_nope_head_dim + d.qk_rope_head_dim)


# ---------------------------------------------------------------------------
# Normalisation and rotation
# ---------------------------------------------------------------------------
def rms_norm(y, gamma, eps):
    """RMSNorm over the last axis: y / sqrt(mean(y^2) + eps) * gamma.

    MLA blog, ``DeepseekV2MLAAttention.__init__`` (``kv_a_layernorm`` =
    RMSNorm(kv_lora_rank, eps=rms_norm_eps)) and the wrapper's forward
    (``q_a_layernorm`` on ``q_c``)."""
    y = _f64(y)
    return y / np.sqrt(np.mean(y * y, axis=-1, keepdims=True) + eps) * _f64(gamma)


def rope_angles(positions, rope_dim, theta):
    """angle[n, i] = pos[n] * theta^(-2i/rope_dim), i in [0, rope_dim/2)."""
    i = np.arange(rope_dim // 2, dtype=F64)
    inv_freq = F64(theta) ** (-2.0 * i / rope_dim)
    return _f64(positions)[:, None] * inv_freq[None, :]


def apply_rope(x, positions, theta, style):
    """Rotate the last axis of ``x`` ([N, ..., rope_dim]) by each row's position.

    Pair k is rotated by angle[n, k]: (a, b) -> (a cos - b sin, b cos + a sin).
    NeoX pairs element k with k + rope_dim/2; interleaved pairs 2k with 2k+1
    and writes the result back in the same interleaved slots.
    Sources: PR #758 Summary ("partial interleaved or NeoX RoPE"); MLA blog,
    wrapper forward (only ``q[..., qk_nope:]`` and ``k_pe`` are rotated)."""
    x = _f64(x)
    rd = x.shape[-1]
    half = rd // 2
    ang = rope_angles(positions, rd, theta)
    shape = (x.shape[0],) + (1,) * (x.ndim - 2) + (half,)
    cos = np.cos(ang).reshape(shape)
    sin = np.sin(ang).reshape(shape)
    if style == "neox":
        ia, ib = slice(0, half), slice(half, rd)
    elif style == "interleaved":
        ia, ib = slice(0, rd, 2), slice(1, rd, 2)
    else:
        raise ValueError(style)
    a, b = x[..., ia], x[..., ib]
    out = np.empty_like(x)
    out[..., ia] = a * cos - b * sin
    out[..., ib] = b * cos + a * sin
    return out


# ---------------------------------------------------------------------------
# Projections
# ---------------------------------------------------------------------------
def kv_a_weight(d, w):
    """The rows producing ``[kv_c | k_pe]``: the last kv_lora_rank+qk_rope rows
    of ``fused_qkv_a_proj`` (its output is split [q_lora_rank, kv_lora_rank +
    qk_rope_head_dim]) or ``kv_a_proj_with_mqa`` when there is no q_lora_rank."""
    if d.q_lora_rank > 0:
        return _f64(w["fused_qkv_a_proj"])[d.q_lora_rank:]
    return _f64(w["kv_a_proj_with_mqa"])


def latent_cache_entries(d, w, hidden, positions):
    """What ``concat_and_cache_mla`` stores per token: ``[RMSNorm(kv_c) | RoPE(k_pe)]``.

    MLA blog, wrapper forward: ``kv_c, k_pe = kv_lora.split([kv_lora_rank,
    qk_rope_head_dim])``; the cache gets the *normed* kv_c; k_pe is rotated
    with the token's own position.  Returns [N, kv_lora_rank + qk_rope]."""
    kv = _f64(hidden) @ kv_a_weight(d, w).T
    c = rms_norm(kv[:, :d.kv_lora_rank], w["kv_a_layernorm"], d.rms_norm_eps)
    k_pe = apply_rope(kv[:, d.kv_lora_rank:], positions, d.rope_theta, d.rope_style)
    return np.concatenate([c, k_pe], axis=1)


def round_to_dtype(d, x):
    """The value a typed tensor of the layer's dtype holds for fp64 ``x``.

    The method stores two tensors in the model dtype: the latent cache (MLA
    blog, ``do_kv_cache_update`` passes ``kv_cache_dtype`` to
    ``concat_and_cache_mla``; ``get_kv_cache_spec`` types the cache with it)
    and the attention output (``MLAAttention.forward`` allocates it with
    ``dtype=q.dtype``).  For bf16 layers each value is rounded to the nearest
    bf16 (8 significant bits, ties to even); fp32 layers keep fp64 here, their
    rounding being far below that configuration's tolerance."""
    x = _f64(x)
    if getattr(d, "dtype", "fp32") != "bf16":
        return x
    m, ex = np.frexp(x)                          # x = m * 2^ex, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), ex - 8)  # 8 significant bits, ties to even


def project_queries(d, w, x, positions):
    """Rotated queries ``[N, H, qk_nope + qk_rope]`` (nope first, rope last).

    MLA blog, wrapper forward: q_c = first q_lora_rank outputs of
    ``fused_qkv_a_proj``; q = q_b_proj(q_a_layernorm(q_c)); otherwise
    q = q_proj(x).  Then view as [tokens, heads, qk_head_dim] and rotate
    ``q[..., qk_nope:]``."""
    x = _f64(x)
    H, dn, dr = d.num_heads, d.qk_nope_head_dim, d.qk_rope_head_dim
    if d.q_lora_rank > 0:
        q_c = x @ _f64(w["fused_qkv_a_proj"])[:d.q_lora_rank].T
        q_c = rms_norm(q_c, w["q_a_layernorm"], d.rms_norm_eps)
        q = q_c @ _f64(w["q_b_proj"]).T
    else:
        q = x @ _f64(w["q_proj"]).T
    q = q.reshape(x.shape[0], H, dn + dr)
    q[..., dn:] = apply_rope(q[..., dn:], positions, d.rope_theta, d.rope_style)
    return q


def expand_keys(d, w, entries):
    """Expand latent cache entries into per-head keys and values.

    MLA blog, ``forward_mha``: ``kv_b_proj(kv_c_normed).view(-1, H, qk_nope +
    v_head)`` split ``[qk_nope, v_head]``; ``_concat_k_nope_k_pe`` appends the
    shared k_pe to every head.  Returns K [H, J, qk_nope+qk_rope] and
    V [H, J, v_head]."""
    e = _f64(entries)
    H, dn, dv, r = d.num_heads, d.qk_nope_head_dim, d.v_head_dim, d.kv_lora_rank
    J = e.shape[0]
    c, k_pe = e[:, :r], e[:, r:]
    kvb = (c @ _f64(w["kv_b_proj"]).T).reshape(J, H, dn + dv)
    k_nope, v = kvb[..., :dn], kvb[..., dn:]
    K = np.concatenate([k_nope, np.broadcast_to(k_pe[:, None, :], (J, H, k_pe.shape[1]))], axis=-1)
    return np.ascontiguousarray(K.transpose(1, 0, 2)), np.ascontiguousarray(v.transpose(1, 0, 2))


# ---------------------------------------------------------------------------
# Masking and attention
# ---------------------------------------------------------------------------
def visibility(positions, kv_len, window, q_visible, num_keys):
    """vis[i, j]: query i (logical position positions[i]) sees key j.

    PR #758 / PR #1026: full or sliding masks applied by logical position and
    fully masked query rows.  Reading: key j is visible iff j < kv_len, and
    window == 0 (full) or positions[i] - j < window, and q_visible[i]."""
    j = np.arange(num_keys)[None, :]
    p = np.asarray(positions, dtype=np.int64)[:, None]
    vis = j < int(kv_len)
    if int(window) > 0:
        vis = vis & ((p - j) < int(window))
    vis = vis & (np.asarray(q_visible).astype(bool)[:, None])
    return np.broadcast_to(vis, (p.shape[0], num_keys)).copy()


def attend(d, q, segments, vis):
    """Scaled dot-product attention of rotated queries over expanded keys.

    q: [T, H, dqk]; segments: list of (K [H, J_s, dqk], V [H, J_s, dv]) whose
    concatenation along J is the key sequence in logical order; vis: [T, J].
    Softmax over the visible keys (max-subtracted); a row with no visible key
    is set to exactly zero (PR #758 Structure: "fully-masked-query zeroing").
    Returns o [T, H, dv]."""
    q = _f64(q)
    qh = q.transpose(1, 0, 2)                                     # [H, T, dqk]
    s = np.concatenate([qh @ K.transpose(0, 2, 1) for K, _ in segments], axis=2)
    s = s * softmax_scale(d)
    s = np.where(vis[None, :, :], s, -np.inf)                     # [H, T, J]
    with np.errstate(invalid="ignore"):
        p = np.exp(s - s.max(axis=2, keepdims=True))              # NaN on rows with no key
        p = p / p.sum(axis=2, keepdims=True)
    o = np.zeros((qh.shape[0], qh.shape[1], segments[0][1].shape[2]))
    start = 0
    for K, V in segments:
        J = K.shape[1]
        o += p[:, :, start:start + J] @ V
        start += J
    o[:, ~vis.any(axis=1), :] = 0.0                               # fully masked queries
    return o.transpose(1, 0, 2)


def output_projection(d, w, x, o):
    """Concatenate heads head-major to [T, H*v_head], apply the optional gate
    (reading: ``o * sigmoid(x @ gate_proj.T)``), then ``o_proj`` (no bias).
    MLA blog, ``DeepseekV2MLAAttention.__init__`` (o_proj: H*v_head -> hidden)
    and wrapper forward (``return self.o_proj(attn_out)``); PR #758 (gate)."""
    T = o.shape[0]
    o = _f64(o).reshape(T, d.num_heads * d.v_head_dim)
    if d.use_output_gate:
        g = _f64(x) @ _f64(w["gate_proj"]).T
        o = o * (1.0 / (1.0 + np.exp(-g)))
    return o @ _f64(w["o_proj"]).T


def block_forward(d, w, x, positions, segments, vis):
    """The draft layer's attention output for one block of queries.

    x [T, D] block hidden states; positions [T]; segments: expanded keys
    (see ``expand_keys``) in logical order; vis [T, J].  Returns [T, D]."""
    q = project_queries(d, w, x, positions)
    o = attend(d, q, segments, vis)
    return output_projection(d, w, x, o)


# ---------------------------------------------------------------------------
# Absorbed form (second route, for the absorbed == expanded invariant only)
# ---------------------------------------------------------------------------
def split_kv_b(d, w):
    """W_UK [H, qk_nope, kv_lora_rank] and W_UV [H, v_head, kv_lora_rank]: the
    per-head row blocks of kv_b_proj viewed [H, qk_nope + v_head, r_kv] and
    split [qk_nope, v_head] (MLA blog, ``forward_mha`` view/split; the MQA
    branch uses them as ``W_UK_T`` and ``_v_up_proj``)."""
    H, dn, dv, r = d.num_heads, d.qk_nope_head_dim, d.v_head_dim, d.kv_lora_rank
    kvb = _f64(w["kv_b_proj"]).reshape(H, dn + dv, r)
    return kvb[:, :dn, :], kvb[:, dn:, :]


def attend_absorbed(d, w, q, entries, vis):
    """MLA blog, ``forward_impl`` MQA branch + ``forward_mqa``: q_nope is
    mapped into the latent space (``q_nope @ W_UK``), scores are taken against
    the raw cache entries [c | k_pe], the output is a latent average of c and
    ``W_UV`` maps it to v_head.  Returns o [T, H, dv]."""
    q = _f64(q)
    e = _f64(entries)
    dn, r = d.qk_nope_head_dim, d.kv_lora_rank
    W_UK, W_UV = split_kv_b(d, w)
    q_lat = np.einsum("thn,hnc->thc", q[..., :dn], W_UK)             # [T, H, r]
    q_abs = np.concatenate([q_lat, q[..., dn:]], axis=-1)             # [T, H, r + dr]
    s = np.einsum("thc,jc->htj", q_abs, e) * softmax_scale(d)
    s = np.where(vis[None], s, -np.inf)
    with np.errstate(invalid="ignore"):
        p = np.exp(s - s.max(axis=2, keepdims=True))
        p = p / p.sum(axis=2, keepdims=True)
    o_lat = np.einsum("htj,jc->thc", p, e[:, :r])
    o = np.einsum("thc,hvc->thv", o_lat, W_UV)
    o[~vis.any(axis=1)] = 0.0
    return o
