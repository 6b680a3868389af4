"""Scalar pure-Python brute force of the MLA draft-layer forward, for tiny dims.

TEST INFRASTRUCTURE (same rules as ``oracle.mla``).  This is a second,
independent transcription of the same definition with explicit loops over
every index and the ``math`` module only: no numpy, no shared helper with
``oracle.mla``.  It exists so that the numpy oracle is checked against
something other than itself; use it for hidden <= 32, heads <= 2,
ranks <= 8.

Sources: "MLA (Multi-Head Latent Attention)" blog (module layout, split
orders, latent cache, kv_b expansion); "Add config-selectable MLA draft
attention" (masks, empty-row zeroing, gate, RoPE styles).
"""
from __future__ import annotations

import math


def _matvec(W, x):
    """y[o] = sum_i W[o][i] * x[i]  (torch.nn.Linear without bias)."""
    out = []
    for row in W:
        acc = 0.0
        for a, b in zip(row, x):
            acc += a * b
        out.append(acc)
    return out


def _rmsnorm(y, g, eps):
    ms = 0.0
    for v in y:
        ms += v * v
    ms /= len(y)
    inv = 1.0 / math.sqrt(ms + eps)
    return [y[i] * inv * g[i] for i in range(len(y))]


def _rope(x, pos, theta, style):
    n = len(x)
    half = n // 2
    out = list(x)
    for k in range(half):
        ang = pos * theta ** (-(2.0 * k) / n)
        c, s = math.cos(ang), math.sin(ang)
        if style == "neox":
            ia, ib = k, k + half
        else:
            ia, ib = 2 * k, 2 * k + 1
        a, b = x[ia], x[ib]
        out[ia] = a * c - b * s
        out[ib] = b * c + a * s
    return out


def _rows(a):
    return [[float(v) for v in r] for r in a]


def cache_entry(d, w, h, pos):
    """[RMSNorm(kv_c) | RoPE(k_pe)] for one hidden vector ``h``."""
    r, L = d.kv_lora_rank, d.kv_lora_rank + d.qk_rope_head_dim
    if d.q_lora_rank > 0:
        Wkv = _rows(w["fused_qkv_a_proj"])[d.q_lora_rank:d.q_lora_rank + L]
    else:
        Wkv = _rows(w["kv_a_proj_with_mqa"])
    kv = _matvec(Wkv, [float(v) for v in h])
    c = _rmsnorm(kv[:r], [float(v) for v in w["kv_a_layernorm"]], d.rms_norm_eps)
    return c + _rope(kv[r:], pos, d.rope_theta, d.rope_style)


def forward(d, w, x_block, positions, entries, kv_len, window, q_visible):
    """Output rows [T][D] of one block.

    ``entries`` are the cache entries of keys 0..J-1 in logical order (lists of
    floats).  Key j is visible to query i iff q_visible[i] and j < kv_len and
    (window == 0 or positions[i] - j < window)."""
    H, dn, dr, dv = d.num_heads, d.qk_nope_head_dim, d.qk_rope_head_dim, d.v_head_dim
    r = d.kv_lora_rank
    scale = d.softmax_scale if getattr(d, "softmax_scale", 0.0) else 1.0 / math.sqrt(dn + dr)
    Wkvb = _rows(w["kv_b_proj"])
    Wo = _rows(w["o_proj"])
    keys_nope, vals, kpes = [], [], []
    for e in entries:
        e = [float(v) for v in e]
        kvb = _matvec(Wkvb, e[:r])
        kn, vv = [], []
        for h in range(H):
            base = h * (dn + dv)
            kn.append(kvb[base:base + dn])
            vv.append(kvb[base + dn:base + dn + dv])
        keys_nope.append(kn)
        vals.append(vv)
        kpes.append(e[r:r + dr])
    out = []
    for i, xi in enumerate(x_block):
        xi = [float(v) for v in xi]
        if d.q_lora_rank > 0:
            Wa = _rows(w["fused_qkv_a_proj"])[:d.q_lora_rank]
            qc = _rmsnorm(_matvec(Wa, xi), [float(v) for v in w["q_a_layernorm"]], d.rms_norm_eps)
            q = _matvec(_rows(w["q_b_proj"]), qc)
        else:
            q = _matvec(_rows(w["q_proj"]), xi)
        o_cat = []
        for h in range(H):
            qh = q[h * (dn + dr):(h + 1) * (dn + dr)]
            q_nope, q_pe = qh[:dn], _rope(qh[dn:], int(positions[i]), d.rope_theta, d.rope_style)
            scores = []
            for j in range(len(entries)):
                vis = (bool(q_visible[i]) and j < kv_len
                       and (window == 0 or int(positions[i]) - j < window))
                if not vis:
                    continue
                s = 0.0
                for t in range(dn):
                    s += q_nope[t] * keys_nope[j][h][t]
                for t in range(dr):
                    s += q_pe[t] * kpes[j][t]
                scores.append((j, s * scale))
            oh = [0.0] * dv
            if scores:
                mx = max(s for _, s in scores)
                den = 0.0
                for _, s in scores:
                    den += math.exp(s - mx)
                for j, s in scores:
                    p = math.exp(s - mx) / den
                    for t in range(dv):
                        oh[t] += p * vals[j][h][t]
            o_cat.extend(oh)
        if d.use_output_gate:
            g = _matvec(_rows(w["gate_proj"]), xi)
            o_cat = [o_cat[k] / (1.0 + math.exp(-g[k])) for k in range(len(o_cat))]
        out.append(_matvec(Wo, o_cat))
    return out
