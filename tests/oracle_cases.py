"""Tiny seeded cases used to check the fp64 oracle against the brute force.

A case is C context tokens (positions 0..C-1) plus one block of T queries at
positions C..C+T-1 that sees keys 0..C+T-1 under the given window / masked
rows.  ``oracle_out(m)`` takes the oracle module as an argument so that the
mutation tests can run it against a copy of the oracle with a planted mistake.
"""
from __future__ import annotations

import math

import numpy as np

from head_latent_attention_qkv_gb300.workloads import MLADims, make_weights
from oracle import brute


def tiny_dims(q_lora=6, style="neox", gate=False, dn=4, dv=4, **kw):
    return MLADims(hidden_size=16, num_heads=2, q_lora_rank=q_lora, kv_lora_rank=8,
                   qk_nope_head_dim=dn, qk_rope_head_dim=4, v_head_dim=dv,
                   rope_style=style, rope_theta=10000.0, use_output_gate=gate,
                   dtype="fp32", **kw)


class TinyCase:
    def __init__(self, d, seed=0, C=5, T=4, window=0, masked=()):
        rng = np.random.Generator(np.random.PCG64(seed))
        self.d = d
        self.w = make_weights(d, rng)
        self.ctx = rng.standard_normal((C, d.hidden_size))
        self.x = rng.standard_normal((T, d.hidden_size))
        self.C, self.T = C, T
        self.pos = np.arange(C, C + T)
        self.kv_len = C + T
        self.window = window
        self.qvis = np.array([0 if i in masked else 1 for i in range(T)], dtype=np.uint8)

    def oracle_out(self, m):
        d, w = self.d, self.w
        ent = m.latent_cache_entries(d, w, np.concatenate([self.ctx, self.x]),
                                     np.arange(self.C + self.T))
        vis = m.visibility(self.pos, self.kv_len, self.window, self.qvis, self.C + self.T)
        return ent, m.block_forward(d, w, self.x, self.pos, [m.expand_keys(d, w, ent)], vis)

    def brute_out(self):
        d, w = self.d, self.w
        hid = np.concatenate([self.ctx, self.x])
        ent = [brute.cache_entry(d, w, hid[j], j) for j in range(self.C + self.T)]
        out = brute.forward(d, w, self.x, self.pos, ent, self.kv_len, self.window, self.qvis)
        return np.array(ent), np.array(out)


def rel_err(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    if a.shape != b.shape or not (np.all(np.isfinite(a)) and np.all(np.isfinite(b))):
        return math.inf
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


BRUTE_CASES = [
    dict(dims=dict(q_lora=6, style="neox"), case=dict(seed=1)),
    dict(dims=dict(q_lora=0, style="interleaved"), case=dict(seed=2)),
    dict(dims=dict(q_lora=6, style="interleaved", gate=True, dv=6), case=dict(seed=3, window=3)),
    dict(dims=dict(q_lora=0, style="neox", gate=True), case=dict(seed=4, window=2, masked=(1,))),
    dict(dims=dict(q_lora=6, style="neox", dn=6, dv=2), case=dict(seed=5, C=7, T=3, window=9)),
]


def brute_cases():
    return [TinyCase(tiny_dims(**c["dims"]), **c["case"]) for c in BRUTE_CASES]
