"""The bench's algorithmic work counts (the numerator of its TFLOP/s and
roofline figures) against an independent count: visible (query, key) pairs
taken from the oracle's visibility mask, projections from the layer's
shapes.  CPU only."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from head_latent_attention_qkv_gb300 import workloads as W  # noqa: E402
from oracle import mla  # noqa: E402


def _visible_pairs(wl, step):
    """Per block, the number of visible (query row, key) pairs, by the
    oracle's mask."""
    T, out = wl.block_len, []
    for b in range(len(step.kv_len)):
        r = slice(b * T, (b + 1) * T)
        n = int(step.kv_len[b])
        vis = mla.visibility(step.block_positions[r], n, int(step.window[b]), step.q_visible[r], n)
        out.append(int(vis.sum()))
    return out


def _expected(wl, shared):
    d = wl.dims
    H, D = d.num_heads, d.hidden_size
    L = d.kv_lora_rank + d.qk_rope_head_dim
    dqk = d.qk_nope_head_dim + d.qk_rope_head_dim
    tok = 2 * D * (d.q_lora_rank + L) + (2 * D * H * d.v_head_dim if d.use_output_gate else 0)
    tok += 2 * d.q_lora_rank * H * dqk                        # q_b
    tok += 2 * H * d.v_head_dim * D                           # o_proj
    if shared:
        tok += 2 * d.kv_lora_rank * H * (d.qk_nope_head_dim + d.v_head_dim)   # the token's own expansion
        per_pair = H * (2 * dqk + 2 * d.v_head_dim)
    else:
        tok += 2 * H * d.qk_nope_head_dim * d.kv_lora_rank + 2 * H * d.kv_lora_rank * d.v_head_dim
        per_pair = H * (2 * L + 2 * d.kv_lora_rank)
    total, attention = 0, []
    for step in wl.steps:
        pairs = sum(_visible_pairs(wl, step))
        attention.append(per_pair * pairs)
        total += tok * len(step.block_positions) + attention[-1]
    ctx = 0 if wl.ctx_hidden is None else len(wl.ctx_hidden)
    total += 2 * D * L * ctx                                  # the context append
    if shared:
        total += 2 * d.kv_lora_rank * H * (d.qk_nope_head_dim + d.v_head_dim) * ctx * len(wl.steps)
    return total, attention


@pytest.mark.parametrize("shared", [False, True])
def test_block_parallel_counts(shared):
    d = W.DEEPSEEK_V3_MLA.replace(num_heads=4, hidden_size=256, q_lora_rank=64)
    wl = W.block_parallel_workload("f", d, 9, batch=2, ctx_len=128, blocks_per_seq=3, block_len=16,
                                   page_size=64, windows=(0, 50))
    s = wl.steps[0]
    qv = s.q_visible.copy()
    qv[[1, 40]] = 0
    import dataclasses
    wl = dataclasses.replace(wl, steps=[dataclasses.replace(s, q_visible=qv)])
    got = bench.algorithmic_flops(wl, shared)
    total, attention = _expected(wl, shared)
    assert got["attention"] == attention
    assert got["total"] == total


def test_deepseek_shaped_totals():
    """The headline's two counts (expanded form 54.4 TFLOP, absorbed 87.0
    TFLOP per step) follow from the same formulas.  The step's structure is
    rebuilt without its tensors: 4 sequences x 1024 proposals of 16 tokens at
    positions 4096..4111 over a 4096-token context, windows 0 / 1024."""
    from types import SimpleNamespace
    nb, T, ctx = 4 * 1024, 16, 4096
    step = SimpleNamespace(block_positions=np.tile(np.arange(ctx, ctx + T), nb),
                           kv_len=np.full(nb, ctx + T), window=np.tile([0, 1024], nb // 2),
                           q_visible=np.ones(nb * T, dtype=np.uint8), append_hidden=None)
    wl = SimpleNamespace(dims=W.DEEPSEEK_V3_MLA, block_len=T, steps=[step],
                         ctx_hidden=np.empty((4 * ctx, 0)))
    for shared, want in ((True, 54.41e12), (False, 87.0e12)):
        got = bench.algorithmic_flops(wl, shared)["total"]
        assert abs(got - want) / want < 2e-3, (shared, got)
