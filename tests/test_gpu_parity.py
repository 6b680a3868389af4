"""CUDA path vs the fp64 oracle on the same seeded inputs (needs a GB300).

Small variants of every workload run whole (ragged contexts, partial pages
and tiles, masked rows, sliding windows, two cached blocks); the full-size
workloads run in the benchmark's launch configuration and are checked on a
seeded sample of blocks the oracle computes one by one.  See tests/parity.py
for the tolerances and the exact checks.
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


@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_small_workload_matches_oracle(name):
    from tests.parity import check_workload
    wl = workloads.make_workload(name, "small")
    check_workload(wl)


def _sample_blocks(wl, per_step, seed=0):
    rng = np.random.default_rng(seed)
    out = []
    for s in wl.steps:
        nb = len(s.kv_len)
        pick = rng.choice(nb, size=min(per_step, nb), replace=False)
        out.append(sorted(int(b) for b in pick))
    return out


FULL = [("tiny_fp32", None), ("qwen3_4b_prefill", None), ("qwen3_4b_sliding_gate", None),
        ("qwen3_4b_cached_decode", 8), ("deepseek_v3_block_parallel", 8), ("qwen3_4b_decode_t1", 8)]


@pytest.mark.parametrize("name,per_step", FULL)
def test_full_size_workload_matches_oracle_on_sampled_blocks(name, per_step):
    from tests.parity import check_workload
    wl = workloads.make_workload(name, "full")
    sample = None if per_step is None else _sample_blocks(wl, per_step)
    if name == "deepseek_v3_block_parallel":
        # keep both mask kinds in the sample: even blocks full, odd blocks sliding
        step = wl.steps[0]
        sample = [sorted(set(sample[0]) | {0, 1, len(step.kv_len) - 1})]
    check_workload(wl, sample)


@pytest.mark.parametrize("case", ["decode_T6", "sliding_T5_gate"])
def test_partial_query_tiles_match_oracle(case):
    """block_len x num_heads not a multiple of the 128-row attention tile: the
    last tile of every block is padded (its extra rows masked and not written)."""
    from tests.parity import check_workload
    W = workloads
    if case == "decode_T6":          # 192 rows per block: one full and one half tile
        wl = W.cached_decode_workload(case, W.QWEN3_4B_MLA, 6, batch=3, prefill_len=256,
                                      len_lo=60, len_hi=250, block_len=6, num_blocks=2,
                                      page_size=64)
    else:                            # 160 rows, sliding window, gate, NeoX, a masked row
        d = W.QWEN3_4B_MLA.replace(use_output_gate=True, rope_style="neox")
        wl = W.prefill_workload(case, d, 7, [300, 129, 17], 5, page_size=128, window=100,
                                masked_rows=lambda s: (1,) if s == 1 else ())
    check_workload(wl)


@pytest.mark.parametrize("page_size", [16, 256])
def test_page_sizes_match_oracle(page_size):
    """Pages smaller than the 128-key tile (one copy per page segment) and
    larger ones (several tiles per page), with ragged contexts and permuted
    physical pages."""
    from tests.parity import check_workload
    W = workloads
    wl = W.prefill_workload(f"pages{page_size}", W.QWEN3_4B_MLA, 9, [150, 40, 333], 16,
                            page_size=page_size)
    check_workload(wl)


@pytest.mark.parametrize("rope", ["neox", "interleaved"])
def test_many_block_tokens_split_queries_in_the_projection(rope):
    """1024 block tokens (64 blocks of 16): the q_b projection runs as the
    persistent GEMM whose epilogue splits the heads and rotates the RoPE dims
    itself (both pairings), instead of the row kernel; sampled blocks against
    the oracle."""
    from tests.parity import check_workload
    W = workloads
    wl = W.cached_decode_workload(f"q_split_{rope}", W.QWEN3_4B_MLA.replace(rope_style=rope), 21,
                                  batch=64, prefill_len=300, len_lo=100, len_hi=300, block_len=16,
                                  num_blocks=1, page_size=128)
    check_workload(wl, _sample_blocks(wl, 6, seed=3))


def _scaled_workload(gain_q, gain_kv, seed=12):
    """Config 1 small with the RMSNorm gains scaled and hidden states carrying
    +-1e3 outliers (bf16-representable values on both sides)."""
    import dataclasses
    W = workloads
    wl = W.make_workload("qwen3_4b_prefill", "small")
    rnd = lambda x: W.bf16_bits_to_f32(W.bf16_bits(np.asarray(x, np.float32)))
    w = dict(wl.weights)
    w["q_a_layernorm"] = rnd(w["q_a_layernorm"] * gain_q)
    w["kv_a_layernorm"] = rnd(w["kv_a_layernorm"] * gain_kv)
    rng = np.random.default_rng(seed)
    ctx = wl.ctx_hidden.copy()
    ctx[rng.integers(0, ctx.shape[0], 40), rng.integers(0, ctx.shape[1], 40)] = rng.choice([-1e3, 1e3], 40)
    step = wl.steps[0]
    blk = step.block_hidden.copy()
    blk[rng.integers(0, blk.shape[0], 8), rng.integers(0, blk.shape[1], 8)] = rng.choice([-1e3, 1e3], 8)
    return dataclasses.replace(wl, name=f"gains{gain_q}x{gain_kv}_outliers", weights=w,
                               ctx_hidden=ctx, steps=[dataclasses.replace(step, block_hidden=blk)])


def test_fp16_intermediates_stay_in_range_with_large_gains_and_outliers():
    """The bf16 layer keeps the normalised q_c, q_nope, o_lat and o (and the
    weights they meet) in fp16, whose largest finite value is 65504.  Bounds
    that follow from the RMSNorm (an element of a normalised row is at most
    sqrt(width) times its gain): |q_c| <= sqrt(q_lora_rank) max|gamma_q|,
    |o_lat| <= sqrt(kv_lora_rank) max|gamma_kv| (a convex combination of
    normalised latents).  With both gains scaled 30x and +-1e3 outliers in the
    hidden states every intermediate stays finite and inside these bounds."""
    from head_latent_attention_qkv_gb300 import _lib, api
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload
    wl = _scaled_workload(30.0, 30.0)
    dev = DeviceWorkload(wl)
    out = dev.run_all()[0]
    torch.cuda.synchronize()
    assert api.mla_get_device_status(dev.handle) == 0
    assert torch.isfinite(out.float()).all()
    d = wl.dims
    M = out.shape[0]
    ws = dev.handle._ws
    oo = api.mla_forward_workspace_offset(dev.handle, M, _lib.MLA_WS_O_LAT)
    qo = api.mla_forward_workspace_offset(dev.handle, M, _lib.MLA_WS_Q_ABS)
    o_lat = ws[oo:oo + M * d.num_heads * d.kv_lora_rank * 2].view(torch.float16).float()
    q_abs = ws[qo:qo + M * d.num_heads * d.cache_dim * 2].view(torch.bfloat16).float()
    assert torch.isfinite(o_lat).all() and torch.isfinite(q_abs).all()
    bound = np.sqrt(d.kv_lora_rank) * float(np.abs(wl.weights["kv_a_layernorm"]).max())
    assert float(o_lat.abs().max()) <= bound * (1 + 2.0 ** -10) < 65504.0
    cache = dev.cache.float()
    assert torch.isfinite(cache[~torch.isnan(cache)]).all()
    dev.handle.close()


def _few_row_case(case):
    """Workloads that run the few-row attention (block_len x heads <= 32,
    128-token pages): ragged lengths leave partial last tiles and many key
    splits per block."""
    import dataclasses
    W = workloads
    if case == "t1_ragged":
        return W.cached_decode_workload(case, W.QWEN3_4B_MLA, 11, batch=5, prefill_len=700,
                                        len_lo=60, len_hi=700, block_len=1, num_blocks=2,
                                        page_size=128)
    if case == "t1_window_masked":
        wl = W.cached_decode_workload(case, W.QWEN3_4B_MLA.replace(rope_style="neox",
                                                                   use_output_gate=True),
                                      12, batch=4, prefill_len=900, len_lo=300, len_hi=900,
                                      block_len=1, num_blocks=1, page_size=128)
        s = wl.steps[0]
        win = s.window.copy()
        win[1], win[3] = 200, 1
        qv = s.q_visible.copy()
        qv[2] = 0
        return dataclasses.replace(wl, steps=[dataclasses.replace(s, window=win, q_visible=qv)])
    if case == "t2_h16":
        return W.cached_decode_workload(case, W.QWEN3_4B_MLA.replace(num_heads=16), 13, batch=4,
                                        prefill_len=600, len_lo=100, len_hi=600, block_len=2,
                                        num_blocks=2, page_size=256)
    if case == "t3_h8":
        return W.prefill_workload(case, W.QWEN3_4B_MLA.replace(num_heads=8), 14, [300, 129, 650],
                                  3, page_size=128)
    raise KeyError(case)


@pytest.mark.parametrize("case", ["t1_ragged", "t1_window_masked", "t2_h16", "t3_h8"])
def test_few_row_blocks_match_oracle(case):
    """Blocks of at most 32 query rows take the few-row kernel (keys in the
    MMA's M dimension, every block's keys split across the SMs and merged by
    log-sum-exp)."""
    from tests.parity import check_workload
    check_workload(_few_row_case(case))


@pytest.mark.parametrize("case", ["T7_ragged_windows_masked", "T16_gate_off", "T40_one_context",
                                  "T32_grouped_masked", "T16_neox_many_tiles"])
def test_shared_context_blocks_match_oracle(case):
    """Blocks that share a context run the expanded form (the context's and
    the blocks' own latents expanded by kv_b_proj, one attention over
    q_nope|q_pe with the own keys as a block-diagonal tile): ragged context
    lengths (not multiples of the 128-key tile), block lengths that leave a
    unit's last rows empty, sliding windows shorter than the context and than
    the block, masked query rows, with and without the output gate.  Block
    lengths that divide the 128-row tile into 8-row multiples (16, 32) take
    each context's full-mask blocks and windowed blocks in separate units, so
    a unit's query and own-key rows come from blocks that are not adjacent.
    With more q_b tiles than SMs (T16_neox_many_tiles) the query projection
    takes the persistent GEMM's staged epilogue with NeoX RoPE."""
    import dataclasses
    from tests.parity import check_workload
    from head_latent_attention_qkv_gb300.runner import shared_contexts
    W = workloads
    d = W.DEEPSEEK_V3_MLA.replace(num_heads=16, hidden_size=1024)
    if case == "T7_ragged_windows_masked":
        wl = W.block_parallel_workload(case, d, 31, batch=3, ctx_len=320, blocks_per_seq=5,
                                       block_len=7, page_size=64, windows=(0, 150, 3))
        s = wl.steps[0]
        qv = s.q_visible.copy()
        qv[[2, 9, 33, 34, 60]] = 0
        wl = dataclasses.replace(wl, steps=[dataclasses.replace(s, q_visible=qv)])
    elif case == "T16_gate_off":
        wl = W.block_parallel_workload(case, d.replace(use_output_gate=False, rope_style="neox"), 32,
                                       batch=2, ctx_len=448, blocks_per_seq=9, block_len=16,
                                       page_size=64, windows=(0, 200))
    elif case == "T32_grouped_masked":
        wl = W.block_parallel_workload(case, d, 34, batch=3, ctx_len=384, blocks_per_seq=7,
                                       block_len=32, page_size=128, windows=(0, 90, 0, 5))
        s = wl.steps[0]
        qv = s.q_visible.copy()
        qv[[0, 31, 70, 300, 671]] = 0
        wl = dataclasses.replace(wl, steps=[dataclasses.replace(s, q_visible=qv)])
    elif case == "T16_neox_many_tiles":
        # 1280 query rows x 32 heads: q_b has more 128-row tiles than the GPU
        # has SMs, so it runs persistent with its staged split epilogue
        # (NeoX pairs (k, k + 32) inside one 64-column group)
        wl = W.block_parallel_workload(case, d.replace(num_heads=32, rope_style="neox"), 35, batch=2,
                                       ctx_len=256, blocks_per_seq=40, block_len=16, page_size=128,
                                       windows=(0, 100))
    else:
        wl = W.block_parallel_workload(case, d, 33, batch=1, ctx_len=256, blocks_per_seq=4,
                                       block_len=40, page_size=128, windows=(0,))
    assert shared_contexts(wl, wl.steps[0]) is not None
    check_workload(wl)


def test_shared_attention_entry_reproduces_the_forwards_output():
    """mla_shared_attention re-runs the expanded attention on the shared
    forward's intermediates: the per-head output o is the same bit for bit."""
    from head_latent_attention_qkv_gb300 import _lib, api
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload
    wl = workloads.make_workload("deepseek_v3_block_parallel", "small")
    dev = DeviceWorkload(wl)
    dev.run_all()
    s = dev.steps[-1]
    assert s["ctx"] is not None
    M = s["hidden"].shape[0]
    d = wl.dims
    ws = dev.handle._ws
    off = api.mla_forward_workspace_offset(dev.handle, M, _lib.MLA_WS_O)
    n = M * d.num_heads * d.v_head_dim
    torch.cuda.synchronize()
    o_fwd = ws[off:off + 2 * n].clone()
    ws[off:off + 2 * n] = 0
    api.mla_shared_attention(dev.handle, s["positions"], s["desc"], s["ctx"])
    torch.cuda.synchronize()
    assert api.mla_get_device_status(dev.handle) == 0
    assert torch.equal(ws[off:off + 2 * n], o_fwd)
    dev.handle.close()
