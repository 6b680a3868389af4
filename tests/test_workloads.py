"""Host checks of the seeded input generator (CPU).

``workloads.py`` feeds both the oracle and the CUDA path, so its layout
contracts are checked directly: the position contract of the boundary
(query i of block b sits at kv_len[b] - T + i), cache slots that are unique
and agree with the page tables, pages in range, the masked rows and windows
each configuration asks for, and seeded reproducibility.
"""
import numpy as np
import pytest

from head_latent_attention_qkv_gb300 import workloads as W

_CACHE = {}


def _small(name):
    if name not in _CACHE:
        _CACHE[name] = W.make_workload(name, "small")
    return _CACHE[name]


SMALL = [_small(n) for n in W.WORKLOADS]


def _slot(table_row, page_size, j):
    return int(table_row[j // page_size]) * page_size + j % page_size


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_block_positions_follow_the_boundary_contract(wl):
    T = wl.block_len
    for s in wl.steps:
        nb = len(s.kv_len)
        pos = s.block_positions.reshape(nb, T)
        expect = s.kv_len[:, None] - T + np.arange(T)[None, :]
        np.testing.assert_array_equal(pos, expect)


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_slots_are_unique_in_range_and_match_the_page_tables(wl):
    n_slots = wl.num_pages * wl.page_size
    written = []
    if wl.ctx_slots is not None:
        written.append(wl.ctx_slots)
    if wl.prefill_slots is not None:
        written.append(wl.prefill_slots)
    T = wl.block_len
    for s in wl.steps:
        assert np.all((s.block_table >= -1) & (s.block_table < wl.num_pages))
        for blk_slots in (s.block_slots, s.append_slots):
            if blk_slots is None:
                continue
            written.append(blk_slots)
            # each block token's slot is the table's slot of its logical position
            for b in range(len(s.kv_len)):
                for i in range(T):
                    j = int(s.block_positions[b * T + i])
                    assert blk_slots[b * T + i] == _slot(s.block_table[b], wl.page_size, j)
    allw = np.concatenate(written)
    assert np.all((allw >= 0) & (allw < n_slots))
    if wl.prefill_slots is None:
        # without a pre-filled cache every slot is written once
        assert len(np.unique(allw)) == len(allw)


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_every_visible_key_has_a_valid_page(wl):
    for s in wl.steps:
        for b in range(len(s.kv_len)):
            pages_needed = -(-int(s.kv_len[b]) // wl.page_size)
            assert np.all(s.block_table[b, :pages_needed] >= 0)


def test_sliding_workload_masks_and_windows():
    wl = _small("qwen3_4b_sliding_gate")
    s = wl.steps[0]
    assert np.all(s.window == 512) and wl.dims.use_output_gate and wl.dims.rope_style == "neox"
    qv = s.q_visible.reshape(-1, wl.block_len)
    for b in range(qv.shape[0]):
        want = np.ones(wl.block_len, dtype=bool)
        if b % 4 == 0:
            want[:4] = False
        np.testing.assert_array_equal(qv[b].astype(bool), want)


def test_block_parallel_workload_alternates_full_and_sliding():
    wl = _small("deepseek_v3_block_parallel")
    s = wl.steps[0]
    per_seq = 3
    for b, win in enumerate(s.window):
        assert win == (0 if (b % per_seq) % 2 == 0 else 100)
    # every proposal of a sequence is anchored right after the shared context
    np.testing.assert_array_equal(s.kv_len, np.full(len(s.kv_len), 192 + wl.block_len))


def test_one_token_decode_has_one_query_token_per_sequence():
    wl = _small("qwen3_4b_decode_t1")
    assert wl.block_len == 1 and len(wl.steps) == 2
    a, b = wl.steps
    np.testing.assert_array_equal(b.kv_len, a.kv_len + 1)


def test_generation_is_seeded():
    a = _small("qwen3_4b_prefill")
    b = W.make_workload("qwen3_4b_prefill", "small")
    np.testing.assert_array_equal(a.ctx_hidden, b.ctx_hidden)
    np.testing.assert_array_equal(a.steps[0].block_table, b.steps[0].block_table)
    for k, v in a.weights.items():
        if v is not None:
            np.testing.assert_array_equal(v, b.weights[k])


def test_bf16_values_are_exactly_representable():
    wl = _small("qwen3_4b_prefill")
    for arr in (wl.ctx_hidden, wl.steps[0].block_hidden, wl.weights["q_b_proj"]):
        rt = W.bf16_bits_to_f32(W.bf16_bits(arr))
        np.testing.assert_array_equal(rt, arr)
