"""Pin of the oracle's paged-cache walk (``oracle/keys.py``), CPU only.

``OracleRun`` turns a block's page table into cache slots, skips pages no
query of the block sees and reuses expanded keys per (page, length) within a
sequence.  Every GPU parity test compares against its output, so it is
checked here against a plain restatement that shares none of that logic:

* the cache is rebuilt slot by slot from the workload's own slot arrays
  (context tokens, pre-filled entries, appended and block tokens);
* key j of block b is read at ``block_table[b][j // P] * P + j % P``
  ("MLA (Multi-Head Latent Attention)" blog, ``MLAAttentionSpec`` /
  ``do_kv_cache_update``: pages of ``page_size`` tokens addressed through the
  block table, entries keyed by slot);
* every key below kv_len is expanded and passed to the attention with the
  visibility mask, no page skipped and nothing memoised.

The two routes agree to 1e-12 relative in fp64 on ragged contexts, permuted
pages of 16, 64, 128 and 256 tokens, sliding windows, masked rows, proposals
sharing one context, and two consecutive cached blocks ("extract GQA/MLA
attention into reusable layers", Accuracy Test: the cached decode).  Three
mistakes planted in copies of ``keys.py`` (page index off by one, a memo key
without the segment length, skipping a page that is only partly visible)
each break the agreement.
"""
import os
import types

import numpy as np
import pytest

from head_latent_attention_qkv_gb300 import workloads as W
from oracle import keys as oracle_keys
from oracle import mla

SMALL_DIMS = W.MLADims(hidden_size=32, num_heads=2, q_lora_rank=16, kv_lora_rank=16,
                       qk_nope_head_dim=8, qk_rope_head_dim=8, v_head_dim=8,
                       rope_style="interleaved", rope_theta=1e4, dtype="bf16")


def _cases():
    d = SMALL_DIMS
    dg = d.replace(use_output_gate=True, rope_style="neox")
    out = []
    for P in (16, 64, 128, 256):
        out.append(W.prefill_workload(f"prefill_p{P}", d, 11 + P, [150, 40, 333, 7], 16,
                                      page_size=P))
    out.append(W.prefill_workload("sliding_masked", dg, 21, [300, 97, 129, 513], 16,
                                  page_size=32, window=100,
                                  masked_rows=lambda s: (0, 1, 2, 3) if s % 2 == 0 else ()))
    out.append(W.prefill_workload("sliding_tiny_window", d, 22, [70, 33], 5, page_size=16,
                                  window=3))
    out.append(W.cached_decode_workload("cached_two_blocks", d, 23, batch=4, prefill_len=200,
                                        len_lo=17, len_hi=150, block_len=16, num_blocks=2,
                                        page_size=32))
    out.append(W.cached_decode_workload("cached_two_steps_t1", d, 24, batch=3, prefill_len=90,
                                        len_lo=10, len_hi=80, block_len=1, num_blocks=2,
                                        page_size=16))
    out.append(W.block_parallel_workload("proposals", dg, 25, batch=2, ctx_len=128,
                                         blocks_per_seq=4, block_len=16, page_size=64,
                                         windows=(0, 50)))
    out.append(_one_step(W.cached_decode_workload("two_blocks_one_step", d, 26, batch=4,
                                                  prefill_len=200, len_lo=17, len_hi=150,
                                                  block_len=16, num_blocks=2, page_size=32)))
    return out


def _one_step(wl):
    """Both cached blocks of every sequence in one step: the second block of a
    sequence sees the first one's tokens, so the two read the same partly
    filled page with different lengths."""
    import dataclasses
    s0, s1 = wl.steps
    cat = np.concatenate
    merged = W.Step(
        append_hidden=cat([s0.append_hidden, s1.append_hidden]),
        append_positions=cat([s0.append_positions, s1.append_positions]),
        append_slots=cat([s0.append_slots, s1.append_slots]),
        block_hidden=cat([s0.block_hidden, s1.block_hidden]),
        block_positions=cat([s0.block_positions, s1.block_positions]),
        block_slots=None, block_table=cat([s0.block_table, s1.block_table]),
        kv_len=cat([s0.kv_len, s1.kv_len]), window=cat([s0.window, s1.window]),
        q_visible=cat([s0.q_visible, s1.q_visible]),
        block_seq=cat([s0.block_seq, s1.block_seq]))
    return dataclasses.replace(wl, steps=[merged])


CASES = _cases()


def _independent_outputs(wl):
    """Per step, {block: fp64 output rows} from a slot-by-slot cache and an
    unskipped, unmemoised key walk."""
    d, w, P, T = wl.dims, wl.weights, wl.page_size, wl.block_len
    cache = {}

    def put(hidden, positions, slots):
        ent = mla.round_to_dtype(d, mla.latent_cache_entries(d, w, hidden, positions))
        for i, sl in enumerate(np.asarray(slots)):
            cache[int(sl)] = ent[i]

    if wl.prefill_slots is not None:
        for i, sl in enumerate(wl.prefill_slots):
            cache[int(sl)] = np.asarray(wl.prefill_values[i], np.float64)
    if wl.ctx_hidden is not None:
        put(wl.ctx_hidden, wl.ctx_positions, wl.ctx_slots)
    outs = []
    for step in wl.steps:
        if step.append_hidden is not None:
            put(step.append_hidden, step.append_positions, step.append_slots)
        if step.block_slots is not None:
            put(step.block_hidden, step.block_positions, step.block_slots)
        res = {}
        for b in range(len(step.kv_len)):
            n = int(step.kv_len[b])
            table = step.block_table[b]
            entries = np.stack([cache[int(table[j // P]) * P + j % P] for j in range(n)])
            rows = slice(b * T, (b + 1) * T)
            pos = step.block_positions[rows]
            vis = mla.visibility(pos, n, int(step.window[b]), step.q_visible[rows], n)
            x = step.block_hidden[rows]
            if not vis.any():
                o = np.zeros((T, d.num_heads, d.v_head_dim))
                res[b] = mla.output_projection(d, w, x, o)
            else:
                res[b] = mla.block_forward(d, w, x, pos, [mla.expand_keys(d, w, entries)], vis)
        outs.append(res)
    return outs


def _oracle_outputs(wl, keys_module):
    run = keys_module.OracleRun(wl)
    if wl.ctx_hidden is not None:
        run.append(wl.ctx_hidden, wl.ctx_positions, wl.ctx_slots)
    outs = []
    for step in wl.steps:
        if step.append_hidden is not None:
            run.append(step.append_hidden, step.append_positions, step.append_slots)
        outs.append(run.forward_blocks(step, range(len(step.kv_len)), round_output=False))
    return outs


def _max_rel(a_outs, b_outs):
    worst = 0.0
    for a, b in zip(a_outs, b_outs):
        assert sorted(a) == sorted(b)
        for k in a:
            scale = max(np.sqrt(np.mean(b[k] ** 2)), 1e-300)
            worst = max(worst, float(np.max(np.abs(a[k] - b[k]))) / scale)
    return worst


@pytest.mark.parametrize("wl", CASES, ids=[w.name for w in CASES])
def test_oracle_walk_equals_independent_slot_gather(wl):
    expect = _independent_outputs(wl)
    got = _oracle_outputs(wl, oracle_keys)
    assert _max_rel(got, expect) < 1e-12
    # masked rows: exactly zero on both routes
    for step, res in zip(wl.steps, got):
        masked = np.nonzero(step.q_visible == 0)[0]
        for m in masked:
            b, i = divmod(int(m), wl.block_len)
            assert np.all(res[b][i] == 0.0)


def test_cases_exercise_page_skipping_and_reuse():
    """The pin is only meaningful if the walk actually skips pages and reuses
    memoised keys somewhere in the cases."""
    skipped = reused = 0
    for wl in CASES:
        run = oracle_keys.OracleRun(wl)
        for step in wl.steps:
            for b in range(len(step.kv_len)):
                vis = run.block_visibility(step, b)
                n = vis.shape[1]
                for pi in range(-(-n // wl.page_size)):
                    if not vis[:, pi * wl.page_size:(pi + 1) * wl.page_size].any():
                        skipped += 1
            seqs = step.block_seq
            reused += len(seqs) - len(set(int(s) for s in seqs))
    assert skipped > 0 and reused > 0


_KEYS_SRC = open(os.path.join(os.path.dirname(oracle_keys.__file__), "keys.py")).read()

MUTATIONS = {
    # page index off by one
    "page_off_by_one": ("pages = step.block_table[b][j // self.P].astype(np.int64)",
                        "pages = step.block_table[b][np.minimum(j // self.P + 1, "
                        "step.block_table.shape[1] - 1)].astype(np.int64)"),
    # memo keyed by page id alone: segments of different length collide
    "memo_key_without_length": ("key = (int(step.block_table[b][pi]), hi - lo)",
                                "key = int(step.block_table[b][pi])"),
    # a page is skipped unless every one of its keys is visible to some query
    "skip_partly_visible_page": ("if not vis[:, lo:hi].any():",
                                 "if not vis[:, lo:hi].any(axis=0).all():"),
}


def _mutant(name):
    old, new = MUTATIONS[name]
    assert _KEYS_SRC.count(old) == 1, name
    mod = types.ModuleType(f"oracle._keys_{name}")
    mod.__package__ = "oracle"
    exec(compile(_KEYS_SRC.replace(old, new), f"<keys mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_walk_mistake_is_caught(name):
    m = _mutant(name)
    caught = False
    for wl in CASES:
        try:
            got = _oracle_outputs(wl, m)
        except (IndexError, ValueError):
            caught = True
            break
        if not _max_rel(got, _independent_outputs(wl)) < 1e-12:
            caught = True
            break
    assert caught, f"mutation {name} went unnoticed"
