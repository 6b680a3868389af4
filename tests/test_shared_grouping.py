"""Host logic of the shared-context grouping (which blocks the runner sends
to mla_draft_forward_shared): CPU only, no kernel runs."""
import dataclasses

import numpy as np

from head_latent_attention_qkv_gb300 import workloads as W
from head_latent_attention_qkv_gb300.runner import shared_contexts


def _wl(**kw):
    d = W.DEEPSEEK_V3_MLA.replace(num_heads=4, hidden_size=256, q_lora_rank=64)
    args = dict(batch=3, ctx_len=128, blocks_per_seq=4, block_len=16, page_size=64, windows=(0, 50))
    args.update(kw)
    return W.block_parallel_workload("g", d, 7, **args)


def test_proposals_over_one_context_are_grouped():
    wl = _wl()
    got = shared_contexts(wl, wl.steps[0])
    assert got is not None
    ctx_len, starts, rows = got
    assert ctx_len.tolist() == [128, 128, 128]
    assert starts.tolist() == [0, 4, 8, 12]
    assert rows == 3 * 128


def test_blocks_out_of_sequence_order_are_not_grouped():
    wl = _wl()
    s = wl.steps[0]
    seq = s.block_seq.copy()
    seq[[3, 4]] = seq[[4, 3]]
    assert shared_contexts(wl, dataclasses.replace(s, block_seq=seq)) is None


def test_a_context_with_one_block_is_not_grouped():
    wl = _wl(blocks_per_seq=1)
    assert shared_contexts(wl, wl.steps[0]) is None
    assert shared_contexts(wl, wl.steps[0], min_blocks=1) is not None


def test_a_block_whose_table_names_other_context_pages_is_not_grouped():
    wl = _wl()
    s = wl.steps[0]
    table = s.block_table.copy()
    table[5, 1] = table[0, 1]           # block 5 (context 1) reads a page of context 0
    assert shared_contexts(wl, dataclasses.replace(s, block_table=table)) is None


def test_a_block_with_a_longer_own_span_is_not_grouped():
    wl = _wl()
    s = wl.steps[0]
    kv = s.kv_len.copy()
    kv[2] -= 1                           # kv_len must be ctx_len + block_len for every block
    assert shared_contexts(wl, dataclasses.replace(s, kv_len=kv)) is None


def test_grouping_preserves_the_context_page_identity_of_the_generator():
    wl = _wl()
    s = wl.steps[0]
    ctx_len, starts, _ = shared_contexts(wl, s)
    for c in range(len(ctx_len)):
        pages = ctx_len[c] // wl.page_size
        rows = np.asarray(s.block_table)[starts[c]:starts[c + 1], :pages]
        assert (rows == rows[0]).all()
