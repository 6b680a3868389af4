"""Drive the fp64 oracle over a whole workload (paged cache, many blocks).

TEST INFRASTRUCTURE (same rules as ``oracle.mla``).  The workload object is
read by attribute only (weights, slots, block tables, lengths, ...); nothing
from the CUDA library is imported.

The oracle keeps its own fp64 latent cache indexed by flat slot, filled the
way the method fills it ("MLA (Multi-Head Latent Attention)" blog,
``do_kv_cache_update``: ``kv_cache[slot] = [kv_c_normed | k_pe]`` keyed by
``slot_mapping``): context tokens are appended from their hidden states
(target-context injection, "Add config-selectable MLA draft attention"), a
pre-filled cache is taken as given, and block latents are written at the
block's slots before the block attends.  Key ``j`` of a block is the entry at
``block_table[j // page_size] * page_size + j % page_size``.
"""
from __future__ import annotations

import numpy as np

from . import mla


class OracleRun:
    def __init__(self, wl):
        self.wl = wl
        self.d = wl.dims
        self.P = wl.page_size
        self.cache = np.zeros((wl.num_pages * wl.page_size, wl.dims.cache_dim))
        self.written = np.zeros(wl.num_pages * wl.page_size, dtype=bool)
        if wl.prefill_slots is not None:
            self.cache[wl.prefill_slots] = wl.prefill_values
            self.written[wl.prefill_slots] = True

    def append(self, hidden, positions, slots, rows=None):
        """Write the oracle's latent entries of ``hidden[rows]`` at ``slots[rows]``."""
        if rows is None:
            rows = np.arange(len(slots))
        rows = np.asarray(rows)
        if rows.size == 0:
            return np.zeros((0, self.d.cache_dim))
        ent = mla.round_to_dtype(
            self.d, mla.latent_cache_entries(self.d, self.wl.weights, hidden[rows], positions[rows]))
        self.cache[slots[rows]] = ent
        self.written[slots[rows]] = True
        return ent

    def key_slots(self, step, b):
        """Flat slots of keys 0..kv_len-1 of block b, in logical order."""
        n = int(step.kv_len[b])
        j = np.arange(n, dtype=np.int64)
        pages = step.block_table[b][j // self.P].astype(np.int64)
        return pages * self.P + j % self.P

    def block_visibility(self, step, b):
        T = self.wl.block_len
        rows = slice(b * T, (b + 1) * T)
        n = int(step.kv_len[b])
        return mla.visibility(step.block_positions[rows], n, int(step.window[b]),
                              step.q_visible[rows], n)

    def needed_slots(self, step, blocks):
        """Slots holding at least one visible key of the given blocks."""
        need = np.zeros(len(self.cache), dtype=bool)
        for b in blocks:
            vis = self.block_visibility(step, b).any(axis=0)
            need[self.key_slots(step, b)[vis]] = True
        return need

    def forward_blocks(self, step, blocks, write_block_latents=True, round_output=True):
        """Oracle output rows [T, D] for each block in ``blocks`` (dict), held
        in the layer dtype (``round_output=False``: the fp64 values before
        that storage rounding)."""
        rnd = (lambda x: mla.round_to_dtype(self.d, x)) if round_output else (lambda x: x)
        d, w, T = self.d, self.wl.weights, self.wl.block_len
        blocks = list(blocks)
        if write_block_latents and step.block_slots is not None and blocks:
            rows = np.concatenate([np.arange(b * T, (b + 1) * T) for b in blocks])
            self.append(step.block_hidden, step.block_positions, step.block_slots, rows)
        memo, memo_seq, out = {}, None, {}
        for b in sorted(blocks, key=lambda b: int(step.block_seq[b])):
            if step.block_seq[b] != memo_seq:
                memo, memo_seq = {}, step.block_seq[b]
            vis = self.block_visibility(step, b)
            slots = self.key_slots(step, b)
            n = len(slots)
            segs, cols = [], []
            for pi in range(-(-n // self.P)):
                lo, hi = pi * self.P, min(n, (pi + 1) * self.P)
                if not vis[:, lo:hi].any():
                    continue
                key = (int(step.block_table[b][pi]), hi - lo)
                if key not in memo:
                    memo[key] = mla.expand_keys(d, w, self.cache[slots[lo:hi]])
                segs.append(memo[key])
                cols.append(np.arange(lo, hi))
            rows = slice(b * T, (b + 1) * T)
            x = step.block_hidden[rows]
            if not segs:
                o = np.zeros((T, d.num_heads, d.v_head_dim))
                out[b] = rnd(mla.output_projection(d, w, x, o))
                continue
            v = vis[:, np.concatenate(cols)]
            out[b] = rnd(mla.block_forward(d, w, x, step.block_positions[rows], segs, v))
        return out


def run_workload(wl, blocks_per_step=None, ctx_all=False, round_output=True):
    """Run the oracle over ``wl``.

    ``blocks_per_step[k]``: blocks of step k to evaluate (default: all).
    Context latents are computed only where a selected block can see them
    unless ``ctx_all``.  ``round_output=False`` returns the fp64 outputs
    before their storage rounding to the layer dtype.  Returns (OracleRun,
    [dict block -> out rows]).
    """
    run = OracleRun(wl)
    outs = []
    for k, step in enumerate(wl.steps):
        blocks = range(len(step.kv_len)) if blocks_per_step is None else blocks_per_step[k]
        if k == 0 and wl.ctx_hidden is not None:
            if ctx_all:
                rows = None
            else:
                need = run.needed_slots(step, blocks)
                rows = np.nonzero(need[wl.ctx_slots])[0]
            run.append(wl.ctx_hidden, wl.ctx_positions, wl.ctx_slots, rows)
        if step.append_hidden is not None:
            run.append(step.append_hidden, step.append_positions, step.append_slots)
        outs.append(run.forward_blocks(step, blocks, round_output=round_output))
    return run, outs
