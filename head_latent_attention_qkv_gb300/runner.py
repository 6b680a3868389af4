"""Drive a synthetic workload through the CUDA library (device side).

Uploads the seeded inputs of ``workloads.Workload`` to the GPU, then runs the
call sequence: prefilled cache entries are copied in, context tokens are
appended with ``mla_latent_cache_append``, and every step appends its tokens
(if any) and calls ``mla_draft_forward`` -- or, when its blocks come in
groups that share one context (consecutive blocks, at least two per
context, each seeing its context and then its own block_len keys),
``mla_draft_forward_shared`` with that context list.  ``run_step_after`` issues a step's
cache appends on a second stream instead, so that the forward's projections
run beside them and only its attention waits (``mla_draft_forward_after``).
Only data movement happens here; all of the layer's arithmetic runs in the
library.
"""
from __future__ import annotations

import numpy as np
import torch

from . import api


def shared_contexts(wl, step, min_blocks=2):
    """(ctx_len [num_ctx], ctx_block_start [num_ctx + 1], ctx_rows) when the
    step's blocks share contexts as mla_draft_forward_shared wants them,
    else None."""
    if wl.ctx_seq is None or step.block_seq is None:
        return None
    seq = np.asarray(step.block_seq)
    n_ctx = int(seq.max()) + 1 if seq.size else 0
    if n_ctx == 0 or np.any(np.diff(seq) < 0) or set(np.unique(seq).tolist()) != set(range(n_ctx)):
        return None
    ctx_len = np.bincount(np.asarray(wl.ctx_seq), minlength=n_ctx)[:n_ctx].astype(np.int32)
    starts = np.searchsorted(seq, np.arange(n_ctx + 1)).astype(np.int32)
    if np.min(np.diff(starts)) < min_blocks:
        return None
    if np.any(step.kv_len != ctx_len[seq] + wl.block_len):
        return None
    # the context keys are read through each context's first block's page
    # table: every block of the context must name the same pages for them
    table = np.asarray(step.block_table)
    for c in range(n_ctx):
        pages = -(-int(ctx_len[c]) // wl.page_size)
        rows = table[starts[c]:starts[c + 1], :pages]
        if np.any(rows != rows[:1]):
            return None
    return ctx_len, starts, int(ctx_len.sum())


def to_dev(a, dtype=None, device="cuda"):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


class DeviceWorkload:
    """Device copies of a workload's inputs, ready for repeated runs."""

    def __init__(self, wl, device="cuda", cache_fill=float("nan")):
        self.wl, self.device = wl, device
        dt = api.torch_dtype(wl.dims)
        self.dtype = dt
        self.weights = {k: to_dev(v, dt, device) for k, v in wl.weights.items() if v is not None}
        self.handle = api.mla_draft_init(wl.dims, self.weights, wl.page_size, device)
        self.cache = torch.full(wl.cache_shape, cache_fill, dtype=dt, device=device)
        self.cache_fill = cache_fill
        self.ctx = None
        if wl.ctx_hidden is not None:
            self.ctx = (to_dev(wl.ctx_hidden, dt, device), to_dev(wl.ctx_positions, None, device),
                        to_dev(wl.ctx_slots, None, device))
        self.prefill = None
        if wl.prefill_slots is not None:
            self.prefill = (to_dev(wl.prefill_slots, None, device),
                            to_dev(wl.prefill_values, dt, device))
        self._side_ws = None
        self.steps = []
        for s in wl.steps:
            d = dict(
                append=None if s.append_hidden is None else (
                    to_dev(s.append_hidden, dt, device), to_dev(s.append_positions, None, device),
                    to_dev(s.append_slots, None, device)),
                hidden=to_dev(s.block_hidden, dt, device),
                positions=to_dev(s.block_positions, None, device),
                slots=to_dev(s.block_slots, None, device),
                block_table=to_dev(s.block_table, None, device),
                kv_len=to_dev(s.kv_len, None, device),
                window=to_dev(s.window, None, device),
                q_visible=to_dev(s.q_visible, None, device),
                vis_stats=torch.full((len(s.block_positions), 3), -7, dtype=torch.int32, device=device),
            )
            d["desc"] = api.make_desc(d["block_table"], d["kv_len"], d["window"], d["q_visible"],
                                      wl.block_len, d["vis_stats"])
            d["out"] = torch.empty(len(s.block_positions), wl.dims.hidden_size, dtype=dt, device=device)
            d["ctx"] = None
            sc = shared_contexts(wl, s)
            if sc is not None:
                d["ctx_len"] = to_dev(sc[0], None, device)
                d["ctx_start"] = to_dev(sc[1], None, device)
                d["ctx"] = api.make_shared_ctx(d["ctx_len"], d["ctx_start"], sc[2])
            self.steps.append(d)

    def reset_cache(self):
        self.cache.fill_(self.cache_fill)
        if self.prefill is not None:
            flat = self.cache.view(-1, self.wl.dims.cache_dim)
            flat[self.prefill[0]] = self.prefill[1]

    def append_context(self):
        if self.ctx is not None:
            api.mla_latent_cache_append(self.handle, *self.ctx, self.cache)

    def run_step(self, k):
        s = self.steps[k]
        if s["append"] is not None:
            api.mla_latent_cache_append(self.handle, *s["append"], self.cache)
        if s["ctx"] is not None:
            api.mla_draft_forward_shared(self.handle, s["hidden"], s["positions"], s["slots"],
                                         self.cache, s["desc"], s["ctx"], out=s["out"])
        else:
            api.mla_draft_forward(self.handle, s["hidden"], s["positions"], s["slots"], self.cache,
                                  s["desc"], out=s["out"])
        return s["out"]

    def run_step_after(self, k, side, with_context=False):
        """Step k with its cache appends (the context first when
        ``with_context``) on stream ``side``, forked from the current stream;
        the forward runs on the current stream and its attention waits for
        the appends, which also joins ``side`` back."""
        s = self.steps[k]
        main = torch.cuda.current_stream()
        appends = []
        if with_context and self.ctx is not None:
            appends.append(self.ctx)
        if s["append"] is not None:
            appends.append(s["append"])
        ready = None
        if appends:
            side.wait_stream(main)
            for a in appends:
                n = a[0].shape[0]
                need = api.lib.mla_append_workspace_bytes(self.handle.h, n)
                if self._side_ws is None or self._side_ws.numel() < need:
                    self._side_ws = api._buf(need, self.device)
                api.mla_latent_cache_append(self.handle, *a, self.cache, stream=side,
                                            workspace=self._side_ws)
            ready = torch.cuda.Event()
            ready.record(side)
        if s["ctx"] is not None:
            api.mla_draft_forward_shared_after(self.handle, s["hidden"], s["positions"], s["slots"],
                                               self.cache, s["desc"], s["ctx"], cache_ready=ready,
                                               out=s["out"])
        else:
            api.mla_draft_forward_after(self.handle, s["hidden"], s["positions"], s["slots"],
                                        self.cache, s["desc"], cache_ready=ready, out=s["out"])
        return s["out"]

    def run_all(self):
        """Fresh cache, context append, every step.  Returns the step outputs."""
        self.reset_cache()
        self.append_context()
        return [self.run_step(k).clone() for k in range(len(self.steps))]
