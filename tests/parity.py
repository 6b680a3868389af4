"""GPU-vs-oracle comparison helpers for the parity tests.

Tolerances (from the layer's contract): outputs max|gpu - ref| <= 2e-2 * rms
and mean|gpu - ref| <= 2e-3 * rms for bf16 (rms over rows that are not fully
masked), 1e-4 for both in the fp32 configuration.  For bf16 tensors the
per-element bound is max(2e-2 * rms, one bf16 ulp of the reference value):
the oracle, like the method, holds the output and the cache in bf16, and one
ulp is the format's resolution.  The floor's reach is bounded by a second
comparison of the layer output against the oracle's fp64 value before its
bf16 rounding: there an element may exceed 2e-2 * rms by at most half a bf16
ulp (the rounding of the GPU's own bf16 result), the mean of what each
element exceeds that half ulp by stays within 2e-3 * rms, and the number of
elements that pass the first comparison only through the floor is reported.  Exact
checks: fully
masked rows are bitwise +0.0; the per-row visible-key count, first and last
visible key reported by the kernel equal the oracle's visibility; the cache
slots written are exactly the slots the calls name (every other slot keeps
its NaN sentinel); written latents are within tolerance of the oracle's.
"""
from __future__ import annotations

import json

import numpy as np
import torch

from head_latent_attention_qkv_gb300 import api
from head_latent_attention_qkv_gb300.runner import DeviceWorkload
from oracle.keys import run_workload
from oracle.mla import round_to_dtype


def tolerances(dims):
    return (1e-4, 1e-4) if dims.dtype == "fp32" else (2e-2, 2e-3)


def compare(got, ref, dims, what, valid_rows=None, ref64=None):
    """Check ``got`` against the oracle's typed value ``ref`` (and, for bf16
    tensors when given, its fp64 value ``ref64`` before storage rounding).
    Returns a dict of the relative errors and the floor count."""
    tmax, tmean = tolerances(dims)
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    sel = slice(None) if valid_rows is None else valid_rows
    rms = np.sqrt(np.mean(ref[sel] ** 2))
    assert np.all(np.isfinite(got[sel])), f"{what}: non-finite values"
    err = np.abs(got[sel] - ref[sel])
    emax, emean = err.max() / rms, err.mean() / rms
    bound = np.full(err.shape, tmax * rms)
    floor_only = 0
    if dims.dtype == "bf16":
        # resolution floor of a bf16 tensor: both sides hold bf16 values, so a
        # difference far below tolerance still shows as one ulp where it
        # straddles a rounding boundary; 1 ulp of an element above ~2.6*rms
        # exceeds 2e-2*rms
        floor_only = int(np.count_nonzero(err > bound))
        bound = np.maximum(bound, bf16_ulp(ref[sel]))
    over = err > bound
    assert not over.any() and emean <= tmean, (
        f"{what}: max {emax:.3e} mean {emean:.3e} (rms {rms:.3e}), "
        f"{int(over.sum())} elements beyond max(tol*rms, 1 ulp)")
    stats = {"what": what, "max_rel": float(emax), "mean_rel": float(emean),
             "elements": int(err.size), "floor_only": floor_only}
    if ref64 is not None and dims.dtype == "bf16":
        # the GPU's output is itself a bf16 tensor: each element may carry half
        # an ulp of its own rounding on top of the kernel's error; the mean bar
        # applies to what is left once that half ulp is taken off
        r64 = np.asarray(ref64, np.float64)[sel]
        e64 = np.abs(got[sel] - r64)
        half = 0.5 * bf16_ulp(r64)
        over64 = e64 > tmax * rms + half
        mean_net = np.maximum(e64 - half, 0.0).mean()
        assert not over64.any() and mean_net <= tmean * rms, (
            f"{what} vs unrounded fp64: max {e64.max() / rms:.3e} mean beyond the half ulp "
            f"{mean_net / rms:.3e}, {int(over64.sum())} elements beyond tol*rms + half an ulp")
        stats.update(max_rel_fp64=float(e64.max() / rms), mean_rel_fp64=float(e64.mean() / rms),
                     mean_rel_fp64_net=float(mean_net / rms),
                     beyond_tol_fp64=int(np.count_nonzero(e64 > tmax * rms)))
    return stats


def bf16_ulp(x):
    """Spacing of bf16 values (8 significant bits) at |x|."""
    ax = np.maximum(np.abs(np.asarray(x, np.float64)), np.finfo(np.float32).tiny)
    return np.ldexp(1.0, np.frexp(ax)[1] - 8)


def vis_expected(run, step, b):
    vis = run.block_visibility(step, b)
    cnt = vis.sum(axis=1)
    first = np.where(cnt > 0, vis.argmax(axis=1), -1)
    last = np.where(cnt > 0, vis.shape[1] - 1 - vis[:, ::-1].argmax(axis=1), -1)
    return np.stack([cnt, first, last], axis=1)


def check_workload(wl, blocks_per_step=None, check_cache=True, dev=None):
    """Run ``wl`` through the library (on ``dev``'s handle when given, else a
    fresh one) and compare with the oracle."""
    dev = DeviceWorkload(wl) if dev is None else dev
    outs_gpu = dev.run_all()
    torch.cuda.synchronize()
    assert api.mla_get_device_status(dev.handle) == 0
    run, outs_64 = run_workload(wl, blocks_per_step, round_output=False)
    T = wl.block_len
    report = []
    for k, step in enumerate(wl.steps):
        blocks = sorted(outs_64[k])
        got = outs_gpu[k].float().cpu().numpy().reshape(-1, T, wl.dims.hidden_size)[blocks]
        ref64 = np.stack([outs_64[k][b] for b in blocks])
        ref = round_to_dtype(wl.dims, ref64)
        qv = step.q_visible.reshape(-1, T)[blocks].astype(bool)
        report.append(compare(got, ref, wl.dims, f"{wl.name} step {k} out", qv, ref64=ref64))
        assert np.all(got[~qv] == 0) and not np.signbit(got[~qv]).any(), "masked rows not +0"
        vs = dev.steps[k]["vis_stats"].cpu().numpy().reshape(-1, T, 3)
        for b in blocks:
            np.testing.assert_array_equal(vs[b], vis_expected(run, step, b),
                                          err_msg=f"{wl.name} step {k} block {b} visibility")
    if check_cache:
        cache = dev.cache.float().cpu().numpy().reshape(-1, wl.dims.cache_dim)
        named = np.zeros(len(cache), dtype=bool)
        for s in (wl.ctx_slots, wl.prefill_slots, *[x.block_slots for x in wl.steps],
                  *[x.append_slots for x in wl.steps]):
            if s is not None:
                named[s] = True
        assert np.all(np.isnan(cache[~named])), "a slot outside the slot mappings was written"
        assert np.all(np.isfinite(cache[named])), "a named slot was not written"
        report.append(compare(cache[run.written], run.cache[run.written], wl.dims,
                              f"{wl.name} cache"))
    dev.handle.close()
    for r in report:
        print("parity", json.dumps(r))
    return report
