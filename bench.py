"""Benchmark of the MLA draft-layer hot path on GB300.

One step = the whole path over one batch of a synthetic workload: the
latent-cache append of the context tokens (target-context injection), then
the draft-layer forward of every query block (its own latents appended by
the forward), captured in one CUDA graph.  The default workload is the
DeepSeek-V3-shaped layer (hidden 7168, 128 heads, gate on): 4 sequences x
1024 proposals of 16 tokens over a 4096-token context, alternating full and
1024-window sliding masks, bf16.  Inputs are seeded synthetic data resident
in HBM; L2 (126 MB) is flushed by writing a 256 MB buffer between timed steps.

The same JSON line carries the roofline of the step's dominant kernel (the
one with the largest event-timed share, timed alone on the step's own
inputs) and, for the default workload, the cached-block decode (64 sequences,
two 16-token blocks over a pre-filled cache) and its one-token variant, each
timed the same way, with the cache bytes they read per second.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

N > 1 runs under torchrun as independent replicas (the forward shards by
sequence with no exchange step): each rank owns a full workload, rank 0
prints one JSON line with the max time over ranks and the summed tokens.
``--impl reference`` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "deepseek_v3_block_parallel"
DECODE_WORKLOADS = ("qwen3_4b_cached_decode", "qwen3_4b_decode_t1")
METRIC = "MLA draft-layer tokens/s (block query tokens; TFLOP/s and %bf16 peak alongside)"
DESC = {"tiny_fp32": "1 x (64 context + 8-token block), fp32",
        "qwen3_4b_prefill": "8 x (2048 context + 16-token block), full mask",
        "qwen3_4b_sliding_gate": "16 x (8192 context + 16), sliding 512, gate, masked rows",
        "qwen3_4b_cached_decode": "64 seqs, cache pre-filled, 2 consecutive 16-token blocks",
        "deepseek_v3_block_parallel": "4 x 1024 proposals of 16 over a 4096 context, gate, "
                                      "alternating full / 1024-window masks",
        "qwen3_4b_decode_t1": "64 seqs, cache pre-filled, 2 consecutive one-token steps"}


def algorithmic_flops(wl, shared=False):
    """Absorbed latent path: per block token 2D(r_q+L) [+2D*H*dv gate] +
    2 r_q H dqk + 2 H dn r_kv + 2 H r_kv dv + 2 H dv D, per visible key
    H (2L + 2 r_kv); per appended token 2 D L.  The expanded form (``shared``:
    blocks sharing a context) instead: no W_UK / W_UV, per gathered latent row
    (each context key once, each block token) 2 r_kv H (dn + dv), per visible
    key H (2 dqk + 2 dv).  Also the cache bytes the attention reads (1152 B
    per key a block can see, once per block)."""
    d = wl.dims
    H, D, L = d.num_heads, d.hidden_size, d.cache_dim
    qdim = d.q_lora_rank if d.q_lora_rank else H * d.qk_head_dim
    per_tok = 2 * D * (qdim + L) + (2 * D * H * d.v_head_dim if d.use_output_gate else 0)
    if d.q_lora_rank:
        per_tok += 2 * d.q_lora_rank * H * d.qk_head_dim
    if not shared:
        per_tok += 2 * H * d.qk_nope_head_dim * d.kv_lora_rank + 2 * H * d.kv_lora_rank * d.v_head_dim
    else:
        per_tok += 2 * d.kv_lora_rank * H * (d.qk_nope_head_dim + d.v_head_dim)   # its own row
    per_tok += 2 * H * d.v_head_dim * D
    per_key = H * (2 * d.qk_head_dim + 2 * d.v_head_dim) if shared else H * (2 * L + 2 * d.kv_lora_rank)
    T = wl.block_len
    total = block_tokens = cache_bytes = 0
    attention = []                             # per step: flops of its attention launch
    appended = 0 if wl.ctx_hidden is None else len(wl.ctx_hidden)
    for step in wl.steps:
        keys = 0
        for b in range(len(step.kv_len)):      # visible keys per query: [lo, kv_len)
            r = slice(b * T, (b + 1) * T)
            n, w = int(step.kv_len[b]), int(step.window[b])
            p = step.block_positions[r].astype(np.int64)
            lo = np.maximum(0, p - w + 1) if w > 0 else np.zeros_like(p)
            keys += int(((n - lo) * step.q_visible[r]).sum())
            cache_bytes += (n - int(lo.min())) * L * 2
        attention.append(per_key * keys)
        total += per_tok * len(step.block_positions) + attention[-1]
        block_tokens += len(step.block_positions)
        if step.append_hidden is not None:
            appended += len(step.append_hidden)
    append = 2 * D * L * (0 if wl.ctx_hidden is None else len(wl.ctx_hidden))
    total += 2 * D * L * (appended - (0 if wl.ctx_hidden is None else len(wl.ctx_hidden))) + append
    if shared:      # each context's keys expanded once per step
        total += 2 * d.kv_lora_rank * H * (d.qk_nope_head_dim + d.v_head_dim) * len(wl.ctx_hidden) * len(wl.steps)
    return dict(total=total, append=append, block_tokens=block_tokens, ctx_tokens=appended,
                cache_bytes=cache_bytes, attention=attention)


def attention_cache_bytes(wl):
    """Cache bytes the last step's attention reads: 1152 per key a block can
    see, once per block (from the first key any of its rows sees)."""
    step, L = wl.steps[-1], wl.dims.cache_dim
    total = 0
    for b in range(len(step.kv_len)):
        r = slice(b * wl.block_len, (b + 1) * wl.block_len)
        w, kv = int(step.window[b]), int(step.kv_len[b])
        lo = max(0, int(step.block_positions[r].min()) - w + 1) if w > 0 else 0
        total += (kv - lo) * L * 2
    return total


def few_row_attention(wl):
    """The library serves blocks of at most 32 query rows (bf16, 128-token
    pages) with the few-row kernel and its segment merge."""
    return (wl.dims.dtype == "bf16" and wl.block_len * wl.dims.num_heads <= 32
            and wl.page_size % 128 == 0)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms by a
    background nvidia-smi while the GPU runs the warm-up, the timed steps and
    untimed replays of the same step just before and after them (started, and
    its first line awaited, before the warm-up)."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.samples, self.index, self.proc, self.reader = [], index, None, None

    def _read(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 6:
                self.samples.append(f)

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 3.0:
                time.sleep(0.01)
            self.samples.clear()          # drop the idle sample taken before the load
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=10)
        except Exception:
            self.proc.kill()
        if self.reader is not None:
            self.reader.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if len(s) > 2 + i and s[2 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


def dram_traffic(kernel, workload):
    """DRAM bytes per launch of ``kernel`` on ``workload`` from the
    machine-readable record of the ncu captures (profiles/dram_traffic.json),
    or None when there is none or the kernel's source changed since."""
    import hashlib
    rec = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(rec):
        return None
    try:
        entry = json.load(open(rec))[kernel][workload]
        src = os.path.join(ROOT, entry["source"])
        if hashlib.sha256(open(src, "rb").read()).hexdigest() != entry["source_sha256"]:
            return None
        return float(entry["bytes_per_launch"])
    except (KeyError, ValueError, OSError, TypeError):
        return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def max_over_ranks(x, world):
    """Largest value of x over the ranks (the job is as fast as its slowest
    replica); works on the process group's backend, gloo or NCCL."""
    if world <= 1:
        return x
    import torch
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_replica, world, seconds):
    """Whole-job throughput: every replica processed its own full workload."""
    return world * tokens_per_replica / seconds


def timed(fn, n, flush, stream):
    """Mean event time (ms) of n runs of fn, L2 flushed (untimed) before each."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for k in range(n):
        flush.fill_(k & 0xFF)
        ev[k][0].record(stream)
        fn()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    t = [e[0].elapsed_time(e[1]) for e in ev]
    return sum(t) / len(t)


def capture(fn):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(2):
        g.replay()
    return g


class Session:
    """One workload on the device: its step, and the two kernels that carry
    most of its work (the context append and the last step's attention) as
    launches of their own on the step's inputs."""

    def __init__(self, name, overlap=False, scale="full"):
        import torch
        from head_latent_attention_qkv_gb300 import _lib, api, workloads
        from head_latent_attention_qkv_gb300.runner import DeviceWorkload
        self.name, self.overlap = name, overlap
        self.wl = workloads.make_workload(name, scale)
        self.dev = DeviceWorkload(self.wl)
        # blocks sharing a context run the expanded form (when the layer allows it)
        self.shared = (self.dev.steps[-1]["ctx"] is not None and self.wl.dims.dtype == "bf16"
                       and self.wl.dims.qk_nope_head_dim == 128 and self.wl.dims.v_head_dim == 128
                       and self.wl.block_len <= 128)
        self.fl = algorithmic_flops(self.wl, self.shared)
        self.side = torch.cuda.Stream()
        self.api, self.lib = api, _lib
        dev = self.dev
        dev.reset_cache()
        torch.cuda.synchronize()
        n0 = api.mla_kernel_launches(dev.handle)
        self.step()
        self.launches = api.mla_kernel_launches(dev.handle) - n0
        # the last step's attention on its own inputs: the forward left Q_abs in
        # its workspace; a copy of it feeds the attention entry point
        s = dev.steps[-1]
        M = s["hidden"].shape[0]
        d = self.wl.dims
        torch.cuda.synchronize()
        off = api.mla_forward_workspace_offset(dev.handle, M, _lib.MLA_WS_Q_ABS)
        esz = 2 if d.dtype == "bf16" else 4
        nq = M * d.num_heads * d.cache_dim
        raw = dev.handle._ws[off:off + nq * esz]
        self.q_abs = raw.view(api.torch_dtype(d)).view(M * d.num_heads, d.cache_dim).clone()
        self.o_lat = torch.empty(M * d.num_heads, d.kv_lora_rank,
                                 dtype=torch.float16 if d.dtype == "bf16" else torch.float32,
                                 device="cuda")
        self.lse = torch.empty(M * d.num_heads, dtype=torch.float32, device="cuda")

    def step(self):
        dev = self.dev
        if self.overlap:
            for k in range(len(dev.steps)):
                dev.run_step_after(k, self.side, with_context=(k == 0))
        else:
            dev.append_context()
            for k in range(len(dev.steps)):
                dev.run_step(k)

    def append(self):
        self.dev.append_context()

    def attention(self):
        s = self.dev.steps[-1]
        if self.shared:
            # the expanded attention on the intermediates the step's forward left
            self.api.mla_shared_attention(self.dev.handle, s["positions"], s["desc"], s["ctx"])
            return
        self.api.mla_latent_attention(self.dev.handle, self.q_abs, s["positions"], self.dev.cache,
                                      s["desc"], o_lat=self.o_lat, lse=self.lse)

    def close(self):
        self.dev.handle.close()


def run_ours(args, rank, world):
    import torch
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    S = Session(args.workload, args.overlap, args.scale)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.__enter__()
    for _ in range(args.warmup):
        S.step()
    run_s, run_a, run_t = S.step, S.append, S.attention
    if not args.no_graph:
        run_s = capture(S.step).replay
        run_a = capture(S.append).replay if S.dev.ctx is not None else None
        run_t = capture(S.attention).replay

    def hold_load(n_more, limit_s=2.0):
        # untimed replays of the same step until the clock sampler (20 ms
        # period) has n_more samples of this load: a short timed region
        # alone can end before its first sample
        if clocks.proc is None:
            return
        target, t0 = len(clocks.samples) + n_more, time.time()
        while len(clocks.samples) < target and time.time() - t0 < limit_s:
            run_s()
            torch.cuda.synchronize()

    hold_load(1)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms = timed(run_s, args.steps, flush, stream)
    # the two largest kernels alone, same protocol (the roofline line takes
    # the one with the larger time)
    kernels = {}
    if S.dev.ctx is not None:
        kernels["append"] = dict(ms=timed(run_a, args.steps, flush, stream), flops=S.fl["append"])
    kernels["attention"] = dict(ms=timed(run_t, args.steps, flush, stream),
                                flops=S.fl["attention"][-1], bytes=attention_cache_bytes(S.wl),
                                few_row=few_row_attention(S.wl), shared=S.shared)
    hold_load(2)
    clocks.__exit__(None, None, None)
    ms = max_over_ranks(ms, world)
    assert S.api.mla_get_device_status(S.dev.handle) == 0, "device status word set"
    e2e_s, h2d, d2h = measure_e2e(args, S.dev, S.step, torch)
    e2e = (max_over_ranks(e2e_s, world), h2d, d2h)
    res = dict(ms=ms, kernels=kernels, flops=S.fl, clocks=clocks.summary(), e2e=e2e,
               graphs=not args.no_graph, launches=S.launches)
    S.close()
    del S
    torch.cuda.empty_cache()
    if args.workload == WORKLOAD and args.scale == "full" and not args.no_decode:
        res["decode"] = [decode_line(name, args, flush, stream) for name in DECODE_WORKLOADS]
    return res


def decode_line(name, args, flush, stream):
    """A cached-decode workload: its whole step (both appends and forwards,
    one graph) and its last attention alone, with the cache bytes read."""
    import torch
    hbm, bf16, _, src = measured_peaks()
    S = Session(name)
    for _ in range(3):
        S.step()
    g, ga = capture(S.step), capture(S.attention)
    n = max(args.steps, 20)
    ms = timed(g.replay, n, flush, stream)
    ms_att = timed(ga.replay, n, flush, stream)
    fl = S.fl
    att_bytes = attention_cache_bytes(S.wl)
    assert S.api.mla_get_device_status(S.dev.handle) == 0
    out = {"workload": name, "shape": DESC[name], "ms_per_step": ms,
           "block_tokens_per_s": fl["block_tokens"] / (ms * 1e-3),
           "tflops": fl["total"] / (ms * 1e-3) / 1e12,
           "pct_bf16_peak": 100 * fl["total"] / (ms * 1e-3) / 1e12 / bf16,
           "cache_read_gbs": fl["cache_bytes"] / (ms * 1e-3) / 1e9,
           "pct_hbm": 100 * fl["cache_bytes"] / (ms * 1e-3) / 1e9 / hbm,
           "attention_alone": {"ms": ms_att,
                               "cache_read_gbs": att_bytes / (ms_att * 1e-3) / 1e9,
                               "pct_hbm": 100 * att_bytes / (ms_att * 1e-3) / 1e9 / hbm,
                               "tflops": fl["attention"][-1] / (ms_att * 1e-3) / 1e12,
                               "pct_bf16_peak": 100 * fl["attention"][-1] / (ms_att * 1e-3) / 1e12 / bf16},
           "peaks": f"{src}: HBM {hbm} GB/s, bf16 {bf16} TFLOP/s burst"}
    S.close()
    del S
    torch.cuda.empty_cache()
    return out


def measure_e2e(args, dev, step, torch):
    """Same step through the C ABI with host buffers: pinned host -> device
    copies of the step's inputs, the appends and forwards, device -> host of
    the outputs, all inside the timed region."""
    pairs = []
    if dev.ctx is not None:
        pairs += list(dev.ctx)
    for s in dev.steps:
        if s["append"] is not None:
            pairs += list(s["append"])
        pairs += [s["hidden"], s["positions"]] + ([s["slots"]] if s["slots"] is not None else [])
    host = [(t.cpu().pin_memory(), t) for t in pairs]
    outs = [(torch.empty(s["out"].shape, dtype=s["out"].dtype).pin_memory(), s["out"]) for s in dev.steps]
    h2d = sum(h.numel() * h.element_size() for h, _ in host)
    d2h = sum(h.numel() * h.element_size() for h, _ in outs)
    times = []
    for k in range(args.warmup + args.steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for h, d in host:
            d.copy_(h, non_blocking=True)
        step()
        for h, d in outs:
            h.copy_(d, non_blocking=True)
        torch.cuda.synchronize()
        if k >= args.warmup:
            times.append(time.perf_counter() - t0)
    return sum(times) / len(times), h2d, d2h


def cpu_baseline(workload=WORKLOAD, budget_s=15.0):
    """The fp64 oracle as it stands, on a bounded sample of the same workload:
    whole blocks (context latents of the block's sequence + the block's
    forward), as many as fit in ``budget_s``.  Returns block tokens/s."""
    from head_latent_attention_qkv_gb300 import workloads
    from oracle.keys import OracleRun
    wl = workloads.make_workload(workload)
    step = wl.steps[0]
    run = OracleRun(wl)
    t0 = time.perf_counter()
    done = 0
    rows = []
    for b in range(len(step.kv_len)):
        if wl.ctx_hidden is not None:
            rows = np.nonzero(wl.ctx_seq == step.block_seq[b])[0]
            run.append(wl.ctx_hidden, wl.ctx_positions, wl.ctx_slots, rows)
        if step.append_hidden is not None:
            r = np.arange(b * wl.block_len, (b + 1) * wl.block_len)
            run.append(step.append_hidden, step.append_positions, step.append_slots, r)
        run.forward_blocks(step, [b])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    return dict(value=done * wl.block_len / dt, unit="tokens/s", cores=cores, kind="oracle",
                sample=f"{done} of {len(step.kv_len)} blocks of the first step (each: "
                       f"{len(rows)} context-token appends, the block's own "
                       f"{wl.block_len if step.append_hidden is not None else 0}-token append "
                       f"and its {wl.block_len}-token forward), fp64 numpy, {dt:.1f} s")


def base_line(args, world):
    return {"metric": METRIC, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "data": "synthetic (seeded N(0,1) hidden, N(0,0.02) weights)",
            "config": {"workload": args.workload if args.scale == "full" else f"{args.workload} ({args.scale})",
                       "shape": DESC.get(args.workload, ""),
                       "parallelism": f"replicas x{world}",
                       "l2": "flushed (256 MB write) between steps",
                       "schedule": "append on a second stream beside the forward's projections"
                       if args.overlap else "append, then forward (one stream, one CUDA graph)"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--overlap", action="store_true",
                    help="append on a second stream beside the forward's projections")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the cached-decode lines of the default workload")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--scale", default="full", choices=["full", "medium"],
                    help="medium: the DeepSeek-V3-shaped layer on 1/64 of its batch (profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        # the reference arm is the fp64 CPU oracle; rank 0 alone runs it
        if rank != 0:
            return
        per = []
        for _ in range(args.steps):
            per.append(cpu_baseline(args.workload, budget_s=max(2.0, 60.0 / max(args.steps, 1))))
        v = statistics.median(p["value"] for p in per)
        line = base_line(args, 1)
        line["config"].update({"schedule": "fp64 oracle, one sampled block at a time, host cores",
                               "l2": "n/a (CPU)"})
        line.update({"impl": "reference", "value": v, "ms_per_step": None,
                     "dtype": "f64", "cpu_baseline": dict(per[-1], value=v),
                     "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                             "d2h_bytes_per_step": 0}})
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl")
    r = run_ours(args, rank, world)
    if rank != 0:
        torch.distributed.destroy_process_group() if world > 1 else None
        return
    hbm, bf16, bf16_sus, src = measured_peaks()
    fl = r["flops"]
    value = job_tokens_per_s(fl["block_tokens"], world, r["ms"] * 1e-3)
    tflops = fl["total"] / (r["ms"] * 1e-3) / 1e12
    names = {"append": "kv_append_tc_kernel: latent-cache append (tcgen05 GEMM N=576 + "
                       "RMSNorm/RoPE/slot scatter), the context's tokens",
             "attention": "latent_attn_tc_kernel: latent attention (tcgen05 QK^T and PV over "
                          "the 576-wide cache), the last step's blocks"}
    if r["kernels"]["attention"].get("shared"):
        names["attention"] = ("expand_attn_kernel: expanded attention (tcgen05 [q_nope|q_pe][k_nope|k_pe]^T "
                              "and P V, head dims 192 / 128) over each context's keys and the blocks' own, "
                              "the last step's blocks")
    dom = max(r["kernels"], key=lambda k: r["kernels"][k]["ms"])
    k = r["kernels"][dom]
    ach = k["flops"] / (k["ms"] * 1e-3) / 1e12
    line = base_line(args, world)
    e2e_s, h2d, d2h = r["e2e"]
    if dom == "attention" and k.get("few_row"):
        # few query rows per block: the cache stream bounds it (60 flop per cache byte at 32 rows)
        gbs = k["bytes"] / (k["ms"] * 1e-3) / 1e9
        roofline = {"kernel": "latent_decode_tc_kernel + decode_merge_kernel: few-row latent attention "
                              "(keys in the MMA's M, 32 rows in N) and its segment merge, the last step's blocks",
                    "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                    "traffic": dram_traffic("decode", args.workload),
                    "launch_ms": k["ms"], "algorithmic_bytes_per_launch": k["bytes"],
                    "share_of_step": k["ms"] / r["ms"],
                    "peak_source": f"{src} HBM copy rate; traffic is the attention kernel's, the merge adds "
                                   f"its fp32 partials"}
    else:
        roofline = {"kernel": names[dom], "bound": "tensor", "achieved": ach, "peak": bf16,
                    "unit": "TFLOP/s", "frac": ach / bf16,
                    "traffic": dram_traffic("expand" if k.get("shared") else dom, args.workload),
                    "launch_ms": k["ms"], "algorithmic_flops_per_launch": k["flops"],
                    "share_of_step": k["ms"] / r["ms"],
                    "peak_source": f"{src} bf16 burst (sustained {bf16_sus}: frac "
                                   f"{ach / bf16_sus if bf16_sus else None})"}
    others = {n: {"launch_ms": v["ms"], "tflops": v["flops"] / (v["ms"] * 1e-3) / 1e12,
                  "frac": v["flops"] / (v["ms"] * 1e-3) / 1e12 / bf16,
                  "traffic": dram_traffic("decode" if v.get("few_row") else n, args.workload)}
              for n, v in r["kernels"].items() if n != dom}
    line.update({
        "value": value, "ms_per_step": r["ms"], "dtype": "bf16",
        "tflops": tflops, "pct_bf16_peak": 100 * tflops / bf16,
        "context_tokens_per_s": world * fl["ctx_tokens"] / (r["ms"] * 1e-3),
        "cache_read_gbs": fl["cache_bytes"] / (r["ms"] * 1e-3) / 1e9,
        "pct_hbm_cache_read": 100 * fl["cache_bytes"] / (r["ms"] * 1e-3) / 1e9 / hbm,
        "roofline": roofline,
        "other_kernels": others,
        "e2e": {"value": job_tokens_per_s(fl["block_tokens"], world, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": r["launches"] * args.steps,
        "cuda_graphs": r["graphs"],
        "clocks": r["clocks"],
    })
    if "decode" in r:
        line["decode"] = r["decode"]
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
