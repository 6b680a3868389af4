"""Benchmark of the MLA draft-layer hot path on GB300.

One step = the whole path over one batch of the Qwen3-4B-sized block-prefill
workload (8 sequences x (2048 context tokens + one 16-token draft block),
bf16): latent-cache append of the 16384 context tokens, then the draft-layer
forward of the 128 block tokens, captured in one CUDA graph (``--overlap``
runs the append on a second stream beside the forward's projections, the
forward's attention waiting for it through ``mla_draft_forward_after``).
Inputs are seeded synthetic data resident in HBM; L2 (126 MB) is flushed by
writing a 256 MB buffer between timed steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

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

WORKLOAD = "qwen3_4b_prefill"
METRIC = "MLA draft-layer tokens/s (block query tokens; TFLOP/s and %bf16 peak alongside)"


def algorithmic_flops(wl):
    """Absorbed latent path: per block token 2D(r_q+L) [+2D*H*dv gate] +
    2 r_q H dqk + 2 H dn r_kv + 2 H r_kv dv + 2 H dv D, per visible key
    H (2L + 2 r_kv); per appended token 2 D L.  Also the cache bytes the
    attention reads (1152 B per key a block can see, once per block)."""
    d = wl.dims
    H, D, L = d.num_heads, d.hidden_size, d.cache_dim
    qdim = d.q_lora_rank if d.q_lora_rank else H * d.qk_head_dim
    per_tok = 2 * D * (qdim + L) + (2 * D * H * d.v_head_dim if d.use_output_gate else 0)
    if d.q_lora_rank:
        per_tok += 2 * d.q_lora_rank * H * d.qk_head_dim
    per_tok += 2 * H * d.qk_nope_head_dim * d.kv_lora_rank + 2 * H * d.kv_lora_rank * d.v_head_dim
    per_tok += 2 * H * d.v_head_dim * D
    T = wl.block_len
    total = block_tokens = cache_bytes = 0
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
        total += per_tok * len(step.block_positions) + H * (2 * L + 2 * d.kv_lora_rank) * keys
        block_tokens += len(step.block_positions)
        if step.append_hidden is not None:
            appended += len(step.append_hidden)
    append = 2 * D * L * (0 if wl.ctx_hidden is None else len(wl.ctx_hidden))
    total += 2 * D * L * (appended - (0 if wl.ctx_hidden is None else len(wl.ctx_hidden))) + append
    return dict(total=total, append=append, block_tokens=block_tokens, ctx_tokens=appended,
                cache_bytes=cache_bytes)


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


def append_traffic():
    """DRAM bytes per launch of the append kernel from the committed ncu
    summary, or None when the kernel source changed since that capture."""
    import hashlib
    src = os.path.join(ROOT, "head_latent_attention_qkv_gb300", "csrc", "append_tc.cu")
    summ = os.path.join(ROOT, "profiles", "ncu_kv_append_qwen3_4b_prefill.md")
    if not (os.path.exists(src) and os.path.exists(summ)):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    vals = {}
    for line in open(summ):
        key = line.strip().lstrip("-* `")
        if ":" in key and key.startswith(("traffic_bytes_per_launch", "kernel_source_sha256")):
            k, v = key.split(":", 1)
            vals[k.strip().strip("`")] = v.strip().strip("` ")
    if vals.get("kernel_source_sha256") != digest:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
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


def run_ours(args, rank, world):
    import torch
    from head_latent_attention_qkv_gb300 import api, workloads
    from head_latent_attention_qkv_gb300.runner import DeviceWorkload

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    wl = workloads.make_workload(args.workload)
    fl = algorithmic_flops(wl)
    dev = DeviceWorkload(wl)
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def append():
        dev.append_context()

    def step():
        # one step: the context append, then each step's appends and forward
        # (--overlap: the appends on a second stream beside the forward's
        # projections; the attention waits for them)
        if args.overlap:
            for k in range(len(dev.steps)):
                dev.run_step_after(k, side, with_context=(k == 0))
        else:
            dev.append_context()
            for k in range(len(dev.steps)):
                dev.run_step(k)

    dev.reset_cache()
    torch.cuda.synchronize()
    n0 = api._lib.lib.mla_kernel_launches(dev.handle.h)
    step()
    launches = int(api._lib.lib.mla_kernel_launches(dev.handle.h) - n0)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.__enter__()
    for _ in range(args.warmup):
        step()
    run_s, run_a = step, append
    if not args.no_graph:
        graphs = []
        for fn in (step, append):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            graphs.append(g)
        for _ in range(2):
            for g in graphs:
                g.replay()
        run_s, run_a = graphs[0].replay, graphs[1].replay

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
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for k in range(args.steps):
        flush.fill_(k & 0xFF)                      # evict L2 between steps (untimed)
        ev[k][0].record(stream)
        run_s()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    t_step = [e[0].elapsed_time(e[1]) for e in ev]
    # the context append alone (its kernel is the roofline line), same protocol
    t_app = []
    if dev.ctx is not None:
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            ev[k][0].record(stream)
            run_a()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        t_app = [e[0].elapsed_time(e[1]) for e in ev]
    hold_load(2)
    clocks.__exit__(None, None, None)
    ms = max_over_ranks(sum(t_step) / len(t_step), world)
    assert api.mla_get_device_status(dev.handle) == 0, "device status word set"
    e2e_s, h2d, d2h = measure_e2e(args, dev, step, torch)
    e2e = (max_over_ranks(e2e_s, world), h2d, d2h)
    return dict(ms=ms, ms_append=sum(t_app) / len(t_app) if t_app else None, flops=fl,
                clocks=clocks.summary(), e2e=e2e, graphs=not args.no_graph, launches=launches)


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
    from head_latent_attention_qkv_gb300 import workloads
    desc = {"tiny_fp32": "1 x (64 context + 8-token block), fp32",
            "qwen3_4b_prefill": "8 x (2048 context + 16-token block), full mask",
            "qwen3_4b_sliding_gate": "16 x (8192 context + 16), sliding 512, gate, masked rows",
            "qwen3_4b_cached_decode": "64 seqs, cache pre-filled, 2 consecutive 16-token blocks",
            "deepseek_v3_block_parallel": "4 x 1024 proposals of 16 over a 4096 context, gate",
            "qwen3_4b_decode_t1": "64 seqs, cache pre-filled, 2 consecutive one-token steps"}
    return {"metric": METRIC, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "data": "synthetic (seeded N(0,1) hidden, N(0,0.02) weights)",
            "config": {"workload": args.workload, "shape": desc.get(args.workload, ""),
                       "parallelism": f"replicas x{world}",
                       "l2": "flushed (256 MB write) between steps",
                       "schedule": "append on a second stream beside the forward's projections"
                       if args.overlap else "append, then forward (one stream, one CUDA graph)"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--overlap", action="store_true",
                    help="append on a second stream beside the forward's projections")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD)
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
    if fl["append"]:
        t_app = r["ms_append"] * 1e-3
        ach, rl_kernel = fl["append"] / t_app / 1e12, "latent-cache append (tcgen05 GEMM N=576 + RMSNorm/RoPE/slot scatter)"
    else:   # no context append in this workload: the whole step against the tensor peak
        ach, rl_kernel = fl["total"] / (r["ms"] * 1e-3) / 1e12, "whole step (appends + forwards)"
    line = base_line(args, world)
    e2e_s, h2d, d2h = r["e2e"]
    line.update({
        "value": value, "ms_per_step": r["ms"], "dtype": "bf16",
        "tflops": tflops, "pct_bf16_peak": 100 * tflops / bf16,
        "context_tokens_per_s": world * fl["ctx_tokens"] / (r["ms"] * 1e-3),
        "cache_read_gbs": fl["cache_bytes"] / (r["ms"] * 1e-3) / 1e9,
        "pct_hbm_cache_read": 100 * fl["cache_bytes"] / (r["ms"] * 1e-3) / 1e9 / hbm,
        "roofline": {"kernel": rl_kernel,
                     "bound": "tensor", "achieved": ach, "peak": bf16, "unit": "TFLOP/s",
                     "frac": ach / bf16,
                     "traffic": append_traffic() if fl["append"] and args.workload == WORKLOAD else None,
                     "peak_source": f"{src} bf16 burst"},
        "e2e": {"value": job_tokens_per_s(fl["block_tokens"], world, e2e_s), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": r["launches"] * args.steps,
        "cuda_graphs": r["graphs"],
        "clocks": r["clocks"],
    })
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
