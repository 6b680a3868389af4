"""Seeded synthetic inputs for the MLA draft-layer forward.

This module only draws random numbers and lays out indices (pages, slots,
positions, lengths).  It holds none of the layer's arithmetic, so both the
CUDA path and the CPU oracle can be fed from it without sharing any compute
code.

Conventions
-----------
* Weights follow ``torch.nn.Linear``: ``W[out, in]``, ``y = x @ W.T``.
* Linear weights ~ N(0, 0.02); RMSNorm gains ~ 1 + N(0, 0.02); hidden states
  ~ N(0, 1).  Values are drawn as fp32 from numpy's PCG64 and, for bf16
  workloads, rounded to the nearest bf16 (ties to even).  Arrays are float32
  holding exactly those values; ``bf16_bits`` gives the device bit patterns.
* Draw order is fixed: weights in ``mla_weights_t`` field order
  (fused_qkv_a_proj, q_a_layernorm, q_b_proj, q_proj, kv_a_proj_with_mqa,
  kv_a_layernorm, kv_b_proj, gate_proj, o_proj), then context hidden, block
  hidden, pre-filled cache, lengths, page permutation.
* The paged latent cache is ``[num_pages, page_size, kv_lora_rank +
  qk_rope_head_dim]``.  Token ``j`` (logical position ``j``) of a sequence
  lives at slot ``page_table[j // page_size] * page_size + j % page_size``.
  Physical page ids are a seeded permutation so that page-table indexing is
  exercised.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np


@dataclass(frozen=True)
class MLADims:
    hidden_size: int
    num_heads: int
    q_lora_rank: int            # 0 == no low-rank query (q_proj + kv_a_proj_with_mqa)
    kv_lora_rank: int
    qk_nope_head_dim: int
    qk_rope_head_dim: int
    v_head_dim: int
    rope_style: str             # "neox" | "interleaved"
    rope_theta: float
    rms_norm_eps: float = 1e-6
    use_output_gate: bool = False
    dtype: str = "bf16"         # "bf16" | "fp32"
    softmax_scale: float = 0.0  # 0 => 1/sqrt(qk_nope_head_dim + qk_rope_head_dim)
    max_position: int = 16384   # rope table length

    @property
    def qk_head_dim(self) -> int:
        return self.qk_nope_head_dim + self.qk_rope_head_dim

    @property
    def cache_dim(self) -> int:
        return self.kv_lora_rank + self.qk_rope_head_dim

    def replace(self, **kw) -> "MLADims":
        return dataclasses.replace(self, **kw)


QWEN3_4B_MLA = MLADims(hidden_size=2560, num_heads=32, q_lora_rank=1536,
                       kv_lora_rank=512, qk_nope_head_dim=128,
                       qk_rope_head_dim=64, v_head_dim=128,
                       rope_style="interleaved", rope_theta=1e6)

DEEPSEEK_V3_MLA = MLADims(hidden_size=7168, num_heads=128, q_lora_rank=1536,
                          kv_lora_rank=512, qk_nope_head_dim=128,
                          qk_rope_head_dim=64, v_head_dim=128,
                          rope_style="interleaved", rope_theta=1e4,
                          use_output_gate=True)

TINY_FP32_MLA = MLADims(hidden_size=256, num_heads=4, q_lora_rank=0,
                        kv_lora_rank=64, qk_nope_head_dim=32,
                        qk_rope_head_dim=16, v_head_dim=32,
                        rope_style="neox", rope_theta=1e4, dtype="fp32")

WEIGHT_FIELDS = ("fused_qkv_a_proj", "q_a_layernorm", "q_b_proj", "q_proj",
                 "kv_a_proj_with_mqa", "kv_a_layernorm", "kv_b_proj",
                 "gate_proj", "o_proj")


def weight_shapes(d: MLADims) -> Dict[str, Optional[tuple]]:
    """Shapes of the layer's parameters (None where the field is unused)."""
    H, D, L = d.num_heads, d.hidden_size, d.cache_dim
    s: Dict[str, Optional[tuple]] = {k: None for k in WEIGHT_FIELDS}
    if d.q_lora_rank > 0:
        s["fused_qkv_a_proj"] = (d.q_lora_rank + L, D)
        s["q_a_layernorm"] = (d.q_lora_rank,)
        s["q_b_proj"] = (H * d.qk_head_dim, d.q_lora_rank)
    else:
        s["q_proj"] = (H * d.qk_head_dim, D)
        s["kv_a_proj_with_mqa"] = (L, D)
    s["kv_a_layernorm"] = (d.kv_lora_rank,)
    s["kv_b_proj"] = (H * (d.qk_nope_head_dim + d.v_head_dim), d.kv_lora_rank)
    if d.use_output_gate:
        s["gate_proj"] = (H * d.v_head_dim, D)
    s["o_proj"] = (D, H * d.v_head_dim)
    return s


# bf16 storage rounding of generated values (a storage format, not layer arithmetic)
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _storage_round(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits_to_f32(bf16_bits(x))
    return np.ascontiguousarray(x, dtype=np.float32)


def _normal(rng: np.random.Generator, shape, std: float, mean: float,
            dtype: str, chunk: int = 1 << 24) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if mean != 0.0:
            v += np.float32(mean)
        out[s:e] = _storage_round(v, dtype)
    return out.reshape(shape)


def make_weights(d: MLADims, rng: np.random.Generator) -> Dict[str, Optional[np.ndarray]]:
    shapes = weight_shapes(d)
    w: Dict[str, Optional[np.ndarray]] = {}
    for name in WEIGHT_FIELDS:
        shp = shapes[name]
        if shp is None:
            w[name] = None
        elif name.endswith("layernorm"):
            w[name] = _normal(rng, shp, 0.02, 1.0, d.dtype)
        else:
            w[name] = _normal(rng, shp, 0.02, 0.0, d.dtype)
    return w


# --------------------------------------------------------------------------
# Workload layout
# --------------------------------------------------------------------------
@dataclass
class Step:
    """One call sequence on the device: optional appends, then one forward."""
    append_hidden: Optional[np.ndarray]      # [n, D] tokens appended before the forward
    append_positions: Optional[np.ndarray]   # [n] int32
    append_slots: Optional[np.ndarray]       # [n] int64
    block_hidden: np.ndarray                 # [nb*T, D]
    block_positions: np.ndarray              # [nb*T] int32
    block_slots: Optional[np.ndarray]        # [nb*T] int64, None => latents already appended
    block_table: np.ndarray                  # [nb, max_pages] int32
    kv_len: np.ndarray                       # [nb] int32
    window: np.ndarray                       # [nb] int32 (0 = full)
    q_visible: np.ndarray                    # [nb*T] uint8
    block_seq: np.ndarray                    # [nb] sequence id of each block


@dataclass
class Workload:
    name: str
    dims: MLADims
    seed: int
    weights: Dict[str, Optional[np.ndarray]]
    page_size: int
    num_pages: int
    block_len: int
    # context injection (target hidden states) appended once before the steps
    ctx_hidden: Optional[np.ndarray]          # [n_ctx, D]
    ctx_positions: Optional[np.ndarray]       # [n_ctx] int32
    ctx_slots: Optional[np.ndarray]           # [n_ctx] int64
    ctx_seq: Optional[np.ndarray]             # [n_ctx] sequence id
    # raw cache entries written before anything runs (cached-decode workloads)
    prefill_slots: Optional[np.ndarray]       # [n_pre] int64
    prefill_values: Optional[np.ndarray]      # [n_pre, L] float32 (storage-rounded)
    steps: List[Step] = field(default_factory=list)
    description: str = ""

    @property
    def cache_shape(self):
        return (self.num_pages, self.page_size, self.dims.cache_dim)


class _PageAllocator:
    def __init__(self, rng: np.random.Generator, total_pages: int):
        self.perm = rng.permutation(total_pages).astype(np.int32)
        self.next = 0

    def take(self, n: int) -> np.ndarray:
        p = self.perm[self.next:self.next + n]
        assert len(p) == n, "page pool exhausted"
        self.next += n
        return p


def _slots(pages: np.ndarray, page_size: int, start: int, n: int) -> np.ndarray:
    j = np.arange(start, start + n, dtype=np.int64)
    return pages[j // page_size].astype(np.int64) * page_size + j % page_size


def _pad_table(rows: List[np.ndarray]) -> np.ndarray:
    width = max(len(r) for r in rows)
    t = np.full((len(rows), width), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        t[i, :len(r)] = r
    return t


def prefill_workload(name: str, d: MLADims, seed: int, ctx_lens, block_len: int,
                     page_size: int, window: int = 0, masked_rows=None,
                     description: str = "") -> Workload:
    """Sequences of ``ctx_lens[s]`` context tokens plus one block of
    ``block_len`` draft tokens anchored right after the context.

    The context latents are appended from their own hidden states (target
    context injection); the block's latents are written by the forward.
    ``masked_rows(s) -> iterable`` lists block rows of sequence s whose query is
    fully masked.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    w = make_weights(d, rng)
    B, T = len(ctx_lens), block_len
    n_ctx = int(sum(ctx_lens))
    ctx_hidden = _normal(rng, (n_ctx, d.hidden_size), 1.0, 0.0, d.dtype)
    block_hidden = _normal(rng, (B * T, d.hidden_size), 1.0, 0.0, d.dtype)
    pages_per_seq = [-(-(c + T) // page_size) for c in ctx_lens]
    total_pages = int(sum(pages_per_seq))
    alloc = _PageAllocator(rng, total_pages)
    ctx_pos, ctx_slots, ctx_seq = [], [], []
    b_pos, b_slots, tables, kv_len = [], [], [], []
    for s, c in enumerate(ctx_lens):
        pages = alloc.take(pages_per_seq[s])
        ctx_pos.append(np.arange(c, dtype=np.int32))
        ctx_slots.append(_slots(pages, page_size, 0, c))
        ctx_seq.append(np.full(c, s, dtype=np.int32))
        b_pos.append(np.arange(c, c + T, dtype=np.int32))
        b_slots.append(_slots(pages, page_size, c, T))
        tables.append(pages)
        kv_len.append(c + T)
    q_vis = np.ones(B * T, dtype=np.uint8)
    if masked_rows is not None:
        for s in range(B):
            for r in masked_rows(s):
                q_vis[s * T + r] = 0
    step = Step(append_hidden=None, append_positions=None, append_slots=None,
                block_hidden=block_hidden, block_positions=np.concatenate(b_pos),
                block_slots=np.concatenate(b_slots), block_table=_pad_table(tables),
                kv_len=np.array(kv_len, dtype=np.int32),
                window=np.full(B, window, dtype=np.int32), q_visible=q_vis,
                block_seq=np.arange(B, dtype=np.int32))
    return Workload(name=name, dims=d, seed=seed, weights=w, page_size=page_size,
                    num_pages=total_pages, block_len=T, ctx_hidden=ctx_hidden,
                    ctx_positions=np.concatenate(ctx_pos), ctx_slots=np.concatenate(ctx_slots),
                    ctx_seq=np.concatenate(ctx_seq), prefill_slots=None, prefill_values=None,
                    steps=[step], description=description)


def block_parallel_workload(name: str, d: MLADims, seed: int, batch: int, ctx_len: int,
                            blocks_per_seq: int, block_len: int, page_size: int,
                            windows=(0,), description: str = "") -> Workload:
    """Each sequence has one context of ``ctx_len`` tokens and
    ``blocks_per_seq`` independent proposals, all anchored right after the
    context (positions ctx_len .. ctx_len+T-1), each with a private page for
    its own latents.  Block j of a sequence uses ``windows[j % len(windows)]``.
    """
    assert ctx_len % page_size == 0, "proposal pages must not share the context's last page"
    rng = np.random.Generator(np.random.PCG64(seed))
    w = make_weights(d, rng)
    T = block_len
    ctx_hidden = _normal(rng, (batch * ctx_len, d.hidden_size), 1.0, 0.0, d.dtype)
    nb = batch * blocks_per_seq
    block_hidden = _normal(rng, (nb * T, d.hidden_size), 1.0, 0.0, d.dtype)
    ctx_pages = ctx_len // page_size
    priv_pages = -(-T // page_size)
    total_pages = batch * (ctx_pages + blocks_per_seq * priv_pages)
    alloc = _PageAllocator(rng, total_pages)
    ctx_pos, ctx_slots, ctx_seq = [], [], []
    b_pos, b_slots, tables, kv_len, win, bseq = [], [], [], [], [], []
    for s in range(batch):
        cp = alloc.take(ctx_pages)
        ctx_pos.append(np.arange(ctx_len, dtype=np.int32))
        ctx_slots.append(_slots(cp, page_size, 0, ctx_len))
        ctx_seq.append(np.full(ctx_len, s, dtype=np.int32))
        for j in range(blocks_per_seq):
            pages = np.concatenate([cp, alloc.take(priv_pages)])
            b_pos.append(np.arange(ctx_len, ctx_len + T, dtype=np.int32))
            b_slots.append(_slots(pages, page_size, ctx_len, T))
            tables.append(pages)
            kv_len.append(ctx_len + T)
            win.append(windows[j % len(windows)])
            bseq.append(s)
    step = Step(append_hidden=None, append_positions=None, append_slots=None,
                block_hidden=block_hidden, block_positions=np.concatenate(b_pos),
                block_slots=np.concatenate(b_slots), block_table=_pad_table(tables),
                kv_len=np.array(kv_len, dtype=np.int32), window=np.array(win, dtype=np.int32),
                q_visible=np.ones(nb * T, dtype=np.uint8), block_seq=np.array(bseq, dtype=np.int32))
    return Workload(name=name, dims=d, seed=seed, weights=w, page_size=page_size,
                    num_pages=total_pages, block_len=T, ctx_hidden=ctx_hidden,
                    ctx_positions=np.concatenate(ctx_pos), ctx_slots=np.concatenate(ctx_slots),
                    ctx_seq=np.concatenate(ctx_seq), prefill_slots=None, prefill_values=None,
                    steps=[step], description=description)


def cached_decode_workload(name: str, d: MLADims, seed: int, batch: int, prefill_len: int,
                           len_lo: int, len_hi: int, block_len: int, num_blocks: int,
                           page_size: int, description: str = "") -> Workload:
    """Latent cache pre-filled with ``prefill_len`` random entries per sequence;
    sequence s keeps the first ``L_s ~ U{len_lo..len_hi}`` of them as context.
    Then ``num_blocks`` consecutive blocks are each appended through the
    latent-append call and attended (the forward does not write latents).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    w = make_weights(d, rng)
    T = block_len
    hid = [_normal(rng, (batch * T, d.hidden_size), 1.0, 0.0, d.dtype) for _ in range(num_blocks)]
    cap = max(prefill_len, len_hi + num_blocks * T)
    pages_per_seq = -(-cap // page_size)
    total_pages = batch * pages_per_seq
    pre_vals = _normal(rng, (batch * prefill_len, d.cache_dim), 1.0, 0.0, d.dtype)
    lens = rng.integers(len_lo, len_hi + 1, size=batch).astype(np.int32)
    alloc = _PageAllocator(rng, total_pages)
    tables = [alloc.take(pages_per_seq) for _ in range(batch)]
    pre_slots = np.concatenate([_slots(tables[s], page_size, 0, prefill_len) for s in range(batch)])
    steps = []
    for k in range(num_blocks):
        pos = np.concatenate([np.arange(lens[s] + k * T, lens[s] + (k + 1) * T, dtype=np.int32)
                              for s in range(batch)])
        slots = np.concatenate([_slots(tables[s], page_size, int(lens[s]) + k * T, T)
                                for s in range(batch)])
        steps.append(Step(append_hidden=hid[k], append_positions=pos, append_slots=slots,
                          block_hidden=hid[k], block_positions=pos, block_slots=None,
                          block_table=_pad_table(tables),
                          kv_len=(lens + (k + 1) * T).astype(np.int32),
                          window=np.zeros(batch, dtype=np.int32),
                          q_visible=np.ones(batch * T, dtype=np.uint8),
                          block_seq=np.arange(batch, dtype=np.int32)))
    return Workload(name=name, dims=d, seed=seed, weights=w, page_size=page_size,
                    num_pages=total_pages, block_len=T, ctx_hidden=None, ctx_positions=None,
                    ctx_slots=None, ctx_seq=None, prefill_slots=pre_slots,
                    prefill_values=pre_vals, steps=steps, description=description)


def attention_inputs(wl: Workload, step: Step, seed: int):
    """Seeded inputs for the latent attention step alone: absorbed query rows
    ``[tokens * heads, cache_dim]`` (token-major, N(0, 1)) and every slot of
    the paged cache ``[num_pages * page_size, cache_dim]`` (N(0, 1)), both
    rounded to the layer dtype."""
    rng = np.random.Generator(np.random.PCG64(seed))
    d = wl.dims
    rows = len(step.block_positions) * d.num_heads
    q = _normal(rng, (rows, d.cache_dim), 1.0, 0.0, d.dtype)
    cache = _normal(rng, (wl.num_pages * wl.page_size, d.cache_dim), 1.0, 0.0, d.dtype)
    return q, cache


def attention_grad_inputs(wl: Workload, step: Step, seed: int):
    """Seeded upstream gradient of the latent attention output:
    ``[tokens * heads, kv_lora_rank]`` float32, N(0, 1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    d = wl.dims
    rows = len(step.block_positions) * d.num_heads
    return _normal(rng, (rows, d.kv_lora_rank), 1.0, 0.0, "fp32")


# --------------------------------------------------------------------------
# The named workloads (full sizes) and their shrunken parity variants
# --------------------------------------------------------------------------
WORKLOADS = ("tiny_fp32", "qwen3_4b_prefill", "qwen3_4b_sliding_gate",
             "qwen3_4b_cached_decode", "deepseek_v3_block_parallel", "qwen3_4b_decode_t1")


def make_workload(name: str, scale: str = "full") -> Workload:
    """Build a named workload.  ``scale='small'`` keeps the layer dims but
    shrinks batch/context so the fp64 oracle runs the whole thing in seconds,
    with ragged context lengths that leave partial tiles and pages;
    ``scale='medium'`` (DeepSeek-V3-shaped layer only) keeps the per-block
    shapes at 1/64 of the batch."""
    small = scale == "small"
    if name == "tiny_fp32":
        return prefill_workload(name, TINY_FP32_MLA, 0, [64], 8, page_size=16,
                                description="fp32; 1 x (64 context + 8-token block), full mask")
    if name == "qwen3_4b_prefill":
        d = QWEN3_4B_MLA
        if small:
            return prefill_workload(name, d, 1, [200, 77, 131], 16, page_size=64,
                                    description="3 x (ragged context + 16-token block), full mask")
        return prefill_workload(name, d, 1, [2048] * 8, 16, page_size=128,
                                description="8 x (2048 context + 16-token block), full mask")
    if name == "qwen3_4b_sliding_gate":
        d = QWEN3_4B_MLA.replace(use_output_gate=True, rope_style="neox")
        masked = lambda s: range(4) if s % 4 == 0 else ()
        if small:
            return prefill_workload(name, d, 2, [700, 300, 97, 1000, 513], 16, page_size=128,
                                    window=512, masked_rows=masked,
                                    description="5 x (ragged context + 16), sliding 512, gate")
        return prefill_workload(name, d, 2, [8192] * 16, 16, page_size=128, window=512,
                                masked_rows=masked,
                                description="16 x (8192 context + 16), sliding 512, gate")
    if name == "qwen3_4b_cached_decode":
        d = QWEN3_4B_MLA
        if small:
            return cached_decode_workload(name, d, 3, batch=5, prefill_len=512, len_lo=100,
                                          len_hi=512, block_len=16, num_blocks=2, page_size=32,
                                          description="5 seqs, prefilled 512, 2 cached blocks")
        return cached_decode_workload(name, d, 3, batch=64, prefill_len=4096, len_lo=1024,
                                      len_hi=4096, block_len=16, num_blocks=2, page_size=128,
                                      description="64 seqs, prefilled 4096, L~U[1024,4096], 2 blocks")
    if name == "qwen3_4b_decode_t1":
        # one query token per step (block_len 1): 32 query rows per sequence, the
        # regime where the cache stream, not the tensor pipe, bounds the attention
        d = QWEN3_4B_MLA
        if small:
            return cached_decode_workload(name, d, 5, batch=5, prefill_len=512, len_lo=100,
                                          len_hi=512, block_len=1, num_blocks=2, page_size=32,
                                          description="5 seqs, prefilled 512, 2 one-token steps")
        return cached_decode_workload(name, d, 5, batch=64, prefill_len=4096, len_lo=1024,
                                      len_hi=4096, block_len=1, num_blocks=2, page_size=128,
                                      description="64 seqs, prefilled 4096, L~U[1024,4096], 2 one-token steps")
    if name == "deepseek_v3_block_parallel":
        d = DEEPSEEK_V3_MLA
        if scale == "medium":
            # the same per-block work (16 x 128 query rows over a 4096-token
            # context) on one sequence of 64 proposals: absorbed queries of
            # 151 MB, more than L2, a few GB in all (profiling captures)
            return block_parallel_workload(name, d, 4, batch=1, ctx_len=4096, blocks_per_seq=64,
                                           block_len=16, page_size=128, windows=(0, 1024),
                                           description="1 x 64 proposals of 16 over 4096 context")
        if small:
            return block_parallel_workload(name, d, 4, batch=2, ctx_len=192, blocks_per_seq=3,
                                           block_len=16, page_size=64, windows=(0, 100),
                                           description="2 seqs x 3 proposals over 192 context")
        return block_parallel_workload(name, d, 4, batch=4, ctx_len=4096, blocks_per_seq=1024,
                                       block_len=16, page_size=128, windows=(0, 1024),
                                       description="4 x 1024 proposals of 16 over 4096 context")
    raise KeyError(name)
