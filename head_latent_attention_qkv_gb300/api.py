"""Python entry points with the C ABI's names, taking torch tensors.

Marshalling only: pointers, sizes and the current CUDA stream are passed to
``libmla_draft.so``; torch allocates the caller-owned device buffers (weight
arena, workspace, outputs).  Tensors must already be on the CUDA device, of the
layer's dtype (weights, hidden, cache, out) or int32/int64/uint8 for indices.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib
from ._lib import check, lib

_TORCH_DTYPE = {"bf16": torch.bfloat16, "fp32": torch.float32}


def torch_dtype(dims) -> torch.dtype:
    return _TORCH_DTYPE[dims.dtype]


def make_config(dims, page_size: int) -> _lib.mla_config_t:
    return _lib.mla_config_t(
        hidden_size=dims.hidden_size, num_heads=dims.num_heads, q_lora_rank=dims.q_lora_rank,
        kv_lora_rank=dims.kv_lora_rank, qk_nope_head_dim=dims.qk_nope_head_dim,
        qk_rope_head_dim=dims.qk_rope_head_dim, v_head_dim=dims.v_head_dim,
        rope=_lib.MLA_ROPE_INTERLEAVED if dims.rope_style == "interleaved" else _lib.MLA_ROPE_NEOX,
        use_output_gate=int(bool(dims.use_output_gate)),
        dtype=_lib.MLA_BF16 if dims.dtype == "bf16" else _lib.MLA_FP32, page_size=page_size,
        max_position=dims.max_position, rope_theta=dims.rope_theta,
        rms_norm_eps=dims.rms_norm_eps, softmax_scale=dims.softmax_scale)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _buf(nbytes: int, device) -> torch.Tensor:
    # 256-byte aligned: the caching allocator hands out 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class Handle:
    """A library handle plus the device buffers the caller owns for it."""

    def __init__(self, dims, weights: dict, page_size: int, device="cuda", stream=None):
        self.dims, self.page_size, self.device = dims, page_size, torch.device(device)
        self.cfg = make_config(dims, page_size)
        self.arena = _buf(lib.mla_weight_arena_bytes(C.byref(self.cfg)), self.device)
        w = _lib.mla_weights_t(**{k: (weights[k].data_ptr() if weights.get(k) is not None else None)
                                  for k in _lib.WEIGHT_FIELDS})
        h = C.c_void_p()
        check(lib.mla_draft_init(C.byref(self.cfg), C.byref(w), _ptr(self.arena),
                                 self.arena.numel(), _stream(stream), C.byref(h)), "mla_draft_init")
        self.h = h
        self._ws = None

    def workspace(self, nbytes: int) -> torch.Tensor:
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = _buf(nbytes, self.device)
        return self._ws

    def close(self):
        if self.h:
            lib.mla_draft_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mla_draft_init(dims, weights: dict, page_size: int, device="cuda", stream=None) -> Handle:
    return Handle(dims, weights, page_size, device, stream)


def mla_latent_cache_append(h: Handle, hidden, positions, slot_mapping, cache, stream=None,
                            workspace=None):
    n = hidden.shape[0]
    need = lib.mla_append_workspace_bytes(h.h, n)
    ws = workspace if workspace is not None else h.workspace(need)
    check(lib.mla_latent_cache_append(h.h, _ptr(hidden), _ptr(positions), _ptr(slot_mapping), n,
                                      _ptr(cache), cache.shape[0], _ptr(ws), ws.numel(),
                                      _stream(stream)), "mla_latent_cache_append")


def make_desc(block_table, kv_len, window=None, q_visible=None, block_len=16, vis_stats=None):
    return _lib.mla_attn_desc_t(
        num_blocks=block_table.shape[0], block_len=block_len, max_pages=block_table.shape[1],
        reserved=0, block_table=block_table.data_ptr(), kv_len=kv_len.data_ptr(),
        window=None if window is None else window.data_ptr(),
        q_visible=None if q_visible is None else q_visible.data_ptr(),
        vis_stats=None if vis_stats is None else vis_stats.data_ptr())


def mla_draft_forward(h: Handle, hidden, positions, block_slot_mapping, cache, desc, out=None,
                      stream=None, workspace=None):
    M = desc.num_blocks * desc.block_len
    if out is None:
        out = torch.empty(M, h.dims.hidden_size, dtype=torch_dtype(h.dims), device=h.device)
    need = lib.mla_forward_workspace_bytes(h.h, M)
    ws = workspace if workspace is not None else h.workspace(need)
    check(lib.mla_draft_forward(h.h, _ptr(hidden), _ptr(positions), _ptr(block_slot_mapping),
                                _ptr(cache), cache.shape[0], C.byref(desc), _ptr(out), _ptr(ws),
                                ws.numel(), _stream(stream)), "mla_draft_forward")
    return out


def make_shared_ctx(ctx_len, ctx_block_start, ctx_rows):
    """Context list for mla_draft_forward_shared: device int32 ``ctx_len``
    [num_ctx] and ``ctx_block_start`` [num_ctx + 1]; ``ctx_rows`` (host int)
    is the sum of ``ctx_len``."""
    return _lib.mla_shared_ctx_t(num_ctx=ctx_len.shape[0], ctx_rows=int(ctx_rows),
                                 ctx_len=ctx_len.data_ptr(), ctx_block_start=ctx_block_start.data_ptr())


def mla_draft_forward_shared(h: Handle, hidden, positions, block_slot_mapping, cache, desc, ctx,
                             out=None, stream=None, workspace=None):
    """mla_draft_forward for blocks that share contexts (``ctx`` from
    make_shared_ctx): the expanded form where the layer allows it."""
    M = desc.num_blocks * desc.block_len
    if out is None:
        out = torch.empty(M, h.dims.hidden_size, dtype=torch_dtype(h.dims), device=h.device)
    need = lib.mla_forward_shared_workspace_bytes(h.h, M, ctx.ctx_rows)
    ws = workspace if workspace is not None else h.workspace(need)
    check(lib.mla_draft_forward_shared(h.h, _ptr(hidden), _ptr(positions), _ptr(block_slot_mapping),
                                       _ptr(cache), cache.shape[0], C.byref(desc), C.byref(ctx),
                                       _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
          "mla_draft_forward_shared")
    return out


def mla_draft_forward_shared_after(h: Handle, hidden, positions, block_slot_mapping, cache, desc,
                                   ctx, cache_ready=None, out=None, stream=None, workspace=None):
    """mla_draft_forward_shared whose attention waits for ``cache_ready``
    (a recorded torch.cuda.Event, or None)."""
    M = desc.num_blocks * desc.block_len
    if out is None:
        out = torch.empty(M, h.dims.hidden_size, dtype=torch_dtype(h.dims), device=h.device)
    need = lib.mla_forward_shared_workspace_bytes(h.h, M, ctx.ctx_rows)
    ws = workspace if workspace is not None else h.workspace(need)
    ev = None if cache_ready is None else C.c_void_p(cache_ready.cuda_event)
    check(lib.mla_draft_forward_shared_after(h.h, _ptr(hidden), _ptr(positions),
                                             _ptr(block_slot_mapping), _ptr(cache), cache.shape[0],
                                             C.byref(desc), C.byref(ctx), _ptr(out), _ptr(ws),
                                             ws.numel(), _stream(stream), ev),
          "mla_draft_forward_shared_after")
    return out


def mla_shared_attention(h: Handle, positions, desc, ctx, workspace=None, stream=None):
    """The expanded attention step alone, on the intermediates the last
    mla_draft_forward_shared left in the workspace (the handle's unless
    given); rewrites that workspace's per-head output o."""
    M = desc.num_blocks * desc.block_len
    need = lib.mla_forward_shared_workspace_bytes(h.h, M, ctx.ctx_rows)
    ws = workspace if workspace is not None else h.workspace(need)
    check(lib.mla_shared_attention(h.h, _ptr(positions), C.byref(desc), C.byref(ctx), _ptr(ws),
                                   ws.numel(), _stream(stream)), "mla_shared_attention")


def mla_draft_forward_after(h: Handle, hidden, positions, block_slot_mapping, cache, desc,
                            cache_ready=None, out=None, stream=None, workspace=None):
    """mla_draft_forward whose attention waits for ``cache_ready`` (a
    recorded torch.cuda.Event, or None)."""
    M = desc.num_blocks * desc.block_len
    if out is None:
        out = torch.empty(M, h.dims.hidden_size, dtype=torch_dtype(h.dims), device=h.device)
    need = lib.mla_forward_workspace_bytes(h.h, M)
    ws = workspace if workspace is not None else h.workspace(need)
    ev = None if cache_ready is None else C.c_void_p(cache_ready.cuda_event)
    check(lib.mla_draft_forward_after(h.h, _ptr(hidden), _ptr(positions), _ptr(block_slot_mapping),
                                      _ptr(cache), cache.shape[0], C.byref(desc), _ptr(out),
                                      _ptr(ws), ws.numel(), _stream(stream), ev),
          "mla_draft_forward_after")
    return out


def mla_latent_attention(h: Handle, q_abs, positions, cache, desc, o_lat=None, lse=None,
                         stream=None, workspace=None):
    """The latent attention step alone: ``o_lat`` [rows, kv_lora_rank] (fp16
    for bf16 layers) and, when ``lse`` is given, its fp32 [rows] log-sum-exp.
    The workspace the few-row kernel needs comes from the handle unless given."""
    rows = desc.num_blocks * desc.block_len * h.dims.num_heads
    if o_lat is None:
        dt = torch.float16 if h.dims.dtype == "bf16" else torch.float32
        o_lat = torch.empty(rows, h.dims.kv_lora_rank, dtype=dt, device=h.device)
    need = lib.mla_latent_attention_workspace_bytes(h.h, C.byref(desc))
    ws = workspace if workspace is not None else (h.workspace(need) if need else None)
    check(lib.mla_latent_attention(h.h, _ptr(q_abs), _ptr(positions), _ptr(cache),
                                   cache.shape[0], C.byref(desc), _ptr(o_lat), _ptr(lse),
                                   _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)),
          "mla_latent_attention")
    return o_lat


def mla_latent_attention_workspace_bytes(h: Handle, desc) -> int:
    return int(lib.mla_latent_attention_workspace_bytes(h.h, C.byref(desc)))


def mla_latent_attention_backward(h: Handle, q_abs, positions, cache, desc, o_lat, lse, d_o_lat,
                                  d_q_abs, d_cache, stream=None):
    """Gradients of the latent attention step: d_q_abs (written) and d_cache
    (added to; fp32, zeroed by the caller)."""
    check(lib.mla_latent_attention_backward(h.h, _ptr(q_abs), _ptr(positions), _ptr(cache),
                                            cache.shape[0], C.byref(desc), _ptr(o_lat), _ptr(lse),
                                            _ptr(d_o_lat), _ptr(d_q_abs), _ptr(d_cache),
                                            _stream(stream)), "mla_latent_attention_backward")


def mla_check_wait_timeout(h: Handle, max_rounds: int, gave_up, stream=None):
    """Self-check of the bounded-wait failure path (``gave_up``: a device
    int32 tensor of one element, set to 1 when the wait gave up)."""
    check(lib.mla_check_wait_timeout(h.h, max_rounds, _ptr(gave_up), _stream(stream)),
          "mla_check_wait_timeout")


def mla_forward_workspace_offset(h: Handle, num_tokens: int, part: int) -> int:
    return int(lib.mla_forward_workspace_offset(h.h, num_tokens, part))


def mla_latent_cache_append_noalloc(h: Handle, hidden, positions, slot_mapping, cache,
                                    stream=None):
    """The allocation-free append (library-owned fixed scratch; at most
    mla_append_noalloc_max_tokens(h) tokens per call)."""
    check(lib.mla_latent_cache_append_noalloc(h.h, _ptr(hidden), _ptr(positions),
                                              _ptr(slot_mapping), hidden.shape[0], _ptr(cache),
                                              cache.shape[0], _stream(stream)),
          "mla_latent_cache_append_noalloc")


def mla_append_noalloc_max_tokens(h: Handle) -> int:
    return int(lib.mla_append_noalloc_max_tokens(h.h))


def mla_kernel_launches(h: Handle) -> int:
    return int(lib.mla_kernel_launches(h.h))


def mla_cache_entry_dim(dims, page_size: int = 64) -> int:
    return int(lib.mla_cache_entry_dim(C.byref(make_config(dims, page_size))))


def mla_cache_page_bytes(dims, page_size: int) -> int:
    return int(lib.mla_cache_page_bytes(C.byref(make_config(dims, page_size))))


def mla_weight_arena_bytes(dims, page_size: int = 64) -> int:
    return int(lib.mla_weight_arena_bytes(C.byref(make_config(dims, page_size))))


def mla_get_device_status(h: Handle, stream=None) -> int:
    bits = C.c_int32(0)
    lib.mla_get_device_status(h.h, _stream(stream), C.byref(bits))
    return bits.value
