"""ctypes binding of ``libmla_draft.so`` (C ABI in ``include/mla_draft.h``).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  torch is used for device memory and streams.  If the shared library
is missing the import of this module fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmla_draft.so")

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA, MLA_ERR_DEVICE_CHECK, MLA_ERR_TIMEOUT = range(6)
MLA_BF16, MLA_FP32 = 0, 1
MLA_ROPE_NEOX, MLA_ROPE_INTERLEAVED = 0, 1
MLA_DEV_BAD_SLOT, MLA_DEV_BAD_POSITION, MLA_DEV_BAD_PAGE, MLA_DEV_TIMEOUT, MLA_DEV_BAD_LENGTH = 1, 2, 4, 8, 16
MLA_DEV_BAD_WINDOW = 32
MLA_WS_Q_ABS, MLA_WS_O_LAT, MLA_WS_O = 0, 1, 2


class mla_config_t(C.Structure):
    _fields_ = [(n, C.c_int32) for n in (
        "hidden_size", "num_heads", "q_lora_rank", "kv_lora_rank", "qk_nope_head_dim",
        "qk_rope_head_dim", "v_head_dim", "rope", "use_output_gate", "dtype", "page_size",
        "max_position")] + [("rope_theta", C.c_double), ("rms_norm_eps", C.c_double),
                            ("softmax_scale", C.c_double)]


WEIGHT_FIELDS = ("fused_qkv_a_proj", "q_a_layernorm", "q_b_proj", "q_proj", "kv_a_proj_with_mqa",
                 "kv_a_layernorm", "kv_b_proj", "gate_proj", "o_proj")


class mla_weights_t(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in WEIGHT_FIELDS]


class mla_attn_desc_t(C.Structure):
    _fields_ = [("num_blocks", C.c_int32), ("block_len", C.c_int32), ("max_pages", C.c_int32),
                ("reserved", C.c_int32), ("block_table", C.c_void_p), ("kv_len", C.c_void_p),
                ("window", C.c_void_p), ("q_visible", C.c_void_p), ("vis_stats", C.c_void_p)]


class mla_shared_ctx_t(C.Structure):
    _fields_ = [("num_ctx", C.c_int32), ("ctx_rows", C.c_int32), ("ctx_len", C.c_void_p),
                ("ctx_block_start", C.c_void_p)]


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: status {status}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with head_latent_attention_qkv_gb300.build")
    lib = C.CDLL(LIB_PATH)
    P, I32, SZ = C.c_void_p, C.c_int32, C.c_size_t
    sig = {
        "mla_status_string": (C.c_char_p, [I32]),
        "mla_last_error": (C.c_char_p, []),
        "mla_cache_entry_dim": (I32, [C.POINTER(mla_config_t)]),
        "mla_cache_page_bytes": (SZ, [C.POINTER(mla_config_t)]),
        "mla_weight_arena_bytes": (SZ, [C.POINTER(mla_config_t)]),
        "mla_draft_init": (I32, [C.POINTER(mla_config_t), C.POINTER(mla_weights_t), P, SZ, P,
                                 C.POINTER(P)]),
        "mla_append_workspace_bytes": (SZ, [P, I32]),
        "mla_forward_workspace_bytes": (SZ, [P, I32]),
        "mla_latent_cache_append": (I32, [P, P, P, P, I32, P, I32, P, SZ, P]),
        "mla_draft_forward": (I32, [P, P, P, P, P, I32, C.POINTER(mla_attn_desc_t), P, P, SZ, P]),
        "mla_draft_forward_after": (I32, [P, P, P, P, P, I32, C.POINTER(mla_attn_desc_t), P, P, SZ,
                                          P, P]),
        "mla_forward_shared_workspace_bytes": (SZ, [P, I32, I32]),
        "mla_draft_forward_shared": (I32, [P, P, P, P, P, I32, C.POINTER(mla_attn_desc_t),
                                           C.POINTER(mla_shared_ctx_t), P, P, SZ, P]),
        "mla_draft_forward_shared_after": (I32, [P, P, P, P, P, I32, C.POINTER(mla_attn_desc_t),
                                                 C.POINTER(mla_shared_ctx_t), P, P, SZ, P, P]),
        "mla_shared_attention": (I32, [P, P, C.POINTER(mla_attn_desc_t), C.POINTER(mla_shared_ctx_t),
                                       P, SZ, P]),
        "mla_get_device_status": (I32, [P, P, C.POINTER(I32)]),
        "mla_draft_destroy": (None, [P]),
        "mla_kernel_launches": (C.c_ulonglong, [P]),
        "mla_latent_cache_append_noalloc": (I32, [P, P, P, P, I32, P, I32, P]),
        "mla_append_noalloc_max_tokens": (C.c_int64, [P]),
        "mla_forward_workspace_offset": (SZ, [P, I32, I32]),
        "mla_latent_attention": (I32, [P, P, P, P, I32, C.POINTER(mla_attn_desc_t), P, P, P, SZ, P]),
        "mla_latent_attention_workspace_bytes": (SZ, [P, C.POINTER(mla_attn_desc_t)]),
        "mla_check_wait_timeout": (I32, [P, C.c_uint32, P, P]),
        "mla_latent_attention_backward": (I32, [P, P, P, P, I32, C.POINTER(mla_attn_desc_t), P, P,
                                                P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib, sig


lib, SIGNATURES = _load()


def check(status: int, where: str):
    if status != MLA_OK:
        raise MLAError(status, where, lib.mla_last_error().decode())
