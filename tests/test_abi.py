"""Host-side checks of the C ABI (no GPU work is launched).

The library must load, export every function ``include/mla_draft.h``
declares, answer the geometry queries with the figures the MLA blog prints
(tests/golden/mla_cache_geometry.json) and reject invalid arguments with the
documented status before touching the device.
"""
import ctypes as C
import json
import os
import re

import pytest

from head_latent_attention_qkv_gb300 import _lib, api
from head_latent_attention_qkv_gb300.workloads import DEEPSEEK_V3_MLA, QWEN3_4B_MLA, TINY_FP32_MLA

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
lib = _lib.lib


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src))
    return names


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert {"mla_draft_init", "mla_latent_cache_append", "mla_draft_forward"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature"


def test_cache_geometry_matches_golden():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "mla_cache_geometry.json")))
    for case in g["cases"]:
        dims = DEEPSEEK_V3_MLA.replace(dtype="bf16" if case["dtype_size"] == 2 else "fp32")
        cfg = api.make_config(dims, case["block_size"])
        assert lib.mla_cache_entry_dim(C.byref(cfg)) == g["cache_entry_dim"]
        assert lib.mla_cache_page_bytes(C.byref(cfg)) == case["mla_page_bytes"]
        # an MLA page is half a full-attention page with one KV head (no K and V copies)
        assert 2 * lib.mla_cache_page_bytes(C.byref(cfg)) == case["full_attention_page_bytes"]


@pytest.mark.parametrize("dims", [TINY_FP32_MLA, QWEN3_4B_MLA, DEEPSEEK_V3_MLA])
def test_arena_bytes_positive_for_valid_configs(dims):
    cfg = api.make_config(dims, 64)
    n = lib.mla_weight_arena_bytes(C.byref(cfg))
    assert n > 0 and n % 256 == 0


@pytest.mark.parametrize("field,value", [("hidden_size", 0), ("num_heads", -1), ("qk_rope_head_dim", 7),
                                         ("page_size", 0), ("dtype", 5), ("rope", 9),
                                         ("q_lora_rank", -3), ("max_position", 0)])
def test_invalid_config_is_rejected(field, value):
    cfg = api.make_config(QWEN3_4B_MLA, 64)
    setattr(cfg, field, value)
    assert lib.mla_weight_arena_bytes(C.byref(cfg)) == 0
    assert lib.mla_cache_entry_dim(C.byref(cfg)) == 0
    w = _lib.mla_weights_t()
    h = C.c_void_p()
    st = lib.mla_draft_init(C.byref(cfg), C.byref(w), C.c_void_p(256), 1 << 40, None, C.byref(h))
    assert st == _lib.MLA_ERR_INVALID_ARG and not h.value
    assert lib.mla_last_error()


@pytest.mark.parametrize("field,value", [("kv_lora_rank", 256), ("qk_rope_head_dim", 32),
                                         ("page_size", 48), ("page_size", 192), ("hidden_size", 2600)])
def test_bf16_shapes_without_a_kernel_are_unsupported_at_init(field, value):
    cfg = api.make_config(QWEN3_4B_MLA, 64)
    setattr(cfg, field, value)
    w = _lib.mla_weights_t(**{k: 256 for k in _lib.WEIGHT_FIELDS})   # non-NULL, never read
    h = C.c_void_p()
    st = lib.mla_draft_init(C.byref(cfg), C.byref(w), C.c_void_p(256), 1 << 40, None, C.byref(h))
    assert st == _lib.MLA_ERR_UNSUPPORTED and not h.value, lib.mla_last_error()


def test_missing_weights_are_rejected_before_any_device_work():
    cfg = api.make_config(QWEN3_4B_MLA, 64)
    w = _lib.mla_weights_t()          # every pointer NULL
    h = C.c_void_p()
    st = lib.mla_draft_init(C.byref(cfg), C.byref(w), C.c_void_p(256), 1 << 40, None, C.byref(h))
    assert st == _lib.MLA_ERR_INVALID_ARG
    assert b"fused_qkv_a_proj" in lib.mla_last_error()


def test_null_handle_calls_return_invalid_arg():
    assert lib.mla_latent_cache_append(None, None, None, None, 4, None, 1, None, 0, None) == _lib.MLA_ERR_INVALID_ARG
    desc = _lib.mla_attn_desc_t(num_blocks=1, block_len=16, max_pages=1)
    assert lib.mla_draft_forward(None, None, None, None, None, 1, C.byref(desc), None, None, 0, None) \
        == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_draft_forward_after(None, None, None, None, None, 1, C.byref(desc), None, None, 0,
                                       None, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_get_device_status(None, None, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_append_workspace_bytes(None, 4) == 0
    ctx = _lib.mla_shared_ctx_t(num_ctx=1, ctx_rows=64)
    assert lib.mla_draft_forward_shared(None, None, None, None, None, 1, C.byref(desc), C.byref(ctx),
                                        None, None, 0, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_draft_forward_shared_after(None, None, None, None, None, 1, C.byref(desc),
                                              C.byref(ctx), None, None, 0, None, None) \
        == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_shared_attention(None, None, C.byref(desc), C.byref(ctx), None, 0, None) \
        == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_forward_shared_workspace_bytes(None, 16, 64) == 0
    lib.mla_draft_destroy(None)


def test_python_binding_has_the_c_names():
    # every entry point the header declares that a Python caller uses directly
    for n in declared_functions() - {"mla_draft_destroy", "mla_status_string", "mla_last_error",
                                      "mla_append_workspace_bytes", "mla_forward_workspace_bytes",
                                      "mla_forward_shared_workspace_bytes"}:
        assert hasattr(api, n), f"api.{n} missing"
    assert api.mla_cache_entry_dim(QWEN3_4B_MLA) == 576
    assert api.mla_cache_page_bytes(QWEN3_4B_MLA, 64) == 64 * 576 * 2
    assert api.mla_weight_arena_bytes(QWEN3_4B_MLA) > 0


def test_status_strings():
    for s in range(6):
        assert lib.mla_status_string(s)
    assert lib.mla_status_string(99) == b"unknown status"
