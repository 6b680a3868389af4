"""Pins of the fp64 oracle against things other than itself (CPU only).

* closed forms of RMSNorm and of the rotation (both pairings);
* the independent scalar brute force (``oracle.brute``) on tiny cases;
* invariants the method fixes: absorbed == expanded, NeoX == interleaved
  under the matching permutation, q_lora_rank=None kv branch, one visible
  key, equal scores, fully masked rows, window covering every key == full,
  cached two-block decode == one-shot forward;
* the cache geometry the MLA blog prints (tests/golden/mla_cache_geometry.json).

Parity of three parts rests on a reading of the pages, not on the pages: the
sliding-window edge (``p - j < window``), the interleaved output layout (pairs
rotated in place) and the gate (``o * sigmoid(x @ gate_proj.T)`` before
o_proj).  Their pins below fix the reading's consequences (window >= kv_len is
full; window 1 keeps only keys at or after the query; a zero gate weight
halves the output), not the reading itself.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import mla
from tests.oracle_cases import TinyCase, brute_cases, rel_err, tiny_dims

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------
def test_rmsnorm_closed_form():
    y = np.array([[3.0, 4.0]])
    out = mla.rms_norm(y, np.array([1.0, 2.0]), 0.0)
    np.testing.assert_allclose(out, [[3 / math.sqrt(12.5), 8 / math.sqrt(12.5)]], rtol=1e-15)
    out_eps = mla.rms_norm(y, np.ones(2), 0.5)
    np.testing.assert_allclose(out_eps, y / math.sqrt(13.0), rtol=1e-15)


def test_rmsnorm_scale_invariance():
    rng = np.random.default_rng(0)
    y, g = rng.standard_normal((3, 64)), 1 + 0.02 * rng.standard_normal(64)
    np.testing.assert_allclose(mla.rms_norm(1000 * y, g, 0.0), mla.rms_norm(y, g, 0.0), rtol=1e-13)


@pytest.mark.parametrize("style", ["neox", "interleaved"])
def test_rope_position_zero_is_identity(style):
    x = np.random.default_rng(1).standard_normal((5, 3, 8))
    np.testing.assert_array_equal(mla.apply_rope(x, np.zeros(5), 1e4, style), x)


@pytest.mark.parametrize("style", ["neox", "interleaved"])
@pytest.mark.parametrize("k", [0, 1, 3])
def test_rope_unit_vector_closed_form(style, k):
    """e_a of pair k at position p -> (cos, sin) of p * theta^(-2k/d) in (a, b)."""
    d, theta, p = 8, 10000.0, 7
    a, b = (k, k + d // 2) if style == "neox" else (2 * k, 2 * k + 1)
    ang = p * theta ** (-2.0 * k / d)
    x = np.zeros((1, d)); x[0, a] = 1.0
    want = np.zeros(d); want[a], want[b] = math.cos(ang), math.sin(ang)
    np.testing.assert_allclose(mla.apply_rope(x, [p], theta, style)[0], want, atol=1e-15)
    x = np.zeros((1, d)); x[0, b] = 1.0
    want = np.zeros(d); want[a], want[b] = -math.sin(ang), math.cos(ang)
    np.testing.assert_allclose(mla.apply_rope(x, [p], theta, style)[0], want, atol=1e-15)


@pytest.mark.parametrize("style", ["neox", "interleaved"])
def test_rope_norm_and_relative_position(style):
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal((1, 16)), rng.standard_normal((1, 16))
    r = lambda v, p: mla.apply_rope(v, [p], 1e4, style)[0]
    np.testing.assert_allclose(np.linalg.norm(r(q, 123)), np.linalg.norm(q), rtol=1e-13)
    base = r(q, 40) @ r(k, 17)
    for delta in (1, 50, 1000):
        np.testing.assert_allclose(r(q, 40 + delta) @ r(k, 17 + delta), base, rtol=1e-10, atol=1e-12)


def test_cache_geometry_golden():
    g = json.load(open(os.path.join(GOLDEN, "mla_cache_geometry.json")))
    d = tiny_dims().replace(kv_lora_rank=g["kv_lora_rank"], qk_rope_head_dim=g["qk_rope_head_dim"],
                            qk_nope_head_dim=g["qk_nope_head_dim"])
    assert d.cache_dim == g["cache_entry_dim"] and d.qk_head_dim == g["q_head_dim"]
    rng = np.random.default_rng(3)
    w = {"kv_a_proj_with_mqa": rng.standard_normal((d.cache_dim, 16)),
         "kv_a_layernorm": np.ones(d.kv_lora_rank)}
    ent = mla.latent_cache_entries(d.replace(q_lora_rank=0), w, rng.standard_normal((2, 16)), [0, 1])
    assert ent.shape == (2, g["cache_entry_dim"])


# --------------------------------------------------------------------------
# Brute force and invariants
# --------------------------------------------------------------------------
@pytest.mark.parametrize("i", range(5))
def test_oracle_matches_brute_force(i):
    case = brute_cases()[i]
    ent_o, out_o = case.oracle_out(mla)
    ent_b, out_b = case.brute_out()
    assert rel_err(ent_o, ent_b) < 1e-13
    assert rel_err(out_o, out_b) < 1e-12


@pytest.mark.parametrize("style", ["neox", "interleaved"])
@pytest.mark.parametrize("window", [0, 3])
def test_absorbed_equals_expanded(style, window):
    case = TinyCase(tiny_dims(q_lora=6, style=style, dn=4, dv=6), seed=7, window=window, masked=(2,))
    d, w = case.d, case.w
    ent = mla.latent_cache_entries(d, w, np.concatenate([case.ctx, case.x]), np.arange(case.kv_len))
    q = mla.project_queries(d, w, case.x, case.pos)
    vis = mla.visibility(case.pos, case.kv_len, window, case.qvis, case.kv_len)
    o_exp = mla.attend(d, q, [mla.expand_keys(d, w, ent)], vis)
    o_abs = mla.attend_absorbed(d, w, q, ent, vis)
    assert rel_err(o_abs, o_exp) < 1e-12


def _perm_rope_rows(W, base, d_r):
    """Reorder rope rows so NeoX slot k takes interleaved slot 2k and slot
    k + d_r/2 takes 2k + 1."""
    W = np.array(W, dtype=np.float64)
    perm = np.concatenate([np.arange(0, d_r, 2), np.arange(1, d_r, 2)])
    W[base:base + d_r] = W[base + perm]
    return W


@pytest.mark.parametrize("q_lora", [6, 0])
def test_interleaved_equals_neox_under_permutation(q_lora):
    case = TinyCase(tiny_dims(q_lora=q_lora, style="interleaved"), seed=8, window=4)
    d, w = case.d, dict(case.w)
    _, out_int = case.oracle_out(mla)
    H, dqk, dn, dr, r = d.num_heads, d.qk_head_dim, d.qk_nope_head_dim, d.qk_rope_head_dim, d.kv_lora_rank
    wn = dict(w)
    qname = "q_b_proj" if q_lora else "q_proj"
    Wq = w[qname]
    for h in range(H):
        Wq = _perm_rope_rows(Wq, h * dqk + dn, dr)
    wn[qname] = Wq
    if q_lora:
        wn["fused_qkv_a_proj"] = _perm_rope_rows(w["fused_qkv_a_proj"], q_lora + r, dr)
    else:
        wn["kv_a_proj_with_mqa"] = _perm_rope_rows(w["kv_a_proj_with_mqa"], r, dr)
    case.d, case.w = d.replace(rope_style="neox"), wn
    _, out_neox = case.oracle_out(mla)
    assert rel_err(out_neox, out_int) < 1e-12


def test_q_lora_none_kv_branch_equals_fused_rows():
    case = TinyCase(tiny_dims(q_lora=6), seed=9)
    d, w = case.d, case.w
    hid = np.concatenate([case.ctx, case.x])
    d0 = d.replace(q_lora_rank=0)
    w0 = {"kv_a_proj_with_mqa": np.array(w["fused_qkv_a_proj"][d.q_lora_rank:]),
          "kv_a_layernorm": w["kv_a_layernorm"]}
    a = mla.latent_cache_entries(d, w, hid, np.arange(len(hid)))
    b = mla.latent_cache_entries(d0, w0, hid, np.arange(len(hid)))
    assert rel_err(a, b) < 1e-15


def test_one_visible_key_gives_its_value():
    case = TinyCase(tiny_dims(), seed=10)
    d, w = case.d, case.w
    ent = mla.latent_cache_entries(d, w, np.concatenate([case.ctx, case.x]), np.arange(case.kv_len))
    K, V = mla.expand_keys(d, w, ent)
    q = mla.project_queries(d, w, case.x, case.pos)
    vis = np.zeros((case.T, case.kv_len), dtype=bool)
    keys = [0, 3, 8, 5]
    for t, j in enumerate(keys):
        vis[t, j] = True
    o = mla.attend(d, q, [(K, V)], vis)
    for t, j in enumerate(keys):
        np.testing.assert_array_equal(o[t], V[:, j, :])


def test_equal_scores_give_mean_of_visible_values():
    case = TinyCase(tiny_dims(), seed=11)
    d, w = case.d, case.w
    ent = mla.latent_cache_entries(d, w, np.concatenate([case.ctx, case.x]), np.arange(case.kv_len))
    K, V = mla.expand_keys(d, w, ent)
    q = np.zeros((case.T, d.num_heads, d.qk_head_dim))
    vis = mla.visibility(case.pos, case.kv_len, 3, np.ones(case.T), case.kv_len)
    o = mla.attend(d, q, [(K, V)], vis)
    for t in range(case.T):
        np.testing.assert_allclose(o[t], V[:, vis[t], :].mean(axis=1), rtol=1e-14)


def test_fully_masked_rows_are_exact_zero():
    case = TinyCase(tiny_dims(gate=True), seed=12, masked=(0, 2))
    _, out = case.oracle_out(mla)
    assert np.all(out[[0, 2]] == 0.0) and not np.signbit(out[[0, 2]]).any()
    assert np.all(np.abs(out[[1, 3]]) > 0)


def test_window_covering_all_keys_equals_full_mask():
    full = TinyCase(tiny_dims(style="interleaved"), seed=13, window=0)
    wide = TinyCase(tiny_dims(style="interleaved"), seed=13, window=full.kv_len)
    np.testing.assert_array_equal(full.oracle_out(mla)[1], wide.oracle_out(mla)[1])


def test_window_one_keeps_keys_at_or_after_the_query():
    vis = mla.visibility(np.arange(5, 9), 9, 1, np.ones(4), 9)
    for t, p in enumerate(range(5, 9)):
        assert list(np.nonzero(vis[t])[0]) == list(range(p, 9))


def test_gate_zero_weight_halves_output():
    """sigmoid(0) = 1/2 multiplies o before the linear o_proj: out halves."""
    case = TinyCase(tiny_dims(gate=True), seed=14)
    case.w = dict(case.w, gate_proj=np.zeros_like(case.w["gate_proj"]))
    gated = case.oracle_out(mla)[1]
    case.d = case.d.replace(use_output_gate=False)
    np.testing.assert_allclose(gated, 0.5 * case.oracle_out(mla)[1], rtol=1e-14)


def test_cached_two_block_decode_equals_one_shot():
    """Block 2 through the cache (context + block-1 latents + its own) ==
    a one-shot forward of [block1; block2] under a block-causal mask, and ==
    a fresh forward of block 2 whose context is prefix + block 1 recomputed
    from hidden states (PR #1026: cached block decoding, two consecutive
    blocks on a cache)."""
    d = tiny_dims(q_lora=6, style="interleaved")
    rng = np.random.Generator(np.random.PCG64(15))
    from head_latent_attention_qkv_gb300.workloads import make_weights
    w = make_weights(d, rng)
    C, T = 6, 3
    ctx, x1, x2 = (rng.standard_normal((n, d.hidden_size)) for n in (C, T, T))
    e_ctx = mla.latent_cache_entries(d, w, ctx, np.arange(C))
    e1 = mla.latent_cache_entries(d, w, x1, np.arange(C, C + T))
    e2 = mla.latent_cache_entries(d, w, x2, np.arange(C + T, C + 2 * T))
    cache = np.concatenate([e_ctx, e1, e2])
    p2 = np.arange(C + T, C + 2 * T)
    J = C + 2 * T
    vis2 = mla.visibility(p2, J, 0, np.ones(T), J)
    out_cached = mla.block_forward(d, w, x2, p2, [mla.expand_keys(d, w, cache)], vis2)
    fresh = mla.latent_cache_entries(d, w, np.concatenate([ctx, x1, x2]), np.arange(J))
    out_fresh = mla.block_forward(d, w, x2, p2, [mla.expand_keys(d, w, fresh)], vis2)
    assert rel_err(out_fresh, out_cached) < 1e-13
    xs = np.concatenate([x1, x2])
    ps = np.arange(C, C + 2 * T)
    vis = np.concatenate([mla.visibility(ps[:T], C + T, 0, np.ones(T), J),
                          mla.visibility(ps[T:], J, 0, np.ones(T), J)])
    out_one = mla.block_forward(d, w, xs, ps, [mla.expand_keys(d, w, cache)], vis)
    assert rel_err(out_one[T:], out_cached) < 1e-13
    vis1 = mla.visibility(ps[:T], C + T, 0, np.ones(T), C + T)
    out1 = mla.block_forward(d, w, x1, ps[:T], [mla.expand_keys(d, w, cache[:C + T])], vis1)
    assert rel_err(out_one[:T], out1) < 1e-13


def test_typed_storage_rounds_to_nearest_bf16_ties_to_even():
    """bf16 keeps 8 significant bits: 1 + 2^-8 is a tie between 1 and
    1 + 2^-7 (goes to the even 1), 1 + 3*2^-8 is a tie between 1 + 2^-7 and
    1 + 2^-6 (goes to the even 1 + 2^-6); representable values stay."""
    from head_latent_attention_qkv_gb300.workloads import QWEN3_4B_MLA, TINY_FP32_MLA
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1.5, 3.0 + 2 ** -7, 1 + 2 ** -9])
    want = np.array([1.0, 1 + 2 ** -6, -1.0, 1.5, 3.0, 1.0])
    np.testing.assert_array_equal(mla.round_to_dtype(QWEN3_4B_MLA, x), want)
    np.testing.assert_array_equal(mla.round_to_dtype(TINY_FP32_MLA, x), x)
