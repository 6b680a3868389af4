"""Planted mistakes in a copy of the oracle must fail its pins (CPU only).

Mirrors the mutation check of "extract GQA/MLA attention into reusable
layers" (Accuracy Test: scaling V or Q by 1+1e-6 and dropping the empty-row
zeroing must each fail the parity test), at fp64 tolerance, plus the other
plausible slips: rotation pairing swapped, window edge off by one, kv_b split
in the wrong order, softmax scale from qk_nope only, a dropped RMSNorm gain,
k_pe rotated with position 0, the gate ignored.  Each mutation is a text
substitution in ``oracle/mla.py`` executed as a fresh module; the real oracle
is never modified.
"""
import os
import types

import numpy as np
import pytest

from oracle import mla
from tests.oracle_cases import TinyCase, brute_cases, rel_err, tiny_dims

SRC = open(os.path.join(os.path.dirname(mla.__file__), "mla.py")).read()

MUTATIONS = {
    "scale_v": [("k_nope, v = kvb[..., :dn], kvb[..., dn:]",
                 "k_nope, v = kvb[..., :dn], kvb[..., dn:] * (1 + 1e-6)")],
    "scale_q": [("q = q.reshape(x.shape[0], H, dn + dr)",
                 "q = q.reshape(x.shape[0], H, dn + dr) * (1 + 1e-6)")],
    "drop_zeroing": [("o[:, ~vis.any(axis=1), :] = 0.0", "pass")],
    "swap_rope_style": [("ia, ib = slice(0, half), slice(half, rd)", "ia, ib = slice(0, rd, 2), slice(1, rd, 2)  # X"),
                        ("ia, ib = slice(0, rd, 2), slice(1, rd, 2)\n", "ia, ib = slice(0, half), slice(half, rd)\n")],
    "window_plus_one": [("((p - j) < int(window))", "((p - j) <= int(window))")],
    "window_minus_one": [("((p - j) < int(window))", "((p - j) < int(window) - 1)")],
    "kv_b_split_v_first": [("k_nope, v = kvb[..., :dn], kvb[..., dn:]",
                            "v, k_nope = kvb[..., :dv], kvb[..., dv:]")],
    "scale_nope_only": [("return 1.0 / np.sqrt(d.qk_nope_head_dim + d.qk_rope_head_dim)",
                         "return 1.0 / np.sqrt(d.qk_nope_head_dim)")],
    "drop_kv_gamma": [('c = rms_norm(kv[:, :d.kv_lora_rank], w["kv_a_layernorm"], d.rms_norm_eps)',
                       'c = rms_norm(kv[:, :d.kv_lora_rank], 1.0, d.rms_norm_eps)')],
    "k_pe_position_zero": [("k_pe = apply_rope(kv[:, d.kv_lora_rank:], positions,",
                            "k_pe = apply_rope(kv[:, d.kv_lora_rank:], np.zeros(len(positions)),")],
    "gate_ignored": [("if d.use_output_gate:", "if False:")],
}


def mutated_oracle(name):
    src = SRC
    for old, new in MUTATIONS[name]:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    mod = types.ModuleType("oracle_mutant_" + name)
    exec(compile(src, mod.__name__, "exec"), mod.__dict__)
    return mod


def pin_failures(m):
    """Run the brute-force and masked-row pins against oracle module ``m``."""
    fails = []
    for i, case in enumerate(brute_cases() + [TinyCase(tiny_dims(gate=True), seed=21, masked=(1,))]):
        try:
            ent_o, out_o = case.oracle_out(m)
        except Exception as e:                      # a mutation may break shapes
            fails.append((i, repr(e)))
            continue
        ent_b, out_b = case.brute_out()
        if rel_err(ent_o, ent_b) >= 1e-13 or rel_err(out_o, out_b) >= 1e-12:
            fails.append(i)
    return fails


def test_unmutated_copy_passes_the_pins():
    m = types.ModuleType("oracle_copy")
    exec(compile(SRC, "oracle_copy", "exec"), m.__dict__)
    assert pin_failures(m) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name):
    assert pin_failures(mutated_oracle(name)), f"mutation {name} passed every pin"
