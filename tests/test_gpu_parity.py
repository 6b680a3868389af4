"""CUDA path vs the fp64 oracle on the same seeded inputs (needs a GB300).

Small variants of every workload run whole (ragged contexts, partial pages
and tiles, masked rows, sliding windows, two cached blocks); the full-size
workloads run in the benchmark's launch configuration and are checked on a
seeded sample of blocks the oracle computes one by one.  See tests/parity.py
for the tolerances and the exact checks.
"""
import numpy as np
import pytest

from head_latent_attention_qkv_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_small_workload_matches_oracle(name):
    from tests.parity import check_workload
    wl = workloads.make_workload(name, "small")
    check_workload(wl)


def _sample_blocks(wl, per_step, seed=0):
    rng = np.random.default_rng(seed)
    out = []
    for s in wl.steps:
        nb = len(s.kv_len)
        pick = rng.choice(nb, size=min(per_step, nb), replace=False)
        out.append(sorted(int(b) for b in pick))
    return out


FULL = [("tiny_fp32", None), ("qwen3_4b_prefill", None), ("qwen3_4b_sliding_gate", None),
        ("qwen3_4b_cached_decode", 8), ("deepseek_v3_block_parallel", 8)]


@pytest.mark.parametrize("name,per_step", FULL)
def test_full_size_workload_matches_oracle_on_sampled_blocks(name, per_step):
    from tests.parity import check_workload
    wl = workloads.make_workload(name, "full")
    sample = None if per_step is None else _sample_blocks(wl, per_step)
    if name == "deepseek_v3_block_parallel":
        # keep both mask kinds in the sample: even blocks full, odd blocks sliding
        step = wl.steps[0]
        sample = [sorted(set(sample[0]) | {0, 1, len(step.kv_len) - 1})]
    check_workload(wl, sample)
