"""bench.py's roofline arithmetic, on the CPU: the algorithmic bytes and FLOPs
it divides by are the per-unit figures of the measurement plan (1,540 bytes per
bf16 token-head at D = 128 plus the fp32 states and checkpoints; 132,612 bytes
and 7 D^2 FLOPs per decode head-step)."""
import importlib.util
import os

import pytest

from linear_attention_serving_k1_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_prefill_bytes_workload2(bench):
    w = workloads.workload(2)
    # 8192 tokens x 32 heads x 1540 B, plus the initial and final state (32 x 64 KiB each)
    assert bench.prefill_algorithmic_bytes(w) == 8192 * 32 * 1540 + 2 * 32 * 128 * 128 * 4 == 407_896_064


def test_prefill_bytes_workload4_counts_checkpoints(bench):
    w = workloads.workload(4)
    n_ck = 131072 // w.ckpt_stride
    assert n_ck == 4
    assert bench.prefill_algorithmic_bytes(w) == 131072 * 32 * 1540 + (2 + n_ck) * 32 * 128 * 128 * 4


def test_prefill_flops_per_token_head(bench):
    w = workloads.workload(2)
    assert bench.prefill_flops(w) == int(8192 * 32 * (5 * 64 * 128 + 6 * 128 * 128 + 64 * 64 / 3))
    assert bench.prefill_flops(w) // (8192 * 32) == 140_629


def test_decode_cost_per_head(bench):
    flops, nbytes = bench.decode_cost_per_head(128)
    assert flops == 7 * 128 * 128
    assert nbytes == 132_612
