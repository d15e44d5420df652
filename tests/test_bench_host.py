"""Host logic of bench.py that needs no GPU: the attention flop count, the
tensor-peak fallback, and the oracle CPU baseline on one thread and on every
host core (spawned processes)."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


@pytest.mark.parametrize("seq", [1, 2, 7, 64])
@pytest.mark.parametrize("causal", [True, False])
def test_attention_flops_count_visible_pairs(seq, causal):
    pairs = sum(1 for i in range(seq) for j in range(seq) if j <= i or not causal)
    assert bench.attn_flops(3, seq, 16, causal) == 4.0 * 3 * 16 * pairs


def test_tensor_peak_falls_back_without_measurements():
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        pytest.skip("measured peaks present")
    assert bench.bf16_peak() == (bench.FALLBACK_BF16_TFLOPS, "fallback")


def test_cpu_baseline_one_thread_and_all_cores():
    r = bench.cpu_baseline(1.0)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s"
    assert r["value_1_thread"] > 0 and r["value"] >= r["value_1_thread"]
    n = len(os.sched_getaffinity(0))
    assert r["cores"] in (1, n)
    if r["cores"] == n and n > 1:
        assert f"{n} processes" in r["sample"]
