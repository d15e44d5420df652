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


def test_step_covers_every_workload_with_its_bytes():
    """The timed step's launch groups: config 2's LayerNorm, config 3's causal
    softmax, the sweep's bf16 LayerNorm cases at 1000, 4097 and 65537 columns
    (fwd and bwd each) and config 4's cross-entropy, with their algorithmic bytes."""
    w = bench.make_inputs(scale_rows=1 / 1024)
    nb = bench.step_bytes(w)
    want = ["ln_fwd", "softmax", "ln_bwd"]
    for c in (1000, 4097, 65537):
        want += [f"ln_bf16_c{c}_fwd", f"ln_bf16_c{c}_bwd"]
    assert list(nb) == want + ["xent"]
    for c in (1000, 4097, 65537):
        r, cc = w[f"lnb{c}"]["x"].shape
        assert cc == c and w[f"lnb{c}"]["x"].dtype.itemsize == 2
        assert nb[f"ln_bf16_c{c}_fwd"] == 2 * r * c * 2 + 2 * c * 2 + 8 * r
        assert nb[f"ln_bf16_c{c}_bwd"] == 3 * r * c * 2 + 3 * c * 2 + 8 * r
