"""GPU parity at the full sizes of the five measured workloads, through the same
entry points (and so the same kernel variants and launch shapes) that bench.py
times:
  1. softmax cross-entropy fwd+bwd, fp32, 64 x 1000
  2. LayerNorm fwd+bwd, fp32, 4096 x 768
  3. causal attention-score softmax, bf16, 65536 x 512
  4. LM-head softmax cross-entropy fwd+bwd, bf16, 16384 x 50304, in place, 5% ignored:
     loss compared on every row, dlogits on a sample of rows, ignored rows all zero
  5. the ragged / extreme sweep, fp32 and bf16, cols in {1, 31, 97, 1000, 4097, 65537},
     rows = floor(2^24 / cols), for softmax cross-entropy and LayerNorm fwd+bwd
"""
import numpy as np
import pytest
import torch

import oracle
from row_reduction_pass_gb300 import synth
import row_reduction_pass_gb300 as rr

from parity import TOL, TOL_F32_OUT, check_ln, check_softmax, check_xent, compare, host, to_dev

pytestmark = pytest.mark.gpu


def test_xent_f32_64x1000():
    d = synth.make("xent_f32_64x1000")
    check_xent(d["logits"], d["labels"], "f32")


def test_layernorm_f32_4096x768():
    d = synth.make("ln_f32_4096x768")
    check_ln(d["x"], d["gamma"], d["beta"], d["dy"], d["eps"], "f32")
    check_ln(d["x"], d["gamma"], d["beta"], d["dy"], d["eps"], "f32", oracle_stats=False)


def test_causal_softmax_bf16_65536x512():
    d = synth.make("softmax_bf16_causal_65536x512")
    check_softmax(d["x"], "bf16")


def test_lm_head_xent_bf16_16384x50304_in_place():
    d = synth.make("xent_bf16_16384x50304")
    logits, labels = d["logits"], d["labels"]
    rows, cols = logits.shape
    xd = to_dev(logits)
    lab = to_dev(labels)
    loss = torch.full((rows,), float("nan"), device=xd.device)
    bad = torch.zeros(1, dtype=torch.int32, device=xd.device)
    rr.rr_softmax_xent_fwd_bwd(xd, lab, loss, xd, ignore_index=d["ignore_index"],
                               bad_label_count=bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == 0
    rloss, _, rbad = oracle.xent(logits, labels, d["ignore_index"], want_dlogits=False)
    assert rbad == 0
    compare("lm-head xent loss (all rows)", host(loss), rloss, *TOL_F32_OUT)
    ignored = np.nonzero(labels == d["ignore_index"])[0]
    assert ignored.size > 0
    sample_ign = torch.from_numpy(ignored[:64]).to(xd.device)
    assert bool((xd.index_select(0, sample_ign) == 0).all())
    rng = np.random.default_rng(4)
    sample = np.unique(np.concatenate([[0, rows - 1], rng.choice(rows, 384, replace=False)]))
    got = host(xd.index_select(0, torch.from_numpy(sample).to(xd.device)))
    _, rdl, _ = oracle.xent(logits[sample], labels[sample], d["ignore_index"])
    rtol, atol = TOL["bf16"]
    compare("lm-head xent dlogits (sampled rows)", got, rdl, rtol, atol)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", synth.SWEEP_COLS)
def test_sweep_xent(cols, dtype):
    d = synth.make(f"sweep_xent_{dtype}_c{cols}")
    check_xent(d["logits"], d["labels"], dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", synth.SWEEP_COLS)
def test_sweep_layernorm(cols, dtype):
    d = synth.make(f"sweep_ln_{dtype}_c{cols}")
    check_ln(d["x"], d["gamma"], d["beta"], d["dy"], d["eps"], dtype)
