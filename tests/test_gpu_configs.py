"""GPU parity at the full sizes of the five measured workloads, through the same
entry points (and so the same kernel variants and launch shapes) that bench.py
times:
  1. softmax cross-entropy fwd+bwd, fp32, 64 x 1000
  2. LayerNorm fwd+bwd, fp32, 4096 x 768
  3. causal attention-score softmax, bf16, 65536 x 512
  4. LM-head softmax cross-entropy fwd+bwd, bf16, 16384 x 50304, in place, 5% ignored:
     loss and dlogits compared on every row, ignored rows all zero
  5. the ragged / extreme sweep, fp32 and bf16, cols in {1, 31, 97, 1000, 4097, 65537},
     rows = floor(2^24 / cols), for softmax cross-entropy and LayerNorm fwd+bwd
"""
import collections
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from row_reduction_pass_gb300 import synth
import row_reduction_pass_gb300 as rr

from parity import (TOL, TOL_F32_OUT, check_guards, check_ln, check_softmax, check_xent, compare,
                    host, out_f32, to_dev, zeros_i32)

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
    """Every row of the full-size workload: loss and all 16384 x 50304 dlogits
    against the oracle (in slabs of rows, so the float64 reference never holds
    more than a few slabs), every ignored row all zero, guard bands intact."""
    d = synth.make("xent_bf16_16384x50304")
    logits, labels = d["logits"], d["labels"]
    ign = d["ignore_index"]
    rows, cols = logits.shape
    xd = to_dev(logits)
    lab = to_dev(labels)
    loss = out_f32(rows)
    bad = zeros_i32(1)
    rr.rr_softmax_xent_fwd_bwd(xd, lab, loss, xd, ignore_index=ign, bad_label_count=bad)
    torch.cuda.synchronize()
    check_guards()
    assert int(bad.item()) == 0
    ignored = np.nonzero(labels == ign)[0]
    assert ignored.size > 0
    assert bool((xd.index_select(0, torch.from_numpy(ignored).to(xd.device)) == 0).all())
    rtol, atol = TOL["bf16"]
    slab = 256

    def reference(s):
        e = min(rows, s + slab)
        rloss, rdl, rbad = oracle.xent(logits[s:e], labels[s:e], ign)
        return s, e, rloss, rdl, rbad

    # the C oracle releases the GIL, so slabs run on a few threads; at most
    # `workers` slabs are in flight
    workers = max(1, min(8, os.cpu_count() or 1))
    starts = list(range(0, rows, slab))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        pending = collections.deque(ex.submit(reference, s) for s in starts[:workers])
        nxt = workers
        while pending:
            s, e, rloss, rdl, rbad = pending.popleft().result()
            if nxt < len(starts):
                pending.append(ex.submit(reference, starts[nxt]))
                nxt += 1
            assert rbad == 0
            compare(f"lm-head xent loss rows {s}..{e}", host(loss[s:e]), rloss, *TOL_F32_OUT)
            compare(f"lm-head xent dlogits rows {s}..{e}", host(xd[s:e]), rdl, rtol, atol)


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
