"""GPU parity with each kernel tier forced through RR_FORCE_TIER, against the
float64 oracle: spans of short rows (T0), a row in registers (T1: engine direct
variants, LayerNorm / RMSNorm row groups), staged rows one per CTA (T2) and
cluster-split rows (T3), each on the shapes it can hold, so every tier is
checked on short, medium and long rows and not only where the planner would
pick it.  Where the forced tier cannot hold a shape the call must fail with
RR_ERR_INVALID_ARG; `holds` states those rules."""
import contextlib
import os

import numpy as np
import pytest
import torch

import oracle
import row_reduction_pass_gb300 as rr
from row_reduction_pass_gb300 import synth

from parity import (TOL, TOL_F32_OUT, check_guards, check_log_softmax, check_norm_bwd,
                    check_softmax, check_softmax_bwd, check_xent, compare, empty_like_dev, host,
                    out_f32, store, to_dev)

pytestmark = pytest.mark.gpu

COLS = [1, 31, 97, 1000, 4097]
ROWS = {1: 2000, 31: 700, 97: 400, 1000: 120, 4097: 40}


@contextlib.contextmanager
def tier(t):
    old = os.environ.get("RR_FORCE_TIER")
    os.environ["RR_FORCE_TIER"] = str(t)
    try:
        yield
    finally:
        if old is None:
            del os.environ["RR_FORCE_TIER"]
        else:
            os.environ["RR_FORCE_TIER"] = old


def holds(op: str, t: int, cols: int, e: int) -> bool:
    """Whether forced tier t takes rows of `cols` elements of e bytes (16-byte
    aligned tensors) for operation `op`."""
    if t == 0:  # rows of a byte length not a multiple of 16, with a limit per operation
        rb = cols * e
        if rb % 16 == 0:
            return False
        if op in ("softmax", "log_softmax"):
            return rb <= 448 and cols <= 160
        if op == "xent":
            return rb <= 448 and cols <= 200
        if op in ("softmax_bwd", "log_softmax_bwd"):
            return rb <= 224
        if op in ("ln_fwd", "rms_fwd"):
            return rb <= 448 and (e == 4 or cols <= 128)
        return rb <= (96 if e == 2 else 64)  # norm backward
    if t == 1:
        return True  # every row length used here fits one row group
    if t == 2:
        return not op.startswith("rms")  # no staged RMSNorm kernel
    # t == 3: a split into K >= 2 slices of whole 16-byte chunks needs a second
    # slice with columns in it
    v = 16 // e
    half = -(-cols // 2)
    return (-(-half // v) * v) < cols


def expect(op, t, cols, dtype, fn):
    e = 2 if dtype == "bf16" else 4
    with tier(t):
        if holds(op, t, cols, e):
            fn()
        else:
            with pytest.raises(rr.RRError, match="INVALID_ARG"):
                fn()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("t", [0, 1, 2, 3])
def test_softmax_family_tiers(t, cols, dtype):
    x, lab = synth.xent_inputs(ROWS[cols], cols, dtype, 3.0, 4000 + cols, ignore_frac=0.05,
                               outlier_frac=0.01, masked_row_every=37)
    expect("softmax", t, cols, dtype, lambda: check_softmax(x, dtype))
    expect("log_softmax", t, cols, dtype, lambda: check_log_softmax(x, dtype))
    expect("xent", t, cols, dtype, lambda: check_xent(x, lab, dtype))
    # backward of the oracle's softmax output with a second input dy
    rng = np.random.default_rng(cols)
    y = store(oracle.softmax(x), dtype)
    dy = store(rng.standard_normal(x.shape), dtype)
    expect("softmax_bwd", t, cols, dtype, lambda: check_softmax_bwd(y, dy, dtype))


def norm_fwd_only(x, g, b, dtype, rms):
    rows = x.shape[0]
    xd, gd = to_dev(x), to_dev(g)
    y = empty_like_dev(x.shape, dtype)
    rstd = out_f32(rows)
    rtol, atol = TOL[dtype]
    if rms:
        rr.rr_rmsnorm_fwd(xd, gd, y, rstd, eps=1e-5)
        torch.cuda.synchronize()
        check_guards()
        ry, rrstd = oracle.rms_fwd(x, g, 1e-5)
    else:
        mean = out_f32(rows)
        rr.rr_layernorm_fwd(xd, gd, to_dev(b), y, mean, rstd, eps=1e-5)
        torch.cuda.synchronize()
        check_guards()
        ry, rmean, rrstd = oracle.ln_fwd(x, g, b, 1e-5)
        compare("ln mean", host(mean), rmean, *TOL_F32_OUT)
    compare("norm y", host(y), ry, rtol, atol)
    compare("norm rstd", host(rstd), rrstd, *TOL_F32_OUT)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cols", COLS)
@pytest.mark.parametrize("t", [0, 1, 2, 3])
def test_norm_tiers(t, cols, dtype):
    x, g, b, dy = synth.ln_inputs(ROWS[cols], cols, dtype, 5000 + cols, row_offset=10.0,
                                  gamma_std=0.1, beta_std=0.1, outlier_frac=0.005,
                                  masked_row_every=41)
    expect("ln_fwd", t, cols, dtype, lambda: norm_fwd_only(x, g, b, dtype, False))
    expect("ln_bwd", t, cols, dtype, lambda: check_norm_bwd(x, g, b, dy, dtype))
    expect("rms_fwd", t, cols, dtype, lambda: norm_fwd_only(x, g, b, dtype, True))
    expect("rms_bwd", t, cols, dtype, lambda: check_norm_bwd(x, g, b, dy, dtype, rms=True))


def test_bad_tier_value_is_rejected():
    x = torch.zeros(4, 8, device="cuda")
    with tier("7"):
        with pytest.raises(rr.RRError, match="INVALID_ARG"):
            rr.rr_softmax_fwd(x, torch.empty_like(x))
