"""GPU parity for rows of one column, which every operation runs on its
elementwise kernels (a one-element row is its own maximum, sum and moments):
softmax, log-softmax, cross-entropy, the softmax / log-softmax backward and the
LayerNorm / RMSNorm forward and backward, against the float64 oracle through
the C ABI.  Row counts from one row to several grid-stride passes over all
resident blocks (three million rows), a ragged last tile, misaligned and
in-place tensors, special values (NaN, +-inf, -0, +-1e8, subnormals),
ignored rows and labels out of range; the norm backward's per-block partials
through both the workspace and the no-allocation entry points."""
import numpy as np
import pytest
import torch

import oracle
import row_reduction_pass_gb300 as rr
from row_reduction_pass_gb300 import synth

from parity import (TOL, check_guards, check_ln, check_log_softmax, check_norm_bwd, check_rms,
                    check_softmax, check_softmax_bwd, check_xent, compare, empty_like_dev, host,
                    store, to_dev)

pytestmark = pytest.mark.gpu

ROWS = [1, 255, 1025, 4097, 3_000_017]


def logits(rows, dtype, seed):
    x, lab = synth.xent_inputs(rows, 1, dtype, 3.0, seed, ignore_frac=0.05, outlier_frac=0.01,
                               masked_row_every=37)
    lab[1::50] = 4                  # out of range -> NaN loss, counted
    lab[2::97] = -7                 # negative, not the ignore index
    return x, lab


def upstream(rows, dtype, seed):
    return store(np.random.default_rng(seed).standard_normal((rows, 1)), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows", ROWS)
def test_softmax_family_one_column(rows, dtype):
    x, lab = logits(rows, dtype, 11 + rows)
    check_softmax(x, dtype)
    check_log_softmax(x, dtype)
    check_xent(x, lab, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows", ROWS)
def test_softmax_bwd_one_column(rows, dtype):
    x, _ = logits(rows, dtype, 21 + rows)
    dy = upstream(rows, dtype, 22 + rows)
    check_softmax_bwd(store(oracle.softmax(x), dtype), dy, dtype)
    check_softmax_bwd(store(oracle.log_softmax(x), dtype), dy, dtype, log=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows", ROWS)
def test_norms_one_column(rows, dtype):
    x, g, b, dy = synth.ln_inputs(rows, 1, dtype, 31 + rows, row_offset=10.0, gamma_std=0.1,
                                  beta_std=0.1, outlier_frac=0.005, masked_row_every=41)
    check_ln(x, g, b, dy, 1e-5, dtype)
    check_ln(x, g, b, dy, 1e-5, dtype, oracle_stats=False)
    check_rms(x, g, dy, 1e-5, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_column_layouts(dtype):
    """Misaligned bases (one element past a 16-byte boundary), in-place
    outputs, statistics off a 16-byte boundary, dx written over an input."""
    rows = 100_003
    x, lab = logits(rows, dtype, 41)
    check_softmax(x, dtype, pad_in=1, pad_out=3)
    check_softmax(x, dtype, pad_in=1, inplace=True)
    check_log_softmax(x, dtype, pad_in=2, inplace=True)
    check_xent(x, lab, dtype, pad_in=3, inplace=True)
    check_xent(x, lab, dtype, pad_in=0, pad_out=1)
    dy = upstream(rows, dtype, 42)
    y = store(oracle.softmax(x), dtype)
    check_softmax_bwd(y, dy, dtype, pads=(1, 2, 3))
    check_softmax_bwd(y, dy, dtype, inplace="dy")
    check_softmax_bwd(store(oracle.log_softmax(x), dtype), dy, dtype, log=True, inplace="y")
    xl, g, b, dyl = synth.ln_inputs(rows, 1, dtype, 43, row_offset=10.0, masked_row_every=41)
    check_ln(xl, g, b, dyl, 1e-5, dtype, pad=(1, 1, 1, 1, 1))
    check_rms(xl, g, dyl, 1e-5, dtype, pad=(3, 1, 1, 2, 1))
    for inplace in ("dy", "x"):
        check_norm_bwd(xl, g, b, dyl, dtype, stat_pad=1, inplace=inplace)
        check_norm_bwd(xl, g, b, dyl, dtype, rms=True, stat_pad=3, inplace=inplace)


# Special values, each at several rows (the kernels take rows in tiles of
# 256 x U, so the positions fall in different lanes and tiles).
# (Logits stay below 2^30 in magnitude, the softmax family's range: beyond it
# the rounding residual of m log2 e can exceed the float32 exponent range.)
_SPECIAL = [np.nan, np.inf, -np.inf, -0.0, 0.0, 1e8, -1e8, 1e-40, -1e-40, 88.0, -104.0]


def _special_column(rows, dtype, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, 1)) * 3.0
    for i, v in enumerate(_SPECIAL):
        x[i::len(_SPECIAL) * 7, 0] = v
    return store(x, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_column_special_values(dtype):
    rows = 70_001
    x = _special_column(rows, dtype, 51)
    lab = np.zeros(rows, np.int32)
    lab[3::5] = -100                # ignored, also on NaN / inf rows
    lab[4::13] = 1                  # out of range, also on masked rows
    lab[6::17] = -2
    check_softmax(x, dtype)
    check_log_softmax(x, dtype)
    check_xent(x, lab, dtype)
    dy = upstream(rows, dtype, 52)
    check_softmax_bwd(store(oracle.softmax(x), dtype), dy, dtype)
    check_softmax_bwd(store(oracle.log_softmax(x), dtype), dy, dtype, log=True)
    g = store(np.array([1.5]), dtype)
    b = store(np.array([-0.25]), dtype)
    xn = _special_column(rows, dtype, 53)
    check_ln(xn, g, b, dy, 1e-5, dtype)
    check_rms(xn, g, dy, 1e-5, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_column_noalloc(dtype):
    """The no-allocation LayerNorm backward at one column, three million rows:
    the per-block partials fit its scratch; two calls in a row agree with the
    oracle."""
    rows = 3_000_017
    x, g, b, dy = synth.ln_inputs(rows, 1, dtype, 61, row_offset=10.0, masked_row_every=97)
    _, m64, r64 = oracle.ln_fwd(x, g, b, 1e-5, want_y=False)
    mean, rstd = to_dev(m64.astype(np.float32)), to_dev(r64.astype(np.float32))
    xd, gd, dyd = to_dev(x), to_dev(g), to_dev(dy)
    odx, odg, odb, sdg, sdb = oracle.ln_bwd(dy, x, host(mean), host(rstd), g)
    rtol, atol = TOL[dtype]
    for _ in range(2):
        dx = empty_like_dev(x.shape, dtype)
        dg, db = empty_like_dev(g.shape, dtype), empty_like_dev(g.shape, dtype)
        rr.rr_layernorm_bwd_noalloc(dyd, xd, mean, rstd, gd, dx, dg, db)
        torch.cuda.synchronize()
        check_guards()
        compare("noalloc dx", host(dx), odx, rtol, atol)
        compare("noalloc dgamma", host(dg), odg, rtol, atol, scale=sdg)
        compare("noalloc dbeta", host(db), odb, rtol, atol, scale=sdb)
