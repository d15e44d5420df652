"""GPU parity of the phase-aligned long-row kernels (rows of at least 8 KB whose
input and output tensors share their address modulo 16) against the float64
oracle: softmax, log-softmax, softmax cross-entropy and the softmax /
log-softmax backward, and LayerNorm /
RMSNorm, on every phase-class count a row length can give (P = 1, 2, 4, 8
classes of rows by start offset), on tensors whose base is not 16-byte aligned
(every row shifted), in place, one block per row and rows split over a cluster,
and with the cross-entropy's edge cases: labels in a row's first and last
column (its shared head / tail chunk), ignored rows, labels outside the row,
fully masked rows and outliers.  Each case also runs with these kernels turned
off (RR_SMX=0 / RR_LNX=0), so the kernels they replace keep their coverage on
the same shapes, and the norms with each of their two long-row designs forced
(RR_LNP=1: rows in shared memory with pipelined merges; RR_LNP=0: rows in
registers)."""
import contextlib
import os

import numpy as np
import pytest
import torch

import oracle
from row_reduction_pass_gb300 import synth

import row_reduction_pass_gb300 as rr
from parity import (TOL, TOL_F32_OUT, check_guards, check_ln, check_log_softmax, check_norm_bwd,
                    check_rms, check_softmax, check_softmax_bwd, check_xent, compare, host,
                    out_f32, store, to_dev)

pytestmark = pytest.mark.gpu


@contextlib.contextmanager
def env(**kv):
    old = {k: os.environ.get(k) for k in kv}
    os.environ.update({k: str(v) for k, v in kv.items()})
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


def phases(cols: int, e: int) -> int:
    rb = cols * e % 16
    return 1 if rb == 0 else 16 // np.gcd(16, rb)


# (dtype, cols, rows): P = 8, 2, 4, 1 classes; one block per row; clusters of
# 2 and 3 ranks (bf16 and fp32 blocks hold up to 32768 / 24576 elements)
SMX_SHAPES = [
    ("bf16", 4097, 45), ("bf16", 4100, 21), ("bf16", 4102, 19), ("bf16", 4104, 9),
    ("bf16", 40001, 7), ("bf16", 65537, 5),
    ("f32", 2049, 33), ("f32", 2050, 17), ("f32", 2052, 6), ("f32", 2051, 1),
    ("f32", 30001, 6), ("f32", 65537, 4),
]


def test_shapes_cover_every_phase_count():
    got = {(d, phases(c, 2 if d == "bf16" else 4)) for d, c, _ in SMX_SHAPES}
    assert {("bf16", p) for p in (1, 2, 4, 8)} <= got
    assert {("f32", p) for p in (1, 2, 4)} <= got


def bwd_case(x, dtype, seed):
    """The backward's inputs: the oracle's softmax and log-softmax of x (as
    stored) and an upstream gradient dy ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    dy = store(rng.standard_normal(x.shape), dtype)
    return store(oracle.softmax(x), dtype), store(oracle.log_softmax(x), dtype), dy


def xent_case(rows, cols, dtype, seed):
    x, lab = synth.xent_inputs(rows, cols, dtype, 4.0, seed, ignore_frac=0.1, outlier_frac=0.002,
                               masked_row_every=5)
    lab = lab.copy()
    # labels in the first / last column of rows (their head / tail chunks,
    # shared with the neighbouring rows), and outside [0, cols)
    edge = [0, cols - 1, cols, -1, 1, cols - 2]
    for i, v in enumerate(edge):
        r = 1 + 2 * i
        if r < rows:
            lab[r] = v
    return x, lab


@pytest.mark.parametrize("on", [True, False], ids=["phase", "off"])
@pytest.mark.parametrize("dtype,cols,rows", SMX_SHAPES)
def test_softmax_family_long_rows(dtype, cols, rows, on):
    x, lab = xent_case(rows, cols, dtype, 7000 + cols)
    y, z, dy = bwd_case(x, dtype, cols)
    # RR_SMB=1: the backward's phase-class kernel for fp32 rows too
    with env(RR_SMX="1" if on else "0", RR_SMB="1"):
        check_softmax(x, dtype)
        check_log_softmax(x, dtype)
        check_xent(x, lab, dtype)
        check_softmax_bwd(y, dy, dtype)
        check_softmax_bwd(z, dy, dtype, log=True)


@pytest.mark.parametrize("pad", [1, 3, 8])
@pytest.mark.parametrize("dtype,cols,rows", [("bf16", 4097, 24), ("f32", 2049, 20),
                                             ("bf16", 65537, 3)])
def test_softmax_family_unaligned_bases(dtype, cols, rows, pad, monkeypatch):
    """Input and output shifted by the same element count: every row's phase
    moves, and the first row's copy reads bytes before the tensor."""
    monkeypatch.setenv("RR_SMB", "1")
    x, lab = xent_case(rows, cols, dtype, 7100 + cols + pad)
    e = 2 if dtype == "bf16" else 4
    po = pad + 16 // e  # the same address modulo 16, another place
    check_softmax(x, dtype, pad_in=pad, pad_out=po)
    check_log_softmax(x, dtype, pad_in=pad, pad_out=po)
    check_xent(x, lab, dtype, pad_in=pad, pad_out=po)
    y, z, dy = bwd_case(x, dtype, pad)
    check_softmax_bwd(y, dy, dtype, pads=(pad, po, pad + 2 * (po - pad)))
    check_softmax_bwd(z, dy, dtype, log=True, pads=(po, pad, pad))


@pytest.mark.parametrize("dtype,cols,rows", [("bf16", 4097, 30), ("f32", 2050, 12),
                                             ("bf16", 40001, 4)])
def test_softmax_family_in_place(dtype, cols, rows, monkeypatch):
    monkeypatch.setenv("RR_SMB", "1")
    x, lab = xent_case(rows, cols, dtype, 7200 + cols)
    check_softmax(x, dtype, pad_in=5, inplace=True)
    check_log_softmax(x, dtype, inplace=True)
    check_xent(x, lab, dtype, pad_in=3, inplace=True)
    y, z, dy = bwd_case(x, dtype, 3)
    check_softmax_bwd(y, dy, dtype, inplace="y")
    check_softmax_bwd(z, dy, dtype, log=True, inplace="dy")


def test_xent_every_label_position_of_a_chunk():
    """Rows of 4097 bf16 columns (8 phase classes): row r has label r mod 16
    or cols - 1 - (r mod 16), so every lane of the head and tail chunks of
    every phase class holds a label somewhere."""
    rows, cols = 64, 4097
    x, lab = synth.xent_inputs(rows, cols, "bf16", 2.0, 7300)
    r = np.arange(rows)
    lab = np.where(r % 2 == 0, (r // 2) % 16, cols - 1 - (r // 2) % 16).astype(np.int32)
    check_xent(x, lab, "bf16")


def test_xent_custom_ignore_index_and_all_rows_ignored():
    rows, cols = 16, 4100
    x, lab = synth.xent_inputs(rows, cols, "bf16", 2.0, 7400)
    lab = lab.copy()
    lab[::3] = -1
    check_xent(x, lab, "bf16", ignore_index=-1)
    check_xent(x, np.full(rows, -100, np.int32), "bf16")


# LayerNorm / RMSNorm on the same phase counts, bases and cluster splits
LN_SHAPES = [("bf16", 4097, 40), ("bf16", 4102, 11), ("f32", 2050, 13), ("f32", 2052, 4),
             ("bf16", 65537, 4), ("f32", 40001, 3), ("bf16", 32771, 21), ("bf16", 32768, 6),
             ("f32", 16387, 9), ("f32", 16389, 1), ("bf16", 32772, 2)]


# routed (default: the column-block kernels for rows of 64 KB and more), the
# column-block kernels for every shape (RR_LNC_MIN=16), the pipelined kernels
# wherever they fit (RR_LNP=1), the row-in-registers ones (RR_LNP=0) and
# neither (RR_LNX=0); all but the first two with the column-block kernels off
NORM_KERNELS = {"routed": {}, "column": {"RR_LNC_MIN": "16"},
                "pipelined": {"RR_LNP": "1", "RR_LNC": "0"},
                "registers": {"RR_LNP": "0", "RR_LNC": "0"},
                "off": {"RR_LNX": "0", "RR_LNC": "0"}}


@pytest.mark.parametrize("kern", list(NORM_KERNELS))
@pytest.mark.parametrize("dtype,cols,rows", LN_SHAPES)
def test_norms_long_rows(dtype, cols, rows, kern):
    x, g, b, dy = synth.ln_inputs(rows, cols, dtype, 7500 + cols, row_offset=10.0, gamma_std=0.1,
                                  beta_std=0.1, outlier_frac=0.002, masked_row_every=7)
    with env(**NORM_KERNELS[kern]):
        check_ln(x, g, b, dy, 1e-5, dtype)
        check_rms(x, g, dy, 1e-5, dtype)
        check_norm_bwd(x, g, b, dy, dtype, inplace="dy")


@pytest.mark.parametrize("kern", ["routed", "pipelined", "column"])
@pytest.mark.parametrize("dtype,cols,rows", [("bf16", 4097, 17), ("f32", 2049, 9),
                                             ("bf16", 32771, 10)])
def test_norms_unaligned_bases(dtype, cols, rows, kern):
    x, g, b, dy = synth.ln_inputs(rows, cols, dtype, 7600 + cols, row_offset=3.0, gamma_std=0.2,
                                  beta_std=0.2)
    e = 2 if dtype == "bf16" else 4
    v = 16 // e
    # x, y, dy and dx at the same address modulo 16, other places; gamma /
    # beta elsewhere
    with env(**NORM_KERNELS[kern]):
        check_ln(x, g, b, dy, 1e-5, dtype, pad=(3, 3 + v, 2, 3 + 2 * v, 3 + v))
        check_norm_bwd(x, g, b, dy, dtype, stat_pad=1)
        check_rms(x, g, dy, 1e-5, dtype, pad=(5, 5 + v, 1, 5, 5 + 2 * v))


@pytest.mark.parametrize("dtype,cols,rows", [("bf16", 32771, 9), ("f32", 16387, 5)])
def test_norm_forward_in_place_long_rows(dtype, cols, rows):
    """y == x for rows the column-block kernels take otherwise (they keep their
    row records in y, so an in-place call goes to the phase-aligned kernels):
    LayerNorm and RMSNorm against the oracle, guard bands intact."""
    x, g, b, _ = synth.ln_inputs(rows, cols, dtype, 7700 + cols, row_offset=5.0, gamma_std=0.1,
                                 beta_std=0.1, outlier_frac=0.002, masked_row_every=4)
    rtol, atol = TOL[dtype]
    ry, rmean, rrstd = oracle.ln_fwd(x, g, b, 1e-5)
    xd, gd, bd = to_dev(x, 3), to_dev(g), to_dev(b)
    mean, rstd = out_f32(rows), out_f32(rows)
    rr.rr_layernorm_fwd(xd, gd, bd, xd, mean, rstd, eps=1e-5)
    torch.cuda.synchronize()
    check_guards()
    compare("ln y in place", host(xd), ry, rtol, atol)
    compare("ln mean", host(mean), rmean, *TOL_F32_OUT)
    compare("ln rstd", host(rstd), rrstd, *TOL_F32_OUT)
    ry, rrstd = oracle.rms_fwd(x, g, 1e-5)
    xd = to_dev(x, 5)
    rstd = out_f32(rows)
    rr.rr_rmsnorm_fwd(xd, gd, xd, rstd, eps=1e-5)
    torch.cuda.synchronize()
    check_guards()
    compare("rms y in place", host(xd), ry, rtol, atol)
    compare("rms rstd", host(rstd), rrstd, *TOL_F32_OUT)
