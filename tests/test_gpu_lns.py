"""GPU parity of the LayerNorm / RMSNorm backward on short rows whose byte
length is not a multiple of 16 (65 bytes to 1 KB): the phase-class kernels
(a warp per row or two, rows grouped by their offset within a 16-byte block),
against the float64 oracle through the C ABI.  Row lengths on both sides of
each variant's limit (16, 32, 64 chunks) and of the tier's (64 bytes below,
~1 KB above), row counts below the number of phase classes (empty classes),
ragged ones and hundreds of thousands, ±1e4 outliers and masked rows, bases
off a 16-byte boundary (the same offset for dy, x and dx, and different ones,
which go to the row-group kernels), statistics off a boundary, dx written
over dy or x, and the no-allocation entry point."""
import numpy as np
import pytest
import torch

import oracle
import row_reduction_pass_gb300 as rr
from row_reduction_pass_gb300 import synth

from parity import TOL, check_guards, compare, empty_like_dev, host, to_dev

pytestmark = pytest.mark.gpu

CASES = [("f32", c) for c in (17, 31, 33, 63, 97, 127, 129, 250, 251)] + \
        [("bf16", c) for c in (33, 47, 97, 127, 129, 255, 257, 499, 503)]


def run(x, g, b, dy, dtype, rms, pads=(0, 0, 0), stat_pad=0, inplace=None):
    """The backward alone on the oracle's float32 statistics; pads = element
    offsets of (x, dy, dx) past a 16-byte boundary."""
    rows = x.shape[0]
    if rms:
        _, r64 = oracle.rms_fwd(x, g, 1e-5, want_y=False)
        m64 = np.zeros(rows)
    else:
        _, m64, r64 = oracle.ln_fwd(x, g, b, 1e-5, want_y=False)
    m32, r32 = m64.astype(np.float32), r64.astype(np.float32)
    md, rd = to_dev(m32, stat_pad), to_dev(r32, stat_pad)
    xd, dyd, gd = to_dev(x, pads[0]), to_dev(dy, pads[1]), to_dev(g)
    dx = {"dy": dyd, "x": xd}.get(inplace) if inplace else empty_like_dev(x.shape, dtype, pads[2])
    dg = empty_like_dev(g.shape, dtype)
    rtol, atol = TOL[dtype]
    if rms:
        rr.rr_rmsnorm_bwd(dyd, xd, rd, gd, dx, dg)
        torch.cuda.synchronize()
        check_guards()
        rdx, rdg, sdg = oracle.rms_bwd(dy, x, r32.astype(np.float64), g)
    else:
        db = empty_like_dev(g.shape, dtype)
        rr.rr_layernorm_bwd(dyd, xd, md, rd, gd, dx, dg, db)
        torch.cuda.synchronize()
        check_guards()
        rdx, rdg, rdb, sdg, sdb = oracle.ln_bwd(dy, x, m32.astype(np.float64),
                                                r32.astype(np.float64), g)
        compare("dbeta", host(db), rdb, rtol, atol, scale=sdb)
    compare("dx", host(dx), rdx, rtol, atol)
    compare("dgamma", host(dg), rdg, rtol, atol, scale=sdg)


def inputs(rows, cols, dtype, seed):
    return synth.ln_inputs(rows, cols, dtype, seed, row_offset=10.0, gamma_std=0.1,
                           beta_std=0.1, outlier_frac=0.005, masked_row_every=41)


@pytest.mark.parametrize("dtype,cols", CASES)
@pytest.mark.parametrize("rows", [1, 3, 5003, 200003])
@pytest.mark.parametrize("rms", [False, True])
def test_short_row_backward(dtype, cols, rows, rms):
    if rows * cols > 30_000_000:
        pytest.skip("oracle time")
    x, g, b, dy = inputs(rows, cols, dtype, 1100 + cols + rows)
    run(x, g, b, dy, dtype, rms)


@pytest.mark.parametrize("dtype,cols", [("f32", 31), ("f32", 97), ("bf16", 97), ("bf16", 255)])
@pytest.mark.parametrize("layout", ["same_offset", "mixed_offsets", "stats_off", "dx_over_dy",
                                    "dx_over_x"])
@pytest.mark.parametrize("rms", [False, True])
def test_short_row_backward_layouts(dtype, cols, layout, rms):
    x, g, b, dy = inputs(20011, cols, dtype, 1300 + cols)
    if layout == "same_offset":
        run(x, g, b, dy, dtype, rms, pads=(3, 3, 3))
    elif layout == "mixed_offsets":
        run(x, g, b, dy, dtype, rms, pads=(1, 2, 0))
    elif layout == "stats_off":
        run(x, g, b, dy, dtype, rms, stat_pad=1)
    elif layout == "dx_over_dy":
        run(x, g, b, dy, dtype, rms, inplace="dy")
    else:
        run(x, g, b, dy, dtype, rms, inplace="x")


@pytest.mark.parametrize("dtype,cols", [("f32", 97), ("bf16", 499)])
def test_short_row_backward_noalloc(dtype, cols):
    """The no-allocation entry point caps the blocks (one partial each) at
    its scratch; two calls in a row against the oracle."""
    rows = 300007
    x, g, b, dy = inputs(rows, cols, dtype, 1400 + cols)
    _, m64, r64 = oracle.ln_fwd(x, g, b, 1e-5, want_y=False)
    md, rd = to_dev(m64.astype(np.float32)), to_dev(r64.astype(np.float32))
    xd, gd, dyd = to_dev(x), to_dev(g), to_dev(dy)
    odx, odg, odb, sdg, sdb = oracle.ln_bwd(dy, x, host(md), host(rd), g)
    rtol, atol = TOL[dtype]
    for _ in range(2):
        dx = empty_like_dev(x.shape, dtype)
        dg, db = empty_like_dev(g.shape, dtype), empty_like_dev(g.shape, dtype)
        rr.rr_layernorm_bwd_noalloc(dyd, xd, md, rd, gd, dx, dg, db)
        torch.cuda.synchronize()
        check_guards()
        compare("noalloc dx", host(dx), odx, rtol, atol)
        compare("noalloc dgamma", host(dg), odg, rtol, atol, scale=sdg)
        compare("noalloc dbeta", host(db), odb, rtol, atol, scale=sdb)
