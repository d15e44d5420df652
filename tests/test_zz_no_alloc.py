"""rr_layernorm_bwd_noalloc: the LayerNorm backward for callers that cannot
allocate device memory when they call it (it keeps its column partials in a
fixed scratch array inside the library instead of a caller workspace).

Called through the C ABI; its outputs must match rr_layernorm_bwd's (which
gets a caller-allocated workspace) and the float64 oracle's on two calls in a
row, since the scratch is shared and keeps the previous call's contents.  The file sorts last so that a
run stopping at the first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import row_reduction_pass_gb300 as rr
from row_reduction_pass_gb300 import synth

from parity import TOL, check_guards, compare, empty_like_dev, host, to_dev

pytestmark = pytest.mark.gpu


def _inputs(rows, cols, dtype, seed):
    x, g, b, dy = synth.ln_inputs(rows, cols, dtype, seed, row_offset=10.0, outlier_frac=0.002,
                                  masked_row_every=97)
    # the saved statistics: the oracle's, rounded to float32 as the forward stores them
    _, m64, r64 = oracle.ln_fwd(x, g, b, 1e-5, want_y=False)
    mean, rstd = to_dev(m64.astype(np.float32)), to_dev(r64.astype(np.float32))
    xd, gd, dyd = to_dev(x), to_dev(g), to_dev(dy)
    return (x, g, dy), (xd, gd, dyd, mean, rstd)


def _call_noalloc(lib, dyd, xd, mean, rstd, gd, dx, dg, db):
    rows, cols = xd.shape
    code = 0 if xd.dtype == torch.float32 else 1
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib.rr_layernorm_bwd_noalloc(p(dyd), p(xd), p(mean), p(rstd), p(gd), p(dx), p(dg),
                                        p(db), rows, cols, code,
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check_twice(rows, cols, dtype, seed):
    """Two no-allocation calls in a row against the workspace entry point and
    against the float64 oracle (given the same float32 mean / rstd)."""
    lib = rr.load_library()
    (x, g, dy), (xd, gd, dyd, mean, rstd) = _inputs(rows, cols, dtype, seed)
    ref_dx = empty_like_dev(x.shape, dtype)
    ref_dg, ref_db = empty_like_dev(g.shape, dtype), empty_like_dev(g.shape, dtype)
    rr.rr_layernorm_bwd(dyd, xd, mean, rstd, gd, ref_dx, ref_dg, ref_db)
    torch.cuda.synchronize()
    rtol, atol = TOL[dtype]
    odx, odg, odb, sdg, sdb = oracle.ln_bwd(dy, x, host(mean), host(rstd), g)
    for _ in range(2):
        dx = empty_like_dev(x.shape, dtype)
        dg, db = empty_like_dev(g.shape, dtype), empty_like_dev(g.shape, dtype)
        st = _call_noalloc(lib, dyd, xd, mean, rstd, gd, dx, dg, db)
        assert st == 0, lib.rr_last_error_detail()
        torch.cuda.synchronize()
        check_guards()
        # dgamma / dbeta are fp32 column sums whose rounding follows the number
        # of row groups; against each other both sides' bounds add up
        compare("noalloc dx vs workspace call", host(dx), host(ref_dx), rtol, atol)
        compare("noalloc dgamma vs workspace call", host(dg), host(ref_dg), rtol, atol,
                scale=2 * sdg)
        compare("noalloc dbeta vs workspace call", host(db), host(ref_db), rtol, atol,
                scale=2 * sdb)
        compare("noalloc dx vs oracle", host(dx), odx, rtol, atol)
        compare("noalloc dgamma vs oracle", host(dg), odg, rtol, atol, scale=sdg)
        compare("noalloc dbeta vs oracle", host(db), odb, rtol, atol, scale=sdb)


# (1000, 9001, f32): rr_layernorm_bwd's plan wants more than 8 MiB of partials,
# so this one runs with fewer row groups than the workspace variant
@pytest.mark.parametrize("rows,cols,dtype", [(4096, 768, "f32"), (3000, 97, "bf16"),
                                             (1000, 2048, "f32"), (777, 4097, "bf16"),
                                             (1000, 9001, "f32")])
def test_noalloc_matches_workspace_variant_twice(rows, cols, dtype):
    _check_twice(rows, cols, dtype, 11 + cols)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_longest_supported_rows(dtype, monkeypatch):
    """The longest rows the LayerNorm backward holds without the column-block
    kernels (which take rows of any length; RR_LNC=0 here), found through the
    workspace size query, which returns 0 for rows no kernel holds: the
    scratch then carries the fewest column partials.  One column beyond, both
    entry points refuse the shape with the same status."""
    monkeypatch.setenv("RR_LNC", "0")
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    lo, hi = 65537, 1 << 20            # supported / not (one partial is 8 MiB at 2^20)
    assert rr.rr_layernorm_bwd_workspace_size(3, lo, tdt) > 0
    assert rr.rr_layernorm_bwd_workspace_size(3, hi, tdt) == 0
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if rr.rr_layernorm_bwd_workspace_size(3, mid, tdt) > 0:
            lo = mid
        else:
            hi = mid
    _check_twice(3, lo, dtype, 5)
    if rr.rr_layernorm_bwd_workspace_size(3, lo + 1, tdt) == 0:
        lib = rr.load_library()
        (_, _, _), (xd, gd, dyd, mean, rstd) = _inputs(3, lo + 1, dtype, 6)
        dx = empty_like_dev(tuple(xd.shape), dtype)
        dg, db = empty_like_dev((lo + 1,), dtype), empty_like_dev((lo + 1,), dtype)
        st = _call_noalloc(lib, dyd, xd, mean, rstd, gd, dx, dg, db)
        with pytest.raises(rr.RRError) as ei:
            rr.rr_layernorm_bwd(dyd, xd, mean, rstd, gd, dx, dg, db,
                                workspace=torch.empty(1 << 24, dtype=torch.uint8,
                                                      device=xd.device))
        assert st == ei.value.status


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = rr.load_library()
    rows, cols = 2, (1 << 20) + 1        # one partial alone is beyond 8 MiB; nothing is launched
    fake = [ctypes.c_void_p((i + 1) << 40) for i in range(8)]
    st = lib.rr_layernorm_bwd_noalloc(*fake, rows, cols, 0, ctypes.c_void_p(0))
    assert st == 4                        # RR_ERR_WORKSPACE_TOO_SMALL
    assert b"8 MiB" in lib.rr_last_error_detail()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_noalloc_column_block_rows(dtype):
    """Rows the column-block kernels take (255 x 65537, the sweep's longest):
    the no-allocation entry point fits their column partials and row records
    in its scratch (with fewer row groups where needed); both entry points
    agree with the oracle."""
    _check_twice(255, 65537, dtype, 7)
