"""rr_layernorm_bwd_noalloc: the LayerNorm backward for callers that cannot
allocate device memory when they call it (it keeps its column partials in a
fixed scratch array inside the library instead of a caller workspace).

Called through the C ABI; its outputs must match rr_layernorm_bwd's (which
gets a caller-allocated workspace) on two calls in a row, since the scratch is
shared and keeps the previous call's contents.  The file sorts last so that a
run stopping at the first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import row_reduction_pass_gb300 as rr
from row_reduction_pass_gb300 import synth

from parity import TOL, compare, host, to_dev

pytestmark = pytest.mark.gpu


def _dev_inputs(rows, cols, dtype, seed):
    x, g, b, dy = synth.ln_inputs(rows, cols, dtype, seed, row_offset=10.0, outlier_frac=0.002,
                                  masked_row_every=97)
    xd, gd, bd, dyd = to_dev(x), to_dev(g), to_dev(b), to_dev(dy)
    y = torch.empty_like(xd)
    mean = torch.empty(rows, device=xd.device)
    rstd = torch.empty(rows, device=xd.device)
    rr.rr_layernorm_fwd(xd, gd, bd, y, mean, rstd, eps=1e-5)
    return xd, gd, dyd, mean, rstd


def _call_noalloc(lib, dyd, xd, mean, rstd, gd, dx, dg, db):
    rows, cols = xd.shape
    code = 0 if xd.dtype == torch.float32 else 1
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.rr_layernorm_bwd_noalloc(p(dyd), p(xd), p(mean), p(rstd), p(gd), p(dx), p(dg), p(db),
                                      rows, cols, code,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.rr_last_error_detail()


# (1000, 9001, f32): rr_layernorm_bwd's plan wants more than 8 MiB of partials,
# so this one runs with fewer row groups than the workspace variant
@pytest.mark.parametrize("rows,cols,dtype", [(4096, 768, "f32"), (3000, 97, "bf16"),
                                             (1000, 2048, "f32"), (777, 4097, "bf16"),
                                             (1000, 9001, "f32")])
def test_noalloc_matches_workspace_variant_twice(rows, cols, dtype):
    lib = rr.load_library()
    xd, gd, dyd, mean, rstd = _dev_inputs(rows, cols, dtype, 11 + cols)
    ref_dx, ref_dg, ref_db = torch.empty_like(xd), torch.empty_like(gd), torch.empty_like(gd)
    rr.rr_layernorm_bwd(dyd, xd, mean, rstd, gd, ref_dx, ref_dg, ref_db)
    torch.cuda.synchronize()
    rtol, atol = TOL[dtype]
    # dgamma / dbeta are fp32 column sums whose rounding follows the number of
    # row groups; both calls are held to the parity bound against sum_r |term_r|
    live = (rstd != 0)[:, None]           # rstd == 0 marks a masked row: no terms
    xh = (xd.double() - mean.double()[:, None]) * rstd.double()[:, None]
    zero = torch.zeros((), dtype=torch.float64, device=xd.device)
    sdg = host(torch.where(live, (dyd.double() * xh).abs(), zero).sum(0))
    sdb = host(torch.where(live, dyd.double().abs(), zero).sum(0))
    for _ in range(2):
        dx = torch.full_like(xd, float("nan"))
        dg = torch.full_like(gd, float("nan"))
        db = torch.full_like(gd, float("nan"))
        _call_noalloc(lib, dyd, xd, mean, rstd, gd, dx, dg, db)
        torch.cuda.synchronize()
        compare("noalloc dx", host(dx), host(ref_dx), rtol, atol)
        compare("noalloc dgamma", host(dg), host(ref_dg), rtol, atol, scale=2 * sdg)
        compare("noalloc dbeta", host(db), host(ref_db), rtol, atol, scale=2 * sdb)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = rr.load_library()
    rows, cols = 2, (1 << 20) + 1        # one partial alone is beyond 8 MiB; nothing is launched
    fake = ctypes.c_void_p(1 << 20)
    st = lib.rr_layernorm_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, rows, cols, 0,
                                      ctypes.c_void_p(0))
    assert st == 4                        # RR_ERR_WORKSPACE_TOO_SMALL
    assert b"8 MiB" in lib.rr_last_error_detail()
