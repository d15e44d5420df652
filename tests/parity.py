"""Helpers shared by the GPU parity tests: host<->device marshalling of the
seeded inputs, the comparison rule, and one call per operation through the C
ABI (via the package binding) next to the float64 oracle on the same inputs.

Comparison rule (elementwise, both sides NaN counts as equal):
    |gpu - ref| <= atol + rtol * |ref|
  outputs in the I/O dtype:  fp32 rtol 1e-5, atol 1e-5;  bf16 rtol 2e-2, atol 1e-5
  float32 outputs (loss, mean, rstd):                   rtol 1e-5, atol 1e-5
  dgamma / dbeta (sums over rows):
    |gpu - ref| <= rtol_io * |ref| + 1e-5 * sum_r |term_r| + 1e-5

Guard bands: every device buffer these helpers make (inputs, outputs, in-place
tensors, per-row statistics, counters) sits inside a larger allocation whose
GUARD elements before it (plus any misalignment padding) and GUARD elements
after it hold a sentinel bit pattern.  check_guards() asserts that no kernel
wrote a byte there; the run_* helpers call it after every launch, and an
autouse fixture (conftest.py) calls it again when each test ends.  This is the
out-of-bounds write check for the ragged, misaligned and in-place paths.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import row_reduction_pass_gb300 as rr
from row_reduction_pass_gb300 import synth

TOL = {"f32": (1e-5, 1e-5), "bf16": (2e-2, 1e-5)}
TOL_F32_OUT = (1e-5, 1e-5)


def dev():
    return torch.device("cuda:0")


GUARD = 64  # sentinel elements before and after every buffer (>= 128 bytes)
# Sentinel bits: a NaN payload no kernel produces (kernels write quiet NaNs
# with the canonical payload, numbers, or nothing).
_SENTINEL = {torch.float32: (torch.int32, 0x7FA5A5A5), torch.bfloat16: (torch.int16, 0x7FA5),
             torch.int32: (torch.int32, 0x7FA5A5A5)}
_GUARDED: list = []


def _guarded(n: int, tdt, pad_elems: int) -> torch.Tensor:
    """A 1-D device buffer of n elements of tdt that starts GUARD + pad_elems
    elements into an allocation filled with the sentinel; registered for
    check_guards().  GUARD * element size is a multiple of 16, so the view's
    alignment modulo 16 is pad_elems * element size."""
    itype, bits = _SENTINEL[tdt]
    start = GUARD + pad_elems
    raw = torch.full((start + n + GUARD,), bits, dtype=itype, device=dev())
    _GUARDED.append((raw, start, n, bits))
    view = raw[start:start + n]
    return view if tdt == torch.int32 else view.view(tdt)


def check_guards(clear: bool = False):
    """Asserts that the guard bands of every registered buffer still hold the
    sentinel (no out-of-bounds write); clear=True forgets the buffers."""
    bad = []
    for raw, start, n, bits in _GUARDED:
        pre = raw[:start] != bits
        post = raw[start + n:] != bits
        if bool(pre.any()) or bool(post.any()):
            i_pre = torch.nonzero(pre).flatten().tolist()
            i_post = torch.nonzero(post).flatten().tolist()
            bad.append(f"buffer of {n} elements: {len(i_pre)} written before it "
                       f"(offsets {[i - start for i in i_pre[:4]]}), {len(i_post)} after it "
                       f"(offsets {[n + i for i in i_post[:4]]})")
    if clear:
        _GUARDED.clear()
    assert not bad, "out-of-bounds writes: " + "; ".join(bad)


def to_dev(a: np.ndarray, pad_elems: int = 0) -> torch.Tensor:
    """Copy a host array (float32, bf16 bits or int32) to the GPU inside a
    guard band.  pad_elems > 0 places it pad_elems elements past a 16-byte
    aligned start (a misaligned base)."""
    if a.dtype == np.uint16:
        flat = torch.from_numpy(np.ascontiguousarray(a).view(np.int16).reshape(-1))
        tdt = torch.bfloat16
    elif a.dtype == np.float32:
        flat = torch.from_numpy(np.ascontiguousarray(a).reshape(-1))
        tdt = torch.float32
    elif a.dtype == np.int32:
        flat = torch.from_numpy(np.ascontiguousarray(a).reshape(-1))
        tdt = torch.int32
    else:
        raise TypeError(a.dtype)
    view = _guarded(a.size, tdt, pad_elems)
    raw = view if tdt != torch.bfloat16 else view.view(torch.int16)
    raw.copy_(flat.to(dev()))
    return view.view(a.shape)


def empty_like_dev(shape, dtype: str, pad_elems: int = 0, fill=float("nan")) -> torch.Tensor:
    """Device output buffer poisoned with NaN (so unwritten outputs are
    caught), inside a guard band."""
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32}[dtype]
    n = int(np.prod(shape))
    view = _guarded(n, tdt, pad_elems)
    view.fill_(fill)
    return view.view(shape)


def out_f32(n: int, pad_elems: int = 0) -> torch.Tensor:
    """A float32 per-row output (loss, mean, rstd) poisoned with NaN, guarded."""
    return empty_like_dev((n,), "f32", pad_elems)


def zeros_i32(n: int) -> torch.Tensor:
    """A zeroed int32 device counter, guarded."""
    return empty_like_dev((n,), "i32", 0, fill=0)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare(name: str, got: np.ndarray, ref: np.ndarray, rtol: float, atol: float,
            scale: np.ndarray | None = None, scale_rtol: float = 1e-5):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} != {ref.shape}"
    both_nan = np.isnan(got) & np.isnan(ref)
    with np.errstate(invalid="ignore"):  # inf - inf where both are infinite
        err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    if scale is not None:
        bound = bound + scale_rtol * scale
    same_inf = np.isinf(got) & np.isinf(ref) & (np.sign(got) == np.sign(ref))
    ok = both_nan | same_inf | (err <= bound)
    if not ok.all():
        idx = np.unravel_index(np.argmax(np.where(ok, -1.0, np.nan_to_num(err, nan=np.inf))),
                               got.shape)
        raise AssertionError(
            f"{name}: {int((~ok).sum())} of {ok.size} outside tolerance; worst at {idx}: "
            f"gpu={got[idx]!r} ref={ref[idx]!r} bound={bound[idx]!r}")
    finite = np.isfinite(got) & np.isfinite(ref)
    return float(err[finite].max()) if finite.any() else 0.0


# ----------------------------------------------------------------- ops ----

def run_softmax(x: np.ndarray, dtype: str, pad_in=0, pad_out=0, inplace=False):
    xd = to_dev(x, pad_in)
    y = xd if inplace else empty_like_dev(x.shape, dtype, pad_out)
    rr.rr_softmax_fwd(xd, y)
    torch.cuda.synchronize()
    check_guards()
    return host(y)


def check_softmax(x, dtype, **kw):
    got = run_softmax(x, dtype, **kw)
    ref = oracle.softmax(x)
    rtol, atol = TOL[dtype]
    compare("softmax y", got, ref, rtol, atol)


def run_xent(logits, labels, dtype, ignore_index=-100, pad_in=0, pad_out=0, inplace=False):
    xd = to_dev(logits, pad_in)
    lab = to_dev(labels)
    loss = out_f32(logits.shape[0])
    dl = xd if inplace else empty_like_dev(logits.shape, dtype, pad_out)
    bad = zeros_i32(1)
    rr.rr_softmax_xent_fwd_bwd(xd, lab, loss, dl, ignore_index=ignore_index, bad_label_count=bad)
    torch.cuda.synchronize()
    check_guards()
    return host(loss), host(dl), int(bad.item())


def check_xent(logits, labels, dtype, ignore_index=-100, **kw):
    loss, dl, bad = run_xent(logits, labels, dtype, ignore_index, **kw)
    rloss, rdl, rbad = oracle.xent(logits, labels, ignore_index)
    rtol, atol = TOL[dtype]
    compare("xent loss", loss, rloss, *TOL_F32_OUT)
    compare("xent dlogits", dl, rdl, rtol, atol)
    assert bad == rbad, f"bad label count {bad} != {rbad}"


def run_ln(x, gamma, beta, dy, eps, dtype, pad=(0, 0, 0, 0, 0), oracle_stats=True):
    """LayerNorm fwd then bwd on the GPU.  pad = element offsets of
    (x, y, gamma/beta, dy, dx).  The backward gets the oracle's mean / rstd
    (rounded to float32) when oracle_stats, else the GPU forward's."""
    xd = to_dev(x, pad[0])
    gd = to_dev(gamma, pad[2])
    bd = to_dev(beta, pad[2])
    y = empty_like_dev(x.shape, dtype, pad[1])
    rows = x.shape[0]
    mean = out_f32(rows)
    rstd = out_f32(rows)
    rr.rr_layernorm_fwd(xd, gd, bd, y, mean, rstd, eps=eps)
    _, rmean, rrstd = oracle.ln_fwd(x, gamma, beta, eps, want_y=False)
    if oracle_stats:
        m_in = to_dev(rmean.astype(np.float32))
        r_in = to_dev(rrstd.astype(np.float32))
    else:
        m_in, r_in = mean, rstd
    dyd = to_dev(dy, pad[3])
    dx = empty_like_dev(x.shape, dtype, pad[4])
    dg = empty_like_dev(gamma.shape, dtype)
    db = empty_like_dev(gamma.shape, dtype)
    rr.rr_layernorm_bwd(dyd, xd, m_in, r_in, gd, dx, dg, db)
    torch.cuda.synchronize()
    check_guards()
    return dict(y=host(y), mean=host(mean), rstd=host(rstd), dx=host(dx), dgamma=host(dg),
                dbeta=host(db), mean_in=m_in.cpu().numpy().astype(np.float64),
                rstd_in=r_in.cpu().numpy().astype(np.float64))


def check_ln(x, gamma, beta, dy, eps, dtype, pad=(0, 0, 0, 0, 0), oracle_stats=True):
    g = run_ln(x, gamma, beta, dy, eps, dtype, pad, oracle_stats)
    ry, rmean, rrstd = oracle.ln_fwd(x, gamma, beta, eps)
    rtol, atol = TOL[dtype]
    compare("ln y", g["y"], ry, rtol, atol)
    compare("ln mean", g["mean"], rmean, *TOL_F32_OUT)
    compare("ln rstd", g["rstd"], rrstd, *TOL_F32_OUT)
    # The backward's own inputs include mean / rstd: the oracle gets exactly the
    # float32 values the GPU was given (the oracle's statistics rounded to
    # float32).  In the chained check (GPU statistics into the GPU backward) the
    # oracle chains its own float64 statistics instead.
    if oracle_stats:
        rdx, rdg, rdb, sdg, sdb = oracle.ln_bwd(dy, x, g["mean_in"], g["rstd_in"], gamma)
    else:
        rdx, rdg, rdb, sdg, sdb = oracle.ln_bwd(dy, x, rmean, rrstd, gamma)
    compare("ln dx", g["dx"], rdx, rtol, atol)
    compare("ln dgamma", g["dgamma"], rdg, rtol, atol, scale=sdg)
    compare("ln dbeta", g["dbeta"], rdb, rtol, atol, scale=sdb)
    return g


def check_norm_bwd(x, gamma, beta, dy, dtype, rms=False, stat_pad=0, inplace=None):
    """The LayerNorm (or RMSNorm) backward alone, given the oracle's statistics
    rounded to float32 and stored stat_pad elements past a 16-byte boundary;
    inplace = "dy" or "x" writes dx over that input."""
    rows = x.shape[0]
    if rms:
        _, rrstd = oracle.rms_fwd(x, gamma, 1e-5, want_y=False)
        rmean = np.zeros(rows)
    else:
        _, rmean, rrstd = oracle.ln_fwd(x, gamma, beta, 1e-5, want_y=False)
    m32, r32 = rmean.astype(np.float32), rrstd.astype(np.float32)
    m_in, r_in = to_dev(m32, stat_pad), to_dev(r32, stat_pad)
    xd, dyd, gd = to_dev(x), to_dev(dy), to_dev(gamma)
    dx = {"dy": dyd, "x": xd}.get(inplace) if inplace else empty_like_dev(x.shape, dtype)
    dg = empty_like_dev(gamma.shape, dtype)
    rtol, atol = TOL[dtype]
    if rms:
        rr.rr_rmsnorm_bwd(dyd, xd, r_in, gd, dx, dg)
        torch.cuda.synchronize()
        check_guards()
        rdx, rdg, sdg = oracle.rms_bwd(dy, x, r32.astype(np.float64), gamma)
    else:
        db = empty_like_dev(gamma.shape, dtype)
        rr.rr_layernorm_bwd(dyd, xd, m_in, r_in, gd, dx, dg, db)
        torch.cuda.synchronize()
        check_guards()
        rdx, rdg, rdb, sdg, sdb = oracle.ln_bwd(dy, x, m32.astype(np.float64),
                                                r32.astype(np.float64), gamma)
        compare("norm bwd dbeta", host(db), rdb, rtol, atol, scale=sdb)
    compare("norm bwd dx", host(dx), rdx, rtol, atol)
    compare("norm bwd dgamma", host(dg), rdg, rtol, atol, scale=sdg)


def run_rms(x, gamma, dy, eps, dtype, pad=(0, 0, 0, 0, 0), oracle_stats=True):
    """RMSNorm fwd then bwd on the GPU; pad as for run_ln (the beta slot unused).
    The backward gets the oracle's rstd rounded to float32 when oracle_stats."""
    xd = to_dev(x, pad[0])
    gd = to_dev(gamma, pad[2])
    y = empty_like_dev(x.shape, dtype, pad[1])
    rows = x.shape[0]
    rstd = out_f32(rows)
    rr.rr_rmsnorm_fwd(xd, gd, y, rstd, eps=eps)
    _, rrstd = oracle.rms_fwd(x, gamma, eps, want_y=False)
    r_in = to_dev(rrstd.astype(np.float32)) if oracle_stats else rstd
    dyd = to_dev(dy, pad[3])
    dx = empty_like_dev(x.shape, dtype, pad[4])
    dg = empty_like_dev(gamma.shape, dtype)
    rr.rr_rmsnorm_bwd(dyd, xd, r_in, gd, dx, dg)
    torch.cuda.synchronize()
    check_guards()
    return dict(y=host(y), rstd=host(rstd), dx=host(dx), dgamma=host(dg),
                rstd_in=r_in.cpu().numpy().astype(np.float64))


def check_rms(x, gamma, dy, eps, dtype, pad=(0, 0, 0, 0, 0), oracle_stats=True):
    g = run_rms(x, gamma, dy, eps, dtype, pad, oracle_stats)
    ry, rrstd = oracle.rms_fwd(x, gamma, eps)
    rtol, atol = TOL[dtype]
    compare("rms y", g["y"], ry, rtol, atol)
    compare("rms rstd", g["rstd"], rrstd, *TOL_F32_OUT)
    rdx, rdg, sdg = oracle.rms_bwd(dy, x, g["rstd_in"] if oracle_stats else rrstd, gamma)
    compare("rms dx", g["dx"], rdx, rtol, atol)
    compare("rms dgamma", g["dgamma"], rdg, rtol, atol, scale=sdg)
    return g


def store(a64: np.ndarray, dtype: str) -> np.ndarray:
    """A float64 host array as stored inputs (float32, or bf16 bits)."""
    a32 = np.ascontiguousarray(a64, np.float32)
    return a32 if dtype == "f32" else synth.bf16_bits(a32)


def check_log_softmax(x, dtype, pad_in=0, pad_out=0, inplace=False):
    xd = to_dev(x, pad_in)
    z = xd if inplace else empty_like_dev(x.shape, dtype, pad_out)
    rr.rr_log_softmax_fwd(xd, z)
    torch.cuda.synchronize()
    check_guards()
    rtol, atol = TOL[dtype]
    compare("log_softmax z", host(z), oracle.log_softmax(x), rtol, atol)


def check_softmax_bwd(y, dy, dtype, log=False, pads=(0, 0, 0), inplace=None):
    """y (softmax output, or log-softmax output z when log) and dy are stored
    inputs; inplace = "y" or "dy" writes dx over that input."""
    yd = to_dev(y, pads[0])
    dyd = to_dev(dy, pads[1])
    if inplace == "y":
        dx = yd
    elif inplace == "dy":
        dx = dyd
    else:
        dx = empty_like_dev(y.shape, dtype, pads[2])
    (rr.rr_log_softmax_bwd if log else rr.rr_softmax_bwd)(yd, dyd, dx)
    torch.cuda.synchronize()
    check_guards()
    ref = oracle.log_softmax_bwd(y, dy) if log else oracle.softmax_bwd(y, dy)
    rtol, atol = TOL[dtype]
    compare("log_softmax dx" if log else "softmax dx", host(dx), ref, rtol, atol)
