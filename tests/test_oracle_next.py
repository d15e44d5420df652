"""Pins for the oracle's softmax backward, log-softmax forward / backward and
RMSNorm forward / backward, each checked against something other than its own
formula: torch / scipy float64 routines and autograd, closed forms worked by
hand, invariants, central finite differences (the gradient check of the
"NexusGrad" README, sec. "Testing") and masked rows.  No GPU needed."""
import math

import numpy as np
import pytest
import scipy.special as sps
import torch

import oracle

RNG = np.random.default_rng(2468)


def f32(a):
    return np.ascontiguousarray(a, np.float32)


def dyadic(shape, scale=1.0, step=2.0 ** -8):
    return f32(np.round(RNG.normal(0, scale, size=shape) / step) * step)


def t64(a):
    return torch.tensor(np.asarray(a, np.float64), dtype=torch.float64)


# ---------------------------------------------------------- softmax backward

@pytest.mark.parametrize("shape", [(1, 1), (3, 5), (4, 97), (2, 1000)])
def test_softmax_bwd_matches_torch_vjp(shape):
    x = f32(RNG.normal(0, 2, size=shape))
    dy = f32(RNG.normal(0, 1, size=shape))
    xt = t64(x).requires_grad_()
    yt = torch.softmax(xt, 1)
    (g,) = torch.autograd.grad(yt, xt, t64(dy))
    # the oracle reads y as stored (float32): equal to the VJP up to that rounding
    dx = oracle.softmax_bwd(f32(yt.detach().numpy()), dy)
    np.testing.assert_allclose(dx, g.numpy(), rtol=2e-6, atol=2e-7)


def test_softmax_bwd_closed_form_and_invariants():
    p = [0.0900305732, 0.2447284711, 0.6652409558]  # softmax([1, 2, 3])
    dx = oracle.softmax_bwd(f32([p]), f32([[1.0, 0.0, 0.0]]))
    np.testing.assert_allclose(dx[0], [p[0] * (1 - p[0]), -p[1] * p[0], -p[2] * p[0]], rtol=1e-6)
    x = f32(RNG.normal(0, 3, size=(5, 40)))
    y = f32(sps.softmax(x.astype(np.float64), axis=1))
    dy = f32(RNG.normal(0, 1, size=(5, 40)))
    dx = oracle.softmax_bwd(y, dy)
    # rows of a Jacobian-vector product of the softmax sum to (almost) zero
    np.testing.assert_allclose(dx.sum(1), 0.0, atol=1e-6)
    # a constant upstream gradient has no effect
    dx = oracle.softmax_bwd(y, f32(np.full((5, 40), 2.5)))
    np.testing.assert_allclose(dx, 0.0, atol=2e-6)
    # a fully masked row (softmax output 0) has a zero gradient
    dx = oracle.softmax_bwd(f32(np.zeros((1, 7))), f32(RNG.normal(0, 1, (1, 7))))
    assert (dx == 0).all()


def test_softmax_bwd_central_differences():
    h = 2.0 ** -12
    x = dyadic((2, 6), scale=2.0)
    dy = dyadic((2, 6))
    dyd = dy.astype(np.float64)

    def L(x_):
        return float((oracle.softmax(x_) * dyd).sum())

    dx = oracle.softmax_bwd(f32(oracle.softmax(x)), dy)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        assert (L(xp) - L(xm)) / (2 * h) == pytest.approx(dx[idx], abs=2e-6)


# ------------------------------------------------------------ log-softmax

@pytest.mark.parametrize("shape", [(1, 1), (3, 7), (5, 64), (2, 50304)])
def test_log_softmax_matches_scipy(shape):
    x = f32(RNG.normal(0, 4, size=shape))
    np.testing.assert_allclose(oracle.log_softmax(x), sps.log_softmax(x.astype(np.float64), 1),
                               rtol=1e-13, atol=1e-13)


def test_log_softmax_closed_forms_and_special_rows():
    z = oracle.log_softmax(f32([[1.0, 2.0, 3.0]]))
    np.testing.assert_allclose(z[0], [-2.4076059644, -1.4076059644, -0.4076059644], rtol=0,
                               atol=5e-11)
    # exp(z) is the softmax: sums to one; shift invariance on a dyadic grid
    x = dyadic((4, 30), scale=3.0)
    z = oracle.log_softmax(x)
    np.testing.assert_allclose(np.exp(z).sum(1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(oracle.log_softmax(f32(x + 64.0)), z, rtol=1e-12, atol=1e-12)
    # one column: 0; masked row: 0; a -inf entry in a live row: -inf
    assert (oracle.log_softmax(f32([[5.0], [-3.0]])) == 0).all()
    z = oracle.log_softmax(f32([[-np.inf, -np.inf], [0.0, -np.inf]]))
    assert (z[0] == 0).all() and z[1, 0] == 0.0 and z[1, 1] == -np.inf


@pytest.mark.parametrize("shape", [(1, 1), (3, 5), (4, 97)])
def test_log_softmax_bwd_matches_torch_vjp(shape):
    x = f32(RNG.normal(0, 2, size=shape))
    dz = f32(RNG.normal(0, 1, size=shape))
    xt = t64(x).requires_grad_()
    zt = torch.log_softmax(xt, 1)
    (g,) = torch.autograd.grad(zt, xt, t64(dz))
    dx = oracle.log_softmax_bwd(f32(zt.detach().numpy()), dz)
    np.testing.assert_allclose(dx, g.numpy(), rtol=2e-6, atol=2e-6)


def test_log_softmax_bwd_closed_form_and_invariants():
    z = f32([[-2.4076059644, -1.4076059644, -0.4076059644]])
    dx = oracle.log_softmax_bwd(z, f32([[1.0, 0.0, 0.0]]))
    np.testing.assert_allclose(dx[0], [1 - 0.0900305732, -0.2447284711, -0.6652409558], rtol=1e-6)
    x = f32(RNG.normal(0, 3, size=(6, 33)))
    z = f32(oracle.log_softmax(x))
    dz = f32(RNG.normal(0, 1, size=(6, 33)))
    np.testing.assert_allclose(oracle.log_softmax_bwd(z, dz).sum(1), 0.0, atol=5e-6)


def test_log_softmax_bwd_central_differences():
    h = 2.0 ** -12
    x = dyadic((2, 6), scale=2.0)
    dz = dyadic((2, 6))
    dzd = dz.astype(np.float64)

    def L(x_):
        return float((oracle.log_softmax(x_) * dzd).sum())

    dx = oracle.log_softmax_bwd(f32(oracle.log_softmax(x)), dz)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        assert (L(xp) - L(xm)) / (2 * h) == pytest.approx(dx[idx], abs=5e-6)


# ---------------------------------------------------------------- RMSNorm

def _torch_rms(x, g, eps):
    xt = t64(x).requires_grad_()
    gt = t64(g).requires_grad_()
    y = torch.nn.functional.rms_norm(xt, (x.shape[1],), gt, eps)
    return xt, gt, y


@pytest.mark.parametrize("shape", [(1, 1), (4, 3), (7, 33), (5, 768)])
def test_rms_fwd_matches_torch(shape):
    x = f32(RNG.normal(0, 1, size=shape) + RNG.uniform(-3, 3, size=(shape[0], 1)))
    g = f32(RNG.normal(1, 0.1, size=shape[1]))
    y, rstd = oracle.rms_fwd(x, g, 1e-5)
    _, _, yt = _torch_rms(x, g, 1e-5)
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-13)
    xd = x.astype(np.float64)
    np.testing.assert_allclose(rstd, 1 / np.sqrt((xd ** 2).mean(1) + 1e-5), rtol=1e-13)


def test_rms_fwd_closed_forms_and_special_rows():
    # x = [1, 2, 3], gamma = 1, eps = 0: mean square 14/3, rstd = sqrt(3/14)
    y, rstd = oracle.rms_fwd(f32([[1.0, 2.0, 3.0]]), f32([1, 1, 1]), 0.0)
    assert rstd[0] == pytest.approx(0.4629100498862757, rel=1e-15)
    np.testing.assert_allclose(y[0], [0.4629100498862757, 0.9258200997725514, 1.3887301496588271],
                               rtol=1e-15)
    # scale invariance (eps = 0, scale a power of two) and unit mean square
    x = dyadic((3, 20), scale=2.0)
    g = f32(np.ones(20))
    y1, _ = oracle.rms_fwd(x, g, 0.0)
    y2, _ = oracle.rms_fwd(f32(x * 8.0), g, 0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-14)
    np.testing.assert_allclose((y1 ** 2).mean(1), 1.0, rtol=1e-13)
    # one column: y = sign(x) * gamma up to eps
    y, _ = oracle.rms_fwd(f32([[3.0], [-0.5]]), f32([2.0]), 0.0)
    np.testing.assert_allclose(y[:, 0], [2.0, -2.0], rtol=1e-15)
    # masked row
    y, rstd = oracle.rms_fwd(f32([[1, np.inf, 2], [1, 2, 2]]), f32([1, 1, 1]), 1e-5)
    assert (y[0] == 0).all() and rstd[0] == 0 and rstd[1] > 0


@pytest.mark.parametrize("shape", [(1, 1), (3, 4), (6, 33), (4, 768)])
def test_rms_bwd_matches_torch_autograd(shape):
    x = f32(RNG.normal(0, 1, size=shape))
    g = f32(RNG.normal(1, 0.1, size=shape[1]))
    dy = f32(RNG.normal(0, 1, size=shape))
    _, rstd = oracle.rms_fwd(x, g, 1e-5)
    dx, dg, dga = oracle.rms_bwd(dy, x, rstd, g)
    xt, gt, y = _torch_rms(x, g, 1e-5)
    (y * t64(dy)).sum().backward()
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert (dga >= np.abs(dg) - 1e-12).all()


def test_rms_bwd_invariants_and_special_rows():
    # eps = 0: the output is invariant to scaling x, so dx is orthogonal to x
    x = f32(RNG.normal(0, 1, size=(4, 25)))
    g = f32(RNG.normal(1, 0.2, size=25))
    dy = f32(RNG.normal(0, 1, size=(4, 25)))
    _, rstd = oracle.rms_fwd(x, g, 0.0)
    dx, _, _ = oracle.rms_bwd(dy, x, rstd, g)
    np.testing.assert_allclose((dx * x.astype(np.float64)).sum(1), 0.0, atol=1e-12)
    # masked row: dx = 0, no contribution to dgamma
    x = f32([[1, 2, 2], [1, np.nan, 3]])
    _, rstd = oracle.rms_fwd(x, f32([1, 1, 1]), 1e-5)
    dx, dg, _ = oracle.rms_bwd(f32([[1, 0, 0], [5, 5, 5]]), x, rstd, f32([1, 1, 1]))
    assert (dx[1] == 0).all()
    np.testing.assert_allclose(dg, [1 * rstd[0], 0, 0], rtol=1e-15)


def test_rms_bwd_central_differences():
    h = 2.0 ** -10
    eps = 1e-5
    x = dyadic((2, 5))
    g = dyadic((5,), scale=0.5) + f32(1.0)
    dy = dyadic((2, 5))
    dyd = dy.astype(np.float64)

    def L(x_, g_):
        y, _ = oracle.rms_fwd(x_, g_, eps)
        return float((y * dyd).sum())

    _, rstd = oracle.rms_fwd(x, g, eps)
    dx, dg, _ = oracle.rms_bwd(dy, x, rstd, g)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        assert (L(xp, g) - L(xm, g)) / (2 * h) == pytest.approx(dx[idx], abs=2e-5)
    for j in range(5):
        gp, gm = g.copy(), g.copy()
        gp[j] += h
        gm[j] -= h
        assert (L(x, gp) - L(x, gm)) / (2 * h) == pytest.approx(dg[j], abs=1e-6)


def test_brute_force_tiny_against_torch():
    for _ in range(30):
        R, C = int(RNG.integers(1, 5)), int(RNG.integers(1, 8))
        x = f32(RNG.normal(0, 2, size=(R, C)))
        d = f32(RNG.normal(0, 1, size=(R, C)))
        xt = t64(x).requires_grad_()
        zt = torch.log_softmax(xt, 1)
        np.testing.assert_allclose(oracle.log_softmax(x), zt.detach().numpy(), rtol=1e-12,
                                   atol=1e-13)
        (gz,) = torch.autograd.grad(zt, xt, t64(d))
        np.testing.assert_allclose(oracle.log_softmax_bwd(f32(zt.detach().numpy()), d), gz.numpy(),
                                   rtol=1e-5, atol=1e-5)
        g = f32(RNG.normal(1, .2, C))
        y, rstd = oracle.rms_fwd(x, g, 1e-5)
        xt, gt, yt = _torch_rms(x, g, 1e-5)
        np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-13)
        (yt * t64(d)).sum().backward()
        dx, dg, _ = oracle.rms_bwd(d, x, rstd, g)
        np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-8, atol=1e-10)
        np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-9, atol=1e-11)
        assert math.isfinite(float(dx.sum()))
