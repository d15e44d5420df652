"""Pins for the float64 oracle, checked against things other than itself:
library routines (scipy, torch CPU float64 autograd), closed forms, invariants,
central finite differences (the gradient check of the "NexusGrad" README,
sec. "Testing"), and brute force on tiny inputs.  No GPU needed."""
import math

import numpy as np
import pytest
import scipy.special as sps
import torch

import oracle
from row_reduction_pass_gb300 import synth

RNG = np.random.default_rng(12345)


def f32(a):
    return np.ascontiguousarray(a, np.float32)


def dyadic(shape, scale=4.0, step=2.0 ** -8):
    """Random values on a 2^-8 grid, so x +- 2^-10 is exact in float32."""
    return f32(np.round(RNG.normal(0, scale, size=shape) / step) * step)


# ---------------------------------------------------------------- softmax ----

@pytest.mark.parametrize("shape", [(1, 1), (3, 7), (5, 64), (4, 1000)])
def test_softmax_matches_scipy(shape):
    x = f32(RNG.normal(0, 3, size=shape))
    y = oracle.softmax(x)
    ref = sps.softmax(x.astype(np.float64), axis=1)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(y.sum(1), 1.0, rtol=1e-13)


def test_softmax_bf16_reads_exact_bits():
    x = f32(RNG.normal(0, 3, size=(6, 33)))
    bits = synth.bf16_bits(x)
    wide = synth.bf16_to_f32(bits).astype(np.float64)
    np.testing.assert_allclose(oracle.softmax(bits), sps.softmax(wide, axis=1), rtol=1e-13)


def test_softmax_shift_invariance_and_special_cases():
    x = dyadic((4, 9), scale=2.0)
    np.testing.assert_allclose(oracle.softmax(x), oracle.softmax(f32(x + 8.0)), rtol=1e-12)
    assert oracle.softmax(f32([[3.5]]))[0, 0] == 1.0
    assert oracle.softmax(f32([[-np.inf]]))[0, 0] == 0.0
    # two elements reduce to the logistic function
    t = 1.75
    y = oracle.softmax(f32([[0.0, t]]))
    assert y[0, 1] == pytest.approx(sps.expit(t), rel=1e-14)
    # fully masked row -> zeros, and a masked row does not disturb its neighbours
    m = f32([[1, 2, 3], [-np.inf] * 3, [0, 0, 0]])
    y = oracle.softmax(m)
    assert (y[1] == 0).all()
    np.testing.assert_allclose(y[2], [1 / 3] * 3, rtol=1e-15)


def test_softmax_causal_row_support():
    x = synth.causal_scores(1, 2, 16, 16, "f32", 4.0, 7)
    y = oracle.softmax(x)
    for r in range(x.shape[0]):
        q = r % 16
        assert (y[r, :q + 1] > 0).all() and (y[r, q + 1:] == 0).all()
    assert (y[::16, 0] == 1.0).all()


def test_online_normaliser_reaches_three_pass():
    """Milakov-Gimelshein online (m, d) equals (max, sum exp(x - max))."""
    for n in (1, 2, 17, 1000):
        x = RNG.normal(0, 5, size=n)
        m, d = oracle.online_softmax_stats(x)
        assert m == x.max()
        assert m + math.log(d) == pytest.approx(sps.logsumexp(x), rel=1e-14, abs=1e-14)
    # merge of two halves equals the whole, including an all -inf half
    x = RNG.normal(0, 5, size=101)
    ma, da = oracle.online_softmax_stats(x[:40])
    mb, db = oracle.online_softmax_stats(x[40:])
    m, d = oracle.online_merge(ma, da, mb, db)
    assert m + math.log(d) == pytest.approx(sps.logsumexp(x), rel=1e-14)
    m2, d2 = oracle.online_merge(ma, da, -math.inf, 0.0)
    assert (m2, d2) == (ma, pytest.approx(da, rel=1e-15))
    m3, d3 = oracle.online_softmax_stats(np.array([-np.inf, -np.inf]))
    assert m3 == -math.inf and d3 == 0.0


# ------------------------------------------------------------- cross-entropy --

def test_xent_matches_logsumexp_and_softmax_minus_onehot():
    x = f32(RNG.normal(0, 2, size=(16, 50)))
    lab = RNG.integers(0, 50, size=16).astype(np.int32)
    loss, dl, bad = oracle.xent(x, lab)
    xd = x.astype(np.float64)
    ref_loss = sps.logsumexp(xd, axis=1) - xd[np.arange(16), lab]
    np.testing.assert_allclose(loss, ref_loss, rtol=1e-13)
    ref_dl = sps.softmax(xd, axis=1)
    ref_dl[np.arange(16), lab] -= 1.0
    np.testing.assert_allclose(dl, ref_dl, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dl.sum(1), 0.0, atol=1e-14)
    assert bad == 0


def test_xent_matches_torch_cross_entropy():
    x = f32(RNG.normal(0, 3, size=(8, 33)))
    lab = RNG.integers(0, 33, size=8).astype(np.int32)
    lab[3] = -100
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    lt = torch.nn.functional.cross_entropy(xt, torch.tensor(lab, dtype=torch.int64),
                                           reduction="none", ignore_index=-100)
    lt.sum().backward()
    loss, dl, _ = oracle.xent(x, lab)
    np.testing.assert_allclose(loss, lt.detach().numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dl, xt.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_xent_gradient_by_central_differences():
    h = 2.0 ** -10
    x = dyadic((3, 7), scale=1.5)
    lab = np.array([0, 3, 6], np.int32)
    _, dl, _ = oracle.xent(x, lab)
    for r in range(3):
        for j in range(7):
            xp, xm = x.copy(), x.copy()
            xp[r, j] += h
            xm[r, j] -= h
            fp = oracle.xent(xp, lab, want_dlogits=False)[0][r]
            fm = oracle.xent(xm, lab, want_dlogits=False)[0][r]
            assert (fp - fm) / (2 * h) == pytest.approx(dl[r, j], abs=2e-6)


def test_xent_shift_invariance_and_special_rows():
    x = dyadic((3, 6), scale=2.0)
    lab = np.array([1, 5, 0], np.int32)
    l1, d1, _ = oracle.xent(x, lab)
    l2, d2, _ = oracle.xent(f32(x - 16.0), lab)
    np.testing.assert_allclose(l1, l2, rtol=1e-12)
    np.testing.assert_allclose(d1, d2, rtol=1e-11, atol=1e-15)
    # ignored row, fully masked row, out-of-range label
    x2 = f32([[1, 2, 3], [-np.inf] * 3, [1, 2, 3], [1, 2, 3]])
    lab2 = np.array([-100, 0, 7, -1], np.int32)
    loss, dl, bad = oracle.xent(x2, lab2)
    assert loss[0] == 0 and (dl[0] == 0).all()
    assert loss[1] == 0 and (dl[1] == 0).all()
    assert math.isnan(loss[2]) and math.isnan(loss[3]) and bad == 2
    np.testing.assert_allclose(dl[2], sps.softmax([1.0, 2.0, 3.0]), rtol=1e-15)
    # a single class: loss 0, gradient 0
    l1c, d1c, _ = oracle.xent(f32([[4.0]]), np.array([0], np.int32))
    assert l1c[0] == 0.0 and d1c[0, 0] == 0.0


# ----------------------------------------------------------------- LayerNorm --

def _torch_ln(x, g, b, eps):
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    gt = torch.tensor(g, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True)
    y = torch.nn.functional.layer_norm(xt, (x.shape[1],), gt, bt, eps)
    return xt, gt, bt, y


@pytest.mark.parametrize("shape", [(1, 1), (4, 3), (7, 33), (5, 768)])
def test_ln_fwd_matches_torch(shape):
    x = f32(RNG.normal(0, 1, size=shape) + RNG.uniform(-10, 10, size=(shape[0], 1)))
    g = f32(RNG.normal(1, 0.1, size=shape[1]))
    b = f32(RNG.normal(0, 0.1, size=shape[1]))
    y, mean, rstd = oracle.ln_fwd(x, g, b, 1e-5)
    _, _, _, yt = _torch_ln(x, g, b, 1e-5)
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-10, atol=1e-12)
    xd = x.astype(np.float64)
    np.testing.assert_allclose(mean, xd.mean(1), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(xd.var(1) + 1e-5), rtol=1e-12)


def test_ln_fwd_closed_forms():
    # one column: y = beta, rstd = eps^-1/2
    y, mean, rstd = oracle.ln_fwd(f32([[3.0], [-7.5]]), f32([2.0]), f32([0.25]), 1e-5)
    assert (y == 0.25).all() and rstd == pytest.approx([1e-5 ** -0.5] * 2, rel=1e-15)
    # shift invariance on a dyadic grid (shift exact in float32)
    x = dyadic((3, 10), scale=1.0)
    g = f32(RNG.normal(1, 0.1, 10))
    b = f32(RNG.normal(0, 0.1, 10))
    y1, _, r1 = oracle.ln_fwd(x, g, b, 1e-5)
    y2, _, r2 = oracle.ln_fwd(f32(x + 32.0), g, b, 1e-5)
    np.testing.assert_allclose(y1, y2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r1, r2, rtol=1e-13)
    # normalised values have zero mean and (almost) unit variance
    y, _, _ = oracle.ln_fwd(x, f32(np.ones(10)), f32(np.zeros(10)), 0.0)
    np.testing.assert_allclose(y.mean(1), 0.0, atol=1e-14)
    np.testing.assert_allclose((y ** 2).mean(1), 1.0, rtol=1e-13)
    # masked row
    y, mean, rstd = oracle.ln_fwd(f32([[1, 2, -np.inf], [1, 2, 3]]), f32([1, 1, 1]),
                                  f32([0, 0, 0]), 1e-5)
    assert (y[0] == 0).all() and mean[0] == 0 and rstd[0] == 0
    assert mean[1] == 2.0


def test_welford_and_chan_reach_two_pass_moments():
    for n in (1, 2, 3, 768, 5000):
        x = RNG.normal(0, 1, size=n) + RNG.uniform(-10, 10)
        mean, m2 = oracle.welford(x)
        assert mean == pytest.approx(x.mean(), rel=1e-12, abs=1e-12)
        assert m2 == pytest.approx(((x - x.mean()) ** 2).sum(), rel=1e-10, abs=1e-12)
    x = RNG.normal(3, 2, size=257)
    a, b = x[:100], x[100:]
    ma, m2a = oracle.welford(a)
    mb, m2b = oracle.welford(b)
    n, mean, m2 = oracle.chan_merge(100, ma, m2a, 157, mb, m2b)
    assert n == 257 and mean == pytest.approx(x.mean(), rel=1e-13)
    assert m2 == pytest.approx(np.var(x) * 257, rel=1e-12)
    # merging with an empty side is the identity
    assert oracle.chan_merge(0, 0.0, 0.0, 100, ma, m2a) == (100, pytest.approx(ma, rel=1e-15),
                                                            pytest.approx(m2a, rel=1e-15))


@pytest.mark.parametrize("shape", [(1, 1), (3, 4), (6, 33), (4, 768)])
def test_ln_bwd_matches_torch_autograd(shape):
    x = f32(RNG.normal(0, 1, size=shape) + RNG.uniform(-5, 5, size=(shape[0], 1)))
    g = f32(RNG.normal(1, 0.1, size=shape[1]))
    b = f32(RNG.normal(0, 0.1, size=shape[1]))
    dy = f32(RNG.normal(0, 1, size=shape))
    _, mean, rstd = oracle.ln_fwd(x, g, b, 1e-5)
    dx, dg, db, dga, dba = oracle.ln_bwd(dy, x, mean, rstd, g)
    xt, gt, bt, y = _torch_ln(x, g, b, 1e-5)
    (y * torch.tensor(dy, dtype=torch.float64)).sum().backward()
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(db, bt.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert (dga >= np.abs(dg) - 1e-12).all() and (dba >= np.abs(db) - 1e-12).all()
    np.testing.assert_allclose(dx.sum(1), 0.0, atol=1e-11)


def test_ln_bwd_central_differences():
    """d/dx, d/dgamma, d/dbeta of L = sum(y * dy) by central differences."""
    h = 2.0 ** -10
    eps = 1e-5
    x = dyadic((2, 5), scale=1.0)
    g = dyadic((5,), scale=0.5) + f32(1.0)
    b = dyadic((5,), scale=0.5)
    dy = dyadic((2, 5), scale=1.0)
    dyd = dy.astype(np.float64)

    def L(x_, g_, b_):
        y, _, _ = oracle.ln_fwd(x_, g_, b_, eps)
        return float((y * dyd).sum())

    _, mean, rstd = oracle.ln_fwd(x, g, b, eps)
    dx, dg, db, _, _ = oracle.ln_bwd(dy, x, mean, rstd, g)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        assert (L(xp, g, b) - L(xm, g, b)) / (2 * h) == pytest.approx(dx[idx], abs=2e-5)
    for j in range(5):
        gp, gm = g.copy(), g.copy()
        gp[j] += h
        gm[j] -= h
        assert (L(x, gp, b) - L(x, gm, b)) / (2 * h) == pytest.approx(dg[j], abs=1e-6)
        bp, bm = b.copy(), b.copy()
        bp[j] += h
        bm[j] -= h
        assert (L(x, g, bp) - L(x, g, bm)) / (2 * h) == pytest.approx(db[j], abs=1e-6)


def test_ln_bwd_special_rows():
    # one column: dx = 0; masked row: dx = 0 and no contribution to dgamma / dbeta
    dx, dg, db, _, _ = oracle.ln_bwd(f32([[1.5]]), f32([[2.0]]), [2.0], [316.0], f32([1.0]))
    assert dx[0, 0] == 0.0 and db[0] == 1.5
    x = f32([[1, 2, 3], [4, -np.inf, 5]])
    dy = f32([[1, 0, 0], [9, 9, 9]])
    _, mean, rstd = oracle.ln_fwd(x, f32([1, 1, 1]), f32([0, 0, 0]), 0.0)
    dx, dg, db, _, _ = oracle.ln_bwd(dy, x, mean, rstd, f32([1, 1, 1]))
    assert (dx[1] == 0).all()
    np.testing.assert_allclose(db, [1, 0, 0])
    np.testing.assert_allclose(dg, [-math.sqrt(1.5), 0, 0], rtol=1e-15)
    np.testing.assert_allclose(dx[0], [1 / (2 * math.sqrt(6)) * 1.0, -1 / math.sqrt(6),
                                       1 / (2 * math.sqrt(6))], rtol=1e-14)


def test_brute_force_tiny_against_torch():
    """Every op on random tiny shapes (R <= 4, C <= 7) against torch float64."""
    for _ in range(40):
        R, C = int(RNG.integers(1, 5)), int(RNG.integers(1, 8))
        x = f32(RNG.normal(0, 2, size=(R, C)))
        np.testing.assert_allclose(oracle.softmax(x), torch.softmax(
            torch.tensor(x, dtype=torch.float64), 1).numpy(), rtol=1e-13)
        lab = RNG.integers(0, C, size=R).astype(np.int32)
        loss, dl, _ = oracle.xent(x, lab)
        xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
        lt = torch.nn.functional.cross_entropy(xt, torch.tensor(lab, dtype=torch.int64),
                                               reduction="none")
        lt.sum().backward()
        np.testing.assert_allclose(loss, lt.detach().numpy(), rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(dl, xt.grad.numpy(), rtol=1e-12, atol=1e-15)
        g, b = f32(RNG.normal(1, .2, C)), f32(RNG.normal(0, .2, C))
        dy = f32(RNG.normal(0, 1, size=(R, C)))
        y, mean, rstd = oracle.ln_fwd(x, g, b, 1e-5)
        dx, dg, db, _, _ = oracle.ln_bwd(dy, x, mean, rstd, g)
        xt, gt, bt, yt = _torch_ln(x, g, b, 1e-5)
        (yt * torch.tensor(dy, dtype=torch.float64)).sum().backward()
        np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-8, atol=1e-10)
        np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(db, bt.grad.numpy(), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- rows of one column ----

def test_one_column_closed_forms():
    """A one-element row is its own maximum, sum and moments: softmax 1,
    log-softmax 0, cross-entropy loss 0 and dlogits 0 at the label (1 for a
    label out of range, whose loss is NaN), a -inf or NaN row masked to 0, +inf
    giving NaN; LayerNorm mean = x, rstd = 1 / sqrt(eps), y = beta; RMSNorm
    rstd = 1 / sqrt(x^2 + eps); the backward's dx = rstd (g - g - xhat g xhat)
    = 0 for LayerNorm.  These are the values the elementwise kernels write."""
    x = f32([[2.5], [-7.0], [0.0], [1e8], [-np.inf], [np.nan], [np.inf]])
    live = slice(0, 4)
    y = oracle.softmax(x)
    z = oracle.log_softmax(x)
    assert np.all(y[live] == 1.0) and np.all(z[live] == 0.0)
    assert np.all(y[4:6] == 0.0) and np.all(z[4:6] == 0.0)
    assert np.isnan(y[6, 0]) and np.isnan(z[6, 0])
    lab = np.array([0, 0, 3, -100, 0, 0, 0], np.int32)
    loss, dl, bad = oracle.xent(x, lab)
    assert loss[0] == 0.0 and loss[1] == 0.0 and dl[0, 0] == 0.0 and dl[1, 0] == 0.0
    assert np.isnan(loss[2]) and dl[2, 0] == 1.0 and bad == 1
    assert loss[3] == 0.0 and dl[3, 0] == 0.0          # ignored
    assert loss[4] == 0.0 and loss[5] == 0.0           # masked rows
    assert np.isnan(loss[6]) and np.isnan(dl[6, 0])    # +inf
    xs = f32([[2.5], [-7.0], [0.25]])
    g, b = f32([1.5]), f32([-0.25])
    yl, mean, rstd = oracle.ln_fwd(xs, g, b, 1e-5)
    assert np.allclose(mean, xs[:, 0], rtol=0, atol=0)
    assert np.allclose(rstd, 1.0 / math.sqrt(1e-5), rtol=1e-12)
    assert np.allclose(yl, -0.25, rtol=0, atol=1e-12)
    yr, rr_ = oracle.rms_fwd(xs, g, 1e-5)
    assert np.allclose(rr_, 1.0 / np.sqrt(xs[:, 0].astype(np.float64) ** 2 + 1e-5), rtol=1e-12)
    assert np.allclose(yr[:, 0], xs[:, 0] * rr_ * 1.5, rtol=1e-12)
    dy = f32([[0.5], [-1.0], [2.0]])
    dx, dg, db, _, _ = oracle.ln_bwd(dy, xs, mean, rstd, g)
    assert np.allclose(dx, 0.0, atol=1e-12)
    assert np.allclose(db, dy.sum(), rtol=1e-12) and np.allclose(dg, 0.0, atol=1e-12)
