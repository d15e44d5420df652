"""The worked 3-element examples in tests/golden/worked_examples.json (written by
tests/golden/make_golden.py from the oracle) pinned by 40-digit closed forms,
and re-derived by the current oracle (regression)."""
import json
import os

import mpmath as mp
import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
mp.mp.dps = 40


@pytest.fixture(scope="module")
def cases():
    with open(GOLDEN) as f:
        return json.load(f)


def close(a, b, rel=1e-14, abs_=1e-15):
    return abs(float(a) - float(b)) <= abs_ + rel * abs(float(b))


def test_softmax_123_closed_form(cases):
    c = cases["softmax_123"]
    z = mp.e ** -2 + mp.e ** -1 + 1          # e^(x - max) summed, max = 3
    want = [mp.e ** -2 / z, mp.e ** -1 / z, 1 / z]
    assert all(close(g, w) for g, w in zip(c["y"][0], want))


@pytest.mark.parametrize("lab", [0, 2])
def test_xent_123_closed_form(cases, lab):
    c = cases[f"xent_123_label{lab}"]
    lse = mp.log(mp.e + mp.e ** 2 + mp.e ** 3)
    assert close(c["loss"][0], lse - (lab + 1))
    p = [mp.e ** k / (mp.e + mp.e ** 2 + mp.e ** 3) for k in (1, 2, 3)]
    p[lab] -= 1
    assert all(close(g, w) for g, w in zip(c["dlogits"][0], p))


@pytest.mark.parametrize("eps", [0.0, 1e-5])
def test_ln_fwd_123_closed_form(cases, eps):
    c = cases[f"ln_fwd_123_eps{eps:g}"]
    var = mp.mpf(2) / 3                      # population variance of 1, 2, 3
    rstd = 1 / mp.sqrt(var + mp.mpf(eps))
    assert c["mean"][0] == 2.0 and close(c["rstd"][0], rstd)
    assert all(close(g, w) for g, w in zip(c["y"][0], [-rstd, 0, rstd]))


def test_ln_bwd_123_closed_form(cases):
    c = cases["ln_bwd_123_dy100"]
    r = mp.sqrt(mp.mpf(3) / 2)               # rstd with eps = 0
    xh = [-r, mp.mpf(0), r]
    g = [1, 0, 0]
    mg = mp.mpf(1) / 3
    mgx = sum(a * b for a, b in zip(g, xh)) / 3
    dx = [r * (g[j] - mg - xh[j] * mgx) for j in range(3)]
    assert all(close(a, b) for a, b in zip(c["dx"][0], dx))
    assert close(c["dgamma"][0], -r) and c["dgamma"][1:] == [0.0, 0.0]
    assert c["dbeta"] == [1.0, 0.0, 0.0]


def test_oracle_reproduces_fixture(cases):
    x = np.array(cases["softmax_123"]["x"], np.float32)
    assert oracle.softmax(x).tolist() == cases["softmax_123"]["y"]
    for lab in (0, 2):
        c = cases[f"xent_123_label{lab}"]
        loss, dl, _ = oracle.xent(x, np.array([lab], np.int32))
        assert loss.tolist() == c["loss"] and dl.tolist() == c["dlogits"]
    c = cases["ln_bwd_123_dy100"]
    dx, dg, db, _, _ = oracle.ln_bwd(np.array(c["dy"], np.float32), x, c["mean"], c["rstd"],
                                     np.ones(3, np.float32))
    assert dx.tolist() == c["dx"] and dg.tolist() == c["dgamma"] and db.tolist() == c["dbeta"]
