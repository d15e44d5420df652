"""Pins of the oracle's attention (scaled dot-product, causal or not) against
what the definition fixes, not against a retyping of it: the first causal row
sees only its own key; equal scores give running means and lse = log(count);
a dominant key selects its value; softmax invariances (a common shift of the
keys moves only lse; jointly permuting keys and values changes nothing when
all keys are visible); linearity in V; a hand-worked two-key case."""
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


def test_first_causal_row_is_its_own_value():
    q, k, v = rnd((2, 9, 8), 1), rnd((2, 9, 8), 2), rnd((2, 9, 8), 3)
    o, lse = oracle.attention(q, k, v, 0.3)
    np.testing.assert_array_equal(o[:, 0], v[:, 0].astype(np.float64))
    np.testing.assert_allclose(lse[:, 0], 0.3 * np.einsum("bc,bc->b", q[:, 0].astype(np.float64),
                                                          k[:, 0].astype(np.float64)),
                               rtol=1e-15, atol=1e-15)


def test_equal_scores_give_running_means():
    q = np.zeros((1, 7, 4), np.float32)           # every score 0
    k, v = rnd((1, 7, 4), 4), rnd((1, 7, 4), 5)
    o, lse = oracle.attention(q, k, v, 1.0)
    for i in range(7):
        np.testing.assert_allclose(o[0, i], v[0, :i + 1].astype(np.float64).mean(axis=0),
                                   rtol=1e-13, atol=1e-14)
        assert lse[0, i] == pytest.approx(math.log(i + 1), abs=1e-14)
    on, lsen = oracle.attention(q, k, v, 1.0, causal=False)
    np.testing.assert_allclose(on[0], np.broadcast_to(v[0].astype(np.float64).mean(axis=0), (7, 4)),
                               rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lsen[0], math.log(7), rtol=1e-15)


def test_dominant_key_selects_its_value():
    # k_j = (j + 1) * e: for a query along +e the largest visible key is the
    # last one (j = i causal, j = s - 1 otherwise); with Q and K swapped every
    # row would see equal scores instead
    s, d = 6, 4
    e = np.zeros(d, np.float32)
    e[1] = 1.0
    k = np.stack([(j + 1) * e for j in range(s)])[None]
    q = np.stack([40.0 * e for _ in range(s)])[None].astype(np.float32)
    v = rnd((1, s, d), 6)
    o, _ = oracle.attention(q, k.astype(np.float32), v, 1.0)
    np.testing.assert_allclose(o[0], v[0].astype(np.float64), rtol=0, atol=1e-12)
    on, _ = oracle.attention(q, k.astype(np.float32), v, 1.0, causal=False)
    np.testing.assert_allclose(on[0], np.broadcast_to(v[0, -1].astype(np.float64), (s, d)),
                               rtol=0, atol=1e-12)


def test_shifting_every_key_moves_only_lse():
    q, v = rnd((1, 8, 8), 7), rnd((1, 8, 8), 9)
    k = (np.round(rnd((1, 8, 8), 8) * 16) / 16).astype(np.float32)  # k + u exact in float32
    u = np.float32(0.25) * np.ones(8, np.float32)
    o1, l1 = oracle.attention(q, k, v, 0.5)
    o2, l2 = oracle.attention(q, k + u, v, 0.5)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    shift = 0.5 * (q[0].astype(np.float64) @ u.astype(np.float64))
    np.testing.assert_allclose(l2[0] - l1[0], shift, rtol=1e-10, atol=1e-12)


def test_joint_permutation_of_keys_and_values():
    q, k, v = rnd((1, 10, 4), 10), rnd((1, 10, 4), 11), rnd((1, 10, 4), 12)
    perm = np.random.default_rng(13).permutation(10)
    o1, l1 = oracle.attention(q, k, v, 0.7, causal=False)
    o2, l2 = oracle.attention(q, k[:, perm], v[:, perm], 0.7, causal=False)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=1e-13)


def test_linear_in_values():
    q, k = rnd((1, 8, 4), 14), rnd((1, 8, 4), 15)
    v1, v2 = rnd((1, 8, 4), 16), rnd((1, 8, 4), 17)
    o1, _ = oracle.attention(q, k, v1, 0.4)
    o2, _ = oracle.attention(q, k, v2, 0.4)
    o12, _ = oracle.attention(q, k, (v1.astype(np.float64) + v2).astype(np.float32), 0.4)
    # v1 + v2 rounded to float32 once: the difference is that rounding, carried linearly
    r = (v1.astype(np.float64) + v2) - (v1.astype(np.float64) + v2).astype(np.float32)
    o_r, _ = oracle.attention(q, k, r.astype(np.float32), 0.4) if np.any(r) else (0.0, None)
    np.testing.assert_allclose(o12, o1 + o2 - o_r, rtol=1e-6, atol=1e-6)


def test_two_keys_by_hand():
    # one head, d = 1: q = (1, 2), k = (0, 1), v = (3, 5), scale 1, causal.
    # row 0: only key 0 -> o = 3, lse = 0.
    # row 1: scores (0, 2): p = (1, e^2) / (1 + e^2); o = (3 + 5 e^2) / (1 + e^2);
    #        lse = log(1 + e^2).
    q = np.array([[[1.0], [2.0]]], np.float32)
    k = np.array([[[0.0], [1.0]]], np.float32)
    v = np.array([[[3.0], [5.0]]], np.float32)
    o, lse = oracle.attention(q, k, v, 1.0)
    e2 = math.exp(2.0)
    assert o[0, 0, 0] == 3.0 and lse[0, 0] == 0.0
    assert o[0, 1, 0] == pytest.approx((3 + 5 * e2) / (1 + e2), rel=1e-15)
    assert lse[0, 1] == pytest.approx(math.log1p(e2), rel=1e-15)


def test_causal_last_row_equals_full_attention_last_row():
    q, k, v = rnd((2, 12, 8), 18), rnd((2, 12, 8), 19), rnd((2, 12, 8), 20)
    oc, lc = oracle.attention(q, k, v, 0.35)
    of, lf = oracle.attention(q, k, v, 0.35, causal=False)
    np.testing.assert_allclose(oc[:, -1], of[:, -1], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lc[:, -1], lf[:, -1], rtol=1e-14)
