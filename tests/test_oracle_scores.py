"""Pins of the oracle's scoring (Eqs. (1)-(5) of the Nexus Sampling paper) to facts
that hold independently of its code: invariants, closed forms and special cases."""
import math

import numpy as np
import pytest


def _rand(T=40, d=16, W=8, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((T, d)) * scale, rng.standard_normal((W, d)) * scale


def test_rows_are_distributions_and_a_sums_to_one(oracle_lib):
    # Eq. (1): every softmax row is a distribution; Eq. (1)/(3): sum_j a_j = 1.
    K, Q = _rand(T=300, d=32, W=16, seed=1, scale=2.0)
    o = oracle_lib.slice_scores(K, Q, walk_len=3)
    assert np.allclose(o["P"].sum(1), 1.0, atol=1e-12)
    assert (o["P"] >= 0).all()
    assert abs(o["a"].sum() - 1.0) < 1e-12
    assert np.allclose(o["a"], o["P"].mean(0), atol=1e-15)


def test_two_key_closed_form_checks_sqrt_d_scale(oracle_lib):
    # one query (2,0,0,0), keys e1 and 0 in d = 4: logits 2/sqrt(4) = 1 and 0, so the
    # softmax row is the logistic pair (e/(e+1), 1/(e+1)).
    K = np.array([[1.0, 0, 0, 0], [0.0, 0, 0, 0]])
    Q = np.array([[2.0, 0, 0, 0]])
    o = oracle_lib.slice_scores(K, Q, walk_len=0)
    e = math.e
    assert np.allclose(o["a"], [e / (e + 1), 1 / (e + 1)], rtol=0, atol=1e-15)
    assert abs(o["rowmax"][0] - 1.0) < 1e-15
    assert abs(o["rowsum"][0] - (1 + 1 / e)) < 1e-15


def test_single_key_and_identical_keys(oracle_lib):
    K, Q = _rand(T=1, d=8, W=4, seed=2)
    o = oracle_lib.slice_scores(K, Q, walk_len=2)
    assert o["a"][0] == 1.0 and abs(o["w"][0] - 1.5) < 1e-7  # s = 1 + lambda * 1
    row = np.random.default_rng(3).standard_normal(8)
    K = np.tile(row, (50, 1))
    o = oracle_lib.slice_scores(K, Q, walk_len=2)
    assert np.allclose(o["a"], 1 / 50, atol=1e-15)
    assert np.allclose(o["ctilde"], 1 / 50, atol=1e-15)


def test_dominant_key_takes_all_mass(oracle_lib):
    rng = np.random.default_rng(4)
    K = rng.standard_normal((64, 16))
    K[17] = 0.0
    K[17, 0] = 400.0
    Q = np.abs(rng.standard_normal((6, 16))) + 1.0  # positive along feature 0
    o = oracle_lib.slice_scores(K, Q, walk_len=3)
    assert o["a"][17] > 1 - 1e-12
    assert o["ctilde"][17] > 1 - 1e-12


def test_shift_invariance(oracle_lib):
    # adding one vector to every key adds a per-row constant to the logits: P unchanged.
    K, Q = _rand(T=100, d=12, W=6, seed=5)
    shift = np.random.default_rng(6).standard_normal(12) * 3
    o1 = oracle_lib.slice_scores(K, Q, walk_len=3)
    o2 = oracle_lib.slice_scores(K + shift, Q, walk_len=3)
    assert np.allclose(o1["a"], o2["a"], rtol=1e-10, atol=1e-15)
    assert np.allclose(o1["ctilde"], o2["ctilde"], rtol=1e-10, atol=1e-15)


def test_zero_step_walk_reproduces_direct_scores(oracle_lib):
    # H = 0: c~ = 0 (empty walk), so s = a exactly and w = a + eps r.
    K, Q = _rand(T=77, d=8, W=5, seed=7)
    o = oracle_lib.slice_scores(K, Q, walk_len=0, lam=0.5, eps_tie=0.0)
    assert (o["ctilde"] == 0).all()
    assert (o["s"] == o["a"]).all()
    assert (o["w"] == o["a"].astype(np.float32)).all()


def test_one_step_walk_is_the_newest_row(oracle_lib):
    # H = 1: C = 1 * P_{W-1}, so c~ = P_{W-1}.
    K, Q = _rand(T=60, d=8, W=5, seed=8)
    o = oracle_lib.slice_scores(K, Q, walk_len=1)
    assert np.allclose(o["ctilde"], o["P"][-1], atol=1e-15)
    assert o["gamma"][0] == 1.0


def test_two_step_walk_closed_form_and_order(oracle_lib):
    # H = 2 over rows r1 = P_{W-2} (older), r2 = P_{W-1}: gamma = (1, 1 + <r1, r2>),
    # c~ = (r1 + gamma_2 r2) / (1 + gamma_2). Swapping the order would weight r1.
    K, Q = _rand(T=40, d=8, W=4, seed=9, scale=1.5)
    o = oracle_lib.slice_scores(K, Q, walk_len=2)
    r1, r2 = o["P"][-2], o["P"][-1]
    g2 = 1 + r1 @ r2
    assert np.allclose(o["gamma"], [1.0, g2], atol=1e-14)
    assert np.allclose(o["ctilde"], (r1 + g2 * r2) / (1 + g2), atol=1e-15)


def test_equal_walk_rows(oracle_lib):
    # All walk rows equal p: c~ = p, gamma_2 = 1 + |p|^2, gamma_3 = 1 + (1 + gamma_2)|p|^2.
    rng = np.random.default_rng(10)
    K = rng.standard_normal((30, 8))
    q = rng.standard_normal(8)
    Q = np.vstack([rng.standard_normal((2, 8)), np.tile(q, (3, 1))])
    o = oracle_lib.slice_scores(K, Q, walk_len=3)
    p = o["P"][-1]
    n2 = p @ p
    assert np.allclose(o["ctilde"], p, atol=1e-15)
    assert np.allclose(o["gamma"], [1.0, 1 + n2, 1 + (2 + n2) * n2], atol=1e-14)


def test_nexus_score_mass_and_tie_ramp(oracle_lib):
    # Eq. (2): sum s = 1 + lambda; Eq. (5): w - s = eps * j / (T - 1).
    K, Q = _rand(T=200, d=16, W=8, seed=11)
    lam, eps = 0.5, 1e-6
    o = oracle_lib.slice_scores(K, Q, walk_len=3, lam=lam, eps_tie=eps)
    assert abs(o["ctilde"].sum() - 1) < 1e-12
    assert abs(o["s"].sum() - (1 + lam)) < 1e-12
    ramp = eps * np.arange(200) / 199
    assert np.allclose(o["w"], (o["s"] + ramp).astype(np.float32), rtol=0, atol=0)


def test_hub_amplification_sign(oracle_lib):
    # Theorem 1 (sign form): with i.i.d. window rows, a token whose mass co-varies with
    # the rows' alignment (a hub) gets E[c~_j] > E[a_j]; mass sums to 1, so the other
    # tokens lose. Rows: with prob. 1/2 the query points at the hub, else it is zero
    # (a uniform row).
    rng = np.random.default_rng(12)
    T, d, W = 64, 16, 8
    K = rng.standard_normal((T, d))
    hub = 5
    unit = K[hub] / np.linalg.norm(K[hub])
    q_al = 2.0 * unit * math.sqrt(d)
    p_al = oracle_lib.slice_scores(K, q_al[None, :], walk_len=0)["a"]
    a_star = 0.5 * p_al + 0.5 / T              # exact mean row of the i.i.d. law
    # The walk reads only the last 3 rows, so its expectation over the i.i.d. law is
    # the exact average over the 2^3 aligned/uniform patterns of those rows.
    c_mean = np.zeros(T)
    for pattern in range(8):
        aligned = np.array([(pattern >> b) & 1 for b in range(3)], bool)
        Q = np.zeros((W, d))
        Q[W - 3:][aligned] = q_al
        c_mean += oracle_lib.slice_scores(K, Q, walk_len=3)["ctilde"] / 8
    assert c_mean[hub] > a_star[hub] * 1.01
    assert np.delete(c_mean - a_star, hub).sum() < 0
    assert abs(c_mean.sum() - 1) < 1e-12
