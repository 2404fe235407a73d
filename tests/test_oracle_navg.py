"""Pins of the oracle's n-averaged reservoir priority (Nexus Sampling paper, §2.3 Eq. (6),
pi_j = (1/n) sum_i (u_j^(i))^(1/w_j), keep the top K by pi_j; n = 5 in §5.1) and of the
specified binary32 exponential its log-domain form uses.

The oracle orders candidates by ln(n pi_j) = M r + ln(sum_i exp((l_i - M) r)) with
l_i = ln u_i, M = max_i l_i, r = 1/w_j. Fixed here against things its code does not
compute: the fp64 exponential, Eq. (6) evaluated directly in fp64, the n -> infinity limit
(App. 8.2: the deterministic limit orders by w_j/(w_j + 1), i.e. top-K by w), and the
exact law of the kept item for two candidates, from the Beta(w, 1) distribution of
u^(1/w) (P(u^(1/w) <= x) = x^w) by numerical convolution.
"""
import math

import numpy as np
import pytest
from scipy.signal import fftconvolve

SEED = 0x243F6A8885A308D3


def test_exp_spec_within_two_ulp_of_exp(oracle_lib):
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-86.0, 0.0, 200001), -rng.random(200000) * 86.0,
                        -rng.random(100000) * 1e-3, [0.0, -1e-30, -0.5, -0.34657359]])
    x = x.astype(np.float32)
    got = oracle_lib.exp_spec(x).astype(np.float64)
    want = np.exp(x.astype(np.float64))
    ulp = np.spacing(want.astype(np.float32)).astype(np.float64)
    err = np.abs(got - want) / ulp
    assert err.max() <= 2.0, (err.max(), x[err.argmax()])
    assert oracle_lib.exp_spec(np.float32([0.0]))[0] == 1.0
    # below the smallest normal scale the result is flushed to zero
    assert (oracle_lib.exp_spec(np.float32([-88.5, -90.0, -1e4])) == 0).all()
    # monotone over a dense sorted sweep
    xs = np.sort(x)
    ys = oracle_lib.exp_spec(xs)
    assert (np.diff(ys.astype(np.float64)) >= 0).all()


def _draws(oracle_lib, pos, step, head, seq, n):
    """The n uniforms of one candidate: word i % 4 of Philox block i // 4, the block
    index in bits 24..31 of counter word 3."""
    out = []
    for g in range((n + 3) // 4):
        words = oracle_lib.philox4x32_10([pos, step, head, (seq & 0xFFFFFF) | (g << 24)],
                                         [SEED & 0xFFFFFFFF, SEED >> 32])
        out += [oracle_lib.uniform(int(wd)) for wd in words]
    return np.array(out[:n], np.float64)


@pytest.mark.parametrize("n", [2, 3, 5, 8, 13])
def test_log_domain_key_equals_eq6_in_double(oracle_lib, n):
    # where (u)^(1/w) does not underflow, ln(n pi) computed directly from Eq. (6) in fp64
    # matches the oracle's binary32 log-domain key to a few binary32 ulps
    rng = np.random.default_rng(n)
    for trial in range(300):
        w = float(np.float32(rng.uniform(0.05, 4.0)))
        pos, step, head, seq = int(rng.integers(0, 1 << 30)), trial, 9, 4
        u = _draws(oracle_lib, pos, step, head, seq, n)
        direct = math.log(np.sum(u ** (1.0 / w)))            # ln(n * pi_j)
        key = oracle_lib.reservoir_key(w, pos, SEED, step, head, seq, n_avg=n)
        assert abs(key - direct) <= 1e-5 * max(1.0, abs(direct)), (w, key, direct)


def test_one_draw_is_the_efraimidis_spirakis_key(oracle_lib):
    rng = np.random.default_rng(1)
    for _ in range(200):
        w = float(np.float32(rng.uniform(1e-6, 1.0)))
        pos = int(rng.integers(0, 1 << 30))
        u = _draws(oracle_lib, pos, 3, 7, 2, 1)[0]
        k1 = oracle_lib.reservoir_key(w, pos, SEED, 3, 7, 2, n_avg=1)
        assert k1 == np.float32(oracle_lib.ln_spec(np.float32([u]))[0] / np.float32(w))


def test_zero_weight_gives_minus_infinity(oracle_lib):
    for n in (1, 2, 5):
        assert oracle_lib.reservoir_key(0.0, 5, SEED, 0, 0, 0, n_avg=n) == -np.inf


def test_large_n_reproduces_topk_by_weight(oracle_lib):
    # App. 8.2: n -> infinity gives pi_j -> E[u^(1/w)] = w / (w + 1), increasing in w, so the
    # reservoir keeps the top K by w. Weights 1.3x apart are far enough apart for n = 1024.
    rng = np.random.default_rng(2)
    T, B = 48, 16
    w = (0.5 * 1.3 ** rng.permutation(T)).astype(np.float32)
    pos = np.arange(T, dtype=np.int32) * 7 + 11
    top = np.sort(np.argsort(-w.astype(np.float64))[:B])
    for step in range(3):
        keep, _ = oracle_lib.select_slice(w, pos, B, 0, 0, oracle_lib.RESERVOIR, SEED, step, 1, 1,
                                          n_avg=1024)
        assert np.array_equal(keep, top), step
    # with n = 1 the same weights are sampled, not sorted
    keep1 = [oracle_lib.select_slice(w, pos, B, 0, 0, oracle_lib.RESERVOIR, SEED, s, 1, 1)[0]
             for s in range(3)]
    assert any(not np.array_equal(k, top) for k in keep1)


def _sum_pmf(w, n, M):
    """pmf of the bin index of sum_i X_i, X_i iid with P(X <= x) = x^w on [0, 1] split
    into M bins (each X put at its bin's midpoint; the offsets cancel in comparisons)."""
    edges = np.linspace(0.0, 1.0, M + 1)
    p = np.diff(edges ** w)
    out = p
    for _ in range(n - 1):
        out = np.clip(fftconvolve(out, p), 0.0, None)
    return out / out.sum()


def _p_second_wins(w1, w2, n, M=20000):
    p1, p2 = _sum_pmf(w1, n, M), _sum_pmf(w2, n, M)
    c1 = np.cumsum(p1)
    below = np.concatenate([[0.0], c1[:-1]])              # P(S1 index < b)
    return float(np.sum(p2 * below) + 0.5 * np.sum(p2 * p1))


@pytest.mark.parametrize("w1,w2,n", [(1.0, 2.0, 2), (1.0, 2.0, 5), (1.5, 3.0, 5), (2.0, 2.5, 3)])
def test_two_candidate_inclusion_matches_the_exact_law(oracle_lib, w1, w2, n):
    exact = _p_second_wins(w1, w2, n)
    draws = 40000
    w = np.array([w1, w2], np.float32)
    pos = np.array([101, 202], np.int32)
    wins = 0
    for step in range(draws):
        keep, _ = oracle_lib.select_slice(w, pos, 1, 0, 0, oracle_lib.RESERVOIR, SEED, step,
                                          5, 6, n_avg=n)
        wins += int(keep[0] == 1)
    emp = wins / draws
    sig = math.sqrt(exact * (1 - exact) / draws)
    assert abs(emp - exact) <= 5 * sig + 5e-4, (emp, exact, sig)
    # n-averaging sharpens the choice toward the heavier candidate (the n -> infinity
    # limit of App. 8.2): the exact law moves away from the n = 1 value w2 / (w1 + w2)
    assert exact > w2 / (w1 + w2)


def test_averaging_count_reaches_every_draw_group(oracle_lib):
    # keys with n = 4 use one Philox block; n = 5 needs a second block (draw group 1):
    # the fifth uniform must change the key of some candidates
    rng = np.random.default_rng(3)
    diff = 0
    for i in range(200):
        w = float(np.float32(rng.uniform(0.5, 2.0)))
        k4 = oracle_lib.reservoir_key(w, i, SEED, 1, 2, 3, n_avg=4)
        k5 = oracle_lib.reservoir_key(w, i, SEED, 1, 2, 3, n_avg=5)
        u5 = _draws(oracle_lib, i, 1, 2, 3, 5)
        assert abs(k5 - math.log(np.sum(u5 ** (1 / w)))) <= 1e-5 * max(1, abs(k5))
        diff += k4 != k5
    assert diff > 150
