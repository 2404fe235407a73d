"""Pins of the oracle's selection (§2.3 of the Nexus Sampling paper, Eq. (6) at n = 1,
Efraimidis-Spirakis keys) against brute-force enumeration, closed forms and the
deterministic special cases."""
import itertools
import math

import numpy as np
import pytest


def _es_set_probs(w, k):
    """Exact law of the kept set under successive weighted sampling without replacement
    (the distribution Efraimidis and Spirakis prove their keys realise)."""
    n = len(w)
    tot = float(np.sum(w))
    probs = {}
    for seq in itertools.permutations(range(n), k):
        p, rem = 1.0, tot
        for i in seq:
            p *= w[i] / rem
            rem -= w[i]
        key = tuple(sorted(seq))
        probs[key] = probs.get(key, 0.0) + p
    return probs


def _draws(oracle_lib, w, k, n_draws, seed=0x1234):
    w32 = np.asarray(w, np.float32)
    pos = np.arange(len(w), dtype=np.int32) + 100
    counts = {}
    for step in range(n_draws):
        keep, _ = oracle_lib.select_slice(w32, pos, k, 0, 0, oracle_lib.RESERVOIR, seed, step, 3, 9)
        key = tuple(int(x) for x in keep)
        counts[key] = counts.get(key, 0) + 1
    return counts


@pytest.mark.parametrize("w,k", [
    ([0.05, 0.1, 0.15, 0.2, 0.5], 2),
    ([3.0, 1.0, 1.0, 0.5, 0.25, 0.125, 2.0, 0.7, 0.01, 1.5], 4),
    ([1e-4, 2e-4, 5e-5, 8e-5, 3e-4, 1e-4], 3),          # token-sized weights
])
def test_reservoir_inclusion_matches_enumeration(oracle_lib, w, k):
    n_draws = 60000
    probs = _es_set_probs(np.asarray(w, np.float64), k)
    counts = _draws(oracle_lib, w, k, n_draws)
    assert all(len(s) == k for s in counts)
    # per-item inclusion within 5 sigma
    incl = np.zeros(len(w))
    for s, p in probs.items():
        incl[list(s)] += p
    emp = np.zeros(len(w))
    for s, c in counts.items():
        emp[list(s)] += c / n_draws
    sig = np.sqrt(incl * (1 - incl) / n_draws)
    assert np.all(np.abs(emp - incl) <= 5 * sig + 1e-12), (emp, incl)
    # chi-square over the sets with expected count >= 5
    chi2, df, rest_o, rest_e = 0.0, -1, 0, 0.0
    for s, p in probs.items():
        e = p * n_draws
        o = counts.get(s, 0)
        if e >= 5:
            chi2 += (o - e) ** 2 / e
            df += 1
        else:
            rest_o += o
            rest_e += e
    if rest_e > 0:
        chi2 += (rest_o - rest_e) ** 2 / max(rest_e, 1e-9)
        df += 1
    # Wilson-Hilferty: chi2/df ~ N(1 - 2/(9df), 2/(9df)); allow 5 sigma
    z = ((chi2 / df) ** (1 / 3) - (1 - 2 / (9 * df))) / math.sqrt(2 / (9 * df))
    assert z < 5, (chi2, df)


def test_inclusion_monotone_and_positive(oracle_lib):
    # App. 8.2: every positive weight has positive inclusion probability, monotone in w.
    w = np.array([0.02, 0.05, 0.1, 0.2, 0.4, 0.8])
    probs = _es_set_probs(w, 2)
    incl = np.zeros(w.size)
    for s, p in probs.items():
        incl[list(s)] += p
    assert (incl > 0).all() and (np.diff(incl) > 0).all()
    counts = _draws(oracle_lib, w, 2, 20000)
    emp = np.zeros(w.size)
    for s, c in counts.items():
        emp[list(s)] += c
    assert (emp > 0).all()


def test_horvitz_thompson_unbiased(oracle_lib):
    # Proposition 2, part 1: sum_j I_j z_j / p_j is unbiased for sum_j z_j.
    w = np.array([0.3, 0.05, 0.2, 0.1, 0.15, 0.2])
    z = np.array([1.0, 4.0, 0.5, 2.0, 3.0, 0.25])
    k, n_draws = 3, 40000
    probs = _es_set_probs(w, k)
    p = np.zeros(w.size)
    for s, pr in probs.items():
        p[list(s)] += pr
    counts = _draws(oracle_lib, w, k, n_draws, seed=99)
    vals, wts = [], []
    for s, c in counts.items():
        vals.append(sum(z[j] / p[j] for j in s))
        wts.append(c)
    vals, wts = np.array(vals), np.array(wts, float)
    mean = (vals * wts).sum() / n_draws
    var = ((vals - mean) ** 2 * wts).sum() / n_draws
    assert abs(mean - z.sum()) < 5 * math.sqrt(var / n_draws)


def test_degenerate_weights_collapse_to_topk(oracle_lib):
    rng = np.random.default_rng(1)
    for trial in range(50):
        T, K = 40, 7
        w = np.zeros(T, np.float32)
        big = rng.choice(T, K, replace=False)
        w[big] = rng.uniform(1, 5, K).astype(np.float32)
        small = np.setdiff1d(np.arange(T), big)
        w[small[: T // 2 - K]] = 1e-30
        keep, _ = oracle_lib.select_slice(w, np.arange(T, dtype=np.int32), K, 0, 0,
                                          oracle_lib.RESERVOIR, seed=trial, step=trial)
        assert np.array_equal(keep, np.sort(big))


def test_topk_mode_is_sorted_weights(oracle_lib):
    # top-K template: the K largest w, ties to the larger slot, plus the forced slots.
    rng = np.random.default_rng(2)
    T, B, ns, nr = 200, 50, 8, 8
    w = rng.integers(0, 20, T).astype(np.float32) / 7   # many ties
    keep, _ = oracle_lib.select_slice(w, np.arange(T, dtype=np.int32), B, ns, nr,
                                      oracle_lib.TOPK)
    forced = set(range(ns)) | set(range(T - nr, T))
    cand = [j for j in range(T) if j not in forced]
    best = sorted(cand, key=lambda j: (-float(w[j]), -j))[: B - ns - nr]
    assert np.array_equal(keep, np.array(sorted(forced | set(best))))


def test_budget_forced_and_identity(oracle_lib):
    rng = np.random.default_rng(3)
    T = 500
    w = rng.random(T).astype(np.float32)
    pos = np.arange(T, dtype=np.int32)
    for B in (64, 65, 100, 499):
        keep, kappa = oracle_lib.select_slice(w, pos, B, 32, 32, seed=7, step=1)
        assert keep.size == B and np.all(np.diff(keep) > 0)
        assert set(range(32)) <= set(keep) and set(range(T - 32, T)) <= set(keep)
        assert np.isnan(kappa[:32]).all() and np.isfinite(kappa[32:T - 32]).all()
        assert (kappa[32:T - 32] < 0).all()
    keep, _ = oracle_lib.select_slice(w, pos, T, 32, 32)
    assert np.array_equal(keep, np.arange(T))
    keep, _ = oracle_lib.select_slice(w[:10], pos[:10], 64, 32, 32)
    assert np.array_equal(keep, np.arange(10))
    with pytest.raises(ValueError):
        oracle_lib.select_slice(w, pos, 40, 32, 32)


def test_key_is_log_uniform_over_weight(oracle_lib):
    # kappa_j = ln_spec(u_j) / w_j with u_j from Philox(pos, step, head, seq; seed), word 0.
    seed, step, head, seq = 0x243F6A8885A308D3, 5, 17, 3
    x = oracle_lib.philox4x32_10([1234, step, head, seq], [seed & 0xFFFFFFFF, seed >> 32])[0]
    u = np.float32(oracle_lib.uniform(int(x)))
    w = np.float32(3.5e-5)
    want = np.float32(oracle_lib.ln_spec(np.array([u], np.float32))[0] / w)
    assert oracle_lib.reservoir_key(w, 1234, seed, step, head, seq) == want
    assert oracle_lib.reservoir_key(0.0, 1234, seed, step, head, seq) == -np.inf


def test_compaction_keeps_rows_in_order(oracle_lib):
    from streaming_kv_cache_step_gb300 import workloads as W
    wl = W.shrink(W.llama3_8b_layer(), lens=np.array([700], np.int32), capacity=700,
                  kv_heads=1, budget=np.array([150], np.int32), n_hubs=8)
    cache, q, over = W.slice_numpy_cache(wl, 0)
    k0, v0, p0 = cache["k"].copy(), cache["v"].copy(), cache["pos"].copy()
    params = dict(window=wl.window, walk_len=wl.walk_len, seed=11, step=0, **over)
    out = oracle_lib.evict_step(cache, q, params)
    keep = out["keep"][0, : out["newlen"][0]]
    assert out["newlen"][0] == 150 and cache["lens"][0, 0, 0] == 150
    assert np.array_equal(cache["k"][0, 0, 0, :150], k0[0, 0, 0, keep])
    assert np.array_equal(cache["v"][0, 0, 0, :150], v0[0, 0, 0, keep])
    assert np.array_equal(cache["pos"][0, 0, 0, :150], p0[0, 0, 0, keep])
    assert np.array_equal(cache["k"][0, 0, 0, 150:], k0[0, 0, 0, 150:])   # tail untouched
