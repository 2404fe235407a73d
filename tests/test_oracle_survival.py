"""Pins of the long-run survival law the paper proves for the selection step (§3 and
App. 8.3, Lemma 1): over a stream of eviction steps, a token's survival under the
reservoir is the product of its per-step inclusion probabilities (strictly positive for a
positive weight), while under deterministic top-K it is the product of indicators, so it
drops to zero at the first step where its weight falls below the cutoff.

The stream here puts one tracked token against N - 1 fresh candidates with fixed weights
at every step (everything else is replaced between steps), so its per-step inclusion
probability q is the same at every step and its E-step survival is exactly q^E; q comes
from enumerating successive weighted sampling without replacement (the law Efraimidis and
Spirakis prove their keys realise), not from the oracle."""
import itertools
import math

import numpy as np
import pytest


def _inclusion(w, k, j):
    """P(item j is among the k kept) under successive weighted sampling w/o replacement."""
    n, tot, p = len(w), float(np.sum(w)), 0.0
    for seq in itertools.permutations(range(n), k):
        if j not in seq:
            continue
        pr, rem = 1.0, tot
        for i in seq:
            pr *= w[i] / rem
            rem -= w[i]
        p += pr
    return p


def _stream(oracle_lib, w, k, steps, mode, seed):
    """Survival (0/1 after each step) of item 0 when every other item is fresh each step."""
    alive, out = True, []
    for e in range(steps):
        if alive:
            pos = np.array([7] + [1000 * (e + 1) + i for i in range(1, len(w))], np.int32)
            keep, _ = oracle_lib.select_slice(np.asarray(w, np.float32), pos, k, 0, 0, mode,
                                              seed, e, 3, 1)
            alive = 0 in keep
        out.append(alive)
    return out


@pytest.mark.parametrize("w0", [0.02, 0.08, 0.2])
def test_reservoir_survival_is_the_product_of_inclusions(oracle_lib, w0):
    w = np.array([w0, 0.3, 0.25, 0.15, 0.1, 0.12], np.float64)
    k, steps, streams = 3, 3, 12000
    q = _inclusion(w, k, 0)
    surv = np.zeros(steps)
    for sd in range(streams):
        surv += _stream(oracle_lib, w, k, steps, oracle_lib.RESERVOIR, 0xBEEF0000 + sd)
    surv /= streams
    for e in range(steps):
        want = q ** (e + 1)
        sig = math.sqrt(want * (1 - want) / streams)
        assert abs(surv[e] - want) <= 5 * sig + 1e-9, (e, surv[e], want)
    assert surv[-1] > 0                     # strictly positive for a positive weight


def test_topk_survival_is_the_product_of_indicators(oracle_lib):
    # below the K-th largest weight: gone at the first step; above it: kept at every step
    k, steps = 3, 5
    below = np.array([0.11, 0.3, 0.25, 0.15, 0.1, 0.12], np.float64)   # 4th largest
    above = np.array([0.16, 0.3, 0.25, 0.15, 0.1, 0.12], np.float64)   # 3rd largest
    for sd in range(20):
        assert _stream(oracle_lib, below, k, steps, oracle_lib.TOPK, sd) == [False] * steps
        assert _stream(oracle_lib, above, k, steps, oracle_lib.TOPK, sd) == [True] * steps
    # the reservoir keeps the below-cutoff token alive at a positive rate at every step
    alive = sum(_stream(oracle_lib, below, k, 2, oracle_lib.RESERVOIR, 0x5000 + sd)[-1]
                for sd in range(2000))
    q = _inclusion(below, k, 0)
    assert abs(alive / 2000 - q * q) <= 5 * math.sqrt(q * q * (1 - q * q) / 2000)
