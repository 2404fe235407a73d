"""The pages' printed defaults (tests/golden/paper_defaults.txt) against the values the
workloads, the oracle and the library are run with."""
import os

import numpy as np

import oracle
from streaming_kv_cache_step_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "paper_defaults.txt")


def _golden() -> dict:
    out = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, v = line.split()
            out[k] = float(v)
    return out


def test_workloads_use_the_printed_mixing_and_tie_break():
    g = _golden()
    for make in W.WORKLOADS.values():
        wl = make()
        assert wl.lam == g["lambda"] and wl.eps_tie == g["eps_tie"], wl.name


def test_printed_window_and_walk_depth_are_the_unset_configs_choice():
    # the tiny and streaming configs name no window; they take the printed W and H
    g = _golden()
    for name in ("tiny", "streaming_paged"):
        wl = W.WORKLOADS[name]()
        assert (wl.window, wl.walk_len) == (g["window"], g["walk_len"]), name


def test_oracle_eps_tie_ramp_matches_the_printed_magnitude(oracle_lib):
    # with identical keys every a_j = 1/T and c~ is uniform too, so w_j - w_0 is the
    # tie-break ramp alone: eps_tie * j / (T - 1) (w is binary32: a few ulp of 1/6)
    g = _golden()
    T, d, Wn = 9, 8, 4
    K = np.ones((T, d))
    Q = np.ones((Wn, d))
    o = oracle.slice_scores(K, Q, 3, g["lambda"], g["eps_tie"])
    ramp = o["w"] - o["w"][0]
    assert np.allclose(ramp, g["eps_tie"] * np.arange(T) / (T - 1), rtol=0, atol=4e-8)
    assert ramp[-1] > 0.9 * g["eps_tie"]
