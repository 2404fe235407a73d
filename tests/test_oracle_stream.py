"""Streaming pins of the oracle: the long-run survival claim of the Nexus Sampling paper
(§3 and Lemma 1: planted bridge tokens survive longer under Nexus scoring with the
reservoir than under deterministic top-K on the direct score), and resumability of
the counter-based stream."""
import math

import numpy as np
import pytest

from streaming_kv_cache_step_gb300 import workloads as W


def run_stream(oracle_lib, wl, steps, mode, walk_len, philox_seed, sid=0):
    """Evict, append fresh tokens, repeat. Returns surviving planted-bridge fractions."""
    cache, q, over = W.slice_numpy_cache(wl, sid)
    bridges = W.plant(wl, sid)["bridges"]
    alive = []
    for step in range(steps):
        if step > 0:
            W.append_tokens(wl, W.numpy_cache_as_torch(cache), step, sids=[sid],
                            slice_index={sid: 0})
            q = W.storage_to_numpy(W.to_storage(
                __import__("torch").as_tensor(W.query_rows(wl, sid, step)), wl.dtype)
            ).reshape(q.shape)
        params = dict(window=wl.window, walk_len=walk_len, mode=mode, seed=philox_seed,
                      step=step, n_sink=wl.n_sink, n_recent=wl.n_recent, **over)
        oracle_lib.evict_step(cache, q, params)
        T = int(cache["lens"].reshape(-1)[0])
        present = np.isin(bridges, cache["pos"].reshape(-1)[:T])
        alive.append(present.mean())
    return np.array(alive)


@pytest.mark.xfail(strict=False, reason=(
    "long-run survival claim not reproduced on the tiny synthetic recipe: planted "
    "bridges sit in the mid-band and die within 2-3 steps under every policy "
    "(32 seeds, 10 steps; measured curves are in the design notes)"))
def test_bridges_survive_longer_under_nexus_than_topk(oracle_lib):
    n_seeds, steps = 32, 10
    nexus, topk = [], []
    for seed in range(n_seeds):
        wl = W.shrink(W.tiny(), seed=W.DATA_SEED_BASE + 1000 + seed)
        nexus.append(run_stream(oracle_lib, wl, steps, oracle_lib.RESERVOIR, 3, 0xA5A5 + seed))
        topk.append(run_stream(oracle_lib, wl, steps, oracle_lib.TOPK, 0, 0xA5A5 + seed))
    nexus, topk = np.array(nexus), np.array(topk)
    # lifetime = area under the survival curve (steps survived per bridge)
    final_n, final_t = nexus.sum(1), topk.sum(1)
    diff = final_n - final_t
    se = diff.std(ddof=1) / math.sqrt(n_seeds) + 1e-12
    # one-sided paired test on the lifetimes
    assert diff.mean() > 0, (final_n.mean(), final_t.mean())
    assert diff.mean() / se > 2.0, (final_n.mean(), final_t.mean(), se)


def test_stream_is_a_function_of_its_state(oracle_lib):
    # Philox is counter-based: the stream depends only on (inputs, step, seed).
    wl = W.shrink(W.tiny(), steps=10)
    full = run_stream(oracle_lib, wl, 10, oracle_lib.RESERVOIR, 3, 77)
    again = run_stream(oracle_lib, wl, 10, oracle_lib.RESERVOIR, 3, 77)
    assert np.array_equal(full, again)
