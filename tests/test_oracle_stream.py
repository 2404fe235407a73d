"""Streaming pins of the oracle: a stream of eviction steps is a function of its state
(the Philox draws are indexed by position, step, head and sequence -- §2.3 -- so a stream
can be resumed or replayed exactly). The survival law of the selection over a stream
(Lemma 1) is pinned in test_oracle_survival.py; the planted-bridge survival study of §3
runs from tests/survival_study.py."""
import numpy as np

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


def test_stream_is_a_function_of_its_state(oracle_lib):
    # Philox is counter-based: the stream depends only on (inputs, step, seed).
    wl = W.shrink(W.tiny(), steps=10)
    full = run_stream(oracle_lib, wl, 10, oracle_lib.RESERVOIR, 3, 77)
    again = run_stream(oracle_lib, wl, 10, oracle_lib.RESERVOIR, 3, 77)
    assert np.array_equal(full, again)
