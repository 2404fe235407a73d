"""Full-size parity: every workload at its full size, in the launch configuration the
benchmark times (one nexus_evict_step over every slice of the cache), checked against the
oracle on sampled slices it computes one by one, plus properties that hold for every
slice; and the streaming runs (fresh tokens between steps) against the oracle's own
stream of the sampled slices."""
import numpy as np
import pytest
import torch

import oracle
from harness import DEV, GpuRun, compare_survivors, oracle_kappa, oracle_params
from streaming_kv_cache_step_gb300 import nexus
from streaming_kv_cache_step_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _sample(wl, n, seed=7):
    if wl.n_slices <= n:
        return list(range(wl.n_slices))
    rng = np.random.default_rng(seed)
    if n < 3:
        return sorted(rng.choice(wl.n_slices, n, replace=False).tolist())
    picks = set(rng.choice(wl.n_slices, n - 2, replace=False).tolist())
    picks |= {0, wl.n_slices - 1}
    return sorted(picks)


def _check_all_slices(run, keep, lens0):
    """Properties every slice satisfies: new length, ascending in-range survivors, forced
    slots kept."""
    wl = run.wl
    lens = run.lens()
    for sid in range(run.cache.n_slices):
        s = wl.slice_coords(sid)[1]
        T, B = int(lens0[sid]), int(wl.budget[s])
        nl = min(T, B)
        assert lens[sid] == nl
        k = keep[sid, :nl]
        assert np.all(np.diff(k) > 0) and (nl == 0 or (k[0] >= 0 and k[-1] < T))
        if T > B:
            assert np.array_equal(k[: wl.n_sink], np.arange(wl.n_sink))
            assert np.array_equal(k[nl - wl.n_recent:], np.arange(T - wl.n_recent, T))


FULL = {"llama3_8b_layer": 8, "batch16_32layers": 10, "long_context": 3, "streaming_paged": 10,
        "prefill_256k": 2}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_step0(name):
    wl = W.WORKLOADS[name]()
    run = GpuRun(wl)
    lens0 = run.lens()
    nexus.evict_step(run.cache, run.q, run.params, run.keep, run.ws, run.status)
    run.check_status()
    keep = run.keep.cpu().numpy()
    _check_all_slices(run, keep, lens0)
    for sid in _sample(wl, FULL[name]):
        c, q, over = W.slice_numpy_cache(wl, sid)
        ref = oracle.evict_step(c, q, oracle_params(wl, over), mutate=False)
        T = int(lens0[sid])
        nl = int(ref["newlen"][0])
        kappa = oracle_kappa(wl, sid, ref["w"][0, :T], c["pos"][0, 0, 0, :T])
        compare_survivors(keep[sid, :nl], ref["keep"][0, :nl], kappa)
        for nm in ("k", "v", "pos"):
            got = W.storage_to_numpy(run.slice_rows(nm, sid, nl))
            assert np.array_equal(got, c[nm][0, 0, 0][keep[sid, :nl]]), (sid, nm)


STREAMS = [("tiny", 10, 1), ("llama3_8b_layer", 21, 2), ("streaming_paged", 200, 3),
           ("long_context", 3, 1)]


@pytest.mark.parametrize("name,steps,n_sampled", STREAMS)
def test_full_size_stream(name, steps, n_sampled):
    """Evict, append fresh tokens, evict again ... on the GPU (all slices) and in the
    oracle (sampled slices, each with its own state). Survivors are compared as sets of
    absolute token positions, step by step."""
    wl = W.WORKLOADS[name]()
    run = GpuRun(wl)
    sids = _sample(wl, n_sampled, seed=11)
    states = {}
    for sid in sids:
        c, q, over = W.slice_numpy_cache(wl, sid, capacity=wl.capacity)
        states[sid] = (c, over)
    worst = 1.0
    for step in range(steps):
        if step > 0:
            W.append_tokens_all(wl, run.d, step)
            run.q = W.queries(wl, step, DEV)
            for sid in sids:
                W.append_tokens(wl, W.numpy_cache_as_torch(states[sid][0]), step, sids=[sid],
                                slice_index={sid: 0})
        run.params.step = step
        nexus.evict_step(run.cache, run.q, run.params, run.keep, run.ws, run.status)
        run.check_status()
        lens = run.lens()
        for sid in sids:
            c, over = states[sid]
            qn = W.storage_to_numpy(W.to_storage(torch.as_tensor(W.query_rows(wl, sid, step)),
                                                 wl.dtype)).reshape(1, 1, wl.group, wl.window,
                                                                    wl.head_dim)
            oracle.evict_step(c, qn, oracle_params(wl, over, step=step), mutate=True)
            nl = int(c["lens"].reshape(-1)[0])
            assert lens[sid] == nl
            want = set(c["pos"][0, 0, 0, :nl].tolist())
            got = set(W.storage_to_numpy(run.slice_rows("pos", sid, nl)).tolist())
            overlap = len(want & got) / max(nl, 1)
            worst = min(worst, overlap)
            assert overlap >= 0.995, (step, sid, overlap)
    print(f"{name}: worst per-step survivor overlap {worst:.5f} over {steps} steps")
