"""The multi-GPU path of bench.py on CPU: world-size-2 gloo ranks exercise its host logic
(every rank evicts its own sequences, a barrier, the slowest rank's time decides the
whole-job rate, only rank 0 runs the reference arm). Slices are independent, so no data
moves between ranks."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from streaming_kv_cache_step_gb300 import workloads as W
        wl = W.WORKLOADS["llama3_8b_layer"]()
        local_ms = 10.0 * (rank + 1)                 # rank 1 is the slower one
        rate, total = bench.job_rate(65536, 5, local_ms, world)
        bench.barrier(world)
        base = bench.rank_seq_base(rank, wl)

        class Args:
            workload, steps, warmup = "llama3_8b_layer", 1, 0
        ref = bench.run_reference(Args, rank, world) if rank != 0 else "skipped"
        out.put((rank, rate, total, base, wl.seqs, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_sequences_and_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, rate0, tot0, base0, seqs, _), (r1, rate1, tot1, base1, _, ref1) = res
    assert (r0, r1) == (0, 1)
    assert tot0 == tot1 == pytest.approx(20.0)           # max over ranks
    assert rate0 == rate1 == pytest.approx(65536 * 5 * 2 / 0.020)
    assert (base0, base1) == (0, seqs)                    # disjoint Philox sequence ids
    assert ref1 is None                                   # only rank 0 runs the reference


def _oracle_cache(d):
    """A make_cache dict (CPU torch tensors) as the oracle's numpy cache."""
    from streaming_kv_cache_step_gb300 import workloads as W
    c = {k: d[k] for k in ("layers", "seqs", "kv_heads", "group", "head_dim", "capacity")}
    for k in ("k", "v"):
        c[k] = W.storage_to_numpy(d[k])
    c["pos"] = d["pos"].numpy().copy()
    c["lens"] = d["lens"].numpy().copy()
    return c


def _shard_workload():
    import numpy as np
    from streaming_kv_cache_step_gb300 import workloads as W
    return W.shrink(W.llama3_8b_layer(), seqs=2, kv_heads=2, lens=np.array([700, 450], np.int32),
                    capacity=704, budget=np.array([150, 120], np.int32), n_hubs=8)


def _oracle_rank(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from streaming_kv_cache_step_gb300 import workloads as W
        wl = _shard_workload()
        c = _oracle_cache(W.make_cache(wl, "cpu"))
        q = W.storage_to_numpy(W.queries(wl, 0, "cpu"))
        params = dict(window=wl.window, walk_len=wl.walk_len, budget=wl.budget,
                      seed=wl.philox_seed, step=0, seq_id_base=bench.rank_seq_base(rank, wl))
        res = oracle.evict_step(c, q, params, mutate=True)
        got = [None] * world
        dist.all_gather_object(got, (rank, res["keep"], res["newlen"], c["k"], c["pos"]))
        if rank == 0:
            out.put(got)
    finally:
        dist.destroy_process_group()


def test_two_ranks_evicting_their_own_sequences_equal_one_process():
    """§8(e) partitioning: every rank evicts its own sequences with its own Philox
    sequence ids (bench.rank_seq_base); together they give exactly what one process
    evicting all the sequences at once gives. Each rank here holds the same generated
    data (as every bench rank does), so the one-process cache is the two shards stacked."""
    import numpy as np
    import oracle
    from streaming_kv_cache_step_gb300 import workloads as W
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_oracle_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=300), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl = _shard_workload()
    d = _oracle_cache(W.make_cache(wl, "cpu"))
    S = wl.seqs
    whole = dict(d, seqs=2 * S)
    for k in ("k", "v", "pos", "lens"):
        whole[k] = np.ascontiguousarray(np.concatenate([d[k], d[k]], axis=1))
    q = W.storage_to_numpy(W.queries(wl, 0, "cpu"))
    q2 = np.ascontiguousarray(np.concatenate([q, q], axis=1))
    params = dict(window=wl.window, walk_len=wl.walk_len, budget=np.tile(wl.budget, 2),
                  seed=wl.philox_seed, step=0, seq_id_base=0)
    res = oracle.evict_step(whole, q2, params, mutate=True)
    per_rank = wl.n_slices                         # slices of one rank, in slice-id order
    for r, keep, newlen, k, pos in got:
        sl = slice(r * per_rank, (r + 1) * per_rank)
        assert np.array_equal(res["keep"][sl], keep), r
        assert np.array_equal(res["newlen"][sl], newlen), r
        assert np.array_equal(whole["k"][:, r * S:(r + 1) * S], k), r
        assert np.array_equal(whole["pos"][:, r * S:(r + 1) * S], pos), r
    # the ranks' draws differ (their sequence ids do), so their survivors differ too
    assert not np.array_equal(got[0][1], got[1][1])
