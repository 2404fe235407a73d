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
