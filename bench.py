#!/usr/bin/env python
"""Throughput of one Nexus Sampling eviction step (scores, walk, reservoir selection,
in-place compaction) on the GB300, through the library's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                    [--workload batch16_32layers]

One step = nexus_evict_step over every slice of the workload's step-0 cache (for the
default workload: 16 sequences x 32 layers x 8 KV heads of 32768 cached rows each, d =
128 bf16, evicted to 6554 rows each -- 134M rows, 68.7 GB of K and V, the largest
single-GPU workload). Before each timed step, untimed: the cache is restored from a
pristine device copy, a buffer twice the L2 size is written and another one as large is
read (L2 then holds neither the cache nor dirty lines), and a sleep kernel keeps the
device busy while the host issues the step. By default the timed loop replays one
CUDA-graph capture of the nexus_evict_step call (--launch eager calls it every step; its
times are reported beside). Rank 0 prints one JSON line.

value   KV rows scored+evicted per second (a row = one cached token of one KV head of
        one layer), all ranks, device-timed with CUDA events on the launching stream.
e2e     the same metric end to end through the C ABI with host buffers: per step the
        cache, queries and lengths are copied from pinned host memory to the device,
        the step runs, and the kept-slot lists and lengths are copied back.
roofline  the dominant kernel: algorithmic bytes per launch / its mean event-timed
        duration, against the measured HBM copy bandwidth; traffic from the counter
        capture recorded under profiles/ while the kernel's source is unchanged.
cpu_baseline  the CPU oracle (C) on every host core (one slice per thread), bounded sample.
--impl reference  runs the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "cached tokens scored+evicted/s per eviction step; % HBM roofline (1×GB300)"
UNIT = "KV rows/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--workload", default="batch16_32layers")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--n-avg", type=int, default=1,
                    help="reservoir averaging count n of Eq. (6) (the paper runs n = 5)")
    ap.add_argument("--block-size", type=int, default=1, choices=(1, 32),
                    help="rows per keep/evict decision; at 32 the workload's budget becomes "
                         "ceil(B / 32) blocks with one sink and one recency block")
    ap.add_argument("--launch", choices=("graph", "eager"), default="graph",
                    help="device-timed loop: replay one CUDA-graph capture of the "
                         "nexus_evict_step call, or call it eagerly every step")
    return ap.parse_args()


# source file of each kernel, for matching the DRAM traffic recorded under profiles/
KERNEL_SOURCES = {"score_tc": "nx_score_tc.cu", "select": "nx_select.cu",
                  "compact": "nx_compact.cu", "prep": "nx_score.cu"}


def _source_digest(kernel: str) -> str | None:
    import hashlib
    name = KERNEL_SOURCES.get(kernel)
    if name is None:
        return None
    path = os.path.join(ROOT, "streaming_kv_cache_step_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str) -> int | None:
    """DRAM bytes (read + write) of one launch, from the counter capture recorded in
    profiles/traffic.txt, when it was taken of this kernel source on this workload; None
    once the kernel has changed since (or when there is no capture)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    digest = _source_digest(kernel)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel \
                    and parts[1] == workload and parts[2] == digest:
                return int(parts[3])
    return None


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), src="measured")
    return dict(hbm_gbs=FALLBACK_HBM_GBS, src="fallback")


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="nx_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self) -> dict:
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["no samples"])

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1])]
        mx = [num(r[2]) for r in rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(mx) if mx else None, reasons=reasons, samples=len(rows),
                    power_w_max=max((num(r[3]) or 0) for r in rows))


# ---------------------------------------------------------------------------
# distributed (one process per GPU; host-side barrier and max only)
# ---------------------------------------------------------------------------

def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allmax(x: float, world: int) -> float:
    """Maximum of x over the ranks (the slowest rank's time decides)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seq_base(rank: int, wl) -> int:
    """First Philox sequence id of this rank: every rank evicts its own sequences."""
    return rank * wl.seqs


def job_rate(rows_per_step: int, steps: int, local_ms: float, world: int) -> tuple:
    """Whole-job rows/s: the rows all ranks processed over the slowest rank's time.
    Returns (rows/s, max-over-ranks milliseconds)."""
    total_ms = allmax(local_ms, world)
    return rows_per_step * steps * world / (total_ms / 1e3), total_ms


# ---------------------------------------------------------------------------
# algorithmic bytes (what the method must move)
# ---------------------------------------------------------------------------

def algorithmic_bytes(wl, lens0: np.ndarray, keep: np.ndarray, newlen: np.ndarray) -> dict:
    """Per step: K read once + pos (scoring), queries, the kept-unit list, and every
    moved row's k, v and pos read and written (compaction). keep holds kept units (rows,
    or blocks of wl.block_size rows); newlen the rows left per slice."""
    eb = 2 if wl.dtype == "bf16" else 4
    row = wl.head_dim * eb
    b = wl.block_size
    rows = int(lens0.sum())
    moved, units = 0, 0
    for i in range(keep.shape[0]):
        n = int(newlen[i])
        nu = -(-n // b)
        units += nu
        u = keep[i, :nu]
        if b == 1:
            moved += int((u != np.arange(nu)).sum())
        else:
            # a block moves whole; the newest block may hold fewer than b rows
            sizes = np.minimum(b, int(lens0[i]) - u * b)
            moved += int(sizes[u != np.arange(nu)].sum())
    qbytes = wl.n_slices * wl.group * wl.window * wl.head_dim * eb
    score = rows * (row + 4) + qbytes
    compact = moved * (4 * row + 8) + units * 4
    return dict(rows=rows, moved=moved, score=score, compact=compact, total=score + compact)


def configured_workload(args):
    """The named workload with the reservoir averaging count and block size asked for."""
    import dataclasses
    from streaming_kv_cache_step_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]()
    over = dict(n_avg=getattr(args, "n_avg", 1))
    b = getattr(args, "block_size", 1)
    if b > 1:
        over.update(block_size=b, n_sink=-(-wl.n_sink // b), n_recent=-(-wl.n_recent // b),
                    budget=(-(-wl.budget // b)).astype(np.int32))
    return dataclasses.replace(wl, **over)


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

_T0 = time.time()


def _log(msg: str) -> None:
    """Progress of the set-up phases on stderr (stdout carries only the JSON line)."""
    print(f"[bench {time.time() - _T0:7.1f} s] {msg}", file=sys.stderr, flush=True)


def run_native(args, rank, world, local):
    from streaming_kv_cache_step_gb300 import nexus
    from streaming_kv_cache_step_gb300 import workloads as W
    import __graft_entry__
    __graft_entry__.build()
    _log("library built and loaded")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = configured_workload(args)
    pristine = W.make_cache(wl, dev)
    _log(f"cache of {wl.name} generated on the device")
    work = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in pristine.items()}
    q = W.queries(wl, 0, dev)
    cache = nexus.Cache.from_dict(work)
    params = nexus.Params(budget=work["budget"], budget_max=int(wl.budget.max()),
                          window=wl.window, walk_len=wl.walk_len, n_sink=wl.n_sink,
                          n_recent=wl.n_recent, lam=wl.lam, eps_tie=wl.eps_tie,
                          seed=wl.philox_seed, step=0, seq_id_base=rank_seq_base(rank, wl),
                          n_avg=wl.n_avg, block_size=wl.block_size)
    ws = nexus.alloc_workspace(cache, params)
    status = nexus.new_status(dev)
    keep = torch.full((cache.n_slices, wl.capacity), -1, dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    clean = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    names = ("k", "v", "pos", "lens")

    def restore():
        for n in names:
            work[n].copy_(pristine[n], non_blocking=True)
        # evict L2: write a buffer twice its size, then read another one as large, so the
        # step starts with a cold L2 that holds no dirty lines to write back
        flush.zero_()
        torch.sum(clean, 0, out=sink)

    def step(events=None):
        arr = nexus.profile_next_call(events) if events else None
        nexus.evict_step(cache, q, params, keep, ws, status)
        del arr

    for _ in range(args.warmup):
        restore()
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    launch_names = nexus.last_launch_names()
    nl = len(launch_names)
    scorer_cfg = nexus.scorer_config() if "score_tc" in launch_names else None

    # ---- timed region ----
    # Each timed step: restore the pristine cache, flush L2, then keep the device busy
    # while the host issues the step, so that the events time the device work.
    def timed(K, graph):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        per = [[] for _ in range(nl)]
        count = 0
        if graph is not None:
            g, kev_g = graph
        for i in range(K):
            restore()
            torch.cuda._sleep(200_000)
            starts[i].record(stream)
            if graph is not None:
                g.replay()
            else:
                kev_g = [torch.cuda.Event(enable_timing=True) for _ in range(nl)]
                step(kev_g)
            ends[i].record(stream)
            count += nl if graph is not None else nexus.last_launch_count()
            ends[i].synchronize()          # the graph's events are re-recorded next step
            for j in range(nl):
                prev = starts[i] if j == 0 else kev_g[j - 1]
                per[j].append(prev.elapsed_time(kev_g[j]))
        torch.cuda.synchronize()
        step_ms = [starts[i].elapsed_time(ends[i]) for i in range(K)]
        per_kernel = {f"{j}:{name}": statistics.mean(per[j]) * 1e3
                      for j, name in enumerate(launch_names)}       # microseconds
        return step_ms, per_kernel, count

    graph = None
    if args.launch == "graph":
        # one capture of the C-ABI call, its per-launch events included; every replay
        # runs the same kernels on the restored inputs
        kev_g = [torch.cuda.Event(enable_timing=True) for _ in range(nl)]
        for e in kev_g:
            e.record(stream)
        restore()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            arr = nexus.profile_next_call(kev_g)
            nexus.evict_step(cache, q, params, keep, ws, status)
            del arr
        torch.cuda.synchronize()
        graph = (g, kev_g)
        for _ in range(2):
            restore()
            g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"device status {int(status.item())}"

    _log("warm-up done")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    barrier(world)
    torch.cuda.synchronize()
    step_ms, per_kernel, launches = timed(K, graph)
    torch.cuda.synchronize()
    barrier(world)
    time.sleep(0.2)
    clocks = sampler.stop()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    local_ms = sum(step_ms)
    eager = None
    if graph is not None:
        # the same step called eagerly through the C ABI (host launch latency included
        # wherever the device outruns the host)
        ke = min(K, 30)
        e_ms, e_kern, _ = timed(ke, None)
        eager = dict(ms_per_step=round(allmax(sum(e_ms), world) / ke, 5), steps=ke,
                     kernels_us={k: round(v, 3) for k, v in e_kern.items()})

    _log("timed loops done")
    # algorithmic bytes of this step (from the kept-slot lists of the last step)
    lens0 = pristine["lens"].reshape(-1).cpu().numpy()
    newlen = work["lens"].reshape(-1).cpu().numpy()
    ab = algorithmic_bytes(wl, lens0, keep.cpu().numpy(), newlen)
    rows_per_step = ab["rows"]
    value, total_ms = job_rate(rows_per_step, K, local_ms, world)

    # dominant kernel and its roofline
    dom = max(per_kernel, key=per_kernel.get)
    dom_name = dom.split(":", 1)[1]
    if "compact" in dom_name:
        dom_bytes = ab["compact"]
    elif "select" in dom_name:
        dom_bytes = rows_per_step * 4 + int(newlen.sum()) * 4
    else:
        dom_bytes = ab["score"]
    peaks = measured_peaks()
    achieved = dom_bytes / (per_kernel[dom] * 1e-6) / 1e9
    step_gbs = ab["total"] / (statistics.mean(step_ms) * 1e-3) / 1e9
    roofline = dict(bound="hbm", kernel=dom_name, achieved=round(achieved, 1),
                    peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=round(achieved / peaks["hbm_gbs"], 4),
                    traffic=recorded_traffic(dom_name, wl.name), alg_bytes=int(dom_bytes),
                    peak_source=peaks["src"],
                    whole_step=dict(achieved=round(step_gbs, 1),
                                    frac=round(step_gbs / peaks["hbm_gbs"], 4),
                                    alg_bytes=ab["total"]))

    # ---- end to end through the C ABI with host buffers ----
    # about 1e11 bytes of host->device copies at most (five steps of the 68.7 GB cache)
    cache_bytes = sum(pristine[n].numel() * pristine[n].element_size() for n in names)
    e2e_steps = args.e2e_steps or max(3, min(K, 50, int(4e11 // max(cache_bytes, 1))))
    host = {n: torch.empty_like(pristine[n], device="cpu").pin_memory() for n in names}
    for n in names:
        host[n].copy_(pristine[n])
    q_host = torch.empty_like(q, device="cpu").pin_memory()
    q_host.copy_(q)
    keep_host = torch.empty_like(keep, device="cpu").pin_memory()
    lens_host = torch.empty_like(pristine["lens"], device="cpu").pin_memory()
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    h2d = sum(host[n].numel() * host[n].element_size() for n in names) + \
        q_host.numel() * q_host.element_size()
    d2h = keep_host.numel() * 4 + lens_host.numel() * 4
    barrier(world)
    torch.cuda.synchronize()
    for i in range(e2e_steps):
        flush.zero_()
        torch.sum(clean, 0, out=sink)
        e_s[i].record(stream)
        for n in names:
            work[n].copy_(host[n], non_blocking=True)
        q.copy_(q_host, non_blocking=True)
        nexus.evict_step(cache, q, params, keep, ws, status)
        keep_host.copy_(keep, non_blocking=True)
        lens_host.copy_(work["lens"], non_blocking=True)
        e_e[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    _log(f"end-to-end loop done ({e2e_steps} steps)")
    e2e_value, _ = job_rate(rows_per_step, e2e_steps,
                            sum(e_s[i].elapsed_time(e_e[i]) for i in range(e2e_steps)), world)

    out = dict(metric=METRIC, value=round(value, 1), unit=UNIT, n_gpus=world, steps=K,
               warmup=args.warmup, ms_per_step=round(total_ms / K, 5), higher_is_better=True,
               scaling="weak", vs_baseline=None, dtype=wl.dtype, data="synthetic",
               config=dict(workload=wl.name, layers=wl.layers, seqs=wl.seqs,
                           q_heads=wl.q_heads, kv_heads=wl.kv_heads, head_dim=wl.head_dim,
                           cache_rows=int(wl.lens.max()), budget=int(wl.budget.max()),
                           window=wl.window, walk=wl.walk_len, n_sink=wl.n_sink,
                           n_recent=wl.n_recent, n_avg=wl.n_avg, block_size=wl.block_size,
                           rows_per_step=rows_per_step,
                           moved_rows=ab["moved"], alg_bytes_per_step=ab["total"],
                           l2="flushed between timed steps (2x L2 written, then 2x L2 read)",
                           launch=("one CUDA-graph capture of the nexus_evict_step call, "
                                   "replayed every step" if graph is not None
                                   else "nexus_evict_step called every step"),
                           parallelism=f"dp{world} (independent sequences per rank)"),
               roofline=roofline,
               e2e=dict(value=round(e2e_value, 1), unit=UNIT, h2d_bytes_per_step=h2d,
                        d2h_bytes_per_step=d2h, steps=e2e_steps),
               ms_per_step_median=round(statistics.median(step_ms), 5),
               per_sequence_tokens_per_s=round(value / (wl.layers * wl.kv_heads), 1),
               gpu_launches=launches, kernels_us={k: round(v, 3) for k, v in per_kernel.items()},
               scorer=scorer_cfg, eager=eager,
               clocks=clocks)
    return out, wl


# ---------------------------------------------------------------------------
# CPU oracle (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def _oracle_slices(wl, n):
    """n sampled step-0 slices of the workload (one per host thread); a workload with
    fewer slices than threads repeats them, so that every core has a slice to score."""
    from streaming_kv_cache_step_gb300 import workloads as W
    made = [W.slice_numpy_cache(wl, sid) for sid in range(min(wl.n_slices, n))]
    return [made[i % len(made)] for i in range(n)]


def _oracle_pass(wl, slices, pool):
    """One pass of the oracle's eviction step over the sampled slices, one host thread
    per slice (ctypes releases the GIL); returns the rows processed."""
    import oracle

    def run_slice(item):
        c, q, over = item
        cc = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in c.items()}
        pr = dict(window=wl.window, walk_len=wl.walk_len, n_sink=wl.n_sink,
                  n_recent=wl.n_recent, lam=wl.lam, eps_tie=wl.eps_tie, seed=wl.philox_seed,
                  step=0, n_avg=wl.n_avg, block_size=wl.block_size, **over)
        oracle.evict_step(cc, q, pr, mutate=True, nthreads=1)
        return int(c["lens"].reshape(-1)[0])

    return sum(pool.map(run_slice, slices))


def oracle_rate(wl, budget_s: float):
    """cpu_baseline: rows/s of the CPU oracle, wall-clock, on a bounded sample."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    slices = _oracle_slices(wl, cores)
    distinct = min(wl.n_slices, cores)
    rows, passes = 0, 0
    with ThreadPoolExecutor(max_workers=len(slices)) as pool:
        t0 = time.perf_counter()
        while True:
            rows += _oracle_pass(wl, slices, pool)
            passes += 1
            dt = time.perf_counter() - t0
            if dt >= budget_s:
                break
    return dict(value=round(rows / dt, 1), unit=UNIT, cores=cores, threads=len(slices),
                kind="oracle",
                sample=f"{passes} passes over {len(slices)} slices ({distinct} distinct) of the "
                       f"{wl.n_slices} step-0 slices of {wl.name} ({rows} rows, {dt:.1f} s "
                       f"wall), one host thread per slice")


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle as it stands, K timed steps after W warm-up steps,
    each step one pass over a bounded sample of the workload's slices."""
    from concurrent.futures import ThreadPoolExecutor
    from streaming_kv_cache_step_gb300 import workloads as W
    if rank != 0:
        return None
    import oracle
    oracle.build()
    wl = configured_workload(args)
    cores = os.cpu_count() or 1
    slices = _oracle_slices(wl, cores)
    with ThreadPoolExecutor(max_workers=len(slices)) as pool:
        for _ in range(args.warmup):
            _oracle_pass(wl, slices, pool)
        t0 = time.perf_counter()
        rows = 0
        for _ in range(args.steps):
            rows += _oracle_pass(wl, slices, pool)
        dt = time.perf_counter() - t0
    value = rows / dt
    sample = (f"{len(slices)} slices ({min(wl.n_slices, cores)} distinct) of the "
              f"{wl.n_slices} step-0 slices of {wl.name} per step, one host thread per slice")
    return dict(metric=METRIC, value=round(value, 1), unit=UNIT, n_gpus=world,
                steps=args.steps, warmup=args.warmup,
                ms_per_step=round(dt / max(args.steps, 1) * 1e3, 3), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                impl="reference",
                config=dict(workload=wl.name, sample_slices=len(slices),
                            rows_per_step=rows // max(args.steps, 1)),
                cpu_baseline=dict(value=round(value, 1), unit=UNIT, cores=cores,
                                  threads=len(slices), kind="oracle", sample=sample),
                e2e=dict(value=round(value, 1), unit=UNIT, h2d_bytes_per_step=0,
                         d2h_bytes_per_step=0))


def main():
    args = parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    out, wl = run_native(args, rank, world, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = oracle_rate(wl, budget_s=10.0)
            _log("cpu baseline done")
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
