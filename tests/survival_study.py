"""Long-run survival of planted bridge tokens under Nexus Sampling against deterministic
top-K on the direct score -- the claim of the paper's §3 ("bridge tokens ... land in the
noisy mid-band"; Nexus scoring lifts them, the reservoir keeps them at a controlled rate)
and Lemma 1 (App. 8.3) -- measured on the CPU oracle, on sampled slices of the seeded
workloads, over many seeds.

    python tests/survival_study.py --recipe tiny --seeds 32
    python tests/survival_study.py --recipe long_context --seeds 32 --steps 50
    python tests/survival_study.py --recipe streaming_paged --seeds 32 --steps 200

Each stream evicts, appends the workload's fresh tokens, and evicts again, with fresh
window queries near the same hubs every step (the workloads' own stream). Policies:
"nexus" = the workload's walk length H with reservoir keys (n = 1), "topk_a" = H = 0 with
the top-K template on the direct score. Every seed changes both the data seed and the
Philox seed; both policies see the same data. Printed: one JSON line with the mean
survival curves, the mean lifetimes (area under the curve, steps survived per bridge), a
one-sided paired t statistic of nexus - topk_a over seeds, and diagnostics of step 0: the
bridges' mean rank percentile under a and under the Nexus weight w (0 = top), and the
budget's percentile (the top-K cutoff).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import multiprocessing as mp
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _workload(recipe: str, seed_index: int):
    from streaming_kv_cache_step_gb300 import workloads as W
    if recipe == "tiny":
        wl = W.tiny()
    elif recipe == "tiny_runs":
        wl = dataclasses.replace(W.tiny(), query_run=4)
    elif recipe == "long_context":
        wl = W.long_context()
    elif recipe == "streaming_paged":
        wl = W.streaming_paged()
    else:
        raise ValueError(recipe)
    return dataclasses.replace(wl, seed=W.DATA_SEED_BASE + 7000 + 131 * seed_index)


def _percentile(values, idx):
    """Rank percentile (0 = largest) of entries idx among values."""
    order = np.argsort(-values, kind="stable")
    rank = np.empty(values.size, np.int64)
    rank[order] = np.arange(values.size)
    return rank[idx] / max(values.size - 1, 1)


def run_stream(args):
    """One (recipe, seed, policy, slice) stream; returns the bridges' survival per step and
    the step-0 diagnostics."""
    recipe, seed_index, policy, sid, steps = args
    import torch
    import oracle
    from streaming_kv_cache_step_gb300 import workloads as W
    torch.set_num_threads(1)
    wl = _workload(recipe, seed_index)
    layer, s, h = wl.slice_coords(sid)
    cap = wl.capacity
    cache, q, over = W.slice_numpy_cache(wl, sid, capacity=cap)
    bridges = W.plant(wl, sid)["bridges"]
    walk = wl.walk_len if policy == "nexus" else 0
    mode = oracle.RESERVOIR if policy == "nexus" else oracle.TOPK
    philox = 0x9E3779B97F4A7C15 ^ (seed_index * 0x100000001B3)
    alive, diag = [], None
    for step in range(steps):
        if step > 0:
            W.append_tokens(wl, W.numpy_cache_as_torch(cache), step, sids=[sid],
                            slice_index={sid: 0})
            q = W.storage_to_numpy(W.to_storage(torch.as_tensor(W.query_rows(wl, sid, step)),
                                                wl.dtype)).reshape(q.shape)
        T = int(cache["lens"].reshape(-1)[0])
        params = dict(window=wl.window, walk_len=walk, mode=mode, seed=philox, step=step,
                      n_sink=wl.n_sink, n_recent=wl.n_recent, **over)
        if step == 0 and bridges.size:
            ref = oracle.evict_step(cache, q, dict(params, walk_len=wl.walk_len,
                                                   mode=oracle.RESERVOIR), mutate=False)
            pos0 = cache["pos"][0, 0, 0, :T]
            slot = np.searchsorted(pos0, bridges)
            B = int(over["budget"][0])
            diag = dict(pct_a=float(_percentile(ref["a"][0, :T], slot).mean()),
                        pct_w=float(_percentile(ref["w"][0, :T].astype(np.float64),
                                                slot).mean()),
                        cutoff=B / T)
        oracle.evict_step(cache, q, params, mutate=True)
        T = int(cache["lens"].reshape(-1)[0])
        present = np.isin(bridges, cache["pos"].reshape(-1)[:T])
        alive.append(float(present.mean()) if bridges.size else float("nan"))
    return dict(recipe=recipe, seed=seed_index, policy=policy, sid=sid, alive=alive, diag=diag)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--recipe", default="tiny")
    ap.add_argument("--seeds", type=int, default=32)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--slices", type=int, default=1, help="sampled slices per seed")
    ap.add_argument("--procs", type=int, default=os.cpu_count() or 1)
    a = ap.parse_args()
    wl0 = _workload(a.recipe, 0)
    steps = a.steps or wl0.steps
    rng = np.random.default_rng(12345)
    sids = sorted(rng.choice(wl0.n_slices, min(a.slices, wl0.n_slices), replace=False).tolist())
    jobs = [(a.recipe, sd, pol, sid, steps) for sd in range(a.seeds) for sid in sids
            for pol in ("nexus", "topk_a")]
    with mp.get_context("spawn").Pool(a.procs) as pool:
        res = pool.map(run_stream, jobs)
    curves = {p: np.array([r["alive"] for r in res if r["policy"] == p]) for p in ("nexus", "topk_a")}
    life = {p: curves[p].sum(1) for p in curves}           # steps survived per bridge
    diff = life["nexus"] - life["topk_a"]
    se = diff.std(ddof=1) / math.sqrt(diff.size) if diff.size > 1 else float("nan")
    diags = [r["diag"] for r in res if r["policy"] == "nexus" and r["diag"]]
    out = dict(recipe=a.recipe, seeds=a.seeds, slices=sids, steps=steps,
               survival={p: [round(float(x), 4) for x in curves[p].mean(0)] for p in curves},
               lifetime={p: round(float(life[p].mean()), 4) for p in life},
               paired_t=round(float(diff.mean() / se), 3) if se and se > 0 else None,
               bridge_pct_a=round(float(np.mean([d["pct_a"] for d in diags])), 4),
               bridge_pct_w=round(float(np.mean([d["pct_w"] for d in diags])), 4),
               budget_pct=round(float(np.mean([d["cutoff"] for d in diags])), 4))
    print(json.dumps(out))


if __name__ == "__main__":
    main()
