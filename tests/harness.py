"""Shared helpers of the GPU parity tests: run the library on a workload, run the oracle
on regenerated slices, and compare with the tolerances the acceptance bar fixes."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from streaming_kv_cache_step_gb300 import nexus
from streaming_kv_cache_step_gb300 import workloads as W

DEV = "cuda:0"
RTOL = 1e-3           # scores: bf16 inputs, fp32 accumulation, vs the fp64 oracle


def round_bf16(x: np.ndarray) -> np.ndarray:
    """The window query of a bf16 model is bf16: round (through binary32) to the nearest
    bfloat16, ties to even, by the bit-level rule; returns float64."""
    b = np.asarray(x, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def score_tol(ref: np.ndarray, T: int) -> np.ndarray:
    """|gpu - oracle| bound per entry: rtol 1e-3, plus 1e-3/T absolute for entries near 0."""
    return RTOL * np.abs(ref) + 1e-3 / max(T, 1)


class GpuRun:
    """A workload's step-0 cache on the GPU with its parameters, workspace and status word."""

    def __init__(self, wl: W.Workload, mode=nexus.MODE_RESERVOIR, walk_len=None, step=0):
        self.wl = wl
        self.dev = torch.device(DEV)
        self.d = W.make_cache(wl, self.dev)
        self.q = W.queries(wl, step, self.dev)
        self.cache = nexus.Cache.from_dict(self.d)
        sb = None if wl.slice_budget is None else torch.as_tensor(
            wl.slice_budget.astype(np.int32), device=self.dev)
        bmax = int(wl.budget.max() if sb is None else wl.slice_budget.max())
        self.params = nexus.Params(
            budget=self.d["budget"], budget_max=bmax, window=wl.window,
            walk_len=wl.walk_len if walk_len is None else walk_len, n_sink=wl.n_sink,
            n_recent=wl.n_recent, mode=mode, lam=wl.lam, eps_tie=wl.eps_tie,
            seed=wl.philox_seed, step=step, n_avg=wl.n_avg, block_size=wl.block_size,
            slice_budget=sb)
        self.ws = nexus.alloc_workspace(self.cache, self.params)
        self.status = nexus.new_status(self.dev)
        S, cap = self.cache.n_slices, wl.capacity
        self.keep = torch.full((S, cap), -1, dtype=torch.int32, device=self.dev)

    def lens(self) -> np.ndarray:
        return self.d["lens"].reshape(-1).cpu().numpy()

    def zero_status(self):
        self.status.zero_()

    def check_status(self, expect=0):
        torch.cuda.synchronize()
        got = int(self.status.item())
        assert got == expect, f"device status {got}"

    def slice_rows(self, name: str, sid: int, n: int) -> torch.Tensor:
        """First n rows (in slot order) of k, v or pos of one slice."""
        t = self.d[name]
        layer, s, h = self.wl.slice_coords(sid)
        if self.wl.page_size:
            ps = self.wl.page_size
            slots = torch.arange(n, device=self.dev)
            pages = self.d["block_table"][s].long()[slots // ps]
            return t[layer, pages, h, slots % ps]
        return t[layer, s, h, :n]


def oracle_params(wl: W.Workload, over: dict, mode=oracle.RESERVOIR, walk_len=None, step=0):
    return dict(window=wl.window, walk_len=wl.walk_len if walk_len is None else walk_len,
                n_sink=wl.n_sink, n_recent=wl.n_recent, mode=mode, lam=wl.lam,
                eps_tie=wl.eps_tie, seed=wl.philox_seed, step=step, n_avg=wl.n_avg,
                block_size=wl.block_size, **over)


def oracle_slice(wl: W.Workload, sid: int, mode=oracle.RESERVOIR, walk_len=None, step=0):
    """Oracle step on the regenerated step-0 slice (never on data from the GPU)."""
    c, q, over = W.slice_numpy_cache(wl, sid, step=step)
    ref = oracle.evict_step(c, q, oracle_params(wl, over, mode, walk_len, step), mutate=False)
    return c, q, over, ref


def compare_survivors(gpu_keep: np.ndarray, ref_keep: np.ndarray, kappa_ref: np.ndarray,
                      min_overlap: float = 0.995):
    """End-to-end bar: >= 99.5% overlap; every disagreement within 1e-3 of the cutoff key."""
    n = ref_keep.size
    assert gpu_keep.size == n
    inter = np.intersect1d(gpu_keep, ref_keep).size
    assert inter >= min_overlap * n, f"overlap {inter}/{n}"
    diff = np.setxor1d(gpu_keep, ref_keep)
    if diff.size:
        cand = kappa_ref[np.isfinite(kappa_ref)]
        kept_cand = kappa_ref[ref_keep][np.isfinite(kappa_ref[ref_keep])]
        cut = kept_cand.min() if kept_cand.size else 0.0
        for j in diff:
            assert abs(kappa_ref[j] - cut) <= 1e-3 * abs(cut), (j, kappa_ref[j], cut)
        del cand
    return inter / max(n, 1)


def slice_budget(wl, sid) -> int:
    s = wl.slice_coords(sid)[1]
    return int(wl.budget[s] if wl.slice_budget is None else wl.slice_budget[sid])


def unit_positions(pos, b):
    """Philox positions of the decision units: a block's is its first row's."""
    return np.ascontiguousarray(pos[::b])


def oracle_kappa(wl, sid, w32, pos, step=0, mode=oracle.RESERVOIR):
    """Keys of every unit (NaN for forced) from the oracle's own weights (w32 per unit,
    pos per row)."""
    layer, s, h = wl.slice_coords(sid)
    _, kappa = oracle.select_slice(w32, unit_positions(pos, wl.block_size), slice_budget(wl, sid),
                                   wl.n_sink, wl.n_recent, mode, wl.philox_seed, step,
                                   layer * wl.kv_heads + h, s, n_avg=wl.n_avg)
    return kappa
