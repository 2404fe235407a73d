"""kv_compact_noalloc: the compaction entry point for callers that cannot allocate device
memory (it takes no workspace; its scratch is a static device array in the library).
Its output must equal kv_compact's, call after call. This file sorts last so that a
stop-at-first-failure run has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from harness import DEV, GpuRun, oracle_slice
from streaming_kv_cache_step_gb300 import nexus
from streaming_kv_cache_step_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc(run, keep, params):
    lib = nexus.load()
    lib.kv_compact_noalloc.argtypes = [ctypes.c_void_p] * 5
    lib.kv_compact_noalloc.restype = ctypes.c_int
    return lib.kv_compact_noalloc(ctypes.byref(run.cache.c_struct()),
                                  ctypes.c_void_p(keep.data_ptr()),
                                  ctypes.byref(params.c_struct()),
                                  ctypes.c_void_p(run.status.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _same_cache(a, b, wl):
    for name in ("k", "v", "pos", "lens"):
        assert torch.equal(a.d[name], b.d[name]), name


def test_noalloc_compaction_equals_kv_compact_twice_in_a_row():
    lens = np.array([3000, 1800, 700], np.int32)
    wl = W.shrink(W.llama3_8b_layer(), seqs=3, kv_heads=4, lens=lens, capacity=3072,
                  budget=np.array([700, 500, 700], np.int32), n_hubs=16)
    ref_run, na_run = GpuRun(wl), GpuRun(wl)       # two identical caches
    S, cap = ref_run.cache.n_slices, wl.capacity
    keep = torch.full((S, cap), -1, dtype=torch.int32, device=DEV)
    for sid in range(S):
        _, _, _, ref = oracle_slice(wl, sid)
        nl = int(ref["newlen"][0])
        keep[sid, :nl] = torch.as_tensor(ref["keep"][0, :nl], device=DEV)
    # call 1: the step-0 eviction
    nexus.compact(ref_run.cache, keep, ref_run.params, ref_run.ws, ref_run.status)
    assert _noalloc(na_run, keep, na_run.params) == nexus.NX_OK
    ref_run.check_status()
    na_run.check_status()
    _same_cache(ref_run, na_run, wl)
    # call 2: a second, smaller budget on the compacted caches (the static scratch still
    # holds call 1's flags and lengths)
    budget2 = torch.tensor([400, 300, 650], dtype=torch.int32, device=DEV)
    p2 = nexus.Params(budget=budget2, budget_max=650, window=wl.window)
    rng = np.random.default_rng(5)
    keep2 = torch.full((S, cap), -1, dtype=torch.int32, device=DEV)
    lens1 = ref_run.lens()
    b2 = budget2.cpu().numpy()
    for sid in range(S):
        s = wl.slice_coords(sid)[1]
        n = int(min(lens1[sid], b2[s]))
        keep2[sid, :n] = torch.as_tensor(np.sort(rng.choice(int(lens1[sid]), n, replace=False)),
                                         device=DEV)
    nexus.compact(ref_run.cache, keep2, p2, ref_run.ws, ref_run.status)
    assert _noalloc(na_run, keep2, p2) == nexus.NX_OK
    ref_run.check_status()
    na_run.check_status()
    _same_cache(ref_run, na_run, wl)
    assert list(na_run.lens()) == [min(int(lens1[i]), int(b2[wl.slice_coords(i)[1]]))
                                   for i in range(S)]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # 4096 slices x ceil(26214 / 32) tiles of flags need ~13 MiB > 4 MiB: rejected on the
    # host, nothing launched.
    lib = nexus.load()
    lib.kv_compact_noalloc.argtypes = [ctypes.c_void_p] * 5
    lib.kv_compact_noalloc.restype = ctypes.c_int
    c = nexus.CCache(1, 512, 8, 4, 128, 32768, 0, 0, 0, nexus.DTYPE_BF16, 1 << 20, 1 << 21,
                     1 << 22, 1 << 23, None)
    p = nexus.CParams(32, 3, 32, 32, 1, 0, 0.5, 1e-6, 1 << 24, 26214, 0, 0, 0, 1, 1, 0, None)
    rc = lib.kv_compact_noalloc(ctypes.byref(c), ctypes.c_void_p(1 << 25), ctypes.byref(p),
                                ctypes.c_void_p(1 << 26), None)
    assert rc == nexus.NX_ERR_WORKSPACE
