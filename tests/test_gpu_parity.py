"""GPU parity: the library's kernels, called through the C ABI, against the CPU oracle on
the same seeded inputs, at sizes the oracle finishes in seconds (several tiles, ragged
tails, paged and contiguous layouts, every dtype and window shape)."""
import numpy as np
import pytest
import torch

import oracle
from harness import (DEV, GpuRun, compare_survivors, oracle_kappa, oracle_slice, round_bf16,
                     score_tol)
from streaming_kv_cache_step_gb300 import nexus
from streaming_kv_cache_step_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _cases():
    paged_lens = np.array([1500, 900, 2048, 100], np.int32)
    return {
        "tiny_f32": W.tiny(),
        "gqa_ragged": W.shrink(W.llama3_8b_layer(), seqs=3, kv_heads=2,
                               lens=np.array([1000, 37, 700], np.int32), capacity=1024,
                               budget=np.array([300, 300, 128], np.int32), n_hubs=16),
        "paged": W.shrink(W.streaming_paged(4), lens=paged_lens, capacity=2048,
                          budget=np.maximum(64, paged_lens * 2 // 10).astype(np.int32)),
        "long_w64_h5": W.shrink(W.long_context(), seqs=1, kv_heads=2,
                                lens=np.array([1500], np.int32), capacity=1536,
                                budget=np.array([300], np.int32), n_hubs=8, n_bridges=8),
        "mixture": W.shrink(W.batch16_32layers(), layers=2, seqs=2, kv_heads=2,
                            lens=np.full(2, 777, np.int32), capacity=800,
                            budget=np.full(2, 160, np.int32)),
        # bf16 head_dim 64 on the tensor-core scorer (its 64-column K boxes, 8 stages)
        "bf16_d64": W.shrink(W.llama3_8b_layer(), head_dim=64, seqs=2, kv_heads=2,
                             lens=np.array([1200, 517], np.int32), capacity=1280,
                             budget=np.array([256, 200], np.int32), n_hubs=8),
        # page sizes other than 16: 8 (sixteen boxes per tile), 32, and 128 (one box per tile)
        "paged_ps8": W.shrink(W.streaming_paged(3), page_size=8, lens=np.array([1300, 77, 1024],
                              np.int32), capacity=1536, budget=np.array([260, 64, 204], np.int32)),
        "paged_ps32": W.shrink(W.streaming_paged(3), page_size=32,
                               lens=np.array([1500, 900, 33], np.int32), capacity=1536,
                               budget=np.array([300, 180, 64], np.int32)),
        "paged_ps128": W.shrink(W.streaming_paged(2), page_size=128,
                                lens=np.array([1900, 1280], np.int32), capacity=2048,
                                budget=np.array([380, 256], np.int32)),
        # a capacity that is not a multiple of four (the selection's scalar key staging)
        "cap_1023": W.shrink(W.llama3_8b_layer(), seqs=2, kv_heads=2,
                             lens=np.array([1023, 611], np.int32), capacity=1023,
                             budget=np.array([205, 150], np.int32), n_hubs=8),
        # walk lengths other than 0, 3 and 5 (the generic walk epilogue)
        "walk_h1_w16": W.shrink(W.llama3_8b_layer(), window=16, walk_len=1, seqs=1, kv_heads=2,
                                lens=np.array([1100], np.int32), capacity=1152,
                                budget=np.array([220], np.int32), n_hubs=8),
        "walk_h2": W.shrink(W.llama3_8b_layer(), walk_len=2, seqs=1, kv_heads=2,
                            lens=np.array([900], np.int32), capacity=1024,
                            budget=np.array([180], np.int32), n_hubs=8),
        "walk_h4": W.shrink(W.llama3_8b_layer(), walk_len=4, seqs=2, kv_heads=1,
                            lens=np.array([1000, 700], np.int32), capacity=1024,
                            budget=np.array([200, 140], np.int32), n_hubs=8),
        "walk_h4_w16": W.shrink(W.llama3_8b_layer(), window=16, walk_len=4, seqs=1,
                                kv_heads=2, lens=np.array([800], np.int32), capacity=896,
                                budget=np.array([160], np.int32), n_hubs=8),
    }


CASES = _cases()

# tensor-core scorer layouts: 0 the automatic choice (one pipeline per CTA at these sizes),
# 2 two pipelines per CTA (windows of up to 32 rows, bf16)
LAYOUTS = [0, 2]


@pytest.fixture
def layout(request):
    lay = request.param
    nexus.scorer_layout(lay)
    yield lay
    nexus.scorer_layout(0)


def _layout_case(name, lay):
    wl = CASES[name]
    if lay == 2 and (wl.window > 32 or wl.dtype != "bf16"):
        pytest.skip("two pipelines per CTA cover bf16 windows of up to 32 rows")
    return wl


def _check_layout_used(lay, wl=None):
    if lay == 2:
        assert nexus.scorer_config()["teams_per_cta"] == 2, nexus.scorer_config()
    if wl is not None:
        # bf16 caches run on the tensor-core scorer, fp32 ones on the CUDA-core scorer
        want = nexus.SCORER_TENSOR_CORE if wl.dtype == "bf16" else nexus.SCORER_CUDA_CORE
        assert nexus.last_scorer() == want, (nexus.last_scorer(), nexus.scorer_config())


def _decode(c, q, wl):
    k = c["k"][0, 0, 0, : int(c["lens"].reshape(-1)[0])]
    if k.dtype == np.uint16:
        k = (k.astype(np.uint32) << 16).view(np.float32)
        qf = (q.astype(np.uint32) << 16).view(np.float32)
    else:
        qf = q
    qbar = qf.reshape(wl.group, wl.window, wl.head_dim).astype(np.float64).mean(0)
    if k.dtype == np.float32 and wl.dtype == "bf16":
        qbar = round_bf16(qbar)         # a bf16 model's head average is bf16
    return k.astype(np.float64), qbar


@pytest.mark.parametrize("layout", LAYOUTS, indirect=True)
@pytest.mark.parametrize("name", list(CASES))
def test_scores_and_walk_match_oracle(name, layout):
    wl = _layout_case(name, layout)
    run = GpuRun(wl)
    S, cap, Wn = run.cache.n_slices, wl.capacity, wl.window
    a = torch.full((S, cap), -1.0, device=DEV)
    stats = torch.zeros((S, Wn, 2), device=DEV)
    w = torch.full((S, cap), -1.0, device=DEV)
    ct = torch.full((S, cap), -1.0, device=DEV)
    nexus.direct_scores(run.cache, run.q, run.params, a, stats, run.ws, run.status)
    nexus.walk(run.cache, run.q, run.params, w, ct, run.ws, run.status)
    run.check_status()
    _check_layout_used(layout, wl)
    a, stats, w, ct = a.cpu().numpy(), stats.cpu().numpy(), w.cpu().numpy(), ct.cpu().numpy()
    lens = run.lens()
    for sid in range(S):
        T = int(lens[sid])
        c, q, over, ref = oracle_slice(wl, sid)
        K, Qb = _decode(c, q, wl)
        o = oracle.slice_scores(K, Qb, wl.walk_len, wl.lam, wl.eps_tie)
        assert np.all(np.abs(a[sid, :T] - ref["a"][0, :T]) <= score_tol(ref["a"][0, :T], T))
        assert np.all(np.abs(w[sid, :T] - ref["w"][0, :T]) <= score_tol(ref["w"][0, :T], T))
        assert np.all(np.abs(ct[sid, :T] - o["ctilde"]) <= score_tol(o["ctilde"], T))
        assert np.allclose(stats[sid, :, 0], o["rowmax"], rtol=1e-5, atol=1e-4)
        assert np.allclose(stats[sid, :, 1], o["rowsum"], rtol=1e-4)
        assert abs(a[sid, :T].astype(np.float64).sum() - 1) < 1e-4
        assert (a[sid, T:] == -1).all() and (w[sid, T:] == -1).all()   # tail untouched


@pytest.mark.parametrize("mode", [nexus.MODE_RESERVOIR, nexus.MODE_TOPK])
@pytest.mark.parametrize("name", list(CASES))
def test_select_bitexact_on_oracle_weights(name, mode):
    wl = CASES[name]
    run = GpuRun(wl, mode=mode)
    S, cap = run.cache.n_slices, wl.capacity
    w_in = torch.zeros((S, cap), device=DEV)
    refs = []
    for sid in range(S):
        _, _, _, ref = oracle_slice(wl, sid, mode=mode)
        refs.append(ref)
        T = int(ref["w"].shape[1])       # the oracle's one-slice cache has capacity T
        w_in[sid, :T] = torch.as_tensor(ref["w"][0], device=DEV)
    nexus.reservoir_select(w_in, run.cache, run.params, run.keep, run.ws, run.status)
    run.check_status()
    keep = run.keep.cpu().numpy()
    for sid, ref in enumerate(refs):
        nl = int(ref["newlen"][0])
        assert np.array_equal(keep[sid, :nl], ref["keep"][0, :nl]), sid
        assert (keep[sid, nl:] == -1).all()


@pytest.mark.parametrize("name", list(CASES))
def test_compact_bitexact_on_oracle_keep(name, compact_kernel):
    wl = CASES[name]
    run = GpuRun(wl)
    S, cap = run.cache.n_slices, wl.capacity
    keep_in = torch.full((S, cap), -1, dtype=torch.int32, device=DEV)
    cs = []
    for sid in range(S):
        c, _, _, ref = oracle_slice(wl, sid)
        nl = int(ref["newlen"][0])
        keep_in[sid, :nl] = torch.as_tensor(ref["keep"][0, :nl], device=DEV)
        oracle.compact_slice(c, 0, ref["keep"][0, :nl])
        cs.append((c, nl))
    k_before = run.d["k"].clone()
    nexus.compact(run.cache, keep_in, run.params, run.ws, run.status)
    run.check_status()
    lens = run.lens()
    for sid, (c, nl) in enumerate(cs):
        assert lens[sid] == nl
        for name_ in ("k", "v", "pos"):
            got = W.storage_to_numpy(run.slice_rows(name_, sid, nl))
            assert np.array_equal(got, c[name_][0, 0, 0, :nl]), (sid, name_)
    if not wl.page_size:   # rows at or beyond the new length are untouched
        for sid, (c, nl) in enumerate(cs):
            layer, s, h = wl.slice_coords(sid)
            assert torch.equal(run.d["k"][layer, s, h, nl:], k_before[layer, s, h, nl:])


@pytest.mark.parametrize("layout", LAYOUTS, indirect=True)
@pytest.mark.parametrize("name", list(CASES))
def test_evict_step_end_to_end(name, layout):
    wl = _layout_case(name, layout)
    run = GpuRun(wl)
    S = run.cache.n_slices
    lens0 = run.lens()
    nexus.evict_step(run.cache, run.q, run.params, run.keep, run.ws, run.status)
    run.check_status()
    _check_layout_used(layout, wl)
    keep = run.keep.cpu().numpy()
    lens = run.lens()
    for sid in range(S):
        c, _, _, ref = oracle_slice(wl, sid)
        nl = int(ref["newlen"][0])
        T = int(lens0[sid])
        assert lens[sid] == nl
        kappa = oracle_kappa(wl, sid, ref["w"][0, :T], c["pos"][0, 0, 0, :T])
        compare_survivors(keep[sid, :nl], ref["keep"][0, :nl], kappa)
        # the compacted rows are exactly the original rows at the kept slots
        for name_ in ("k", "v", "pos"):
            got = W.storage_to_numpy(run.slice_rows(name_, sid, nl))
            assert np.array_equal(got, c[name_][0, 0, 0][keep[sid, :nl]]), (sid, name_)


def test_zero_walk_gives_direct_scores_and_budget_edges():
    # H = 0 reproduces the direct score; B = n_sink + n_recent keeps the forced slots only;
    # T <= B is an identity; T = 1 and T = 0 slices are handled.
    wl = W.shrink(W.llama3_8b_layer(), seqs=4, kv_heads=1, walk_len=0,
                  lens=np.array([600, 1, 0, 64], np.int32), capacity=640,
                  budget=np.array([64, 64, 64, 64], np.int32), n_hubs=4)
    run = GpuRun(wl)
    S, cap = run.cache.n_slices, wl.capacity
    a = torch.zeros((S, cap), device=DEV)
    w = torch.zeros((S, cap), device=DEV)
    nexus.direct_scores(run.cache, run.q, run.params, a, None, run.ws, run.status)
    nexus.walk(run.cache, run.q, run.params, w, None, run.ws, run.status)
    run.check_status()
    T = 600
    ramp = (np.arange(T) / (T - 1)).astype(np.float32) * np.float32(wl.eps_tie)
    assert np.allclose(w[0, :T].cpu().numpy(), a[0, :T].cpu().numpy() + ramp, rtol=1e-6,
                       atol=1e-9)
    assert a[1, 0].item() == pytest.approx(1.0, abs=1e-6)
    nexus.evict_step(run.cache, run.q, run.params, run.keep, run.ws, run.status)
    run.check_status()
    keep = run.keep.cpu().numpy()
    assert np.array_equal(keep[0, :64], np.r_[np.arange(32), np.arange(600 - 32, 600)])
    assert keep[1, 0] == 0 and np.array_equal(keep[3, :64], np.arange(64))
    assert list(run.lens()) == [64, 1, 0, 64]


def test_device_argument_faults_are_flagged_not_fatal():
    wl = W.shrink(W.llama3_8b_layer(), seqs=2, kv_heads=1, lens=np.array([500, 500], np.int32),
                  capacity=512, budget=np.array([100, 40], np.int32), n_hubs=4)
    run = GpuRun(wl)
    before = run.d["k"].clone()
    nexus.evict_step(run.cache, run.q, run.params, run.keep, run.ws, run.status)
    torch.cuda.synchronize()
    assert int(run.status.item()) & nexus.NX_DEV_BAD_BUDGET       # 40 < 32 + 32
    assert run.lens()[1] == 500                                    # that slice untouched
    assert torch.equal(run.d["k"][0, 1, 0], before[0, 1, 0])
    assert run.lens()[0] == 100                                    # the other one evicted
    run.zero_status()
    run.d["lens"].view(-1)[1] = 9999                               # > capacity
    nexus.evict_step(run.cache, run.q, run.params, run.keep, run.ws, run.status)
    torch.cuda.synchronize()
    assert int(run.status.item()) & nexus.NX_DEV_BAD_LEN


def test_bounded_wait_times_out_and_context_survives():
    # A compaction tile that never publishes "read done" (test hook) makes the later tiles
    # that depend on it give up after the bounded wait: NX_DEV_TIMEOUT, no hang, and the
    # next clean call on the same context succeeds.
    wl = W.shrink(W.llama3_8b_layer(), seqs=1, kv_heads=1, lens=np.array([8192], np.int32),
                  capacity=8192, budget=np.array([1638], np.int32), n_hubs=8)
    run = GpuRun(wl)
    _, _, _, ref = oracle_slice(wl, 0)
    keep_in = torch.full((1, wl.capacity), -1, dtype=torch.int32, device=DEV)
    keep_in[0, :1638] = torch.as_tensor(ref["keep"][0, :1638], device=DEV)
    lib = nexus.load()
    import ctypes
    rc = lib.nexus_debug_compact(ctypes.byref(run.cache.c_struct()),
                                 ctypes.c_void_p(keep_in.data_ptr()),
                                 ctypes.byref(run.params.c_struct()),
                                 ctypes.c_void_p(run.ws.data_ptr()), ctypes.c_size_t(run.ws.numel()),
                                 ctypes.c_void_p(run.status.data_ptr()),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                 ctypes.c_longlong(1))
    assert rc == 0
    torch.cuda.synchronize()
    assert int(run.status.item()) & nexus.NX_DEV_TIMEOUT
    # the context is still usable: a fresh, clean step succeeds
    run2 = GpuRun(wl)
    nexus.evict_step(run2.cache, run2.q, run2.params, run2.keep, run2.ws, run2.status)
    run2.check_status()
    assert run2.lens()[0] == 1638


@pytest.mark.parametrize("name", ["gqa_ragged", "paged", "long_w64_h5", "mixture", "bf16_d64",
                                  "walk_h4"])
def test_tensor_core_scorer_matches_cuda_core_scorer(name):
    # the bf16 shapes run on the tcgen05 scorer by default; the CUDA-core scorer is an
    # independent kernel on the same inputs: both must agree within the score tolerance
    wl = CASES[name]
    run = GpuRun(wl)
    S, cap = run.cache.n_slices, wl.capacity
    outs = []
    for simt in (False, True):
        nexus.force_simt(simt)
        try:
            w = torch.full((S, cap), -1.0, device=DEV)
            ct = torch.full((S, cap), -1.0, device=DEV)
            nexus.walk(run.cache, run.q, run.params, w, ct, run.ws, run.status)
            run.check_status()
            names = nexus.last_launch_names()
            cfg = nexus.scorer_config()
        finally:
            nexus.force_simt(False)
        assert ("score_tc" in names) != simt, (names, cfg)
        outs.append((w.cpu().numpy(), ct.cpu().numpy()))
    (w_tc, c_tc), (w_si, c_si) = outs
    lens = run.lens()
    for sid in range(S):
        T = int(lens[sid])
        assert np.all(np.abs(w_tc[sid, :T] - w_si[sid, :T]) <= 2 * score_tol(w_si[sid, :T], T))
        assert np.all(np.abs(c_tc[sid, :T] - c_si[sid, :T]) <= 2 * score_tol(c_si[sid, :T], T))


@pytest.mark.parametrize("name", ["gqa_ragged", "paged"])
def test_evict_step_replays_from_a_cuda_graph(name):
    """nexus_evict_step captured once in a CUDA graph and replayed on the restored cache
    gives, every replay, exactly what the eager call gives."""
    wl = CASES[name]
    run = GpuRun(wl)
    pristine = {k: run.d[k].clone() for k in ("k", "v", "pos", "lens")}

    def restore():
        for k, t in pristine.items():
            run.d[k].copy_(t)

    run.keep.fill_(-1)
    nexus.evict_step(run.cache, run.q, run.params, run.keep, run.ws, run.status)
    run.check_status()
    want = {k: run.d[k].clone() for k in pristine}
    want_keep = run.keep.clone()
    restore()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        nexus.evict_step(run.cache, run.q, run.params, run.keep, run.ws, run.status)
    for _ in range(3):
        restore()
        run.keep.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        run.check_status()
        assert torch.equal(run.keep, want_keep)
        for k in pristine:
            assert torch.equal(run.d[k], want[k]), k


# degenerate lengths: an empty slice, one and two rows (the ramp's T - 1 = 0 case), exactly
# the forced slots, one row past them, and a small eviction
EDGE = W.shrink(W.llama3_8b_layer(), seqs=6, kv_heads=1,
                lens=np.array([0, 1, 2, 64, 65, 200], np.int32), capacity=256,
                budget=np.array([64, 64, 64, 64, 64, 100], np.int32), n_hubs=4)


@pytest.mark.parametrize("layout", LAYOUTS, indirect=True)
def test_degenerate_lengths_end_to_end(layout):
    wl = EDGE
    run = GpuRun(wl)
    S, cap = run.cache.n_slices, wl.capacity
    lens0 = run.lens()
    w = torch.full((S, cap), -1.0, device=DEV)
    ct = torch.full((S, cap), -1.0, device=DEV)
    nexus.walk(run.cache, run.q, run.params, w, ct, run.ws, run.status)
    run.check_status()
    w = w.cpu().numpy()
    nexus.evict_step(run.cache, run.q, run.params, run.keep, run.ws, run.status)
    run.check_status()
    _check_layout_used(layout, wl)
    keep = run.keep.cpu().numpy()
    lens = run.lens()
    for sid in range(S):
        c, _, _, ref = oracle_slice(wl, sid)
        T, nl = int(lens0[sid]), int(ref["newlen"][0])
        assert lens[sid] == nl, (sid, lens[sid], nl)
        assert np.all(np.abs(w[sid, :T] - ref["w"][0, :T]) <= score_tol(ref["w"][0, :T], T))
        assert (w[sid, T:] == -1).all()
        if nl:
            kappa = oracle_kappa(wl, sid, ref["w"][0, :T], c["pos"][0, 0, 0, :T])
            compare_survivors(keep[sid, :nl], ref["keep"][0, :nl], kappa)
            for name_ in ("k", "v", "pos"):
                got = W.storage_to_numpy(run.slice_rows(name_, sid, nl))
                assert np.array_equal(got, c[name_][0, 0, 0][keep[sid, :nl]]), (sid, name_)


def _select_on_given_weights(wl, w_np, mode):
    """nexus_reservoir_select on caller-given weights against the oracle's select_slice,
    slice by slice (bit-exact)."""
    run = GpuRun(wl, mode=mode)
    S, cap = run.cache.n_slices, wl.capacity
    w_in = torch.zeros((S, cap), device=DEV)
    lens = run.lens()
    for sid in range(S):
        T = int(lens[sid])
        w_in[sid, :T] = torch.as_tensor(w_np[sid, :T], device=DEV)
    nexus.reservoir_select(w_in, run.cache, run.params, run.keep, run.ws, run.status)
    run.check_status()
    keep = run.keep.cpu().numpy()
    for sid in range(S):
        layer, s, h = wl.slice_coords(sid)
        T = int(lens[sid])
        pos = np.arange(T, dtype=np.int32)      # step-0 caches hold position j at slot j
        ref, _ = oracle.select_slice(w_np[sid, :T], pos, int(wl.budget[s]), wl.n_sink,
                                     wl.n_recent, mode, wl.philox_seed, 0,
                                     layer * wl.kv_heads + h, s)
        assert np.array_equal(keep[sid, :ref.size], ref), sid
        assert (keep[sid, ref.size:] == -1).all()


TIES = W.shrink(W.llama3_8b_layer(), seqs=3, kv_heads=2,
                lens=np.array([3000, 1999, 640], np.int32), capacity=3072,
                budget=np.array([600, 400, 128], np.int32), n_hubs=4)


def test_select_topk_heavily_tied_weights_bitexact():
    # weights on a grid of 20 values: the threshold key is tied many times over, so the
    # selection resolves the cutoff by the slot passes (the newer slot wins)
    rng = np.random.default_rng(21)
    S, cap = TIES.n_slices, TIES.capacity
    w = (rng.integers(0, 20, (S, cap)) / 7).astype(np.float32)
    _select_on_given_weights(TIES, w, nexus.MODE_TOPK)


def test_select_reservoir_with_zero_weights_bitexact():
    # zero weights give the key ln(u)/0 = -inf: when fewer positive-weight candidates
    # remain than the budget asks for, the -inf keys tie at the cutoff
    rng = np.random.default_rng(22)
    S, cap = TIES.n_slices, TIES.capacity
    w = rng.random((S, cap)).astype(np.float32) * 1e-3
    lens = TIES.lens
    for sid in range(S):
        s = TIES.slice_coords(sid)[1]
        T, B = int(lens[s]), int(TIES.budget[s])
        zero = rng.choice(np.arange(32, T - 32), T - 64 - (B - 64) // 2, replace=False)
        w[sid, zero] = 0.0      # only (B - 64) / 2 candidates keep a positive weight
    _select_on_given_weights(TIES, w, nexus.MODE_RESERVOIR)


# Few slices longer than one block's shared memory holds (over 48K units, two SMs per
# slice) take the multi-block selection: every slice split into co-resident segments that
# merge their digit histograms through global memory. Ragged lengths, a slice within its
# budget (kept whole), ties at the cutoff, reservoir and top-K.
MULTI = W.shrink(W.llama3_8b_layer(), seqs=3, kv_heads=2,
                 lens=np.array([60000, 52222, 800], np.int32), capacity=61440,
                 budget=np.array([12000, 10444, 900], np.int32), n_hubs=8)


@pytest.mark.parametrize("mode", [nexus.MODE_RESERVOIR, nexus.MODE_TOPK])
def test_select_multi_block_bitexact(mode):
    rng = np.random.default_rng(31)
    S, cap = MULTI.n_slices, MULTI.capacity
    w = (rng.random((S, cap)) * 1e-3 + 1e-6).astype(np.float32)
    _select_on_given_weights(MULTI, w, mode)
    assert nexus.last_launch_names()[-1] == "select_multi", nexus.last_launch_names()


def test_select_multi_block_heavily_tied_bitexact():
    rng = np.random.default_rng(32)
    S, cap = MULTI.n_slices, MULTI.capacity
    w = (rng.integers(0, 12, (S, cap)) / 5).astype(np.float32)
    _select_on_given_weights(MULTI, w, nexus.MODE_TOPK)
    assert nexus.last_launch_names()[-1] == "select_multi", nexus.last_launch_names()


@pytest.mark.parametrize("lens,window", [((160_000,), 32), ((170_000, 3000), 32),
                                         ((158_000,), 64), ((157_000,), 16)])
def test_slices_beyond_the_single_pass_residency_limit(lens, window):
    # Slices longer than the single tensor-core pass holds on chip (152 pipelines x 8 tiles x
    # 128 rows) take the two-pass tensor-core scorer (records first, then the finish): the
    # results are the oracle's, and the call says which scorer it used.
    lens = np.array(lens, np.int32)
    cap = int(lens.max())
    wl = W.shrink(W.llama3_8b_layer(), seqs=lens.size, kv_heads=1, lens=lens, capacity=cap,
                  budget=(lens // 5).astype(np.int32), n_hubs=16, window=window,
                  walk_len=5 if window == 64 else 3)
    run = GpuRun(wl)
    S = run.cache.n_slices
    w = torch.full((S, cap), -1.0, device=DEV)
    nexus.walk(run.cache, run.q, run.params, w, None, run.ws, run.status)
    run.check_status()
    assert nexus.last_scorer() == nexus.SCORER_TENSOR_CORE_TWO_PASS, nexus.scorer_config()
    assert nexus.last_launch_names()[1:3] == ["score_tc_records", "score_tc"]
    nexus.evict_step(run.cache, run.q, run.params, run.keep, run.ws, run.status)
    run.check_status()
    assert nexus.last_scorer() == nexus.SCORER_TENSOR_CORE_TWO_PASS
    w = w.cpu().numpy()
    keep = run.keep.cpu().numpy()
    for sid in range(S):
        T = int(lens[sid])
        c, _, _, ref = oracle_slice(wl, sid)
        assert np.all(np.abs(w[sid, :T] - ref["w"][0, :T]) <= score_tol(ref["w"][0, :T], T))
        nl = int(ref["newlen"][0])
        kappa = oracle_kappa(wl, sid, ref["w"][0, :T], c["pos"][0, 0, 0, :T])
        compare_survivors(keep[sid, :nl], ref["keep"][0, :nl], kappa)
        got = W.storage_to_numpy(run.slice_rows("k", sid, nl))
        assert np.array_equal(got, c["k"][0, 0, 0][keep[sid, :nl]])
