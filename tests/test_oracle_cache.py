"""Pins of the oracle's whole-cache driver (the per-step loop over every (layer,
sequence, KV head) slice of a cache) against its single-slice pieces, fed by hand:

* the window query of a KV group is the mean of that group's G query heads (Nexus
  Sampling paper, §2.1: the window queries are "head-averaged representations";
  query head h*G + g belongs to KV head h), in the model's dtype: for a bf16 cache the
  mean rounded once to bf16 (here by a float32 bit-level rounding written
  independently of the oracle's);
* the Philox stream of a slice is indexed by head id (layer_id_base + l)*Hkv + h and
  sequence id seq_id_base + s (§2.3: the uniforms u_j of Eq. (6) are independent
  per candidate, so every slice draws from its own stream);
* a paged cache (rows scattered over a shuffled page pool through a block table) gives
  the same result as the same rows stored contiguously;
* the in-place compaction keeps, in order, the rows at the kept slots (§2.1: inference
  continues with K_S, V_S).

A mistake in the driver -- a query head taken as g*Hkv + h, a sum instead of a mean, a
Philox id built from the wrong coordinate, a page looked up for the wrong sequence --
changes at least one of the compared quantities.
"""
import numpy as np
import pytest

L, S, HKV, G, D, W, H = 2, 3, 2, 4, 64, 8, 3
CAP = 160
LENS = np.array([150, 97, 160], np.int32)
BUDGET = np.array([90, 80, 70], np.int32)
N_SINK, N_RECENT = 4, 6


def _bf16_bits(x):
    """Round binary32 to bfloat16 (nearest even), as uint16 bit patterns."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _decode(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _contiguous_cache(seed=0, dtype="bf16"):
    rng = np.random.default_rng(seed)
    kf = rng.standard_normal((L, S, HKV, CAP, D)).astype(np.float32)
    vf = rng.standard_normal((L, S, HKV, CAP, D)).astype(np.float32)
    # a few strong keys so that the attention rows are far from uniform
    kf[:, :, :, 40] *= 3.0
    kf[:, :, :, 77] *= 2.5
    qf = rng.standard_normal((L, S, HKV * G, W, D)).astype(np.float32) * 1.5
    if dtype == "bf16":
        k, v, q = _bf16_bits(kf), _bf16_bits(vf), _bf16_bits(qf)
    else:
        k, v, q = kf, vf, qf
    pos = np.full((L, S, HKV, CAP), -1, np.int32)
    for s in range(S):
        # absolute positions that differ between sequences and are not the slot index
        pos[:, s, :, :LENS[s]] = 1000 * (s + 1) + 3 * np.arange(LENS[s])
    lens = np.repeat(LENS[None, :, None], L, 0).repeat(HKV, 2).astype(np.int32)
    cache = dict(layers=L, seqs=S, kv_heads=HKV, group=G, head_dim=D, capacity=CAP,
                 k=k, v=v, pos=pos, lens=lens)
    return cache, q


def _paged_copy(cache, page_size, seed=1):
    """The same rows in a shuffled page pool [L][pages][Hkv][page][d]."""
    mp = CAP // page_size
    npages = S * mp + 5                      # a few pages nobody uses
    perm = np.random.default_rng(seed).permutation(npages).astype(np.int32)
    bt = perm[: S * mp].reshape(S, mp).copy()
    k = np.zeros((L, npages, HKV, page_size, D), cache["k"].dtype)
    v = np.zeros_like(k)
    pos = np.full((L, npages, HKV, page_size), -7, np.int32)
    for s in range(S):
        for p in range(mp):
            rows = slice(p * page_size, (p + 1) * page_size)
            k[:, bt[s, p]] = cache["k"][:, s, :, rows]
            v[:, bt[s, p]] = cache["v"][:, s, :, rows]
            pos[:, bt[s, p]] = cache["pos"][:, s, :, rows]
    out = dict(cache, k=k, v=v, pos=pos, lens=cache["lens"].copy(), page_size=page_size,
               num_pages=npages, max_pages_per_seq=mp, block_table=bt)
    return out


def _params(**over):
    p = dict(window=W, walk_len=H, n_sink=N_SINK, n_recent=N_RECENT, lam=0.5, eps_tie=1e-6,
             budget=BUDGET, seed=0x1234ABCD5678EF01, step=7, seq_id_base=11, layer_id_base=5)
    p.update(over)
    return p


def _slice_rows(cache, name, sid, n):
    h, s, l = sid % HKV, (sid // HKV) % S, sid // (HKV * S)
    t = cache[name]
    if cache.get("page_size", 0):
        ps = cache["page_size"]
        j = np.arange(n)
        return t[l, cache["block_table"][s][j // ps], h, j % ps]
    return t[l, s, h, :n]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_group_mean_query_and_slice_scores(oracle_lib, dtype):
    cache, q = _contiguous_cache(dtype=dtype)
    p = _params()
    out = oracle_lib.evict_step(cache, q, p, mutate=False)
    dec = _decode if dtype == "bf16" else (lambda a: a.astype(np.float64))
    for sid in range(L * S * HKV):
        h, s, l = sid % HKV, (sid // HKV) % S, sid // (HKV * S)
        T = int(LENS[s])
        K = dec(cache["k"][l, s, h, :T])
        # KV head h owns query heads h*G .. h*G + G - 1; its window query is their mean,
        # a tensor of the model's dtype (bf16: the mean rounded once to bf16)
        Qbar = dec(q[l, s, h * G:(h + 1) * G]).mean(axis=0)
        if dtype == "bf16":
            Qbar = _decode(_bf16_bits(Qbar))
        o = oracle_lib.slice_scores(K, Qbar, H, 0.5, 1e-6)
        # the same additions in the same order: bit-equal
        assert np.array_equal(out["a"][sid, :T], o["a"]), sid
        assert np.array_equal(out["w"][sid, :T], o["w"]), sid
        assert out["newlen"][sid] == min(T, int(BUDGET[s]))


def test_wrong_query_grouping_would_be_detected(oracle_lib):
    # the pin above separates the two plausible groupings on this cache: the mean over
    # heads g*Hkv + h gives visibly different scores from the mean over h*G + g
    cache, q = _contiguous_cache()
    l, s, h = 1, 2, 1
    T = int(LENS[s])
    K = _decode(cache["k"][l, s, h, :T])
    right = _decode(q[l, s, h * G:(h + 1) * G]).mean(axis=0)
    wrong = _decode(q[l, s, [g * HKV + h for g in range(G)]]).mean(axis=0)
    a_r = oracle_lib.slice_scores(K, right, H)["a"]
    a_w = oracle_lib.slice_scores(K, wrong, H)["a"]
    a_sum = oracle_lib.slice_scores(K, right * G, H)["a"]          # a sum, not a mean
    assert np.abs(a_r - a_w).max() > 1e-3 * a_r.max()
    assert np.abs(a_r - a_sum).max() > 1e-3 * a_r.max()


@pytest.mark.parametrize("mode", [0, 1])
def test_survivors_follow_the_slice_philox_ids(oracle_lib, mode):
    cache, q = _contiguous_cache(seed=3)
    p = _params(mode=mode)
    out = oracle_lib.evict_step(cache, q, p, mutate=False)
    for sid in range(L * S * HKV):
        h, s, l = sid % HKV, (sid // HKV) % S, sid // (HKV * S)
        T = int(LENS[s])
        head_id = (p["layer_id_base"] + l) * HKV + h
        seq_id = p["seq_id_base"] + s
        keep, _ = oracle_lib.select_slice(out["w"][sid, :T], cache["pos"][l, s, h, :T],
                                          int(BUDGET[s]), N_SINK, N_RECENT, mode, p["seed"],
                                          p["step"], head_id, seq_id)
        nl = int(out["newlen"][sid])
        assert np.array_equal(out["keep"][sid, :nl], keep), sid


def test_philox_ids_change_the_reservoir_draw(oracle_lib):
    # every id of the counter reaches the draw: another layer base, sequence base, step
    # or seed changes some slice's survivors (top-K mode ignores all of them)
    cache, q = _contiguous_cache(seed=4)
    base = oracle_lib.evict_step(cache, q, _params(), mutate=False)["keep"]
    for over in (dict(layer_id_base=6), dict(seq_id_base=12), dict(step=8),
                 dict(seed=0x1234ABCD5678EF02)):
        other = oracle_lib.evict_step(cache, q, _params(**over), mutate=False)["keep"]
        differs = [not np.array_equal(base[i], other[i]) for i in range(L * S * HKV)]
        assert sum(differs) >= L * S * HKV - 1, over
    t0 = oracle_lib.evict_step(cache, q, _params(mode=1), mutate=False)["keep"]
    t1 = oracle_lib.evict_step(cache, q, _params(mode=1, layer_id_base=6, seq_id_base=12,
                                                 step=8), mutate=False)["keep"]
    assert np.array_equal(t0, t1)


@pytest.mark.parametrize("page_size", [8, 16, 32])
def test_paged_layout_equals_contiguous(oracle_lib, page_size):
    cache, q = _contiguous_cache(seed=5)
    paged = _paged_copy(cache, page_size, seed=page_size)
    p = _params()
    a = oracle_lib.evict_step(cache, q, p, mutate=True)
    b = oracle_lib.evict_step(paged, q, p, mutate=True)
    for key in ("keep", "w", "a", "newlen"):
        assert np.array_equal(a[key], b[key]), key
    assert np.array_equal(cache["lens"], paged["lens"])
    for sid in range(L * S * HKV):
        nl = int(a["newlen"][sid])
        for name in ("k", "v", "pos"):
            assert np.array_equal(_slice_rows(cache, name, sid, nl),
                                  _slice_rows(paged, name, sid, nl)), (sid, name)


def test_paged_compaction_moves_the_kept_rows(oracle_lib):
    cache, q = _contiguous_cache(seed=6)
    paged = _paged_copy(cache, 16, seed=9)
    before = {n: paged[n].copy() for n in ("k", "v", "pos")}
    out = oracle_lib.evict_step(paged, q, _params(), mutate=True)
    bt = paged["block_table"]
    for sid in range(L * S * HKV):
        h, s, l = sid % HKV, (sid // HKV) % S, sid // (HKV * S)
        nl = int(out["newlen"][sid])
        keep = out["keep"][sid, :nl]
        for name in ("k", "v", "pos"):
            want = before[name][l, bt[s][keep // 16], h, keep % 16]
            assert np.array_equal(_slice_rows(paged, name, sid, nl), want), (sid, name)
        assert paged["lens"][l, s, h] == nl
    # the block table is not modified and pages outside every table are untouched
    unused = np.setdiff1d(np.arange(paged["num_pages"]), bt.reshape(-1))
    assert np.array_equal(paged["k"][:, unused], before["k"][:, unused])


def test_bf16_rounding_of_the_window_queries(oracle_lib):
    # the oracle's rounding of the head average (to 8 significant bits, ties to even,
    # binary32's exponent range) against the bit-level rule on binary32 inputs: random
    # values, exact halfway cases either side of even, subnormals, and the float32 range
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(20000) * 3,
                        rng.standard_normal(2000) * 1e-30,
                        rng.standard_normal(2000) * 1e-39,            # binary32 subnormals
                        rng.standard_normal(2000) * 1e30]).astype(np.float32)
    base = _bf16_bits(rng.standard_normal(4000).astype(np.float32))
    half = ((base.astype(np.uint32) << 16) | 0x8000).view(np.float32)  # exactly between two
    x = np.concatenate([x, half, -half, np.float32([0.0, -0.0, 1.0, 65504.0])])
    got = oracle_lib.round_bf16(x.astype(np.float64))
    want = _decode(_bf16_bits(x))
    assert np.array_equal(got, want)
    # ties went to the even neighbour, so a halfway value never rounds the same way twice
    ev = _bf16_bits(half)
    assert ((ev & 1) == 0).all()
