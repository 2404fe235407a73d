"""Pins of the oracle at block granularity (Nexus Sampling paper, §2.1 "Block
granularity" and Eq. (1): S = rownorm(BlockSum_b(softmax(Q K^T / sqrt(D)))) over
N_k = ceil(T_k / b) blocks; §2.2 Eqs. (2)-(5) over blocks, the tie-break ramp over the
block index; §5.1: b = 32), and of per-slice budgets (§10: a head-adaptive allocation
hands every head its own budget; the eviction step takes it as given).

Checked against the token-level oracle and closed forms: block scores are sums of token
scores where the method is linear (Eq. (3)), the walk takes inner products between block
rows (not token rows), and a step keeps whole blocks."""
import numpy as np
import pytest


def _rand(T, d=16, W=8, seed=0, scale=1.5):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((T, d)) * scale
    K[T // 3] *= 2.5
    return K, rng.standard_normal((W, d)) * scale


def _bsum(x, b):
    T = x.shape[-1]
    N = -(-T // b)
    pad = np.zeros(x.shape[:-1] + (N * b - T,))
    return np.concatenate([x, pad], axis=-1).reshape(x.shape[:-1] + (N, b)).sum(-1)


@pytest.mark.parametrize("T,b", [(256, 32), (300, 32), (100, 32), (33, 32), (31, 32),
                                 (250, 16), (97, 1)])
def test_block_rows_are_block_sums_of_token_rows(oracle_lib, T, b):
    K, Q = _rand(T, seed=T + b)
    tok = oracle_lib.slice_scores(K, Q, 3)
    blk = oracle_lib.block_scores(K, Q, 3, b)
    N = -(-T // b)
    assert blk["a"].shape == (N,)
    # BlockSum of Eq. (1), then rownorm (an identity on distributions up to rounding)
    assert np.allclose(blk["Pb"], _bsum(tok["P"], b), rtol=1e-12, atol=1e-15)
    assert np.allclose(blk["Pb"].sum(1), 1.0, atol=1e-14)
    # Eq. (3) is linear: a block's direct score is the sum of its tokens'
    assert np.allclose(blk["a"], _bsum(tok["a"], b), rtol=1e-12, atol=1e-15)
    assert abs(blk["a"].sum() - 1) < 1e-12
    assert abs(blk["ctilde"].sum() - 1) < 1e-12
    assert abs(blk["s"].sum() - 1.5) < 1e-12
    # Eq. (5): the ramp runs over the block index j / (N_k - 1)
    ramp = 1e-6 * (np.arange(N) / (N - 1) if N > 1 else np.zeros(1))
    assert np.array_equal(blk["w"], (blk["s"] + ramp).astype(np.float32))


def test_block_walk_uses_block_inner_products(oracle_lib):
    # H = 2 over block rows r1 (older), r2: gamma = (1, 1 + <r1, r2>) with the inner
    # product over blocks, c~ = (r1 + gamma_2 r2) / (1 + gamma_2). The token-level inner
    # product is smaller (it misses the cross-token terms inside a block), so a walk over
    # token rows summed afterwards gives a different c~.
    K, Q = _rand(320, seed=5)
    b = 32
    blk = oracle_lib.block_scores(K, Q, 2, b)
    r1, r2 = blk["Pb"][-2], blk["Pb"][-1]
    g2 = 1 + r1 @ r2
    assert np.allclose(blk["gamma"], [1.0, g2], atol=1e-14)
    assert np.allclose(blk["ctilde"], (r1 + g2 * r2) / (1 + g2), atol=1e-15)
    tok = oracle_lib.slice_scores(K, Q, 2)
    assert tok["gamma"][1] < g2 - 1e-6
    assert not np.allclose(_bsum(tok["ctilde"], b), blk["ctilde"], rtol=1e-6, atol=0)
    # H = 1: c~ is the newest block row itself
    one = oracle_lib.block_scores(K, Q, 1, b)
    assert np.allclose(one["ctilde"], blk["Pb"][-1], atol=1e-15)


def _slice_cache(T, d=32, W=8, G=2, seed=0, cap=None):
    rng = np.random.default_rng(seed)
    cap = cap or T
    k = np.zeros((1, 1, 1, cap, d), np.float32)
    k[0, 0, 0, :T] = rng.standard_normal((T, d)) * 1.5
    v = np.zeros_like(k)
    v[0, 0, 0, :T] = rng.standard_normal((T, d))
    pos = np.full((1, 1, 1, cap), -1, np.int32)
    pos[0, 0, 0, :T] = 5000 + 2 * np.arange(T)
    q = (rng.standard_normal((1, 1, G, W, d)) * 1.5).astype(np.float32)
    cache = dict(layers=1, seqs=1, kv_heads=1, group=G, head_dim=d, capacity=cap, k=k, v=v,
                 pos=pos, lens=np.array([[[T]]], np.int32))
    return cache, q


@pytest.mark.parametrize("T", [640, 650, 609])
def test_block_step_keeps_whole_blocks(oracle_lib, T):
    b, B, ns, nr = 32, 8, 1, 1          # units: blocks
    cache, q = _slice_cache(T, seed=T)
    k0, v0, p0 = (cache[n].copy() for n in ("k", "v", "pos"))
    params = dict(window=8, walk_len=3, n_sink=ns, n_recent=nr, budget=np.array([B], np.int32),
                  seed=77, step=3, seq_id_base=2, layer_id_base=1, block_size=b)
    out = oracle_lib.evict_step(cache, q, params, mutate=True)
    N = -(-T // b)
    keep = out["keep"][0, :B]
    assert np.all(np.diff(keep) > 0) and keep[0] == 0 and keep[-1] == N - 1
    rows = np.concatenate([np.arange(u * b, min(T, (u + 1) * b)) for u in keep])
    assert out["newlen"][0] == rows.size == cache["lens"][0, 0, 0]
    assert rows.size == (B - 1) * b + (T - (N - 1) * b)      # the newest block is partial
    for name, before in (("k", k0), ("v", v0), ("pos", p0)):
        assert np.array_equal(cache[name][0, 0, 0, :rows.size], before[0, 0, 0, rows]), name
    # the same survivors as the selection fed the block weights and block positions
    # (a block's position is its first token's), with the slice's Philox ids
    Kd = k0[0, 0, 0, :T].astype(np.float64)
    Qb = q[0, 0].astype(np.float64).mean(0)
    blk = oracle_lib.block_scores(Kd, Qb, 3, b)
    assert np.array_equal(out["w"][0, :N], blk["w"])
    bpos = p0[0, 0, 0, np.arange(N) * b]
    ref, _ = oracle_lib.select_slice(blk["w"], bpos, B, ns, nr, oracle_lib.RESERVOIR, 77, 3,
                                     1 * 1 + 0, 2)
    assert np.array_equal(keep, ref)


def test_block_step_identity_when_within_budget(oracle_lib):
    cache, q = _slice_cache(200, seed=1)
    params = dict(window=8, walk_len=3, n_sink=1, n_recent=1, budget=np.array([7], np.int32),
                  block_size=32)
    out = oracle_lib.evict_step(cache, q, params, mutate=True)
    assert out["newlen"][0] == 200 and np.array_equal(out["keep"][0, :7], np.arange(7))


def test_per_slice_budgets_override_the_sequence_budget(oracle_lib):
    # two sequences x three KV heads, every slice with its own budget
    rng = np.random.default_rng(4)
    L, S, Hk, G, d, W, T = 1, 2, 3, 2, 32, 8, 300
    k = rng.standard_normal((L, S, Hk, T, d)).astype(np.float32)
    cache = dict(layers=L, seqs=S, kv_heads=Hk, group=G, head_dim=d, capacity=T, k=k,
                 v=rng.standard_normal((L, S, Hk, T, d)).astype(np.float32),
                 pos=np.tile(np.arange(T, dtype=np.int32), (L, S, Hk, 1)),
                 lens=np.full((L, S, Hk), T, np.int32))
    q = rng.standard_normal((L, S, Hk * G, W, d)).astype(np.float32)
    sb = np.array([70, 120, 64, 250, 90, 300], np.int32)
    base = dict(window=W, walk_len=3, budget=np.array([100, 100], np.int32), seed=9)
    per = oracle_lib.evict_step(dict(cache), q, dict(base, slice_budget=sb), mutate=False)
    assert list(per["newlen"]) == list(np.minimum(sb, T))
    for sid in range(S * Hk):
        h, s = sid % Hk, sid // Hk
        keep, _ = oracle_lib.select_slice(per["w"][sid, :T], cache["pos"][0, s, h], int(sb[sid]),
                                          32, 32, oracle_lib.RESERVOIR, 9, 0, h, s)
        assert np.array_equal(per["keep"][sid, :keep.size], keep)
    same = oracle_lib.evict_step(dict(cache), q, dict(base, slice_budget=np.full(6, 100, np.int32)),
                                 mutate=False)
    seq = oracle_lib.evict_step(dict(cache), q, base, mutate=False)
    assert np.array_equal(same["keep"], seq["keep"])
