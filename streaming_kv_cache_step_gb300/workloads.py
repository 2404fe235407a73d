"""Seeded synthetic inputs for the eviction step.

This module serves both the CUDA path (tests, bench) and the CPU oracle (tests,
baseline). It holds none of the method's arithmetic: it only draws keys, values,
window queries, positions, lengths, budgets and page tables.

Bit-identical on CPU and GPU. Every cache element is a pure function of
(workload seed, tensor tag, slice id, absolute token position, feature index):

* A 32-bit integer hash (multiply-xorshift on int64 tensors, with no overflow)
  gives two words per element.
* The four 16-bit halves give uniforms u_i = (v_i + 1/2) / 2^16.
* z = (u_1 + u_2 + u_3 + u_4 - 2) * sqrt(3) is an Irwin-Hall approximation of
  N(0, 1). The sum is exact in binary32, so only the final multiply rounds.

Planted rows (hubs, bridges, chains), per-row scales and the window queries are
drawn with numpy on the host, then copied. So a sampled slice regenerated on the
CPU has the same bits as the full cache generated on the GPU.

The recipes follow the workloads the eviction step is measured on:

* tiny: one fp32 head with d = 64, 512 keys, 4 hubs and 8 bridges.
* llama3_8b_layer: a Llama-3-8B-shaped layer with 8192 keys and Zipf(1.1) hub mass.
* batch16_32layers: 16 sequences x 32 layers with 32768 keys drawn from a
  64-topic mixture.
* long_context: 4 sequences with 131072 keys, heavy-tailed (log-normal) key
  norms and 256 planted query->hub->bridge chains.
* streaming_paged: 256 ragged sequences with 16-token pages, evicted every
  decode token.
* prefill_256k: a one-shot eviction at the end of a 262144-token prefill.

Each recipe is described in full where it is defined below.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

M32 = 0xFFFFFFFF
_HMUL = 0x45D9F3B          # < 2^27: products with 32-bit words stay below 2^59
SQRT3 = float(np.float32(math.sqrt(3.0)))
DATA_SEED_BASE = 0x5EED0
PHILOX_SEED = 0x243F6A8885A308D3

TAG_K, TAG_V, TAG_TOPIC, TAG_SCALE = 1, 2, 3, 4


def _mix32_int(x: int) -> int:
    x &= M32
    x = (((x >> 16) ^ x) * _HMUL) & M32
    x = (((x >> 16) ^ x) * _HMUL) & M32
    return ((x >> 16) ^ x) & M32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    x = (((x >> 16) ^ x) * _HMUL) & M32
    x = (((x >> 16) ^ x) * _HMUL) & M32
    return (x >> 16) ^ x


def stream_key(seed: int, tag: int, slice_id: int) -> int:
    """Per (workload seed, tensor tag, slice) hash key, a 32-bit Python int."""
    k = _mix32_int(seed ^ 0x6A09E667)
    k = _mix32_int(k ^ (tag * 0x3C6EF372 & M32))
    return _mix32_int(k ^ (slice_id * 0x9E3779B1 & M32))


def hash_words(key: torch.Tensor, idx: torch.Tensor) -> torch.Tensor:
    """32-bit hash of int64 element indices (< 2^40) under int64 keys (< 2^32)."""
    lo = idx & M32
    hi = idx >> 32
    x = _mix32(lo ^ key)
    return _mix32(x ^ ((hi * 0x9E37 + 0x7F4A7C15) & M32))


def normal_from_hash(key: torch.Tensor, idx: torch.Tensor) -> torch.Tensor:
    """Irwin-Hall(4) approximately-normal binary32 values, exact-bit reproducible."""
    h1 = hash_words(key, 2 * idx)
    h2 = hash_words(key, 2 * idx + 1)
    s = None
    for part in (h1 & 0xFFFF, h1 >> 16, h2 & 0xFFFF, h2 >> 16):
        u = (part.to(torch.float32) + 0.5) / 65536.0
        s = u if s is None else s + u
    return (s - 2.0) * SQRT3


def uniform_int_from_hash(key: torch.Tensor, idx: torch.Tensor, n: int) -> torch.Tensor:
    return hash_words(key, idx) % n


def to_storage(x: torch.Tensor, dtype: str) -> torch.Tensor:
    """binary32 -> storage dtype (bf16 by round-to-nearest-even, or f32 unchanged)."""
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


def storage_to_numpy(x: torch.Tensor) -> np.ndarray:
    """Storage tensor -> numpy (bf16 as its uint16 bit pattern)."""
    x = x.detach().to("cpu").contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy()


# ---------------------------------------------------------------------------
# Workload description
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    layers: int
    seqs: int
    kv_heads: int
    group: int
    head_dim: int
    dtype: str                   # "bf16" or "f32"
    lens: np.ndarray             # int32 [S] initial cached tokens per sequence
    capacity: int                # rows per slice (multiple of page_size when paged)
    window: int
    walk_len: int
    budget: np.ndarray           # int32 [S]
    page_size: int = 0
    n_sink: int = 32
    n_recent: int = 32
    steps: int = 1
    append_per_step: int = 0     # tokens appended before every step after the first
    key_kind: str = "normal"     # normal | mixture | lognormal
    n_hubs: int = 0              # hub slots per slice (query targets)
    hub_norm: float = 1.0        # hub keys are scaled by this
    n_bridges: int = 0           # bridge slots per slice
    query_gain: float = 8.0      # gain of the hub direction in a window query
    query_run: int = 1           # window rows come in runs of this many rows on one pair
                                 # of adjacent hubs (alternating between the two), so
                                 # consecutive rows co-attend the pair's bridges
    zipf: float = 0.0            # > 0: hub rank of a query ~ Zipf(zipf)
    n_topics: int = 0
    lognormal_sigma: float = 0.0
    seed: int = DATA_SEED_BASE
    philox_seed: int = PHILOX_SEED
    lam: float = 0.5
    eps_tie: float = 1e-6
    n_avg: int = 1               # reservoir averaging count n of Eq. (6)
    block_size: int = 1          # b: rows per keep/evict decision (budgets count blocks)
    slice_budget: np.ndarray | None = None   # int32 [L*S*Hkv]: per-slice budgets (optional)

    @property
    def n_slices(self) -> int:
        return self.layers * self.seqs * self.kv_heads

    @property
    def q_heads(self) -> int:
        return self.kv_heads * self.group

    def slice_coords(self, sid: int):
        h = sid % self.kv_heads
        s = (sid // self.kv_heads) % self.seqs
        layer = sid // (self.kv_heads * self.seqs)
        return layer, s, h

    def max_pages_per_seq(self) -> int:
        return self.capacity // self.page_size if self.page_size else 0

    def rows_per_step0(self) -> int:
        return int(self.lens.astype(np.int64).sum()) * self.layers * self.kv_heads


def _rng(wl: Workload, *salt) -> np.random.Generator:
    return np.random.default_rng([wl.seed, *[int(x) & M32 for x in salt]])


# ---------------------------------------------------------------------------
# Planted structure (host, numpy) -- hubs, bridges, chains
# ---------------------------------------------------------------------------

def plant(wl: Workload, sid: int) -> dict:
    """Planted positions of one slice: hub and bridge absolute positions.

    Hubs and bridges sit at distinct positions outside the forced sink and
    recency slots of the first step.
    """
    return _memo("plant", wl, sid, lambda: _plant(wl, sid))


def _plant(wl: Workload, sid: int) -> dict:
    layer, s, h = wl.slice_coords(sid)
    T = int(wl.lens[s])
    lo, hi = wl.n_sink, max(wl.n_sink + 1, T - wl.n_recent)
    rng = _rng(wl, 11, sid)
    n = wl.n_hubs + wl.n_bridges
    n = min(n, hi - lo)
    picks = rng.choice(np.arange(lo, hi), size=n, replace=False) if n > 0 else np.zeros(0, int)
    hubs = np.sort(picks[: min(wl.n_hubs, n)])
    bridges = np.sort(picks[min(wl.n_hubs, n):])
    return dict(hubs=hubs.astype(np.int64), bridges=bridges.astype(np.int64))


def _base_rows(wl: Workload, sid: int, positions: np.ndarray) -> np.ndarray:
    """Unplanted binary32 key rows of one slice at the given absolute positions (host)."""
    pos = torch.as_tensor(np.asarray(positions, dtype=np.int64))
    return _key_rows(wl, torch.tensor([sid], dtype=torch.int64), pos[None, :],
                     "cpu")[0].numpy()


def _planted_rows(wl: Workload, sid: int) -> tuple[np.ndarray, np.ndarray]:
    """(positions, binary32 rows) that replace the base keys of one slice."""
    return _memo("rows", wl, sid, lambda: _planted_rows_uncached(wl, sid))


def _planted_rows_uncached(wl: Workload, sid: int) -> tuple[np.ndarray, np.ndarray]:
    pl = plant(wl, sid)
    d = wl.head_dim
    hubs, bridges = pl["hubs"], pl["bridges"]
    if hubs.size == 0 and bridges.size == 0:
        return np.zeros(0, np.int64), np.zeros((0, d), np.float32)
    base_h = _base_rows(wl, sid, hubs).astype(np.float64)
    rows, where = [], []
    rows.append(base_h * wl.hub_norm)
    where.append(hubs)
    if bridges.size:
        base_b = _base_rows(wl, sid, bridges).astype(np.float64)
        unit_h = base_h / np.linalg.norm(base_h, axis=1, keepdims=True)
        nb = bridges.size
        out = np.zeros((nb, d))
        for i in range(nb):
            if wl.key_kind == "lognormal":
                # chain i: bridge with cosine ~0.6 to its hub, normal norm.
                hv = unit_h[i % hubs.size]
                noise = base_b[i] - (base_b[i] @ hv) * hv
                noise /= max(np.linalg.norm(noise), 1e-12)
                out[i] = math.sqrt(d) * (0.6 * hv + 0.8 * noise)
            else:
                # bridge between hubs i and i+1: the mean direction plus noise.
                a, b = unit_h[i % hubs.size], unit_h[(i + 1) % hubs.size]
                dirn = (a + b) / max(np.linalg.norm(a + b), 1e-12)
                noise = base_b[i] / max(np.linalg.norm(base_b[i]), 1e-12)
                v = 0.8 * dirn + 0.6 * noise
                out[i] = math.sqrt(d) * v / np.linalg.norm(v)
        rows.append(out)
        where.append(bridges)
    return (np.concatenate(where).astype(np.int64),
            np.concatenate(rows).astype(np.float32))


# ---------------------------------------------------------------------------
# Keys and values (device-agnostic, exact-bit)
# ---------------------------------------------------------------------------

def _row_scale(wl: Workload, sids: torch.Tensor, pos: torch.Tensor, device) -> torch.Tensor | None:
    """Log-normal row norms exp(sigma * zeta), zeta ~ Irwin-Hall(4) drawn per (slice,
    position) from the hash. The sum m of four 16-bit words indexes a 4096-entry binary32
    table of exp(sigma * zeta(m)) built by numpy, so CPU and GPU get the same bits."""
    if wl.key_kind != "lognormal":
        return None
    keys = torch.tensor([stream_key(wl.seed, TAG_SCALE, int(s)) for s in sids.cpu().tolist()],
                        dtype=torch.int64, device=device)[:, None]
    h1 = hash_words(keys, 2 * pos)
    h2 = hash_words(keys, 2 * pos + 1)
    m = (h1 & 0xFFFF) + (h1 >> 16) + (h2 & 0xFFFF) + (h2 >> 16)        # [0, 4 * 65535]
    centers = (np.arange(4096, dtype=np.float64) * 64 + 31.5 + 2.0) / 65536.0
    table = np.exp(wl.lognormal_sigma * (centers - 2.0) * math.sqrt(3.0)).astype(np.float32)
    return torch.as_tensor(table, device=device)[m >> 6]


_CACHE: dict = {}


def _memo(kind: str, wl: Workload, sid: int, fn):
    key = (kind, sid, repr(sorted((k, v) for k, v in vars(wl).items()
                                  if not isinstance(v, np.ndarray))),
           wl.lens.tobytes())
    if key not in _CACHE:
        if len(_CACHE) > 200000:
            _CACHE.clear()
        _CACHE[key] = fn()
    return _CACHE[key]


def _centroids(wl: Workload, layer: int, h: int) -> np.ndarray:
    def make():
        rng = _rng(wl, 31, layer, h)
        return rng.standard_normal((wl.n_topics, wl.head_dim)).astype(np.float32)
    return _memo("mu", wl, layer * 65536 + h, make)


def _key_rows(wl: Workload, sids: torch.Tensor, pos: torch.Tensor, device) -> torch.Tensor:
    """Unplanted binary32 keys, shape [n_sid, n_pos, d], for absolute positions pos[n_sid, n_pos]."""
    d = wl.head_dim
    sids = sids.to(device)
    pos = pos.to(device)
    keys = torch.tensor([stream_key(wl.seed, TAG_K, int(s)) for s in sids.cpu().tolist()],
                        dtype=torch.int64, device=device)[:, None, None]
    kk = torch.arange(d, dtype=torch.int64, device=device)[None, None, :]
    idx = pos[:, :, None] * d + kk
    z = normal_from_hash(keys, idx)
    if wl.key_kind == "mixture":
        # token topic uniform over n_topics; k = (mu_topic + 0.5 z) / sqrt(1.25)
        tkeys = torch.tensor([stream_key(wl.seed, TAG_TOPIC, int(s)) for s in sids.cpu().tolist()],
                             dtype=torch.int64, device=device)[:, None]
        topic = uniform_int_from_hash(tkeys, pos, wl.n_topics)
        mus = []
        for s in sids.cpu().tolist():
            layer, _, h = wl.slice_coords(int(s))
            mus.append(_centroids(wl, layer, h))
        mu = torch.as_tensor(np.stack(mus), device=device)          # [n, topics, d]
        sel = torch.gather(mu, 1, topic[:, :, None].expand(-1, -1, d))
        z = (sel + z * 0.5) * float(np.float32(1.0 / math.sqrt(1.25)))
    sc = _row_scale(wl, sids, pos, device)
    if sc is not None:
        z = z * sc[:, :, None]
    return z


def value_rows(wl: Workload, sids: torch.Tensor, pos: torch.Tensor, device) -> torch.Tensor:
    d = wl.head_dim
    keys = torch.tensor([stream_key(wl.seed, TAG_V, int(s)) for s in sids.cpu().tolist()],
                        dtype=torch.int64, device=device)[:, None, None]
    kk = torch.arange(d, dtype=torch.int64, device=device)[None, None, :]
    return normal_from_hash(keys, pos.to(device)[:, :, None] * d + kk)


def key_rows(wl: Workload, sids, pos, device) -> torch.Tensor:
    """Binary32 keys (planted rows included) for slices sids at absolute positions pos."""
    sids = torch.as_tensor(sids, dtype=torch.int64)
    pos = torch.as_tensor(pos, dtype=torch.int64)
    z = _key_rows(wl, sids, pos, device)
    if wl.n_hubs or wl.n_bridges:
        pmin = pos.amin(dim=1).tolist() if pos.numel() else []
        for i, sid in enumerate(sids.tolist()):
            if pmin and pmin[i] >= int(wl.lens[wl.slice_coords(sid)[1]]):
                continue            # appended tokens are never planted
            where, rows = _planted_rows(wl, sid)
            if where.size == 0:
                continue
            p_np = pos[i].numpy()
            mask = np.isin(p_np, where)
            if mask.any():
                lut = {int(pw): r for r, pw in enumerate(where)}
                cols_np = np.nonzero(mask)[0]
                rsel = [lut[int(p_np[c])] for c in cols_np]
                cols = torch.as_tensor(cols_np, dtype=torch.int64, device=z.device)
                z[i, cols] = torch.as_tensor(rows[rsel], device=z.device)
    return z


# ---------------------------------------------------------------------------
# Window queries (host, numpy)
# ---------------------------------------------------------------------------

def query_rows(wl: Workload, sid: int, step: int) -> np.ndarray:
    """Binary32 window queries of one slice: [G, W, d] for the G query heads of the group."""
    layer, s, h = wl.slice_coords(sid)
    G, W, d = wl.group, wl.window, wl.head_dim
    rng = _rng(wl, 41, sid, step)
    noise = rng.standard_normal((G, W, d))
    if wl.key_kind == "mixture":
        mu = _centroids(wl, layer, h).astype(np.float64)
        q = np.zeros((G, W, d))
        for w in range(W):
            m = int(rng.integers(1, 4))
            topics = rng.choice(wl.n_topics, size=m, replace=False)
            q[:, w] = 0.5 * mu[topics].sum(0) / math.sqrt(m) + 0.5 * noise[:, w]
        return q.astype(np.float32)
    pl = plant(wl, sid)
    hubs = pl["hubs"]
    if hubs.size == 0:
        return noise.astype(np.float32)
    def make_unit():
        hk = key_rows(wl, [sid], hubs[None, :], "cpu")[0].numpy().astype(np.float64)
        return hk / np.linalg.norm(hk, axis=1, keepdims=True)
    unit = _memo("unit", wl, sid, make_unit)
    if wl.zipf > 0:
        ranks = np.arange(1, hubs.size + 1, dtype=np.float64)
        p = ranks ** (-wl.zipf)
        p /= p.sum()
        target = rng.choice(hubs.size, size=W, p=p)
    else:
        target = rng.integers(0, hubs.size, size=W)
    if wl.query_run > 1:
        # runs of rows on one adjacent hub pair (i, i + 1), alternating between the two
        for r0 in range(0, W, wl.query_run):
            i = int(rng.integers(0, hubs.size))
            for r in range(r0, min(W, r0 + wl.query_run)):
                target[r] = (i + (r - r0) % 2) % hubs.size
    q = noise + wl.query_gain * unit[target][None, :, :]
    return q.astype(np.float32)


def queries(wl: Workload, step: int, device, sids=None) -> torch.Tensor:
    """Window queries [L][S][Hq][W][d] in storage dtype (all slices), or [n][G][W][d] for sids."""
    G, W, d = wl.group, wl.window, wl.head_dim
    if sids is not None:
        q = np.stack([query_rows(wl, int(s), step) for s in sids])
        return to_storage(torch.as_tensor(q), wl.dtype).to(device)
    q = np.empty((wl.layers, wl.seqs, wl.kv_heads, G, W, d), np.float32)
    for sid in range(wl.n_slices):
        layer, s, h = wl.slice_coords(sid)
        q[layer, s, h] = query_rows(wl, sid, step)
    q = q.reshape(wl.layers, wl.seqs, wl.q_heads, W, d)
    return to_storage(torch.as_tensor(q), wl.dtype).to(device)


# ---------------------------------------------------------------------------
# Whole cache
# ---------------------------------------------------------------------------

def page_table(wl: Workload) -> tuple[np.ndarray, int]:
    """Shuffled page pool: block_table [S][max_pages] (-1 unused) and the pool size."""
    mp = wl.max_pages_per_seq()
    need = [int(math.ceil(wl.capacity / wl.page_size)) for _ in range(wl.seqs)]
    total = int(sum(need))
    perm = _rng(wl, 51).permutation(total).astype(np.int32)
    bt = np.full((wl.seqs, mp), -1, np.int32)
    o = 0
    for s in range(wl.seqs):
        bt[s, : need[s]] = perm[o: o + need[s]]
        o += need[s]
    return bt, total


def make_cache(wl: Workload, device, chunk_rows: int = 1 << 22) -> dict:
    """The full step-0 cache on `device`: token j of every slice at slot j, pos = j."""
    L, S, Hk, d, cap = wl.layers, wl.seqs, wl.kv_heads, wl.head_dim, wl.capacity
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    out = dict(layers=L, seqs=S, kv_heads=Hk, group=wl.group, head_dim=d, capacity=cap,
               page_size=wl.page_size, num_pages=0, max_pages_per_seq=wl.max_pages_per_seq())
    lens = np.repeat(wl.lens[None, :, None], L, 0).repeat(Hk, 2).astype(np.int32)
    if wl.page_size:
        bt, npages = page_table(wl)
        out["num_pages"] = npages
        out["block_table"] = torch.as_tensor(bt, device=device)
        k = torch.zeros((L, npages, Hk, wl.page_size, d), dtype=tdt, device=device)
        v = torch.zeros_like(k)
        pos = torch.full((L, npages, Hk, wl.page_size), -1, dtype=torch.int32, device=device)
    else:
        k = torch.zeros((L, S, Hk, cap, d), dtype=tdt, device=device)
        v = torch.zeros_like(k)
        pos = torch.full((L, S, Hk, cap), -1, dtype=torch.int32, device=device)
    for sid in range(wl.n_slices):
        layer, s, h = wl.slice_coords(sid)
        T = int(wl.lens[s])
        for j0 in range(0, T, max(1, chunk_rows // d)):
            j1 = min(T, j0 + max(1, chunk_rows // d))
            p = torch.arange(j0, j1, dtype=torch.int64)[None, :]
            kr = to_storage(key_rows(wl, [sid], p, device)[0], wl.dtype)
            vr = to_storage(value_rows(wl, torch.tensor([sid]), p, device)[0], wl.dtype)
            pr = torch.arange(j0, j1, dtype=torch.int32, device=device)
            if wl.page_size:
                ps = wl.page_size
                slots = torch.arange(j0, j1, device=device)
                pages = out["block_table"][s].long()[slots // ps]
                k[layer, pages, h, slots % ps] = kr
                v[layer, pages, h, slots % ps] = vr
                pos[layer, pages, h, slots % ps] = pr
            else:
                k[layer, s, h, j0:j1] = kr
                v[layer, s, h, j0:j1] = vr
                pos[layer, s, h, j0:j1] = pr
    out.update(k=k, v=v, pos=pos, lens=torch.as_tensor(lens, device=device),
               budget=torch.as_tensor(wl.budget.astype(np.int32), device=device))
    return out


def slice_numpy_cache(wl: Workload, sid: int, positions=None, step: int = 0,
                      capacity: int | None = None) -> tuple[dict, np.ndarray, dict]:
    """A one-slice contiguous numpy cache (oracle input) holding `positions` in order,
    with room for `capacity` rows (default: exactly the positions given).

    Returns (cache, queries [1][1][G][W][d] storage-dtype numpy, params overrides with
    seq_id_base / layer_id_base so the Philox stream matches the full cache).
    """
    layer, s, h = wl.slice_coords(sid)
    if positions is None:
        positions = np.arange(int(wl.lens[s]))
    positions = np.asarray(positions, dtype=np.int64)
    T = positions.size
    cap = max(T, 1) if capacity is None else max(capacity, T, 1)
    kr = to_storage(key_rows(wl, [sid], positions[None, :], "cpu")[0], wl.dtype)
    vr = to_storage(value_rows(wl, torch.tensor([sid]), torch.as_tensor(positions)[None, :], "cpu")[0],
                    wl.dtype)
    k = np.zeros((1, 1, 1, cap, wl.head_dim), dtype=np.uint16 if wl.dtype == "bf16" else np.float32)
    v = np.zeros_like(k)
    k[0, 0, 0, :T] = storage_to_numpy(kr)
    v[0, 0, 0, :T] = storage_to_numpy(vr)
    pos = np.full((1, 1, 1, cap), -1, np.int32)
    pos[0, 0, 0, :T] = positions
    cache = dict(layers=1, seqs=1, kv_heads=1, group=wl.group, head_dim=wl.head_dim, capacity=cap,
                 k=k, v=v, pos=pos, lens=np.array([[[T]]], np.int32))
    qn = storage_to_numpy(to_storage(torch.as_tensor(query_rows(wl, sid, step)), wl.dtype))
    qn = qn.reshape(1, 1, wl.group, wl.window, wl.head_dim)
    B = wl.budget[s] if wl.slice_budget is None else wl.slice_budget[sid]
    over = dict(seq_id_base=s, layer_id_base=layer * wl.kv_heads + h,
                budget=np.array([B], np.int32))
    return cache, qn, over


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def tiny() -> Workload:
    """One fp32 head (G = 1, d = 64), 512 keys ~ N(0,1); 4 hubs with norm x4 and 8 bridges
    along the mean direction of two adjacent hubs; 16 window queries aimed at hubs with
    gain 2 (hub logit ~8); B = 128, H = 3; 10 steps refilling to 512."""
    return Workload(name="tiny", layers=1, seqs=1, kv_heads=1, group=1, head_dim=64, dtype="f32",
                    lens=np.array([512], np.int32), capacity=512, window=16, walk_len=3,
                    budget=np.array([128], np.int32), steps=10, append_per_step=384,
                    n_hubs=4, hub_norm=4.0, n_bridges=8, query_gain=2.0,
                    seed=DATA_SEED_BASE + 0)


def llama3_8b_layer() -> Workload:
    """One Llama-3-8B-shaped layer: 32 q / 8 kv heads, d = 128 bf16, batch 1, 8192 keys
    ~ N(0,1), 64 hub positions per head; each window query aims at a hub whose rank is
    Zipf(1.1); W = 32, B = 1638 (80% evicted), H = 3; evict every 64 decode tokens."""
    return Workload(name="llama3_8b_layer", layers=1, seqs=1, kv_heads=8, group=4, head_dim=128,
                    dtype="bf16", lens=np.array([8192], np.int32), capacity=8192, window=32,
                    walk_len=3, budget=np.array([1638], np.int32), steps=21, append_per_step=64,
                    n_hubs=64, query_gain=8.0, zipf=1.1, seed=DATA_SEED_BASE + 1)


def batch16_32layers() -> Workload:
    """16 sequences x 32 layers x (32 q / 8 kv heads, d = 128 bf16), 32768 keys per slice
    from a mixture of 64 topic centroids; queries near 1-3 centroids; W = 32, B = 6554,
    H = 3."""
    return Workload(name="batch16_32layers", layers=32, seqs=16, kv_heads=8, group=4,
                    head_dim=128, dtype="bf16", lens=np.full(16, 32768, np.int32),
                    capacity=32768, window=32, walk_len=3, budget=np.full(16, 6554, np.int32),
                    key_kind="mixture", n_topics=64, seed=DATA_SEED_BASE + 2)


def long_context() -> Workload:
    """4 sequences, 32 q / 8 kv heads, d = 128 bf16, 131072 keys with log-normal norms
    (heavy-tailed attention), 32 planted chains per head (256 per sequence): a hub and a
    bridge at cosine 0.6 to it; each window row aims at one chain's hub. W = 64,
    B = 26214, H = 5, 50 steps."""
    return Workload(name="long_context", layers=1, seqs=4, kv_heads=8, group=4, head_dim=128,
                    dtype="bf16", lens=np.full(4, 131072, np.int32), capacity=131072, window=64,
                    walk_len=5, budget=np.full(4, 26214, np.int32), steps=50,
                    append_per_step=131072 - 26214, key_kind="lognormal", lognormal_sigma=0.5,
                    n_hubs=32, hub_norm=1.5, n_bridges=32, query_gain=8.0,
                    seed=DATA_SEED_BASE + 3)


def streaming_paged(n_seqs: int = 256) -> Workload:
    """256 sequences with lengths ~ U[1024, 65536], 16-token pages from a shuffled pool,
    8 kv heads (G = 4), d = 128 bf16, W = 16, H = 3, B = floor(0.2 len); step 0 evicts to
    B, then each of 199 steps appends one token and evicts back to B; 4 hubs and 16
    bridges per head."""
    rng = np.random.default_rng([DATA_SEED_BASE + 4, 61])
    lens = rng.integers(1024, 65537, size=n_seqs).astype(np.int32)
    return Workload(name="streaming_paged", layers=1, seqs=n_seqs, kv_heads=8, group=4,
                    head_dim=128, dtype="bf16", lens=lens, capacity=65536, window=16,
                    walk_len=3, budget=(lens * 2 // 10).astype(np.int32), page_size=16,
                    steps=200, append_per_step=1, n_hubs=4, hub_norm=4.0, n_bridges=16,
                    query_gain=2.0, seed=DATA_SEED_BASE + 4)


def prefill_256k() -> Workload:
    """One-shot eviction at the end of a long prefill (the paper's §2.1 streaming view: a
    long prompt can trigger one eviction when prefill ends): 2 sequences x 8 kv heads
    (32 q heads), d = 128 bf16, 262144 prompt tokens per slice, the window being the last
    32 prompt rows, H = 3, keep 20% (B = 52428), one step; 64 Zipf(1.1) hubs per head as
    in the Llama layer. Longer than one on-chip pass of the tensor-core scorer."""
    return Workload(name="prefill_256k", layers=1, seqs=2, kv_heads=8, group=4, head_dim=128,
                    dtype="bf16", lens=np.full(2, 262144, np.int32), capacity=262144,
                    window=32, walk_len=3, budget=np.full(2, 52428, np.int32), steps=1,
                    n_hubs=64, query_gain=8.0, zipf=1.1, seed=DATA_SEED_BASE + 5)


def batch16_1layer() -> Workload:
    """One layer of the 16-sequence batch (128 slices, 1 GiB of keys): a profiling case
    larger than L2 that a counter capture replays quickly."""
    return dataclasses.replace(batch16_32layers(), name="batch16_1layer", layers=1)


WORKLOADS = {
    "tiny": tiny,
    "llama3_8b_layer": llama3_8b_layer,
    "batch16_32layers": batch16_32layers,
    "long_context": long_context,
    "streaming_paged": streaming_paged,
    "prefill_256k": prefill_256k,
    "batch16_1layer": batch16_1layer,
}


def shrink(wl: Workload, **kw) -> Workload:
    """A smaller copy of a workload (for oracle-sized tests)."""
    return dataclasses.replace(wl, **kw)


# ---------------------------------------------------------------------------
# Streaming: fresh tokens between eviction steps
# ---------------------------------------------------------------------------

def first_new_position(wl: Workload, s: int, step: int) -> int:
    """Absolute position of the first token appended before `step` (step >= 1)."""
    return int(wl.lens[s]) + (step - 1) * wl.append_per_step


def append_tokens(wl: Workload, cache: dict, step: int, sids=None, slice_index=None) -> None:
    """Append `append_per_step` fresh tokens to every listed slice (in place).

    ``cache`` holds torch tensors (any device) in the layout of ``make_cache`` or,
    with ``slice_index`` = {sid: row in the cache}, one-slice-per-row contiguous
    caches such as the oracle's. New tokens go to slots len .. len + n - 1 with the
    next absolute positions; their keys and values are the workload's own rows.
    """
    n = wl.append_per_step
    if n <= 0:
        return
    k, v, pos, lens = cache["k"], cache["v"], cache["pos"], cache["lens"]
    dev = k.device
    sids = range(wl.n_slices) if sids is None else sids
    lens_flat = lens.reshape(-1)
    for sid in sids:
        layer, s, h = wl.slice_coords(int(sid))
        row = int(sid) if slice_index is None else slice_index[int(sid)]
        cur = int(lens_flat[row])
        if cur + n > wl.capacity:
            raise ValueError("append would exceed the slice capacity")
        p0 = first_new_position(wl, s, step)
        p = torch.arange(p0, p0 + n, dtype=torch.int64)[None, :]
        kr = to_storage(key_rows(wl, [int(sid)], p, dev)[0], wl.dtype)
        vr = to_storage(value_rows(wl, torch.tensor([int(sid)]), p, dev)[0], wl.dtype)
        pr = torch.arange(p0, p0 + n, dtype=torch.int32, device=dev)
        slots = torch.arange(cur, cur + n, device=dev)
        if slice_index is None and wl.page_size:
            ps = wl.page_size
            pages = cache["block_table"][s].long()[slots // ps]
            k[layer, pages, h, slots % ps] = kr.to(k.dtype)
            v[layer, pages, h, slots % ps] = vr.to(v.dtype)
            pos[layer, pages, h, slots % ps] = pr
        elif slice_index is None:
            k[layer, s, h, cur:cur + n] = kr.to(k.dtype)
            v[layer, s, h, cur:cur + n] = vr.to(v.dtype)
            pos[layer, s, h, cur:cur + n] = pr
        else:
            kf = k.reshape(-1, k.shape[-2], k.shape[-1])
            vf = v.reshape(-1, v.shape[-2], v.shape[-1])
            pf = pos.reshape(-1, pos.shape[-1])
            kf[row, cur:cur + n] = kr.to(k.dtype)
            vf[row, cur:cur + n] = vr.to(v.dtype)
            pf[row, cur:cur + n] = pr
        lens_flat[row] = cur + n


def append_tokens_all(wl: Workload, cache: dict, step: int) -> None:
    """append_tokens for every slice of a make_cache cache at once (same bits)."""
    n = wl.append_per_step
    if n <= 0:
        return
    batch = max(1, (1 << 26) // (n * wl.head_dim))     # bound the hash temporaries
    k, v, pos, lens = cache["k"], cache["v"], cache["pos"], cache["lens"]
    dev = k.device
    lens_flat = lens.reshape(-1)
    ns = wl.n_slices
    sids = np.arange(ns)
    s_of = (sids // wl.kv_heads) % wl.seqs
    l_of = sids // (wl.kv_heads * wl.seqs)
    h_of = sids % wl.kv_heads
    p0 = wl.lens[s_of].astype(np.int64) + (step - 1) * n
    ar = torch.arange(n, device=dev)
    if int(lens_flat.max()) + n > wl.capacity:
        raise ValueError("append would exceed the slice capacity")
    for b0 in range(0, ns, batch):
        b1 = min(ns, b0 + batch)
        P = torch.as_tensor(p0[b0:b1, None] + np.arange(n)[None, :])
        kr = to_storage(key_rows(wl, sids[b0:b1], P, dev), wl.dtype).to(k.dtype)
        vr = to_storage(value_rows(wl, torch.as_tensor(sids[b0:b1]), P, dev), wl.dtype).to(v.dtype)
        pr = P.to(device=dev, dtype=torch.int32)
        slots = lens_flat[b0:b1].long()[:, None] + ar[None, :]
        li = torch.as_tensor(l_of[b0:b1], device=dev)[:, None].expand(-1, n)
        hi = torch.as_tensor(h_of[b0:b1], device=dev)[:, None].expand(-1, n)
        si = torch.as_tensor(s_of[b0:b1], device=dev)[:, None].expand(-1, n)
        if wl.page_size:
            ps = wl.page_size
            pages = cache["block_table"].long()[si, slots // ps]
            k[li, pages, hi, slots % ps] = kr
            v[li, pages, hi, slots % ps] = vr
            pos[li, pages, hi, slots % ps] = pr
        else:
            k[li, si, hi, slots] = kr
            v[li, si, hi, slots] = vr
            pos[li, si, hi, slots] = pr
        lens_flat[b0:b1] += n


def numpy_cache_as_torch(cache: dict) -> dict:
    """Torch CPU views (shared memory) of a numpy cache dict, bf16 bits viewed as bf16."""
    out = dict(cache)
    for name in ("k", "v"):
        a = cache[name]
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        out[name] = t.view(torch.bfloat16) if a.dtype == np.uint16 else t
    for name in ("pos", "lens"):
        out[name] = torch.from_numpy(cache[name])
    return out
