"""CPU oracle for one Nexus Sampling eviction step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference arm may import this package. The product path (the CUDA library and
its binding) never does; the two share no code.

The arithmetic lives in ``nexus_oracle.c`` (plain loops, doubles for the
scores, an exactly specified binary32 key path). This module compiles it with
gcc and marshals numpy arrays through ctypes. Every function follows
"Forget Without Compromise: Nexus Sampling for Streaming KV-Cache Eviction Under
Fixed Budgets": §2.1 Eq. (1) (block size b = 1, or b > 1 with BlockSum and
rownorm), §2.2 Eqs. (2)-(5), §2.3 Eq. (6) (n = 1: Efraimidis & Spirakis (IPL
2006) keys; n > 1: the n-averaged priority in the log domain), plus Salmon et al.
(SC'11) for Philox4x32-10 and Cody & Waite (1980) argument reduction for the
specified binary32 logarithm and exponential.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nexus_oracle.c")
_LIB = os.path.join(_HERE, "libnexus_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
RESERVOIR, TOPK = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libnexus_oracle.so`` (gcc, OpenMP, no FP contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", _LIB + ".tmp", _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            c_p = ctypes.c_void_p
            lib.nxo_slice_scores.argtypes = [ctypes.c_int] * 4 + [ctypes.c_double] * 2 + [c_p] * 10
            lib.nxo_slice_scores.restype = ctypes.c_int
            lib.nxo_philox4x32_10.argtypes = [c_p, c_p, c_p]
            lib.nxo_uniform.argtypes = [ctypes.c_uint32]
            lib.nxo_uniform.restype = ctypes.c_float
            lib.nxo_ln_spec.argtypes = [ctypes.c_float]
            lib.nxo_ln_spec.restype = ctypes.c_float
            lib.nxo_ln_spec_many.argtypes = [ctypes.c_int64, c_p, c_p]
            lib.nxo_exp_spec.argtypes = [ctypes.c_float]
            lib.nxo_exp_spec.restype = ctypes.c_float
            lib.nxo_exp_spec_many.argtypes = [ctypes.c_int64, c_p, c_p]
            lib.nxo_round_bf16_many.argtypes = [ctypes.c_int64, c_p, c_p]
            lib.nxo_block_scores.argtypes = ([ctypes.c_int] * 5 + [ctypes.c_double] * 2
                                             + [c_p] * 8)
            lib.nxo_block_scores.restype = ctypes.c_int
            lib.nxo_reservoir_key_n.argtypes = [ctypes.c_float, ctypes.c_int32, ctypes.c_uint64,
                                                ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                                ctypes.c_int]
            lib.nxo_reservoir_key_n.restype = ctypes.c_float
            lib.nxo_philox_many.argtypes = [ctypes.c_int64, c_p, c_p, c_p]
            lib.nxo_reservoir_key.argtypes = [ctypes.c_float, ctypes.c_int32, ctypes.c_uint64,
                                              ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
            lib.nxo_reservoir_key.restype = ctypes.c_float
            lib.nxo_select_slice.argtypes = ([ctypes.c_int, c_p, c_p] + [ctypes.c_int] * 4
                                             + [ctypes.c_uint64] + [ctypes.c_uint32] * 3
                                             + [ctypes.c_int, c_p, c_p])
            lib.nxo_select_slice.restype = ctypes.c_int
            lib.nxo_evict_step.argtypes = [c_p, c_p, c_p, ctypes.c_int, c_p, c_p, c_p, c_p, c_p,
                                           ctypes.c_int, ctypes.c_int]
            lib.nxo_evict_step.restype = ctypes.c_int
            lib.nxo_compact_slice.argtypes = [c_p, ctypes.c_int, c_p, ctypes.c_int]
            lib.nxo_compact_slice.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# Single-slice pieces
# --------------------------------------------------------------------------

def slice_scores(K, Qbar, walk_len, lam=0.5, eps_tie=1e-6):
    """Eqs. (1)-(5) for one slice at block size 1, in double.

    K: (T, d) keys; Qbar: (W, d) window queries. Returns a dict with P (W, T),
    a, ctilde, s (double, length T), w (binary32), rowmax, rowsum (W,), gamma (H,).
    """
    lib = _load()
    K = np.ascontiguousarray(K, dtype=np.float64)
    Qbar = np.ascontiguousarray(Qbar, dtype=np.float64)
    T, d = K.shape
    W = Qbar.shape[0]
    out = dict(P=np.zeros((W, T)), a=np.zeros(T), ctilde=np.zeros(T), s=np.zeros(T),
               w=np.zeros(T, np.float32), rowmax=np.zeros(W), rowsum=np.zeros(W),
               gamma=np.zeros(max(walk_len, 1)))
    rc = lib.nxo_slice_scores(T, d, W, walk_len, lam, eps_tie, _ptr(K), _ptr(Qbar),
                              _ptr(out["P"]), _ptr(out["a"]), _ptr(out["ctilde"]), _ptr(out["s"]),
                              _ptr(out["w"]), _ptr(out["rowmax"]), _ptr(out["rowsum"]),
                              _ptr(out["gamma"]))
    if rc != 0:
        raise ValueError("nxo_slice_scores rejected its arguments")
    out["gamma"] = out["gamma"][:walk_len]
    return out


def block_scores(K, Qbar, walk_len, block, lam=0.5, eps_tie=1e-6):
    """Eq. (1) with BlockSum over blocks of ``block`` slots and rownorm, then Eqs.
    (2)-(5) over the N_k = ceil(T / block) blocks, in double. Returns a dict with Pb
    (W, N_k), a, ctilde, s (double), w (binary32), gamma (H,)."""
    lib = _load()
    K = np.ascontiguousarray(K, dtype=np.float64)
    Qbar = np.ascontiguousarray(Qbar, dtype=np.float64)
    T, d = K.shape
    W = Qbar.shape[0]
    N = -(-T // block)
    out = dict(Pb=np.zeros((W, N)), a=np.zeros(N), ctilde=np.zeros(N), s=np.zeros(N),
               w=np.zeros(N, np.float32), gamma=np.zeros(max(walk_len, 1)))
    rc = lib.nxo_block_scores(T, d, W, walk_len, block, lam, eps_tie, _ptr(K), _ptr(Qbar),
                              _ptr(out["Pb"]), _ptr(out["a"]), _ptr(out["ctilde"]),
                              _ptr(out["s"]), _ptr(out["w"]), _ptr(out["gamma"]))
    if rc != N:
        raise ValueError("nxo_block_scores rejected its arguments")
    out["gamma"] = out["gamma"][:walk_len]
    return out


def philox4x32_10(ctr, key):
    """Philox4x32-10 of one counter (4 words) under one key (2 words)."""
    lib = _load()
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    o = np.zeros(4, np.uint32)
    lib.nxo_philox4x32_10(_ptr(c), _ptr(k), _ptr(o))
    return o


def philox_many(ctrs, key):
    """Philox4x32-10 of an (n, 4) array of counters under one key."""
    lib = _load()
    c = np.ascontiguousarray(ctrs, dtype=np.uint32).reshape(-1, 4)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    o = np.zeros_like(c)
    lib.nxo_philox_many(c.shape[0], _ptr(c), _ptr(k), _ptr(o))
    return o


def uniform(x: int) -> float:
    return float(_load().nxo_uniform(int(x) & 0xFFFFFFFF))


def ln_spec(u):
    """The specified binary32 logarithm, elementwise over a float32 array."""
    lib = _load()
    u = np.ascontiguousarray(u, dtype=np.float32)
    o = np.zeros_like(u)
    lib.nxo_ln_spec_many(u.size, _ptr(u), _ptr(o))
    return o


def exp_spec(x):
    """The specified binary32 exponential, elementwise over a float32 array."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    o = np.zeros_like(x)
    lib.nxo_exp_spec_many(x.size, _ptr(x), _ptr(o))
    return o


def round_bf16(x):
    """The window queries of a bf16 model as the oracle forms them: each value rounded to
    the nearest bfloat16 (ties to even), elementwise over a float64 array."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    o = np.zeros_like(x)
    lib.nxo_round_bf16_many(x.size, _ptr(x), _ptr(o))
    return o


def reservoir_key(w, pos, seed, step, head_id, seq_id, n_avg=1) -> float:
    """Order key of one candidate: ln(u)/w (n_avg = 1) or ln(n pi) of Eq. (6)."""
    return float(_load().nxo_reservoir_key_n(float(np.float32(w)), int(pos), int(seed),
                                             int(step), int(head_id), int(seq_id),
                                             int(n_avg)))


def select_slice(w32, pos, B, n_sink, n_recent, mode=RESERVOIR, seed=0, step=0, head_id=0,
                 seq_id=0, n_avg=1):
    """§2.3 retention set of one slice over its decision units (slots, or blocks).
    Returns (kept units ascending, keys per unit)."""
    lib = _load()
    w32 = np.ascontiguousarray(w32, dtype=np.float32)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    T = w32.shape[0]
    keep = np.zeros(max(T, 1), np.int32)
    kappa = np.zeros(max(T, 1), np.float32)
    nl = lib.nxo_select_slice(T, _ptr(w32), _ptr(pos), B, n_sink, n_recent, mode, seed, step,
                              head_id, seq_id, n_avg, _ptr(keep), _ptr(kappa))
    if nl < 0:
        raise ValueError("nxo_select_slice rejected its arguments")
    return keep[:nl].copy(), kappa[:T].copy()


# --------------------------------------------------------------------------
# Whole-cache step
# --------------------------------------------------------------------------

class _Cache(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("layers", "seqs", "kv_heads", "group", "head_dim", "capacity", "page_size",
                 "num_pages", "max_pages_per_seq", "dtype")] + [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pos", ctypes.c_void_p),
        ("lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p)]


class _Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("window", "walk_len", "n_sink", "n_recent", "mode")] + [
        ("lam", ctypes.c_double), ("eps_tie", ctypes.c_double), ("budget", ctypes.c_void_p),
        ("seed", ctypes.c_uint64), ("step", ctypes.c_uint32), ("seq_id_base", ctypes.c_int32),
        ("layer_id_base", ctypes.c_int32), ("n_avg", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("slice_budget", ctypes.c_void_p)]


def evict_step(cache: dict, q, params: dict, slices=None, mutate=True, nthreads=0):
    """One eviction step over numpy cache arrays (modified in place when mutate).

    ``cache`` keys: k, v (uint16 bf16 bits or float32), pos, lens, budget-independent
    geometry (layers, seqs, kv_heads, group, head_dim, capacity, page_size, num_pages,
    max_pages_per_seq, block_table). ``params`` keys: window, walk_len, n_sink,
    n_recent, mode, lam, eps_tie, budget (int32[S]), seed, step, seq_id_base,
    layer_id_base, n_avg (default 1), block_size (default 1), slice_budget (optional
    int32[L*S*Hkv], overrides budget per slice). Budgets and forced counts are in
    decision units (blocks when block_size > 1). Returns dict(keep (kept units), w, a
    (per unit), newlen (rows left)) for the listed slices.
    """
    lib = _load()
    k, v = cache["k"], cache["v"]
    dtype = BF16 if k.dtype == np.uint16 else F32
    for name in ("k", "v", "pos", "lens"):
        if not cache[name].flags["C_CONTIGUOUS"]:
            raise ValueError(f"cache[{name!r}] must be C-contiguous")
    bt = cache.get("block_table")
    c = _Cache(cache["layers"], cache["seqs"], cache["kv_heads"], cache["group"],
               cache["head_dim"], cache["capacity"], cache.get("page_size", 0),
               cache.get("num_pages", 0), cache.get("max_pages_per_seq", 0), dtype,
               k.ctypes.data, v.ctypes.data, cache["pos"].ctypes.data, cache["lens"].ctypes.data,
               None if bt is None else bt.ctypes.data)
    budget = np.ascontiguousarray(params["budget"], dtype=np.int32)
    sb = params.get("slice_budget")
    sb = None if sb is None else np.ascontiguousarray(sb, dtype=np.int32)
    p = _Params(params["window"], params["walk_len"], params.get("n_sink", 32),
                params.get("n_recent", 32), params.get("mode", RESERVOIR),
                params.get("lam", 0.5), params.get("eps_tie", 1e-6), budget.ctypes.data,
                params.get("seed", 0), params.get("step", 0), params.get("seq_id_base", 0),
                params.get("layer_id_base", 0), params.get("n_avg", 1),
                params.get("block_size", 1), None if sb is None else sb.ctypes.data)
    n_all = cache["layers"] * cache["seqs"] * cache["kv_heads"]
    sel = None if slices is None else np.ascontiguousarray(slices, dtype=np.int32)
    n = n_all if sel is None else sel.size
    cap = cache["capacity"]
    keep = np.full((n, cap), -1, np.int32)
    w = np.zeros((n, cap), np.float32)
    a = np.zeros((n, cap), np.float64)
    newlen = np.zeros(n, np.int32)
    q = np.ascontiguousarray(q)
    rc = lib.nxo_evict_step(ctypes.byref(c), q.ctypes.data, ctypes.byref(p), n, _ptr(sel),
                            _ptr(keep), _ptr(w), _ptr(a), _ptr(newlen), 1 if mutate else 0,
                            nthreads)
    if rc != 0:
        raise ValueError("nxo_evict_step failed")
    return dict(keep=keep, w=w, a=a, newlen=newlen)


def compact_slice(cache: dict, sid: int, keep) -> None:
    """Out-of-place definition of the compaction of one slice (in the numpy arrays)."""
    lib = _load()
    k = cache["k"]
    dtype = BF16 if k.dtype == np.uint16 else F32
    bt = cache.get("block_table")
    c = _Cache(cache["layers"], cache["seqs"], cache["kv_heads"], cache["group"],
               cache["head_dim"], cache["capacity"], cache.get("page_size", 0),
               cache.get("num_pages", 0), cache.get("max_pages_per_seq", 0), dtype,
               k.ctypes.data, cache["v"].ctypes.data, cache["pos"].ctypes.data,
               cache["lens"].ctypes.data, None if bt is None else bt.ctypes.data)
    keep = np.ascontiguousarray(keep, dtype=np.int32)
    if lib.nxo_compact_slice(ctypes.byref(c), int(sid), _ptr(keep), keep.size) != 0:
        raise MemoryError("nxo_compact_slice")


def cpu_count() -> int:
    return os.cpu_count() or 1
