"""Thin ctypes binding of libnexus.so (include/nexus.h). Argument marshalling only:
every step of the eviction path runs in the library's CUDA kernels.

Tensors are torch CUDA tensors; the stream is torch's current stream unless given.
The library must be built (``__graft_entry__.build()`` or
``python -m streaming_kv_cache_step_gb300.build``); if it is missing, every call
raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnexus.so")

NX_OK, NX_ERR_INVALID_ARG, NX_ERR_UNSUPPORTED, NX_ERR_CUDA = 0, 1, 2, 3
NX_ERR_TIMEOUT, NX_ERR_WORKSPACE, NX_ERR_DEVICE_FAULT = 4, 5, 6
NX_DEV_TIMEOUT, NX_DEV_BAD_LEN, NX_DEV_BAD_BUDGET, NX_DEV_BAD_PAGE = 1, 2, 4, 8
DTYPE_F32, DTYPE_BF16 = 0, 1
MODE_RESERVOIR, MODE_TOPK = 0, 1

SYMBOLS = ("nexus_workspace_bytes", "nexus_direct_scores", "nexus_walk",
           "nexus_reservoir_select", "kv_compact", "nexus_evict_step", "nx_status_string",
           "nexus_last_launch_count", "nexus_debug_compact", "nexus_last_launch_name",
           "nexus_profile_next_call", "nexus_debug_force_simt", "nexus_debug_set_trace",
           "nexus_debug_scorer_config", "nexus_debug_scorer_layout", "kv_compact_noalloc",
           "nexus_last_scorer", "nexus_debug_compact_kernel")
SCORER_NONE, SCORER_TENSOR_CORE, SCORER_CUDA_CORE, SCORER_TENSOR_CORE_TWO_PASS = 0, 1, 2, 3


class NexusError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class CCache(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("layers", "seqs", "kv_heads", "group", "head_dim", "capacity", "page_size",
                 "num_pages", "max_pages_per_seq", "dtype")] + [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pos", ctypes.c_void_p),
        ("lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p)]


class CParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("window", "walk_len", "n_sink", "n_recent", "n_avg", "mode")] + [
        ("lam", ctypes.c_float), ("eps_tie", ctypes.c_float), ("budget", ctypes.c_void_p),
        ("budget_max", ctypes.c_int32), ("seq_id_base", ctypes.c_int32),
        ("layer_id_base", ctypes.c_int32), ("step", ctypes.c_uint32), ("seed", ctypes.c_uint64),
        ("block_size", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("slice_budget", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load libnexus.so once; raise if it is not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libnexus.so is not built ({path}); run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            lib.nexus_workspace_bytes.argtypes = [P, P]
            lib.nexus_workspace_bytes.restype = ctypes.c_size_t
            lib.nexus_direct_scores.argtypes = [P, P, P, P, P, P, ctypes.c_size_t, P, P]
            lib.nexus_walk.argtypes = [P, P, P, P, P, P, ctypes.c_size_t, P, P]
            lib.nexus_reservoir_select.argtypes = [P, P, P, P, P, ctypes.c_size_t, P, P]
            lib.kv_compact.argtypes = [P, P, P, P, ctypes.c_size_t, P, P]
            lib.nexus_evict_step.argtypes = [P, P, P, P, P, ctypes.c_size_t, P, P]
            for name in ("nexus_direct_scores", "nexus_walk", "nexus_reservoir_select",
                         "kv_compact", "nexus_evict_step"):
                getattr(lib, name).restype = ctypes.c_int
            lib.nexus_debug_compact.argtypes = [P, P, P, P, ctypes.c_size_t, P, P,
                                                ctypes.c_longlong]
            lib.nexus_debug_compact.restype = ctypes.c_int
            lib.nx_status_string.argtypes = [ctypes.c_int]
            lib.nx_status_string.restype = ctypes.c_char_p
            lib.nexus_last_scorer.argtypes = []
            lib.nexus_last_scorer.restype = ctypes.c_int32
            lib.nexus_last_launch_count.argtypes = []
            lib.nexus_last_launch_count.restype = ctypes.c_int32
            lib.nexus_last_launch_name.argtypes = [ctypes.c_int32]
            lib.nexus_last_launch_name.restype = ctypes.c_char_p
            lib.nexus_profile_next_call.argtypes = [ctypes.c_void_p, ctypes.c_int32]
            lib.nexus_profile_next_call.restype = None
            lib.nexus_debug_force_simt.argtypes = [ctypes.c_int32]
            lib.nexus_debug_force_simt.restype = None
            lib.nexus_debug_compact_kernel.argtypes = [ctypes.c_int32]
            lib.nexus_debug_compact_kernel.restype = None
            lib.nexus_debug_scorer_layout.argtypes = [ctypes.c_int32]
            lib.nexus_debug_scorer_layout.restype = None
            lib.nexus_debug_set_trace.argtypes = [ctypes.c_void_p]
            lib.nexus_debug_set_trace.restype = None
            lib.nexus_debug_scorer_config.argtypes = [ctypes.c_void_p]
            lib.nexus_debug_scorer_config.restype = None
            _lib = lib
    return _lib


def force_simt(on: bool) -> None:
    """Route scoring to the CUDA-core scorer even where the tensor-core one applies."""
    load().nexus_debug_force_simt(1 if on else 0)


COMPACT_AUTO, COMPACT_TILES, COMPACT_SLICES = 0, 1, 2


def compact_kernel(which: int) -> None:
    """Testing hook: the compaction kernel, process-wide (COMPACT_TILES, COMPACT_SLICES or
    COMPACT_AUTO)."""
    load().nexus_debug_compact_kernel(int(which))


def scorer_layout(teams: int) -> None:
    """Tensor-core scorer layout: 2 or 1 pipelines per CTA, 0 for the automatic choice."""
    load().nexus_debug_scorer_layout(int(teams))


def scorer_config() -> dict:
    """Configuration of the last tensor-core scorer launch made from this thread."""
    out = (ctypes.c_int32 * 8)()
    load().nexus_debug_scorer_config(out)
    keys = ("teams_per_cta", "occupancy_api", "grid", "tiles_per_chunk", "tmem_buffers",
            "chunks_per_slice", "tmem_cols", "smem_bytes")
    return dict(zip(keys, list(out)))


def set_trace(buf) -> None:
    """Install (int64 CUDA tensor) or remove (None) the scorer's phase-trace buffer."""
    load().nexus_debug_set_trace(None if buf is None else ctypes.c_void_p(buf.data_ptr()))


def status_string(status: int) -> str:
    return load().nx_status_string(int(status)).decode()


def last_scorer() -> int:
    """SCORER_TENSOR_CORE, SCORER_CUDA_CORE or SCORER_NONE for the last call of this thread."""
    return int(load().nexus_last_scorer())


def last_launch_count() -> int:
    return int(load().nexus_last_launch_count())


def last_launch_names() -> list[str]:
    lib = load()
    return [lib.nexus_last_launch_name(i).decode() for i in range(last_launch_count())]


def profile_next_call(events) -> object:
    """Arm per-launch events (torch.cuda.Event with timing) for the next call; returns
    the ctypes array, which the caller keeps alive until that call returns."""
    for e in events:
        if not e.cuda_event:          # torch creates the CUDA event on first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    load().nexus_profile_next_call(arr, len(events))
    return arr


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


@dataclass
class Cache:
    """Device KV cache in the layouts of include/nexus.h (tensors stay owned by torch)."""
    k: torch.Tensor
    v: torch.Tensor
    pos: torch.Tensor
    lens: torch.Tensor
    layers: int
    seqs: int
    kv_heads: int
    group: int
    head_dim: int
    capacity: int
    page_size: int = 0
    num_pages: int = 0
    max_pages_per_seq: int = 0
    block_table: torch.Tensor | None = None

    @classmethod
    def from_dict(cls, d: dict) -> "Cache":
        return cls(k=d["k"], v=d["v"], pos=d["pos"], lens=d["lens"], layers=d["layers"],
                   seqs=d["seqs"], kv_heads=d["kv_heads"], group=d["group"],
                   head_dim=d["head_dim"], capacity=d["capacity"],
                   page_size=d.get("page_size", 0), num_pages=d.get("num_pages", 0),
                   max_pages_per_seq=d.get("max_pages_per_seq", 0),
                   block_table=d.get("block_table"))

    @property
    def n_slices(self) -> int:
        return self.layers * self.seqs * self.kv_heads

    def c_struct(self) -> CCache:
        dt = DTYPE_BF16 if self.k.dtype == torch.bfloat16 else DTYPE_F32
        for t in (self.k, self.v, self.pos, self.lens):
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError("cache tensors must be contiguous CUDA tensors")
        if self.pos.dtype != torch.int32 or self.lens.dtype != torch.int32:
            raise ValueError("pos and lens must be int32")
        return CCache(self.layers, self.seqs, self.kv_heads, self.group, self.head_dim,
                      self.capacity, self.page_size, self.num_pages, self.max_pages_per_seq, dt,
                      self.k.data_ptr(), self.v.data_ptr(), self.pos.data_ptr(),
                      self.lens.data_ptr(),
                      None if self.block_table is None else self.block_table.data_ptr())


@dataclass
class Params:
    """Step parameters (nx_params). Budgets and forced counts are in decision units:
    rows at block_size 1, blocks of 32 rows at block_size 32."""
    budget: torch.Tensor           # int32 [seqs] on the device
    budget_max: int
    window: int
    walk_len: int = 3
    n_sink: int = 32
    n_recent: int = 32
    n_avg: int = 1
    mode: int = MODE_RESERVOIR
    lam: float = 0.5
    eps_tie: float = 1e-6
    seed: int = 0
    step: int = 0
    seq_id_base: int = 0
    layer_id_base: int = 0
    block_size: int = 1
    slice_budget: torch.Tensor | None = None   # int32 [slices] on the device (optional)

    def c_struct(self) -> CParams:
        if self.budget.dtype != torch.int32 or not self.budget.is_cuda:
            raise ValueError("budget must be an int32 CUDA tensor")
        sb = self.slice_budget
        if sb is not None and (sb.dtype != torch.int32 or not sb.is_cuda):
            raise ValueError("slice_budget must be an int32 CUDA tensor")
        return CParams(self.window, self.walk_len, self.n_sink, self.n_recent, self.n_avg,
                       self.mode, self.lam, self.eps_tie, self.budget.data_ptr(),
                       self.budget_max, self.seq_id_base, self.layer_id_base,
                       self.step & 0xFFFFFFFF, self.seed & 0xFFFFFFFFFFFFFFFF,
                       self.block_size, 0, None if sb is None else sb.data_ptr())


def _check(status: int, where: str):
    if status != NX_OK:
        raise NexusError(status, where)


def workspace_bytes(cache: Cache, params: Params) -> int:
    n = load().nexus_workspace_bytes(ctypes.byref(cache.c_struct()), ctypes.byref(params.c_struct()))
    if n == 0:
        raise NexusError(NX_ERR_INVALID_ARG, "nexus_workspace_bytes")
    return int(n)


def alloc_workspace(cache: Cache, params: Params) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks, above the 256 required
    return torch.empty(workspace_bytes(cache, params), dtype=torch.uint8, device=cache.k.device)


def new_status(device) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


def direct_scores(cache: Cache, q, params: Params, a_out, row_stats_out, ws, dev_status,
                  stream=None):
    _check(load().nexus_direct_scores(ctypes.byref(cache.c_struct()), _ptr(q),
                                      ctypes.byref(params.c_struct()), _ptr(a_out),
                                      _ptr(row_stats_out), _ptr(ws), ws.numel(),
                                      _ptr(dev_status), _stream(stream)),
           "nexus_direct_scores")


def walk(cache: Cache, q, params: Params, w_out, ctilde_out, ws, dev_status, stream=None):
    _check(load().nexus_walk(ctypes.byref(cache.c_struct()), _ptr(q),
                             ctypes.byref(params.c_struct()), _ptr(w_out), _ptr(ctilde_out),
                             _ptr(ws), ws.numel(), _ptr(dev_status), _stream(stream)),
           "nexus_walk")


def reservoir_select(w, cache: Cache, params: Params, keep_idx, ws, dev_status, stream=None):
    _check(load().nexus_reservoir_select(_ptr(w), ctypes.byref(cache.c_struct()),
                                         ctypes.byref(params.c_struct()), _ptr(keep_idx),
                                         _ptr(ws), ws.numel(), _ptr(dev_status),
                                         _stream(stream)),
           "nexus_reservoir_select")


def compact(cache: Cache, keep_idx, params: Params, ws, dev_status, stream=None):
    _check(load().kv_compact(ctypes.byref(cache.c_struct()), _ptr(keep_idx),
                             ctypes.byref(params.c_struct()), _ptr(ws), ws.numel(),
                             _ptr(dev_status), _stream(stream)),
           "kv_compact")


def evict_step(cache: Cache, q, params: Params, keep_idx_out, ws, dev_status, stream=None):
    _check(load().nexus_evict_step(ctypes.byref(cache.c_struct()), _ptr(q),
                                   ctypes.byref(params.c_struct()), _ptr(keep_idx_out),
                                   _ptr(ws), ws.numel(), _ptr(dev_status), _stream(stream)),
           "nexus_evict_step")
