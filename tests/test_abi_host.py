"""Host-side tests of the C ABI (no GPU): the library builds for sm_103a, loads, exports
every symbol include/nexus.h declares, and rejects invalid arguments before any CUDA
call."""
import ctypes
import os
import re
import shutil

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from streaming_kv_cache_step_gb300 import build, nexus
    build.build()
    return nexus.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "nexus.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[a-z_0-9 \*]+?\b([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_symbols_exported(lib):
    names = _declared_functions()
    assert {"nexus_workspace_bytes", "nexus_direct_scores", "nexus_walk",
            "nexus_reservoir_select", "kv_compact", "nexus_evict_step",
            "nx_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from streaming_kv_cache_step_gb300 import nexus
    assert nexus.status_string(0) == "NX_OK"
    assert nexus.status_string(1) == "NX_ERR_INVALID_ARG"
    assert nexus.status_string(99) == "NX_UNKNOWN_STATUS"


def _structs(**over):
    from streaming_kv_cache_step_gb300 import nexus
    c = dict(layers=1, seqs=2, kv_heads=8, group=4, head_dim=128, capacity=8192, page_size=0,
             num_pages=0, max_pages_per_seq=0, dtype=nexus.DTYPE_BF16, k=0x10000, v=0x20000,
             pos=0x30000, lens=0x40000, block_table=None)
    p = dict(window=32, walk_len=3, n_sink=32, n_recent=32, n_avg=1, mode=0, lam=0.5,
             eps_tie=1e-6, budget=0x50000, budget_max=1638, seq_id_base=0, layer_id_base=0,
             step=0, seed=1, block_size=1, reserved=0, slice_budget=None)
    for k, v in over.items():
        (c if k in c else p)[k] = v
    cc = nexus.CCache(*[c[n] for n, _ in nexus.CCache._fields_])
    pp = nexus.CParams(*[p[n] for n, _ in nexus.CParams._fields_])
    return cc, pp


def test_workspace_bytes_and_validation(lib):
    c, p = _structs()
    n = lib.nexus_workspace_bytes(ctypes.byref(c), ctypes.byref(p))
    assert n > 2 * 16 * 8192 * 4   # keys + kept slots at least
    bad = [dict(head_dim=96), dict(window=0), dict(window=65), dict(walk_len=33),
           dict(walk_len=9), dict(k=0x10008), dict(budget_max=63), dict(budget_max=9000),
           dict(page_size=12), dict(dtype=7), dict(seq_id_base=(1 << 24) - 1),
           dict(lam=-1.0), dict(n_avg=0), dict(n_avg=1025), dict(block_size=0),
           dict(block_size=16), dict(block_size=32, budget_max=257),
           dict(block_size=32, n_sink=1, n_recent=0, budget_max=100), dict(reserved=1)]
    for b in bad:
        c, p = _structs(**b)
        assert lib.nexus_workspace_bytes(ctypes.byref(c), ctypes.byref(p)) == 0, b
    # the paper's n = 5 and b = 32 (budgets in blocks: 8192 rows hold 256 blocks)
    for good in (dict(n_avg=5), dict(n_avg=1024),
                 dict(block_size=32, n_sink=1, n_recent=1, budget_max=52)):
        c, p = _structs(**good)
        assert lib.nexus_workspace_bytes(ctypes.byref(c), ctypes.byref(p)) > 0, good


def test_entry_points_reject_before_touching_the_gpu(lib):
    from streaming_kv_cache_step_gb300 import nexus
    P = ctypes.c_void_p
    c, p = _structs(window=0)
    ws, st = P(0x100000), P(0x200000)
    assert lib.nexus_evict_step(ctypes.byref(c), P(0x60000), ctypes.byref(p), None, ws,
                                1 << 40, st, None) == nexus.NX_ERR_INVALID_ARG
    c, p = _structs(block_size=16, n_sink=1, n_recent=1, budget_max=100)
    assert lib.nexus_evict_step(ctypes.byref(c), P(0x60000), ctypes.byref(p), None, ws,
                                1 << 40, st, None) == nexus.NX_ERR_UNSUPPORTED
    c, p = _structs()
    assert lib.nexus_evict_step(ctypes.byref(c), P(0x60000), ctypes.byref(p), None, ws, 16,
                                st, None) == nexus.NX_ERR_WORKSPACE
    assert lib.nexus_evict_step(ctypes.byref(c), P(0x60000), ctypes.byref(p), None, P(0x100010),
                                1 << 40, st, None) == nexus.NX_ERR_WORKSPACE
    assert lib.nexus_direct_scores(ctypes.byref(c), P(0x60004), ctypes.byref(p), P(0x70000),
                                   None, ws, 1 << 40, st, None) == nexus.NX_ERR_INVALID_ARG
    assert lib.kv_compact(ctypes.byref(c), None, ctypes.byref(p), ws, 1 << 40, st,
                          None) == nexus.NX_ERR_INVALID_ARG
    assert lib.nexus_reservoir_select(None, ctypes.byref(c), ctypes.byref(p), P(0x70000), ws,
                                      1 << 40, st, None) == nexus.NX_ERR_INVALID_ARG
    assert lib.nexus_walk(ctypes.byref(c), P(0x60000), ctypes.byref(p), P(0x70000), None, ws,
                          1 << 40, None, None) == nexus.NX_ERR_INVALID_ARG   # no status word


def test_binding_refuses_cpu_tensors(lib):
    from streaming_kv_cache_step_gb300 import nexus
    t = torch.zeros(4)
    cache = nexus.Cache(k=t, v=t, pos=t.int(), lens=t.int(), layers=1, seqs=1, kv_heads=1,
                        group=1, head_dim=64, capacity=4)
    with pytest.raises(ValueError):
        cache.c_struct()


def test_product_path_does_not_import_the_oracle():
    # the package and its binding never import or read the oracle
    pkg = os.path.join(ROOT, "streaming_kv_cache_step_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "nexus_oracle" not in src, f
