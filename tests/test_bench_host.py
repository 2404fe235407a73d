"""Host-side accounting of bench.py: algorithmic bytes per step and the recorded DRAM
traffic lookup (no GPU involved)."""
import hashlib
import importlib.util
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_algorithmic_bytes_counts_only_moved_rows():
    b = _bench()
    from streaming_kv_cache_step_gb300 import workloads as W
    wl = W.shrink(W.llama3_8b_layer(), seqs=1, kv_heads=2, lens=np.array([10], np.int32),
                  capacity=16, budget=np.array([6], np.int32))
    lens0 = np.array([10, 4])
    newlen = np.array([6, 4])
    keep = np.full((2, 16), -1)
    keep[0, :6] = [0, 1, 2, 5, 8, 9]      # slots 3..5 of the output move
    keep[1, :4] = [0, 1, 2, 3]            # nothing evicted, nothing moves
    ab = b.algorithmic_bytes(wl, lens0, keep, newlen)
    row = wl.head_dim * 2
    assert ab["rows"] == 14 and ab["moved"] == 3
    q = wl.n_slices * wl.group * wl.window * wl.head_dim * 2
    assert ab["score"] == 14 * (row + 4) + q
    assert ab["compact"] == 3 * (4 * row + 8) + 10 * 4
    assert ab["total"] == ab["score"] + ab["compact"]


def test_recorded_traffic_requires_the_captured_source(tmp_path, monkeypatch):
    b = _bench()
    src = tmp_path / "streaming_kv_cache_step_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "nx_score_tc.cu").write_text("// kernel v1\n")
    digest = hashlib.sha256(b"// kernel v1\n").hexdigest()[:16]
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.txt").write_text(f"# comment\nscore_tc wl_a {digest} 1234\n"
                                      f"score_tc wl_b 0000000000000000 99\n")
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    assert b.recorded_traffic("score_tc", "wl_a") == 1234
    assert b.recorded_traffic("score_tc", "wl_b") is None      # other source
    assert b.recorded_traffic("score_tc", "wl_c") is None      # never captured
    (src / "nx_score_tc.cu").write_text("// kernel v2\n")      # the kernel changed since
    assert b.recorded_traffic("score_tc", "wl_a") is None
