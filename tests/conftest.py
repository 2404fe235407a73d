import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running")


def pytest_collection_modifyitems(config, items):
    # keep the library-free oracle tests first and the allocation-free entry point last
    pass


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(params=[1, 2], ids=["tiles", "slices"])
def compact_kernel(request):
    """Both compaction kernels (the tile kernel and the warp-per-slice one), process-wide
    for the test, the automatic choice restored afterwards."""
    from streaming_kv_cache_step_gb300 import nexus
    nexus.compact_kernel(request.param)
    yield request.param
    nexus.compact_kernel(nexus.COMPACT_AUTO)
