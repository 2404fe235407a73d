"""GB300-native (sm_103a) per-step eviction of Nexus Sampling.

The compute lives in ``libnexus.so`` (hand-written CUDA behind a C ABI, declared
in ``include/nexus.h``); :mod:`.nexus` is its thin ctypes binding and
:mod:`.workloads` draws seeded synthetic inputs. Importing this package does not
load the library; the binding loads it on first use and fails loudly if it is
missing.
"""
