"""Pins of the oracle's key path: Philox4x32-10 against cuRAND's host generator (a
library routine that runs on the CPU), the uniform map, and ln_spec against a
double-precision logarithm within its error bound."""
import ctypes
import ctypes.util
import math
import os

import numpy as np
import pytest


def _curand_host():
    for name in ("/usr/local/cuda/lib64/libcurand.so", ctypes.util.find_library("curand")):
        if name and (os.path.exists(name) or not name.startswith("/")):
            try:
                return ctypes.CDLL(name)
            except OSError:
                pass
    return None


def test_philox_matches_curand_host_generator(oracle_lib):
    # cuRAND's host PHILOX4_32_10 generator with seed s, asked for 2^20 words, emits
    # for output block i = a * 65536 + c the four words of
    # Philox4x32-10(counter = (a, 0, c, 0), key = s).
    lib = _curand_host()
    if lib is None:
        pytest.skip("libcurand not available")
    for seed in (0x243F6A8885A308D3, 0xFFFFFFFFFFFFFFFF, 12345):
        gen = ctypes.c_void_p()            # a fresh generator: offset 0 for every seed
        if lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:
            pytest.skip("cuRAND host generator unavailable")
        try:
            assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
            n = 1 << 20
            out = np.zeros(n, np.uint32)
            assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p),
                                      ctypes.c_size_t(n)) == 0
        finally:
            lib.curandDestroyGenerator(gen)
        blocks = np.arange(n // 4)
        ctr = np.zeros((blocks.size, 4), np.uint32)
        ctr[:, 0] = blocks // 65536
        ctr[:, 2] = blocks % 65536
        got = oracle_lib.philox_many(ctr, [seed & 0xFFFFFFFF, seed >> 32])
        assert np.array_equal(got, out.reshape(-1, 4)), hex(seed)


def test_philox_counter_words_all_matter(oracle_lib):
    base = oracle_lib.philox4x32_10([1, 2, 3, 4], [5, 6])
    for i in range(4):
        c = [1, 2, 3, 4]
        c[i] ^= 1 << 17
        assert not np.array_equal(oracle_lib.philox4x32_10(c, [5, 6]), base)
    assert not np.array_equal(oracle_lib.philox4x32_10([1, 2, 3, 4], [5, 7]), base)


def test_uniform_range_and_exactness(oracle_lib):
    assert oracle_lib.uniform(0) == 2.0 ** -24
    assert oracle_lib.uniform(0xFFFFFFFF) == 1 - 2.0 ** -24
    assert oracle_lib.uniform(0x80000000) == 0.5 + 2.0 ** -24
    assert oracle_lib.uniform(511) == 2.0 ** -24          # low 9 bits are dropped


def test_uniform_power_mean_matches_closed_form(oracle_lib):
    # E[u^(1/w)] = w / (w + 1) for u ~ U(0,1) (the n -> infinity limit in App. 8.2).
    n = 1 << 18
    ctr = np.zeros((n, 4), np.uint32)
    ctr[:, 0] = np.arange(n)
    ctr[:, 1] = 7
    words = oracle_lib.philox_many(ctr, [0x85A308D3, 0x243F6A88])[:, 0]
    u = (2.0 * (words >> 9).astype(np.float64) + 1) * 2.0 ** -24
    assert abs(u.mean() - 0.5) < 5 * math.sqrt(1 / 12 / n)
    for w in (0.05, 0.5, 1.0, 3.0):
        x = u ** (1 / w)
        assert abs(x.mean() - w / (w + 1)) < 5 * x.std() / math.sqrt(n)


def test_ln_spec_error_bound_over_every_uniform(oracle_lib):
    # Every uniform the key path can see, (2k+1) 2^-24 for k < 2^23: the specified
    # logarithm is within 2 ulp of the double-precision logarithm.
    k = np.arange(1 << 23, dtype=np.float64)
    u64 = (2 * k + 1) * 2.0 ** -24
    u = u64.astype(np.float32)
    assert np.array_equal(u.astype(np.float64), u64)
    got = oracle_lib.ln_spec(u).astype(np.float64)
    ref = np.log(u64)
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64)
    err = np.abs(got - ref) / ulp
    assert err.max() <= 2.0, err.max()
    # and it is monotone non-decreasing in u
    assert (np.diff(got) >= 0).all()


def test_ln_spec_exact_powers_of_two(oracle_lib):
    u = np.array([0.5, 0.25, 2.0 ** -24, 2.0 ** -10], np.float32)
    got = oracle_lib.ln_spec(u)
    ref = np.log(u.astype(np.float64)).astype(np.float32)
    assert np.all(np.abs(got - ref) <= np.spacing(np.abs(ref)))
