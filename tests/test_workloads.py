"""Seeded input generators: sizes, structure and determinism (CPU only)."""
import numpy as np
import pytest

import workloads as wl


def _coo(indptr, indices):
    dst = np.repeat(np.arange(len(indptr) - 1), np.diff(indptr))
    return indices.astype(np.int64), dst


def _check_csr(w):
    assert w.indptr.dtype == np.int32 and w.indices.dtype == np.int32
    assert w.indptr[0] == 0 and np.all(np.diff(w.indptr) >= 0)
    assert w.indices.min() >= 0 and w.indices.max() < w.N
    for a in (w.Q, w.K, w.V):
        assert a.shape == (w.N, w.H, w.D) and a.dtype == np.float32


def _self_loops_once(w):
    src, dst = _coo(w.indptr, w.indices)
    loops = np.bincount(dst[src == dst], minlength=w.N)
    return np.all(loops == 1)


def _symmetric(w):
    src, dst = _coo(w.indptr, w.indices)
    a = np.sort(src * w.N + dst)
    b = np.sort(dst * w.N + src)
    return np.array_equal(a, b)


def _no_duplicates(w):
    src, dst = _coo(w.indptr, w.indices)
    k = np.sort(dst * w.N + src)
    return bool(np.all(k[1:] != k[:-1]))


def test_bf16_round_nearest_even():
    # bf16 keeps 7 fraction bits: the spacing just above 1.0 is 2^-7
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-9, -2.5, 1.0 + 2**-9, 1.0 + 2**-7 + 2**-8],
                 np.float32)
    # ties (1+2^-8, 1+2^-7+2^-8) go to the even neighbour; others to the nearest
    want = np.array([1.0, 1.0, 1.0 + 2**-7, -2.5, 1.0, 1.0 + 2**-6], np.float32)
    v, bits = wl.bf16_round(x)
    np.testing.assert_array_equal(v, want)
    assert bits[0] == 0x3F80 and bits[3] == 0xC020
    assert np.array_equal(wl.bf16_bits_to_f32(bits), v)


def test_tiny_random():
    w = wl.make_workload("tiny_random")
    _check_csr(w)
    assert (w.N, w.nnz, w.H, w.D, w.dtype) == (30, 100, 8, 64, "f32")
    assert _no_duplicates(w)
    w2 = wl.make_workload("tiny_random")
    assert np.array_equal(w.indices, w2.indices) and np.array_equal(w.Q, w2.Q)


def test_molecules():
    w = wl.make_workload("molecules")
    _check_csr(w)
    assert (w.H, w.D, w.dtype) == (8, 10, "f32")
    assert 128 * 10 <= w.N <= 128 * 50
    assert _symmetric(w) and _self_loops_once(w) and _no_duplicates(w)
    deg = np.diff(w.indptr)
    assert deg.max() <= 5 and deg.min() >= 2      # max degree 4 plus the self-loop


def test_erdos_renyi():
    w = wl.make_workload("erdos_renyi")
    _check_csr(w)
    assert (w.N, w.nnz, w.H, w.D, w.dtype) == (100_000, 1_700_000, 8, 64, "bf16")
    assert _symmetric(w) and _self_loops_once(w) and _no_duplicates(w)
    assert np.array_equal(wl.bf16_bits_to_f32(w.bits["K"]).reshape(w.K.shape), w.K)


@pytest.mark.slow
def test_rmat_full():
    w = wl.make_workload("rmat")
    _check_csr(w)
    assert w.N == 1 << 20 and (w.H, w.D, w.dtype) == (4, 32, "bf16")
    assert 16_500_000 < w.nnz < 17_500_000
    assert _self_loops_once(w) and _no_duplicates(w)
    deg = np.diff(w.indptr)
    assert deg.max() > 20_000 and np.median(deg) <= 3


def test_rmat_small_structure():
    w = wl.small_workload("rmat")
    _check_csr(w)
    assert _self_loops_once(w) and _no_duplicates(w)
    deg = np.diff(w.indptr)
    assert deg.max() > 20 * np.median(deg)


def test_dense_blocks():
    w = wl.make_workload("dense_blocks", n_blocks=3, block=64)
    _check_csr(w)
    assert w.nnz == 3 * 64 * 64
    src, dst = _coo(w.indptr, w.indices)
    assert np.all(src // 64 == dst // 64)
    assert _self_loops_once(w) and _no_duplicates(w)
    assert abs(w.Q.std() - 0.5) < 0.05


def test_csr_by_destination_keeps_duplicates():
    ip, ix = wl.csr_by_destination([0, 0, 2], [1, 1, 1], 3)
    assert list(ip) == [0, 0, 3, 3] and list(ix) == [0, 0, 2]
