"""gtattn_fwd_noalloc: the forward for callers that cannot allocate device
memory (allocator callbacks, fixed-budget runtimes, frameworks that own the
device heap).  Its temporaries live in the library's fixed device array; its
results must be the fp64 oracle's within the parity tolerances, like every
other path, and agree with gtattn_fwd's.

The calls run in a row on different graphs, shapes and output types, so what
one call left in the shared array would show up in the next.  Collected last
(file name) so that a failure here does not hide the other tests.
"""
import numpy as np
import pytest

import workloads as wl
from gpu_helpers import assert_close, oracle_rows, out_to_numpy, sample_rows, to_device

torch = pytest.importorskip("torch")
gt = pytest.importorskip("graph_transformer_sparse_gb300")

pytestmark = pytest.mark.gpu


def _call(lib, name, w, d, dt, s):
    d["out"].fill_(float("nan"))
    st = getattr(lib, name)(d["indptr"].data_ptr(), d["indices"].data_ptr(), d["Q"].data_ptr(),
                            d["K"].data_ptr(), d["V"].data_ptr(), d["out"].data_ptr(), w.N, w.nnz, w.H, w.D,
                            w.scale, dt, s)
    assert st == gt.GTATTN_OK, (name, gt.gtattn_status_string(st), lib.gtattn_last_error())
    torch.cuda.synchronize()
    return out_to_numpy(d["out"])


def _both(w, out32):
    """(gtattn_fwd_noalloc output, gtattn_fwd output) through the C ABI."""
    d = to_device(w, out32=out32)
    dt = gt._dtype_code(d["Q"], d["out"])
    lib = gt.load()
    s = torch.cuda.current_stream().cuda_stream
    a = _call(lib, "gtattn_fwd_noalloc", w, d, dt, s)
    b = _call(lib, "gtattn_fwd", w, d, dt, s)
    return a, b


def _generic_shape_graph():
    """H = 3, D = 5 (rows the vector kernel cannot tile: the generic kernel),
    N above the one-block binning limit (the three-launch binning path), and
    hub rows of more than 1024 entries (split into chunks)."""
    rng = np.random.default_rng(77)
    n, H, D = 6000, 3, 5
    ip, ix = wl.random_csr(rng, n, 150_000, self_loops=True, degree_skew=1.1)
    assert np.diff(ip).max() > 1024
    Q, K, V = (rng.standard_normal((n, H, D), dtype=np.float32) for _ in range(3))
    return wl.Workload("generic_3x5", n, H, D, "f32", ip, ix, Q, K, V, float(np.float32(1 / np.sqrt(D))))


def _check(w, got, rows, ref, out32, what):
    rounded = w.dtype == "bf16" and not out32
    assert_close(got[rows], ref, w.dtype, what, rounded_bf16=rounded)


@pytest.mark.parametrize("out32", [True, False])
def test_noalloc_matches_oracle_and_gtattn_fwd_calls_in_a_row(out32):
    # a skewed graph with rows far above the 1024-entry split (chunks and
    # partials in the fixed array), then the generic kernel on another shape,
    # then a different, smaller graph
    big = wl.make_workload("rmat", scale=16, draws=1 << 20)
    assert np.diff(big.indptr).max() > 3000
    cases = [(big, out32), (_generic_shape_graph(), False), (wl.make_workload("molecules"), False)]
    for w, o32 in cases:
        a, b = _both(w, o32)
        assert np.isfinite(a).all(), w.name
        rows = sample_rows(w, n_random=800, n_top=48) if w.N > 4000 else np.arange(w.N)
        ref = oracle_rows(w, rows=rows)["out"]
        _check(w, a, rows, ref, o32, f"{w.name}: noalloc vs oracle (out32={o32})")
        _check(w, b, rows, ref, o32, f"{w.name}: gtattn_fwd vs oracle (out32={o32})")
        # against the plan-less forward on every row: both within the parity
        # tolerance of the oracle, so within twice it of each other
        rtol, atol = (2e-3, 1e-5) if w.dtype == "bf16" else (1e-5, 1e-6)
        err = np.abs(a - b)
        bound = 2 * (rtol * np.abs(b) + atol)
        if w.dtype == "bf16" and not o32:
            bound += np.ldexp(1.0, np.frexp(np.abs(b))[1] - 8)   # one bf16 ulp: either side's rounding
        assert (err <= bound).all(), f"{w.name}: noalloc vs gtattn_fwd, max excess {(err - bound).max()}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = gt.load()
    # 16.8M entries of 8x64 bf16 would need ~70 MB of partials: rejected
    # before any GPU work (the pointers are never touched)
    st = lib.gtattn_fwd_noalloc(256, 256, 256, 256, 256, 256, 32768, 16_777_216, 8, 64, 0.125,
                                gt.GTATTN_BF16, None)
    assert st == gt.GTATTN_ERR_UNSUPPORTED
    assert b"needs" in lib.gtattn_last_error()
