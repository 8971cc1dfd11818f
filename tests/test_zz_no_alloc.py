"""gtattn_fwd_noalloc: the forward for callers that cannot allocate device
memory (allocator callbacks, fixed-budget runtimes, frameworks that own the
device heap).  It must give gtattn_fwd's results while keeping its
temporaries in the library's fixed device array.

Two calls in a row on different graphs check that what the first call left
in the shared array does not leak into the second.  Collected last (file
name) so that a failure here does not hide the other tests.
"""
import numpy as np
import pytest

import workloads as wl
from gpu_helpers import assert_close, out_to_numpy, to_device

torch = pytest.importorskip("torch")
gt = pytest.importorskip("graph_transformer_sparse_gb300")

pytestmark = pytest.mark.gpu


def _both(w, out32):
    """(gtattn_fwd_noalloc output, gtattn_fwd output) through the C ABI."""
    d = to_device(w, out32=out32)
    dt = gt._dtype_code(d["Q"], d["out"])
    lib = gt.load()
    s = torch.cuda.current_stream().cuda_stream
    d["out"].fill_(float("nan"))
    st = lib.gtattn_fwd_noalloc(d["indptr"].data_ptr(), d["indices"].data_ptr(), d["Q"].data_ptr(),
                                d["K"].data_ptr(), d["V"].data_ptr(), d["out"].data_ptr(), w.N, w.nnz, w.H,
                                w.D, w.scale, dt, s)
    assert st == gt.GTATTN_OK, gt.gtattn_status_string(st)
    torch.cuda.synchronize()
    a = out_to_numpy(d["out"])
    d["out"].fill_(float("nan"))
    st = lib.gtattn_fwd(d["indptr"].data_ptr(), d["indices"].data_ptr(), d["Q"].data_ptr(), d["K"].data_ptr(),
                        d["V"].data_ptr(), d["out"].data_ptr(), w.N, w.nnz, w.H, w.D, w.scale, dt, s)
    assert st == gt.GTATTN_OK
    torch.cuda.synchronize()
    return a, out_to_numpy(d["out"])


def test_noalloc_matches_gtattn_fwd_two_calls():
    # first: a skewed graph with rows far above the 1024-entry split (chunks
    # and partials in the fixed array); second: a different, smaller graph
    big = wl.make_workload("rmat", scale=16, draws=1 << 20)
    assert np.diff(big.indptr).max() > 3000
    small = wl.make_workload("molecules")
    for w, out32 in ((big, True), (small, False)):
        a, b = _both(w, out32)
        assert np.isfinite(a).all()
        # the tolerance the parity tests use for this output type
        assert_close(a, b, "f32", f"{w.name}: noalloc vs gtattn_fwd")


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = gt.load()
    # 16.8M entries of 8x64 bf16 would need ~70 MB of partials: rejected
    # before any GPU work (the pointers are never touched)
    st = lib.gtattn_fwd_noalloc(256, 256, 256, 256, 256, 256, 32768, 16_777_216, 8, 64, 0.125,
                                gt.GTATTN_BF16, None)
    assert st == gt.GTATTN_ERR_UNSUPPORTED
    assert b"needs" in lib.gtattn_last_error()
