"""The checking build (``GTATTN_DEBUG``, ``lib/libgtattn_debug.so``): every
call that takes a CSR validates it on the device before anything else runs
and returns GTATTN_ERR_BAD_CSR for offsets that do not run from 0 to nnz
without decreasing or for indices outside [0, N).

The feature arrays carry a padding row on each side, so that even an index
of -1 or N would read inside the allocation; the build is first shown to be
the checking one on a CSR whose bad offset keeps every access in bounds."""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as wl

torch = pytest.importorskip("torch")
gt = pytest.importorskip("graph_transformer_sparse_gb300")
from graph_transformer_sparse_gb300 import _build  # noqa: E402

pytestmark = pytest.mark.gpu

OK, BAD = gt.GTATTN_OK, gt.GTATTN_ERR_BAD_CSR


@pytest.fixture(scope="module")
def dlib():
    lib = ctypes.CDLL(_build.build(debug=True))
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    for name, args in {
        "gtattn_fwd": [vp] * 6 + [i64, i64, i32, i32, f32, i32, vp],
        "gtattn_fwd_noalloc": [vp] * 6 + [i64, i64, i32, i32, f32, i32, vp],
        "gtattn_fwd_probs": [vp] * 8 + [i64, i64, i32, i32, f32, i32, vp],
        "gtattn_bwd": [vp] * 9 + [i64, i64, i32, i32, f32, i32, vp],
        "gtattn_csr_build": [vp, vp, i64, i64, vp, vp, vp],
        "gtattn_plan_destroy": [vp],
        "gtattn_fwd_plan": [vp] * 7 + [i32, i32, f32, i32, vp],
    }.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = i32
    return lib


def _case(seed=3, n=300, H=4, D=32):
    rng = np.random.default_rng(seed)
    ip, ix = wl.random_csr(rng, n, 4000, self_loops=True, degree_skew=1.0)
    QKV = [rng.standard_normal((n + 2, H, D)).astype(np.float32) for _ in range(3)]
    dev = [torch.from_numpy(a).cuda() for a in QKV]
    return ip, ix, QKV, dev, n, H, D


def _p(t, row=0):
    return t.data_ptr() + row * t[0].numel() * t.element_size() if row else t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _fwd(lib, ip_t, ix_t, dev, out, n, nnz, H, D, name="gtattn_fwd"):
    # rows 1..n of the padded arrays are the graph's nodes
    return getattr(lib, name)(ip_t.data_ptr(), ix_t.data_ptr(), _p(dev[0], 1), _p(dev[1], 1), _p(dev[2], 1),
                              _p(out, 1), n, nnz, H, D, float(1 / np.sqrt(D)), gt.GTATTN_F32, _stream())


def test_checking_build_runs_and_matches(dlib):
    ip, ix, QKV, dev, n, H, D = _case()
    ip_t, ix_t = torch.from_numpy(ip).cuda(), torch.from_numpy(ix).cuda()
    out = torch.full((n + 2, H, D), float("nan"), device="cuda")
    assert _fwd(dlib, ip_t, ix_t, dev, out, n, len(ix), H, D) == OK
    torch.cuda.synchronize()
    ref = oracle.sparse_mha(ip, ix, QKV[0][1:-1], QKV[1][1:-1], QKV[2][1:-1], np.float32(1 / np.sqrt(D)))["out"]
    got = out[1:-1].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-5 * np.abs(ref) + 1e-6)
    # the normal build gives the same bits
    out2 = torch.full_like(out, float("nan"))
    gt.gtattn_fwd(ip_t, ix_t, dev[0][1:-1], dev[1][1:-1], dev[2][1:-1], out2[1:-1], n, len(ix), H, D,
                  float(1 / np.sqrt(D)), gt.GTATTN_F32)
    torch.cuda.synchronize()
    assert torch.equal(out[1:-1], out2[1:-1])


def test_bad_csr_is_refused_before_any_gather(dlib):
    ip, ix, QKV, dev, n, H, D = _case(seed=4)
    nnz = len(ix)
    out = torch.full((n + 2, H, D), float("nan"), device="cuda")
    # (1) first offset 1 instead of 0: every access stays in bounds either
    # way; only the checking build refuses it
    ip1 = ip.copy()
    ip1[0] = 1
    assert _fwd(dlib, torch.from_numpy(ip1).cuda(), torch.from_numpy(ix).cuda(), dev, out, n, nnz, H, D) == BAD
    torch.cuda.synchronize()
    assert torch.isnan(out).all(), "a refused call wrote its output"
    # (2) indices one past either end (the padding rows keep even those in bounds)
    for bad in (n, -1):
        ix2 = ix.copy()
        ix2[nnz // 2] = bad
        ix_t, ip_t = torch.from_numpy(ix2).cuda(), torch.from_numpy(ip).cuda()
        for name in ("gtattn_fwd", "gtattn_fwd_noalloc"):
            assert _fwd(dlib, ip_t, ix_t, dev, out, n, nnz, H, D, name) == BAD, (name, bad)
        lg = torch.empty(nnz, H, device="cuda")
        assert dlib.gtattn_fwd_probs(ip_t.data_ptr(), ix_t.data_ptr(), _p(dev[0], 1), _p(dev[1], 1),
                                     _p(dev[2], 1), _p(out, 1), lg.data_ptr(), lg.data_ptr(), n, nnz, H, D,
                                     0.5, gt.GTATTN_F32, _stream()) == BAD
        g = [torch.zeros(n + 2, H, D, device="cuda") for _ in range(3)]
        assert dlib.gtattn_bwd(ip_t.data_ptr(), ix_t.data_ptr(), _p(dev[0], 1), _p(dev[1], 1), _p(dev[2], 1),
                               _p(dev[0], 1), _p(g[0], 1), _p(g[1], 1), _p(g[2], 1), n, nnz, H, D, 0.5,
                               gt.GTATTN_F32, _stream()) == BAD
        plan = ctypes.c_void_p()
        assert dlib.gtattn_csr_build(ip_t.data_ptr(), ix_t.data_ptr(), n, nnz, None, ctypes.byref(plan),
                                     _stream()) == BAD
        assert not plan.value
    # (3) decreasing offsets
    ip3 = ip.copy()
    ip3[n // 2] = ip3[n // 2 + 1] + 1
    assert _fwd(dlib, torch.from_numpy(ip3).cuda(), torch.from_numpy(ix).cuda(), dev, out, n, nnz, H, D) == BAD
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    # (4) a valid call afterwards runs normally
    assert _fwd(dlib, torch.from_numpy(ip).cuda(), torch.from_numpy(ix).cuda(), dev, out, n, nnz, H, D) == OK
    torch.cuda.synchronize()
    assert torch.isfinite(out[1:-1]).all()
