"""GB300 sparse multi-head attention: Python binding of ``libgtattn.so``.

A thin ctypes layer over the C ABI declared in ``include/gtattn.h``: each
function has the C entry point's name and arguments, takes torch CUDA tensors
(or raw device pointers as ints) and raises :class:`GtattnError` on a non-OK
status.  It only marshals arguments; every step runs in the library's CUDA
kernels.  There is no CPU fallback: without the built library (or without a
GPU) the calls raise.

    out[i,h,:] = sum_{e in row i} softmax_e(scale * q_i . k_j) v_j

over a CSR graph keyed by destination (row i attends over
indices[indptr[i]:indptr[i+1]]); empty rows give zeros.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB, build

__all__ = [
    "GtattnError", "Plan", "build", "load", "gtattn_fwd", "gtattn_fwd_plan", "gtattn_fwd_probs", "gtattn_fwd_bias", "gtattn_fwd_weighted", "gtattn_bwd", "gtattn_fwd_ndh",
    "gtattn_fwd_noalloc", "gtattn_fwd_host", "gtattn_fwd_proj", "gtattn_device_errors", "gtattn_bwd_plan",
    "gtattn_fwd_plan_stats", "gtattn_csr_build",
    "gtattn_plan_destroy", "gtattn_plan_get_info", "gtattn_coo_to_csr",
    "gtattn_csr_validate", "gtattn_status_string", "gtattn_profile_enable", "gtattn_profile_read",
    "sparse_mha", "GTATTN_F32", "GTATTN_BF16", "GTATTN_BF16_OUT_F32",
    "GTATTN_KERNEL_AUTO", "GTATTN_KERNEL_VECTOR", "GTATTN_KERNEL_GENERIC", "GTATTN_KERNEL_NARROW",
    "EXPORTED_SYMBOLS",
]

GTATTN_OK, GTATTN_ERR_INVALID_ARG, GTATTN_ERR_BAD_CSR, GTATTN_ERR_UNSUPPORTED = 0, 1, 2, 3
GTATTN_ERR_CUDA, GTATTN_ERR_NO_MEMORY, GTATTN_ERR_TIMEOUT = 4, 5, 6
GTATTN_F32, GTATTN_BF16, GTATTN_BF16_OUT_F32 = 0, 1, 2
GTATTN_KERNEL_AUTO, GTATTN_KERNEL_VECTOR, GTATTN_KERNEL_GENERIC, GTATTN_KERNEL_NARROW = 0, 1, 2, 3

EXPORTED_SYMBOLS = (
    "gtattn_status_string", "gtattn_last_error", "gtattn_csr_build", "gtattn_plan_destroy",
    "gtattn_plan_get_info", "gtattn_fwd", "gtattn_fwd_plan", "gtattn_fwd_probs",
    "gtattn_coo_to_csr", "gtattn_csr_validate", "gtattn_profile_enable", "gtattn_profile_read",
    "gtattn_fwd_noalloc", "gtattn_fwd_host", "gtattn_fwd_bias", "gtattn_fwd_weighted", "gtattn_bwd",
    "gtattn_fwd_ndh", "gtattn_fwd_proj", "gtattn_device_errors", "gtattn_bwd_plan", "gtattn_fwd_plan_stats",
)
KCAT_NAMES = ("bin", "rows", "combine", "softmax", "dense", "gemm")


class GtattnError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = f"{what}: {gtattn_status_string(status)} ({status})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


class PlanOpts(ctypes.Structure):
    _fields_ = [("long_row_min", ctypes.c_int32), ("chunk_edges", ctypes.c_int32),
                ("detect_dense", ctypes.c_int32), ("kernel", ctypes.c_int32), ("wait_cycles", ctypes.c_int32),
                ("test_stall", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("nnz", ctypes.c_int64), ("n_long_rows", ctypes.c_int32),
                ("n_chunks", ctypes.c_int32), ("n_dense_blocks", ctypes.c_int32),
                ("n_dense_rows", ctypes.c_int32), ("n_empty_rows", ctypes.c_int32),
                ("max_degree", ctypes.c_int32), ("n_buckets", ctypes.c_int32),
                ("bucket_rows", ctypes.c_int32 * 64), ("device_error", ctypes.c_int32)]

    def as_dict(self):
        d = {k: getattr(self, k) for k, _ in self._fields_ if k != "bucket_rows"}
        d["bucket_rows"] = list(self.bucket_rows)[: self.n_buckets]
        return d


class Profile(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int32 * 8), ("groups", ctypes.c_int32 * 8),
                ("ms", ctypes.c_double * 8)]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load ``libgtattn.so`` (building it first if it is missing) and
    declare the C signatures.  Raises if it cannot be built or loaded."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB
        if not os.path.exists(p):
            build()
        lib = ctypes.CDLL(p)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        sig = {
            "gtattn_status_string": ([i32], ctypes.c_char_p),
            "gtattn_last_error": ([], ctypes.c_char_p),
            "gtattn_csr_build": ([vp, vp, i64, i64, vp, vp, vp], i32),
            "gtattn_plan_destroy": ([vp], i32),
            "gtattn_plan_get_info": ([vp, vp], i32),
            "gtattn_fwd": ([vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp], i32),
            "gtattn_fwd_plan": ([vp, vp, vp, vp, vp, vp, vp, i32, i32, f32, i32, vp], i32),
            "gtattn_fwd_probs": ([vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp], i32),
            "gtattn_fwd_bias": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp], i32),
            "gtattn_fwd_weighted": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp], i32),
            "gtattn_bwd": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp], i32),
            "gtattn_fwd_ndh": ([vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp], i32),
            "gtattn_coo_to_csr": ([vp, vp, i64, i64, vp, vp, vp], i32),
            "gtattn_csr_validate": ([vp, vp, i64, i64, vp], i32),
            "gtattn_fwd_noalloc": ([vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp], i32),
            "gtattn_fwd_host": ([vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, f32, i32, vp], i32),
            "gtattn_fwd_proj": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i32, i32, i32, i32, i32, f32,
                                 i32, vp], i32),
            "gtattn_device_errors": ([vp, i32], i32),
            "gtattn_bwd_plan": ([vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, f32, i32, vp], i32),
            "gtattn_fwd_plan_stats": ([vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, f32, i32, vp], i32),
            "gtattn_profile_enable": ([i32], i32),
            "gtattn_profile_read": ([vp, i32], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def gtattn_status_string(status: int) -> str:
    try:
        return load().gtattn_status_string(int(status)).decode()
    except OSError:
        return str(status)


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------
def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if x.numel() and not x.is_cuda:
            raise ValueError("expected a CUDA tensor")
        if not x.is_contiguous():
            raise ValueError("expected a contiguous tensor")
        return x.data_ptr() or None
    raise TypeError(f"cannot take a device pointer of {type(x)}")


def _host_ptr(x):
    """Pointer of a contiguous host (CPU) tensor, or None."""
    if x is None:
        return None
    if getattr(x, "is_cuda", False):
        raise ValueError("expected a host (CPU) tensor")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr() or None


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(q, out=None):
    """gtattn_dtype of (Q, out): fp32/fp32, bf16/bf16 or bf16/fp32."""
    import torch
    if q.dtype == torch.float32 and (out is None or out.dtype == torch.float32):
        return GTATTN_F32
    if q.dtype == torch.bfloat16 and (out is None or out.dtype == torch.bfloat16):
        return GTATTN_BF16
    if q.dtype == torch.bfloat16 and out.dtype == torch.float32:
        return GTATTN_BF16_OUT_F32
    raise ValueError(f"unsupported dtypes {q.dtype} -> {None if out is None else out.dtype}")


def _check(status, what):
    if status != GTATTN_OK:
        detail = load().gtattn_last_error().decode() if status == GTATTN_ERR_CUDA else ""
        raise GtattnError(status, what, detail)


# --------------------------------------------------------------------------
# the C entry points
# --------------------------------------------------------------------------
def gtattn_fwd(indptr, indices, Q, K, V, out, N, nnz, H, D, scale, dtype, stream=None):
    _check(load().gtattn_fwd(_ptr(indptr), _ptr(indices), _ptr(Q), _ptr(K), _ptr(V), _ptr(out),
                             int(N), int(nnz), int(H), int(D), float(scale), int(dtype),
                             _stream(stream)), "gtattn_fwd")


def gtattn_fwd_noalloc(indptr, indices, Q, K, V, out, N, nnz, H, D, scale, dtype, stream=None):
    """gtattn_fwd for callers that cannot allocate device memory: temporaries
    live in the library's fixed 32 MiB device array (see include/gtattn.h for
    the size limit and why overlapping calls race)."""
    _check(load().gtattn_fwd_noalloc(_ptr(indptr), _ptr(indices), _ptr(Q), _ptr(K), _ptr(V), _ptr(out),
                                     int(N), int(nnz), int(H), int(D), float(scale), int(dtype),
                                     _stream(stream)), "gtattn_fwd_noalloc")


def gtattn_fwd_host(indptr, indices, Q, K, V, out, N, nnz, H, D, scale, dtype, stream=None):
    """gtattn_fwd on host (CPU, preferably pinned) tensors: copies in,
    computes and copies the output back, overlapped, ordered on `stream`;
    `out` is complete once `stream` has passed the call."""
    _check(load().gtattn_fwd_host(_host_ptr(indptr), _host_ptr(indices), _host_ptr(Q), _host_ptr(K),
                                  _host_ptr(V), _host_ptr(out),
                                  int(N), int(nnz), int(H), int(D), float(scale), int(dtype),
                                  _stream(stream)), "gtattn_fwd_host")


def gtattn_fwd_proj(indptr, indices, X, Wqkv, bqkv, Wo, bo, Y, N, nnz, F_in, H, D, F_out, scale, dtype,
                    heads_inner=False, qkv=None, attn=None, stream=None):
    """The attention block with its projections: q, k, v = X Wqkv^T + bqkv
    (weights of the three maps stacked, nn.Linear layout), the sparse
    attention, Y = o Wo^T + bo.  bqkv / bo: fp32 device tensors or None;
    qkv ([3, N, H, D]) and attn ([N, H, D]) optionally receive the
    intermediates; heads_inner: SparseMHA's feature order (d*H + h)."""
    _check(load().gtattn_fwd_proj(_ptr(indptr), _ptr(indices), _ptr(X), _ptr(Wqkv), _ptr(bqkv), _ptr(Wo), _ptr(bo),
                                  _ptr(Y), _ptr(qkv), _ptr(attn), int(N), int(nnz), int(F_in), int(H), int(D),
                                  int(F_out), 1 if heads_inner else 0, float(scale), int(dtype), _stream(stream)),
           "gtattn_fwd_proj")


def gtattn_bwd_plan(plan, indptr, indices, Q, K, V, dO, dQ, dK, dV, H, D, scale, dtype, O=None, stats=None,
                    stream=None):
    """gtattn_bwd on a plan's binning; the plan keeps the source-major
    pattern built by its first backward call.  O and stats: the fp32 output
    and row statistics of gtattn_fwd_plan_stats (both or neither); given,
    the forward is not recomputed."""
    _check(load().gtattn_bwd_plan(plan.handle if isinstance(plan, Plan) else plan, _ptr(indptr), _ptr(indices),
                                  _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(stats), _ptr(dO), _ptr(dQ), _ptr(dK),
                                  _ptr(dV), int(H), int(D), float(scale), int(dtype), _stream(stream)),
           "gtattn_bwd_plan")


def gtattn_device_errors(reset: bool = True) -> int:
    """Error codes recorded on the current device by the plan-less
    tensor-core kernels (1: a bounded wait gave up); synchronises."""
    code = ctypes.c_int(0)
    _check(load().gtattn_device_errors(ctypes.byref(code), 1 if reset else 0), "gtattn_device_errors")
    return code.value


def gtattn_fwd_plan(plan, indptr, indices, Q, K, V, out, H, D, scale, dtype, stream=None):
    _check(load().gtattn_fwd_plan(plan.handle if isinstance(plan, Plan) else plan, _ptr(indptr),
                                  _ptr(indices), _ptr(Q), _ptr(K), _ptr(V), _ptr(out), int(H), int(D),
                                  float(scale), int(dtype), _stream(stream)), "gtattn_fwd_plan")


def gtattn_fwd_plan_stats(plan, indptr, indices, Q, K, V, out, stats, H, D, scale, dtype, stream=None):
    """gtattn_fwd_plan that also writes the rows' log2-sum-exp (fp32 [N, H])."""
    _check(load().gtattn_fwd_plan_stats(plan.handle if isinstance(plan, Plan) else plan, _ptr(indptr),
                                        _ptr(indices), _ptr(Q), _ptr(K), _ptr(V), _ptr(out), _ptr(stats), int(H),
                                        int(D), float(scale), int(dtype), _stream(stream)),
           "gtattn_fwd_plan_stats")


def gtattn_fwd_probs(indptr, indices, Q, K, V, out, logits, probs, N, nnz, H, D, scale, dtype,
                     stream=None):
    _check(load().gtattn_fwd_probs(_ptr(indptr), _ptr(indices), _ptr(Q), _ptr(K), _ptr(V), _ptr(out),
                                   _ptr(logits), _ptr(probs), int(N), int(nnz), int(H), int(D),
                                   float(scale), int(dtype), _stream(stream)), "gtattn_fwd_probs")


def gtattn_fwd_bias(indptr, indices, Q, K, V, bias, out, N, nnz, H, D, scale, dtype, logits=None, probs=None,
                    stream=None):
    """Forward with a per-edge, per-head additive bias (fp32 [nnz, H] device
    tensor); logits/probs (optional) select the unfused path."""
    _check(load().gtattn_fwd_bias(_ptr(indptr), _ptr(indices), _ptr(Q), _ptr(K), _ptr(V), _ptr(bias), _ptr(out),
                                  _ptr(logits), _ptr(probs), int(N), int(nnz), int(H), int(D), float(scale),
                                  int(dtype), _stream(stream)), "gtattn_fwd_bias")


def gtattn_fwd_weighted(indptr, indices, values, Q, K, V, out, N, nnz, H, D, scale, dtype, logits=None, probs=None,
                        stream=None):
    """Forward on a weighted adjacency (values: fp32 [nnz] device tensor, A's
    stored values); logits/probs (optional) select the unfused path."""
    _check(load().gtattn_fwd_weighted(_ptr(indptr), _ptr(indices), _ptr(values), _ptr(Q), _ptr(K), _ptr(V),
                                      _ptr(out), _ptr(logits), _ptr(probs), int(N), int(nnz), int(H), int(D),
                                      float(scale), int(dtype), _stream(stream)), "gtattn_fwd_weighted")


def gtattn_bwd(indptr, indices, Q, K, V, dO, dQ, dK, dV, N, nnz, H, D, scale, dtype, stream=None):
    """Gradients of sum(out * dO) with respect to Q, K, V (fp32 device tensors
    dQ, dK, dV, overwritten)."""
    _check(load().gtattn_bwd(_ptr(indptr), _ptr(indices), _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ), _ptr(dK),
                             _ptr(dV), int(N), int(nnz), int(H), int(D), float(scale), int(dtype), _stream(stream)),
           "gtattn_bwd")


def gtattn_fwd_ndh(indptr, indices, Q, K, V, out, N, nnz, H, D, scale, dtype, stream=None):
    """gtattn_fwd on head-innermost [N, D, H] tensors."""
    _check(load().gtattn_fwd_ndh(_ptr(indptr), _ptr(indices), _ptr(Q), _ptr(K), _ptr(V), _ptr(out), int(N), int(nnz),
                                 int(H), int(D), float(scale), int(dtype), _stream(stream)), "gtattn_fwd_ndh")


def gtattn_csr_build(indptr, indices, N, nnz, opts=None, stream=None):
    """Returns a raw plan handle (int); prefer :class:`Plan`."""
    h = ctypes.c_void_p()
    o = ctypes.byref(opts) if opts is not None else None
    _check(load().gtattn_csr_build(_ptr(indptr), _ptr(indices), int(N), int(nnz), o, ctypes.byref(h),
                                   _stream(stream)), "gtattn_csr_build")
    return h.value


def gtattn_plan_destroy(handle):
    _check(load().gtattn_plan_destroy(handle), "gtattn_plan_destroy")


def gtattn_plan_get_info(handle) -> dict:
    info = PlanInfo()
    _check(load().gtattn_plan_get_info(handle, ctypes.byref(info)), "gtattn_plan_get_info")
    return info.as_dict()


def gtattn_coo_to_csr(src, dst, nnz, N, indptr, indices, stream=None):
    _check(load().gtattn_coo_to_csr(_ptr(src), _ptr(dst), int(nnz), int(N), _ptr(indptr), _ptr(indices),
                                    _stream(stream)), "gtattn_coo_to_csr")


def gtattn_csr_validate(indptr, indices, N, nnz, stream=None) -> bool:
    """True for a well-formed CSR, False for GTATTN_ERR_BAD_CSR; raises otherwise."""
    st = load().gtattn_csr_validate(_ptr(indptr), _ptr(indices), int(N), int(nnz), _stream(stream))
    if st == GTATTN_ERR_BAD_CSR:
        return False
    _check(st, "gtattn_csr_validate")
    return True


def gtattn_profile_enable(on: bool = True):
    _check(load().gtattn_profile_enable(int(bool(on))), "gtattn_profile_enable")


def gtattn_profile_read(reset: bool = True) -> dict:
    """Per-category kernel launches and summed CUDA-event milliseconds
    recorded while profiling was enabled."""
    pr = Profile()
    _check(load().gtattn_profile_read(ctypes.byref(pr), int(bool(reset))), "gtattn_profile_read")
    return {name: dict(launches=pr.launches[k], groups=pr.groups[k], ms=pr.ms[k])
            for k, name in enumerate(KCAT_NAMES)}


class Plan:
    """Owns a plan built by ``gtattn_csr_build`` (freed on close/GC)."""

    def __init__(self, indptr, indices, N=None, nnz=None, long_row_min=0, chunk_edges=0,
                 detect_dense=False, kernel=GTATTN_KERNEL_AUTO, wait_cycles=0, test_stall=False,
                 stream=None):
        N = int(indptr.numel() - 1) if N is None else int(N)
        nnz = int(indices.numel()) if nnz is None else int(nnz)
        self.opts = PlanOpts(int(long_row_min), int(chunk_edges), int(bool(detect_dense)), int(kernel),
                             int(wait_cycles), int(bool(test_stall)))
        self.handle = gtattn_csr_build(indptr, indices, N, nnz, self.opts, stream)
        self.N, self.nnz = N, nnz
        self._keep = (indptr, indices)

    def info(self) -> dict:
        return gtattn_plan_get_info(self.handle)

    def close(self):
        if getattr(self, "handle", None):
            gtattn_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def sparse_mha(indptr, indices, Q, K, V, scale=None, out=None, plan=None, stream=None):
    """Convenience wrapper: allocates ``out`` and calls ``gtattn_fwd`` (or
    ``gtattn_fwd_plan`` when a :class:`Plan` is given)."""
    import torch
    N, H, D = Q.shape
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty_like(Q)
    dt = _dtype_code(Q, out)
    if plan is not None:
        gtattn_fwd_plan(plan, indptr, indices, Q, K, V, out, H, D, scale, dt, stream)
    else:
        gtattn_fwd(indptr, indices, Q, K, V, out, N, indices.numel(), H, D, scale, dt, stream)
    return out
