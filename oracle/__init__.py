"""fp64 CPU oracle for sparse multi-head attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs anything here, and this
package imports nothing from the product.

The arithmetic lives in ``oracle.c`` (plain C, double precision); this module
compiles it with gcc on first use and wraps it with ctypes.  See ``oracle.c``
for the passages each function follows and the readings taken.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
brute-force dense masked softmax, closed forms and invariants; the linear
layer against a hand-worked example and a library matmul, the storage
rounding against a nearest-neighbour search, the projected block against a
dense numpy route (no function is unpinned).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``oracle/_build/liboracle.so`` (gcc, -O2,
    IEEE semantics: no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_double
            lib.gto_check_csr.argtypes = [i64, i64, vp, vp]
            lib.gto_check_csr.restype = ctypes.c_int
            lib.gto_sparse_mha_rows.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, vp, dbl,
                                                vp, i64, vp, vp, vp]
            lib.gto_sparse_mha_rows.restype = ctypes.c_int
            lib.gto_dense_attention.argtypes = [i64, i32, i32, vp, vp, vp, dbl, vp]
            lib.gto_dense_attention.restype = ctypes.c_int
            lib.gto_sparse_mha_bwd.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, dbl, vp, vp, vp]
            lib.gto_sparse_mha_bwd.restype = ctypes.c_int
            lib.gto_linear.argtypes = [i64, i32, i32, vp, vp, vp, vp]
            lib.gto_linear.restype = ctypes.c_int
            lib.gto_round_store.argtypes = [i64, vp, i32, vp]
            lib.gto_round_store.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


def check_csr(indptr, indices, n: int) -> bool:
    """True when indptr runs monotonically from 0 to nnz and every index is
    in [0, n)."""
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    return _load().gto_check_csr(n, int(indptr[-1]), _ptr(indptr), _ptr(indices)) == 0


def sparse_mha(indptr, indices, Q, K, V, scale, rows=None, want_probs=False,
               threads: int = 1, bias=None, values=None):
    """Sparse MHA forward in fp64.

    ``indptr`` int32 [N+1], ``indices`` int32 [nnz] (CSR by destination),
    ``Q, K, V`` float32 [N, H, D] (bf16 inputs passed as their exact float32
    values), ``scale`` the float32 scale (promoted to double).  ``rows``
    limits the computation to a list of rows (outputs then follow that list).
    Returns ``dict(out=[R,H,D] f64, logits=[nnz,H] f64 | None, probs=... )``;
    logits/probs entries of rows not computed stay NaN.
    ``threads`` > 1 splits the rows over host threads (each thread calls the
    same single-threaded C routine on a contiguous slice of rows).
    ``bias``: optional float32 [nnz, H] added to each logit (per-edge,
    per-head additive bias; -inf removes an entry).
    ``values``: optional float32 [nnz], the weighted adjacency's stored
    values; each logit is scale * (q.k * value).
    """
    lib = _load()
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    N, H, D = Q.shape
    nnz = int(indptr[-1])
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        if bias.shape != (nnz, H):
            raise OracleError(f"bias must be [nnz, H] = {(nnz, H)}, got {bias.shape}")
    if values is not None:
        values = np.ascontiguousarray(values, dtype=np.float32)
        if values.shape != (nnz,):
            raise OracleError(f"values must be [nnz] = {(nnz,)}, got {values.shape}")
    if rows is None:
        rows_arr = np.arange(N, dtype=np.int64)
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
    R = len(rows_arr)
    out = np.zeros((R, H, D), dtype=np.float64)
    logits = np.full((nnz, H), np.nan) if want_probs else None
    probs = np.full((nnz, H), np.nan) if want_probs else None
    s = float(np.float32(scale))

    def run(r0, r1):
        rc = lib.gto_sparse_mha_rows(
            N, nnz, H, D, _ptr(indptr), _ptr(indices), _ptr(Q), _ptr(K), _ptr(V), _ptr(values), _ptr(bias), s,
            _ptr(rows_arr[r0:r1]), r1 - r0, _ptr(out[r0:r1]),
            _ptr(logits), _ptr(probs))
        if rc != 0:
            raise OracleError(f"gto_sparse_mha_rows failed with code {rc}")

    threads = max(1, min(int(threads), R if R > 0 else 1))
    if threads == 1:
        run(0, R)
    else:
        # split by edge count so each thread gets a similar amount of work
        deg = (indptr[1:].astype(np.int64) - indptr[:-1])[rows_arr] + 1
        cum = np.cumsum(deg)
        cuts = [0] + [int(np.searchsorted(cum, cum[-1] * t / threads)) for t in range(1, threads)] + [R]
        errs = []

        def worker(a, b):
            try:
                if b > a:
                    run(a, b)
            except Exception as exc:  # pragma: no cover - re-raised below
                errs.append(exc)

        ts = [threading.Thread(target=worker, args=(cuts[t], cuts[t + 1])) for t in range(threads)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        if errs:
            raise errs[0]
    return dict(out=out, logits=logits, probs=probs)


def dense_attention(Q, K, V, scale):
    """All-pairs attention softmax(scale * Q K^T) V per head, fp64.
    ``Q, K, V`` float32 [n, H, D]; returns float64 [n, H, D]."""
    lib = _load()
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    n, H, D = Q.shape
    out = np.zeros((n, H, D), dtype=np.float64)
    rc = lib.gto_dense_attention(n, H, D, _ptr(Q), _ptr(K), _ptr(V),
                                 float(np.float32(scale)), _ptr(out))
    if rc != 0:
        raise OracleError(f"gto_dense_attention failed with code {rc}")
    return out


def sparse_mha_bwd(indptr, indices, Q, K, V, dO, scale):
    """Gradients of sum(out * dO) with respect to Q, K, V (fp64), for the
    sparse forward with binary A.  Returns ``dict(dQ=, dK=, dV=)``, each
    float64 [N, H, D]."""
    lib = _load()
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    Q, K, V, dO = (np.ascontiguousarray(x, dtype=np.float32) for x in (Q, K, V, dO))
    N, H, D = Q.shape
    dQ, dK, dV = (np.zeros((N, H, D), dtype=np.float64) for _ in range(3))
    rc = lib.gto_sparse_mha_bwd(N, int(indptr[-1]), H, D, _ptr(indptr), _ptr(indices), _ptr(Q), _ptr(K), _ptr(V),
                                _ptr(dO), float(np.float32(scale)), _ptr(dQ), _ptr(dK), _ptr(dV))
    if rc != 0:
        raise OracleError(f"gto_sparse_mha_bwd failed with code {rc}")
    return dict(dQ=dQ, dK=dK, dV=dV)


def linear(X, W, b=None, threads: int = 1):
    """Y = X W^T + b in fp64 (``gto_linear``): X float32 [M, Kin], W float32
    [Nout, Kin] (nn.Linear's weight), b float32 [Nout] or None.  Returns
    float64 [M, Nout].  ``threads`` > 1 splits the rows over host threads."""
    lib = _load()
    X = np.ascontiguousarray(X, dtype=np.float32)
    W = np.ascontiguousarray(W, dtype=np.float32)
    M, Kin = X.shape
    Nout, K2 = W.shape
    if K2 != Kin:
        raise OracleError(f"W must be [Nout, {Kin}], got {W.shape}")
    if b is not None:
        b = np.ascontiguousarray(b, dtype=np.float32)
        if b.shape != (Nout,):
            raise OracleError(f"b must be [{Nout}], got {b.shape}")
    Y = np.zeros((M, Nout), dtype=np.float64)

    def run(r0, r1):
        rc = lib.gto_linear(r1 - r0, Kin, Nout, _ptr(X[r0:r1]), _ptr(W), _ptr(b), _ptr(Y[r0:r1]))
        if rc != 0:
            raise OracleError(f"gto_linear failed with code {rc}")

    threads = max(1, min(int(threads), M if M > 0 else 1))
    if threads == 1:
        run(0, M)
    else:
        cuts = [M * t // threads for t in range(threads + 1)]
        ts = [threading.Thread(target=run, args=(cuts[t], cuts[t + 1])) for t in range(threads)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
    return Y


def round_store(x, precision: str):
    """The value an intermediate holds once stored (``gto_round_store``):
    "f32" the nearest float32; "bf16" that float32, then the nearest bf16
    (as float32).  Returns float32 of the same shape."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float32)
    mode = {"f32": 0, "bf16": 1}[precision]
    rc = lib.gto_round_store(x.size, _ptr(x), mode, _ptr(out))
    if rc != 0:
        raise OracleError(f"gto_round_store failed with code {rc}")
    return out


def _split_heads(Y, H, D, heads_inner):
    """[M, H*D] projection output -> [M, H, D].  Heads-major features
    (f = h*D + d): TransLayer's view(-1, h, d_qkv).  Heads-inner features
    (f = d*H + h): SparseMHA's reshape(N, head_dim, num_heads)."""
    M = Y.shape[0]
    if heads_inner:
        return Y.reshape(M, D, H).transpose(0, 2, 1)
    return Y.reshape(M, H, D)


def _merge_heads(O, heads_inner):
    """[M, H, D] -> [M, H*D] in the same feature order (the out projection's
    input: out.reshape(N, -1) / wv.view(-1, h * d_qkv))."""
    M, H, D = O.shape
    if heads_inner:
        return O.transpose(0, 2, 1).reshape(M, D * H)
    return O.reshape(M, H * D)


def sparse_mha_proj(indptr, indices, X, Wq, Wk, Wv, Wo, bq, bk, bv, bo, H, D, scale,
                    heads_inner=False, store="f32", rows=None, threads: int = 1):
    """The attention block with its projections, in fp64:

        q, k, v = X Wq^T + bq, X Wk^T + bk, X Wv^T + bv   (split into H heads of D)
        o       = SparseAttn(q, k, v, A)                    (sparse_mha)
        Y       = o Wo^T + bo                               (o's heads merged back)

    -- SparseMHA.forward of "Graph Transformer in a Nutshell" (nn.Linear maps
    with biases, features split head-inner: ``heads_inner=True``) and the
    attention part of TransLayer.forward in "Efficient Sparse Transformer
    implementation with DGL's builtin operators" (bias=False: pass None;
    head-major view).  The scale is an argument applied to q.k, as in
    sparse_mha (SparseMHA folds head_dim**-0.5 into q; the product is the
    same).

    ``store``: the precision the intermediates q, k, v and o are held in
    between the stages ("f32" or "bf16", see ``round_store``); the arithmetic
    of every stage is fp64.  ``rows``: compute Y for these rows only (the
    projections of their neighbours are computed, nothing else).
    Returns float64 [len(rows) or N, Nout]."""
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    X = np.ascontiguousarray(X, dtype=np.float32)
    N = X.shape[0]
    if rows is None:
        need = np.arange(N, dtype=np.int64)
        sel = np.arange(N, dtype=np.int64)
        lindptr, lindices = indptr, indices
    else:
        rows = np.asarray(rows, dtype=np.int64)
        starts, ends = indptr[rows].astype(np.int64), indptr[rows + 1].astype(np.int64)
        nbr = np.concatenate([indices[a:b] for a, b in zip(starts, ends)] + [np.zeros(0, np.int32)])
        need = np.unique(np.concatenate([rows, nbr.astype(np.int64)]))
        local = np.full(N, -1, dtype=np.int64)
        local[need] = np.arange(len(need))
        # a CSR over the needed nodes: the sampled rows keep their entries,
        # the other needed nodes (neighbours only) get none
        deg = np.zeros(len(need), dtype=np.int64)
        deg[local[rows]] = ends - starts
        lindptr = np.zeros(len(need) + 1, dtype=np.int64)
        np.cumsum(deg, out=lindptr[1:])
        lindices = np.empty(int(lindptr[-1]), dtype=np.int32)
        for r, a, b in zip(rows, starts, ends):
            o = lindptr[local[r]]
            lindices[o:o + (b - a)] = local[indices[a:b]]
        lindptr = lindptr.astype(np.int32)
        sel = local[rows]
    Xn = X[need]
    q, k, v = (round_store(_split_heads(linear(Xn, W, b, threads), H, D, heads_inner), store)
               for W, b in ((Wq, bq), (Wk, bk), (Wv, bv)))
    o = sparse_mha(lindptr, lindices, q, k, v, scale, rows=sel, threads=threads)["out"]
    o = round_store(o, store)
    return linear(_merge_heads(o, heads_inner), Wo, bo, threads)
