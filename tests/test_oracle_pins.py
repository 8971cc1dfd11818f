"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things other than itself:
  * a hand-derived worked example (tests/golden/hand_worked_example.json);
  * brute-force dense masked softmax attention on tiny graphs, built from the
    COO edge list (not the CSR) -- the masked-softmax pattern of the GAT
    comparison in "Graph Transformer theory, derivation and implementation"
    and its b_inf = -inf reading of disconnected pairs;
  * closed forms: complete graph == dense attention (scipy's softmax),
    single neighbour -> v_j exactly, q = 0 or scale = 0 -> neighbour mean,
    V constant -> constant, empty row -> exact 0, duplicate entries weigh
    twice;
  * invariants: probabilities sum to one; permutation equivariance (same
    page, "permutation equivariant"); invariance to shifting every key by
    one vector;
  * mutation checks: plausible mistakes planted in a copy of oracle.c (the
    query taken from the wrong node, a dropped scale, a wrong head offset,
    values gathered from the destination, a sign error in the exponent, a
    missing normalisation, a dropped last edge) each fail the brute-force
    pin.
"""
import json
import math
import os
import re
import subprocess
import tempfile
import ctypes

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_example.json")


# --------------------------------------------------------------------------
# helpers (independent of the oracle's code)
# --------------------------------------------------------------------------
def _val(x):
    if isinstance(x, str):
        table = {"ln3": math.log(3.0), "-ln3": -math.log(3.0)}
        if x in table:
            return table[x]
        num, den = x.split("/")
        return float(num) / float(den)
    return float(x)


def _arr(nested):
    if isinstance(nested, list):
        return [_arr(v) for v in nested]
    return _val(nested)


def brute_force(src, dst, n, Q, K, V, scale):
    """Dense route: count matrix A[i, j] = #edges j -> i, logits
    scale * q_i.k_j (+ log count), non-edges -inf, row softmax, times V.
    Rows without edges give 0."""
    A = np.zeros((n, n))
    np.add.at(A, (np.asarray(dst), np.asarray(src)), 1.0)
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
    logits = scale * np.einsum("ihd,jhd->hij", q, k)
    with np.errstate(divide="ignore"):
        logits = logits + np.log(A)[None]          # log 0 = -inf masks non-edges
    has = (A.sum(1) > 0)
    out = np.zeros_like(q)
    lg = logits[:, has, :]
    m = lg.max(axis=2, keepdims=True)
    w = np.exp(lg - m)
    p = w / w.sum(axis=2, keepdims=True)
    out[has] = np.einsum("hij,jhd->ihd", p, v)
    return out


def brute_force_bias(indptr, indices, n, Q, K, V, scale, bias):
    """Dense route with a per-edge additive bias: B[h, i, j] = bias of the
    entry j -> i (graphs without duplicate entries), non-edges -inf; logits
    scale * q_i.k_j + B, row softmax, times V; rows whose logits are all
    -inf give 0."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
    H = q.shape[1]
    B = np.full((H, n, n), -np.inf)
    dst = np.repeat(np.arange(n), np.diff(indptr))
    for e in range(len(indices)):
        B[:, dst[e], indices[e]] = np.asarray(bias, dtype=np.float64)[e]
    logits = scale * np.einsum("ihd,jhd->hij", q, k) + B
    out = np.zeros_like(q)
    for h in range(H):
        for i in range(n):
            row = logits[h, i]
            if not np.isfinite(row).any():
                continue
            w = np.exp(row - row[np.isfinite(row)].max())
            out[i, h] = (w / w.sum()) @ v[:, h]
    return out


def _csr_coo(indptr, indices):
    dst = np.repeat(np.arange(len(indptr) - 1), np.diff(indptr))
    return np.asarray(indices, dtype=np.int64), dst


def _rand_feats(rng, n, h, d, std=1.0):
    return [(rng.standard_normal((n, h, d)) * std).astype(np.float32) for _ in range(3)]


# --------------------------------------------------------------------------
# the worked example
# --------------------------------------------------------------------------
def test_hand_worked_example():
    g = json.load(open(GOLDEN))
    Q = np.array(_arr(g["Q"]), dtype=np.float32)
    K = np.array(_arr(g["K"]), dtype=np.float32)
    V = np.array(_arr(g["V"]), dtype=np.float32)
    r = oracle.sparse_mha(np.array(g["indptr"]), np.array(g["indices"]), Q, K, V,
                          g["scale"], want_probs=True)
    np.testing.assert_allclose(r["out"], np.array(_arr(g["expected_out"])), rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(r["probs"], np.array(_arr(g["expected_probs"])), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(r["logits"], np.array(_arr(g["expected_logits"])), rtol=1e-6, atol=1e-7)
    # the empty row is exactly zero, the single-neighbour row is v exactly
    assert np.all(r["out"][1] == 0.0)
    assert np.array_equal(r["out"][2], V[2].astype(np.float64))


# --------------------------------------------------------------------------
# brute force
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(6))
def test_brute_force_random_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(2, 48))
    e = int(rng.integers(0, n * n // 2 + 1))
    H = int(rng.integers(1, 5))
    D = int(rng.integers(1, 9))
    pick = rng.choice(n * n, size=e, replace=False)
    src, dst = pick // n, pick % n
    indptr, indices = wl.csr_by_destination(src, dst, n)
    Q, K, V = _rand_feats(rng, n, H, D)
    scale = float(np.float32(1 / math.sqrt(D)))
    got = oracle.sparse_mha(indptr, indices, Q, K, V, scale)["out"]
    ref = brute_force(src, dst, n, Q, K, V, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_brute_force_tiny_random_workload():
    w = wl.make_workload("tiny_random")
    src, dst = _csr_coo(w.indptr, w.indices)
    got = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale)["out"]
    ref = brute_force(src, dst, w.N, w.Q, w.K, w.V, w.scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_duplicates_count_twice():
    rng = np.random.default_rng(7)
    n, H, D = 9, 3, 4
    src = rng.integers(0, n, 40)
    dst = rng.integers(0, n, 40)                 # with repeats
    indptr, indices = wl.csr_by_destination(src, dst, n)
    Q, K, V = _rand_feats(rng, n, H, D)
    got = oracle.sparse_mha(indptr, indices, Q, K, V, 0.5)["out"]
    ref = brute_force(src, dst, n, Q, K, V, 0.5)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_direction_matters():
    """Row i attends over its sources j (edges j -> i): a one-way edge
    0 -> 1 gives row 1 = v_0 and leaves row 0 empty."""
    rng = np.random.default_rng(3)
    Q, K, V = _rand_feats(rng, 2, 2, 3)
    indptr, indices = wl.csr_by_destination([0], [1], 2)
    out = oracle.sparse_mha(indptr, indices, Q, K, V, 1.0)["out"]
    assert np.all(out[0] == 0)
    assert np.array_equal(out[1], V[0].astype(np.float64))


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def test_complete_graph_equals_dense_attention():
    rng = np.random.default_rng(11)
    n, H, D = 23, 3, 16
    Q, K, V = _rand_feats(rng, n, H, D)
    scale = float(np.float32(1 / math.sqrt(D)))
    indptr, indices, _ = wl.dense_block_csr(n_blocks=1, block=n)
    got = oracle.sparse_mha(indptr, indices, Q, K, V, scale)["out"]
    # library route: scipy softmax over all pairs, per head
    S = scale * np.einsum("ihd,jhd->hij", Q.astype(np.float64), K.astype(np.float64))
    ref = np.einsum("hij,jhd->ihd", sp_softmax(S, axis=2), V.astype(np.float64))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)
    dense = oracle.dense_attention(Q, K, V, scale)
    np.testing.assert_allclose(dense, ref, rtol=1e-12, atol=1e-13)


def test_dense_blocks_equal_blockwise_dense_attention():
    w = wl.make_workload("dense_blocks", n_blocks=2, block=32)
    got = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale)["out"]
    for b in range(2):
        sl = slice(32 * b, 32 * (b + 1))
        S = w.scale * np.einsum("ihd,jhd->hij", w.Q[sl].astype(np.float64), w.K[sl].astype(np.float64))
        ref = np.einsum("hij,jhd->ihd", sp_softmax(S, axis=2), w.V[sl].astype(np.float64))
        np.testing.assert_allclose(got[sl], ref, rtol=1e-12, atol=1e-13)


def test_single_neighbour_is_exact():
    rng = np.random.default_rng(5)
    n, H, D = 50, 4, 7
    Q, K, V = _rand_feats(rng, n, H, D, std=30.0)
    src = rng.integers(0, n, n)
    indptr, indices = wl.csr_by_destination(src, np.arange(n), n)
    out = oracle.sparse_mha(indptr, indices, Q, K, V, 0.125)["out"]
    assert np.array_equal(out, V[src].astype(np.float64))


@pytest.mark.parametrize("how", ["q_zero", "scale_zero"])
def test_uniform_weights_give_neighbour_mean(how):
    rng = np.random.default_rng(9)
    w = wl.make_workload("molecules", n_graphs=6)
    Q, K, V = w.Q.copy(), w.K, w.V
    scale = w.scale
    if how == "q_zero":
        Q[:] = 0
    else:
        scale = 0.0
    out = oracle.sparse_mha(w.indptr, w.indices, Q, K, V, scale)["out"]
    ref = np.zeros_like(out)
    for i in range(w.N):
        nb = w.indices[w.indptr[i]:w.indptr[i + 1]]
        if len(nb):
            ref[i] = V[nb].astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-14)


def test_constant_values_and_empty_rows():
    rng = np.random.default_rng(12)
    indptr, indices = wl.random_csr(rng, 40, 90, self_loops=True)
    Q, K, _ = _rand_feats(rng, 40, 2, 5)
    V = np.full((40, 2, 5), 1.75, dtype=np.float32)
    out = oracle.sparse_mha(indptr, indices, Q, K, V, 0.4)["out"]
    deg = np.diff(indptr)
    assert (deg == 0).any()
    assert np.all(out[deg == 0] == 0.0)
    np.testing.assert_allclose(out[deg > 0], 1.75, rtol=1e-14)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def test_probs_sum_to_one():
    w = wl.small_workload("rmat")
    r = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, want_probs=True)
    p = r["probs"]
    assert np.all(p > 0) and np.all(p <= 1)
    sums = np.add.reduceat(p, w.indptr[:-1][np.diff(w.indptr) > 0], axis=0)
    np.testing.assert_allclose(sums, 1.0, rtol=0, atol=1e-14)
    # logits are scale * q.k at the CSR position
    dst = np.repeat(np.arange(w.N), np.diff(w.indptr))
    lref = w.scale * np.einsum("ehd,ehd->eh", w.Q[dst].astype(np.float64),
                               w.K[w.indices].astype(np.float64))
    np.testing.assert_allclose(r["logits"], lref, rtol=1e-12, atol=1e-12)


def test_permutation_equivariance():
    rng = np.random.default_rng(21)
    w = wl.small_workload("molecules")
    src, dst = _csr_coo(w.indptr, w.indices)
    perm = rng.permutation(w.N)                      # node i -> perm[i]
    inv = np.argsort(perm)
    ip2, ix2 = wl.csr_by_destination(perm[src], perm[dst], w.N)
    Q2, K2, V2 = w.Q[inv], w.K[inv], w.V[inv]
    a = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale)["out"]
    b = oracle.sparse_mha(ip2, ix2, Q2, K2, V2, w.scale)["out"]
    np.testing.assert_allclose(b[perm], a, rtol=1e-12, atol=1e-14)


def test_key_shift_invariance():
    rng = np.random.default_rng(22)
    indptr, indices = wl.random_csr(rng, 60, 400, self_loops=True)
    Q, K, V = _rand_feats(rng, 60, 3, 8)
    # keys and shift on coarse grids so that K + u is exact in float32
    K = (np.round(K * 64) / 64).astype(np.float32)
    u = np.round(rng.standard_normal((1, 3, 8)) * 4) / 4
    a = oracle.sparse_mha(indptr, indices, Q, K, V, 0.3)["out"]
    K2 = (K.astype(np.float64) + u).astype(np.float32)
    assert np.array_equal(K2.astype(np.float64), K.astype(np.float64) + u)
    b = oracle.sparse_mha(indptr, indices, Q, K2, V, 0.3)["out"]
    np.testing.assert_allclose(b, a, rtol=1e-10, atol=1e-12)


def test_rows_subset_matches_full():
    w = wl.small_workload("erdos_renyi")
    full = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, threads=4)["out"]
    rows = np.array([0, 17, 4000, 5999, 17])
    part = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, rows=rows)["out"]
    assert np.array_equal(part, full[rows])


def test_bad_csr_is_rejected():
    indptr = np.array([0, 2, 1], dtype=np.int32)
    assert not oracle.check_csr(indptr, np.array([0, 1], dtype=np.int32), 2)
    assert not oracle.check_csr(np.array([0, 1, 2], dtype=np.int32), np.array([0, 5], dtype=np.int32), 2)
    assert oracle.check_csr(np.array([0, 1, 2], dtype=np.int32), np.array([0, 1], dtype=np.int32), 2)
    Q = np.zeros((2, 1, 1), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.sparse_mha(indptr, np.array([0, 1], dtype=np.int32), Q, Q, Q, 1.0)


# --------------------------------------------------------------------------
# mutation checks: each planted mistake must fail a pin
# --------------------------------------------------------------------------
MUTATIONS = {
    # q_i . k_j with the operands' node indices swapped (transposed product)
    "swap_qk_nodes": ("const float* q = Q + i * HD + (int64_t)h * D;",
                      "const float* q = Q + (int64_t)indices[beg] * HD + (int64_t)h * D;"),
    "drop_scale": ("l[k] = scale * dot;", "l[k] = dot;"),
    "wrong_head_offset": ("const float* kj = K + j * HD + (int64_t)h * D;",
                          "const float* kj = K + j * HD;"),
    "values_from_destination": ("const float* vj = V + j * HD + (int64_t)h * D;",
                                "const float* vj = V + i * HD + (int64_t)h * D;"),
    "sign_error": ("p[k] = exp(l[k] - m);", "p[k] = exp(m - l[k]);"),
    "no_normalisation": ("for (int64_t k = 0; k < deg; ++k) p[k] /= S;", ""),
    "last_edge_dropped": ("for (int64_t k = 0; k < deg; ++k) {\n                const int64_t j = indices[beg + k];\n                const float* vj",
                          "for (int64_t k = 0; k + 1 < deg; ++k) {\n                const int64_t j = indices[beg + k];\n                const float* vj"),
}


def _compile_mutant(src_text, tmpdir, name):
    path = os.path.join(tmpdir, name + ".c")
    with open(path, "w") as f:
        f.write(src_text)
    so = os.path.join(tmpdir, name + ".so")
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", path, "-o", so, "-lm"], check=True)
    lib = ctypes.CDLL(so)
    i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_double
    lib.gto_sparse_mha_rows.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, vp, dbl, vp, i64, vp, vp, vp]
    lib.gto_sparse_mha_rows.restype = ctypes.c_int
    return lib


def _run_mutant(lib, indptr, indices, Q, K, V, scale, bias=None, values=None):
    N, H, D = Q.shape
    out = np.zeros((N, H, D))
    p = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    indptr = np.ascontiguousarray(indptr, np.int32)
    indices = np.ascontiguousarray(indices, np.int32)
    rc = lib.gto_sparse_mha_rows(N, int(indptr[-1]), H, D, p(indptr), p(indices), p(Q), p(K), p(V), p(values), p(bias),
                                 float(scale), None, N, p(out), None, None)
    assert rc == 0
    return out


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(name):
    text = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTATIONS[name]
    # plant the mistake in the sparse routine (the first occurrence)
    assert 0 <= text.find(old) < text.index("int gto_dense_attention("), f"anchor for {name} missing"
    mutant = text.replace(old, new, 1)
    rng = np.random.default_rng(1234)
    n, H, D = 17, 3, 5
    pick = rng.choice(n * n, size=80, replace=False)
    src, dst = pick // n, pick % n
    indptr, indices = wl.csr_by_destination(src, dst, n)
    Q, K, V = _rand_feats(rng, n, H, D)
    ref = brute_force(src, dst, n, Q, K, V, 0.7)
    with tempfile.TemporaryDirectory() as td:
        lib = _compile_mutant(mutant, td, name)
        got = _run_mutant(lib, indptr, indices, Q, K, V, 0.7)
    assert not np.allclose(got, ref, rtol=1e-9, atol=1e-12), f"pin missed mutation {name}"


# --------------------------------------------------------------------------
# per-edge additive bias (Graphormer spatial encoding)
# --------------------------------------------------------------------------
def _bias_graph(rng, n, e, H, D):
    pick = rng.choice(n * n, size=e, replace=False)
    indptr, indices = wl.csr_by_destination(pick // n, pick % n, n)
    Q, K, V = _rand_feats(rng, n, H, D)
    return indptr, indices, Q, K, V


@pytest.mark.parametrize("seed", range(4))
def test_bias_brute_force(seed):
    rng = np.random.default_rng(300 + seed)
    n, H, D = int(rng.integers(3, 40)), int(rng.integers(1, 5)), int(rng.integers(1, 9))
    indptr, indices, Q, K, V = _bias_graph(rng, n, int(rng.integers(1, n * n // 2 + 1)), H, D)
    bias = (rng.standard_normal((len(indices), H)) * 2).astype(np.float32)
    bias[rng.random(bias.shape) < 0.15] = -np.inf          # some pairs removed
    scale = float(np.float32(1 / math.sqrt(D)))
    got = oracle.sparse_mha(indptr, indices, Q, K, V, scale, bias=bias)["out"]
    ref = brute_force_bias(indptr, indices, n, Q, K, V, scale, bias)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_zero_bias_is_no_bias():
    rng = np.random.default_rng(310)
    indptr, indices, Q, K, V = _bias_graph(rng, 30, 300, 3, 8)
    a = oracle.sparse_mha(indptr, indices, Q, K, V, 0.35, want_probs=True)
    b = oracle.sparse_mha(indptr, indices, Q, K, V, 0.35, want_probs=True,
                          bias=np.zeros((len(indices), 3), np.float32))
    for key in ("out", "logits", "probs"):
        assert np.array_equal(a[key], b[key]), key


def test_row_constant_bias_cancels():
    # softmax is shift-invariant: a bias constant over a row's entries (per head)
    # changes the logits but not the probabilities or the output
    rng = np.random.default_rng(311)
    n, H = 30, 3
    indptr, indices, Q, K, V = _bias_graph(rng, n, 320, H, 8)
    c = rng.standard_normal((n, H)).astype(np.float32) * 3
    bias = np.repeat(c, np.diff(indptr), axis=0)
    a = oracle.sparse_mha(indptr, indices, Q, K, V, 0.35, want_probs=True)
    b = oracle.sparse_mha(indptr, indices, Q, K, V, 0.35, want_probs=True, bias=bias)
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["probs"], a["probs"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(b["logits"] - a["logits"], bias.astype(np.float64), rtol=0, atol=1e-12)


def test_minus_inf_bias_removes_entries():
    # b = -inf removes the pair: the same as deleting those CSR entries; a row
    # with every entry removed gives zeros and probabilities 0
    rng = np.random.default_rng(312)
    n, H = 25, 2
    indptr, indices, Q, K, V = _bias_graph(rng, n, 200, H, 6)
    deg = np.diff(indptr)
    keep = rng.random(len(indices)) < 0.6
    row_of = np.repeat(np.arange(n), deg)
    full_row = int(np.argmax(deg))
    keep[row_of == full_row] = False                         # one row loses every entry
    bias = np.where(keep[:, None], 0.0, -np.inf).astype(np.float32).repeat(H, axis=1)
    got = oracle.sparse_mha(indptr, indices, Q, K, V, 0.4, want_probs=True, bias=bias)
    kept_ptr = np.zeros(n + 1, np.int64)
    np.cumsum(np.bincount(row_of[keep], minlength=n), out=kept_ptr[1:])
    ref = oracle.sparse_mha(kept_ptr.astype(np.int32), indices[keep], Q, K, V, 0.4, want_probs=True)
    np.testing.assert_allclose(got["out"], ref["out"], rtol=1e-12, atol=1e-14)
    assert np.all(got["out"][full_row] == 0.0)
    assert np.all(got["probs"][~keep] == 0.0)
    np.testing.assert_allclose(got["probs"][keep], ref["probs"], rtol=1e-12, atol=1e-15)


def test_log_weight_bias_with_zero_query_is_weighted_mean():
    # q = 0: the logit is the bias alone, so b = ln w gives out = sum w v / sum w
    rng = np.random.default_rng(313)
    n, H, D = 20, 2, 4
    indptr, indices, Q, K, V = _bias_graph(rng, n, 150, H, D)
    Q[:] = 0
    w = rng.uniform(0.1, 5.0, (len(indices), H))
    got = oracle.sparse_mha(indptr, indices, Q, K, V, 0.5, bias=np.log(w).astype(np.float32))["out"]
    wf = np.exp(np.log(w).astype(np.float32).astype(np.float64))
    ref = np.zeros((n, H, D))
    for i in range(n):
        b, e = indptr[i], indptr[i + 1]
        if e > b:
            for h in range(H):
                ref[i, h] = (wf[b:e, h, None] * V[indices[b:e], h].astype(np.float64)).sum(0) / wf[b:e, h].sum()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


BIAS_MUTATIONS = {
    "bias_sign": ("if (bias) l[k] += (double)bias[(beg + k) * H + h];",
                  "if (bias) l[k] -= (double)bias[(beg + k) * H + h];"),
    "bias_transposed_index": ("if (bias) l[k] += (double)bias[(beg + k) * H + h];",
                              "if (bias) l[k] += (double)bias[(int64_t)h * nnz + beg + k];"),
    "bias_scaled_with_dot": ("if (bias) l[k] += (double)bias[(beg + k) * H + h];",
                             "if (bias) l[k] += scale * (double)bias[(beg + k) * H + h];"),
}


@pytest.mark.parametrize("name", sorted(BIAS_MUTATIONS))
def test_bias_pins_catch_planted_mistakes(name):
    text = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = BIAS_MUTATIONS[name]
    assert text.count(old) == 1, f"anchor for {name} missing"
    mutant = text.replace(old, new, 1)
    rng = np.random.default_rng(4321)
    n, H, D = 17, 3, 5
    indptr, indices, Q, K, V = _bias_graph(rng, n, 90, H, D)
    bias = (rng.standard_normal((len(indices), H)) * 3).astype(np.float32)
    ref = brute_force_bias(indptr, indices, n, Q, K, V, 0.7, bias)
    with tempfile.TemporaryDirectory() as td:
        lib = _compile_mutant(mutant, td, name)
        got = _run_mutant(lib, indptr, indices, Q, K, V, 0.7, bias)
    assert not np.allclose(got, ref, rtol=1e-9, atol=1e-12), f"pin missed mutation {name}"


# --------------------------------------------------------------------------
# weighted adjacency: logits scale * (q.k * a_e)
# --------------------------------------------------------------------------
def brute_force_weighted(indptr, indices, n, Q, K, V, scale, values):
    """Dense route: A[i, j] = stored value of the entry j -> i (no duplicate
    entries), logits scale * (q_i.k_j) * A[i, j] on stored entries, the others
    -inf, row softmax, times V; rows without entries give 0."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
    A = np.zeros((n, n))
    M = np.zeros((n, n), bool)
    dst = np.repeat(np.arange(n), np.diff(indptr))
    A[dst, indices] = np.asarray(values, dtype=np.float64)
    M[dst, indices] = True
    logits = scale * np.einsum("ihd,jhd->hij", q, k) * A[None]
    logits[:, ~M] = -np.inf
    out = np.zeros_like(q)
    has = M.any(1)
    lg = logits[:, has, :]
    w = np.exp(lg - lg.max(axis=2, keepdims=True))
    out[has] = np.einsum("hij,jhd->ihd", w / w.sum(axis=2, keepdims=True), v)
    return out


@pytest.mark.parametrize("seed", range(4))
def test_weighted_brute_force(seed):
    rng = np.random.default_rng(400 + seed)
    n, H, D = int(rng.integers(3, 40)), int(rng.integers(1, 5)), int(rng.integers(1, 9))
    indptr, indices, Q, K, V = _bias_graph(rng, n, int(rng.integers(1, n * n // 2 + 1)), H, D)
    values = rng.uniform(0.0, 1.0, len(indices)).astype(np.float32)
    values[rng.random(len(values)) < 0.1] = 0.0                # stored zeros stay in the softmax
    scale = float(np.float32(1 / math.sqrt(D)))
    got = oracle.sparse_mha(indptr, indices, Q, K, V, scale, values=values)["out"]
    ref = brute_force_weighted(indptr, indices, n, Q, K, V, scale, values)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_unit_values_are_binary_adjacency():
    rng = np.random.default_rng(410)
    indptr, indices, Q, K, V = _bias_graph(rng, 30, 300, 3, 8)
    a = oracle.sparse_mha(indptr, indices, Q, K, V, 0.35, want_probs=True)
    b = oracle.sparse_mha(indptr, indices, Q, K, V, 0.35, want_probs=True,
                          values=np.ones(len(indices), np.float32))
    for key in ("out", "logits", "probs"):
        assert np.array_equal(a[key], b[key]), key


def test_zero_values_give_neighbour_mean():
    # every stored value 0: every logit 0, uniform weights over the stored entries
    rng = np.random.default_rng(411)
    n, H, D = 25, 2, 5
    indptr, indices, Q, K, V = _bias_graph(rng, n, 200, H, D)
    got = oracle.sparse_mha(indptr, indices, Q, K, V, 0.5, values=np.zeros(len(indices), np.float32))["out"]
    ref = np.zeros((n, H, D))
    for i in range(n):
        if indptr[i + 1] > indptr[i]:
            ref[i] = V[indices[indptr[i]:indptr[i + 1]]].astype(np.float64).mean(0)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_constant_values_rescale_the_logits():
    # A = c on every stored entry: the same as the binary graph with scale * c
    rng = np.random.default_rng(412)
    indptr, indices, Q, K, V = _bias_graph(rng, 30, 280, 3, 6)
    c = np.float32(0.375)
    got = oracle.sparse_mha(indptr, indices, Q, K, V, 0.5, values=np.full(len(indices), c))["out"]
    ref = oracle.sparse_mha(indptr, indices, Q, K, V, 0.5 * float(c))["out"]
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


WEIGHT_MUTATIONS = {
    "value_of_source_node": ("if (values) dot *= (double)values[beg + k];",
                             "if (values) dot *= (double)values[indices[beg + k] % (int64_t)nnz];"),
    "value_added": ("if (values) dot *= (double)values[beg + k];",
                    "if (values) dot += (double)values[beg + k];"),
    "zero_value_removes_entry": ("if (values) dot *= (double)values[beg + k];",
                                 "if (values) dot = values[beg + k] == 0.0f ? -INFINITY : dot * (double)values[beg + k];"),
}


@pytest.mark.parametrize("name", sorted(WEIGHT_MUTATIONS))
def test_weight_pins_catch_planted_mistakes(name):
    text = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = WEIGHT_MUTATIONS[name]
    assert text.count(old) == 1, f"anchor for {name} missing"
    mutant = text.replace(old, new, 1)
    rng = np.random.default_rng(4322)
    n, H, D = 17, 3, 5
    indptr, indices, Q, K, V = _bias_graph(rng, n, 90, H, D)
    values = rng.uniform(0.0, 1.0, len(indices)).astype(np.float32)
    values[::7] = 0.0
    ref = brute_force_weighted(indptr, indices, n, Q, K, V, 0.7, values)
    with tempfile.TemporaryDirectory() as td:
        lib = _compile_mutant(mutant, td, name)
        got = _run_mutant(lib, indptr, indices, Q, K, V, 0.7, values=values)
    assert not np.allclose(got, ref, rtol=1e-9, atol=1e-12), f"pin missed mutation {name}"


# --------------------------------------------------------------------------
# backward pass: gradients of sum(out * dO)
# --------------------------------------------------------------------------
def _loss(indptr, indices, Q, K, V, G, scale):
    return float((oracle.sparse_mha(indptr, indices, Q, K, V, scale)["out"] * G.astype(np.float64)).sum())


def _fd_grads(indptr, indices, Q, K, V, G, scale):
    """Central differences of the forward oracle at every element of Q, K, V
    (the step actually taken is the difference of the two float32 values)."""
    res = {}
    for name, X in (("dQ", Q), ("dK", K), ("dV", V)):
        fd = np.zeros(X.shape)
        for idx in np.ndindex(X.shape):
            x0 = X[idx]
            xp, xm = np.float32(x0 + 1e-3), np.float32(x0 - 1e-3)
            X[idx] = xp
            lp = _loss(indptr, indices, Q, K, V, G, scale)
            X[idx] = xm
            lm = _loss(indptr, indices, Q, K, V, G, scale)
            X[idx] = x0
            fd[idx] = (lp - lm) / (float(xp) - float(xm))
        res[name] = fd
    return res


@pytest.mark.parametrize("seed", range(2))
def test_backward_matches_finite_differences(seed):
    rng = np.random.default_rng(500 + seed)
    n, H, D = 7, 2, 3
    indptr, indices, Q, K, V = _bias_graph(rng, n, 20, H, D)
    G = rng.standard_normal((n, H, D)).astype(np.float32)
    got = oracle.sparse_mha_bwd(indptr, indices, Q, K, V, G, 0.6)
    fd = _fd_grads(indptr, indices, Q, K, V, G, 0.6)
    for name in fd:
        np.testing.assert_allclose(got[name], fd[name], rtol=1e-5, atol=1e-6, err_msg=name)


def test_backward_single_neighbour_and_constant_values():
    rng = np.random.default_rng(510)
    n, H, D = 12, 2, 4
    src = rng.integers(0, n, n)
    indptr, indices = wl.csr_by_destination(src, np.arange(n), n)   # one entry per row
    Q, K, V = _rand_feats(rng, n, H, D)
    G = rng.standard_normal((n, H, D)).astype(np.float32)
    r = oracle.sparse_mha_bwd(indptr, indices, Q, K, V, G, 0.5)
    assert np.all(r["dQ"] == 0.0) and np.all(r["dK"] == 0.0)     # p = 1 whatever the logits
    ref = np.zeros((n, H, D))
    np.add.at(ref, indices, G.astype(np.float64))                  # dV_j = sum of dO_i over i <- j
    np.testing.assert_allclose(r["dV"], ref, rtol=0, atol=1e-15)
    # constant V: out does not depend on the weights, so dQ = dK = 0
    indptr, indices, Q, K, V = _bias_graph(rng, n, 60, H, D)
    V[:] = 0.75
    r = oracle.sparse_mha_bwd(indptr, indices, Q, K, V, G, 0.5)
    np.testing.assert_allclose(r["dQ"], 0.0, atol=1e-14)
    np.testing.assert_allclose(r["dK"], 0.0, atol=1e-14)


def test_backward_invariants_on_a_larger_graph():
    # exact consequences of the chain rule at sizes finite differences cannot
    # reach: for every row with entries sum_j p_ij = 1 and sum_j ds_ij = 0, so
    #   sum_j dV_j = sum over rows with entries of dO_i,
    #   sum_j dK_j = scale sum_i q_i sum_j ds_ij = 0,
    # and adding one vector c to every K row shifts each row's logits by a
    # constant (softmax unchanged: same dV) while dQ_i gains
    # scale c sum_j ds_ij = 0 (same dQ).
    rng = np.random.default_rng(530)
    n, H, D, m = 300, 3, 8, 280            # rows m..n-1 have no entries
    src = rng.integers(0, n, 4000)
    dst = rng.integers(0, m, 4000)
    indptr, indices = wl.csr_by_destination(src, dst, n)
    Q, K, V = _rand_feats(rng, n, H, D)
    # K and the shift on a 2^-10 grid, so K + c is exact in float32 and the
    # logits move by exactly scale q_i.c
    K = (np.round(np.clip(K, -4, 4) * 1024) / 1024).astype(np.float32)
    c = (rng.integers(-256, 257, (1, H, D)) / 1024).astype(np.float32)
    G = rng.standard_normal((n, H, D)).astype(np.float32)
    r = oracle.sparse_mha_bwd(indptr, indices, Q, K, V, G, 0.4)
    has = np.diff(indptr) > 0
    assert not has[m:].any() and has[:m].sum() > 250
    np.testing.assert_allclose(r["dV"].sum(axis=0), G[has].astype(np.float64).sum(axis=0), rtol=1e-12, atol=1e-11)
    assert np.all(np.abs(r["dK"].sum(axis=0)) <= 1e-12 * np.abs(r["dK"]).sum(axis=0) + 1e-13)
    r2 = oracle.sparse_mha_bwd(indptr, indices, Q, (K + c).astype(np.float32), V, G, 0.4)
    np.testing.assert_allclose(r2["dV"], r["dV"], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(r2["dQ"], r["dQ"], rtol=1e-10, atol=1e-12)


BWD_MUTATIONS = {
    "softmax_jacobian_without_mean": ("const double ds = p[k] * (dp[k] - Dlt);", "const double ds = p[k] * dp[k];"),
    "dk_to_the_row": ("double* dk = dK + j * HD + (int64_t)h * D;", "double* dk = dK + i * HD + (int64_t)h * D;"),
    "dq_without_scale": ("dq[d] += scale * ds * (double)kj[d];", "dq[d] += ds * (double)kj[d];"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTATIONS))
def test_backward_pins_catch_planted_mistakes(name):
    text = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = BWD_MUTATIONS[name]
    assert text.count(old) == 1, f"anchor for {name} missing"
    mutant = text.replace(old, new, 1)
    rng = np.random.default_rng(520)
    n, H, D = 7, 2, 3
    indptr, indices, Q, K, V = _bias_graph(rng, n, 20, H, D)
    G = rng.standard_normal((n, H, D)).astype(np.float32)
    ref = _fd_grads(indptr, indices, Q, K, V, G, 0.6)   # the independent pin
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, name + ".c")
        open(path, "w").write(mutant)
        so = os.path.join(td, name + ".so")
        subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", path, "-o", so, "-lm"], check=True)
        lib = ctypes.CDLL(so)
        i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_double
        lib.gto_sparse_mha_bwd.argtypes = [i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, dbl, vp, vp, vp]
        out = {k: np.zeros((n, H, D)) for k in ("dQ", "dK", "dV")}
        p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
        ip, ix = np.ascontiguousarray(indptr, np.int32), np.ascontiguousarray(indices, np.int32)
        assert lib.gto_sparse_mha_bwd(n, int(ip[-1]), H, D, p(ip), p(ix), p(Q), p(K), p(V), p(G), 0.6,
                                      p(out["dQ"]), p(out["dK"]), p(out["dV"])) == 0
    assert any(not np.allclose(out[k], ref[k], rtol=1e-5, atol=1e-6) for k in out), f"pin missed mutation {name}"


# --------------------------------------------------------------------------
# projections around the attention (SparseMHA's q/k/v/out_proj, TransLayer's
# proj_q/k/v/o): the linear layer, the storage rounding, the whole block
# --------------------------------------------------------------------------
def test_linear_hand_example():
    # [1 2] times W^T with W = [[3, 4], [5, 6]], plus b = [7, 8]: [18, 25]
    X = np.array([[1.0, 2.0]], np.float32)
    W = np.array([[3.0, 4.0], [5.0, 6.0]], np.float32)
    b = np.array([7.0, 8.0], np.float32)
    assert oracle.linear(X, W, b).tolist() == [[18.0, 25.0]]
    assert oracle.linear(X, W).tolist() == [[11.0, 17.0]]


@pytest.mark.parametrize("seed", [0, 1])
def test_linear_matches_library_matmul(seed):
    rng = np.random.default_rng(seed)
    M, Kin, Nout = 37, 19, 23
    X = rng.standard_normal((M, Kin)).astype(np.float32)
    W = rng.standard_normal((Nout, Kin)).astype(np.float32)
    b = rng.standard_normal(Nout).astype(np.float32)
    ref = X.astype(np.float64) @ W.astype(np.float64).T + b.astype(np.float64)
    assert np.allclose(oracle.linear(X, W, b), ref, rtol=1e-13, atol=1e-13)
    assert np.allclose(oracle.linear(X, W, b, threads=4), ref, rtol=1e-13, atol=1e-13)
    # identity weights give X back
    assert np.array_equal(oracle.linear(X, np.eye(Kin, dtype=np.float32)), X.astype(np.float64))


def _nearest_bf16(x64):
    """Nearest bf16 of the nearest float32 of x (ties to even), by comparing
    the two bf16 neighbours of the float32 value (not bit arithmetic)."""
    f = np.float32(x64)
    if not np.isfinite(f):
        return f
    bits = np.array([f], np.float32).view(np.uint32)[0]
    down = np.array([bits & np.uint32(0xFFFF0000)], np.uint32).view(np.float32)[0]
    step = np.array([(bits & np.uint32(0xFFFF0000)) + np.uint32(0x10000)], np.uint32).view(np.float32)[0]
    lo, hi = (down, step) if abs(step) >= abs(down) else (step, down)
    dl, dh = abs(float(f) - float(lo)), abs(float(hi) - float(f))
    if dl < dh:
        return lo
    if dh < dl:
        return hi
    lo_even = (np.array([lo], np.float32).view(np.uint32)[0] >> 16) % 2 == 0
    return lo if lo_even else hi


def test_round_store_matches_nearest_neighbour_search():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-6, 6, 4000),
                        [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.0, -0.0,
                         3.3895313892515355e38, 1e300, -np.inf, np.inf]])
    got = oracle.round_store(x, "bf16")
    ref = np.array([_nearest_bf16(v) for v in x], np.float32)
    assert np.array_equal(got, ref)
    # the ties: 1 + 2^-8 rounds down to 1 (even), 1 + 3 * 2^-8 up to 1 + 2^-6
    assert got[4000] == 1.0 and got[4001] == 1.0 + 2.0 ** -6
    assert np.array_equal(oracle.round_store(x, "f32"), x.astype(np.float32))
    assert np.isnan(oracle.round_store(np.array([np.nan]), "bf16")[0])


def _proj_case(rng, n, e, d_in, H, D, d_out, bias=True):
    pick = rng.choice(n * n, size=e, replace=False)
    src, dst = pick // n, pick % n
    indptr, indices = wl.csr_by_destination(src, dst, n)
    X = rng.standard_normal((n, d_in)).astype(np.float32)
    Ws = [(rng.standard_normal((H * D, d_in)) / np.sqrt(d_in)).astype(np.float32) for _ in range(3)]
    Wo = (rng.standard_normal((d_out, H * D)) / np.sqrt(H * D)).astype(np.float32)
    bs = [rng.standard_normal(H * D).astype(np.float32) * 0.1 if bias else None for _ in range(3)]
    bo = rng.standard_normal(d_out).astype(np.float32) * 0.1 if bias else None
    return src, dst, indptr, indices, X, Ws, Wo, bs, bo


def _brute_proj(src, dst, n, X, Ws, Wo, bs, bo, H, D, scale, heads_inner, store):
    """The block by dense numpy: projections by matmul, heads split by
    reshape, masked dense softmax attention, heads merged, out projection;
    intermediates stored as float32 (or bf16 by neighbour search)."""
    def st(a):
        if store == "f32":
            return a.astype(np.float32)
        return np.vectorize(_nearest_bf16, otypes=[np.float32])(a)

    X64 = X.astype(np.float64)

    def lin(W, b):
        # products summed over the inputs in index order, then the bias, so
        # that both sides hold the same double before rounding it for storage
        acc = np.zeros((X64.shape[0], W.shape[0]))
        for k in range(X64.shape[1]):
            acc += np.outer(X64[:, k], W[:, k].astype(np.float64))
        return (0.0 if b is None else b.astype(np.float64)) + acc

    qkv = []
    for W, b in zip(Ws, bs):
        y = lin(W, b)
        y = y.reshape(n, D, H).transpose(0, 2, 1) if heads_inner else y.reshape(n, H, D)
        qkv.append(st(y))
    o = st(brute_force(src, dst, n, *qkv, scale))
    of = o.transpose(0, 2, 1).reshape(n, D * H) if heads_inner else o.reshape(n, H * D)
    return of.astype(np.float64) @ Wo.astype(np.float64).T + (0.0 if bo is None else bo.astype(np.float64))


@pytest.mark.parametrize("heads_inner", [False, True])
@pytest.mark.parametrize("store", ["f32", "bf16"])
@pytest.mark.parametrize("bias", [True, False])
def test_proj_block_brute_force(heads_inner, store, bias):
    rng = np.random.default_rng(7)
    n, H, D, d_in, d_out = 19, 3, 4, 10, 6
    src, dst, indptr, indices, X, Ws, Wo, bs, bo = _proj_case(rng, n, 90, d_in, H, D, d_out, bias)
    scale = 0.625   # exact in float32 (the oracle takes the scale as a float32 value)
    got = oracle.sparse_mha_proj(indptr, indices, X, *Ws, Wo, *bs, bo, H, D, scale, heads_inner=heads_inner,
                                 store=store)
    ref = _brute_proj(src, dst, n, X, Ws, Wo, bs, bo, H, D, scale, heads_inner, store)
    # the stored intermediates are rounded alike on both sides; what is left
    # is double rounding order
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_proj_layouts_are_a_feature_permutation():
    # a heads-inner block equals the heads-major block whose q/k/v weight
    # rows and out-projection columns are permuted by f = d*H + h -> h*D + d
    rng = np.random.default_rng(8)
    n, H, D, d_in, d_out = 15, 2, 3, 5, 4
    src, dst, indptr, indices, X, Ws, Wo, bs, bo = _proj_case(rng, n, 60, d_in, H, D, d_out)
    perm = np.array([d * H + h for h in range(H) for d in range(D)])   # major position -> inner feature
    inner = oracle.sparse_mha_proj(indptr, indices, X, *Ws, Wo, *bs, bo, H, D, 0.5, heads_inner=True)
    major = oracle.sparse_mha_proj(indptr, indices, X, *[W[perm] for W in Ws], Wo[:, perm], *[b[perm] for b in bs],
                                   bo, H, D, 0.5, heads_inner=False)
    assert np.allclose(inner, major, rtol=1e-13, atol=1e-13)
    # ... and differs from the unpermuted heads-major block
    plain = oracle.sparse_mha_proj(indptr, indices, X, *Ws, Wo, *bs, bo, H, D, 0.5, heads_inner=False)
    assert not np.allclose(inner, plain, rtol=1e-6, atol=1e-6)


def test_proj_rows_subset_matches_full():
    rng = np.random.default_rng(9)
    n, H, D, d_in, d_out = 40, 2, 4, 8, 8
    src, dst, indptr, indices, X, Ws, Wo, bs, bo = _proj_case(rng, n, 300, d_in, H, D, d_out)
    full = oracle.sparse_mha_proj(indptr, indices, X, *Ws, Wo, *bs, bo, H, D, 0.375, store="bf16")
    rows = np.array([0, 3, 17, 39, 22])
    sub = oracle.sparse_mha_proj(indptr, indices, X, *Ws, Wo, *bs, bo, H, D, 0.375, store="bf16", rows=rows)
    assert np.array_equal(sub, full[rows])


LINEAR_MUTATIONS = {
    # W read as [Kin, Nout] (a transposed weight)
    "transposed_weight": ("const float* w = W + (int64_t)n * Kin;", "const float* w = W + n;"),
    "bias_dropped": ("Y[m * Nout + n] = (b ? (double)b[n] : 0.0) + acc;", "Y[m * Nout + n] = acc;"),
    "last_input_dropped": ("for (int32_t k = 0; k < Kin; ++k) acc +=", "for (int32_t k = 0; k + 1 < Kin; ++k) acc +="),
    "ties_away_from_zero": ("if (low > 0x8000u || (low == 0x8000u && lsb)) hi += 0x10000u;",
                            "if (low >= 0x8000u) hi += 0x10000u;"),
}


@pytest.mark.parametrize("name", sorted(LINEAR_MUTATIONS))
def test_proj_pins_catch_planted_mistakes(name):
    text = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = LINEAR_MUTATIONS[name]
    assert text.count(old) == 1, f"anchor for {name} missing"
    mutant = text.replace(old, new)
    rng = np.random.default_rng(11)
    M, Kin, Nout = 9, 7, 5
    X = rng.standard_normal((M, Kin)).astype(np.float32)
    W = rng.standard_normal((Nout, Kin)).astype(np.float32)
    b = rng.standard_normal(Nout).astype(np.float32)
    ties = np.array([1.0 + 2.0 ** -8, 2.0 + 2.0 ** -7, -(4.0 + 2.0 ** -6)])
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, name + ".c")
        open(path, "w").write(mutant)
        so = os.path.join(td, name + ".so")
        subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", path, "-o", so, "-lm"], check=True)
        lib = ctypes.CDLL(so)
        vp = ctypes.c_void_p
        lib.gto_linear.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, vp, vp, vp, vp]
        lib.gto_round_store.argtypes = [ctypes.c_int64, vp, ctypes.c_int32, vp]
        Y = np.zeros((M, Nout))
        lib.gto_linear(M, Kin, Nout, X.ctypes.data_as(vp), W.ctypes.data_as(vp), b.ctypes.data_as(vp),
                       Y.ctypes.data_as(vp))
        r = np.zeros(3, np.float32)
        lib.gto_round_store(3, ties.ctypes.data_as(vp), 1, r.ctypes.data_as(vp))
    ok_linear = np.allclose(Y, X.astype(np.float64) @ W.astype(np.float64).T + b, rtol=1e-12, atol=1e-12)
    ok_round = np.array_equal(r, np.array([_nearest_bf16(v) for v in ties], np.float32))
    assert not (ok_linear and ok_round), f"pin missed mutation {name}"
