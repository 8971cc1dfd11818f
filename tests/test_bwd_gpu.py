"""Backward pass (gtattn_bwd): the gradients of sum(out * dO) with respect to
Q, K, V from the CUDA path against the fp64 oracle backward (itself pinned
by finite differences of the forward oracle) on the same inputs.

Tolerance (the pages state none for gradients), per element and aware of
the sums' conditioning: |g - o| <= 3e-5 * cond + 1e-7, where cond is the
sum of the magnitudes the element is made of, with each term's own error
source included.  Per entry e = (i <- j) and head: p the probability,
dp = dO_i . v_j, Dlt_i = dO_i . O_i, ds = p (dp - Dlt); the dot products
carry errors relative to A = sum_d |dO_i||v_j|, B = sum_d |dO_i||O_i| and
C = scale sum_d |q_i||k_j| (C also bounds the log-domain error of p), so
ds is known to T = p (A + B + |dp - Dlt| C), and
  cond dQ_i = scale sum_e (T + |ds|) |k_j|,   cond dK_j = scale sum_e (T + |ds|) |q_i|,
  cond dV_j = sum_e p (1 + C) |dO_i|.
3e-5 is about 500 fp32 unit roundoffs: sums of up to ~10^5 terms in fp32
(random-walk growth sqrt(n) 2^-24) with the products' own rounding."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import to_device

torch = pytest.importorskip("torch")
gt = pytest.importorskip("graph_transformer_sparse_gb300")

pytestmark = pytest.mark.gpu

GRAD_RTOL = 3e-5


def _segment_add(out, keys, vals):
    """out[k] += sum of vals over the entries with key k (keys sorted)."""
    if len(keys) == 0:
        return
    starts = np.flatnonzero(np.r_[True, keys[1:] != keys[:-1]])
    out[keys[starts]] += np.add.reduceat(vals, starts, axis=0)


def _bwd_cond(indptr, indices, Q, K, V, dO, scale, chunk=20_000):
    """Condition sums (see the module docstring) of dQ, dK, dV, float64
    [N, H, D]; entries processed in chunks to bound memory."""
    fw = oracle.sparse_mha(indptr, indices, Q, K, V, scale, want_probs=True, threads=8)
    P, O = fw["probs"], fw["out"]
    N, H, D = Q.shape
    nnz = len(indices)
    row = np.repeat(np.arange(N), np.diff(indptr))
    Q64, K64, V64, G64 = (np.asarray(x, np.float64) for x in (Q, K, V, dO))
    Dlt = np.einsum("nhd,nhd->nh", G64, O)
    B = np.einsum("nhd,nhd->nh", np.abs(G64), np.abs(O))
    # per entry and head: the weights of |k_j| (dQ), |q_i| (dK) and |dO_i| (dV)
    wq = np.zeros((nnz, H))
    wv = np.zeros((nnz, H))
    for a in range(0, nnz, chunk):
        i, j = row[a:a + chunk], indices[a:a + chunk]
        p = P[a:a + chunk]
        dp = np.einsum("ehd,ehd->eh", G64[i], V64[j])
        A = np.einsum("ehd,ehd->eh", np.abs(G64[i]), np.abs(V64[j]))
        C = scale * np.einsum("ehd,ehd->eh", np.abs(Q64[i]), np.abs(K64[j]))
        ds = p * (dp - Dlt[i])
        T = p * (A + B[i] + np.abs(dp - Dlt[i]) * C)
        wq[a:a + chunk] = scale * (T + np.abs(ds))
        wv[a:a + chunk] = p * (1 + C)
    cq, ck, cv = (np.zeros((N, H, D)) for _ in range(3))
    for a in range(0, nnz, chunk):   # by destination row (entries are in row order)
        i, j = row[a:a + chunk], indices[a:a + chunk]
        _segment_add(cq, i, wq[a:a + chunk, :, None] * np.abs(K64[j]))
    order = np.argsort(indices, kind="stable")   # by source
    for a in range(0, nnz, chunk):
        e = order[a:a + chunk]
        i, j = row[e], indices[e]
        _segment_add(ck, j, wq[e, :, None] * np.abs(Q64[i]))
        _segment_add(cv, j, wv[e, :, None] * np.abs(G64[i]))
    return {"dQ": cq, "dK": ck, "dV": cv}


def _grad_close(got, ref, cond, what):
    bound = GRAD_RTOL * cond + 1e-7
    err = np.abs(got - ref)
    bad = err > bound
    k = np.argmax(err - bound)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside; worst got {got.flat[k]!r} "
                           f"ref {ref.flat[k]!r} cond {cond.flat[k]!r}")


def _dO(w, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((w.N, w.H, w.D)).astype(np.float32)
    if w.dtype == "bf16":
        vals, bits = wl.bf16_round(g)
        return vals, torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    return g, torch.from_numpy(g).cuda()


def _bwd(w, d, dO_t):
    grads = {k: torch.full((w.N, w.H, w.D), float("nan"), device="cuda") for k in ("dQ", "dK", "dV")}
    dt = gt.GTATTN_F32 if w.dtype == "f32" else gt.GTATTN_BF16
    gt.gtattn_bwd(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], dO_t, grads["dQ"], grads["dK"], grads["dV"],
                  w.N, w.nnz, w.H, w.D, w.scale, dt)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy().astype(np.float64) for k, v in grads.items()}


@pytest.mark.parametrize("name", ["tiny_random", "molecules", "erdos_renyi", "rmat", "dense_blocks"])
def test_backward_matches_oracle(name):
    w = wl.small_workload(name)
    g, g_t = _dO(w, seed=sum(map(ord, name)))
    ref = oracle.sparse_mha_bwd(w.indptr, w.indices, w.Q, w.K, w.V, g, w.scale)
    cond = _bwd_cond(w.indptr, w.indices, w.Q, w.K, w.V, g, w.scale)
    got = _bwd(w, to_device(w), g_t)
    for k in ("dQ", "dK", "dV"):
        _grad_close(got[k], ref[k], cond[k], f"{name} {k}")
    # rows without entries have no query gradient
    empty = np.diff(w.indptr) == 0
    assert np.all(got["dQ"][empty] == 0.0)


def test_backward_single_neighbour_rows():
    # p = 1 exactly: no query or key gradient, dV_j the sum of dO_i over i <- j
    rng = np.random.default_rng(3)
    n, H, D = 500, 4, 32
    src = rng.integers(0, n, n)
    indptr, indices = wl.csr_by_destination(src, np.arange(n), n)
    Q, K, V = (rng.standard_normal((n, H, D)).astype(np.float32) for _ in range(3))
    w = wl.Workload("single", n, H, D, "f32", indptr.astype(np.int32), indices.astype(np.int32), Q, K, V, 0.2)
    g, g_t = _dO(w, 4)
    got = _bwd(w, to_device(w), g_t)
    assert np.all(got["dQ"] == 0.0) and np.all(got["dK"] == 0.0)
    ref = np.zeros((n, H, D))
    np.add.at(ref, indices, g.astype(np.float64))
    cond = np.zeros((n, H, D))
    np.add.at(cond, indices, np.abs(g.astype(np.float64)))
    _grad_close(got["dV"], ref, cond, "single-neighbour dV")


def _hub_graph(n, seed):
    # random entries, one destination fed by n/2 sources (a split row), one
    # source feeding n/2 destinations (a split source), nodes past 0.95 n
    # without entries either way
    rng = np.random.default_rng(seed)
    m = int(0.95 * n)
    src = np.concatenate([rng.integers(0, m, 6 * n), rng.integers(0, m, n // 2), np.full(n // 2, 1)])
    dst = np.concatenate([rng.integers(0, m, 6 * n), np.zeros(n // 2, np.int64), rng.integers(0, m, n // 2)])
    key = np.unique(dst * n + src)
    return wl.csr_by_destination(key % n, key // n, n)


@pytest.mark.parametrize("H,D,dtype", [(8, 32, "f32"), (2, 128, "bf16"), (16, 64, "bf16"), (4, 256, "f32"),
                                       (4, 32, "bf16"), (8, 64, "f32")])
def test_backward_shapes_with_hubs(H, D, dtype):
    # every lane width of the two passes (4, 8, 16, 32 features per lane),
    # split rows and split sources, rows and sources without entries
    n = 3000
    indptr, indices = _hub_graph(n, H * D)
    rng = np.random.default_rng(D)
    feats = {k: rng.standard_normal((n, H, D)).astype(np.float32) for k in ("Q", "K", "V")}
    bits = {}
    if dtype == "bf16":
        for k in feats:
            feats[k], bits[k] = wl.bf16_round(feats[k])
    w = wl.Workload("hubs", n, H, D, dtype, indptr.astype(np.int32), indices.astype(np.int32), feats["Q"],
                    feats["K"], feats["V"], float(np.float32(1.0 / np.sqrt(D))), bits)
    g, g_t = _dO(w, 7)
    ref = oracle.sparse_mha_bwd(w.indptr, w.indices, w.Q, w.K, w.V, g, w.scale)
    cond = _bwd_cond(w.indptr, w.indices, w.Q, w.K, w.V, g, w.scale)
    got = _bwd(w, to_device(w), g_t)
    for k in ("dQ", "dK", "dV"):
        _grad_close(got[k], ref[k], cond[k], f"H={H} D={D} {dtype} {k}")
    no_in = np.bincount(w.indices, minlength=n) == 0
    assert np.all(got["dK"][no_in] == 0.0) and np.all(got["dV"][no_in] == 0.0)
    assert np.all(got["dQ"][np.diff(w.indptr) == 0] == 0.0)


def test_backward_no_entries():
    n, H, D = 100, 4, 32
    rng = np.random.default_rng(5)
    Q, K, V = (rng.standard_normal((n, H, D)).astype(np.float32) for _ in range(3))
    w = wl.Workload("empty", n, H, D, "f32", np.zeros(n + 1, np.int32), np.zeros(0, np.int32), Q, K, V, 0.2)
    g, g_t = _dO(w, 6)
    got = _bwd(w, to_device(w), g_t)
    for k in ("dQ", "dK", "dV"):
        assert np.all(got[k] == 0.0), k


def test_backward_argument_errors():
    w = wl.make_workload("tiny_random")
    d = to_device(w)
    z = torch.zeros((w.N, 200, 1), device="cuda")
    with pytest.raises(gt.GtattnError) as e:   # more heads than the backward supports
        gt.gtattn_bwd(d["indptr"], d["indices"], z, z, z, z, z, z, z, w.N, w.nnz, 200, 1, 1.0, gt.GTATTN_F32)
    assert e.value.status == gt.GTATTN_ERR_INVALID_ARG


def _sampled_sources(w, n_random=200, n_top=8, seed=1):
    rng = np.random.default_rng(seed)
    cdeg = np.bincount(w.indices, minlength=w.N)
    top = np.argsort(cdeg)[-n_top:]
    rnd = rng.choice(w.N, size=min(n_random, w.N), replace=False)
    return np.unique(np.concatenate([top, rnd]))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["erdos_renyi", "rmat"])
def test_backward_full_size_sampled(name):
    # Full-size workload on the GPU; the oracle on the subgraph of every
    # destination row that a sampled output depends on: dQ_i needs row i's
    # entries, dK_j and dV_j every row holding source j (each with all its
    # entries, for that row's softmax), so on that subgraph the sampled
    # outputs are exact.
    w = wl.make_workload(name)
    deg = np.diff(w.indptr)
    q_rows = np.unique(np.concatenate([np.argsort(deg)[-16:], np.flatnonzero(deg == 1)[:32],
                                       np.random.default_rng(2).choice(w.N, 300, replace=False)]))
    srcs = _sampled_sources(w)
    row_of = np.repeat(np.arange(w.N), deg)
    keep = np.zeros(w.N, bool)
    keep[q_rows] = True
    keep[row_of[np.isin(w.indices, srcs)]] = True
    sub_deg = np.where(keep, deg, 0)
    sub_ptr = np.zeros(w.N + 1, np.int64)
    np.cumsum(sub_deg, out=sub_ptr[1:])
    sub_idx = w.indices[np.repeat(keep, deg)]
    g, g_t = _dO(w, seed=11)
    ref = oracle.sparse_mha_bwd(sub_ptr.astype(np.int32), sub_idx, w.Q, w.K, w.V, g, w.scale)
    cond = _bwd_cond(sub_ptr.astype(np.int32), sub_idx, w.Q, w.K, w.V, g, w.scale)
    got = _bwd(w, to_device(w), g_t)
    _grad_close(got["dQ"][q_rows], ref["dQ"][q_rows], cond["dQ"][q_rows], f"{name} dQ (sampled rows)")
    for k in ("dK", "dV"):
        _grad_close(got[k][srcs], ref[k][srcs], cond[k][srcs], f"{name} {k} (sampled sources)")
    for k in ("dQ", "dK", "dV"):
        assert np.isfinite(got[k]).all(), k


def _bwd_plan(w, d, dO_t, plan, O=None, stats=None):
    grads = {k: torch.full((w.N, w.H, w.D), float("nan"), device="cuda") for k in ("dQ", "dK", "dV")}
    dt = gt.GTATTN_F32 if w.dtype == "f32" else gt.GTATTN_BF16
    gt.gtattn_bwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], dO_t, grads["dQ"], grads["dK"],
                       grads["dV"], w.H, w.D, w.scale, dt, O=O, stats=stats)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy().astype(np.float64) for k, v in grads.items()}


@pytest.mark.parametrize("name", ["rmat", "erdos_renyi", "tiny_random"])
def test_backward_is_deterministic_and_the_plan_agrees(name):
    # two calls give the same bits; the planned backward (its first call
    # builds the source-major pattern, the second reuses it) gives the same
    # bits as the plan-less one; and the result matches the oracle
    w = wl.small_workload(name)
    g, g_t = _dO(w, 13)
    d = to_device(w)
    a = _bwd(w, d, g_t)
    b = _bwd(w, d, g_t)
    plan = gt.Plan(d["indptr"], d["indices"])
    c1 = _bwd_plan(w, d, g_t, plan)
    c2 = _bwd_plan(w, d, g_t, plan)
    plan.close()
    for k in ("dQ", "dK", "dV"):
        assert np.array_equal(a[k], b[k]), f"{name} {k}: two calls differ"
        assert np.array_equal(a[k], c1[k]) and np.array_equal(a[k], c2[k]), f"{name} {k}: plan differs"
    ref = oracle.sparse_mha_bwd(w.indptr, w.indices, w.Q, w.K, w.V, g, w.scale)
    cond = _bwd_cond(w.indptr, w.indices, w.Q, w.K, w.V, g, w.scale)
    for k in ("dQ", "dK", "dV"):
        _grad_close(a[k], ref[k], cond[k], f"{name} {k}")


def test_backward_deterministic_with_hubs_and_long_segments():
    # a source feeding 5000 destinations (its segment sorted through the
    # merge passes of the segment sort) and a destination fed by 5000
    # sources: split rows and sources summed in chunk order
    n = 12000
    rng = np.random.default_rng(17)
    src = np.concatenate([rng.integers(0, n, 4 * n), np.full(5000, 7), rng.integers(0, n, 5000)])
    dst = np.concatenate([rng.integers(0, n, 4 * n), rng.integers(0, n, 5000), np.full(5000, 11)])
    key = np.unique(dst * n + src)
    indptr, indices = wl.csr_by_destination(key % n, key // n, n)
    H, D = 4, 32
    Q, K, V = (rng.standard_normal((n, H, D)).astype(np.float32) for _ in range(3))
    w = wl.Workload("hubs", n, H, D, "f32", indptr.astype(np.int32), indices.astype(np.int32), Q, K, V, 0.17)
    g, g_t = _dO(w, 19)
    d = to_device(w)
    runs = [_bwd(w, d, g_t) for _ in range(3)]
    for k in ("dQ", "dK", "dV"):
        assert all(np.array_equal(runs[0][k], r[k]) for r in runs[1:]), k
    ref = oracle.sparse_mha_bwd(w.indptr, w.indices, w.Q, w.K, w.V, g, w.scale)
    cond = _bwd_cond(w.indptr, w.indices, w.Q, w.K, w.V, g, w.scale)
    for k in ("dQ", "dK", "dV"):
        _grad_close(runs[0][k], ref[k], cond[k], f"hubs {k}")


def test_backward_plan_with_dense_blocks():
    # a plan that found complete blocks lists their rows in its dense
    # segment; the backward walks those rows too
    w = wl.small_workload("dense_blocks")
    g, g_t = _dO(w, 23)
    d = to_device(w)
    plan = gt.Plan(d["indptr"], d["indices"], detect_dense=True)
    assert plan.info()["n_dense_blocks"] > 0
    got = _bwd_plan(w, d, g_t, plan)
    plan.close()
    ref = oracle.sparse_mha_bwd(w.indptr, w.indices, w.Q, w.K, w.V, g, w.scale)
    cond = _bwd_cond(w.indptr, w.indices, w.Q, w.K, w.V, g, w.scale)
    for k in ("dQ", "dK", "dV"):
        _grad_close(got[k], ref[k], cond[k], f"dense blocks {k}")


def _row_log2sumexp(indptr, logits):
    # natural log-sum-exp of each row's logits over ln 2; -inf for empty rows
    N, H = len(indptr) - 1, logits.shape[1]
    deg = np.diff(indptr)
    out = np.full((N, H), -np.inf)
    rows = np.flatnonzero(deg > 0)
    if len(rows):
        starts = indptr[:-1][rows]
        m = np.maximum.reduceat(logits, starts, axis=0)
        row_of = np.repeat(np.arange(len(rows)), deg[rows])
        ssum = np.add.reduceat(np.exp(logits - m[row_of]), starts, axis=0)
        out[rows] = (m + np.log(ssum)) / np.log(2.0)
    return out


@pytest.mark.parametrize("name", ["rmat", "erdos_renyi", "tiny_random", "dense_blocks"])
def test_backward_reuses_the_saved_forward(name):
    # the forward with row statistics: its output equals the plain planned
    # forward's (fp32 output), its statistics the rows' log2-sum-exp from the
    # oracle's logits; the backward given both skips the recompute and gives
    # the same bits as the backward without them
    w = wl.small_workload(name)
    g, g_t = _dO(w, 29)
    d = to_device(w)
    plan = gt.Plan(d["indptr"], d["indices"], detect_dense=True)
    if name == "dense_blocks":
        assert plan.info()["n_dense_blocks"] > 0
    dt = gt.GTATTN_F32 if w.dtype == "f32" else gt.GTATTN_BF16_OUT_F32
    O = torch.full((w.N, w.H, w.D), float("nan"), device="cuda")
    stats = torch.full((w.N, w.H), float("nan"), device="cuda")
    gt.gtattn_fwd_plan_stats(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], O, stats, w.H, w.D,
                             w.scale, dt)
    plain = torch.full_like(O, float("nan"))
    gt.gtattn_fwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], plain, w.H, w.D, w.scale, dt)
    recomputed = _bwd_plan(w, d, g_t, plan)
    reused = _bwd_plan(w, d, g_t, plan, O=O, stats=stats)
    with pytest.raises(gt.GtattnError):   # one without the other
        _bwd_plan(w, d, g_t, plan, O=O)
    plan.close()
    for k in ("dQ", "dK", "dV"):
        assert np.array_equal(recomputed[k], reused[k]), f"{name} {k}: saved forward changes the bits"
    ref = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, want_probs=True)
    O_h = O.cpu().numpy().astype(np.float64)
    if name != "dense_blocks":   # (there the plain forward takes the dense kernel)
        assert np.array_equal(O_h, plain.cpu().numpy().astype(np.float64))
    assert np.allclose(O_h, ref["out"], rtol=1e-4, atol=1e-5)
    want = _row_log2sumexp(w.indptr, ref["logits"])
    got = stats.cpu().numpy().astype(np.float64)
    empty = np.isinf(want)
    assert (got[empty] == -np.inf).all()
    err = np.abs(got[~empty] - want[~empty])
    assert (err <= 1e-5 * (1 + np.abs(want[~empty]))).all(), float(err.max())
