"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Reduced-size versions of the five workloads run through every path (plan-less
fused, planned fused, every row split into chunks, the generic kernel, the
unfused SDDMM/softmax/SpMM trio) and are compared element by element; the
full-size workloads are compared on sampled rows (hub rows included).
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import (PROB_TOL, TOL, assert_close, oracle_rows, out_to_numpy, sample_rows,
                         to_device)

torch = pytest.importorskip("torch")
gt = pytest.importorskip("graph_transformer_sparse_gb300")

pytestmark = pytest.mark.gpu

NAMES = ["tiny_random", "molecules", "erdos_renyi", "rmat", "dense_blocks"]
_small_cache = {}


def small(name):
    if name not in _small_cache:
        _small_cache[name] = wl.small_workload(name)
    return _small_cache[name]


def _dt(d):
    return gt._dtype_code(d["Q"], d["out"])


def check_out(w, got, ref, what="out", out32=False):
    """bf16 workloads: the fp32-output variant meets the stated tolerance
    (rel 2e-3 / abs 1e-5); the bf16 output may in addition be off by its own
    rounding (half a bf16 ulp)."""
    assert_close(got, ref, w.dtype, what, rounded_bf16=(w.dtype == "bf16" and not out32))


def run(w, d, path, **plan_kw):
    """Run one path; returns (out as float64 numpy, logits, probs)."""
    H, D = w.H, w.D
    d["out"].fill_(float("nan"))
    logits = probs = None
    if path == "fwd":
        gt.gtattn_fwd(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz, H, D,
                      w.scale, _dt(d))
    elif path == "plan":
        plan = gt.Plan(d["indptr"], d["indices"], **plan_kw)
        gt.gtattn_fwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], H, D,
                           w.scale, _dt(d))
        torch.cuda.synchronize()
        plan.close()
    elif path == "probs":
        logits = torch.full((w.nnz, H), float("nan"), device="cuda")
        probs = torch.full((w.nnz, H), float("nan"), device="cuda")
        gt.gtattn_fwd_probs(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], logits, probs,
                            w.N, w.nnz, H, D, w.scale, _dt(d))
    else:
        raise ValueError(path)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy() if logits is not None else None
    pr = probs.cpu().numpy() if probs is not None else None
    return out_to_numpy(d["out"]), lg, pr


PATHS = [
    ("fwd", {}),
    ("plan", {}),
    ("plan", dict(long_row_min=-1, chunk_edges=3)),          # every non-empty row split into chunks
    ("plan", dict(long_row_min=8, chunk_edges=5)),           # mixed: short rows whole, others split
    ("plan", dict(kernel=gt.GTATTN_KERNEL_GENERIC)),         # generic row kernel
    ("plan", dict(kernel=gt.GTATTN_KERNEL_GENERIC, long_row_min=4, chunk_edges=3)),
    ("plan", dict(detect_dense=True)),
    ("probs", {}),
]


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("path,kw", PATHS, ids=lambda x: str(x) if not isinstance(x, dict) else
                         ",".join(f"{k}={v}" for k, v in x.items()) or "default")
def test_small_workloads_all_paths(name, path, kw):
    w = small(name)
    ref = oracle_rows(w, want_probs=(path == "probs"))
    if w.dtype == "bf16":
        got32, _, _ = run(w, to_device(w, out32=True), path, **kw)
        check_out(w, got32, ref["out"], "out (fp32 output)", out32=True)
    d = to_device(w)
    got, lg, pr = run(w, d, path, **kw)
    check_out(w, got, ref["out"])
    if path == "probs":
        assert_close(pr, ref["probs"], w.dtype, "probs", PROB_TOL)
        # logits: condition-aware bound 1e-5 * scale * sum|q k| + 1e-6
        dst = np.repeat(np.arange(w.N), np.diff(w.indptr))
        cond = w.scale * np.einsum("ehd,ehd->eh", np.abs(w.Q[dst].astype(np.float64)),
                                   np.abs(w.K[w.indices].astype(np.float64)))
        err = np.abs(lg - ref["logits"])
        assert np.all(err <= 1e-5 * cond + 1e-6), float((err - 1e-5 * cond).max())


def test_probs_split_row_boundaries():
    # degrees on both sides of the default 1024-entry split threshold and of
    # chunk boundaries (the unfused softmax merges chunk statistics per split
    # row)
    rng = np.random.default_rng(21)
    degs = [0, 1, 2, 255, 256, 257, 1023, 1024, 1025, 2048, 2049, 3000, 3]
    n = 2400
    indptr = np.zeros(n + 1, np.int64)
    deg = np.zeros(n, np.int64)
    deg[: len(degs)] = degs
    deg[len(degs):] = rng.integers(0, 6, n - len(degs))
    np.cumsum(deg, out=indptr[1:])
    indices = rng.integers(0, n, int(indptr[-1])).astype(np.int32)
    Q, K, V = (rng.standard_normal((n, 4, 16)) for _ in range(3))
    Q *= 2.0   # sharper distributions: chunk maxima differ
    w = _mk(indptr, indices, Q, K, V, "f32")
    ref = oracle_rows(w, want_probs=True)
    got, _, pr = run(w, to_device(w), "probs")
    check_out(w, got, ref["out"])
    assert_close(pr, ref["probs"], w.dtype, "probs", PROB_TOL)
    # each stored row's probabilities sum to 1 per head
    for i in range(len(degs)):
        if degs[i]:
            s = pr[indptr[i]:indptr[i + 1]].astype(np.float64).sum(axis=0)
            assert np.allclose(s, 1.0, atol=1e-5), (i, s)


@pytest.mark.parametrize("name", ["tiny_random", "molecules"])
def test_full_small_configs_exact_oracle(name):
    # these two are small enough for the oracle at full size
    w = wl.make_workload(name)
    d = to_device(w)
    ref = oracle_rows(w)
    for path in ("fwd", "plan"):
        got, _, _ = run(w, d, path)
        check_out(w, got, ref["out"])


@pytest.mark.slow
@pytest.mark.parametrize("name", ["erdos_renyi", "rmat", "dense_blocks"])
def test_full_size_sampled_rows(name):
    w = wl.make_workload(name)
    rows = sample_rows(w)
    ref = oracle_rows(w, rows=rows)["out"]
    for out32 in (True, False):
        d = to_device(w, out32=out32)
        for path, kw in (("fwd", {}), ("plan", dict(detect_dense=True))):
            got, _, _ = run(w, d, path, **kw)
            check_out(w, got[rows], ref, f"{name}/{path}/out32={out32}", out32=out32)
        del d
    # every output is finite and every row was written
    assert np.isfinite(got).all()


# ---------------------------------------------------------------------------
# closed forms and edge cases on the GPU
# ---------------------------------------------------------------------------
def _mk(indptr, indices, Q, K, V, dtype="f32"):
    n, H, D = Q.shape
    w = wl.Workload("case", n, H, D, "f32", np.asarray(indptr, np.int32), np.asarray(indices, np.int32),
                    Q.astype(np.float32), K.astype(np.float32), V.astype(np.float32),
                    float(np.float32(1 / np.sqrt(D))))
    if dtype == "bf16":
        w.dtype = "bf16"
        for name in ("Q", "K", "V"):
            vals, bits = wl.bf16_round(getattr(w, name))
            setattr(w, name, vals)
            w.bits[name] = bits
    return w


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("path", ["fwd", "probs"])
def test_single_neighbour_is_exact(dtype, path):
    rng = np.random.default_rng(1)
    n, H, D = 300, 8, 64
    Q, K, V = (rng.standard_normal((n, H, D)) * 4 for _ in range(3))
    src = rng.integers(0, n, n)
    ip, ix = wl.csr_by_destination(src, np.arange(n), n)
    w = _mk(ip, ix, Q, K, V, dtype)
    got, _, _ = run(w, to_device(w), path)
    assert np.array_equal(got, w.V[src].astype(np.float64))


def test_empty_graph_and_empty_rows():
    rng = np.random.default_rng(2)
    n, H, D = 50, 4, 32
    Q, K, V = (rng.standard_normal((n, H, D)) for _ in range(3))
    w = _mk(np.zeros(n + 1), np.zeros(0), Q, K, V)
    for path in ("fwd", "plan", "probs"):
        got, _, _ = run(w, to_device(w), path)
        assert np.all(got == 0.0)
    # N == 0 is a no-op
    z = torch.zeros(0, 4, 32, device="cuda")
    gt.gtattn_fwd(torch.zeros(1, dtype=torch.int32, device="cuda"), None, z, z, z, z, 0, 0, 4, 32, 1.0,
                  gt.GTATTN_F32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zero_query_gives_neighbour_mean(dtype):
    w = wl.small_workload("erdos_renyi") if dtype == "bf16" else wl.make_workload("tiny_random")
    Q0 = np.zeros_like(w.Q)
    w2 = _mk(w.indptr, w.indices, Q0, w.K, w.V, dtype)
    got, _, _ = run(w2, to_device(w2, out32=True), "fwd")
    ref = np.zeros_like(got)
    for i in range(w2.N):
        nb = w2.indices[w2.indptr[i]:w2.indptr[i + 1]]
        if len(nb):
            ref[i] = w2.V[nb].astype(np.float64).mean(axis=0)
    assert_close(got, ref, dtype)


@pytest.mark.parametrize("H,D,dtype", [(3, 5, "f32"), (1, 1, "f32"), (16, 64, "bf16"), (8, 128, "bf16"),
                                        (2, 512, "f32"), (1, 1024, "bf16"), (4, 16, "f32"), (32, 32, "bf16"),
                                        (7, 12, "bf16")])
def test_shapes(H, D, dtype):
    rng = np.random.default_rng(H * 1000 + D)
    n = 700
    ip, ix = wl.random_csr(rng, n, 9000, self_loops=True, degree_skew=1.1)
    Q, K, V = (rng.standard_normal((n, H, D)) for _ in range(3))
    w = _mk(ip, ix, Q, K, V, dtype)
    ref = oracle_rows(w)["out"]
    d = to_device(w)
    for path, kw in (("fwd", {}), ("plan", dict(long_row_min=40, chunk_edges=17)), ("probs", {})):
        got, _, _ = run(w, d, path, **kw)
        check_out(w, got, ref, f"H={H} D={D} {path}")


def test_duplicate_entries_weigh_twice():
    rng = np.random.default_rng(4)
    n, H, D = 40, 2, 16
    src = rng.integers(0, n, 400)
    dst = rng.integers(0, n, 400)
    ip, ix = wl.csr_by_destination(src, dst, n)
    Q, K, V = (rng.standard_normal((n, H, D)) for _ in range(3))
    w = _mk(ip, ix, Q, K, V)
    ref = oracle_rows(w)["out"]
    for path in ("fwd", "probs"):
        got, _, _ = run(w, to_device(w), path)
        assert_close(got, ref, "f32")


def test_misaligned_features_take_the_generic_kernel():
    w = wl.make_workload("tiny_random")
    d = to_device(w)
    HD = w.H * w.D
    # views offset by one element: 4-byte aligned, not 16-byte aligned
    buf = {k: torch.empty(w.N * HD + 1, device="cuda") for k in ("Q", "K", "V", "out")}
    views = {}
    for k in ("Q", "K", "V"):
        buf[k][1:].copy_(d[k].reshape(-1))
        views[k] = buf[k][1:].view(w.N, w.H, w.D)
    views["out"] = buf["out"][1:].view(w.N, w.H, w.D)
    gt.gtattn_fwd(d["indptr"], d["indices"], views["Q"], views["K"], views["V"], views["out"], w.N, w.nnz,
                  w.H, w.D, w.scale, gt.GTATTN_F32)
    torch.cuda.synchronize()
    assert_close(views["out"].cpu().numpy(), oracle_rows(w)["out"], "f32")


def test_guard_bands_untouched():
    w = small("rmat")
    d = to_device(w)
    HD = w.H * w.D
    pad = 4096
    big = torch.full((w.N * HD + 2 * pad,), 12345, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    out = big[pad:pad + w.N * HD].view(w.N, w.H, w.D)
    for long_min in (0, -1):
        plan = gt.Plan(d["indptr"], d["indices"], long_row_min=long_min, chunk_edges=7)
        gt.gtattn_fwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], out, w.H, w.D, w.scale,
                           gt.GTATTN_BF16)
        torch.cuda.synchronize()
        plan.close()
    raw = big.view(torch.int16)
    assert torch.all(raw[:pad] == 12345) and torch.all(raw[-pad:] == 12345)


def test_deterministic():
    w = small("rmat")
    d = to_device(w)
    a, _, _ = run(w, d, "fwd")
    b, _, _ = run(w, d, "fwd")
    assert np.array_equal(a, b)


def test_fused_equals_unfused():
    # both in fp32 output: the fused online softmax and the three-stage path
    # agree to the stated tolerance
    w = small("erdos_renyi")
    d = to_device(w, out32=True)
    a, _, _ = run(w, d, "fwd")
    b, _, _ = run(w, d, "probs")
    assert_close(a, b, "bf16", "fused vs unfused")


# ---------------------------------------------------------------------------
# plan, CSR helpers
# ---------------------------------------------------------------------------
def test_plan_bins_match_degree_histogram():
    w = wl.make_workload("rmat", scale=14, draws=1 << 18)
    d = to_device(w)
    plan = gt.Plan(d["indptr"], d["indices"], long_row_min=100, chunk_edges=64)
    info = plan.info()
    plan.close()
    deg = np.diff(w.indptr)
    long = deg > 100
    assert info["n_long_rows"] == int(long.sum())
    assert info["n_chunks"] == int(((deg[long] + 63) // 64).sum())
    assert info["max_degree"] == int(deg.max())
    assert info["n_empty_rows"] == int((deg == 0).sum())
    hist = np.bincount(np.minimum(deg[~long], 33), minlength=34)
    assert info["bucket_rows"][:33] == hist[:33].tolist()
    assert sum(info["bucket_rows"]) == int((~long).sum())


def test_dense_blocks_detected():
    w = small("dense_blocks")
    d = to_device(w)
    plan = gt.Plan(d["indptr"], d["indices"], detect_dense=True)
    info = plan.info()
    plan.close()
    assert info["n_dense_blocks"] == 3 and info["n_dense_rows"] == w.N


def test_coo_to_csr_matches_host():
    rng = np.random.default_rng(8)
    for n, e in ((1, 0), (100, 5000), (3000, 200_000)):
        src = rng.integers(0, n, e).astype(np.int32)
        dst = (rng.zipf(1.5, e) % n).astype(np.int32)
        ip_ref, ix_ref = wl.csr_by_destination(src, dst, n)
        ip = torch.empty(n + 1, dtype=torch.int32, device="cuda")
        ix = torch.empty(max(e, 1), dtype=torch.int32, device="cuda")
        gt.gtattn_coo_to_csr(torch.from_numpy(src).cuda() if e else None,
                             torch.from_numpy(dst).cuda() if e else None, e, n, ip, ix)
        torch.cuda.synchronize()
        assert np.array_equal(ip.cpu().numpy(), ip_ref)
        assert np.array_equal(ix.cpu().numpy()[:e], ix_ref)


def test_csr_validate():
    w = wl.make_workload("tiny_random")
    d = to_device(w)
    assert gt.gtattn_csr_validate(d["indptr"], d["indices"], w.N, w.nnz)
    bad = d["indices"].clone()
    bad[5] = w.N
    assert not gt.gtattn_csr_validate(d["indptr"], bad, w.N, w.nnz)
    badp = d["indptr"].clone()
    badp[3] = badp[4] + 1
    assert not gt.gtattn_csr_validate(badp, d["indices"], w.N, w.nnz)
    assert not gt.gtattn_csr_validate(d["indptr"], d["indices"], w.N, w.nnz - 1)


def test_bad_arguments_raise():
    w = wl.make_workload("tiny_random")
    d = to_device(w)
    with pytest.raises(gt.GtattnError) as e:
        gt.gtattn_fwd(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz, w.H, 2000,
                      w.scale, gt.GTATTN_F32)
    assert e.value.status == gt.GTATTN_ERR_INVALID_ARG


# ---------------------------------------------------------------------------
# dense-block tensor-core path
# ---------------------------------------------------------------------------
def _mixed_dense_graph(rng, sizes, n_sparse, sparse_edges):
    """Complete blocks of the given sizes (self-loops included) followed by
    `n_sparse` rows of a random sparse graph that also points into the
    blocks; returns COO (src, dst) and n."""
    src, dst = [], []
    base = 0
    for n in sizes:
        r = np.arange(base, base + n)
        src.append(np.tile(r, n))
        dst.append(np.repeat(r, n))
        base += n
    n_total = base + n_sparse
    s = rng.integers(0, n_total, sparse_edges)
    d = rng.integers(base, n_total, sparse_edges)
    src.append(s)
    dst.append(d)
    return np.concatenate(src), np.concatenate(dst), n_total


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("out32", [True, False])
def test_dense_path_mixed_graph(out32, D):
    rng = np.random.default_rng(77)
    src, dst, n = _mixed_dense_graph(rng, [128, 384, 256], 500, 6000)
    ip, ix = wl.csr_by_destination(src, dst, n)
    Q, K, V = (0.5 * rng.standard_normal((n, 8, D)) for _ in range(3))
    w = _mk(ip, ix, Q, K, V, "bf16")
    ref = oracle_rows(w)["out"]
    d = to_device(w, out32=out32)
    plan = gt.Plan(d["indptr"], d["indices"], detect_dense=True)
    info = plan.info()
    assert info["n_dense_blocks"] == 3 and info["n_dense_rows"] == 768
    gt.gtattn_profile_enable(True)
    gt.gtattn_profile_read(reset=True)
    d["out"].fill_(float("nan"))
    gt.gtattn_fwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], 8, D, w.scale,
                       _dt(d))
    torch.cuda.synchronize()
    prof = gt.gtattn_profile_read(reset=True)
    gt.gtattn_profile_enable(False)
    assert prof["dense"]["launches"] == 1, prof
    assert plan.info()["device_error"] == 0
    plan.close()
    got = out_to_numpy(d["out"])
    check_out(w, got, ref, f"mixed dense+sparse D={D} out32={out32}", out32=out32)


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_dense_path_ragged_blocks(sign, D):
    # complete blocks whose sizes are not multiples of the 128-row tile: the
    # last key tile of each is masked (a negative scale flips the mask's
    # sign), rows past a block's end in its last query tile are not stored
    rng = np.random.default_rng(78)
    sizes = [200, 128, 300, 511, 129]
    src, dst, n = _mixed_dense_graph(rng, sizes, 400, 5000)
    ip, ix = wl.csr_by_destination(src, dst, n)
    Q, K, V = (0.5 * rng.standard_normal((n, 8, D)) for _ in range(3))
    w = _mk(ip, ix, Q, K, V, "bf16")
    scale = sign * w.scale
    ref = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, scale, threads=8)["out"]
    for out32 in (True, False):
        d = to_device(w, out32=out32)
        plan = gt.Plan(d["indptr"], d["indices"], detect_dense=True)
        info = plan.info()
        assert info["n_dense_blocks"] == len(sizes) and info["n_dense_rows"] == sum(sizes)
        gt.gtattn_profile_enable(True)
        gt.gtattn_profile_read(reset=True)
        d["out"].fill_(float("nan"))
        gt.gtattn_fwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], 8, D, scale, _dt(d))
        torch.cuda.synchronize()
        prof = gt.gtattn_profile_read(reset=True)
        gt.gtattn_profile_enable(False)
        assert prof["dense"]["launches"] == 1, prof
        assert plan.info()["device_error"] == 0
        plan.close()
        check_out(w, out_to_numpy(d["out"]), ref, f"ragged dense blocks D={D} sign={sign} out32={out32}",
                  out32=out32)


@pytest.mark.parametrize("D", [32, 64, 128])
def test_dense_path_large_scores(D):
    # logits spread over a wide range: the running max is raised mid-row and
    # O is rescaled
    rng = np.random.default_rng(5)
    n = 512
    src, dst, _ = _mixed_dense_graph(rng, [n], 0, 0)
    ip, ix = wl.csr_by_destination(src, dst, n)
    Q = rng.standard_normal((n, 2, D)) * 3 * np.sqrt(64 / D)
    K = rng.standard_normal((n, 2, D)) * 3
    K[:, :, :] *= np.linspace(0.1, 2.0, n)[:, None, None]     # later keys larger: max grows across tiles
    V = rng.standard_normal((n, 2, D))
    w = _mk(ip, ix, Q, K, V, "bf16")
    ref = oracle_rows(w)["out"]
    d = to_device(w, out32=True)
    plan = gt.Plan(d["indptr"], d["indices"], detect_dense=True)
    gt.gtattn_fwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], 2, D, w.scale,
                       _dt(d))
    torch.cuda.synchronize()
    assert plan.info()["device_error"] == 0
    plan.close()
    check_out(w, out_to_numpy(d["out"]), ref, f"dense large scores D={D}", out32=True)


@pytest.mark.parametrize("n", [4096, 4097])
def test_small_graph_binning_threshold(n):
    # one-block binning (n <= 4096) and the three-kernel binning (n > 4096),
    # with hub rows that are split into chunks, empty rows and degree-1 rows
    rng = np.random.default_rng(n)
    deg = rng.integers(0, 6, n)
    deg[rng.choice(n, 6, replace=False)] = [257, 300, 512, 513, 1000, 2500]
    deg[:3] = [0, 1, 0]
    indptr = np.zeros(n + 1, np.int64)
    np.cumsum(deg, out=indptr[1:])
    indices = rng.integers(0, n, int(indptr[-1])).astype(np.int32)
    H, D = 2, 16
    Q, K, V = (rng.standard_normal((n, H, D)).astype(np.float32) for _ in range(3))
    w = wl.Workload("threshold", n, H, D, "f32", indptr.astype(np.int32), indices, Q, K, V,
                    float(np.float32(1 / np.sqrt(D))))
    ref = oracle_rows(w, want_probs=True)
    for path in ("fwd", "probs", "plan"):
        got, _, pr = run(w, to_device(w), path)
        check_out(w, got, ref["out"], f"n={n} {path}")
        if path == "probs":
            assert_close(pr, ref["probs"], w.dtype, "probs", PROB_TOL)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_wide_logit_range_raises_running_max(dtype):
    # logits spread over tens of log2 units inside rows, in random order: the
    # row kernels' running maximum (raised only past a slack) moves mid-row,
    # in whole rows, in split rows' chunks and across edge slots
    rng = np.random.default_rng(21)
    n, H, D = 3000, 4, 32
    deg = rng.integers(1, 48, n)
    deg[rng.choice(n, 20, replace=False)] = rng.integers(257, 1500, 20)
    indptr = np.zeros(n + 1, np.int64)
    np.cumsum(deg, out=indptr[1:])
    indices = rng.integers(0, n, int(indptr[-1]))
    Q = rng.standard_normal((n, H, D))
    K = rng.standard_normal((n, H, D)) * np.linspace(0.2, 4.0, n)[:, None, None]
    V = rng.standard_normal((n, H, D))
    w = _mk(indptr, indices, Q, K, V, dtype)
    # the spread this gives, in log2 units, inside the longer rows
    dst = np.repeat(np.arange(n), deg)
    lg = np.einsum("ehd,ehd->eh", w.Q[dst].astype(np.float64), w.K[w.indices].astype(np.float64)) * w.scale
    spans = [np.ptp(lg[indptr[r]:indptr[r + 1]]) * np.log2(np.e) for r in range(n) if deg[r] >= 20]
    assert np.median(spans) > 16
    ref = oracle_rows(w, want_probs=True)
    for path, kw in (("fwd", {}), ("plan", dict(long_row_min=8, chunk_edges=5)), ("probs", {})):
        d = to_device(w, out32=(dtype == "bf16"))
        got, _, pr = run(w, d, path, **kw)
        check_out(w, got, ref["out"], f"wide logits {path}", out32=True)
        if path == "probs":
            assert_close(pr, ref["probs"], w.dtype, "probs", PROB_TOL)


def test_dense_wait_timeout_is_reported_and_a_later_call_is_correct():
    # The plan's test hook makes the dense-block kernel's softmax warps wait
    # first on a barrier nothing completes, with every wait for another
    # warp's data bounded by 2000 SM cycles: that wait runs out, the MMA
    # warp's waits for P and the TMA warp's waits for free stages run out in
    # turn, each CTA drains the copies and products it issued (those waits
    # keep their own half-second bound), frees its tensor memory and returns.
    # The call returns, the plan reports the timeout once (the record is
    # cleared when read), and the context stays usable: a plan without the
    # hook then gives the oracle's result.
    w = small("dense_blocks")
    d = to_device(w, out32=True)
    plan = gt.Plan(d["indptr"], d["indices"], detect_dense=True, wait_cycles=2000, test_stall=True)
    assert plan.info()["n_dense_blocks"] > 0
    gt.gtattn_fwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], w.H, w.D, w.scale,
                       _dt(d))
    torch.cuda.synchronize()
    assert plan.info()["device_error"] == 1
    assert plan.info()["device_error"] == 0
    plan.close()
    got, _, _ = run(w, d, "plan", detect_dense=True)
    check_out(w, got, oracle_rows(w)["out"], "dense after a timeout", out32=True)


@pytest.mark.parametrize("H,D,dtype", [(4, 32, "bf16"), (8, 64, "f32"), (3, 5, "f32"), (2, 8, "bf16")])
def test_small_graph_one_launch_with_split_rows(H, D, dtype):
    # N <= 4096 and nnz <= 65536: the plan-less forward is one cooperative
    # launch that bins in shared memory; rows of more than 1024 entries (the
    # default threshold) are split into chunks whose partials are combined
    # after the grid-wide sync
    rng = np.random.default_rng(H * 100 + D)
    n = 3000
    src = np.concatenate([rng.integers(0, n, 12000), rng.integers(0, n, 2500), rng.integers(0, n, 4000)])
    dst = np.concatenate([rng.integers(0, n, 12000), np.full(2500, 5), np.full(4000, 2999)])
    key = np.unique(dst * n + src)
    ip, ix = wl.csr_by_destination(key % n, key // n, n)
    assert np.sort(np.diff(ip))[-2] > 1024 and ip[-1] <= 65536
    Q, K, V = (rng.standard_normal((n, H, D)) for _ in range(3))
    w = _mk(ip, ix, Q, K, V, dtype)
    ref = oracle_rows(w)["out"]
    for out32 in ((True, False) if dtype == "bf16" else (False,)):
        d = to_device(w, out32=out32)
        gt.gtattn_profile_enable(True)
        gt.gtattn_profile_read(reset=True)
        got, _, _ = run(w, d, "fwd")
        prof = gt.gtattn_profile_read(reset=True)
        gt.gtattn_profile_enable(False)
        assert prof["rows"]["launches"] == 1 and prof["bin"]["launches"] == 0 and prof["combine"]["launches"] == 0
        check_out(w, got, ref, f"one-launch H={H} D={D} {dtype} out32={out32}", out32=out32)


@pytest.mark.parametrize("H,D,dtype", [(8, 10, "f32"), (8, 10, "bf16"), (5, 7, "f32"), (32, 16, "bf16"),
                                        (1, 2, "f32"), (3, 1, "bf16"), (16, 3, "f32")])
def test_narrow_head_kernel(H, D, dtype):
    # one lane per head (heads of at most 16 features): rows whole, rows of
    # many entries over several lane groups, rows split into chunks, the
    # one-launch small-graph path, and the row statistics
    rng = np.random.default_rng(H * 37 + D)
    n = 900
    ip, ix = wl.random_csr(rng, n, 14000, self_loops=True, degree_skew=1.2)
    assert np.diff(ip).max() > 256
    Q, K, V = (rng.standard_normal((n, H, D)) for _ in range(3))
    w = _mk(ip, ix, Q, K, V, dtype)
    ref = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, want_probs=True)
    d = to_device(w)
    runs = [("fwd", {}), ("plan", {}), ("plan", dict(kernel=gt.GTATTN_KERNEL_NARROW)),
            ("plan", dict(kernel=gt.GTATTN_KERNEL_NARROW, long_row_min=30, chunk_edges=11)),
            ("plan", dict(kernel=gt.GTATTN_KERNEL_NARROW, long_row_min=-1, chunk_edges=4))]
    for path, kw in runs:
        got, _, _ = run(w, d, path, **kw)
        check_out(w, got, ref["out"], f"narrow H={H} D={D} {dtype} {path} {kw}")
    # statistics: log2-sum-exp of each row's logits
    plan = gt.Plan(d["indptr"], d["indices"], kernel=gt.GTATTN_KERNEL_NARROW, long_row_min=30, chunk_edges=11)
    o32 = torch.full((n, H, D), float("nan"), device="cuda")
    stats = torch.full((n, H), float("nan"), device="cuda")
    gt.gtattn_fwd_plan_stats(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], o32, stats, H, D, w.scale,
                             gt.GTATTN_F32 if dtype == "f32" else gt.GTATTN_BF16_OUT_F32)
    torch.cuda.synchronize()
    plan.close()
    check_out(w, o32.cpu().numpy().astype(np.float64), ref["out"], "narrow stats-forward output", out32=True)
    lg = ref["logits"]
    deg = np.diff(w.indptr)
    want = np.full((n, H), -np.inf)
    rows = np.flatnonzero(deg > 0)
    m = np.maximum.reduceat(lg, w.indptr[:-1][rows], axis=0)
    ssum = np.add.reduceat(np.exp(lg - np.repeat(m, deg[rows], axis=0)), w.indptr[:-1][rows], axis=0)
    want[rows] = (m + np.log(ssum)) / np.log(2.0)
    got = stats.cpu().numpy().astype(np.float64)
    assert (got[deg == 0] == -np.inf).all()
    err = np.abs(got[rows] - want[rows])
    assert (err <= 1e-5 * (1 + np.abs(want[rows]))).all(), float(err.max())


def test_narrow_kernel_refuses_wide_shapes():
    # forcing the narrow kernel on heads wider than 16 or more than 32 heads
    rng = np.random.default_rng(3)
    n = 64
    ip, ix = wl.random_csr(rng, n, 300, self_loops=True)
    for H, D in ((2, 17), (33, 4)):
        Q = rng.standard_normal((n, H, D))
        w = _mk(ip, ix, Q, Q, Q)
        d = to_device(w)
        plan = gt.Plan(d["indptr"], d["indices"], kernel=gt.GTATTN_KERNEL_NARROW)
        with pytest.raises(gt.GtattnError):
            gt.gtattn_fwd_plan(plan, d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], H, D, w.scale,
                               gt.GTATTN_F32)
        plan.close()


def test_head_groups_on_a_graph_whose_k_and_v_exceed_the_l2():
    # K and V together above 85 % of the L2, 1 KB rows: the forward runs the
    # heads in groups (one launch of the row kernel per group), each group
    # reading its columns of the rows, and one combine for the split rows of
    # every group (three hub rows of a few thousand entries); sampled rows
    # (the hubs among them) against the oracle, and the same bits from the
    # host-buffer path (its row chunks decide the groups from the whole graph)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    H, D = 8, 64
    n = int(0.5 * l2 / (H * D * 2)) + 1000   # K + V = 2 n H D 2 bytes: about the whole L2
    rng = np.random.default_rng(91)
    src = np.concatenate([rng.integers(0, n, 6 * n), rng.integers(0, n, 9000)])
    dst = np.concatenate([rng.integers(0, n, 6 * n), np.repeat([7, n // 2, n - 3], 3000)])
    key = np.unique(dst.astype(np.int64) * n + src)
    ip, ix = wl.csr_by_destination(key % n, key // n, n)
    assert np.sort(np.diff(ip))[-3] > 2048
    Q, K, V = (rng.standard_normal((n, H, D)).astype(np.float32) for _ in range(3))
    w = _mk(ip, ix, Q, K, V, "bf16")
    d = to_device(w, out32=True)
    gt.gtattn_profile_enable(True)
    gt.gtattn_profile_read(reset=True)
    got, _, _ = run(w, d, "fwd")
    prof = gt.gtattn_profile_read(reset=True)
    gt.gtattn_profile_enable(False)
    kv = 2 * n * H * D * 2
    groups = 1
    while kv / groups > 0.85 * l2 and H % (2 * groups) == 0 and H * D * 2 / (2 * groups) >= 512:
        groups *= 2
    assert groups > 1 and prof["rows"]["launches"] == groups, (groups, prof["rows"])
    assert prof["combine"]["launches"] == 1, prof["combine"]
    rows = np.union1d(sample_rows(w, n_random=800), [7, n // 2, n - 3])
    ref = oracle_rows(w, rows=rows)["out"]
    check_out(w, got[rows], ref, f"head groups x{groups}", out32=True)
    # the host-buffer call: same bits
    out_h = torch.empty(n, H, D, dtype=torch.float32).pin_memory()
    qh, kh, vh = (d[k].cpu().pin_memory() for k in ("Q", "K", "V"))
    gt.gtattn_fwd_host(torch.from_numpy(w.indptr), torch.from_numpy(w.indices), qh, kh, vh, out_h, n, w.nnz, H, D,
                       w.scale, gt.GTATTN_BF16_OUT_F32)
    torch.cuda.synchronize()
    assert np.array_equal(out_h.numpy().astype(np.float64), got)
