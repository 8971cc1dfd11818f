"""GPU parity of the projected attention block (gtattn_fwd_proj) against the
fp64 oracle: q, k, v = X W^T + b, the sparse attention, Y = o Wo^T + bo --
SparseMHA.forward of "Graph Transformer in a Nutshell" (biases, head-inner
features) and the attention part of TransLayer.forward of "Efficient Sparse
Transformer implementation with DGL's builtin operators" (no biases,
head-major features).

Each stage is checked against the oracle on the inputs that stage actually
received (the GPU's own q, k, v and o, read back through the optional
outputs), so the bound of each comparison is that of one stage:

* a linear map accumulates K products in fp32: |err| <= 2e-5 * sum_k |x_k w_k|
  + |b| terms (K * 2^-24 = 3.1e-5 is the worst case for K = 512; ordered
  sums stay far below it), plus half a bf16 ulp of the value when the
  result is stored as bf16;
* the attention: the parity tolerances of the forward (fp32 rel 1e-5 /
  abs 1e-6; bf16 rel 2e-3 / abs 1e-5 plus the output's own rounding).

End to end (fp32 only): the oracle's whole block in fp64 with q, k, v and o
held as float32 between the stages, within 2e-4 of the output map's
condition sum_f |o_f||Wo_jf| + |bo_j| -- the two maps' worst-case 3e-5
relative errors moving the logits by at most ~1e-4 (|scale q.k| sums of a
few units) and the softmax output by as much.
"""
import zlib

import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import assert_close, half_ulp_bf16, out_to_numpy, sample_rows

torch = pytest.importorskip("torch")
gt = pytest.importorskip("graph_transformer_sparse_gb300")

pytestmark = pytest.mark.gpu

LIN_RTOL = 2e-5


def _dev(x, bf16):
    """float32 numpy -> device tensor (bf16 bits when bf16)."""
    if bf16:
        _, bits = wl.bf16_round(x)
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def _params(rng, N, F_in, H, D, F_out, bf16, biases):
    """X ~ N(0, 1); weights and biases ~ U(-1/sqrt(fan_in), 1/sqrt(fan_in))
    (nn.Linear's default initialisation); bf16 operands rounded to bf16."""
    HD = H * D
    X = rng.standard_normal((N, F_in), dtype=np.float32)
    a1, a2 = 1 / np.sqrt(F_in), 1 / np.sqrt(HD)
    W = rng.uniform(-a1, a1, (3 * HD, F_in)).astype(np.float32)
    Wo = rng.uniform(-a2, a2, (F_out, HD)).astype(np.float32)
    b = rng.uniform(-a1, a1, 3 * HD).astype(np.float32) if biases else None
    bo = rng.uniform(-a2, a2, F_out).astype(np.float32) if biases else None
    if bf16:
        X, W, Wo = (wl.bf16_round(t)[0] for t in (X, W, Wo))
    return X, W, b, Wo, bo


def _check_linear(got, X, W, b, stored_bf16, what, rows=None):
    """got [R, Nout] against oracle.linear(X[rows], W, b) within the fp32
    accumulation bound (plus the bf16 storage rounding)."""
    Xs = X if rows is None else X[rows]
    ref = oracle.linear(Xs, W, b)
    cond = oracle.linear(np.abs(Xs), np.abs(W), None if b is None else np.abs(b))
    bound = LIN_RTOL * cond + 1e-7
    if stored_bf16:
        bound = bound + half_ulp_bf16(ref)
    err = np.abs(np.asarray(got, np.float64) - ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside; worst excess "
                           f"{(err - bound).max():.3g} at {np.unravel_index(np.argmax(err - bound), err.shape)}")


def _merge(O, heads_inner):
    """[R, H, D] -> [R, H*D] in the block's feature order (head-inner:
    feature d*H + h; head-major: h*D + d)."""
    R, H, D = O.shape
    return O.transpose(0, 2, 1).reshape(R, D * H) if heads_inner else O.reshape(R, H * D)


def _run(indptr, indices, N, X, W, b, Wo, bo, H, D, F_out, scale, dtype, heads_inner):
    bf = dtype != "f32"
    code = {"f32": gt.GTATTN_F32, "bf16": gt.GTATTN_BF16, "bf16_out_f32": gt.GTATTN_BF16_OUT_F32}[dtype]
    HD, F_in = H * D, X.shape[1]
    d = dict(indptr=torch.from_numpy(indptr).cuda(), indices=torch.from_numpy(indices).cuda(),
             X=_dev(X, bf), W=_dev(W, bf), Wo=_dev(Wo, bf),
             b=None if b is None else torch.from_numpy(b).cuda(),
             bo=None if bo is None else torch.from_numpy(bo).cuda())
    et = torch.bfloat16 if bf else torch.float32
    yt = torch.bfloat16 if dtype == "bf16" else torch.float32
    qkv = torch.full((3, N, H, D), float("nan"), dtype=et, device="cuda")
    attn = torch.full((N, H, D), float("nan"), dtype=et, device="cuda")
    Y = torch.full((N, F_out), float("nan"), dtype=yt, device="cuda")
    gt.gtattn_fwd_proj(d["indptr"], d["indices"], d["X"], d["W"], d["b"], d["Wo"], d["bo"], Y, N,
                       int(indptr[-1]), F_in, H, D, F_out, scale, code, heads_inner=heads_inner, qkv=qkv,
                       attn=attn)
    torch.cuda.synchronize()
    assert gt.gtattn_device_errors() == 0
    return out_to_numpy(qkv).astype(np.float32), out_to_numpy(attn).astype(np.float32), out_to_numpy(Y)


def _check_block(indptr, indices, X, W, b, Wo, bo, H, D, F_out, dtype, heads_inner, rows=None, seed_tag=""):
    N = X.shape[0]
    HD = H * D
    scale = float(np.float32(1 / np.sqrt(D)))
    bf = dtype != "f32"
    qkv, attn, Y = _run(indptr, indices, N, X, W, b, Wo, bo, H, D, F_out, scale, dtype, heads_inner)
    sel = np.arange(N) if rows is None else rows
    # (1) q, k, v: each map against the oracle's linear layer, in head-major [N, H, D]
    for g, name in enumerate("qkv"):
        Wg = W[g * HD:(g + 1) * HD]
        bg = None if b is None else b[g * HD:(g + 1) * HD]
        # the oracle's [R, HD] in the block's feature order, as [R, H, D]
        got = _merge(qkv[g][sel], heads_inner)
        _check_linear(got, X, Wg, bg, bf, f"{seed_tag} {name} map", rows=sel)
    # (2) the attention on the GPU's own q, k, v
    ref = oracle.sparse_mha(indptr, indices, qkv[0], qkv[1], qkv[2], scale, rows=sel, threads=8)["out"]
    assert_close(attn[sel], ref, "bf16" if bf else "f32", f"{seed_tag} attention", rounded_bf16=bf)
    # (3) the out map on the GPU's own o, merged in the block's feature order
    _check_linear(Y[sel], _merge(attn, heads_inner), Wo, bo, dtype == "bf16", f"{seed_tag} out map", rows=sel)
    return qkv, attn, Y, scale


CASES = [
    # workload (small version), H, D, F_in, F_out, dtype, heads_inner, biases
    ("tiny_random", 8, 64, 512, 512, "f32", True, True),
    ("molecules", 8, 10, 80, 80, "f32", True, True),          # SparseMHA's defaults: hidden 80, 8 heads
    ("erdos_renyi", 8, 64, 512, 512, "bf16", False, False),   # TransLayer: no biases, head-major
    ("erdos_renyi", 8, 64, 512, 512, "bf16_out_f32", True, True),
    ("rmat", 4, 32, 128, 128, "bf16", True, True),
    ("dense_blocks", 8, 64, 512, 512, "bf16", False, True),
    ("rmat", 3, 8, 40, 56, "bf16", True, True),               # ragged: N, K and column tails
    ("rmat", 4, 16, 96, 48, "bf16_out_f32", False, True),     # F_in, H*D, F_out all different
    ("molecules", 2, 6, 20, 12, "bf16", True, True),          # F_in, H*D not multiples of 8: CUDA cores
]


@pytest.mark.parametrize("name,H,D,F_in,F_out,dtype,heads_inner,biases", CASES)
def test_proj_block_stages(name, H, D, F_in, F_out, dtype, heads_inner, biases):
    w = wl.small_workload(name)
    rng = np.random.default_rng(zlib.crc32(repr((name, H, D, F_in, F_out, dtype, heads_inner)).encode()))
    X, W, b, Wo, bo = _params(rng, w.N, F_in, H, D, F_out, dtype != "f32", biases)
    _check_block(w.indptr, w.indices, X, W, b, Wo, bo, H, D, F_out, dtype, heads_inner, seed_tag=name)


@pytest.mark.parametrize("name,heads_inner", [("tiny_random", True), ("molecules", True), ("molecules", False)])
def test_proj_block_end_to_end_f32(name, heads_inner):
    w = wl.make_workload(name)
    H, D = w.H, w.D
    F = H * D
    rng = np.random.default_rng(5)
    X, W, b, Wo, bo = _params(rng, w.N, F, H, D, F, False, True)
    qkv, attn, Y, scale = _check_block(w.indptr, w.indices, X, W, b, Wo, bo, H, D, F, "f32", heads_inner,
                                       seed_tag=name)
    HD = H * D
    ref = oracle.sparse_mha_proj(w.indptr, w.indices, X, W[:HD], W[HD:2 * HD], W[2 * HD:], Wo, b[:HD],
                                 b[HD:2 * HD], b[2 * HD:], bo, H, D, scale, heads_inner=heads_inner, store="f32",
                                 threads=8)
    cond = oracle.linear(np.abs(_merge(attn, heads_inner)), np.abs(Wo), np.abs(bo))
    err = np.abs(Y - ref)
    assert (err <= 2e-4 * cond + 1e-6).all(), float((err - 2e-4 * cond).max())


def test_proj_heads_inner_is_the_permuted_block():
    # the same weights read with head-inner features equal the head-major
    # block on weights whose rows (q, k, v) and columns (out) are permuted
    w = wl.small_workload("rmat")
    H, D = 4, 32
    HD = H * D
    rng = np.random.default_rng(11)
    X, W, b, Wo, bo = _params(rng, w.N, HD, H, D, HD, True, True)
    f = np.arange(HD)
    perm = (f % D) * H + f // D          # head-major feature h*D + d <- head-inner d*H + h
    Wp = np.concatenate([W[g * HD:(g + 1) * HD][perm] for g in range(3)])
    bp = np.concatenate([b[g * HD:(g + 1) * HD][perm] for g in range(3)])
    _, a1, y1 = _run(w.indptr, w.indices, w.N, X, W, b, Wo, bo, H, D, HD, 0.125, "bf16", True)
    _, a2, y2 = _run(w.indptr, w.indices, w.N, X, Wp, bp, Wo[:, perm], bo, H, D, HD, 0.125, "bf16", False)
    assert np.array_equal(a1, a2) and np.array_equal(y1, y2)


def test_proj_empty_graph_and_bad_arguments():
    lib = gt.load()
    INV = gt.GTATTN_ERR_INVALID_ARG
    f = lib.gtattn_fwd_proj
    # heads_inner 2, F_in 0, misaligned bf16 X: rejected before any GPU work
    assert f(16, 16, 16, 16, None, 16, None, 16, None, None, 4, 4, 8, 2, 4, 8, 2, 1.0, 1, None) == INV
    assert f(16, 16, 16, 16, None, 16, None, 16, None, None, 4, 4, 0, 2, 4, 8, 0, 1.0, 1, None) == INV
    assert f(16, 16, 17, 16, None, 16, None, 16, None, None, 4, 4, 8, 2, 4, 8, 0, 1.0, 1, None) == INV
    assert f(16, 16, 16, 16, 18, 16, None, 16, None, None, 4, 4, 8, 2, 4, 8, 0, 1.0, 1, None) == INV
    # N = 0: nothing to do
    z = torch.zeros(16, device="cuda")
    assert f(z.data_ptr(), None, None, None, None, None, None, None, None, None, 0, 0, 8, 2, 4, 8, 0, 1.0, 0,
             None) == gt.GTATTN_OK
    # a graph with no entries: attention rows are zero, Y = bo
    N, H, D = 50, 2, 8
    rng = np.random.default_rng(3)
    X, W, b, Wo, bo = _params(rng, N, 16, H, D, 24, False, True)
    _, attn, Y = _run(np.zeros(N + 1, np.int32), np.zeros(0, np.int32), N, X, W, b, Wo, bo, H, D, 24, 0.3,
                      "f32", False)
    assert np.all(attn == 0)
    assert np.allclose(Y, np.broadcast_to(bo, Y.shape), rtol=0, atol=0)


@pytest.mark.slow
def test_proj_block_full_size_rmat_sampled_rows():
    # the bench's configuration: R-MAT at full size, 4 x 32 bf16, hidden 128,
    # SparseMHA's head-inner features with biases; sampled rows (hubs included)
    w = wl.make_workload("rmat")
    H, D = w.H, w.D
    HD = H * D
    rng = np.random.default_rng(21)
    X, W, b, Wo, bo = _params(rng, w.N, HD, H, D, HD, True, True)
    rows = sample_rows(w, n_random=600, n_top=32)
    _check_block(w.indptr, w.indices, X, W, b, Wo, bo, H, D, HD, "bf16", True, rows=rows, seed_tag="rmat full")
