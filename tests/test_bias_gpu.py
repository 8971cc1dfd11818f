"""Per-edge additive bias (gtattn_fwd_bias): the logit of CSR entry e, head h
is scale * q.k + bias[e, h] (the Graphormer spatial-encoding bias of the
"Graph Transformer theory, derivation and implementation" page; -inf removes
the pair).  The CUDA path against the fp64 oracle on the same inputs, and
against the plain forward where the bias reduces to it."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import PROB_TOL, assert_close, out_to_numpy, to_device

torch = pytest.importorskip("torch")
gt = pytest.importorskip("graph_transformer_sparse_gb300")

pytestmark = pytest.mark.gpu

_cache = {}


def small(name):
    if name not in _cache:
        _cache[name] = wl.small_workload(name)
    return _cache[name]


def _dt(w, out32):
    if w.dtype == "f32":
        return gt.GTATTN_F32
    return gt.GTATTN_BF16_OUT_F32 if out32 else gt.GTATTN_BF16


def _bias(w, seed, minus_inf=0.1, removed_row=True):
    """fp32 [nnz, H]: N(0, 1) values, a fraction set to -inf, and (optionally)
    one row of degree >= 2 with every entry removed."""
    rng = np.random.default_rng(seed)
    b = rng.standard_normal((w.nnz, w.H)).astype(np.float32)
    b[rng.random(b.shape) < minus_inf] = -np.inf
    if removed_row:
        deg = np.diff(w.indptr)
        r = int(np.flatnonzero(deg >= 2)[0])
        b[w.indptr[r]:w.indptr[r + 1]] = -np.inf
    return b


def _run(w, d, bias_t, unfused=False):
    d["out"].fill_(float("nan"))
    lg = pr = None
    if unfused:
        lg = torch.full((w.nnz, w.H), float("nan"), device="cuda")
        pr = torch.full((w.nnz, w.H), float("nan"), device="cuda")
    gt.gtattn_fwd_bias(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], bias_t, d["out"], w.N, w.nnz, w.H,
                       w.D, w.scale, _dt(w, d["out"].dtype == torch.float32 and w.dtype == "bf16"),
                       logits=lg, probs=pr)
    torch.cuda.synchronize()
    return (out_to_numpy(d["out"]), None if lg is None else lg.cpu().numpy(),
            None if pr is None else pr.cpu().numpy())


@pytest.mark.parametrize("name", ["tiny_random", "molecules", "erdos_renyi", "rmat", "dense_blocks"])
@pytest.mark.parametrize("unfused", [False, True], ids=["fused", "unfused"])
def test_bias_matches_oracle(name, unfused):
    w = small(name)
    bias = _bias(w, seed=sum(map(ord, name)))
    ref = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, want_probs=True, threads=8, bias=bias)
    d = to_device(w, out32=(w.dtype == "bf16"))
    got, lg, pr = _run(w, d, torch.from_numpy(bias).cuda(), unfused)
    assert_close(got, ref["out"], w.dtype, f"{name} bias out")
    if unfused:
        assert_close(pr, ref["probs"], w.dtype, "bias probs", PROB_TOL)
        fin = np.isfinite(ref["logits"])
        assert np.array_equal(np.isfinite(lg), fin)
        dst = np.repeat(np.arange(w.N), np.diff(w.indptr))
        cond = w.scale * np.einsum("ehd,ehd->eh", np.abs(w.Q[dst].astype(np.float64)),
                                   np.abs(w.K[w.indices].astype(np.float64))) + np.abs(bias)
        err = np.abs(lg[fin] - ref["logits"][fin])
        assert np.all(err <= 1e-5 * cond[fin] + 1e-6)
    # the row with every entry removed is exactly zero
    r = int(np.flatnonzero(np.diff(w.indptr) >= 2)[0])
    assert np.all(got[r] == 0.0)


@pytest.mark.parametrize("name", ["tiny_random", "molecules", "rmat"])
def test_zero_bias_is_bit_exact_plain_forward(name):
    w = small(name)
    d = to_device(w)
    zero = torch.zeros((w.nnz, w.H), device="cuda")
    got, _, _ = _run(w, d, zero)
    d["out"].fill_(float("nan"))
    gt.gtattn_fwd(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz, w.H, w.D, w.scale,
                  _dt(w, False))
    torch.cuda.synchronize()
    assert np.array_equal(got, out_to_numpy(d["out"]))


def test_minus_inf_bias_equals_removed_entries():
    w = small("rmat")
    rng = np.random.default_rng(17)
    keep = rng.random(w.nnz) < 0.7
    bias = np.where(keep, 0.0, -np.inf).astype(np.float32)[:, None].repeat(w.H, axis=1)
    d = to_device(w, out32=True)
    got, _, _ = _run(w, d, torch.from_numpy(bias).cuda())
    row_of = np.repeat(np.arange(w.N), np.diff(w.indptr))
    kp = np.zeros(w.N + 1, np.int64)
    np.cumsum(np.bincount(row_of[keep], minlength=w.N), out=kp[1:])
    wk = wl.Workload("kept", w.N, w.H, w.D, w.dtype, kp.astype(np.int32), w.indices[keep], w.Q, w.K, w.V, w.scale)
    wk.bits = w.bits
    dk = to_device(wk, out32=True)
    gt.gtattn_fwd(dk["indptr"], dk["indices"], dk["Q"], dk["K"], dk["V"], dk["out"], wk.N, wk.nnz, wk.H, wk.D,
                  wk.scale, gt.GTATTN_BF16_OUT_F32)
    torch.cuda.synchronize()
    ref = oracle.sparse_mha(wk.indptr, wk.indices, wk.Q, wk.K, wk.V, wk.scale, threads=8)["out"]
    assert_close(out_to_numpy(dk["out"]), ref, w.dtype, "kept entries, plain forward")
    assert_close(got, ref, w.dtype, "-inf bias")


def test_bias_argument_errors():
    w = small("tiny_random")
    d = to_device(w)
    with pytest.raises(gt.GtattnError) as e:
        gt.gtattn_fwd_bias(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], None, d["out"], w.N, w.nnz, w.H, w.D,
                           w.scale, gt.GTATTN_F32)
    assert e.value.status == gt.GTATTN_ERR_INVALID_ARG
    buf = torch.zeros(w.nnz * w.H + 1, device="cuda")
    with pytest.raises(gt.GtattnError) as e:
        gt.gtattn_fwd_bias(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], buf.data_ptr() + 2, d["out"], w.N,
                           w.nnz, w.H, w.D, w.scale, gt.GTATTN_F32)
    assert e.value.status == gt.GTATTN_ERR_INVALID_ARG
