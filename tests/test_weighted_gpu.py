"""Weighted adjacency (gtattn_fwd_weighted): the logit of CSR entry e is
scale * (q.k) * a_e, the Hadamard product with A's stored values of
"Graph Transformer in a Nutshell" (Sparse Multi-head Attention).  The CUDA
path against the fp64 oracle on the same inputs, and against the plain
forward where the values reduce to it."""
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


def _values(w, seed):
    rng = np.random.default_rng(seed)
    a = rng.uniform(0.0, 1.0, w.nnz).astype(np.float32)
    a[rng.random(w.nnz) < 0.1] = 0.0          # stored zeros stay in the softmax
    return a


def _run(w, d, values_t, unfused=False, scale=None):
    d["out"].fill_(float("nan"))
    lg = pr = None
    if unfused:
        lg = torch.full((w.nnz, w.H), float("nan"), device="cuda")
        pr = torch.full((w.nnz, w.H), float("nan"), device="cuda")
    out32 = d["out"].dtype == torch.float32 and w.dtype == "bf16"
    gt.gtattn_fwd_weighted(d["indptr"], d["indices"], values_t, d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz, w.H,
                           w.D, w.scale if scale is None else scale, _dt(w, out32), logits=lg, probs=pr)
    torch.cuda.synchronize()
    return (out_to_numpy(d["out"]), None if lg is None else lg.cpu().numpy(),
            None if pr is None else pr.cpu().numpy())


@pytest.mark.parametrize("name", ["tiny_random", "molecules", "erdos_renyi", "rmat", "dense_blocks"])
@pytest.mark.parametrize("unfused", [False, True], ids=["fused", "unfused"])
def test_weighted_matches_oracle(name, unfused):
    w = small(name)
    values = _values(w, seed=sum(map(ord, name)) + 7)
    ref = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, want_probs=True, threads=8,
                            values=values)
    d = to_device(w, out32=(w.dtype == "bf16"))
    got, lg, pr = _run(w, d, torch.from_numpy(values).cuda(), unfused)
    assert_close(got, ref["out"], w.dtype, f"{name} weighted out")
    if unfused:
        assert_close(pr, ref["probs"], w.dtype, "weighted probs", PROB_TOL)
        dst = np.repeat(np.arange(w.N), np.diff(w.indptr))
        cond = w.scale * np.einsum("ehd,ehd->eh", np.abs(w.Q[dst].astype(np.float64)),
                                   np.abs(w.K[w.indices].astype(np.float64))) * values[:, None]
        assert np.all(np.abs(lg - ref["logits"]) <= 1e-5 * cond + 1e-6)


@pytest.mark.parametrize("name", ["tiny_random", "molecules", "rmat"])
def test_unit_values_are_bit_exact_plain_forward(name):
    w = small(name)
    d = to_device(w)
    got, _, _ = _run(w, d, torch.ones(w.nnz, device="cuda"))
    d["out"].fill_(float("nan"))
    gt.gtattn_fwd(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz, w.H, w.D, w.scale,
                  _dt(w, False))
    torch.cuda.synchronize()
    assert np.array_equal(got, out_to_numpy(d["out"]))


def test_constant_values_rescale_the_logits():
    w = small("erdos_renyi")
    c = 0.375
    d = to_device(w, out32=True)
    got, _, _ = _run(w, d, torch.full((w.nnz,), c, device="cuda"))
    ref = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, float(np.float32(w.scale * c)), threads=8)["out"]
    assert_close(got, ref, w.dtype, "constant values")


def test_weighted_argument_errors():
    w = small("tiny_random")
    d = to_device(w)
    with pytest.raises(gt.GtattnError) as e:
        gt.gtattn_fwd_weighted(d["indptr"], d["indices"], None, d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz, w.H,
                               w.D, w.scale, gt.GTATTN_F32)
    assert e.value.status == gt.GTATTN_ERR_INVALID_ARG
    buf = torch.zeros(w.nnz + 1, device="cuda")
    with pytest.raises(gt.GtattnError) as e:
        gt.gtattn_fwd_weighted(d["indptr"], d["indices"], buf.data_ptr() + 2, d["Q"], d["K"], d["V"], d["out"], w.N,
                               w.nnz, w.H, w.D, w.scale, gt.GTATTN_F32)
    assert e.value.status == gt.GTATTN_ERR_INVALID_ARG
