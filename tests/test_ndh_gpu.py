"""Head-innermost node rows (gtattn_fwd_ndh): Q, K, V and out as [N, D, H],
the layout SparseMHA of "Graph Transformer in a Nutshell" reshapes its
projections to.  The result, permuted back to [N, H, D], must meet the
oracle's tolerance on the same inputs (split hub rows included)."""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_helpers import assert_close, out_to_numpy

torch = pytest.importorskip("torch")
gt = pytest.importorskip("graph_transformer_sparse_gb300")

pytestmark = pytest.mark.gpu


def _ndh_device(w, out32):
    d = dict(indptr=torch.from_numpy(w.indptr).cuda(), indices=torch.from_numpy(w.indices).cuda())
    for name in ("Q", "K", "V"):
        if w.dtype == "bf16":
            bits = np.ascontiguousarray(w.bits[name].transpose(0, 2, 1)).view(np.int16)
            d[name] = torch.from_numpy(bits).cuda().view(torch.bfloat16)
        else:
            d[name] = torch.from_numpy(np.ascontiguousarray(getattr(w, name).transpose(0, 2, 1))).cuda()
    d["out"] = torch.full(d["Q"].shape, float("nan"), dtype=torch.float32 if out32 else d["Q"].dtype, device="cuda")
    return d


@pytest.mark.parametrize("name", ["tiny_random", "molecules", "erdos_renyi", "rmat"])
@pytest.mark.parametrize("out32", [False, True])
def test_ndh_matches_oracle(name, out32):
    w = wl.small_workload(name)
    if out32 and w.dtype == "f32":
        pytest.skip("fp32 inputs have fp32 output already")
    d = _ndh_device(w, out32)
    dt = gt.GTATTN_F32 if w.dtype == "f32" else (gt.GTATTN_BF16_OUT_F32 if out32 else gt.GTATTN_BF16)
    gt.gtattn_fwd_ndh(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz, w.H, w.D, w.scale, dt)
    torch.cuda.synchronize()
    got = out_to_numpy(d["out"]).transpose(0, 2, 1)          # back to [N, H, D]
    ref = oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, threads=8)["out"]
    assert_close(got, ref, w.dtype, f"{name} [N, D, H]", rounded_bf16=(w.dtype == "bf16" and not out32))
