"""gtattn_fwd_host: the forward on host buffers (copies in, compute, copy out,
overlapped over row chunks) must give exactly gtattn_fwd's output on the same
inputs -- every row is computed by the same kernels whatever the chunking --
and meet the oracle's tolerance on a small case."""
import numpy as np
import pytest

import workloads as wl
from gpu_helpers import assert_close, oracle_rows, out_to_numpy, to_device

torch = pytest.importorskip("torch")
gt = pytest.importorskip("graph_transformer_sparse_gb300")

pytestmark = pytest.mark.gpu


def _host(w, out32=False):
    """Pinned host tensors of the workload and a host output buffer."""
    h = dict(indptr=torch.from_numpy(w.indptr).pin_memory(), indices=torch.from_numpy(w.indices).pin_memory())
    for name in ("Q", "K", "V"):
        if w.dtype == "bf16":
            h[name] = torch.from_numpy(w.bits[name].view(np.int16)).view(torch.bfloat16).pin_memory()
        else:
            h[name] = torch.from_numpy(getattr(w, name)).pin_memory()
    h["out"] = torch.empty(h["Q"].shape, dtype=torch.float32 if out32 else h["Q"].dtype).pin_memory()
    return h


def _dt(w, out32):
    if w.dtype == "f32":
        return gt.GTATTN_F32
    return gt.GTATTN_BF16_OUT_F32 if out32 else gt.GTATTN_BF16


def _host_out(w, out32=False):
    h = _host(w, out32)
    h["out"].fill_(float("nan"))
    gt.gtattn_fwd_host(h["indptr"], h["indices"], h["Q"], h["K"], h["V"], h["out"], w.N, w.nnz, w.H, w.D,
                       w.scale, _dt(w, out32))
    torch.cuda.synchronize()
    return h["out"]


def _device_out(w, out32=False):
    d = to_device(w, out32=out32)
    d["out"].fill_(float("nan"))
    gt.gtattn_fwd(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz, w.H, w.D, w.scale,
                  _dt(w, out32))
    torch.cuda.synchronize()
    return d["out"].cpu()


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


@pytest.mark.parametrize("name", ["tiny_random", "molecules"])
def test_host_matches_device_small(name):
    w = wl.make_workload(name)
    assert _same_bits(_host_out(w), _device_out(w))


def test_host_meets_oracle():
    w = wl.small_workload("erdos_renyi")
    got = out_to_numpy(_host_out(w, out32=True))
    assert_close(got, oracle_rows(w)["out"], w.dtype, "host path vs oracle")


@pytest.mark.parametrize("out32", [False, True])
def test_host_many_chunks_bitexact(out32):
    # ~3.4 M entries: several row chunks, hub rows (split into partials),
    # and empty rows
    rng = np.random.default_rng(11)
    n = 200_000
    deg = np.minimum(rng.zipf(1.6, n), 4000).astype(np.int64)
    deg[rng.random(n) < 0.05] = 0
    indptr = np.zeros(n + 1, np.int64)
    np.cumsum(deg, out=indptr[1:])
    indices = rng.integers(0, n, int(indptr[-1])).astype(np.int32)
    H, D = 2, 32
    Q, K, V = (rng.standard_normal((n, H, D)).astype(np.float32) for _ in range(3))
    w = wl.Workload("chunks", n, H, D, "f32", indptr.astype(np.int32), indices, Q, K, V,
                    float(np.float32(1 / np.sqrt(D))))
    w.dtype = "bf16"
    for name in ("Q", "K", "V"):
        vals, bits = wl.bf16_round(getattr(w, name))
        setattr(w, name, vals)
        w.bits[name] = bits
    assert w.nnz > 3 * (1 << 20)
    got, ref = _host_out(w, out32), _device_out(w, out32)
    assert _same_bits(got, ref)
    empty = deg == 0
    assert torch.all(got[torch.from_numpy(empty)].float() == 0)


def test_host_rejects_inconsistent_csr():
    w = wl.make_workload("tiny_random")
    h = _host(w)
    with pytest.raises(gt.GtattnError) as e:
        gt.gtattn_fwd_host(h["indptr"], h["indices"], h["Q"], h["K"], h["V"], h["out"], w.N, w.nnz - 1, w.H,
                           w.D, w.scale, gt.GTATTN_F32)
    assert e.value.status == gt.GTATTN_ERR_BAD_CSR
    with pytest.raises(ValueError):
        d = to_device(w)
        gt.gtattn_fwd_host(d["indptr"], d["indices"], d["Q"], d["K"], d["V"], d["out"], w.N, w.nnz, w.H, w.D,
                           w.scale, gt.GTATTN_F32)
