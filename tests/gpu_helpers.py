"""Shared helpers for the GPU parity tests: device copies of a workload,
tolerance checks against the fp64 oracle."""
import numpy as np

import oracle
import workloads as wl

# Tolerances (|gpu - oracle| <= rtol*|oracle| + atol), per output dtype.
# fp32 out: rel 1e-5 / abs 1e-6; bf16 out: rel 2e-3 / abs 1e-5 against the
# oracle run on the same bf16-rounded inputs (bf16 rounding of the output
# alone costs up to 2^-9 = 1.95e-3 relative).
TOL = {"f32": (1e-5, 1e-6), "bf16": (2e-3, 1e-5)}
PROB_TOL = (1e-5, 1e-6)


def torch_mod():
    import torch
    return torch


def to_device(w: wl.Workload, dev="cuda", out32=False):
    """Device copies of the workload; ``out32`` gives an fp32 output buffer
    for bf16 inputs (the GTATTN_BF16_OUT_F32 variant)."""
    torch = torch_mod()
    d = dict(indptr=torch.from_numpy(w.indptr).to(dev), indices=torch.from_numpy(w.indices).to(dev))
    for name in ("Q", "K", "V"):
        if w.dtype == "bf16":
            bits = w.bits[name].view(np.int16)
            d[name] = torch.from_numpy(bits).to(dev).view(torch.bfloat16)
        else:
            d[name] = torch.from_numpy(getattr(w, name)).to(dev)
    d["out"] = torch.empty(d["Q"].shape, dtype=torch.float32 if out32 else d["Q"].dtype, device=dev)
    return d


def out_to_numpy(t):
    torch = torch_mod()
    if t.dtype == torch.bfloat16:
        bits = t.view(torch.int16).cpu().numpy().view(np.uint16)
        return wl.bf16_bits_to_f32(bits).astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def half_ulp_bf16(x):
    """Half the bf16 spacing at |x| (bf16 keeps 8 significant bits): the
    largest error of rounding x to bf16."""
    m, e = np.frexp(np.abs(np.asarray(x, dtype=np.float64)))
    return np.ldexp(1.0, e - 9) * (m > 0)


def assert_close(got, ref, dtype, what="out", tol=None, rounded_bf16=False):
    """|got - ref| <= rtol*|ref| + atol.  With ``rounded_bf16`` the output was
    rounded to bf16 after the arithmetic, so the bound also allows that
    rounding: half a bf16 ulp of ref (up to 2^-8 relative)."""
    rtol, atol = tol or TOL[dtype]
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = rtol * np.abs(ref) + atol
    if rounded_bf16:
        bound = bound + half_ulp_bf16(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        worst = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside rtol={rtol} atol={atol}; "
            f"first {idx.tolist()}; worst at {worst}: got {got[worst]!r} ref {ref[worst]!r}")


def oracle_rows(w: wl.Workload, rows=None, want_probs=False, threads=8):
    return oracle.sparse_mha(w.indptr, w.indices, w.Q, w.K, w.V, w.scale, rows=rows,
                             want_probs=want_probs, threads=threads)


def sample_rows(w: wl.Workload, n_random=1500, n_top=64, seed=0):
    """Rows for sampled full-size checks: the highest-degree rows, some
    empty/degree-1 rows if present, and uniformly random rows."""
    rng = np.random.default_rng(seed)
    deg = np.diff(w.indptr)
    top = np.argsort(deg)[-n_top:]
    low = np.flatnonzero(deg <= 1)[:32]
    rnd = rng.choice(w.N, size=min(n_random, w.N), replace=False)
    return np.unique(np.concatenate([top, low, rnd]))
