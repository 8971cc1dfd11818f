"""Seeded synthetic inputs for sparse multi-head attention.

This module only *generates data*: graphs in CSR-by-destination form and
random Q/K/V feature tensors.  It holds none of the attention arithmetic, so
both the fp64 oracle (``oracle/``) and the CUDA path use it without sharing
any of the method's computation.

Every generator is deterministic for a given seed (numpy ``PCG64``).  The five
named workloads follow the shapes and structure of the pages' workloads:

* ``tiny_random``  -- the ``rand_graph(30, 100)`` smoke graph of "Efficient
  Sparse Transformer implementation with DGL's builtin operators"
  (``__main__`` of dgl-transformer.py): 30 nodes, 100 distinct directed
  edges, 8 heads of width 64, fp32.
* ``molecules``    -- batched molecule-like graphs standing in for the
  ogbg-molhiv batches of "Graph Transformer in a Nutshell" (hidden size 80,
  8 heads, so head width 10), fp32.
* ``erdos_renyi``  -- N=100,000, 800,000 undirected pairs symmetrised, plus a
  self-loop per node; 8x64 bf16.
* ``rmat``         -- R-MAT with 2^20 nodes and 2^24 draws (a,b,c,d =
  .57,.19,.19,.05), deduplicated, self-loops replaced by one per node;
  4x32 bf16.  Heavily skewed in-degree.
* ``dense_blocks`` -- 64 disjoint complete graphs of 512 nodes (self-loops
  included); 8x64 bf16, features scaled by 0.5.

bf16 workloads draw fp32 normals and round them to bf16 with round-to-
nearest-even; the returned ``float32`` arrays then hold exactly the bf16
values, and ``*_bits`` hold the raw bf16 bit patterns (``uint16``).
"""
from __future__ import annotations

import math
import sys
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "bf16_round", "bf16_bits_to_f32", "csr_by_destination",
    "tiny_random_edges", "molecule_edges", "erdos_renyi_edges", "rmat_edges",
    "dense_block_csr", "make_features", "make_workload", "WORKLOADS",
    "small_workload", "random_csr",
]


# ---------------------------------------------------------------------------
# bf16 helpers (data preparation only)
# ---------------------------------------------------------------------------
def bf16_round(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Round float32 values to bf16, round-to-nearest-even.

    Returns ``(values_f32, bits_u16)``: the rounded values widened back to
    float32 (exact) and the bf16 bit patterns.  NaN/Inf are not produced by
    the generators and are not handled specially.
    """
    assert sys.byteorder == "little"
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    t = u >> np.uint32(16)
    t &= np.uint32(1)                    # lsb of the kept half: ties to even
    t += np.uint32(0x7FFF)
    t += u                               # wraps only for NaN payloads, never drawn
    t &= np.uint32(0xFFFF0000)
    vals = t.view(np.float32).reshape(x.shape)
    bits = np.ascontiguousarray(t.view(np.uint16).reshape(-1)[1::2]).reshape(x.shape)
    return vals, bits


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    assert sys.byteorder == "little"
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    w = np.zeros(b.size, dtype=np.uint32)
    w.view(np.uint16)[1::2] = b.reshape(-1)
    return w.view(np.float32).reshape(b.shape)


# ---------------------------------------------------------------------------
# CSR construction (data structure only)
# ---------------------------------------------------------------------------
def csr_by_destination(src: np.ndarray, dst: np.ndarray, n: int):
    """COO edge list (src -> dst) to CSR keyed by destination.

    Row ``i`` lists the sources ``j`` of the edges ``j -> i``, sorted by
    ``j``; duplicates are kept as separate entries.  Returns int32
    ``indptr[n+1]`` and ``indices[nnz]``.
    """
    src = np.asarray(src, dtype=np.int64)
    dst = np.asarray(dst, dtype=np.int64)
    if src.shape != dst.shape:
        raise ValueError("src and dst differ in length")
    if len(src) and (min(src.min(), dst.min()) < 0 or max(src.max(), dst.max()) >= n):
        raise ValueError("node id out of range")
    key = dst * np.int64(n) + src
    order = np.argsort(key, kind="stable")
    indices = src[order].astype(np.int32)
    counts = np.bincount(dst, minlength=n)
    indptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(counts, out=indptr[1:])
    if indptr[-1] >= 2**31:
        raise ValueError("nnz exceeds int32")
    return indptr.astype(np.int32), indices


def _unique_sorted(keys: np.ndarray) -> np.ndarray:
    keys = np.sort(keys)
    if len(keys) == 0:
        return keys
    keep = np.empty(len(keys), dtype=bool)
    keep[0] = True
    np.not_equal(keys[1:], keys[:-1], out=keep[1:])
    return keys[keep]


# ---------------------------------------------------------------------------
# Graph generators (return COO src, dst and n)
# ---------------------------------------------------------------------------
def tiny_random_edges(rng: np.random.Generator, n: int = 30, e: int = 100):
    """``e`` distinct directed pairs drawn uniformly without replacement from
    the ``n*n`` ordered pairs (self-loops allowed)."""
    pick = rng.choice(n * n, size=e, replace=False)
    return pick // n, pick % n, n


def molecule_edges(rng: np.random.Generator, n_graphs: int = 128,
                   n_min: int = 10, n_max: int = 50, max_deg: int = 4):
    """Block-diagonal union of molecule-like graphs.

    Each graph: ``n ~ U{n_min..n_max}`` atoms; 1-3 rings of 5 or 6 atoms laid
    out as cycles on consecutive ids, linked into a chain; the remaining atoms
    attach either to the previous atom (backbone) or to a random earlier atom
    with degree below ``max_deg`` (branch).  Edges are made symmetric and one
    self-loop is added per atom.
    """
    src, dst = [], []
    base = 0
    for _ in range(n_graphs):
        n = int(rng.integers(n_min, n_max + 1))
        deg = np.zeros(n, dtype=np.int64)
        und = []

        def link(a, b):
            und.append((a, b))
            deg[a] += 1
            deg[b] += 1

        pos = 0
        for _r in range(int(rng.integers(1, 4))):
            size = int(rng.integers(5, 7))
            if pos + size > n:
                break
            for k in range(size):
                link(pos + k, pos + (k + 1) % size)
            if pos > 0:
                link(pos - 1, pos)
            pos += size
        for v in range(max(pos, 1), n):
            prev = v - 1
            if rng.random() < 0.5 and deg[prev] < max_deg:
                u = prev
            else:
                cand = np.flatnonzero(deg[:v] < max_deg)
                u = int(cand[rng.integers(0, len(cand))]) if len(cand) else prev
            link(u, v)
        for a, b in und:
            src += [base + a, base + b]
            dst += [base + b, base + a]
        src += list(range(base, base + n))
        dst += list(range(base, base + n))
        base += n
    return np.array(src, dtype=np.int64), np.array(dst, dtype=np.int64), base


def erdos_renyi_edges(rng: np.random.Generator, n: int = 100_000, pairs: int = 800_000,
                      self_loops: bool = True):
    """``pairs`` distinct unordered pairs {u != v} drawn uniformly (duplicates
    redrawn), made symmetric, plus one self-loop per node."""
    have = np.empty(0, dtype=np.int64)
    while len(have) < pairs:
        need = pairs - len(have)
        u = rng.integers(0, n, size=int(need * 1.1) + 16)
        v = rng.integers(0, n, size=len(u))
        ok = u != v
        lo = np.minimum(u[ok], v[ok])
        hi = np.maximum(u[ok], v[ok])
        have = _unique_sorted(np.concatenate([have, lo * np.int64(n) + hi]))
        if len(have) > pairs:
            have = have[rng.permutation(len(have))[:pairs]]
    lo, hi = have // n, have % n
    src = np.concatenate([lo, hi])
    dst = np.concatenate([hi, lo])
    if self_loops:
        loops = np.arange(n, dtype=np.int64)
        src = np.concatenate([src, loops])
        dst = np.concatenate([dst, loops])
    return src, dst, n


def rmat_edges(rng: np.random.Generator, scale: int = 20, draws: int = 1 << 24,
               a: float = 0.57, b: float = 0.19, c: float = 0.19):
    """R-MAT: each of ``draws`` edges picks one quadrant per bit level with
    probabilities (a, b, c, 1-a-b-c); u takes the row bit (c or d), v the
    column bit (b or d).  Edge u -> v.  Duplicates and u == v are dropped,
    then one self-loop per node is added.  Returns edges already unique."""
    n = 1 << scale
    u = np.zeros(draws, dtype=np.int64)
    v = np.zeros(draws, dtype=np.int64)
    t_ab, t_abc = a + b, a + b + c
    for lvl in range(scale):
        r = rng.random(draws, dtype=np.float32)
        ubit = r >= t_ab
        vbit = ((r >= a) & (r < t_ab)) | (r >= t_abc)
        sh = scale - 1 - lvl
        u |= ubit.astype(np.int64) << sh
        v |= vbit.astype(np.int64) << sh
    keep = u != v
    loops = np.arange(n, dtype=np.int64)
    key = np.concatenate([v[keep] * np.int64(n) + u[keep], loops * np.int64(n) + loops])
    key = _unique_sorted(key)            # sorted by (dst, src)
    return key % n, key // n, n


def dense_block_csr(n_blocks: int = 64, block: int = 512):
    """CSR of ``n_blocks`` disjoint complete graphs (every ordered pair in a
    block, self-loops included), rows sorted."""
    n = n_blocks * block
    indptr = (np.arange(n + 1, dtype=np.int64) * block)
    if indptr[-1] >= 2**31:
        raise ValueError("nnz exceeds int32")
    row = np.repeat(np.arange(n, dtype=np.int64), block)
    k = np.tile(np.arange(block, dtype=np.int64), n)
    indices = (row // block) * block + k
    return indptr.astype(np.int32), indices.astype(np.int32), n


# ---------------------------------------------------------------------------
# Features
# ---------------------------------------------------------------------------
def make_features(rng: np.random.Generator, n: int, h: int, d: int, dtype: str,
                  std: float = 1.0):
    """Q, K, V ~ std * N(0, 1), shape [n, h, d].  For ``bf16`` the values are
    rounded to bf16 (RNE).  Returns dict with float32 arrays ``Q, K, V`` and,
    for bf16, ``Q_bits, K_bits, V_bits`` (uint16)."""
    out = {}
    for name in ("Q", "K", "V"):
        x = rng.standard_normal((n, h, d), dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if dtype == "bf16":
            vals, bits = bf16_round(x)
            out[name] = vals.reshape(n, h, d)
            out[name + "_bits"] = bits.reshape(n, h, d)
        elif dtype == "f32":
            out[name] = x
        else:
            raise ValueError(dtype)
    return out


@dataclass
class Workload:
    name: str
    N: int
    H: int
    D: int
    dtype: str                 # "f32" or "bf16"
    indptr: np.ndarray         # int32 [N+1]
    indices: np.ndarray        # int32 [nnz]
    Q: np.ndarray              # float32 [N,H,D] (bf16-exact when dtype == "bf16")
    K: np.ndarray
    V: np.ndarray
    scale: float               # float32 value 1/sqrt(D)
    bits: dict = field(default_factory=dict)   # bf16 bit patterns
    desc: str = ""

    @property
    def nnz(self) -> int:
        return int(self.indptr[-1])

    def features(self, name: str) -> np.ndarray:
        """The array handed to the device: float32 or bf16 bits (uint16)."""
        return self.bits[name] if self.dtype == "bf16" else getattr(self, name)


WORKLOADS = {
    "tiny_random": dict(seed=1, H=8, D=64, dtype="f32",
                        desc="30 nodes, 100 distinct directed edges, 8x64 fp32"),
    "molecules": dict(seed=2, H=8, D=10, dtype="f32",
                      desc="128 molecule-like graphs of 10-50 atoms, 8x10 fp32"),
    "erdos_renyi": dict(seed=3, H=8, D=64, dtype="bf16",
                        desc="Erdos-Renyi N=100000, 1.6M symmetric edges + self-loops, 8x64 bf16"),
    "rmat": dict(seed=4, H=4, D=32, dtype="bf16",
                 desc="R-MAT 2^20 nodes, 2^24 draws (.57/.19/.19/.05), dedup + self-loops, 4x32 bf16"),
    "dense_blocks": dict(seed=5, H=8, D=64, dtype="bf16", std=0.5,
                         desc="64 disjoint complete graphs of 512 nodes, 8x64 bf16, 0.5*N(0,1)"),
}


def _scale_for(d: int) -> float:
    return float(np.float32(1.0 / math.sqrt(d)))


def make_workload(name: str, **over) -> Workload:
    """Build one of the five named workloads (see the module docstring).

    Keyword overrides change graph sizes for reduced-size parity cases:
    ``tiny_random(n, e)``, ``molecules(n_graphs)``, ``erdos_renyi(n, pairs)``,
    ``rmat(scale, draws)``, ``dense_blocks(n_blocks, block)``; ``H, D, dtype,
    seed`` override the feature shape.
    """
    spec = dict(WORKLOADS[name])
    spec.update({k: over.pop(k) for k in list(over) if k in ("seed", "H", "D", "dtype", "std")})
    rng = np.random.default_rng(spec["seed"])
    if name == "tiny_random":
        src, dst, n = tiny_random_edges(rng, **over)
        indptr, indices = csr_by_destination(src, dst, n)
    elif name == "molecules":
        src, dst, n = molecule_edges(rng, **over)
        indptr, indices = csr_by_destination(src, dst, n)
    elif name == "erdos_renyi":
        src, dst, n = erdos_renyi_edges(rng, **over)
        indptr, indices = csr_by_destination(src, dst, n)
    elif name == "rmat":
        src, dst, n = rmat_edges(rng, **over)
        counts = np.bincount(dst, minlength=n)
        indptr = np.zeros(n + 1, dtype=np.int64)
        np.cumsum(counts, out=indptr[1:])
        indptr, indices = indptr.astype(np.int32), src.astype(np.int32)
    elif name == "dense_blocks":
        indptr, indices, n = dense_block_csr(**over)
    else:
        raise KeyError(name)
    feats = make_features(rng, n, spec["H"], spec["D"], spec["dtype"], spec.get("std", 1.0))
    bits = {k[0]: v for k, v in feats.items() if k.endswith("_bits")}
    return Workload(name=name, N=n, H=spec["H"], D=spec["D"], dtype=spec["dtype"],
                    indptr=indptr, indices=indices, Q=feats["Q"], K=feats["K"], V=feats["V"],
                    scale=_scale_for(spec["D"]), bits=bits, desc=spec["desc"])


def small_workload(name: str) -> Workload:
    """Reduced-size versions of the five workloads: same structure and
    feature shapes, sizes the fp64 oracle finishes in seconds."""
    small = {
        "tiny_random": {},
        "molecules": {},
        "erdos_renyi": dict(n=6000, pairs=48_000),
        "rmat": dict(scale=13, draws=1 << 17),
        "dense_blocks": dict(n_blocks=3, block=256),
    }
    return make_workload(name, **small[name])


def random_csr(rng: np.random.Generator, n: int, nnz: int, self_loops: bool = False,
               duplicates: bool = False, degree_skew: float = 0.0):
    """A random CSR-by-destination graph for edge cases: ``nnz`` edges with
    destinations drawn uniformly (or Zipf-like when ``degree_skew`` > 0),
    sources uniform; duplicates are removed unless ``duplicates``."""
    if degree_skew > 0:
        w = 1.0 / np.arange(1, n + 1) ** degree_skew
        dst = rng.choice(n, size=nnz, p=w / w.sum())
    else:
        dst = rng.integers(0, n, size=nnz)
    src = rng.integers(0, n, size=nnz)
    if not self_loops:
        ok = src != dst
        src, dst = src[ok], dst[ok]
    if not duplicates:
        key = _unique_sorted(dst * np.int64(n) + src)
        src, dst = key % n, key // n
    return csr_by_destination(src, dst, n)
