"""The bench's algorithmic byte and FLOP models (CPU): the formulas written
out independently on the workloads' exact sizes, and their relations."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

# R-MAT as generated (2^20 nodes, 17,133,085 entries after dedup and
# self-loops), 4 x 32 bf16: a node row is 256 bytes
RMAT = dict(N=1 << 20, nnz=17_133_085, H=4, D=32, esize=2)
# Erdos-Renyi: 100,000 nodes, 1.6 M symmetric entries + 100,000 self-loops, 8 x 64 bf16
ER = dict(N=100_000, nnz=1_700_000, H=8, D=64, esize=2)


def test_compulsory_and_unique_bytes_rmat():
    N, nnz, row = RMAT["N"], RMAT["nnz"], 4 * 32 * 2
    # indptr + indices + Q and out once per node + K and V once per entry
    want_c = 4 * (N + 1) + 4 * nnz + 2 * N * row + 2 * nnz * row
    # each array once: indptr, indices, Q, K, V, out
    want_u = 4 * (N + 1) + 4 * nnz + 4 * N * row
    assert bench.compulsory_bytes(**RMAT) == want_c == 9_381_737_080
    assert bench.unique_bytes(**RMAT) == want_u == 1_146_468_472


def test_erdos_renyi_bytes():
    assert bench.compulsory_bytes(**ER) == 4 * 100_001 + 4 * 1_700_000 + 2 * 100_000 * 1024 + 2 * 1_700_000 * 1024
    assert bench.unique_bytes(**ER) == 4 * 100_001 + 4 * 1_700_000 + 4 * 100_000 * 1024


@pytest.mark.parametrize("w", [RMAT, ER])
def test_path_bytes_add_what_each_variant_moves(w):
    N, nnz, H, D, es = w["N"], w["nnz"], w["H"], w["D"], w["esize"]
    c0, u0 = bench.path_bytes("fwd", N, nnz, H, D, es)
    assert (c0, u0) == (bench.compulsory_bytes(N, nnz, H, D, es), bench.unique_bytes(N, nnz, H, D, es))
    nhd = N * H * D
    # an fp32 bias [nnz, H]; fp32 adjacency values [nnz]; logits and probs written
    assert bench.path_bytes("bias", N, nnz, H, D, es) == (c0 + 4 * nnz * H, u0 + 4 * nnz * H)
    assert bench.path_bytes("weighted", N, nnz, H, D, es) == (c0 + 4 * nnz, u0 + 4 * nnz)
    assert bench.path_bytes("probs", N, nnz, H, D, es) == (c0 + 8 * nnz * H, u0 + 8 * nnz * H)
    # the backward: dO read, three fp32 gradients written
    assert bench.path_bytes("bwd", N, nnz, H, D, es) == (c0 + nhd * es + 12 * nhd, u0 + nhd * es + 12 * nhd)
    # given the saved forward: its fp32 output and statistics read instead of
    # the output written; the training step adds the forward that writes them
    saved = bench.path_bytes("bwd_saved", N, nnz, H, D, es)
    assert saved == (c0 - nhd * es + 4 * nhd + 4 * N * H + nhd * es + 12 * nhd,
                     u0 - nhd * es + 4 * nhd + 4 * N * H + nhd * es + 12 * nhd)
    train = bench.path_bytes("train", N, nnz, H, D, es)
    fwd_stats = (c0 - nhd * es + 4 * nhd + 4 * N * H, u0 - nhd * es + 4 * nhd + 4 * N * H)
    assert train == (fwd_stats[0] + saved[0], fwd_stats[1] + saved[1])


def test_dense_flops():
    # 4 n^2 D per block and head: 64 blocks of 512, 8 heads, D = 64
    assert bench.dense_flops(64, 512, 8, 64) == 4 * 512 * 512 * 64 * 64 * 8 == 34_359_738_368


def test_proj_flops():
    # q/k/v map (N x F by F x 3F) and output map (N x F by F x F), 2 flops a multiply-add
    N, H, D = 1 << 20, 4, 32
    F = H * D
    assert bench.proj_flops(N, H, D) == 2 * N * F * 3 * F + 2 * N * F * F


def test_job_throughput_single_rank():
    # one rank: units over its own time
    value, worst, total = bench.job_throughput(68_532_340.0 * 20, 17.9)
    assert worst == pytest.approx(17.9) and total == pytest.approx(68_532_340.0 * 20)
    assert value == pytest.approx(68_532_340.0 * 20 / 17.9e-3)
