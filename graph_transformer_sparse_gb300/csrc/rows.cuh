// rows.cuh -- launch interface of the row kernels (fused, SpMM, SDDMM modes),
// the split-row combine and the unfused edge softmax.
#pragma once

#include "common.cuh"

namespace gt {

struct RowParams {
    const int* indptr;
    const int* indices;
    const void* Q;
    const void* K;
    const void* V;
    void* out;
    const float* probs;     // SpMM mode: fp32 [nnz, H]
    const float* bias;      // fused / SDDMM modes: fp32 [nnz, H] added to the logits, or null
    const float* values;    // fused / SDDMM modes: fp32 [nnz] multiplying the dot products, or null
    int ndh;                // 1: node rows are [D, H] (head innermost; generic kernel only)
    float* lse;             // fused mode: fp32 [N, H] row log-sum-exp (log2 units) written for every
                            // row (-inf for a row without entries), or null
    float* logits;          // SDDMM mode: fp32 [nnz, H]
    float qscale;           // fused: scale*log2(e); SDDMM: scale
    int N, H, D, HD;
    int groups;             // combine: head groups (1 but for one launch after several groups' rows);
    int64_t gstep_m, gstep_acc;   // group gi's partials at m/s + gi*gstep_m, acc + gi*gstep_acc
    int gstep_out;          // and its output columns at out + gi*gstep_out (elements)
    int ld;                 // row stride of Q, K, V and out in elements (HD, or more for a head group
                            // of wider rows: vector kernel, combine); an int, so that index * ld is
                            // one widening multiply
    int G, lph;             // vector kernel: lanes per feature row, lanes per head
    TaskLists lists;
    Partials part;
    int task_bound;         // upper bound on the warp tasks of the lists (<= 0: unknown)
    // Small graphs in one launch (launch_rows_small): `lists` is unused;
    // every block bins the rows itself into shared memory (rows of more
    // than long_min entries split into lists.chunk_edges-entry chunks, at
    // most small_max_chunks chunks and small_max_long split rows), and when
    // a row is split the grid -- launched cooperatively -- synchronises and
    // the split rows are combined in the same launch.
    int long_min;
    int small_max_chunks, small_max_long;
    int small_no_split;     // nnz <= long_min: no row is split (the blocks skip the check)
};

// Bounds of the one-launch path: rows, entries, and the shared-memory lists
// (chunks and split rows) each block builds.
constexpr int kSmallMaxRows = 4096;
constexpr int kSmallMaxNnz = 65536;
constexpr int kSmallMaxChunks = 512;
constexpr int kSmallMaxLong = 256;

// Upper bound on the warp tasks binning makes: a task is one row or more
// (rows of up to long_min entries), or one chunk of a split row (at most
// nnz / chunk + 1 per row).
inline int row_task_bound(int64_t N, int64_t nnz, int chunk) {
    const int64_t b = N + nnz / (chunk > 0 ? chunk : 1) + 1;
    return b > 0x7fffffff ? 0x7fffffff : static_cast<int>(b);
}

enum class RowKernel { kVector, kGeneric, kNarrow };

struct RowChoice {
    RowKernel kind;
    int vpl;    // 16-byte vectors per lane (vector kernel); narrow kernel: 1 = features read in pairs
    int G, lph;
};

// Widest head the narrow-head kernel takes (one lane per head).
constexpr int kNarrowMaxD = 16;

// Picks the row kernel for a shape; `force` is a gtattn_kernel value.
// Returns false when no kernel supports the shape (or the forced one does not).
bool choose_row_kernel(int H, int D, gtattn_dtype dt, const void* Q, const void* K, const void* V,
                       const void* out, int force, RowChoice* c);

// Launches the persistent row kernel over every task of `p.lists`.
gtattn_status launch_rows(Mode mode, gtattn_dtype dt, const RowChoice& c, const RowParams& p,
                          cudaStream_t s);

// The fused forward in one launch for a small graph (p.small set by the
// caller; N <= kSmallMaxRows, nnz <= kSmallMaxNnz, worst-case chunk and
// split-row counts within the shared-memory lists).
gtattn_status launch_rows_small(gtattn_dtype dt, const RowChoice& c, const RowParams& p, cudaStream_t s);

// Combines split-row partials into `out` for every split row (mode kFused or kSpmm).
gtattn_status launch_combine(Mode mode, gtattn_dtype dt, const RowParams& p, cudaStream_t s);

// Unfused edge softmax: probs[e,h] from logits[e,h] over each row's entries.
gtattn_status launch_edge_softmax(const int* indptr, int N, int H, const TaskLists& L, const Partials& part,
                                  const float* logits, float* probs, cudaStream_t s);

}  // namespace gt
