// bwd.cuh -- backward pass launchers (bwd.cu); the entry point is in api.cu.
#pragma once

#include "common.cuh"

namespace gt {

constexpr int kBwdMaxHeads = 128;

// One warp per destination row, two walks over its entries (any shape with
// H <= kBwdMaxHeads).
gtattn_status launch_bwd_rows(const int* indptr, const int* indices, const void* Q, const void* K, const void* V,
                              const void* dO, float* dQ, float* dK, float* dV, int N, int H, int D, float scale,
                              gtattn_dtype dtype, cudaStream_t s);

// Whether the two-pass backward handles the shape: H*D = 32 E with E in
// {4, 8, 16, 32}, D a multiple of E with D/E a power of two, every pointer
// 16-byte aligned.
bool bwd_tasks_supported(int H, int D, gtattn_dtype dtype, const void* const* ptrs, int n_ptrs);

// Tiles of the scan that lays out the source-major pattern (the size of its
// tile-sum array).
int64_t bwd_scan_tiles(int64_t N);

// Source-major copy of the pattern on stream s: colptr [N+1] over sources and
// rowid [nnz], the destination row of each entry, ascending within a source
// (so the copy, and every sum over it, is the same on every run), and the
// binning of the sources into C (split threshold long_min, C.chunk_edges).
// cursor [N], tsum [bwd_scan_tiles(N)] and tmp [nnz] are scratch; L are the
// destination binning's task lists.
gtattn_status build_csc(const int* indptr, const int* indices, const TaskLists& L, int N, int64_t nnz,
                        int* colptr, int* cursor, int* tsum, int* rowid, int* tmp, const TaskLists& C,
                        int long_min, cudaStream_t s);

// The two passes, given the forward's fp32 output O and row log-sum-exp
// (log2 units): dQ by destination row over `rows`, dK and dV by source over
// `cols` (the binning of colptr).  LD [N*H] is scratch, (L_i, Dlt_i) per row
// and head.  Chunks of split rows and sources store partial sums (part_dq
// [rows' chunks * H*D], part_dk and part_dv [cols' chunks * H*D], scratch),
// which a last step adds in chunk order.  Every row of dQ, dK and dV is
// written, and the result does not depend on the order the GPU runs the
// work in.
gtattn_status launch_bwd_passes(const int* indptr, const int* indices, const TaskLists& rows, const int* colptr,
                                const int* rowid, const TaskLists& cols, const void* Q, const void* K, const void* V,
                                const void* dO, const float* O, const float* lse, float2* LD, float* dQ, float* dK,
                                float* dV, float* part_dq, float* part_dk, float* part_dv, int N, int64_t nnz, int H,
                                int D, float scale, gtattn_dtype dtype, cudaStream_t s);

}  // namespace gt
