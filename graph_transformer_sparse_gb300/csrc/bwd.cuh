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

// Whether the task-parallel backward handles the shape: H*D = 32 E with E in
// {4, 8, 16, 32}, D a multiple of E with D/E a power of two, every pointer
// 16-byte aligned.
bool bwd_tasks_supported(int H, int D, gtattn_dtype dtype, const void* const* ptrs, int n_ptrs);

// Task-parallel backward over the binning's task lists, given the forward's
// fp32 output O and row log-sum-exp (log2 units).  dQ, dK, dV are added to
// (zero them first).
gtattn_status launch_bwd_tasks(const int* indptr, const int* indices, const TaskLists& L, const void* Q,
                               const void* K, const void* V, const void* dO, const float* O, const float* lse,
                               float* dQ, float* dK, float* dV, int N, int H, int D, float scale, gtattn_dtype dtype,
                               cudaStream_t s);

}  // namespace gt
