// dense.cuh -- dense-block attention (complete blocks) on the tensor cores.
#pragma once

#include "common.cuh"

namespace gt {

// True when launch_dense handles this shape: bf16, D == 64, 16-byte aligned.
bool dense_supported(int H, int D, gtattn_dtype dt, const void* Q, const void* K, const void* V,
                     const void* out);

// out_b = softmax(scale * Q_b K_b^T) V_b per head for each block b =
// (first row, size) in `blocks` (device array of n_blocks entries).
gtattn_status launch_dense(const int2* blocks, int n_blocks, const void* Q, const void* K,
                           const void* V, void* out, int H, int D, float scale, cudaStream_t s);

}  // namespace gt
