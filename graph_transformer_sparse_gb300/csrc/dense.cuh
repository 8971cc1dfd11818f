// dense.cuh -- dense-block attention (complete blocks) on the tensor cores.
#pragma once

#include "common.cuh"

namespace gt {

// True when launch_dense handles this shape: bf16 inputs (bf16 or fp32 out),
// D of 32, 64 or 128, 16-byte aligned pointers.
bool dense_supported(int H, int D, gtattn_dtype dt, const void* Q, const void* K, const void* V,
                     const void* out);

// out = softmax(scale * Q K^T) V per head over complete blocks on a
// persistent grid (one CTA per SM).  tiles: device array of work items
// (first row of the block, block size, first row of the item's query rows,
// number of 128-row query tiles (1 or 2)); tiles1: the same blocks as items
// of one query tile each (taken for D = 128); blocks of at least 128 rows, a
// ragged last tile masked.
// A bounded device wait that times out ORs an error code into *err and the
// CTA drains what it issued and returns.  wait_cycles bounds each wait for
// data from another warp (SM clock cycles; <= 0: about one second); the
// drains keep their own bound of about half a second.  test_stall != 0
// (tests only): the softmax warps first wait on a barrier nothing completes,
// so every CTA takes the timeout path.
gtattn_status launch_dense(const int4* tiles, const int4* tiles1, int n_tiles, int n_tiles1, int64_t N,
                           const void* Q, const void* K, const void* V, void* out, int H, int D, float scale,
                           gtattn_dtype dt, int* err, long long wait_cycles, int test_stall, cudaStream_t s);

}  // namespace gt
