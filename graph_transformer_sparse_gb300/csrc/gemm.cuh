// gemm.cuh -- the linear maps around the attention (gemm.cu): Y = A B^T + b
// with A [M, K] and B [Nn, K] row-major (an nn.Linear weight), used by the
// projected attention block.
#pragma once

#include "common.cuh"

namespace gt {

// Where column c of Y goes: output matrix c / cols_per_split (matrices
// split_stride elements apart), column c % cols_per_split of it, rows ld
// elements apart.  One matrix: cols_per_split = Nn, split_stride = 0.
struct GemmOut {
    void* base;
    int64_t split_stride;
    int cols_per_split;
    int64_t ld;
};

// True when the tensor-core kernel takes the problem: bf16 A and B, K a
// multiple of 8 (16-byte rows for TMA), 16-byte aligned A, B and output,
// output chunks of 16 bytes inside one output matrix.
bool gemm_tc_supported(const void* A, const void* B, int K, const GemmOut& o, bool out_f32);

// tcgen05 kernel: bf16 A, B; fp32 accumulation in tensor memory; bias fp32
// [Nn] or null; output bf16 (round to nearest even) or fp32.
gtattn_status launch_gemm_tc(const void* A, const void* B, const float* bias, int64_t M, int Nn, int K,
                             const GemmOut& o, bool out_f32, cudaStream_t s);

// CUDA-core kernel for any shape: A, B fp32 or bf16 (same type), fp32
// accumulation, output of the type out_f32 names.
gtattn_status launch_gemm_simt(const void* A, const void* B, const float* bias, int64_t M, int Nn, int K,
                               bool in_bf16, const GemmOut& o, bool out_f32, cudaStream_t s);

// Head-inner to head-major feature order (f = d*H + h -> h*D + d):
// rows of W [groups * H*D, K] (and of bias [groups * H*D], if any), or
// columns of W [rows, H*D].  esz: element size of W (2 or 4).
gtattn_status launch_permute_rows(const void* W, void* Wp, const float* b, float* bp, int groups, int H, int D,
                                  int K, int esz, cudaStream_t s);
gtattn_status launch_permute_cols(const void* W, void* Wp, int rows, int H, int D, int esz, cudaStream_t s);

}  // namespace gt
