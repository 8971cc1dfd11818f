// common.cuh -- internal definitions shared by the library's CUDA sources.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "gtattn.h"

namespace gt {

// ---------------------------------------------------------------------------
// Degree buckets.  Rows with degree 0..32 get one bucket per degree; larger
// degrees fall into roughly x1.5 steps.  Bucket ids grow with degree; row
// lists are laid out from the highest bucket down so heavy rows start first.
// ---------------------------------------------------------------------------
constexpr int kExactBuckets = 33;
constexpr int kLogBuckets = 15;
constexpr int kNumBuckets = kExactBuckets + kLogBuckets;   // 48
constexpr int kMaxHD = 1024;
constexpr int kDenseTile = 128;   // dense blocks: tiles of this many rows (blocks of at least one)

// upper bounds (inclusive) of the log buckets
__host__ __device__ inline int log_bucket_hi(int k) {
    switch (k) {
        case 0: return 48;    case 1: return 64;    case 2: return 96;    case 3: return 128;
        case 4: return 192;   case 5: return 256;   case 6: return 384;   case 7: return 512;
        case 8: return 768;   case 9: return 1024;  case 10: return 1536; case 11: return 2048;
        case 12: return 3072; case 13: return 4096; default: return 0x7fffffff;
    }
}

__host__ __device__ inline int bucket_of(int deg) {
    if (deg < kExactBuckets) return deg;
    int k = 0;
    while (k < kLogBuckets - 1 && deg > log_bucket_hi(k)) ++k;
    return kExactBuckets + k;
}

__host__ __device__ inline int bucket_lo(int b) {
    if (b < kExactBuckets) return b;
    return b == kExactBuckets ? kExactBuckets : log_bucket_hi(b - kExactBuckets - 1) + 1;
}

// Device-side plan header (int32 words).
struct HdrLayout {
    static constexpr int kLong = 0;          // rows split into chunks
    static constexpr int kChunks = 1;        // chunks over split rows
    static constexpr int kDenseRows = 2;     // rows in the dense segment
    static constexpr int kDenseBlocks = 3;   // complete blocks found
    static constexpr int kMaxDeg = 4;
    static constexpr int kCount = 8;                           // [NB] rows per bucket
    static constexpr int kOffset = kCount + kNumBuckets;       // [NB] start in row list
    static constexpr int kCursor = kOffset + kNumBuckets;      // [NB] scatter cursors
    static constexpr int kCurLong = kCursor + kNumBuckets;     // cursor: long rows
    static constexpr int kCurChunk = kCurLong + 1;             // cursor: chunks
    static constexpr int kCurDense = kCurChunk + 1;            // cursor: dense rows
    static constexpr int kDenseSeg = kCurDense + 1;            // start of dense segment in row list
    static constexpr int kErr = kDenseSeg + 1;                 // device-side error bits (bounded waits)
    static constexpr int kBig = kDenseSeg + 2;                 // split rows of more than kBigChunks chunks
    static constexpr int kCurBig = kDenseSeg + 3;              // cursor: those rows
    static constexpr int kWords = kDenseSeg + 8;
};
// Split rows of more than this many chunks are listed first in the split-row
// list (combined a block per row, its threads over the chunks); the others a
// warp per row, whose lanes walk the chunks one after another for each 32
// output elements (R-MAT, 1024-entry chunks: 32 chunks a warp left the
// combine 26 us long on a few such rows; 8 a warp cut it to the launch).
constexpr int kBigChunks = 8;

// Work lists consumed by the row kernels.
struct TaskLists {
    const int* hdr;          // HdrLayout words (device)
    const int* rows;         // bucketed row list, then the dense segment
    const int2* chunks;      // (row, first entry) per chunk
    const int2* longs;       // (row, first chunk) per split row
    int chunk_edges;
    int include_dense;       // 1: the dense segment is processed by the row kernels
};

// Split-row partial results: per chunk c, m[c*H+h], s[c*H+h] (log2 domain
// running max and sum) and acc[c*HD + t].
struct Partials {
    float* m;
    float* s;
    float* acc;
};

enum Mode { kFused = 0, kSpmm = 1, kSddmm = 2 };

// ---------------------------------------------------------------------------
// small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {   // 2^x, PTX ex2.approx (ftz)
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float load_elem(const float* p, int64_t i) { return __ldg(p + i); }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_elem(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, int64_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

constexpr float kLog2e = 1.4426950408889634f;

// c + a.lo*b.lo + a.hi*b.hi for two packed bf16 pairs: products of bf16
// values are exact in fp32, the sums are fp32 (mixed-precision FMA).
__device__ __forceinline__ float dot2_bf16(uint32_t a, uint32_t b, float c) {
    float r;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %3;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "=f"(r)
        : "r"(a), "r"(b), "f"(c));
    return r;
}
// (a0, a1) += w * (v.lo, v.hi) for a packed bf16 pair v: one f32x2 FMA.
__device__ __forceinline__ void axpy2_bf16(float& a0, float& a1, float w, uint32_t v) {
    asm("{\n\t.reg .b64 rv, rw, ra;\n\t.reg .b32 lo, hi;\n\t"
        "shl.b32 lo, %3, 16;\n\tand.b32 hi, %3, 0xffff0000;\n\t"
        "mov.b64 rv, {lo, hi};\n\tmov.b64 rw, {%2, %2};\n\tmov.b64 ra, {%0, %1};\n\t"
        "fma.rn.f32x2 ra, rv, rw, ra;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(w), "r"(v));
}
// (a0, a1) += (x0, x1) * (y0, y1): one f32x2 FMA.
__device__ __forceinline__ void fma2(float& a0, float& a1, float x0, float x1, float y0, float y1) {
    asm("{\n\t.reg .b64 rx, ry, ra;\n\t"
        "mov.b64 rx, {%2, %3};\n\tmov.b64 ry, {%4, %5};\n\tmov.b64 ra, {%0, %1};\n\t"
        "fma.rn.f32x2 ra, rx, ry, ra;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}

}  // namespace gt

// ---------------------------------------------------------------------------
// host-side helpers (defined in api.cu)
// ---------------------------------------------------------------------------
namespace gt {
gtattn_status cuda_status(cudaError_t e);
void set_last_error(const char* msg);
int num_sms();
cudaMemPool_t pool();
gtattn_status pool_alloc(void** p, size_t bytes, cudaStream_t s);
void pool_free(void* p, cudaStream_t s);
// Host-side argument checks of the forward entry points (null pointers,
// sizes, dtype, alignment): GTATTN_OK or GTATTN_ERR_INVALID_ARG.
gtattn_status check_fwd(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                        const void* V, const void* out, int64_t N, int64_t nnz, int H, int D, gtattn_dtype dtype);
// The checking build (GTATTN_DEBUG): validates a device CSR (offsets from 0
// to nnz, non-decreasing; indices in [0, N)) before the call's first other
// kernel, synchronously, and returns GTATTN_ERR_BAD_CSR if it fails; one
// flag in device memory, so concurrent calls race on it.  Defined in plan.cu.
gtattn_status debug_csr_check(const int32_t* indptr, const int32_t* indices, int64_t N, int64_t nnz,
                              cudaStream_t s);
// gtattn_fwd without that check, for calls on views of a checked CSR (the
// host-buffer path's row chunks); n_src: the rows of K and V (the whole
// graph's), which the kernel choices depend on as in the whole call.
// Defined in api.cu.
gtattn_status fwd_view(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K, const void* V,
                       void* out, int64_t N, int64_t nnz, int H, int D, float scale, gtattn_dtype dtype,
                       int64_t n_src, cudaStream_t stream);

// Benchmark instrumentation: brackets a launch group with CUDA events when
// profiling is enabled (see gtattn_profile_enable).
class ProfScope {
  public:
    ProfScope(int category, int launches, cudaStream_t s);
    ~ProfScope();
  private:
    int cat_;
    cudaStream_t s_;
    void* start_;
};
}  // namespace gt

#define GT_CUDA(call)                                           \
    do {                                                        \
        cudaError_t _e = (call);                                \
        if (_e != cudaSuccess) return gt::cuda_status(_e);      \
    } while (0)

#define GT_TRY(call)                                            \
    do {                                                        \
        gtattn_status _s = (call);                              \
        if (_s != GTATTN_OK) return _s;                         \
    } while (0)

// CSR check of the checking build at an entry point (nothing otherwise).
#ifdef GTATTN_DEBUG
#define GT_DEBUG_CSR(indptr, indices, N, nnz, s)                                        \
    do {                                                                                \
        if ((N) > 0) GT_TRY(gt::debug_csr_check((indptr), (indices), (N), (nnz), (s)));  \
    } while (0)
#else
#define GT_DEBUG_CSR(indptr, indices, N, nnz, s) do { } while (0)
#endif
