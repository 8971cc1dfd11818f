// gemm.cu -- the linear maps around the attention: Y = A B^T + b, with B an
// nn.Linear weight [out features, in features].  These are the q/k/v and
// output projections of SparseMHA ("Graph Transformer in a Nutshell",
// section "Sparse Multi-head Attention": q_proj, k_proj, v_proj, out_proj,
// with biases) and of TransLayer ("Efficient Sparse Transformer
// implementation with DGL's builtin operators": proj_q, proj_k, proj_v,
// proj_o, bias=False).
//
// bf16 operands run on the 5th-generation tensor cores, in a persistent
// kernel (one CTA per SM walking the 128 x 128 output tiles): one thread
// streams 128 x 64 tiles of A and B by TMA (128-byte swizzle) through a
// four-stage ring, one elected lane of a converged warp issues tcgen05.mma
// (kind::f16, M = 128, N = 128, four K steps of 16 per stage) into one of
// two fp32 accumulators in tensor memory, and eight epilogue warps read the
// other accumulator back (tcgen05.ld), add the bias, round, and store the
// tile through a bank-conflict-free shared-memory staging area so that each
// warp store instruction writes whole 64- or 128-byte row pieces -- the
// loads and products of one tile overlap the epilogue of the one before.
// Every mbarrier wait is bounded; a wait that gives up records error code 1
// in a per-device word (gtattn_device_errors), drains the copies and
// products the CTA issued and returns.
//
// Other shapes and fp32 operands take a CUDA-core kernel (64 x 64 tiles,
// 4 x 4 outputs a thread, fp32 FMAs in ascending k).
#include "gemm.cuh"
#include "tc.cuh"

#include <algorithm>
#include <cstdio>
#include <mutex>

namespace gt {

// Error codes recorded by the projection kernels (1: a bounded wait gave up);
// read and cleared by gtattn_device_errors.
__device__ int g_gemm_errors;

namespace {

constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr int kGemmStages = 4;
constexpr uint32_t kTileA = kBM * kBK * 2;   // 16 KB of bf16
constexpr uint32_t kTileB = kBN * kBK * 2;
constexpr uint32_t kStageBytes = kTileA + kTileB;
constexpr int kEpiWarps = 8;                  // epilogue warps: two per tensor-memory lane quarter (column halves)
constexpr int kGemmThreads = (2 + kEpiWarps) * 32;
constexpr uint32_t kStageOut = 4096;          // epilogue staging per warp (32 rows x 128 bytes)
constexpr int kBiasSmem = 4096;               // biases of up to this many columns staged in shared memory
constexpr size_t kGemmSmem = kGemmStages * kStageBytes + kEpiWarps * kStageOut + kBiasSmem * 4 + 1024;
constexpr uint32_t kAccCols = 2 * kBN;        // two accumulators in tensor memory

struct GemmBars {
    uint64_t full[kGemmStages];    // stage loaded (TMA -> MMA)
    uint64_t empty[kGemmStages];   // stage consumed (MMA -> TMA)
    uint64_t acc_full[2];          // accumulator b holds a finished tile (MMA -> epilogue)
    uint64_t acc_empty[2];         // accumulator b read out (epilogue -> MMA, kEpiWarps arrivals)
    uint64_t drain;                // products issued before a give-up finished
};

// D (+)= A B^T over one 64-wide K block: four K steps of 16 elements (32
// bytes: descriptor start + 2 per step), one elected lane of the warp.
__device__ __forceinline__ void mma_kblock(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\tsetp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %3, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %3, q;\n\t}"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc), "l"(a + 2), "l"(b + 2), "l"(a + 4), "l"(b + 4), "l"(a + 6),
          "l"(b + 6)
        : "memory");
}

template <typename TO>
__device__ __forceinline__ TO* out_ptr(const GemmOut& o, int64_t m, int c) {
    const int g = c / o.cols_per_split;
    return static_cast<TO*>(o.base) + g * o.split_stride + m * o.ld + (c - g * o.cols_per_split);
}

// Persistent, warp-specialised: one CTA per SM walks the output tiles
// (column tiles fastest, so neighbouring CTAs share A's rows in the L2).
//   warp 0      TMA: A and B tiles into a four-stage ring, running ahead
//               across tiles
//   warp 1      MMA issue (converged warp, one elected lane) into one of two
//               tensor-memory accumulators, alternating per tile
//   warps 2-9   epilogue: wait for a finished accumulator, read it out
//               (tcgen05.ld; each warp its lane quarter and half the
//               columns), free it for the tile after next, add the bias (in
//               shared memory), round, store through a per-warp staging area
//               as whole row pieces
// so the loads and products of tile t+1 overlap the epilogue of tile t.
template <typename TO>
__global__ void __launch_bounds__(kGemmThreads, 1)
k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
          const float* __restrict__ bias, int64_t M, int Nn, int K, GemmOut o, int64_t n_tiles) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) GemmBars bars;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = (Nn + kBN - 1) / kBN;
    const int KB = (K + kBK - 1) / kBK;
    auto sA = [&](int st) { return smem + st * kStageBytes; };
    auto sB = [&](int st) { return smem + st * kStageBytes + kTileA; };

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&s_tmem)),
                     "r"(kAccCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 32) {
        s_abort = 0;
        for (int i = 0; i < kGemmStages; ++i) {
            mbar_init(&bars.full[i], 1);
            mbar_init(&bars.empty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.acc_full[b], 1);
            mbar_init(&bars.acc_empty[b], kEpiWarps);
        }
        mbar_init(&bars.drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the bias, staged once (columns beyond kBiasSmem read it from global memory)
    // (zeros past Nn up to the next 32-column chunk)
    float* s_bias = reinterpret_cast<float*>(smem + kGemmStages * kStageBytes + kEpiWarps * kStageOut);
    for (int c = threadIdx.x; c < min((Nn + 31) & ~31, kBiasSmem); c += kGemmThreads)
        s_bias[c] = (bias && c < Nn) ? bias[c] : 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ---- TMA producer (one thread) ----
        if (lane == 0) {
            bool ok = true;
            int64_t it = 0;   // k-blocks issued over all tiles
            for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
                const int n0 = static_cast<int>(t % NT) * kBN;
                const int m0 = static_cast<int>((t / NT) * kBM);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int st = static_cast<int>(it % kGemmStages);
                    const int64_t use = it / kGemmStages;
                    if (use > 0 && !mbar_wait(&bars.empty[st], static_cast<uint32_t>((use - 1) & 1))) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&bars.full[st], kStageBytes);
                    tma_load_2d(sA(st), &tmA, kb * kBK, m0, &bars.full[st]);
                    tma_load_2d(sB(st), &tmB, kb * kBK, n0, &bars.full[st]);
                }
            }
            if (!ok) {
                atomicOr(&g_gemm_errors, 1);
                atomicExch(&s_abort, 1);
                // the copies issued must land before the CTA exits (bounded)
                for (int st = 0; st < kGemmStages; ++st) {
                    const int64_t uses = it / kGemmStages + (st < it % kGemmStages ? 1 : 0);
                    if (uses > 0) mbar_wait(&bars.full[st], static_cast<uint32_t>((uses - 1) & 1), kTcWaitCycles / 4);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issue (the converged warp, one elected lane) ----
        const uint32_t idesc = idesc_bf16(kBM, kBN, 0);
        bool ok = true;
        int64_t it = 0;
        int lt = 0;   // tiles of this CTA so far
        for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++lt) {
            const int b = lt & 1;
            // accumulator b was last used by tile lt-2: its epilogue must have read it
            if (lt >= 2 && !mbar_wait_warp(&bars.acc_empty[b], static_cast<uint32_t>(((lt >> 1) - 1) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + static_cast<uint32_t>(b * kBN);
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int st = static_cast<int>(it % kGemmStages);
                if (!mbar_wait_warp(&bars.full[st], static_cast<uint32_t>((it / kGemmStages) & 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                mma_kblock(d, smem_desc_sw128(su32(sA(st)), 16, 1024), smem_desc_sw128(su32(sB(st)), 16, 1024),
                           idesc, kb > 0 ? 1u : 0u);
                tc_commit(&bars.empty[st]);
            }
            if (ok) tc_commit(&bars.acc_full[b]);
        }
        if (!ok) {
            if (lane == 0) {
                atomicOr(&g_gemm_errors, 1);
                atomicExch(&s_abort, 1);
            }
        }
        // every product issued finishes before tensor memory is freed
        tc_commit(&bars.drain);
        mbar_wait_warp(&bars.drain, 0, kTcWaitCycles / 4);
    } else {
        // ---- epilogue (warps 2..9: lane quarter warp % 4, column half (warp - 2) / 4) ----
        const int q4 = warp & 3;
        const int c_half = (warp - 2) >> 2;
        constexpr int kCols = kBN / 2;                            // columns a warp reads out
        constexpr int kVec = 16 / static_cast<int>(sizeof(TO));   // elements per 16-byte piece
        constexpr int nq = 32 / kVec;                             // pieces per row of a 32-column chunk
        constexpr int rows_per_store = 32 / nq;
        constexpr int rows_per_line = 8 / nq;                     // rows sharing one 128-byte bank line
        unsigned char* stage = smem + kGemmStages * kStageBytes + (warp - 2) * kStageOut;
        int lt = 0;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++lt) {
            const int b = lt & 1;
            bool ok = mbar_wait(&bars.acc_full[b], static_cast<uint32_t>((lt >> 1) & 1));
            ok = __all_sync(0xffffffffu, ok) && *reinterpret_cast<volatile int*>(&s_abort) == 0;
            if (!ok) {
                if (lane == 0) atomicExch(&s_abort, 1);
                break;
            }
            tc_fence_after();
            const int n0 = static_cast<int>(t % NT) * kBN + c_half * kCols;
            const int64_t m0 = (t / NT) * kBM;
            const int n_chunks = Nn - n0 > 0 ? (min(kCols, Nn - n0) + 31) / 32 : 0;
            // this lane's row of the warp's column half into registers, then free it
            uint32_t r[kCols];
            const uint32_t trow = tmem + static_cast<uint32_t>(b * kBN + c_half * kCols) +
                                  (static_cast<uint32_t>(q4 * 32) << 16);
#pragma unroll
            for (int c4 = 0; c4 < kCols / 32; ++c4)
                if (c4 < n_chunks) tmem_ld32(trow + 32 * c4, r + 32 * c4);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.acc_empty[b]);
#pragma unroll
            for (int c4 = 0; c4 < kCols / 32; ++c4) {
                if (c4 >= n_chunks) break;
                const int cb = n0 + 32 * c4;   // first column of the chunk
                // the chunk's 32 biases (the same for every lane)
                float bb[32];
                if (cb + 32 <= kBiasSmem) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 f = reinterpret_cast<const float4*>(s_bias + cb)[k];
                        bb[4 * k] = f.x; bb[4 * k + 1] = f.y; bb[4 * k + 2] = f.z; bb[4 * k + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 32; ++u) bb[u] = (bias && cb + u < Nn) ? __ldg(bias + cb + u) : 0.f;
                }
                // this lane's row into the staging area: piece q at slot (q + lane / rows_per_line) % nq
#pragma unroll
                for (int q = 0; q < nq; ++q) {
                    const uint32_t* x = r + 32 * c4 + q * kVec;
                    const float* b = bb + q * kVec;
                    uint4 v;
                    if constexpr (sizeof(TO) == 2) {
                        v = make_uint4(pack2_bf16(__uint_as_float(x[0]) + b[0], __uint_as_float(x[1]) + b[1]),
                                       pack2_bf16(__uint_as_float(x[2]) + b[2], __uint_as_float(x[3]) + b[3]),
                                       pack2_bf16(__uint_as_float(x[4]) + b[4], __uint_as_float(x[5]) + b[5]),
                                       pack2_bf16(__uint_as_float(x[6]) + b[6], __uint_as_float(x[7]) + b[7]));
                    } else {
                        v = make_uint4(__float_as_uint(__uint_as_float(x[0]) + b[0]),
                                       __float_as_uint(__uint_as_float(x[1]) + b[1]),
                                       __float_as_uint(__uint_as_float(x[2]) + b[2]),
                                       __float_as_uint(__uint_as_float(x[3]) + b[3]));
                    }
                    const int slot = (q + lane / rows_per_line) % nq;
                    *reinterpret_cast<uint4*>(stage + (lane * nq + slot) * 16) = v;
                }
                __syncwarp();
                // coalesced stores: rows_per_store rows of nq pieces per instruction; this
                // lane's piece is column c of every row it stores
                const int q = lane % nq;
                const int c = cb + q * kVec;
                if (c < Nn) {
                    TO* col = out_ptr<TO>(o, 0, c);
#pragma unroll
                    for (int i = 0; i < 32 / rows_per_store; ++i) {
                        const int rr = i * rows_per_store + lane / nq;
                        const int slot = (q + rr / rows_per_line) % nq;
                        const uint4 v = *reinterpret_cast<const uint4*>(stage + (rr * nq + slot) * 16);
                        const int64_t m = m0 + q4 * 32 + rr;
                        if (m < M) *reinterpret_cast<uint4*>(col + m * o.ld) = v;
                    }
                }
                __syncwarp();
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kAccCols) : "memory");
    }
}

// ---- CUDA-core kernel ------------------------------------------------------
constexpr int kSimtTile = 64, kSimtK = 16;

template <typename T>
__device__ __forceinline__ float as_float(T x) {
    if constexpr (sizeof(T) == 2) return __bfloat162float(x);
    else return x;
}

template <typename T, typename TO>
__global__ void __launch_bounds__(256)
k_gemm_simt(const T* __restrict__ A, const T* __restrict__ B, const float* __restrict__ bias, int64_t M, int Nn,
            int K, GemmOut o) {
    __shared__ float sA[kSimtK][kSimtTile + 4];
    __shared__ float sB[kSimtK][kSimtTile + 4];
    const int NT = (Nn + kSimtTile - 1) / kSimtTile;
    const int n0 = static_cast<int>(blockIdx.x % NT) * kSimtTile;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x / NT) * kSimtTile;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += kSimtK) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = threadIdx.x + 256 * i;
            const int rr = e / kSimtK, kk = e % kSimtK;
            const int64_t m = m0 + rr;
            const int n = n0 + rr, k = k0 + kk;
            sA[kk][rr] = (m < M && k < K) ? as_float(A[m * K + k]) : 0.f;
            sB[kk][rr] = (n < Nn && k < K) ? as_float(B[static_cast<int64_t>(n) * K + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kSimtK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = sA[kk][ty + 16 * i];
                b[i] = sB[kk][tx + 16 * i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + ty + 16 * i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx + 16 * j;
            if (n >= Nn) continue;
            const float v = acc[i][j] + (bias ? bias[n] : 0.f);
            TO* p = out_ptr<TO>(o, m, n);
            if constexpr (sizeof(TO) == 2) *p = __float2bfloat16_rn(v);
            else *p = v;
        }
    }
}

// ---- head-order permutations -----------------------------------------------
// Row r = g*HD + h*D + d of the result is row g*HD + d*H + h of W.
template <typename T>
__global__ void k_permute_rows(const T* __restrict__ W, T* __restrict__ Wp, const float* __restrict__ b,
                               float* __restrict__ bp, int groups, int H, int D, int K) {
    const int HD = H * D;
    const int64_t total = static_cast<int64_t>(groups) * HD * K;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / K;
        const int k = static_cast<int>(i - r * K);
        const int g = static_cast<int>(r / HD), f = static_cast<int>(r - static_cast<int64_t>(g) * HD);
        const int h = f / D, d = f - h * D;
        const int64_t src = static_cast<int64_t>(g) * HD + d * H + h;
        Wp[i] = W[src * K + k];
        if (b && k == 0) bp[r] = b[src];
    }
}

// Column h*D + d of the result is column d*H + h of W.
template <typename T>
__global__ void k_permute_cols(const T* __restrict__ W, T* __restrict__ Wp, int rows, int H, int D) {
    const int HD = H * D;
    const int64_t total = static_cast<int64_t>(rows) * HD;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / HD;
        const int f = static_cast<int>(i - r * HD);
        const int h = f / D, d = f - h * D;
        Wp[i] = W[r * HD + d * H + h];
    }
}

// [rows, cols] bf16 row-major, box 64 columns x 128 rows, 128-byte swizzle
// (out-of-range rows and columns read as zero).
bool make_map_2d(CUtensorMap* m, const void* base, int64_t rows, int cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {kBK, 128};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int grid_1d(int64_t total, int threads) {
    const int64_t b = (total + threads - 1) / threads;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(b, static_cast<int64_t>(num_sms()) * 16)));
}

}  // namespace

bool gemm_tc_supported(const void* A, const void* B, int K, const GemmOut& o, bool out_f32) {
    const int vec = out_f32 ? 4 : 8;
    const uintptr_t al = reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
                         reinterpret_cast<uintptr_t>(o.base);
    return (al & 15u) == 0 && K % 8 == 0 && K > 0 && o.cols_per_split % vec == 0 && o.ld % vec == 0 &&
           o.split_stride % vec == 0 && encode_fn() != nullptr;
}

gtattn_status launch_gemm_tc(const void* A, const void* B, const float* bias, int64_t M, int Nn, int K,
                             const GemmOut& o, bool out_f32, cudaStream_t s) {
    if (M == 0 || Nn == 0) return GTATTN_OK;
    CUtensorMap ma, mb;
    if (!make_map_2d(&ma, A, M, K) || !make_map_2d(&mb, B, Nn, K)) return GTATTN_ERR_UNSUPPORTED;
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((Nn + kBN - 1) / kBN);
    if ((M + kBM - 1) / kBM * kBM > 0x7fffffff) return GTATTN_ERR_UNSUPPORTED;   // TMA row coordinates are int
    const int grid = static_cast<int>(std::min<int64_t>(tiles, num_sms()));   // persistent: one CTA per SM
    cudaError_t e;
    auto go = [&](auto kernel) {
        cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kGemmSmem));
        if (r != cudaSuccess) return r;
        kernel<<<grid, kGemmThreads, kGemmSmem, s>>>(ma, mb, bias, M, Nn, K, o, tiles);
        return cudaGetLastError();
    };
    e = out_f32 ? go(k_gemm_tc<float>) : go(k_gemm_tc<__nv_bfloat16>);
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

gtattn_status launch_gemm_simt(const void* A, const void* B, const float* bias, int64_t M, int Nn, int K,
                               bool in_bf16, const GemmOut& o, bool out_f32, cudaStream_t s) {
    if (M == 0 || Nn == 0) return GTATTN_OK;
    const int64_t tiles = ((M + kSimtTile - 1) / kSimtTile) * ((Nn + kSimtTile - 1) / kSimtTile);
    if (tiles > 0x7fffffff) return GTATTN_ERR_UNSUPPORTED;
    const unsigned g = static_cast<unsigned>(tiles);
    if (in_bf16) {
        using T = __nv_bfloat16;
        if (out_f32)
            k_gemm_simt<T, float><<<g, 256, 0, s>>>(static_cast<const T*>(A), static_cast<const T*>(B), bias, M, Nn,
                                                    K, o);
        else
            k_gemm_simt<T, T><<<g, 256, 0, s>>>(static_cast<const T*>(A), static_cast<const T*>(B), bias, M, Nn, K,
                                                o);
    } else {
        if (out_f32)
            k_gemm_simt<float, float><<<g, 256, 0, s>>>(static_cast<const float*>(A), static_cast<const float*>(B),
                                                        bias, M, Nn, K, o);
        else
            return GTATTN_ERR_UNSUPPORTED;
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

gtattn_status launch_permute_rows(const void* W, void* Wp, const float* b, float* bp, int groups, int H, int D,
                                  int K, int esz, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(groups) * H * D * K;
    if (total == 0) return GTATTN_OK;
    const int grid = grid_1d(total, 256);
    if (esz == 2)
        k_permute_rows<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(W),
                                                           static_cast<__nv_bfloat16*>(Wp), b, bp, groups, H, D, K);
    else
        k_permute_rows<float><<<grid, 256, 0, s>>>(static_cast<const float*>(W), static_cast<float*>(Wp), b, bp,
                                                   groups, H, D, K);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

gtattn_status launch_permute_cols(const void* W, void* Wp, int rows, int H, int D, int esz, cudaStream_t s) {
    const int64_t total = static_cast<int64_t>(rows) * H * D;
    if (total == 0) return GTATTN_OK;
    const int grid = grid_1d(total, 256);
    if (esz == 2)
        k_permute_cols<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(W),
                                                           static_cast<__nv_bfloat16*>(Wp), rows, H, D);
    else
        k_permute_cols<float><<<grid, 256, 0, s>>>(static_cast<const float*>(W), static_cast<float*>(Wp), rows, H,
                                                   D);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

}  // namespace gt

using namespace gt;

extern "C" gtattn_status gtattn_device_errors(int* code, int reset) {
    if (!code) return GTATTN_ERR_INVALID_ARG;
    *code = 0;
    GT_CUDA(cudaDeviceSynchronize());
    GT_CUDA(cudaMemcpyFromSymbol(code, g_gemm_errors, sizeof(int)));
    if (reset) {
        const int zero = 0;
        GT_CUDA(cudaMemcpyToSymbol(g_gemm_errors, &zero, sizeof(int)));
    }
    return GTATTN_OK;
}
