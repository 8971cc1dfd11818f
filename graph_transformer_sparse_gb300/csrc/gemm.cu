// gemm.cu -- the linear maps around the attention: Y = A B^T + b, with B an
// nn.Linear weight [out features, in features].  These are the q/k/v and
// output projections of SparseMHA ("Graph Transformer in a Nutshell",
// section "Sparse Multi-head Attention": q_proj, k_proj, v_proj, out_proj,
// with biases) and of TransLayer ("Efficient Sparse Transformer
// implementation with DGL's builtin operators": proj_q, proj_k, proj_v,
// proj_o, bias=False).
//
// bf16 operands run on the 5th-generation tensor cores: a CTA computes one
// 128 x 128 tile of Y; one thread loads 128 x 64 tiles of A and B by TMA
// (128-byte swizzle) into a three-stage ring, one elected lane of a
// converged warp issues tcgen05.mma (kind::f16, fp32 accumulators in tensor
// memory, M = 128, N = 128, four K steps of 16 per stage), and all four warps
// read the accumulators back (tcgen05.ld), add the bias, round, and store
// the tile through a bank-conflict-free shared-memory staging area so that
// each warp store instruction writes whole 64- or 128-byte row pieces.  Two
// CTAs fit an SM, so one's epilogue overlaps the other's main loop.  Every
// mbarrier wait is bounded; a wait that gives up records error code 1 in a
// per-device word (gtattn_device_errors), drains the copies and products the
// CTA issued and returns.
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
constexpr int kGemmStages = 3;
constexpr uint32_t kTileA = kBM * kBK * 2;   // 16 KB of bf16
constexpr uint32_t kTileB = kBN * kBK * 2;
constexpr uint32_t kStageBytes = kTileA + kTileB;
constexpr size_t kGemmSmem = kGemmStages * kStageBytes + 1024;   // + alignment to 1024
constexpr int kGemmThreads = 128;
static_assert(4 * 4096 <= kGemmStages * kStageBytes, "the epilogue staging fits in the ring");

struct GemmBars {
    uint64_t full[kGemmStages];    // stage loaded (TMA -> MMA)
    uint64_t empty[kGemmStages];   // stage consumed (MMA -> TMA)
    uint64_t done;                 // every product of the tile finished (MMA -> epilogue)
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

template <typename TO>
__global__ void __launch_bounds__(kGemmThreads, 1)
k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
          const float* __restrict__ bias, int64_t M, int Nn, int K, GemmOut o) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) GemmBars bars;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ float s_bias[kBN];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = (Nn + kBN - 1) / kBN;
    const int nt = static_cast<int>(blockIdx.x % NT);
    const int64_t m0 = static_cast<int64_t>(blockIdx.x / NT) * kBM;
    const int n0 = nt * kBN;
    const int KB = (K + kBK - 1) / kBK;
    auto sA = [&](int st) { return smem + st * kStageBytes; };
    auto sB = [&](int st) { return smem + st * kStageBytes + kTileA; };

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&s_tmem)),
                     "r"(kBN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (threadIdx.x == 32) {
        s_abort = 0;
        for (int i = 0; i < kGemmStages; ++i) {
            mbar_init(&bars.full[i], 1);
            mbar_init(&bars.empty[i], 1);
        }
        mbar_init(&bars.done, 1);
        mbar_init(&bars.drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int c = threadIdx.x; c < kBN; c += kGemmThreads) s_bias[c] = (bias && n0 + c < Nn) ? bias[n0 + c] : 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 0) {
        // ---- TMA producer (one thread) ----
        if (lane == 0) {
            bool ok = true;
            int kb = 0;
            for (; kb < KB; ++kb) {
                const int st = kb % kGemmStages, use = kb / kGemmStages;
                if (use > 0 && !mbar_wait(&bars.empty[st], (use - 1) & 1)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&bars.full[st], kStageBytes);
                tma_load_2d(sA(st), &tmA, kb * kBK, static_cast<int>(m0), &bars.full[st]);
                tma_load_2d(sB(st), &tmB, kb * kBK, n0, &bars.full[st]);
            }
            if (!ok) {
                atomicOr(&g_gemm_errors, 1);
                atomicExch(&s_abort, 1);
                // the copies issued must land before the CTA exits (bounded)
                for (int st = 0; st < kGemmStages; ++st) {
                    const int uses = kb / kGemmStages + (st < kb % kGemmStages ? 1 : 0);
                    if (uses > 0) mbar_wait(&bars.full[st], (uses - 1) & 1, kTcWaitCycles / 4);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issue (the converged warp, one elected lane) ----
        const uint32_t idesc = idesc_bf16(kBM, kBN, 0);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
            const int st = kb % kGemmStages;
            if (!mbar_wait_warp(&bars.full[st], (kb / kGemmStages) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            mma_kblock(tmem, smem_desc_sw128(su32(sA(st)), 16, 1024), smem_desc_sw128(su32(sB(st)), 16, 1024),
                       idesc, kb > 0 ? 1u : 0u);
            tc_commit(&bars.empty[st]);
        }
        if (ok) {
            tc_commit(&bars.done);
        } else {
            if (lane == 0) {
                atomicOr(&g_gemm_errors, 1);
                atomicExch(&s_abort, 1);
            }
            // the products issued must finish before tensor memory is freed
            tc_commit(&bars.drain);
            mbar_wait_warp(&bars.drain, 0, kTcWaitCycles / 4);
        }
    }

    // ---- epilogue: warp w holds rows 32w..32w+31 (tensor-memory lanes) ----
    bool ok = mbar_wait(&bars.done, 0);
    if (!ok) atomicExch(&s_abort, 1);
    ok = __all_sync(0xffffffffu, ok) && *reinterpret_cast<volatile int*>(&s_abort) == 0;
    if (ok) {
        tc_fence_after();
        constexpr int kVec = 16 / static_cast<int>(sizeof(TO));   // elements per 16-byte piece
        constexpr int nq = 32 / kVec;                             // pieces per row of a 32-column chunk
        constexpr int rows_per_store = 32 / nq;
        constexpr int rows_per_line = 8 / nq;                     // rows sharing one 128-byte bank line
        unsigned char* stage = smem + warp * 4096;
        const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        for (int c4 = 0; c4 < kBN / 32; ++c4) {
            if (n0 + 32 * c4 >= Nn) break;   // uniform over the CTA
            uint32_t r[32];
            tmem_ld32(trow + 32 * c4, r);
            tmem_ld_wait();
            // this lane's row into the staging area: piece q at slot (q + lane / rows_per_line) % nq
#pragma unroll
            for (int q = 0; q < nq; ++q) {
                uint4 v;
                if constexpr (sizeof(TO) == 2) {
                    const float* b = s_bias + 32 * c4 + 8 * q;
                    const uint32_t* x = r + 8 * q;
                    v = make_uint4(pack2_bf16(__uint_as_float(x[0]) + b[0], __uint_as_float(x[1]) + b[1]),
                                   pack2_bf16(__uint_as_float(x[2]) + b[2], __uint_as_float(x[3]) + b[3]),
                                   pack2_bf16(__uint_as_float(x[4]) + b[4], __uint_as_float(x[5]) + b[5]),
                                   pack2_bf16(__uint_as_float(x[6]) + b[6], __uint_as_float(x[7]) + b[7]));
                } else {
                    const float* b = s_bias + 32 * c4 + 4 * q;
                    const uint32_t* x = r + 4 * q;
                    v = make_uint4(__float_as_uint(__uint_as_float(x[0]) + b[0]),
                                   __float_as_uint(__uint_as_float(x[1]) + b[1]),
                                   __float_as_uint(__uint_as_float(x[2]) + b[2]),
                                   __float_as_uint(__uint_as_float(x[3]) + b[3]));
                }
                const int slot = (q + lane / rows_per_line) % nq;
                *reinterpret_cast<uint4*>(stage + (lane * nq + slot) * 16) = v;
            }
            __syncwarp();
            // coalesced stores: rows_per_store rows of nq pieces per instruction
#pragma unroll
            for (int i = 0; i < 32 / rows_per_store; ++i) {
                const int rr = i * rows_per_store + lane / nq, q = lane % nq;
                const int slot = (q + rr / rows_per_line) % nq;
                const uint4 v = *reinterpret_cast<const uint4*>(stage + (rr * nq + slot) * 16);
                const int64_t m = m0 + warp * 32 + rr;
                const int c = n0 + 32 * c4 + q * kVec;
                if (m < M && c < Nn) *reinterpret_cast<uint4*>(out_ptr<TO>(o, m, c)) = v;
            }
            __syncwarp();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kBN) : "memory");
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
    if (tiles > 0x7fffffff) return GTATTN_ERR_UNSUPPORTED;
    cudaError_t e;
    auto go = [&](auto kernel) {
        cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kGemmSmem));
        if (r != cudaSuccess) return r;
        kernel<<<static_cast<unsigned>(tiles), kGemmThreads, kGemmSmem, s>>>(ma, mb, bias, M, Nn, K, o);
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
