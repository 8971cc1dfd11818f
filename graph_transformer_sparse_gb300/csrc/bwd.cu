// bwd.cu -- backward pass of the sparse attention forward (binary A).
//
// Gradients of L = sum out * dO with respect to Q, K and V.  The pages train
// this block ("Graph Transformer in a Nutshell": the molhiv loop calls
// loss.backward() through SparseMHA) but print no backward; this is the chain
// rule on the forward's definition, per row i and head h, s_e = scale q_i.k_j,
// p_e the row softmax:
//   dp_e = dO_i . v_j,   Dlt = sum_e p_e dp_e,   ds_e = p_e (dp_e - Dlt)
//   dQ_i = scale sum_e ds_e k_j,   dK_j += scale ds_e q_i,   dV_j += p_e dO_i
//
// One warp per destination row (CSR by destination), lanes over the row's
// H*D features (KPL per lane), per-head dot products summed through shared
// memory.  Two walks over the row's entries: the first recomputes the
// softmax statistics online (max m, sum l, and a = sum exp(s - m) dp, so
// Dlt = a / l without storing anything per entry); the second forms p and
// ds per entry, accumulates dQ_i in registers (written once) and scatters
// dK_j and dV_j with fp32 atomic adds (a source row gathers from all the
// rows it feeds).  The gradients are fp32 whatever the input type.
#include "common.cuh"

#include <algorithm>

namespace gt {
namespace {

constexpr int kBwdWarps = 4;
constexpr int kBwdMaxH = 128;   // per-head state in shared memory

template <typename T, int KPL>
__global__ void __launch_bounds__(kBwdWarps * 32)
k_bwd_rows(const int* __restrict__ indptr, const int* __restrict__ indices, const T* __restrict__ Q,
           const T* __restrict__ K, const T* __restrict__ V, const T* __restrict__ dO, float* __restrict__ dQ,
           float* __restrict__ dK, float* __restrict__ dV, int N, int H, int D, float scale) {
    __shared__ float sm_a[kBwdWarps][KPL * 32];   // q * k products
    __shared__ float sm_b[kBwdWarps][KPL * 32];   // dO * v products
    __shared__ float sm_h[kBwdWarps][5][kBwdMaxH];   // per head: m, l, a then Dlt, p, ds
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HD = H * D;
    float* pa = sm_a[wid];
    float* pb = sm_b[wid];
    float* hm = sm_h[wid][0];
    float* hl = sm_h[wid][1];
    float* hx = sm_h[wid][2];   // walk 1: a = sum exp(s - m) dp; then Dlt = a / l
    float* hp = sm_h[wid][3];   // walk 2: p of the current entry
    float* hy = sm_h[wid][4];   // walk 2: ds of the current entry
    // per-head sums of a product buffer (eight interleaved partial sums)
    auto head_sum = [&](const float* buf, int h) {
        const float* r = buf + h * D;
        float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        int d = 0;
        for (; d + 8 <= D; d += 8) {
#pragma unroll
            for (int k = 0; k < 8; ++k) a[k] += r[d + k];
        }
        for (; d < D; ++d) a[0] += r[d];
        return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
    };
    for (int row = blockIdx.x * kBwdWarps + wid; row < N; row += gridDim.x * kBwdWarps) {
        const int beg = indptr[row], end = indptr[row + 1];
        float q[KPL], g[KPL], dq[KPL];
#pragma unroll
        for (int k = 0; k < KPL; ++k) {
            const int el = lane + 32 * k;
            q[k] = el < HD ? load_elem(Q, (int64_t)row * HD + el) : 0.f;
            g[k] = el < HD ? load_elem(dO, (int64_t)row * HD + el) : 0.f;
            dq[k] = 0.f;
        }
        for (int h = lane; h < H; h += 32) { hm[h] = -INFINITY; hl[h] = 0.f; hx[h] = 0.f; }
        __syncwarp();
        // the per-head score s and dp of entry e, into the product buffers
        auto products = [&](int64_t j) {
#pragma unroll
            for (int k = 0; k < KPL; ++k) {
                const int el = lane + 32 * k;
                if (el < HD) {
                    pa[el] = q[k] * load_elem(K, j * HD + el);
                    pb[el] = g[k] * load_elem(V, j * HD + el);
                }
            }
            __syncwarp();
        };
        // walk 1: m, l and a per head, online
        for (int e = beg; e < end; ++e) {
            products(__ldg(indices + e));
            for (int h = lane; h < H; h += 32) {
                const float s = scale * head_sum(pa, h), dp = head_sum(pb, h);
                const float mo = hm[h], mn = fmaxf(mo, s);
                const float c = expf(mo - mn), w = expf(s - mn);
                hl[h] = hl[h] * c + w;
                hx[h] = hx[h] * c + w * dp;
                hm[h] = mn;
            }
            __syncwarp();
        }
        // Dlt = a / l per head, kept in hx
        for (int h = lane; h < H; h += 32) hx[h] = hl[h] > 0.f ? hx[h] / hl[h] : 0.f;
        __syncwarp();
        // walk 2: p, ds; dQ in registers, dK and dV scattered
        for (int e = beg; e < end; ++e) {
            const int64_t j = __ldg(indices + e);
            products(j);
            for (int h = lane; h < H; h += 32) {
                const float s = scale * head_sum(pa, h), dp = head_sum(pb, h);
                const float p = expf(s - hm[h]) / hl[h];
                hp[h] = p;
                hy[h] = p * (dp - hx[h]);
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < KPL; ++k) {
                const int el = lane + 32 * k;
                if (el < HD) {
                    const int h = el / D;
                    const float ds = hy[h], p = hp[h];
                    dq[k] += scale * ds * load_elem(K, j * HD + el);
                    atomicAdd(dK + j * HD + el, scale * ds * q[k]);
                    atomicAdd(dV + j * HD + el, p * g[k]);
                }
            }
            __syncwarp();
        }
#pragma unroll
        for (int k = 0; k < KPL; ++k) {
            const int el = lane + 32 * k;
            if (el < HD) dQ[(int64_t)row * HD + el] = dq[k];
        }
        __syncwarp();
    }
}

template <typename T>
gtattn_status launch_bwd_t(const int* indptr, const int* indices, const void* Q, const void* K, const void* V,
                           const void* dO, float* dQ, float* dK, float* dV, int N, int H, int D, float scale,
                           cudaStream_t s) {
    const int kpl = (H * D + 31) / 32;
    const int blocks = std::max(1, std::min((N + kBwdWarps - 1) / kBwdWarps, num_sms() * 16));
    auto go = [&](auto kernel) {
        kernel<<<blocks, kBwdWarps * 32, 0, s>>>(indptr, indices, static_cast<const T*>(Q), static_cast<const T*>(K),
                                                  static_cast<const T*>(V), static_cast<const T*>(dO), dQ, dK, dV, N,
                                                  H, D, scale);
        return cudaGetLastError();
    };
    const cudaError_t e = kpl <= 4 ? go(k_bwd_rows<T, 4>) : kpl <= 8 ? go(k_bwd_rows<T, 8>) : go(k_bwd_rows<T, 32>);
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

}  // namespace
}  // namespace gt

using namespace gt;

extern "C" gtattn_status gtattn_bwd(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                                    const void* V, const void* dO, float* dQ, float* dK, float* dV, int64_t N,
                                    int64_t nnz, int H, int D, float scale, gtattn_dtype dtype,
                                    cudaStream_t stream) {
    if (N < 0 || nnz < 0 || N >= (1ll << 31) - 1 || nnz >= (1ll << 31) - 1) return GTATTN_ERR_INVALID_ARG;
    if (H < 1 || D < 1 || (int64_t)H * D > kMaxHD || H > kBwdMaxH) return GTATTN_ERR_INVALID_ARG;
    if (dtype != GTATTN_F32 && dtype != GTATTN_BF16 && dtype != GTATTN_BF16_OUT_F32) return GTATTN_ERR_INVALID_ARG;
    if (!indptr) return GTATTN_ERR_INVALID_ARG;
    if (N > 0 && (!Q || !dO || !dQ || !dK || !dV)) return GTATTN_ERR_INVALID_ARG;
    if (nnz > 0 && (!indices || !K || !V)) return GTATTN_ERR_INVALID_ARG;
    const uintptr_t esz = dtype == GTATTN_F32 ? 4 : 2;
    const uintptr_t in_al = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                            reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(dO);
    const uintptr_t out_al = reinterpret_cast<uintptr_t>(dQ) | reinterpret_cast<uintptr_t>(dK) |
                             reinterpret_cast<uintptr_t>(dV) | reinterpret_cast<uintptr_t>(indptr) |
                             reinterpret_cast<uintptr_t>(indices);
    if ((in_al & (esz - 1)) || (out_al & 3u)) return GTATTN_ERR_INVALID_ARG;
    if (N == 0) return GTATTN_OK;
    const size_t bytes = sizeof(float) * static_cast<size_t>(N) * H * D;
    cudaError_t e = cudaMemsetAsync(dK, 0, bytes, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(dV, 0, bytes, stream);
    if (e != cudaSuccess) return cuda_status(e);
    ProfScope ps(GTATTN_KCAT_ROWS, 1, stream);
    if (dtype == GTATTN_F32)
        return launch_bwd_t<float>(indptr, indices, Q, K, V, dO, dQ, dK, dV, (int)N, H, D, scale, stream);
    return launch_bwd_t<__nv_bfloat16>(indptr, indices, Q, K, V, dO, dQ, dK, dV, (int)N, H, D, scale, stream);
}
