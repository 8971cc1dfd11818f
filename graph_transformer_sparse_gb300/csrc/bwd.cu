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
#include "bwd.cuh"

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


// ---------------------------------------------------------------------------
// task-parallel backward (the shapes the fused row kernel tiles)
// ---------------------------------------------------------------------------
// With the forward's output O and row log-sum-exp L (log2 units) at hand,
//   p_e = 2^(s_e log2 e - L),   Dlt = sum_e p_e dp_e = dO_i . O_i,
// so each entry's p and ds need only that entry: the work splits like the
// forward's -- ordinary rows whole, rows above the split threshold in
// 256-entry chunks -- one task per warp.  A lane holds E contiguous
// features of a row (lph = D/E lanes per head, dot products reduced by xor
// shuffles), loads them as 16-byte vectors and adds its dQ, dK, dV pieces
// with float4 atomics (dQ once per task, dK_j and dV_j per entry).  A row of
// one entry has p = 1 and ds = 0 (the forward wrote no L for it).
template <typename T> struct Vec;
template <> struct Vec<float> {
    template <int E> __device__ static void load(const float* p, float* x) {
#pragma unroll
        for (int k = 0; k < E / 4; ++k) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(p) + k);
            x[4 * k] = v.x; x[4 * k + 1] = v.y; x[4 * k + 2] = v.z; x[4 * k + 3] = v.w;
        }
    }
};
template <> struct Vec<__nv_bfloat16> {
    template <int E> __device__ static void load(const __nv_bfloat16* p, float* x) {
        if constexpr (E == 4) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
            x[0] = bf16lo(v.x); x[1] = bf16hi(v.x); x[2] = bf16lo(v.y); x[3] = bf16hi(v.y);
        } else {
#pragma unroll
            for (int k = 0; k < E / 8; ++k) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + k);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) { x[8 * k + 2 * u] = bf16lo(w[u]); x[8 * k + 2 * u + 1] = bf16hi(w[u]); }
            }
        }
    }
};

template <int E>
__device__ __forceinline__ void atomic_add_vec(float* dst, const float* x, float c) {
#pragma unroll
    for (int k = 0; k < E / 4; ++k)
        atomicAdd(reinterpret_cast<float4*>(dst) + k,
                  make_float4(c * x[4 * k], c * x[4 * k + 1], c * x[4 * k + 2], c * x[4 * k + 3]));
}

constexpr int kTaskWarps = 8;

template <typename T, int E>
__global__ void __launch_bounds__(kTaskWarps * 32)
k_bwd_tasks(const int* __restrict__ indptr, const int* __restrict__ indices, const int* __restrict__ hdr,
            const int* __restrict__ rows, const int2* __restrict__ chunks, int chunk_edges,
            const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V, const T* __restrict__ dO,
            const float* __restrict__ O, const float* __restrict__ L, float* __restrict__ dQ,
            float* __restrict__ dK, float* __restrict__ dV, int H, int lph, float scale) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int HD = 32 * E;
    const int head = lane / lph;
    const float sl2 = scale * kLog2e;
    const int n_rows = hdr[HdrLayout::kDenseSeg];   // the bucketed rows (no dense segment here)
    const int n_tasks = n_rows + hdr[HdrLayout::kChunks];
    auto reduce = [&](float v) {
        for (int o = 1; o < lph; o <<= 1) v += __shfl_xor_sync(full, v, o);
        return v;
    };
    for (int t = blockIdx.x * kTaskWarps + (threadIdx.x >> 5); t < n_tasks; t += gridDim.x * kTaskWarps) {
        int row, beg, end;
        if (t < n_rows) {
            row = rows[t];
            beg = indptr[row];
            end = indptr[row + 1];
        } else {
            const int2 c = chunks[t - n_rows];
            row = c.x;
            beg = c.y;
            end = min(beg + chunk_edges, indptr[row + 1]);
        }
        if (end <= beg) continue;   // uniform over the warp (one task per warp)
        const bool single = indptr[row + 1] - indptr[row] == 1;
        const int64_t off = static_cast<int64_t>(row) * HD + lane * E;
        float q[E], g[E], o[E], dq[E];
        Vec<T>::template load<E>(Q + off, q);
        Vec<T>::template load<E>(dO + off, g);
        Vec<float>::template load<E>(O + off, o);
        // Dlt = dO_i . O_i (this head), summed exactly as dp below, so that a
        // row of one entry (O_i = v_j) gets dp - Dlt = 0 exactly
        float la = 0.f, lb = 0.f;
#pragma unroll
        for (int k = 0; k < E; k += 2) {
            la = fmaf(g[k], o[k], la);
            lb = fmaf(g[k + 1], o[k + 1], lb);
        }
#pragma unroll
        for (int k = 0; k < E; ++k) dq[k] = 0.f;
        const float dl = reduce(la + lb);
        const float lse = single ? 0.f : L[static_cast<int64_t>(row) * H + head];
        int jn = __ldg(indices + beg);
        for (int e = beg; e < end; ++e) {
            const int64_t j = jn;
            if (e + 1 < end) jn = __ldg(indices + e + 1);      // the next index, off the critical path
            float kx[E], vx[E];
            Vec<T>::template load<E>(K + j * HD + lane * E, kx);
            Vec<T>::template load<E>(V + j * HD + lane * E, vx);
            float sa = 0.f, sb = 0.f, da = 0.f, db = 0.f;
#pragma unroll
            for (int k = 0; k < E; k += 2) {
                sa = fmaf(q[k], kx[k], sa);
                sb = fmaf(q[k + 1], kx[k + 1], sb);
                da = fmaf(g[k], vx[k], da);
                db = fmaf(g[k + 1], vx[k + 1], db);
            }
            const float s = reduce(sa + sb), dp = reduce(da + db);
            const float p = single ? 1.f : exp2f(s * sl2 - lse);
            const float ds = p * (dp - dl);
#pragma unroll
            for (int k = 0; k < E; ++k) dq[k] = fmaf(ds, kx[k], dq[k]);
            atomic_add_vec<E>(dK + j * HD + lane * E, q, scale * ds);
            atomic_add_vec<E>(dV + j * HD + lane * E, g, p);
        }
        atomic_add_vec<E>(dQ + off, dq, scale);
    }
}
}  // namespace
}  // namespace gt

namespace gt {

gtattn_status launch_bwd_rows(const int* indptr, const int* indices, const void* Q, const void* K, const void* V,
                              const void* dO, float* dQ, float* dK, float* dV, int N, int H, int D, float scale,
                              gtattn_dtype dtype, cudaStream_t s) {
    if (dtype == GTATTN_F32) return launch_bwd_t<float>(indptr, indices, Q, K, V, dO, dQ, dK, dV, N, H, D, scale, s);
    return launch_bwd_t<__nv_bfloat16>(indptr, indices, Q, K, V, dO, dQ, dK, dV, N, H, D, scale, s);
}

bool bwd_tasks_supported(int H, int D, gtattn_dtype dtype, const void* const* ptrs, int n_ptrs) {
    const int HD = H * D;
    if (HD % 32 != 0) return false;
    const int E = HD / 32;
    if ((E != 4 && E != 8 && E != 16 && E != 32) || D % E != 0) return false;
    const int lph = D / E;
    if (lph & (lph - 1)) return false;
    if (dtype == GTATTN_F32 && E < 4) return false;
    uintptr_t al = 0;
    for (int i = 0; i < n_ptrs; ++i) al |= reinterpret_cast<uintptr_t>(ptrs[i]);
    return (al & 15u) == 0;
}

gtattn_status launch_bwd_tasks(const int* indptr, const int* indices, const TaskLists& L, const void* Q,
                               const void* K, const void* V, const void* dO, const float* O, const float* lse,
                               float* dQ, float* dK, float* dV, int N, int H, int D, float scale, gtattn_dtype dtype,
                               cudaStream_t s) {
    const int E = H * D / 32, lph = D / E;
    const int blocks = num_sms() * 8;
    auto go = [&](auto kernel, auto tag) {
        using T = decltype(tag);
        kernel<<<blocks, kTaskWarps * 32, 0, s>>>(indptr, indices, L.hdr, L.rows, L.chunks, L.chunk_edges,
                                                   static_cast<const T*>(Q), static_cast<const T*>(K),
                                                   static_cast<const T*>(V), static_cast<const T*>(dO), O, lse, dQ,
                                                   dK, dV, H, lph, scale);
        return cudaGetLastError();
    };
    cudaError_t e;
    if (dtype == GTATTN_F32) {
        e = E == 4 ? go(k_bwd_tasks<float, 4>, float{}) : E == 8 ? go(k_bwd_tasks<float, 8>, float{})
          : E == 16 ? go(k_bwd_tasks<float, 16>, float{}) : go(k_bwd_tasks<float, 32>, float{});
    } else {
        using B = __nv_bfloat16;
        e = E == 4 ? go(k_bwd_tasks<B, 4>, B{}) : E == 8 ? go(k_bwd_tasks<B, 8>, B{})
          : E == 16 ? go(k_bwd_tasks<B, 16>, B{}) : go(k_bwd_tasks<B, 32>, B{});
    }
    (void)N;
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

}  // namespace gt
