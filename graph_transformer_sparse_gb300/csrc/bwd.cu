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
// The gradients are fp32 whatever the input type.  Two implementations:
//  * the two passes (second half of this file), for rows that split into
//    lane groups of 4..32 features a lane: the forward's output and
//    log-sum-exp make every entry's p and ds local, so dQ is summed by
//    destination row and dK, dV by source over a source-major copy of the
//    pattern, each in registers and stored once;
//  * for other shapes, a warp per destination row, lanes over the row's H*D
//    features (KPL a lane), per-head dot products summed through shared
//    memory, two walks over the row's entries: the first recomputes the
//    softmax statistics online (max m, sum l, and a = sum exp(s - m) dp, so
//    Dlt = a / l without storing anything per entry); the second forms p and
//    ds per entry, accumulates dQ_i in registers (written once) and scatters
//    dK_j and dV_j with fp32 atomic adds.
#include "bwd.cuh"

#include <algorithm>
#include <mutex>
#include <type_traits>
#include <unordered_map>

#include "plan.cuh"
#include "rows.cuh"

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
// two passes (the shapes the fused row kernel tiles)
// ---------------------------------------------------------------------------
// With the forward's output O and row log-sum-exp L (log2 units) at hand,
//   p_e = 2^(s_e log2 e - L_i),   Dlt_i = sum_e p_e dp_e = dO_i . O_i,
// so each entry's p and ds need only that entry and its row's (L_i, Dlt_i).
// The gradients then split by where they are summed:
//   pass 1, over destination rows (the forward's task lists): Dlt_i and
//           dQ_i = scale sum_e ds_e k_j, summed in registers;
//   pass 2, over source nodes, on a source-major copy of the pattern (colptr
//           over sources, the destination row of every entry):
//           dK_j = scale sum_e ds_e q_i and dV_j = sum_e p_e dO_i, summed in
//           registers.
// No gradient is scattered entry by entry.  Rows and sources above the split
// threshold come in 256-entry chunks whose partial sums are added with float4
// atomics (one per lane per chunk) onto rows zeroed beforehand; all others
// are stored.  A row of one entry has p = 1 and ds = 0 exactly: pass 1 stores
// dQ_i = 0 without reading K or V and marks the row with L_i = +inf, which
// pass 2 reads as p = 1, ds = 0.
//
// A lane holds E contiguous features of a node row, loaded as 8- or 16-byte
// vectors; a row spans G = H D / E lanes (a lane group), a head lph = D / E
// of them, and per-head dot products are reduced by xor shuffles within the
// group.

// E features of one node row as loaded (bf16 stays packed: dot products as
// mixed bf16 x bf16 -> fp32 FMAs, accumulation as f32x2 FMAs).
template <typename T, int E> struct Raw;
template <int E> struct Raw<float, E> {
    float w[E];
    __device__ __forceinline__ void load(const float* p) {
#pragma unroll
        for (int k = 0; k < E / 4; ++k) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(p) + k);
            w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
        }
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int k = 0; k < E; ++k) w[k] = 0.f;
    }
    __device__ __forceinline__ float operator[](int k) const { return w[k]; }
    // this . b (two interleaved fp32 sums)
    __device__ __forceinline__ float dot(const Raw& b) const {
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int k = 0; k < E; k += 2) fma2(x, y, w[k], w[k + 1], b.w[k], b.w[k + 1]);
        return x + y;
    }
    // acc += c * this
    __device__ __forceinline__ void axpy(float* acc, float c) const {
#pragma unroll
        for (int k = 0; k < E; k += 2) fma2(acc[k], acc[k + 1], c, c, w[k], w[k + 1]);
    }
};
template <int E> struct Raw<__nv_bfloat16, E> {
    uint32_t w[E / 2];
    __device__ __forceinline__ void load(const __nv_bfloat16* p) {
        if constexpr (E == 4) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
            w[0] = v.x; w[1] = v.y;
        } else {
#pragma unroll
            for (int k = 0; k < E / 8; ++k) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + k);
                w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
            }
        }
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int k = 0; k < E / 2; ++k) w[k] = 0u;
    }
    __device__ __forceinline__ float operator[](int k) const {
        return (k & 1) ? bf16hi(w[k >> 1]) : bf16lo(w[k >> 1]);
    }
    __device__ __forceinline__ float dot(const Raw& b) const {
        float x = 0.f, y = 0.f;
#pragma unroll
        for (int k = 0; k < E / 2; k += 2) {
            x = dot2_bf16(w[k], b.w[k], x);
            y = dot2_bf16(w[k + 1], b.w[k + 1], y);
        }
        return x + y;
    }
    __device__ __forceinline__ void axpy(float* acc, float c) const {
#pragma unroll
        for (int k = 0; k < E / 2; ++k) axpy2_bf16(acc[2 * k], acc[2 * k + 1], c, w[k]);
    }
};

template <int E>
__device__ __forceinline__ void store_vec(float* dst, const float* x, float c) {
#pragma unroll
    for (int k = 0; k < E / 4; ++k)
        reinterpret_cast<float4*>(dst)[k] =
            make_float4(c * x[4 * k], c * x[4 * k + 1], c * x[4 * k + 2], c * x[4 * k + 3]);
}

constexpr int kTaskWarps = 8;
// the two passes: 128-thread blocks; with bf16 rows of up to 16 features a
// lane, pass 1 is capped at 96 registers (five blocks, 20 warps an SM) and
// pass 2, which holds twice the accumulators, at 128 (four blocks; at 96 it
// spills and runs slower)
constexpr int kPassWarps = 4;
template <typename T, int E, int PASS> constexpr int pass_min_blocks() {
    return sizeof(T) == 2 && E <= 16 ? (PASS == 1 ? 5 : 4) : 2;
}

// One task of a binning's lists: a whole row (t < n_rows) or one chunk of a
// split row.  `whole` is false for chunks; `first` for whole rows and the
// first chunk of a split row.
struct Task {
    int row, beg, end;
    bool whole, first;
    int chunk;   // index in the chunk list (split rows), else -1
};
__device__ __forceinline__ Task task_at(int t, int n_rows, const int* __restrict__ ptr, const int* __restrict__ rows,
                                        const int2* __restrict__ chunks, int chunk_edges) {
    Task k;
    if (t < n_rows) {
        k.row = rows[t];
        k.beg = ptr[k.row];
        k.end = ptr[k.row + 1];
        k.whole = k.first = true;
        k.chunk = -1;
    } else {
        k.chunk = t - n_rows;
        const int2 c = chunks[k.chunk];
        k.row = c.x;
        k.beg = c.y;
        const int re = ptr[c.x + 1];
        k.end = min(c.y + chunk_edges, re);
        k.whole = false;
        k.first = c.y == ptr[c.x];
    }
    return k;
}

// ---- source-major copy of the pattern -------------------------------------
// entries per source: cnt[j] += 1 (cnt zeroed); indices outside [0, N) are
// skipped here and by the scatter alike
__global__ void k_col_count(const int* __restrict__ indices, int64_t nnz, int N, int* __restrict__ cnt) {
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < nnz; e += (int64_t)gridDim.x * blockDim.x) {
        const int j = __ldg(indices + e);
        if ((unsigned)j < (unsigned)N) atomicAdd(cnt + j, 1);
    }
}

constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;

// exclusive scan of one value per thread over a kScanThreads block; *total
// receives the block's sum
__device__ __forceinline__ int block_exclusive_scan(int v, int* total) {
    __shared__ int warp_sum[kScanThreads / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sum[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int w = lane < kScanThreads / 32 ? warp_sum[lane] : 0;
#pragma unroll
        for (int o = 1; o < kScanThreads / 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kScanThreads / 32) warp_sum[lane] = w;   // inclusive warp prefix
    }
    __syncthreads();
    const int before = wid > 0 ? warp_sum[wid - 1] : 0;
    *total = warp_sum[kScanThreads / 32 - 1];
    __syncthreads();   // warp_sum is reused by the next call
    return before + x - v;
}

// per-tile sums of cnt
__global__ void __launch_bounds__(kScanThreads) k_scan_sums(const int* __restrict__ cnt, int N, int* __restrict__ tsum) {
    const int64_t base = (int64_t)blockIdx.x * kScanTile + threadIdx.x * kScanItems;
    int v = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k)
        if (base + k < N) v += cnt[base + k];
    int total;
    block_exclusive_scan(v, &total);
    if (threadIdx.x == 0) tsum[blockIdx.x] = total;
}

// exclusive scan of the tile sums in place (one block); colptr[N] = total
__global__ void __launch_bounds__(kScanThreads) k_scan_top(int* __restrict__ tsum, int n_tiles,
                                                          int* __restrict__ colptr, int N) {
    int carry = 0;
    for (int b0 = 0; b0 < n_tiles; b0 += kScanTile) {
        const int base = b0 + threadIdx.x * kScanItems;
        int x[kScanItems], v = 0;
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            x[k] = base + k < n_tiles ? tsum[base + k] : 0;
            v += x[k];
        }
        int total;
        int run = carry + block_exclusive_scan(v, &total);
#pragma unroll
        for (int k = 0; k < kScanItems; ++k) {
            if (base + k < n_tiles) tsum[base + k] = run;
            run += x[k];
        }
        carry += total;
    }
    if (threadIdx.x == 0) colptr[N] = carry;
}

// colptr[j] = cursor[j] = exclusive prefix of cnt (cnt may alias cursor)
__global__ void __launch_bounds__(kScanThreads) k_scan_apply(const int* cnt, int N, const int* __restrict__ tsum,
                                                            int* __restrict__ colptr, int* cursor) {
    const int64_t base = (int64_t)blockIdx.x * kScanTile + threadIdx.x * kScanItems;
    int x[kScanItems], v = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        x[k] = base + k < N ? cnt[base + k] : 0;
        v += x[k];
    }
    int total;
    int run = tsum[blockIdx.x] + block_exclusive_scan(v, &total);
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        if (base + k < N) {
            colptr[base + k] = run;
            cursor[base + k] = run;
        }
        run += x[k];
    }
}

// rowid[slot] = destination row of each entry, slots taken per source from
// cursor (the order within a source is that of the slot claims; the
// segment sort below makes it ascending)
__global__ void __launch_bounds__(kTaskWarps * 32)
k_csc_scatter(const int* __restrict__ indptr, const int* __restrict__ indices, const int* __restrict__ hdr,
              const int* __restrict__ rows, const int2* __restrict__ chunks, int chunk_edges, int N,
              int* __restrict__ cursor, int* __restrict__ rowid) {
    const int lane = threadIdx.x & 31;
    const int n_rows = hdr[HdrLayout::kDenseSeg] + hdr[HdrLayout::kDenseRows];   // the dense segment too
    const int n_tasks = n_rows + hdr[HdrLayout::kChunks];
    for (int t = blockIdx.x * kTaskWarps + (threadIdx.x >> 5); t < n_tasks; t += gridDim.x * kTaskWarps) {
        const Task k = task_at(t, n_rows, indptr, rows, chunks, chunk_edges);
        for (int e0 = k.beg + lane; e0 < k.end; e0 += 4 * 32) {   // four slots in flight a lane
            int j[4], at[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) j[u] = e0 + 32 * u < k.end ? __ldg(indices + e0 + 32 * u) : -1;
#pragma unroll
            for (int u = 0; u < 4; ++u) at[u] = (unsigned)j[u] < (unsigned)N ? atomicAdd(cursor + j[u], 1) : -1;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (at[u] >= 0) rowid[at[u]] = k.row;
        }
    }
}

// ---- segment sort: each source's destination rows in ascending order ------
// The slot claims of the scatter come in no fixed order; sorted segments make
// the source-major pattern, and so every sum pass 2 forms, the same on every
// run.  Bitonic sorting networks, by segment length:
//   <= 32      a warp each, one value a lane (shuffles)
//   <= 256     a warp each, eight values a lane (shuffles and registers)
//   <= 2048    a block each, in shared memory
//   longer     a block each, runs of 32768 in shared memory; runs merged
//              pairwise through `tmp` (merge path: each thread finds its share
//              of the merged output by a binary search of the two runs)
constexpr int kSortThreads = 256;
constexpr int kSortMid = 2048;      // segments a block sorts in static shared memory
constexpr int kSortRun = 32768;     // runs a block sorts in dynamic shared memory (128 KB)
constexpr int kSortBigThreads = 1024;   // threads of the blocks sorting those

// Bitonic sort of the warp's 32*R values, value index x = r*32 + lane.
template <int R>
__device__ __forceinline__ void warp_bitonic(int (&v)[R], int lane) {
#pragma unroll
    for (int k = 2; k <= 32 * R; k <<= 1) {
#pragma unroll
        for (int m = k >> 1; m > 0; m >>= 1) {
            if (m >= 32) {   // partner in register r ^ (m / 32), same lane
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int p = r ^ (m >> 5);
                    if (p > r) {
                        const bool up = ((r * 32 + lane) & k) == 0;
                        const int a = v[r], b = v[p];
                        if ((a > b) == up) { v[r] = b; v[p] = a; }
                    }
                }
            } else {         // partner in lane lane ^ m, same register
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int o = __shfl_xor_sync(0xffffffffu, v[r], m);
                    const bool lower = (lane & m) == 0, up = ((r * 32 + lane) & k) == 0;
                    v[r] = (lower == up) ? min(v[r], o) : max(v[r], o);
                }
            }
        }
    }
}

// A warp per source with lo < length <= 32*R.
template <int R>
__global__ void __launch_bounds__(256)
k_seg_sort_warp(const int* __restrict__ colptr, int N, int lo, int* __restrict__ rowid) {
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); j < N; j += warps) {
        const int beg = colptr[j], len = colptr[j + 1] - beg;
        if (len <= lo || len > 32 * R) continue;   // uniform over the warp
        int v[R];
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = r * 32 + lane < len ? rowid[beg + r * 32 + lane] : 0x7fffffff;
        warp_bitonic<R>(v, lane);
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (r * 32 + lane < len) rowid[beg + r * 32 + lane] = v[r];
    }
}

// position in the merge of sorted a[0, na) and b[0, nb) at which output
// index d falls: the number of elements taken from a (ties: a first)
__device__ __forceinline__ int merge_split(const int* a, int na, const int* b, int nb, int d) {
    int lo = max(0, d - nb), hi = min(d, na);
    while (lo < hi) {
        const int m = (lo + hi) >> 1;
        if (a[m] <= b[d - m - 1]) lo = m + 1;
        else hi = m;
    }
    return lo;
}

// Bitonic sort of buf[0, p2) (p2 a power of two) by the block's THREADS threads.
template <int THREADS>
__device__ __forceinline__ void block_bitonic(int* buf, int p2) {
    for (int k = 2; k <= p2; k <<= 1) {
        for (int m = k >> 1; m > 0; m >>= 1) {
            const int lm = __ffs(m) - 1;   // m = 2^lm
            for (int i = threadIdx.x; i < p2 / 2; i += THREADS) {
                // the i-th pair of this step: lower index x, partner x + m
                const int x = ((i >> lm) << (lm + 1)) + (i & (m - 1));
                const int a = buf[x], b = buf[x + m];
                const bool up = (x & k) == 0;
                if ((a > b) == up) {
                    buf[x] = b;
                    buf[x + m] = a;
                }
            }
            __syncthreads();
        }
    }
}

// List positions, in a binning's row list (heaviest bucket first), of the
// rows of degree lo+1 .. hi (hi = 0: no upper limit): [first, last).
__device__ __forceinline__ int2 bucket_span(const int* hdr, int lo, int hi) {
    auto end_of = [&](int b) { return hdr[HdrLayout::kOffset + b] + hdr[HdrLayout::kCount + b]; };
    const int last = end_of(bucket_of(lo + 1));
    const int first = hi > 0 && hi + 1 <= 0x3fffffff ? end_of(bucket_of(hi + 1)) : 0;
    return make_int2(hi > 0 ? first : 0, last);
}

// A block per source of degree lo+1 .. hi (hi = 0: any above lo), taken from
// the source binning: its split sources (the longs list) and the sources of
// its row list's buckets in that degree range; runs of RUN values sorted in
// shared memory (static for RUN <= kSortMid, else dynamic), merged pairwise
// through tmp when the segment is longer than one run.
template <int RUN, int THREADS>
__global__ void __launch_bounds__(THREADS)
k_seg_sort_block(const int* __restrict__ colptr, const int* __restrict__ hdr, const int* __restrict__ cols,
                 const int2* __restrict__ longs, int lo, int hi, int* __restrict__ rowid, int* __restrict__ tmp) {
    extern __shared__ int dyn[];
    __shared__ int stat[RUN <= kSortMid ? RUN : 1];
    int* buf = RUN <= kSortMid ? stat : dyn;
    const int n_long = hdr[HdrLayout::kLong];
    const int2 span = bucket_span(hdr, lo, hi);
    const int n_sel = n_long + (span.y - span.x);
    for (int t = blockIdx.x; t < n_sel; t += gridDim.x) {
        const int j = t < n_long ? longs[t].x : cols[span.x + t - n_long];
        const int beg = colptr[j], len = colptr[j + 1] - beg;
        if (len <= lo || (hi > 0 && len > hi)) continue;   // uniform over the block
        for (int r0 = 0; r0 < len; r0 += RUN) {
            const int n = min(RUN, len - r0);
            int p2 = 64;
            while (p2 < n) p2 <<= 1;
            for (int i = threadIdx.x; i < p2; i += THREADS) buf[i] = i < n ? rowid[beg + r0 + i] : 0x7fffffff;
            __syncthreads();
            block_bitonic<THREADS>(buf, p2);
            for (int i = threadIdx.x; i < n; i += THREADS) rowid[beg + r0 + i] = buf[i];
            __syncthreads();
        }
        // merge runs pairwise: width w -> 2w, alternating rowid and tmp
        int* src = rowid + beg;
        int* dst = tmp + beg;
        for (int w = RUN; w < len; w <<= 1) {
            for (int a0 = 0; a0 < len; a0 += 2 * w) {
                const int na = min(w, len - a0), nb = max(0, min(w, len - a0 - w));
                const int tot = na + nb;
                const int* A = src + a0;
                const int* B = A + na;
                const int per = (tot + THREADS - 1) / THREADS;
                const int d0 = min(tot, static_cast<int>(threadIdx.x) * per), d1 = min(tot, d0 + per);
                int ia = merge_split(A, na, B, nb, d0);
                int ib = d0 - ia;
                for (int d = d0; d < d1; ++d) {
                    const bool take_a = ib >= nb || (ia < na && A[ia] <= B[ib]);
                    dst[a0 + d] = take_a ? A[ia++] : B[ib++];
                }
            }
            __syncthreads();
            int* t = src;
            src = dst;
            dst = t;
        }
        if (src != rowid + beg)   // the last merge landed in tmp
            for (int i = threadIdx.x; i < len; i += THREADS) rowid[beg + i] = src[i];
        __syncthreads();
    }
}

// Both passes give each lane group (G lanes, E features a lane) a task of
// its own: the warp takes S = 32 / G consecutive tasks -- split-row chunks
// first, then the rows from the heaviest bucket down, so the S tasks have
// nearly the same length -- and walks them side by side in one warp-uniform
// loop, U entries a group per step with the next step's indices in flight.
// A group whose task is shorter (or absent) runs its remaining steps with
// every load predicated off.
__device__ __forceinline__ Task group_task(int t, int n_tasks, int n_chunks, const int* __restrict__ ptr,
                                           const int* __restrict__ rows, const int2* __restrict__ chunks,
                                           int chunk_edges) {
    if (t >= n_tasks) return Task{-1, 0, 0, false, false};
    if (t < n_chunks) return task_at(n_tasks + t - n_chunks, n_tasks - n_chunks, ptr, rows, chunks, chunk_edges);
    return task_at(t - n_chunks, n_tasks - n_chunks, ptr, rows, chunks, chunk_edges);
}

// ---- pass 1: by destination row ------------------------------------------
// A chunk of a split row stores its partial sum in part_dq[chunk]; the
// combine adds a row's chunks in chunk order.
template <typename T, int E, int U>
__global__ void __launch_bounds__(kPassWarps * 32, pass_min_blocks<T, E, 1>())
k_bwd_dq(const int* __restrict__ indptr, const int* __restrict__ indices, const int* __restrict__ hdr,
         const int* __restrict__ rows, const int2* __restrict__ chunks, int chunk_edges, const T* __restrict__ Q,
         const T* __restrict__ K, const T* __restrict__ V, const T* __restrict__ dO, const float* __restrict__ O,
         const float* __restrict__ L, float2* __restrict__ LD, float* __restrict__ dQ, float* __restrict__ part_dq,
         int H, int G, int lph, float scale) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gl = lane & (G - 1), slot = lane / G, S = 32 / G;
    const int HD = G * E;
    const int head = gl / lph;
    const bool head_lead = gl % lph == 0;
    const float sl2 = scale * kLog2e;
    auto reduce = [&](float v) {
        for (int o = 1; o < lph; o <<= 1) v += __shfl_xor_sync(full, v, o);
        return v;
    };
    const int n_chunks = hdr[HdrLayout::kChunks];
    const int n_tasks = hdr[HdrLayout::kDenseSeg] + hdr[HdrLayout::kDenseRows] + n_chunks;
    for (int t0 = (blockIdx.x * kPassWarps + warp) * S; t0 < n_tasks; t0 += gridDim.x * kPassWarps * S) {
        Task k = group_task(t0 + slot, n_tasks, n_chunks, indptr, rows, chunks, chunk_edges);
        const int64_t off = static_cast<int64_t>(k.row) * HD + gl * E;
        const int deg = k.row >= 0 ? indptr[k.row + 1] - indptr[k.row] : 0;
        if (k.row >= 0 && deg <= 1) {   // never split: dQ_i = 0; a row of one entry is marked for pass 2
            float z[E];
#pragma unroll
            for (int u = 0; u < E; ++u) z[u] = 0.f;
            store_vec<E>(dQ + off, z, 0.f);
            if (deg == 1 && head_lead) LD[static_cast<int64_t>(k.row) * H + head] = make_float2(INFINITY, 0.f);
        }
        const bool walk = deg > 1;
        if (!walk) k.beg = k.end = 0;
        Raw<T, E> q, g;
        Raw<float, E> o;
        float lse = 0.f;
        if (walk) {
            q.load(Q + off);
            g.load(dO + off);
            o.load(O + off);
            lse = L[static_cast<int64_t>(k.row) * H + head];
        } else {
            q.zero();
            g.zero();
            o.zero();
        }
        // Dlt = dO_i . O_i (this head)
        float dl;
        {
            float x = 0.f, y = 0.f;
#pragma unroll
            for (int u = 0; u < E; u += 2) {
                x = fmaf(g[u], o[u], x);
                y = fmaf(g[u + 1], o[u + 1], y);
            }
            dl = reduce(x + y);
        }
        if (walk && k.first && head_lead) LD[static_cast<int64_t>(k.row) * H + head] = make_float2(lse, dl);
        float dq[E];
#pragma unroll
        for (int u = 0; u < E; ++u) dq[u] = 0.f;
        const int steps = __reduce_max_sync(full, (k.end - k.beg + U - 1) / U);
        int jn[U];
#pragma unroll
        for (int u = 0; u < U; ++u) jn[u] = k.beg + u < k.end ? __ldg(indices + k.beg + u) : -1;
        for (int it = 0; it < steps; ++it) {
            const int b = k.beg + it * U;
            int j[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                j[u] = jn[u];
                jn[u] = b + U + u < k.end ? __ldg(indices + b + U + u) : -1;
            }
            Raw<T, E> kx[U], vx[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (j[u] >= 0) {
                    kx[u].load(K + static_cast<int64_t>(j[u]) * HD + gl * E);
                    vx[u].load(V + static_cast<int64_t>(j[u]) * HD + gl * E);
                } else {
                    kx[u].zero();
                    vx[u].zero();
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float s = reduce(q.dot(kx[u])), dp = reduce(g.dot(vx[u]));
                const float p = exp2f(s * sl2 - lse);
                const float ds = j[u] >= 0 ? p * (dp - dl) : 0.f;
                kx[u].axpy(dq, ds);
            }
        }
        if (walk) {
            if (k.whole) store_vec<E>(dQ + off, dq, scale);
            else store_vec<E>(part_dq + static_cast<int64_t>(k.chunk) * HD + gl * E, dq, scale);
        }
    }
}

// ---- pass 2: by source node ------------------------------------------------
template <typename T, int E, int U>
__global__ void __launch_bounds__(kPassWarps * 32, pass_min_blocks<T, E, 2>())
k_bwd_dkv(const int* __restrict__ colptr, const int* __restrict__ rowid, const int* __restrict__ hdr,
          const int* __restrict__ cols, const int2* __restrict__ chunks, int chunk_edges,
          const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V, const T* __restrict__ dO,
          const float2* __restrict__ LD, float* __restrict__ dK, float* __restrict__ dV, float* __restrict__ part_dk,
          float* __restrict__ part_dv, int H, int G, int lph, float scale) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gl = lane & (G - 1), slot = lane / G, S = 32 / G;
    const int HD = G * E;
    const int head = gl / lph;
    const float sl2 = scale * kLog2e;
    auto reduce = [&](float v) {
        for (int o = 1; o < lph; o <<= 1) v += __shfl_xor_sync(full, v, o);
        return v;
    };
    const int n_chunks = hdr[HdrLayout::kChunks];
    const int n_tasks = hdr[HdrLayout::kDenseSeg] + hdr[HdrLayout::kDenseRows] + n_chunks;
    for (int t0 = (blockIdx.x * kPassWarps + warp) * S; t0 < n_tasks; t0 += gridDim.x * kPassWarps * S) {
        const Task k = group_task(t0 + slot, n_tasks, n_chunks, colptr, cols, chunks, chunk_edges);
        const int64_t off = static_cast<int64_t>(k.row) * HD + gl * E;
        float dk[E], dv[E];
#pragma unroll
        for (int u = 0; u < E; ++u) dk[u] = dv[u] = 0.f;
        Raw<T, E> kj, vj;
        if (k.end > k.beg) {
            kj.load(K + off);
            vj.load(V + off);
        } else {
            kj.zero();
            vj.zero();
        }
        const int steps = __reduce_max_sync(full, (k.end - k.beg + U - 1) / U);
        int in[U];
#pragma unroll
        for (int u = 0; u < U; ++u) in[u] = k.beg + u < k.end ? __ldg(rowid + k.beg + u) : -1;
        for (int it = 0; it < steps; ++it) {
            const int b = k.beg + it * U;
            int i[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                i[u] = in[u];
                in[u] = b + U + u < k.end ? __ldg(rowid + b + U + u) : -1;
            }
            Raw<T, E> qx[U], gx[U];
            float2 ld[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (i[u] >= 0) {
                    qx[u].load(Q + static_cast<int64_t>(i[u]) * HD + gl * E);
                    gx[u].load(dO + static_cast<int64_t>(i[u]) * HD + gl * E);
                    ld[u] = __ldg(LD + static_cast<int64_t>(i[u]) * H + head);
                } else {
                    qx[u].zero();
                    gx[u].zero();
                    ld[u] = make_float2(0.f, 0.f);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float s = reduce(qx[u].dot(kj)), dp = reduce(gx[u].dot(vj));
                const bool single = ld[u].x == INFINITY;
                float p = single ? 1.f : exp2f(s * sl2 - ld[u].x);
                float ds = single ? 0.f : p * (dp - ld[u].y);
                if (i[u] < 0) p = ds = 0.f;
                qx[u].axpy(dk, ds);
                gx[u].axpy(dv, p);
            }
        }
        if (k.row >= 0) {
            if (k.whole) {
                store_vec<E>(dK + off, dk, scale);
                store_vec<E>(dV + off, dv, 1.f);
            } else {   // a chunk of a split source: its partial sums
                const int64_t po = static_cast<int64_t>(k.chunk) * HD + gl * E;
                store_vec<E>(part_dk + po, dk, scale);
                store_vec<E>(part_dv + po, dv, 1.f);
            }
        }
    }
}

// ---- split rows and sources: their chunks' partial sums, in chunk order ----
// A warp per split row (longs: (row, first chunk)); out[row] = sum over the
// row's chunks of part[chunk], a float4 a lane.  Up to two arrays at once
// (dK and dV of a split source).
__global__ void __launch_bounds__(256)
k_bwd_chunk_sum(const int* __restrict__ ptr, const int* __restrict__ hdr, const int2* __restrict__ longs,
                int chunk_edges, int HD, const float* __restrict__ part0, float* __restrict__ out0,
                const float* __restrict__ part1, float* __restrict__ out1) {
    const int lane = threadIdx.x & 31;
    const int n_long = hdr[HdrLayout::kLong];
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int li = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); li < n_long; li += warps) {
        const int2 lr = longs[li];
        const int nch = (ptr[lr.x + 1] - ptr[lr.x] + chunk_edges - 1) / chunk_edges;
        for (int q = lane; q < HD / 4; q += 32) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            for (int c = 0; c < nch; ++c) {
                const int64_t o = static_cast<int64_t>(lr.y + c) * HD;
                const float4 x = reinterpret_cast<const float4*>(part0 + o)[q];
                a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
                if (part1) {
                    const float4 y = reinterpret_cast<const float4*>(part1 + o)[q];
                    b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
                }
            }
            reinterpret_cast<float4*>(out0 + static_cast<int64_t>(lr.x) * HD)[q] = a;
            if (part1) reinterpret_cast<float4*>(out1 + static_cast<int64_t>(lr.x) * HD)[q] = b;
        }
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

// Features a lane holds (E) and lanes a node row spans (G = H D / E): 16
// features where the row is 16 to 512 wide and splits into whole heads of
// power-of-two lane counts, else the row over the whole warp.
static bool bwd_layout(int H, int D, int* E, int* G) {
    auto pow2 = [](int x) { return x > 0 && (x & (x - 1)) == 0; };
    const int HD = H * D;
    for (int e : {16, 32}) {
        if (HD % e == 0 && D % e == 0 && pow2(HD / e) && HD / e <= 32 && pow2(D / e)) {
            *E = e;
            *G = HD / e;
            return true;
        }
    }
    if (HD % 32 != 0) return false;
    const int e = HD / 32;
    if ((e != 4 && e != 8) || D % e != 0 || !pow2(D / e)) return false;
    *E = e;
    *G = 32;
    return true;
}

bool bwd_tasks_supported(int H, int D, gtattn_dtype dtype, const void* const* ptrs, int n_ptrs) {
    int E, G;
    if (!bwd_layout(H, D, &E, &G)) return false;
    (void)dtype;
    uintptr_t al = 0;
    for (int i = 0; i < n_ptrs; ++i) al |= reinterpret_cast<uintptr_t>(ptrs[i]);
    return (al & 15u) == 0;
}

int64_t bwd_scan_tiles(int64_t N) { return (N + kScanTile - 1) / kScanTile; }

// resident blocks of `kernel` (blocks of `warps` warps) on the whole GPU,
// cached per kernel, capped by the tasks there can be (at least one a warp)
template <typename Kern>
static int task_grid(Kern kernel, int task_bound, int warps) {
    static std::mutex mu;
    static std::unordered_map<const void*, int> cache;
    int grid;
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(reinterpret_cast<const void*>(kernel));
        if (it != cache.end()) {
            grid = it->second;
        } else {
            int per_sm = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, warps * 32, 0) != cudaSuccess ||
                per_sm < 1)
                per_sm = 1;
            grid = per_sm * num_sms();
            cache[reinterpret_cast<const void*>(kernel)] = grid;
        }
    }
    const int64_t need = (static_cast<int64_t>(task_bound) + warps - 1) / warps;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(grid, need)));
}

gtattn_status build_csc(const int* indptr, const int* indices, const TaskLists& L, int N, int64_t nnz,
                        int* colptr, int* cursor, int* tsum, int* rowid, int* tmp, const TaskLists& C,
                        int long_min, cudaStream_t s) {
    GT_CUDA(cudaMemsetAsync(cursor, 0, sizeof(int) * static_cast<size_t>(N), s));
    if (nnz > 0) {
        const int64_t want = (nnz + 255) / 256;
        const int blocks = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(num_sms()) * 8));
        k_col_count<<<blocks, 256, 0, s>>>(indices, nnz, N, cursor);
        GT_CUDA(cudaGetLastError());
    }
    const int nt = static_cast<int>(bwd_scan_tiles(N));
    k_scan_sums<<<nt, kScanThreads, 0, s>>>(cursor, N, tsum);
    GT_CUDA(cudaGetLastError());
    k_scan_top<<<1, kScanThreads, 0, s>>>(tsum, nt, colptr, N);
    GT_CUDA(cudaGetLastError());
    k_scan_apply<<<nt, kScanThreads, 0, s>>>(cursor, N, tsum, colptr, cursor);
    GT_CUDA(cudaGetLastError());
    const int grid = task_grid(k_csc_scatter, row_task_bound(N, nnz, L.chunk_edges), kTaskWarps);
    k_csc_scatter<<<grid, kTaskWarps * 32, 0, s>>>(indptr, indices, L.hdr, L.rows, L.chunks, L.chunk_edges, N,
                                                   cursor, rowid);
    GT_CUDA(cudaGetLastError());
    // the source binning, whose degree buckets pick the segments of each sort class
    GT_TRY(bin_rows(colptr, N, long_min, C.chunk_edges, nullptr, const_cast<int*>(C.hdr), const_cast<int*>(C.rows),
                    const_cast<int2*>(C.chunks), const_cast<int2*>(C.longs), s));
    if (nnz > 0 && N > 0) {   // segment sort, by length class
        const int wg = static_cast<int>(std::min<int64_t>((N + 7) / 8, static_cast<int64_t>(num_sms()) * 16));
        k_seg_sort_warp<1><<<wg, 256, 0, s>>>(colptr, N, 1, rowid);
        k_seg_sort_warp<8><<<wg, 256, 0, s>>>(colptr, N, 32, rowid);
        k_seg_sort_block<kSortMid, kSortThreads><<<num_sms() * 8, kSortThreads, 0, s>>>(colptr, C.hdr, C.rows,
                                                                                        C.longs, 256, kSortMid,
                                                                                        rowid, tmp);
        GT_CUDA(cudaGetLastError());
        static std::mutex mu;
        static bool set[64] = {};
        int dev = 0;
        GT_CUDA(cudaGetDevice(&dev));
        {
            std::lock_guard<std::mutex> g(mu);
            if (dev < 0 || dev >= 64 || !set[dev]) {
                GT_CUDA(cudaFuncSetAttribute(k_seg_sort_block<kSortRun, kSortBigThreads>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(sizeof(int) * kSortRun)));
                if (dev >= 0 && dev < 64) set[dev] = true;
            }
        }
        k_seg_sort_block<kSortRun, kSortBigThreads><<<num_sms(), kSortBigThreads, sizeof(int) * kSortRun, s>>>(
            colptr, C.hdr, C.rows, C.longs, kSortMid, 0, rowid, tmp);
        GT_CUDA(cudaGetLastError());
    }
    return GTATTN_OK;
}

gtattn_status launch_bwd_passes(const int* indptr, const int* indices, const TaskLists& rows, const int* colptr,
                                const int* rowid, const TaskLists& cols, const void* Q, const void* K, const void* V,
                                const void* dO, const float* O, const float* lse, float2* LD, float* dQ, float* dK,
                                float* dV, float* part_dq, float* part_dk, float* part_dv, int N, int64_t nnz, int H,
                                int D, float scale, gtattn_dtype dtype, cudaStream_t s) {
    int E = 0, G = 0;
    if (!bwd_layout(H, D, &E, &G)) return GTATTN_ERR_UNSUPPORTED;
    const int lph = D / E;
    const int bound_r = row_task_bound(N, nnz, rows.chunk_edges), bound_c = row_task_bound(N, nnz, cols.chunk_edges);
    auto go = [&](auto tag, auto e_tag) -> cudaError_t {
        using T = decltype(tag);
        constexpr int EE = decltype(e_tag)::value;
        // entries in flight per lane group: the registers of U packed rows
        constexpr int U = sizeof(T) == 2 ? (EE <= 16 ? 2 : 1) : (EE <= 8 ? 2 : 1);
        const T* q = static_cast<const T*>(Q);
        const T* k = static_cast<const T*>(K);
        const T* v = static_cast<const T*>(V);
        const T* g = static_cast<const T*>(dO);
        auto k1 = k_bwd_dq<T, EE, U>;
        k1<<<task_grid(k1, bound_r, kPassWarps), kPassWarps * 32, 0, s>>>(
            indptr, indices, rows.hdr, rows.rows, rows.chunks, rows.chunk_edges, q, k, v, g, O, lse, LD, dQ, part_dq,
            H, G, lph, scale);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        auto k2 = k_bwd_dkv<T, EE, U>;
        k2<<<task_grid(k2, bound_c, kPassWarps), kPassWarps * 32, 0, s>>>(
            colptr, rowid, cols.hdr, cols.rows, cols.chunks, cols.chunk_edges, q, k, v, g, LD, dK, dV, part_dk,
            part_dv, H, G, lph, scale);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        // split rows and sources: their chunks summed in chunk order
        const int cg = num_sms() * 4;
        k_bwd_chunk_sum<<<cg, 256, 0, s>>>(indptr, rows.hdr, rows.longs, rows.chunk_edges, G * EE, part_dq, dQ,
                                           nullptr, nullptr);
        k_bwd_chunk_sum<<<cg, 256, 0, s>>>(colptr, cols.hdr, cols.longs, cols.chunk_edges, G * EE, part_dk, dK,
                                           part_dv, dV);
        return cudaGetLastError();
    };
    using B = __nv_bfloat16;
    using I4 = std::integral_constant<int, 4>;
    using I8 = std::integral_constant<int, 8>;
    using I16 = std::integral_constant<int, 16>;
    using I32 = std::integral_constant<int, 32>;
    cudaError_t e;
    if (dtype == GTATTN_F32) {
        e = E == 4 ? go(float{}, I4{}) : E == 8 ? go(float{}, I8{}) : E == 16 ? go(float{}, I16{}) : go(float{}, I32{});
    } else {
        e = E == 4 ? go(B{}, I4{}) : E == 8 ? go(B{}, I8{}) : E == 16 ? go(B{}, I16{}) : go(B{}, I32{});
    }
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

}  // namespace gt
