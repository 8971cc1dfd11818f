// plan.cu -- degree binning (the plan), dense-block detection, CSR helpers.
//
// The pages define only the operation (sparse attention over the stored
// entries of each row); how rows are grouped for the GPU is this library's
// design: rows are counted into degree buckets, laid out from the heaviest
// bucket down, rows above a threshold are cut into fixed-size chunks whose
// partial softmax states a second kernel combines, and complete blocks can
// be routed to the dense tensor-core kernel.
#include "plan.cuh"

#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

namespace gt {

// ---------------------------------------------------------------------------
// binning kernels
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool is_long(int deg, int long_min) { return deg > 0 && deg > long_min; }

// The three binning steps as block-level functions over blocks bid of nb,
// run as three kernels (large graphs) or all three by one block (small ones).
__device__ __forceinline__ void bin_count_part(const int* __restrict__ indptr, int N, int long_min, int chunk,
                                               const int* __restrict__ dense_flag, int* __restrict__ hdr, int bid,
                                               int nb) {
    __shared__ int hist[kNumBuckets];
    __shared__ int s_long, s_chunks, s_dense, s_max, s_big;
    for (int b = threadIdx.x; b < kNumBuckets; b += blockDim.x) hist[b] = 0;
    if (threadIdx.x == 0) { s_long = 0; s_chunks = 0; s_dense = 0; s_max = 0; s_big = 0; }
    __syncthreads();
    for (int i = bid * blockDim.x + threadIdx.x; i < N; i += nb * blockDim.x) {
        int deg = indptr[i + 1] - indptr[i];
        atomicMax(&s_max, deg);
        if (dense_flag && dense_flag[i]) {
            atomicAdd(&s_dense, 1);
        } else if (is_long(deg, long_min)) {
            const int nch = (deg + chunk - 1) / chunk;
            atomicAdd(&s_long, 1);
            atomicAdd(&s_chunks, nch);
            if (nch > kBigChunks) atomicAdd(&s_big, 1);
        } else {
            atomicAdd(&hist[bucket_of(deg)], 1);
        }
    }
    __syncthreads();
    for (int b = threadIdx.x; b < kNumBuckets; b += blockDim.x)
        if (hist[b]) atomicAdd(&hdr[HdrLayout::kCount + b], hist[b]);
    if (threadIdx.x == 0) {
        if (s_long) atomicAdd(&hdr[HdrLayout::kLong], s_long);
        if (s_chunks) atomicAdd(&hdr[HdrLayout::kChunks], s_chunks);
        if (s_dense) atomicAdd(&hdr[HdrLayout::kDenseRows], s_dense);
        if (s_big) atomicAdd(&hdr[HdrLayout::kBig], s_big);
        atomicMax(&hdr[HdrLayout::kMaxDeg], s_max);
    }
}

__global__ void k_bin_count(const int* __restrict__ indptr, int N, int long_min, int chunk,
                            const int* __restrict__ dense_flag, int* __restrict__ hdr) {
    bin_count_part(indptr, N, long_min, chunk, dense_flag, hdr, blockIdx.x, gridDim.x);
}

__device__ __forceinline__ void bin_offsets_part(int* hdr) {   // one thread
    int off = 0;
    for (int b = kNumBuckets - 1; b >= 0; --b) {
        hdr[HdrLayout::kOffset + b] = off;
        off += hdr[HdrLayout::kCount + b];
    }
    hdr[HdrLayout::kDenseSeg] = off;
}

__global__ void k_bin_offsets(int* hdr) {
    if (threadIdx.x == 0 && blockIdx.x == 0) bin_offsets_part(hdr);
}

// Scatter of rows into the bucket lists, the split-row list and the dense
// segment, one tile of blockDim rows at a time: the tile's rows are counted
// per key in shared memory, each key present reserves its range with one
// global atomic, and rows take their place from shared-memory cursors (about
// 25 global atomics per 512 rows instead of one per warp and key).
constexpr int kScatterThreads = 512;
// keys: buckets, split rows of at most kBigChunks chunks (NB), the dense
// segment (NB + 2), split rows of more chunks (NB + 3); NB + 1 is unused (its
// cursor word counts chunks)
constexpr int kKeyBig = kNumBuckets + 3;
constexpr int kScatterKeys = kNumBuckets + 4;
__device__ __forceinline__ int cursor_word(int key) {
    return key == kKeyBig ? HdrLayout::kCurBig : HdrLayout::kCursor + key;
}

__device__ __forceinline__ void bin_scatter_part(const int* __restrict__ indptr, int N, int long_min, int chunk,
                                                 const int* __restrict__ dense_flag, int* __restrict__ hdr,
                                                 int* __restrict__ rows, int2* __restrict__ chunks,
                                                 int2* __restrict__ longs, int bid, int nb) {
    __shared__ int cnt[kScatterKeys], base[kScatterKeys];
    __shared__ int s_chunks, s_chunk_base;
    for (int t0 = bid * blockDim.x; t0 < N; t0 += nb * blockDim.x) {
        for (int k = threadIdx.x; k < kScatterKeys; k += blockDim.x) cnt[k] = 0;
        if (threadIdx.x == 0) s_chunks = 0;
        __syncthreads();
        const int i = t0 + threadIdx.x;
        int key = -1, local = 0, beg = 0, nch = 0, chunk_local = 0;
        if (i < N) {
            beg = indptr[i];
            const int deg = indptr[i + 1] - beg;
            // key: bucket id, NB (split row) or NB+2 (dense segment); the
            // cursors are laid out the same way
            if (dense_flag && dense_flag[i]) key = kNumBuckets + 2;
            else if (is_long(deg, long_min)) key = (deg + chunk - 1) / chunk > kBigChunks ? kKeyBig : kNumBuckets;
            else key = bucket_of(deg);
            local = atomicAdd(&cnt[key], 1);
            if (key == kNumBuckets || key == kKeyBig) {
                nch = (deg + chunk - 1) / chunk;
                chunk_local = atomicAdd(&s_chunks, nch);
            }
        }
        __syncthreads();
        for (int k = threadIdx.x; k < kScatterKeys; k += blockDim.x)
            if (cnt[k]) base[k] = atomicAdd(&hdr[cursor_word(k)], cnt[k]);
        if (threadIdx.x == 0 && s_chunks) s_chunk_base = atomicAdd(&hdr[HdrLayout::kCurChunk], s_chunks);
        __syncthreads();
        if (key >= 0) {
            const int pos = base[key] + local;
            if (key < kNumBuckets) {
                rows[hdr[HdrLayout::kOffset + key] + pos] = i;
            } else if (key == kNumBuckets || key == kKeyBig) {
                // split rows of many chunks first, then the others
                const int c0 = s_chunk_base + chunk_local;
                longs[key == kKeyBig ? pos : hdr[HdrLayout::kBig] + pos] = make_int2(i, c0);
                for (int c = 0; c < nch; ++c) chunks[c0 + c] = make_int2(i, beg + c * chunk);
            } else {
                rows[hdr[HdrLayout::kDenseSeg] + pos] = i;
            }
        }
        __syncthreads();   // cnt / base are reset for the next tile
    }
}

__global__ void __launch_bounds__(kScatterThreads)
k_bin_scatter(const int* __restrict__ indptr, int N, int long_min, int chunk,
              const int* __restrict__ dense_flag, int* __restrict__ hdr,
              int* __restrict__ rows, int2* __restrict__ chunks, int2* __restrict__ longs) {
    bin_scatter_part(indptr, N, long_min, chunk, dense_flag, hdr, rows, chunks, longs, blockIdx.x, gridDim.x);
}

// Small graphs (N <= kBinSmallRows): one block of kSmallThreads bins every
// row in one launch.  Each thread keeps kSmallRowsPerThread rows in
// registers (their indptr loads all in flight at once); counts, offsets and
// cursors stay in shared memory, and the header is written whole (the same
// words the three-kernel path leaves), so no memset is needed.
constexpr int kSmallThreads = 1024;
constexpr int kSmallRowsPerThread = kBinSmallRows / kSmallThreads;
static_assert(kSmallRowsPerThread * kSmallThreads == kBinSmallRows, "small binning covers kBinSmallRows");

__global__ void __launch_bounds__(kSmallThreads)
k_bin_small(const int* __restrict__ indptr, int N, int long_min, int chunk, int* __restrict__ hdr,
            int* __restrict__ rows, int2* __restrict__ chunks, int2* __restrict__ longs) {
    // rows per bucket, then split rows of at most kBigChunks chunks, then the others
    __shared__ int cnt[kNumBuckets + 2];
    __shared__ int off[kNumBuckets];
    __shared__ int s_chunks, s_max;
    for (int k = threadIdx.x; k < kNumBuckets + 2; k += blockDim.x) cnt[k] = 0;
    if (threadIdx.x == 0) { s_chunks = 0; s_max = 0; }
    __syncthreads();
    int beg[kSmallRowsPerThread], deg[kSmallRowsPerThread];
#pragma unroll
    for (int r = 0; r < kSmallRowsPerThread; ++r) {
        const int i = threadIdx.x + r * blockDim.x;
        beg[r] = i < N ? indptr[i] : 0;
        deg[r] = i < N ? indptr[i + 1] - beg[r] : -1;
    }
    int key[kSmallRowsPerThread], pos[kSmallRowsPerThread], c0[kSmallRowsPerThread];
#pragma unroll
    for (int r = 0; r < kSmallRowsPerThread; ++r) {
        key[r] = -1;
        pos[r] = c0[r] = 0;
        if (deg[r] < 0) continue;
        atomicMax(&s_max, deg[r]);
        const int nch = (deg[r] + chunk - 1) / chunk;
        key[r] = is_long(deg[r], long_min) ? (nch > kBigChunks ? kNumBuckets + 1 : kNumBuckets) : bucket_of(deg[r]);
        pos[r] = atomicAdd(&cnt[key[r]], 1);
        if (key[r] >= kNumBuckets) c0[r] = atomicAdd(&s_chunks, nch);
    }
    __syncthreads();
    if (threadIdx.x == 0) {   // bucket lists laid out from the heaviest bucket down
        int o = 0;
        for (int b = kNumBuckets - 1; b >= 0; --b) {
            off[b] = o;
            o += cnt[b];
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < HdrLayout::kWords; k += blockDim.x) {
        int v = 0;
        if (k == HdrLayout::kLong) v = cnt[kNumBuckets] + cnt[kNumBuckets + 1];
        else if (k == HdrLayout::kCurLong) v = cnt[kNumBuckets];
        else if (k == HdrLayout::kBig || k == HdrLayout::kCurBig) v = cnt[kNumBuckets + 1];
        else if (k == HdrLayout::kChunks || k == HdrLayout::kCurChunk) v = s_chunks;
        else if (k == HdrLayout::kMaxDeg) v = s_max;
        else if (k >= HdrLayout::kCount && k < HdrLayout::kCount + kNumBuckets) v = cnt[k - HdrLayout::kCount];
        else if (k >= HdrLayout::kOffset && k < HdrLayout::kOffset + kNumBuckets) v = off[k - HdrLayout::kOffset];
        else if (k >= HdrLayout::kCursor && k < HdrLayout::kCursor + kNumBuckets) v = cnt[k - HdrLayout::kCursor];
        else if (k == HdrLayout::kDenseSeg) v = off[0] + cnt[0];
        hdr[k] = v;
    }
#pragma unroll
    for (int r = 0; r < kSmallRowsPerThread; ++r) {
        const int i = threadIdx.x + r * blockDim.x;
        if (key[r] < 0) continue;
        if (key[r] < kNumBuckets) {
            rows[off[key[r]] + pos[r]] = i;
        } else {   // split rows of many chunks first, then the others
            longs[key[r] == kNumBuckets + 1 ? pos[r] : cnt[kNumBuckets + 1] + pos[r]] = make_int2(i, c0[r]);
            const int nch = (deg[r] + chunk - 1) / chunk;
            for (int c = 0; c < nch; ++c) chunks[c0[r] + c] = make_int2(i, beg[r] + c * chunk);
        }
    }
}
static_assert(HdrLayout::kCurLong == HdrLayout::kCursor + kNumBuckets, "cursor layout");
static_assert(HdrLayout::kCurDense == HdrLayout::kCursor + kNumBuckets + 2, "cursor layout");

// ---------------------------------------------------------------------------
// dense-block detection: a block is rows r0..r0+n-1 whose entries are exactly
// r0, r0+1, ..., r0+n-1 (a complete graph with self-loops, sorted), n at
// least kDenseTile (the kernel masks a ragged last tile).
// ---------------------------------------------------------------------------
__global__ void k_dense_candidates(const int* __restrict__ indptr, const int* __restrict__ indices,
                                   int N, int* __restrict__ cand) {
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < N; i += warps) {
        int beg = indptr[i], deg = indptr[i + 1] - beg;
        int first = -1;
        if (deg >= kDenseTile) {
            int f = indices[beg];
            bool ok = (i >= f) && (i < f + deg);
            for (int k = lane; ok && k < deg; k += 32) ok = indices[beg + k] == f + k;
            ok = __all_sync(0xffffffffu, ok);
            if (ok) first = f;
        }
        if (lane == 0) cand[i] = first;
    }
}

__global__ void k_dense_blocks(const int* __restrict__ indptr, int N, const int* __restrict__ cand,
                               int* __restrict__ hdr, int2* __restrict__ blocks,
                               int* __restrict__ dense_flag) {
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < N; r += warps) {
        if (cand[r] != r) continue;
        int n = indptr[r + 1] - indptr[r];
        if ((long long)r + n > N) continue;
        bool ok = true;
        for (int k = lane; ok && k < n; k += 32)
            ok = cand[r + k] == r && (indptr[r + k + 1] - indptr[r + k]) == n;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) continue;
        int b = 0;
        if (lane == 0) b = atomicAdd(&hdr[HdrLayout::kDenseBlocks], 1);
        b = __shfl_sync(0xffffffffu, b, 0);
        if (lane == 0) blocks[b] = make_int2(r, n);
        for (int k = lane; k < n; k += 32) dense_flag[r + k] = 1;
    }
}

// ---------------------------------------------------------------------------
// host: bin rows into caller-provided arrays (no host synchronisation)
// ---------------------------------------------------------------------------
static int grid_for(int64_t work, int threads) {
    int64_t blocks = (work + threads - 1) / threads;
    int64_t cap = (int64_t)num_sms() * 8;
    return (int)std::max<int64_t>(1, std::min(blocks, cap));
}

int bin_launches(int N, const int* dense_flag) { return N <= kBinSmallRows && !dense_flag ? 1 : 3; }

gtattn_status bin_rows(const int* indptr, int N, int long_min, int chunk, const int* dense_flag,
                       int* hdr, int* rows, int2* chunks, int2* longs, cudaStream_t s) {
    if (N <= kBinSmallRows && !dense_flag) {
        k_bin_small<<<1, kSmallThreads, 0, s>>>(indptr, N, long_min, chunk, hdr, rows, chunks, longs);
        GT_CUDA(cudaGetLastError());
        return GTATTN_OK;
    }
    GT_CUDA(cudaMemsetAsync(hdr, 0, sizeof(int) * HdrLayout::kWords, s));
    if (N == 0) return GTATTN_OK;
    const int T = 256;
    k_bin_count<<<grid_for(N, T), T, 0, s>>>(indptr, N, long_min, chunk, dense_flag, hdr);
    k_bin_offsets<<<1, 32, 0, s>>>(hdr);
    k_bin_scatter<<<grid_for(N, kScatterThreads), kScatterThreads, 0, s>>>(indptr, N, long_min, chunk,
                                                                          dense_flag, hdr, rows, chunks, longs);
    GT_CUDA(cudaGetLastError());
    return GTATTN_OK;
}

void resolve_opts(const gtattn_plan_opts* in, gtattn_plan_opts* out) {
    gtattn_plan_opts o;
    std::memset(&o, 0, sizeof(o));
    if (in) o = *in;
    if (o.long_row_min == 0) o.long_row_min = kDefaultLongMin;
    if (o.long_row_min < -1) o.long_row_min = -1;
    if (o.chunk_edges <= 0) o.chunk_edges = kDefaultChunk;
    *out = o;
}

// worst-case list sizes when the counts are only known on the device
void worst_case_sizes(int64_t N, int64_t nnz, int long_min, int chunk, int64_t* n_long,
                      int64_t* n_chunks) {
    int64_t per = std::max<int64_t>(1, (int64_t)long_min + 1);
    int64_t nl = std::min<int64_t>(N, nnz / per);
    *n_long = nl;
    *n_chunks = nnz / chunk + nl;
}

}  // namespace gt

using namespace gt;

// ---------------------------------------------------------------------------
// the plan object
// ---------------------------------------------------------------------------
extern "C" gtattn_status gtattn_csr_build(const int32_t* indptr, const int32_t* indices, int64_t N,
                                          int64_t nnz, const gtattn_plan_opts* opts,
                                          gtattn_plan** plan_out, cudaStream_t stream) {
    if (!plan_out) return GTATTN_ERR_INVALID_ARG;
    *plan_out = nullptr;
    if (N < 0 || nnz < 0 || N >= (1ll << 31) - 1 || nnz >= (1ll << 31) - 1) return GTATTN_ERR_INVALID_ARG;
    if (!indptr || (nnz > 0 && !indices)) return GTATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(indptr) | reinterpret_cast<uintptr_t>(indices)) & 3u)
        return GTATTN_ERR_INVALID_ARG;
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);

    gtattn_plan* p = new (std::nothrow) gtattn_plan();
    if (!p) return GTATTN_ERR_NO_MEMORY;
    p->N = N;
    p->nnz = nnz;
    resolve_opts(opts, &p->opts);
    GT_CUDA(cudaGetDevice(&p->device));
    p->stream = stream;

    gtattn_status st = GTATTN_OK;
    int* cand = nullptr;
    auto fail = [&](gtattn_status s) {
        if (cand) cudaFree(cand);
        gtattn_plan_destroy(p);
        return s;
    };
    auto chk = [&](cudaError_t e) { return e == cudaSuccess ? GTATTN_OK : cuda_status(e); };

    const int n = (int)N;
    if ((st = chk(cudaMalloc(&p->hdr, sizeof(int) * HdrLayout::kWords))) != GTATTN_OK) return fail(st);
    if ((st = chk(cudaMalloc(&p->rows, sizeof(int) * std::max<int64_t>(N, 1)))) != GTATTN_OK) return fail(st);
    int* dense_flag = nullptr;
    if (p->opts.detect_dense && N > 0) {
        if ((st = chk(cudaMalloc(&p->dense_flag, sizeof(int) * N))) != GTATTN_OK) return fail(st);
        if ((st = chk(cudaMalloc(&cand, sizeof(int) * N))) != GTATTN_OK) return fail(st);
        int64_t max_blocks = std::max<int64_t>(1, N / kDenseTile);
        if ((st = chk(cudaMalloc(&p->blocks, sizeof(int2) * max_blocks))) != GTATTN_OK) return fail(st);
        if ((st = chk(cudaMemsetAsync(p->dense_flag, 0, sizeof(int) * N, stream))) != GTATTN_OK) return fail(st);
        dense_flag = p->dense_flag;
    }
    // pass 1: counts only (lists sized afterwards); dense detection needs the
    // header zeroed first, so detection runs after the memset inside bin_rows
    if ((st = chk(cudaMemsetAsync(p->hdr, 0, sizeof(int) * HdrLayout::kWords, stream))) != GTATTN_OK)
        return fail(st);
    if (N > 0) {
        const int T = 256;
        if (dense_flag) {
            int g = grid_for((int64_t)N * 32, T);
            k_dense_candidates<<<g, T, 0, stream>>>(indptr, indices, n, cand);
            k_dense_blocks<<<g, T, 0, stream>>>(indptr, n, cand, p->hdr, p->blocks, dense_flag);
        }
        k_bin_count<<<grid_for(N, T), T, 0, stream>>>(indptr, n, p->opts.long_row_min,
                                                        p->opts.chunk_edges, dense_flag, p->hdr);
        if ((st = chk(cudaGetLastError())) != GTATTN_OK) return fail(st);
    }
    if ((st = chk(cudaMemcpyAsync(p->hdr_host, p->hdr, sizeof(int) * HdrLayout::kWords,
                                  cudaMemcpyDeviceToHost, stream))) != GTATTN_OK)
        return fail(st);
    if ((st = chk(cudaStreamSynchronize(stream))) != GTATTN_OK) return fail(st);
    if (cand) { cudaFree(cand); cand = nullptr; }

    const int n_long = p->hdr_host[HdrLayout::kLong];
    const int n_chunks = p->hdr_host[HdrLayout::kChunks];
    if ((st = chk(cudaMalloc(&p->chunks, sizeof(int2) * std::max(1, n_chunks)))) != GTATTN_OK) return fail(st);
    if ((st = chk(cudaMalloc(&p->longs, sizeof(int2) * std::max(1, n_long)))) != GTATTN_OK) return fail(st);
    if (N > 0) {
        // pass 2: offsets and scatter (counts and dense blocks stay in the header)
        k_bin_offsets<<<1, 32, 0, stream>>>(p->hdr);
        k_bin_scatter<<<grid_for(N, kScatterThreads), kScatterThreads, 0, stream>>>(
            indptr, n, p->opts.long_row_min, p->opts.chunk_edges, dense_flag, p->hdr, p->rows, p->chunks,
            p->longs);
        if ((st = chk(cudaGetLastError())) != GTATTN_OK) return fail(st);
    }
    if ((st = chk(cudaMemcpyAsync(p->hdr_host, p->hdr, sizeof(int) * HdrLayout::kWords,
                                  cudaMemcpyDeviceToHost, stream))) != GTATTN_OK)
        return fail(st);
    if ((st = chk(cudaStreamSynchronize(stream))) != GTATTN_OK) return fail(st);
    // dense blocks -> one work item per 128-row query tile
    const int nb = p->hdr_host[HdrLayout::kDenseBlocks];
    if (nb > 0) {
        std::vector<int2> hb(nb);
        if ((st = chk(cudaMemcpy(hb.data(), p->blocks, sizeof(int2) * nb, cudaMemcpyDeviceToHost))) != GTATTN_OK)
            return fail(st);
        // one work item per pair of 128-row query tiles: (block row, block size,
        // first query row, query tiles in the item)
        std::vector<int4> tiles, tiles1;
        for (const int2& b : hb) {
            for (int q0 = b.x; q0 < b.x + b.y; q0 += 2 * kDenseTile)
                tiles.push_back(make_int4(b.x, b.y, q0, std::min(2, (b.x + b.y - q0 + kDenseTile - 1) / kDenseTile)));
            // (the widest heads take one query tile per item)
            for (int q0 = b.x; q0 < b.x + b.y; q0 += kDenseTile) tiles1.push_back(make_int4(b.x, b.y, q0, 1));
        }
        if ((st = chk(cudaMalloc(&p->dense_tiles, sizeof(int4) * tiles.size()))) != GTATTN_OK) return fail(st);
        if ((st = chk(cudaMemcpy(p->dense_tiles, tiles.data(), sizeof(int4) * tiles.size(),
                                 cudaMemcpyHostToDevice))) != GTATTN_OK)
            return fail(st);
        p->n_dense_tiles = static_cast<int>(tiles.size());
        if ((st = chk(cudaMalloc(&p->dense_tiles1, sizeof(int4) * tiles1.size()))) != GTATTN_OK) return fail(st);
        if ((st = chk(cudaMemcpy(p->dense_tiles1, tiles1.data(), sizeof(int4) * tiles1.size(),
                                 cudaMemcpyHostToDevice))) != GTATTN_OK)
            return fail(st);
        p->n_dense_tiles1 = static_cast<int>(tiles1.size());
    }
    *plan_out = p;
    return GTATTN_OK;
}

extern "C" gtattn_status gtattn_plan_destroy(gtattn_plan* p) {
    if (!p) return GTATTN_OK;
    int cur = -1;
    cudaGetDevice(&cur);
    if (p->device >= 0 && cur != p->device) cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    cudaFree(p->hdr);
    cudaFree(p->rows);
    cudaFree(p->chunks);
    cudaFree(p->longs);
    cudaFree(p->blocks);
    cudaFree(p->dense_tiles);
    cudaFree(p->dense_tiles1);
    cudaFree(p->dense_flag);
    if (p->ws) cudaFree(p->ws);
    if (p->bwd_pattern) cudaFree(p->bwd_pattern);
    if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    delete p;
    return GTATTN_OK;
}

extern "C" gtattn_status gtattn_plan_get_info(const gtattn_plan* p, gtattn_plan_info* info) {
    if (!p || !info) return GTATTN_ERR_INVALID_ARG;
    std::memset(info, 0, sizeof(*info));
    info->N = p->N;
    info->nnz = p->nnz;
    info->n_long_rows = p->hdr_host[HdrLayout::kLong];
    info->n_chunks = p->hdr_host[HdrLayout::kChunks];
    info->n_dense_blocks = p->hdr_host[HdrLayout::kDenseBlocks];
    info->n_dense_rows = p->hdr_host[HdrLayout::kDenseRows];
    info->n_empty_rows = p->hdr_host[HdrLayout::kCount + 0];
    info->max_degree = p->hdr_host[HdrLayout::kMaxDeg];
    info->n_buckets = kNumBuckets;
    for (int b = 0; b < kNumBuckets; ++b) info->bucket_rows[b] = p->hdr_host[HdrLayout::kCount + b];
    int dev_err = 0;
    cudaError_t e = cudaMemcpy(&dev_err, p->hdr + HdrLayout::kErr, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    info->device_error = dev_err;
    if (dev_err != 0) {   // read and cleared: a later call's record starts empty
        e = cudaMemset(p->hdr + HdrLayout::kErr, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_status(e);
    }
    return GTATTN_OK;
}

// ---------------------------------------------------------------------------
// CSR validation
// ---------------------------------------------------------------------------
__global__ void k_validate(const int* __restrict__ indptr, const int* __restrict__ indices, int N,
                           int nnz, int* __restrict__ bad) {
    const int stride = gridDim.x * blockDim.x;
    int local = 0;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= N; i += stride) {
        int v = indptr[i];
        if (i == 0 && v != 0) local = 1;
        if (i == N && v != nnz) local = 1;
        if (i < N && indptr[i + 1] < v) local = 1;
    }
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += stride) {
        int j = indices[e];
        if (j < 0 || j >= N) local = 1;
    }
    if (local) atomicOr(bad, 1);
}

#ifdef GTATTN_DEBUG
__device__ int g_debug_bad_csr;   // the checking build's validation flag

gtattn_status gt::debug_csr_check(const int32_t* indptr, const int32_t* indices, int64_t N, int64_t nnz,
                              cudaStream_t s) {
    int* bad = nullptr;
    GT_CUDA(cudaGetSymbolAddress(reinterpret_cast<void**>(&bad), g_debug_bad_csr));
    GT_CUDA(cudaMemsetAsync(bad, 0, sizeof(int), s));
    k_validate<<<grid_for(std::max<int64_t>(N + 1, nnz), 256), 256, 0, s>>>(indptr, indices, (int)N, (int)nnz, bad);
    GT_CUDA(cudaGetLastError());
    int h_bad = 0;
    GT_CUDA(cudaMemcpyAsync(&h_bad, bad, sizeof(int), cudaMemcpyDeviceToHost, s));
    GT_CUDA(cudaStreamSynchronize(s));
    if (h_bad) {
        set_last_error("checking build: the CSR failed validation (offsets from 0 to nnz, non-decreasing; "
                       "indices in [0, N)); nothing else ran");
        return GTATTN_ERR_BAD_CSR;
    }
    return GTATTN_OK;
}
#endif

extern "C" gtattn_status gtattn_csr_validate(const int32_t* indptr, const int32_t* indices,
                                             int64_t N, int64_t nnz, cudaStream_t stream) {
    if (N < 0 || nnz < 0 || N >= (1ll << 31) - 1 || nnz >= (1ll << 31) - 1) return GTATTN_ERR_INVALID_ARG;
    if (!indptr || (nnz > 0 && !indices)) return GTATTN_ERR_INVALID_ARG;
    int* bad = nullptr;
    GT_TRY(pool_alloc((void**)&bad, sizeof(int), stream));
    gtattn_status st = GTATTN_OK;
    int h_bad = 0;
    cudaError_t e = cudaMemsetAsync(bad, 0, sizeof(int), stream);
    if (e == cudaSuccess) {
        k_validate<<<grid_for(std::max<int64_t>(N + 1, nnz), 256), 256, 0, stream>>>(
            indptr, indices, (int)N, (int)nnz, bad);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h_bad, bad, sizeof(int), cudaMemcpyDeviceToHost, stream);
    pool_free(bad, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) st = cuda_status(e);
    else if (h_bad) st = GTATTN_ERR_BAD_CSR;
    return st;
}

// ---------------------------------------------------------------------------
// COO -> CSR by destination: count, scan, scatter, sort each row by source
// ---------------------------------------------------------------------------
__global__ void k_coo_count(const int* __restrict__ dst, int nnz, int N, int* __restrict__ cnt) {
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += gridDim.x * blockDim.x) {
        int d = dst[e];
        if (d >= 0 && d < N) atomicAdd(&cnt[d], 1);    // out-of-range edges are dropped
    }
}

// exclusive scan of cnt[0..N) into indptr[0..N], single pass per block of
// 1024 elements plus a block-sum carry done serially by one block.
__global__ void k_block_scan(const int* __restrict__ in, int n, int* __restrict__ out,
                             int* __restrict__ block_sums) {
    __shared__ int s[1024];
    int i = blockIdx.x * 1024 + threadIdx.x;
    int v = i < n ? in[i] : 0;
    s[threadIdx.x] = v;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {
        int t = threadIdx.x >= o ? s[threadIdx.x - o] : 0;
        __syncthreads();
        s[threadIdx.x] += t;
        __syncthreads();
    }
    if (i < n) out[i] = s[threadIdx.x] - v;   // exclusive within block
    if (threadIdx.x == 1023) block_sums[blockIdx.x] = s[1023];
}

__global__ void k_scan_sums(int* __restrict__ sums, int nb, int* __restrict__ total) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int run = 0;
    for (int b = 0; b < nb; ++b) { int v = sums[b]; sums[b] = run; run += v; }
    *total = run;
}

__global__ void k_scan_add(int* __restrict__ out, int n, const int* __restrict__ sums) {
    int i = blockIdx.x * 1024 + threadIdx.x;
    if (i < n) out[i] += sums[blockIdx.x];
}

__global__ void k_coo_scatter(const int* __restrict__ src, const int* __restrict__ dst, int nnz, int N,
                              const int* __restrict__ indptr, int* __restrict__ cursor,
                              int* __restrict__ indices) {
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += gridDim.x * blockDim.x) {
        int d = dst[e];
        if (d < 0 || d >= N) continue;
        int pos = indptr[d] + atomicAdd(&cursor[d], 1);
        indices[pos] = src[e];
    }
}

// sort each row's entries ascending: bitonic network over the row, one block
// per row; rows up to 4096 entries sort in shared memory, longer rows in place
// in global memory (rare: hub rows).
__global__ void k_row_sort(const int* __restrict__ indptr, int N, int* __restrict__ indices) {
    __shared__ int s[4096];
    for (int r = blockIdx.x; r < N; r += gridDim.x) {
        int beg = indptr[r], deg = indptr[r + 1] - beg;
        if (deg < 2) continue;
        int n2 = 1;
        while (n2 < deg) n2 <<= 1;
        if (n2 <= 4096) {
            for (int k = threadIdx.x; k < n2; k += blockDim.x) s[k] = k < deg ? indices[beg + k] : 0x7fffffff;
            __syncthreads();
            for (int size = 2; size <= n2; size <<= 1)
                for (int stride = size >> 1; stride > 0; stride >>= 1) {
                    for (int k = threadIdx.x; k < n2; k += blockDim.x) {
                        int partner = k ^ stride;
                        if (partner > k) {
                            bool up = (k & size) == 0;
                            int a = s[k], b = s[partner];
                            if ((a > b) == up) { s[k] = b; s[partner] = a; }
                        }
                    }
                    __syncthreads();
                }
            for (int k = threadIdx.x; k < deg; k += blockDim.x) indices[beg + k] = s[k];
            __syncthreads();
        } else {
            // odd-even transposition passes on global memory, deg passes
            for (int pass = 0; pass < deg; ++pass) {
                for (int k = 2 * threadIdx.x + (pass & 1); k + 1 < deg; k += 2 * blockDim.x) {
                    int a = indices[beg + k], b = indices[beg + k + 1];
                    if (a > b) { indices[beg + k] = b; indices[beg + k + 1] = a; }
                }
                __syncthreads();
            }
        }
    }
}

extern "C" gtattn_status gtattn_coo_to_csr(const int32_t* src, const int32_t* dst, int64_t nnz,
                                           int64_t N, int32_t* indptr, int32_t* indices,
                                           cudaStream_t stream) {
    if (N < 0 || nnz < 0 || N >= (1ll << 31) - 1 || nnz >= (1ll << 31) - 1) return GTATTN_ERR_INVALID_ARG;
    if (!indptr || (nnz > 0 && (!src || !dst || !indices))) return GTATTN_ERR_INVALID_ARG;
    const int n = (int)N, m = (int)nnz;
    if (N == 0) {
        GT_CUDA(cudaMemsetAsync(indptr, 0, sizeof(int), stream));
        return GTATTN_OK;
    }
    int nb = (n + 1023) / 1024;
    int *cnt = nullptr, *sums = nullptr;
    GT_TRY(pool_alloc((void**)&cnt, sizeof(int) * (size_t)n, stream));
    gtattn_status st = pool_alloc((void**)&sums, sizeof(int) * (size_t)nb, stream);
    if (st != GTATTN_OK) { pool_free(cnt, stream); return st; }
    cudaError_t e = cudaMemsetAsync(cnt, 0, sizeof(int) * (size_t)n, stream);
    if (e == cudaSuccess) {
        if (m > 0) k_coo_count<<<grid_for(m, 256), 256, 0, stream>>>(dst, m, n, cnt);
        k_block_scan<<<nb, 1024, 0, stream>>>(cnt, n, indptr, sums);
        k_scan_sums<<<1, 32, 0, stream>>>(sums, nb, indptr + n);
        k_scan_add<<<nb, 1024, 0, stream>>>(indptr, n, sums);
        e = cudaMemsetAsync(cnt, 0, sizeof(int) * (size_t)n, stream);
    }
    if (e == cudaSuccess && m > 0) {
        k_coo_scatter<<<grid_for(m, 256), 256, 0, stream>>>(src, dst, m, n, indptr, cnt, indices);
        k_row_sort<<<std::min(n, num_sms() * 8), 256, 0, stream>>>(indptr, n, indices);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    pool_free(cnt, stream);
    pool_free(sums, stream);
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}
