// noalloc.cu -- gtattn_fwd_noalloc: the plan-less fused forward without any
// allocation.
//
// Some callers cannot allocate device memory at the point where they run the
// attention: code inside a custom allocator or memory-pool callback, runtimes
// that forbid cudaMalloc after start-up (fixed memory budgets, pre-planned
// arenas), or hosts whose framework owns the whole device heap.  For them this
// entry point keeps its temporaries -- the degree-bucket header, the row and
// chunk lists and the split-row partials -- in one file-scope device array of
// fixed size instead of the library's memory pool.  The row kernels, the
// binning kernels and the combine kernel are the same ones gtattn_fwd uses;
// only where their temporaries live differs.
#include "plan.cuh"
#include "rows.cuh"

#include <algorithm>
#include <cstdio>
#include <mutex>

namespace gt {

// The scratch array.  Every GPU that loads the library holds it until the
// process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB
// Split threshold and chunk size of this variant: larger than gtattn_fwd's
// defaults so that the worst-case partials fit the fixed array.
constexpr int kNoAllocLongMin = 1024;
constexpr int kNoAllocChunk = 1024;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Bytes of scratch one call needs (worst case over graphs with N rows and nnz
// entries: every split row is cut into at most ceil(deg/chunk) chunks).
static size_t noalloc_bytes(int64_t N, int64_t nnz, int H, int HD, int64_t* n_long, int64_t* n_chunks) {
    worst_case_sizes(N, nnz, kNoAllocLongMin, kNoAllocChunk, n_long, n_chunks);
    size_t b = up256(sizeof(int) * HdrLayout::kWords);
    b += up256(sizeof(int) * (size_t)N);
    b += up256(sizeof(int2) * (size_t)*n_chunks);
    b += up256(sizeof(int2) * (size_t)*n_long);
    b += 2 * up256(sizeof(float) * (size_t)*n_chunks * H);
    b += up256(sizeof(float) * (size_t)*n_chunks * HD);
    return b;
}

// Device address of the scratch array, looked up once per device with that
// device current (in host code the array's name is only a host-side handle).
static gtattn_status scratch_address(unsigned char** out) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static unsigned char* addr[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDev) return GTATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> g(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        addr[dev] = static_cast<unsigned char*>(p);
    }
    *out = addr[dev];
    return GTATTN_OK;
}

}  // namespace gt

using namespace gt;

extern "C" gtattn_status gtattn_fwd_noalloc(const int32_t* indptr, const int32_t* indices, const void* Q,
                                            const void* K, const void* V, void* out, int64_t N, int64_t nnz,
                                            int H, int D, float scale, gtattn_dtype dtype,
                                            cudaStream_t stream) {
    // the same argument rules as gtattn_fwd
    if (N < 0 || nnz < 0 || N >= (1ll << 31) - 1 || nnz >= (1ll << 31) - 1) return GTATTN_ERR_INVALID_ARG;
    if (H < 1 || D < 1 || (int64_t)H * D > kMaxHD) return GTATTN_ERR_INVALID_ARG;
    if (dtype != GTATTN_F32 && dtype != GTATTN_BF16 && dtype != GTATTN_BF16_OUT_F32)
        return GTATTN_ERR_INVALID_ARG;
    if (!indptr || (N > 0 && (!Q || !out)) || (nnz > 0 && (!indices || !K || !V))) return GTATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(indptr) | reinterpret_cast<uintptr_t>(indices)) & 3u)
        return GTATTN_ERR_INVALID_ARG;
    const uintptr_t esz = dtype == GTATTN_F32 ? 4 : 2;
    const uintptr_t osz = dtype == GTATTN_BF16 ? 2 : 4;
    if (((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V)) &
         (esz - 1)) || (reinterpret_cast<uintptr_t>(out) & (osz - 1)))
        return GTATTN_ERR_INVALID_ARG;

    const int HD = H * D;
    int64_t n_long = 0, n_chunks = 0;
    const size_t need = noalloc_bytes(N, nnz, H, HD, &n_long, &n_chunks);
    if (need > kNoAllocScratchBytes) {
        char msg[192];
        std::snprintf(msg, sizeof(msg),
                      "gtattn_fwd_noalloc: this problem needs %zu bytes of scratch; the fixed array holds %zu",
                      need, kNoAllocScratchBytes);
        set_last_error(msg);
        return GTATTN_ERR_UNSUPPORTED;
    }
    RowChoice c;
    if (!choose_row_kernel(H, D, dtype, Q, K, V, out, GTATTN_KERNEL_AUTO, &c)) return GTATTN_ERR_UNSUPPORTED;
    if (N == 0) return GTATTN_OK;

    unsigned char* base = nullptr;
    GT_TRY(scratch_address(&base));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        unsigned char* p = base + off;
        off += up256(bytes);
        return p;
    };
    int* hdr = reinterpret_cast<int*>(take(sizeof(int) * HdrLayout::kWords));
    int* rows = reinterpret_cast<int*>(take(sizeof(int) * (size_t)N));
    int2* chunks = reinterpret_cast<int2*>(take(sizeof(int2) * (size_t)n_chunks));
    int2* longs = reinterpret_cast<int2*>(take(sizeof(int2) * (size_t)n_long));
    Partials part;
    part.m = reinterpret_cast<float*>(take(sizeof(float) * (size_t)n_chunks * H));
    part.s = reinterpret_cast<float*>(take(sizeof(float) * (size_t)n_chunks * H));
    part.acc = reinterpret_cast<float*>(take(sizeof(float) * (size_t)n_chunks * HD));

    // bin_rows zeroes the header (counts and cursors) first, so nothing left
    // in the array by an earlier call is read; lists and partials are written
    // before they are read.
    gtattn_status st = bin_rows(indptr, (int)N, kNoAllocLongMin, kNoAllocChunk, nullptr, hdr, rows, chunks,
                                longs, stream);
    if (st != GTATTN_OK) return st;
    RowParams p{};
    p.indptr = indptr;
    p.indices = indices;
    p.Q = Q;
    p.K = K;
    p.V = V;
    p.out = out;
    p.qscale = scale * kLog2e;
    p.N = (int)N;
    p.H = H;
    p.D = D;
    p.HD = HD;
    p.G = c.G;
    p.lph = c.lph;
    p.lists = TaskLists{hdr, rows, chunks, longs, kNoAllocChunk, 1};
    p.part = part;
    p.task_bound = row_task_bound(N, nnz, kNoAllocChunk);
    st = launch_rows(kFused, dtype, c, p, stream);
    // no row can be split when nnz is at most the split threshold
    if (st == GTATTN_OK && nnz > kNoAllocLongMin) st = launch_combine(kFused, dtype, p, stream);
    return st;
}
