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

#include <cuda.h>

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

// Device address of the scratch array in the current context.  In host code
// the array's name is only a host-side handle; its device address is looked
// up (cudaGetSymbolAddress) with the device current and kept per device
// together with the id of the context it belongs to (cuCtxGetId: unique for
// the life of the process, never reused).  When the device's primary context
// has been torn down and made again (cudaDeviceReset, or a context destroyed
// through the driver API), the module is loaded anew and the array may sit
// elsewhere: the new context's id differs, the lookup runs again, and a stale
// address is never used.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
static Fn driver_fn(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        p = nullptr;
    return reinterpret_cast<Fn>(p);
}

// Id of the current context, 0 when none is current (or it cannot be read).
static unsigned long long current_ctx_id() {
    static const CtxGetCurrentFn get = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get || !get_id || get(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

static gtattn_status scratch_address(unsigned char** out) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static unsigned char* addr[kMaxDev] = {};
    static unsigned long long ctx_of[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDev) return GTATTN_ERR_UNSUPPORTED;
    // (on a thread that has made no runtime call on this device no context
    // is current yet, id 0: the symbol lookup below sets up the primary one)
    unsigned long long id = current_ctx_id();
    std::lock_guard<std::mutex> g(mu);
    if (id == 0 || !addr[dev] || ctx_of[dev] != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        id = current_ctx_id();
        if (id == 0) {
            set_last_error("gtattn_fwd_noalloc: the current CUDA context could not be identified");
            return GTATTN_ERR_CUDA;
        }
        addr[dev] = static_cast<unsigned char*>(p);
        ctx_of[dev] = id;
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
    GT_TRY(check_fwd(indptr, indices, Q, K, V, out, N, nnz, H, D, dtype));
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);   // (the checking build: a device flag, no allocation)

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
    p.ld = HD;
    p.groups = 1;
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
