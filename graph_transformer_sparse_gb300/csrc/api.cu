// api.cu -- the C ABI: argument checks, temporaries, dispatch.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "dense.cuh"
#include "gemm.cuh"
#include "plan.cuh"
#include "rows.cuh"
#include "bwd.cuh"

namespace gt {

static thread_local char g_last_error[256] = "";

void set_last_error(const char* msg) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg ? msg : "");
}

gtattn_status cuda_status(cudaError_t e) {
    set_last_error(cudaGetErrorString(e));
    if (e == cudaErrorMemoryAllocation) return GTATTN_ERR_NO_MEMORY;
    return GTATTN_ERR_CUDA;
}

constexpr int kMaxDevices = 64;

int num_sms() {
    static int cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

// L2 bytes of the current device (cached per device); when unknown, a size
// no graph exceeds (the head groups then stay one).
static int64_t l2_bytes() {
    constexpr int64_t kUnknown = int64_t(1) << 50;
    static int64_t cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kUnknown;
    if (cache[dev] == 0) {
        int n = 0;
        cache[dev] = cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, dev) == cudaSuccess && n > 0 ? n : kUnknown;
    }
    return cache[dev];
}

// One library-owned memory pool per device; freed blocks stay cached in the
// pool (release threshold: unlimited) so per-call temporaries cost no
// driver allocation after the first call.
cudaMemPool_t pool() {
    static std::mutex mu;
    static cudaMemPool_t pools[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> g(mu);
    if (!pools[dev]) {
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) != cudaSuccess) return nullptr;
        uint64_t thresh = ~0ull;
        cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &thresh);
        pools[dev] = p;
    }
    return pools[dev];
}

gtattn_status pool_alloc(void** p, size_t bytes, cudaStream_t s) {
    *p = nullptr;
    cudaMemPool_t mp = pool();
    if (!mp) return GTATTN_ERR_CUDA;
    cudaError_t e = cudaMallocFromPoolAsync(p, std::max<size_t>(bytes, 256), mp, s);
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

void pool_free(void* p, cudaStream_t s) {
    if (p) cudaFreeAsync(p, s);
}

// ---------------------------------------------------------------------------
// benchmark instrumentation
// ---------------------------------------------------------------------------
struct ProfRecord {
    int cat;
    cudaEvent_t a, b;
};
static std::mutex g_prof_mu;
static bool g_prof_on = false;
static std::vector<ProfRecord> g_prof;
static int g_prof_launches[GTATTN_KCAT_COUNT] = {};

ProfScope::ProfScope(int category, int launches, cudaStream_t s) : cat_(category), s_(s), start_(nullptr) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (!g_prof_on) return;
    g_prof_launches[category] += launches;
    cudaEvent_t a;
    if (cudaEventCreate(&a) != cudaSuccess) return;
    cudaEventRecord(a, s);
    start_ = a;
}

ProfScope::~ProfScope() {
    if (!start_) return;
    std::lock_guard<std::mutex> g(g_prof_mu);
    cudaEvent_t b;
    if (cudaEventCreate(&b) != cudaSuccess) return;
    cudaEventRecord(b, s_);
    g_prof.push_back(ProfRecord{cat_, static_cast<cudaEvent_t>(start_), b});
}

static size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

// Checks shared by the forward entry points (gtattn_fwd_noalloc too).
gtattn_status check_fwd(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                        const void* V, const void* out, int64_t N, int64_t nnz, int H, int D, gtattn_dtype dtype) {
    if (N < 0 || nnz < 0 || N >= (1ll << 31) - 1 || nnz >= (1ll << 31) - 1) return GTATTN_ERR_INVALID_ARG;
    if (H < 1 || D < 1 || (int64_t)H * D > kMaxHD) return GTATTN_ERR_INVALID_ARG;
    if (dtype != GTATTN_F32 && dtype != GTATTN_BF16 && dtype != GTATTN_BF16_OUT_F32)
        return GTATTN_ERR_INVALID_ARG;
    if (!indptr) return GTATTN_ERR_INVALID_ARG;
    if (N > 0 && (!Q || !out)) return GTATTN_ERR_INVALID_ARG;
    if (nnz > 0 && (!indices || !K || !V)) return GTATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(indptr) | reinterpret_cast<uintptr_t>(indices)) & 3u)
        return GTATTN_ERR_INVALID_ARG;
    const uintptr_t esz = dtype == GTATTN_F32 ? 4 : 2;
    const uintptr_t osz = dtype == GTATTN_BF16 ? 2 : 4;
    const uintptr_t al = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                         reinterpret_cast<uintptr_t>(V);
    if ((al & (esz - 1)) || (reinterpret_cast<uintptr_t>(out) & (osz - 1))) return GTATTN_ERR_INVALID_ARG;
    return GTATTN_OK;
}

// Stream-ordered temporaries of a plan-less call: one pool block carved up.
struct Scratch {
    void* base = nullptr;
    TaskLists lists{};
    Partials part{};
    int64_t part_chunks = 0;   // chunk slots of the partials
    float* logits = nullptr;
    float* probs = nullptr;
};

static gtattn_status scratch_alloc(int64_t N, int64_t nnz, int H, int HD, int long_min, int chunk,
                                   bool need_logits, bool need_probs, Scratch* sc, int** hdr,
                                   int** rows, int2** chunks, int2** longs, cudaStream_t s) {
    int64_t n_long = 0, n_chunks = 0;
    worst_case_sizes(N, nnz, long_min, chunk, &n_long, &n_chunks);
    size_t off = 0;
    const size_t o_hdr = off; off = align_up(off + sizeof(int) * HdrLayout::kWords);
    const size_t o_rows = off; off = align_up(off + sizeof(int) * (size_t)N);
    const size_t o_chunks = off; off = align_up(off + sizeof(int2) * (size_t)n_chunks);
    const size_t o_longs = off; off = align_up(off + sizeof(int2) * (size_t)n_long);
    const size_t o_m = off; off = align_up(off + sizeof(float) * (size_t)n_chunks * H);
    const size_t o_s = off; off = align_up(off + sizeof(float) * (size_t)n_chunks * H);
    const size_t o_acc = off; off = align_up(off + sizeof(float) * (size_t)n_chunks * HD);
    const size_t o_lg = off; if (need_logits) off = align_up(off + sizeof(float) * (size_t)nnz * H);
    const size_t o_pr = off; if (need_probs) off = align_up(off + sizeof(float) * (size_t)nnz * H);
    GT_TRY(pool_alloc(&sc->base, off, s));
    char* b = static_cast<char*>(sc->base);
    *hdr = reinterpret_cast<int*>(b + o_hdr);
    *rows = reinterpret_cast<int*>(b + o_rows);
    *chunks = reinterpret_cast<int2*>(b + o_chunks);
    *longs = reinterpret_cast<int2*>(b + o_longs);
    sc->part.m = reinterpret_cast<float*>(b + o_m);
    sc->part.s = reinterpret_cast<float*>(b + o_s);
    sc->part.acc = reinterpret_cast<float*>(b + o_acc);
    sc->part_chunks = n_chunks;
    if (need_logits) sc->logits = reinterpret_cast<float*>(b + o_lg);
    if (need_probs) sc->probs = reinterpret_cast<float*>(b + o_pr);
    sc->lists = TaskLists{*hdr, *rows, *chunks, *longs, chunk, 1};
    return GTATTN_OK;
}

static RowParams make_params(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                             const void* V, void* out, int64_t N, int64_t nnz, int H, int D, float qscale,
                             const RowChoice& c, const TaskLists& L, const Partials& part) {
    RowParams p{};
    p.indptr = indptr;
    p.indices = indices;
    p.Q = Q;
    p.K = K;
    p.V = V;
    p.out = out;
    p.qscale = qscale;
    p.N = (int)N;
    p.H = H;
    p.D = D;
    p.HD = H * D;
    p.ld = H * D;
    p.groups = 1;
    p.G = c.G;
    p.lph = c.lph;
    p.lists = L;
    p.part = part;
    p.task_bound = row_task_bound(N, nnz, L.chunk_edges);
    return p;
}

}  // namespace gt

using namespace gt;

extern "C" const char* gtattn_status_string(gtattn_status s) {
    switch (s) {
        case GTATTN_OK: return "ok";
        case GTATTN_ERR_INVALID_ARG: return "invalid argument";
        case GTATTN_ERR_BAD_CSR: return "malformed CSR";
        case GTATTN_ERR_UNSUPPORTED: return "unsupported";
        case GTATTN_ERR_CUDA: return "CUDA error";
        case GTATTN_ERR_NO_MEMORY: return "out of memory";
        case GTATTN_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

extern "C" const char* gtattn_last_error(void) { return g_last_error; }

extern "C" gtattn_status gtattn_profile_enable(int on) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    g_prof_on = on != 0;
    return GTATTN_OK;
}

extern "C" gtattn_status gtattn_profile_read(gtattn_profile* out, int reset) {
    if (!out) return GTATTN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(g_prof_mu);
    std::memset(out, 0, sizeof(*out));
    gtattn_status st = GTATTN_OK;
    for (auto& r : g_prof) {
        float ms = 0.f;
        cudaError_t e = cudaEventSynchronize(r.b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.a, r.b);
        if (e != cudaSuccess) st = cuda_status(e);
        out->ms[r.cat] += ms;
        out->groups[r.cat] += 1;
    }
    for (int c = 0; c < GTATTN_KCAT_COUNT; ++c) out->launches[c] = g_prof_launches[c];
    if (reset) {
        for (auto& r : g_prof) { cudaEventDestroy(r.a); cudaEventDestroy(r.b); }
        g_prof.clear();
        std::memset(g_prof_launches, 0, sizeof(g_prof_launches));
    }
    return st;
}

// The fused forward on the fly (binning, fused rows, combine), with an
// optional per-entry additive bias or per-entry adjacency values.
// Head groups run one after another over the same rows (each head's softmax
// is its own, so the groups are independent).  A group's gathers touch only
// its columns of the K and V rows, so when K and V together exceed the L2 a
// group's share may fit and its gathers stop going to DRAM once per entry
// (Erdos-Renyi, 8 x 64 bf16, 205 MB of K and V: one pass 0.464 ms, two
// passes 0.410).  Groups are halved while K and V exceed 85 % of the L2 and
// a group's share of a row stays at least 512 bytes: rows of a few hundred
// bytes lose more to the repeated task set-up than the L2 wins (R-MAT, 256-
// byte rows: 0.96 ms in one pass, 1.24 in two).  Vector kernel, plain fused
// forward (no bias, values, head-innermost rows or row statistics).
static int head_passes(int64_t n_src, int H, int D, gtattn_dtype dtype, const RowChoice& c, const float* bias,
                       const float* values, int ndh) {
    if (bias || values || ndh || c.kind != RowKernel::kVector) return 1;
    const double row = static_cast<double>(H) * D * (dtype == GTATTN_F32 ? 4 : 2);
    const double kv = 2.0 * static_cast<double>(n_src) * row;
    const double budget = 0.85 * static_cast<double>(l2_bytes());
    int n = 1;
    while (kv / n > budget && H % (2 * n) == 0 && row / (2 * n) >= 512.0) n *= 2;
    return n;
}

// The fused rows and (when a row may be split) the combine, over head groups
// (head_passes; one group when row statistics are written).
static gtattn_status rows_in_groups(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                                    const void* V, void* out, int64_t N, int64_t nnz, int H, int D, float scale,
                                    gtattn_dtype dtype, const RowChoice& c, const TaskLists& L, const Partials& part,
                                    int64_t part_chunks, const float* bias, const float* values, int ndh, float* lse,
                                    bool run_rows, bool run_combine, int64_t n_src, cudaStream_t stream) {
    // (n_src: the rows of K and V the entries point into, which decide the
    // head groups; a call on a view of some rows passes the whole graph's.
    // part_chunks: the chunk slots `part` holds at H heads; each group's
    // partials take a block of its own, so one combine after all the groups'
    // rows serves them all)
    int passes = lse ? 1 : head_passes(n_src, H, D, dtype, c, bias, values, ndh);
    RowChoice cs = c;
    if (passes > 1 && !choose_row_kernel(H / passes, D, dtype, Q, K, V, out, GTATTN_KERNEL_VECTOR, &cs)) passes = 1;
    const int Hs = H / passes;
    const size_t esz = dtype == GTATTN_F32 ? 4 : 2, osz = dtype == GTATTN_BF16 ? 2 : 4;
    const int64_t step_m = part_chunks * Hs, step_acc = part_chunks * Hs * D;
    const RowChoice& cg = passes > 1 ? cs : c;
    auto group_params = [&](int g) {
        // head group g: heads g*Hs .. g*Hs+Hs-1, the same rows at the full stride
        const size_t off = static_cast<size_t>(g) * Hs * D;
        const Partials pg{part.m ? part.m + g * step_m : nullptr, part.s ? part.s + g * step_m : nullptr,
                          part.acc ? part.acc + g * step_acc : nullptr};
        RowParams p = make_params(indptr, indices, static_cast<const char*>(Q) + off * esz,
                                  static_cast<const char*>(K) + off * esz, static_cast<const char*>(V) + off * esz,
                                  static_cast<char*>(out) + off * osz, N, nnz, Hs, D, scale * kLog2e, cg, L, pg);
        p.ld = H * D;
        p.bias = bias;
        p.values = values;
        p.ndh = ndh;
        p.lse = lse;
        return p;
    };
    gtattn_status st = GTATTN_OK;
    for (int g = 0; g < passes && st == GTATTN_OK && run_rows; ++g) {
        RowParams p = group_params(g);
        ProfScope ps(GTATTN_KCAT_ROWS, 1, stream);
        st = launch_rows(kFused, dtype, cg, p, stream);
    }
    if (st == GTATTN_OK && run_combine) {
        RowParams p = group_params(0);
        p.groups = passes;
        p.gstep_m = step_m;
        p.gstep_acc = step_acc;
        p.gstep_out = Hs * D;
        ProfScope ps(GTATTN_KCAT_COMBINE, 1, stream);
        st = launch_combine(kFused, dtype, p, stream);
    }
    return st;
}

static gtattn_status fwd_fused(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                               const void* V, const float* values, const float* bias, void* out, int64_t N,
                               int64_t nnz, int H, int D, float scale, gtattn_dtype dtype, cudaStream_t stream,
                               int ndh = 0, int64_t n_src = -1) {
    GT_TRY(check_fwd(indptr, indices, Q, K, V, out, N, nnz, H, D, dtype));
    RowChoice c;
    // head-innermost rows ([N, D, H]): the generic kernel (the vector kernel's
    // lane groups assume head-major rows)
    if (!choose_row_kernel(H, D, dtype, Q, K, V, out, ndh ? GTATTN_KERNEL_GENERIC : GTATTN_KERNEL_AUTO, &c))
        return GTATTN_ERR_UNSUPPORTED;
    if (N == 0) return GTATTN_OK;
    gtattn_plan_opts o;
    resolve_opts(nullptr, &o);
    {
        // small graphs: one cooperative launch that bins in shared memory and
        // combines split rows itself (no binning or combine launches)
        int64_t nl = 0, nc = 0;
        worst_case_sizes(N, nnz, o.long_row_min, o.chunk_edges, &nl, &nc);
        if (N <= kSmallMaxRows && nnz <= kSmallMaxNnz && nc <= kSmallMaxChunks && nl <= kSmallMaxLong) {
            const int HD = H * D;
            void* part_buf = nullptr;
            Partials part{};
            if (nnz > o.long_row_min) {   // a row may be split: its chunks' partials
                const size_t a = align_up(sizeof(float) * static_cast<size_t>(nc) * H);
                GT_TRY(pool_alloc(&part_buf, 2 * a + sizeof(float) * static_cast<size_t>(nc) * HD, stream));
                char* b = static_cast<char*>(part_buf);
                part = Partials{reinterpret_cast<float*>(b), reinterpret_cast<float*>(b + a),
                                reinterpret_cast<float*>(b + 2 * a)};
            }
            TaskLists none{nullptr, nullptr, nullptr, nullptr, o.chunk_edges, 1};
            RowParams p = make_params(indptr, indices, Q, K, V, out, N, nnz, H, D, scale * kLog2e, c, none, part);
            p.bias = bias;
            p.values = values;
            p.ndh = ndh;
            p.long_min = o.long_row_min;
            p.small_max_chunks = kSmallMaxChunks;
            p.small_max_long = kSmallMaxLong;
            p.small_no_split = nnz <= o.long_row_min;
            gtattn_status st;
            {
                ProfScope ps(GTATTN_KCAT_ROWS, 1, stream);
                st = launch_rows_small(dtype, c, p, stream);
            }
            pool_free(part_buf, stream);
            return st;
        }
    }
    Scratch sc;
    int *hdr, *rows;
    int2 *chunks, *longs;
    GT_TRY(scratch_alloc(N, nnz, H, H * D, o.long_row_min, o.chunk_edges, false, false, &sc, &hdr, &rows,
                         &chunks, &longs, stream));
    gtattn_status st;
    {
        ProfScope ps(GTATTN_KCAT_BIN, bin_launches((int)N, nullptr), stream);
        st = bin_rows(indptr, (int)N, o.long_row_min, o.chunk_edges, nullptr, hdr, rows, chunks, longs, stream);
    }
    if (st == GTATTN_OK)
        st = rows_in_groups(indptr, indices, Q, K, V, out, N, nnz, H, D, scale, dtype, c, sc.lists, sc.part,
                            sc.part_chunks, bias, values, ndh, nullptr, true, nnz > o.long_row_min,
                            n_src < 0 ? N : n_src, stream);
    pool_free(sc.base, stream);
    return st;
}

extern "C" gtattn_status gtattn_fwd(const int32_t* indptr, const int32_t* indices, const void* Q,
                                    const void* K, const void* V, void* out, int64_t N, int64_t nnz,
                                    int H, int D, float scale, gtattn_dtype dtype, cudaStream_t stream) {
    GT_TRY(check_fwd(indptr, indices, Q, K, V, out, N, nnz, H, D, dtype));
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);
    return fwd_fused(indptr, indices, Q, K, V, nullptr, nullptr, out, N, nnz, H, D, scale, dtype, stream);
}

gtattn_status gt::fwd_view(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                           const void* V, void* out, int64_t N, int64_t nnz, int H, int D, float scale,
                           gtattn_dtype dtype, int64_t n_src, cudaStream_t stream) {
    return fwd_fused(indptr, indices, Q, K, V, nullptr, nullptr, out, N, nnz, H, D, scale, dtype, stream, 0, n_src);
}

// Row-local transpose between [N, D, H] and [N, H, D] (to_hd: from the
// former).  A warp moves R = kMaxHD / (H D) consecutive node rows at a time:
// one contiguous span read into shared memory with 16-byte loads, then each
// lane gathers 16 bytes of a permuted row through the block's permutation
// table and stores them at once (rows of 16-byte multiples, 16-byte
// aligned: the shapes the vector row kernel takes).
template <typename T>
__global__ void __launch_bounds__(256)
k_transpose_rows(const T* __restrict__ src, T* __restrict__ dst, int64_t n, int H, int D, int to_hd) {
    constexpr int kPer = 16 / sizeof(T);   // elements per 16-byte piece
    __shared__ __align__(16) T sm[8][kMaxHD];
    __shared__ short perm[kMaxHD];          // source element of each destination element
    const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HD = H * D, R = kMaxHD / HD, per_row = HD / kPer;
    for (int el = threadIdx.x; el < HD; el += blockDim.x) {
        int from;
        if (to_hd) { const int h = el / D, d = el - h * D; from = d * H + h; }
        else { const int d = el / H, h = el - d * H; from = h * D + d; }
        perm[el] = static_cast<short>(from);
    }
    __syncthreads();
    T* buf = sm[wid];
    const int64_t spans = (n + R - 1) / R;
    for (int64_t sp = blockIdx.x * 8 + wid; sp < spans; sp += static_cast<int64_t>(gridDim.x) * 8) {
        const int64_t row0 = sp * R;
        const int pieces = static_cast<int>(min(static_cast<int64_t>(R), n - row0)) * per_row;
        const uint4* s4 = reinterpret_cast<const uint4*>(src + row0 * HD);
        for (int i = lane; i < pieces; i += 32) reinterpret_cast<uint4*>(buf)[i] = __ldg(s4 + i);
        __syncwarp();
        uint4* d4 = reinterpret_cast<uint4*>(dst + row0 * HD);
        for (int i = lane; i < pieces; i += 32) {
            const int r = i / per_row, el0 = (i - r * per_row) * kPer;
            const T* rs = buf + r * HD;
            __align__(16) T v[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) v[u] = rs[perm[el0 + u]];
            d4[i] = *reinterpret_cast<const uint4*>(v);
        }
        __syncwarp();
    }
}

template <typename T>
static cudaError_t transpose_rows(const void* src, void* dst, int64_t n, int H, int D, int to_hd, cudaStream_t s) {
    const int64_t spans = (n + kMaxHD / (H * D) - 1) / (kMaxHD / (H * D));
    const int blocks = static_cast<int>(std::min<int64_t>((spans + 7) / 8, static_cast<int64_t>(num_sms()) * 8));
    k_transpose_rows<T><<<std::max(blocks, 1), 256, 0, s>>>(static_cast<const T*>(src), static_cast<T*>(dst), n, H, D,
                                                              to_hd);
    return cudaGetLastError();
}

extern "C" gtattn_status gtattn_fwd_ndh(const int32_t* indptr, const int32_t* indices, const void* Q,
                                        const void* K, const void* V, void* out, int64_t N, int64_t nnz, int H,
                                        int D, float scale, gtattn_dtype dtype, cudaStream_t stream) {
    GT_TRY(check_fwd(indptr, indices, Q, K, V, out, N, nnz, H, D, dtype));
    if (N == 0) return GTATTN_OK;
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);
    // Shapes the vector or narrow-head kernel takes: transpose to [N, H, D]
    // in scratch, the head-major forward, transpose the output back (four
    // row-local copies, far cheaper than the generic kernel on head-innermost
    // rows).  Others: the generic kernel reads the [N, D, H] rows directly.
    const size_t esz = dtype == GTATTN_F32 ? 4 : 2, osz = dtype == GTATTN_BF16 ? 2 : 4;
    const size_t in_bytes = align_up(esz * static_cast<size_t>(N) * H * D);
    const size_t out_bytes = align_up(osz * static_cast<size_t>(N) * H * D);
    RowChoice c;
    void* buf = nullptr;
    if (!choose_row_kernel(H, D, dtype, Q, K, V, out, GTATTN_KERNEL_AUTO, &c) || c.kind == RowKernel::kGeneric ||
        pool_alloc(&buf, 3 * in_bytes + out_bytes, stream) != GTATTN_OK)
        return fwd_fused(indptr, indices, Q, K, V, nullptr, nullptr, out, N, nnz, H, D, scale, dtype, stream, 1);
    char* b = static_cast<char*>(buf);
    void *q2 = b, *k2 = b + in_bytes, *v2 = b + 2 * in_bytes, *o2 = b + 3 * in_bytes;
    auto tr = [&](const void* src, void* dst, size_t sz, int to_hd) {
        return sz == 4 ? transpose_rows<float>(src, dst, N, H, D, to_hd, stream)
                       : transpose_rows<__nv_bfloat16>(src, dst, N, H, D, to_hd, stream);
    };
    cudaError_t e = tr(Q, q2, esz, 1);
    if (e == cudaSuccess) e = tr(K, k2, esz, 1);
    if (e == cudaSuccess) e = tr(V, v2, esz, 1);
    gtattn_status st = e == cudaSuccess ? GTATTN_OK : cuda_status(e);
    if (st == GTATTN_OK) st = fwd_fused(indptr, indices, q2, k2, v2, nullptr, nullptr, o2, N, nnz, H, D, scale, dtype, stream);
    if (st == GTATTN_OK) {
        e = tr(o2, out, osz, 0);
        if (e != cudaSuccess) st = cuda_status(e);
    }
    pool_free(buf, stream);
    return st;
}

static gtattn_status fwd_plan(const gtattn_plan* plan, const int32_t* indptr, const int32_t* indices, const void* Q,
                              const void* K, const void* V, void* out, float* stats, int H, int D, float scale,
                              gtattn_dtype dtype, cudaStream_t stream);

extern "C" gtattn_status gtattn_fwd_plan(const gtattn_plan* plan, const int32_t* indptr,
                                         const int32_t* indices, const void* Q, const void* K,
                                         const void* V, void* out, int H, int D, float scale,
                                         gtattn_dtype dtype, cudaStream_t stream) {
    return fwd_plan(plan, indptr, indices, Q, K, V, out, nullptr, H, D, scale, dtype, stream);
}

extern "C" gtattn_status gtattn_fwd_plan_stats(const gtattn_plan* plan, const int32_t* indptr,
                                               const int32_t* indices, const void* Q, const void* K,
                                               const void* V, void* out, float* stats, int H, int D, float scale,
                                               gtattn_dtype dtype, cudaStream_t stream) {
    if (!stats || (reinterpret_cast<uintptr_t>(stats) & 3u)) return GTATTN_ERR_INVALID_ARG;
    return fwd_plan(plan, indptr, indices, Q, K, V, out, stats, H, D, scale, dtype, stream);
}

static gtattn_status fwd_plan(const gtattn_plan* plan, const int32_t* indptr, const int32_t* indices, const void* Q,
                              const void* K, const void* V, void* out, float* stats, int H, int D, float scale,
                              gtattn_dtype dtype, cudaStream_t stream) {
    if (!plan) return GTATTN_ERR_INVALID_ARG;
    const int64_t N = plan->N, nnz = plan->nnz;
    GT_TRY(check_fwd(indptr, indices, Q, K, V, out, N, nnz, H, D, dtype));
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);
    RowChoice c;
    if (!choose_row_kernel(H, D, dtype, Q, K, V, out, plan->opts.kernel, &c)) return GTATTN_ERR_UNSUPPORTED;
    if (N == 0) return GTATTN_OK;
    const int HD = H * D;
    const int n_chunks = plan->hdr_host[HdrLayout::kChunks];
    const int n_long = plan->hdr_host[HdrLayout::kLong];
    const int n_blocks = plan->hdr_host[HdrLayout::kDenseBlocks];
    // (the dense-block kernel writes no row statistics: with stats, every row
    // goes through the row kernels)
    const bool dense = n_blocks > 0 && !stats && dense_supported(H, D, dtype, Q, K, V, out);

    Partials part{};
    if (n_chunks > 0) {
        const size_t need = align_up(sizeof(float) * (size_t)n_chunks * H) * 2 +
                            align_up(sizeof(float) * (size_t)n_chunks * HD);
        if (plan->ws_bytes < need) {
            pool_free(plan->ws, stream);
            plan->ws = nullptr;
            plan->ws_bytes = 0;
            GT_TRY(pool_alloc(&plan->ws, need, stream));
            plan->ws_bytes = need;
        }
        char* b = static_cast<char*>(plan->ws);
        part.m = reinterpret_cast<float*>(b);
        part.s = reinterpret_cast<float*>(b + align_up(sizeof(float) * (size_t)n_chunks * H));
        part.acc = reinterpret_cast<float*>(b + 2 * align_up(sizeof(float) * (size_t)n_chunks * H));
    }
    TaskLists L{plan->hdr, plan->rows, plan->chunks, plan->longs, plan->opts.chunk_edges, dense ? 0 : 1};
    gtattn_status st = GTATTN_OK;
    if (dense) {
        ProfScope ps(GTATTN_KCAT_DENSE, 1, stream);
        st = launch_dense(plan->dense_tiles, plan->dense_tiles1, plan->n_dense_tiles, plan->n_dense_tiles1, N, Q, K,
                          V, out, H, D, scale, dtype,
                          plan->hdr + HdrLayout::kErr, plan->opts.wait_cycles, plan->opts.test_stall, stream);
    }
    int row_tasks = n_chunks + (dense ? 0 : plan->hdr_host[HdrLayout::kDenseRows]);
    for (int b = 0; b < kNumBuckets; ++b) row_tasks += plan->hdr_host[HdrLayout::kCount + b];
    if (st == GTATTN_OK && (row_tasks > 0 || n_long > 0))
        st = rows_in_groups(indptr, indices, Q, K, V, out, N, nnz, H, D, scale, dtype, c, L, part, n_chunks, nullptr,
                            nullptr, 0, stats, row_tasks > 0, n_long > 0, N, stream);
    return st;
}

// The unfused trio (SDDMM, edge softmax, SpMM), with an optional per-entry
// additive bias or per-entry adjacency values in the SDDMM.
static gtattn_status fwd_unfused(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                                 const void* V, const float* values, const float* bias, void* out, float* logits,
                                 float* probs, int64_t N, int64_t nnz, int H, int D, float scale,
                                 gtattn_dtype dtype, cudaStream_t stream) {
    GT_TRY(check_fwd(indptr, indices, Q, K, V, out, N, nnz, H, D, dtype));
    if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(probs)) & 3u)
        return GTATTN_ERR_INVALID_ARG;
    RowChoice c;
    if (!choose_row_kernel(H, D, dtype, Q, K, V, out, GTATTN_KERNEL_AUTO, &c)) return GTATTN_ERR_UNSUPPORTED;
    if (N == 0) return GTATTN_OK;
    gtattn_plan_opts o;
    resolve_opts(nullptr, &o);
    Scratch sc;
    int *hdr, *rows;
    int2 *chunks, *longs;
    GT_TRY(scratch_alloc(N, nnz, H, H * D, o.long_row_min, o.chunk_edges, logits == nullptr,
                         probs == nullptr, &sc, &hdr, &rows, &chunks, &longs, stream));
    float* lg = logits ? logits : sc.logits;
    float* pr = probs ? probs : sc.probs;
    gtattn_status st;
    {
        ProfScope ps(GTATTN_KCAT_BIN, bin_launches((int)N, nullptr), stream);
        st = bin_rows(indptr, (int)N, o.long_row_min, o.chunk_edges, nullptr, hdr, rows, chunks, longs, stream);
    }
    RowParams p = make_params(indptr, indices, Q, K, V, out, N, nnz, H, D, scale, c, sc.lists, sc.part);
    p.logits = lg;
    p.probs = pr;
    p.bias = bias;
    p.values = values;
    // (1) SDDMM: logits
    if (st == GTATTN_OK && nnz > 0) {
        ProfScope ps(GTATTN_KCAT_ROWS, 1, stream);
        st = launch_rows(kSddmm, dtype, c, p, stream);
    }
    // (2) edge softmax: probs
    if (st == GTATTN_OK && nnz > 0) {
        ProfScope ps(GTATTN_KCAT_SOFTMAX, 4, stream);
        st = launch_edge_softmax(indptr, (int)N, H, sc.lists, sc.part, lg, pr, stream);
    }
    // (3) SpMM: out
    if (st == GTATTN_OK) {
        ProfScope ps(GTATTN_KCAT_ROWS, 1, stream);
        st = launch_rows(kSpmm, dtype, c, p, stream);
    }
    if (st == GTATTN_OK && nnz > o.long_row_min) {   // else no row is split
        ProfScope ps(GTATTN_KCAT_COMBINE, 1, stream);
        st = launch_combine(kSpmm, dtype, p, stream);
    }
    pool_free(sc.base, stream);
    return st;
}

extern "C" gtattn_status gtattn_fwd_probs(const int32_t* indptr, const int32_t* indices, const void* Q,
                                          const void* K, const void* V, void* out, float* logits,
                                          float* probs, int64_t N, int64_t nnz, int H, int D, float scale,
                                          gtattn_dtype dtype, cudaStream_t stream) {
    GT_TRY(check_fwd(indptr, indices, Q, K, V, out, N, nnz, H, D, dtype));
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);
    return fwd_unfused(indptr, indices, Q, K, V, nullptr, nullptr, out, logits, probs, N, nnz, H, D, scale, dtype,
                       stream);
}

extern "C" gtattn_status gtattn_fwd_bias(const int32_t* indptr, const int32_t* indices, const void* Q,
                                         const void* K, const void* V, const float* bias, void* out,
                                         float* logits, float* probs, int64_t N, int64_t nnz, int H, int D,
                                         float scale, gtattn_dtype dtype, cudaStream_t stream) {
    if ((nnz > 0 && !bias) || (reinterpret_cast<uintptr_t>(bias) & 3u)) return GTATTN_ERR_INVALID_ARG;
    GT_TRY(check_fwd(indptr, indices, Q, K, V, out, N, nnz, H, D, dtype));
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);
    if (logits || probs)
        return fwd_unfused(indptr, indices, Q, K, V, nullptr, bias, out, logits, probs, N, nnz, H, D, scale, dtype,
                           stream);
    return fwd_fused(indptr, indices, Q, K, V, nullptr, bias, out, N, nnz, H, D, scale, dtype, stream);
}

extern "C" gtattn_status gtattn_fwd_weighted(const int32_t* indptr, const int32_t* indices, const float* values,
                                             const void* Q, const void* K, const void* V, void* out, float* logits,
                                             float* probs, int64_t N, int64_t nnz, int H, int D, float scale,
                                             gtattn_dtype dtype, cudaStream_t stream) {
    if ((nnz > 0 && !values) || (reinterpret_cast<uintptr_t>(values) & 3u)) return GTATTN_ERR_INVALID_ARG;
    GT_TRY(check_fwd(indptr, indices, Q, K, V, out, N, nnz, H, D, dtype));
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);
    if (logits || probs)
        return fwd_unfused(indptr, indices, Q, K, V, values, nullptr, out, logits, probs, N, nnz, H, D, scale, dtype,
                           stream);
    return fwd_fused(indptr, indices, Q, K, V, values, nullptr, out, N, nnz, H, D, scale, dtype, stream);
}


// ---------------------------------------------------------------------------
// backward
// ---------------------------------------------------------------------------
// The source-major copy of a graph's pattern (colptr over sources, rowid:
// the destination rows, ascending within a source) and the binning of its
// sources, carved from one block; and the scratch its build needs.
struct SourceMajor {
    int* colptr = nullptr;
    int* rowid = nullptr;
    TaskLists cols{};
    int64_t max_chunks = 0;   // capacity of the source chunk list
    // the destination rows binned with the same thresholds, for the
    // by-destination pass (rows cut into chunks of the backward's size: a
    // lane group walks a task's entries in order, so long tasks become a tail)
    TaskLists dq{};
    int64_t dq_chunks = 0;    // capacity of its chunk list
};

static size_t source_major_carve(char* base, int64_t N, int64_t nnz, const gtattn_plan_opts& o, SourceMajor* sm) {
    int64_t n_long = 0, n_chunks = 0;
    worst_case_sizes(N, nnz, o.long_row_min, o.chunk_edges, &n_long, &n_chunks);
    size_t off = 0;
    const size_t o_cp = off; off = align_up(off + sizeof(int) * static_cast<size_t>(N + 1));
    const size_t o_rid = off; off = align_up(off + sizeof(int) * static_cast<size_t>(nnz));
    const size_t o_h = off; off = align_up(off + sizeof(int) * HdrLayout::kWords);
    const size_t o_r = off; off = align_up(off + sizeof(int) * static_cast<size_t>(N));
    const size_t o_c = off; off = align_up(off + sizeof(int2) * static_cast<size_t>(n_chunks));
    const size_t o_l = off; off = align_up(off + sizeof(int2) * static_cast<size_t>(n_long));
    const size_t o_dh = off; off = align_up(off + sizeof(int) * HdrLayout::kWords);
    const size_t o_dr = off; off = align_up(off + sizeof(int) * static_cast<size_t>(N));
    const size_t o_dc = off; off = align_up(off + sizeof(int2) * static_cast<size_t>(n_chunks));
    const size_t o_dl = off; off = align_up(off + sizeof(int2) * static_cast<size_t>(n_long));
    if (base && sm) {
        sm->colptr = reinterpret_cast<int*>(base + o_cp);
        sm->rowid = reinterpret_cast<int*>(base + o_rid);
        sm->cols = TaskLists{reinterpret_cast<int*>(base + o_h), reinterpret_cast<int*>(base + o_r),
                             reinterpret_cast<int2*>(base + o_c), reinterpret_cast<int2*>(base + o_l), o.chunk_edges, 1};
        sm->max_chunks = n_chunks;
        sm->dq = TaskLists{reinterpret_cast<int*>(base + o_dh), reinterpret_cast<int*>(base + o_dr),
                           reinterpret_cast<int2*>(base + o_dc), reinterpret_cast<int2*>(base + o_dl), o.chunk_edges, 1};
        sm->dq_chunks = n_chunks;   // (same thresholds, N and nnz: the same worst case)
    }
    return off;
}

// Builds *sm (carved already) from the destination binning `rows`: counts,
// scan, scatter, segment sort, the source binning, then the destination
// rows binned again with the source thresholds (for the by-destination
// pass).  Scratch from the pool.
static gtattn_status source_major_build(const int32_t* indptr, const int32_t* indices, const TaskLists& rows,
                                        int64_t N, int64_t nnz, const gtattn_plan_opts& o, const SourceMajor& sm,
                                        cudaStream_t stream) {
    size_t off = 0;
    const size_t o_cur = off; off = align_up(off + sizeof(int) * static_cast<size_t>(N));
    const size_t o_ts = off; off = align_up(off + sizeof(int) * static_cast<size_t>(bwd_scan_tiles(N) + 1));
    const size_t o_tmp = off; off = align_up(off + sizeof(int) * static_cast<size_t>(nnz));
    void* scr = nullptr;
    GT_TRY(pool_alloc(&scr, off, stream));
    char* b = static_cast<char*>(scr);
    gtattn_status st;
    {
        ProfScope ps(GTATTN_KCAT_BIN, 5 + (nnz > 0) + 4 * (nnz > 0) + bin_launches((int)N, nullptr), stream);
        st = build_csc(indptr, indices, rows, (int)N, nnz, sm.colptr, reinterpret_cast<int*>(b + o_cur),
                       reinterpret_cast<int*>(b + o_ts), sm.rowid, reinterpret_cast<int*>(b + o_tmp), sm.cols,
                       o.long_row_min, stream);
    }
    if (st == GTATTN_OK) {
        ProfScope ps(GTATTN_KCAT_BIN, bin_launches((int)N, nullptr), stream);
        // (the lists are this pattern's own memory, carved writable)
        st = bin_rows(indptr, (int)N, o.long_row_min, o.chunk_edges, nullptr, const_cast<int*>(sm.dq.hdr),
                      const_cast<int*>(sm.dq.rows), const_cast<int2*>(sm.dq.chunks), const_cast<int2*>(sm.dq.longs),
                      stream);
    }
    pool_free(scr, stream);
    return st;
}

// The source binning's split thresholds: the backward's own (a task per
// source of up to kBwdLongMin entries, kBwdChunk-entry chunks above) unless
// the plan's thresholds were set away from the forward's defaults.
static gtattn_plan_opts source_opts(const gtattn_plan_opts& o) {
    gtattn_plan_opts s = o;
    if (s.long_row_min == kDefaultLongMin && s.chunk_edges == kDefaultChunk) {
        s.long_row_min = kBwdLongMin;
        s.chunk_edges = kBwdChunk;
    }
    return s;
}

// Host-side checks of the backward entry points.
static gtattn_status check_bwd(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                               const void* V, const void* dO, const float* dQ, const float* dK, const float* dV,
                               int64_t N, int64_t nnz, int H, int D, gtattn_dtype dtype) {
    if (N < 0 || nnz < 0 || N >= (1ll << 31) - 1 || nnz >= (1ll << 31) - 1) return GTATTN_ERR_INVALID_ARG;
    if (H < 1 || D < 1 || (int64_t)H * D > kMaxHD || H > kBwdMaxHeads) return GTATTN_ERR_INVALID_ARG;
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
    return GTATTN_OK;
}

// The two-pass backward given the forward's destination binning (rows, with
// row_chunks chunk slots) and the source-major pattern: the forward again for
// its fp32 output and log-sum-exp (unless the caller saved both), then the
// passes (by destination over the pattern's own destination binning, by
// source over its source binning).
static gtattn_status bwd_run(const int32_t* indptr, const int32_t* indices, const TaskLists& rows, int64_t row_chunks,
                             const SourceMajor& sm, const void* Q, const void* K, const void* V, const float* O_saved,
                             const float* stats_saved, const void* dO, float* dQ, float* dK, float* dV, int64_t N,
                             int64_t nnz, int H, int D, float scale, gtattn_dtype dtype, const RowChoice& c,
                             cudaStream_t stream) {
    const int HD = H * D;
    const gtattn_dtype fdt = dtype == GTATTN_F32 ? GTATTN_F32 : GTATTN_BF16_OUT_F32;   // fp32 forward output
    const size_t grad_bytes = sizeof(float) * static_cast<size_t>(N) * HD;
    size_t off = 0;
    const bool saved = O_saved != nullptr;
    const size_t o_O = off; if (!saved) off = align_up(off + grad_bytes);
    const size_t o_L = off; if (!saved) off = align_up(off + sizeof(float) * static_cast<size_t>(N) * H);
    const size_t o_LD = off; off = align_up(off + sizeof(float2) * static_cast<size_t>(N) * H);
    const int64_t fwd_chunks = saved ? 0 : row_chunks;   // the forward's partials
    const size_t o_m = off; off = align_up(off + sizeof(float) * static_cast<size_t>(fwd_chunks) * H);
    const size_t o_s = off; off = align_up(off + sizeof(float) * static_cast<size_t>(fwd_chunks) * H);
    const size_t o_acc = off; off = align_up(off + sizeof(float) * static_cast<size_t>(fwd_chunks) * HD);
    const size_t o_pq = off; off = align_up(off + sizeof(float) * static_cast<size_t>(sm.dq_chunks) * HD);
    const size_t o_pk = off; off = align_up(off + sizeof(float) * static_cast<size_t>(sm.max_chunks) * HD);
    const size_t o_pv = off; off = align_up(off + sizeof(float) * static_cast<size_t>(sm.max_chunks) * HD);
    void* buf = nullptr;
    GT_TRY(pool_alloc(&buf, off, stream));
    char* b = static_cast<char*>(buf);
    float* O = reinterpret_cast<float*>(b + o_O);
    float* lse = reinterpret_cast<float*>(b + o_L);
    Partials part{reinterpret_cast<float*>(b + o_m), reinterpret_cast<float*>(b + o_s),
                  reinterpret_cast<float*>(b + o_acc)};
    gtattn_status st = GTATTN_OK;
    if (saved) {   // the forward's fp32 output and row statistics, kept by the caller
        O = const_cast<float*>(O_saved);
        lse = const_cast<float*>(stats_saved);
    } else {          // the forward again
        RowParams p = make_params(indptr, indices, Q, K, V, O, N, nnz, H, D, scale * kLog2e, c, rows, part);
        p.lse = lse;
        {
            ProfScope ps(GTATTN_KCAT_ROWS, 1, stream);
            st = launch_rows(kFused, fdt, c, p, stream);
        }
        if (st == GTATTN_OK && row_chunks > 0) {
            ProfScope ps(GTATTN_KCAT_COMBINE, 1, stream);
            st = launch_combine(kFused, fdt, p, stream);
        }
    }
    if (st == GTATTN_OK) {
        ProfScope ps(GTATTN_KCAT_ROWS, 4, stream);
        st = launch_bwd_passes(indptr, indices, sm.dq, sm.colptr, sm.rowid, sm.cols, Q, K, V, dO, O, lse,
                               reinterpret_cast<float2*>(b + o_LD), dQ, dK, dV, reinterpret_cast<float*>(b + o_pq),
                               reinterpret_cast<float*>(b + o_pk), reinterpret_cast<float*>(b + o_pv), (int)N, nnz, H,
                               D, scale, dtype, stream);
    }
    pool_free(buf, stream);
    return st;
}

// Shapes the two passes do not take: a warp per row with scalar atomics.
static gtattn_status bwd_fallback(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                                  const void* V, const void* dO, float* dQ, float* dK, float* dV, int64_t N, int H,
                                  int D, float scale, gtattn_dtype dtype, cudaStream_t stream) {
    const size_t grad_bytes = sizeof(float) * static_cast<size_t>(N) * H * D;
    GT_CUDA(cudaMemsetAsync(dQ, 0, grad_bytes, stream));
    GT_CUDA(cudaMemsetAsync(dK, 0, grad_bytes, stream));
    GT_CUDA(cudaMemsetAsync(dV, 0, grad_bytes, stream));
    ProfScope ps(GTATTN_KCAT_ROWS, 1, stream);
    return launch_bwd_rows(indptr, indices, Q, K, V, dO, dQ, dK, dV, (int)N, H, D, scale, dtype, stream);
}

static bool bwd_two_pass(int H, int D, gtattn_dtype dtype, const void* Q, const void* K, const void* V,
                         const void* dO, const float* dQ, const float* dK, const float* dV, RowChoice* c) {
    const void* ptrs[7] = {Q, K, V, dO, dQ, dK, dV};
    const gtattn_dtype fdt = dtype == GTATTN_F32 ? GTATTN_F32 : GTATTN_BF16_OUT_F32;
    return bwd_tasks_supported(H, D, dtype, ptrs, 7) &&
           choose_row_kernel(H, D, fdt, Q, K, V, dQ, GTATTN_KERNEL_AUTO, c);
}

extern "C" gtattn_status gtattn_bwd(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                                    const void* V, const void* dO, float* dQ, float* dK, float* dV, int64_t N,
                                    int64_t nnz, int H, int D, float scale, gtattn_dtype dtype,
                                    cudaStream_t stream) {
    GT_TRY(check_bwd(indptr, indices, Q, K, V, dO, dQ, dK, dV, N, nnz, H, D, dtype));
    if (N == 0) return GTATTN_OK;
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);
    RowChoice c;
    if (!bwd_two_pass(H, D, dtype, Q, K, V, dO, dQ, dK, dV, &c))
        return bwd_fallback(indptr, indices, Q, K, V, dO, dQ, dK, dV, N, H, D, scale, dtype, stream);
    gtattn_plan_opts o;
    resolve_opts(nullptr, &o);
    const gtattn_plan_opts so = source_opts(o);
    Scratch sc;
    int *hdr, *rows;
    int2 *chunks, *longs;
    GT_TRY(scratch_alloc(N, nnz, H, H * D, o.long_row_min, o.chunk_edges, false, false, &sc, &hdr, &rows, &chunks,
                         &longs, stream));
    int64_t n_long = 0, row_chunks = 0;
    worst_case_sizes(N, nnz, o.long_row_min, o.chunk_edges, &n_long, &row_chunks);
    void* smb = nullptr;
    gtattn_status st = pool_alloc(&smb, source_major_carve(nullptr, N, nnz, so, nullptr), stream);
    SourceMajor sm;
    if (st == GTATTN_OK) {
        source_major_carve(static_cast<char*>(smb), N, nnz, so, &sm);
        ProfScope ps(GTATTN_KCAT_BIN, bin_launches((int)N, nullptr), stream);
        st = bin_rows(indptr, (int)N, o.long_row_min, o.chunk_edges, nullptr, hdr, rows, chunks, longs, stream);
    }
    if (st == GTATTN_OK) st = source_major_build(indptr, indices, sc.lists, N, nnz, so, sm, stream);
    if (st == GTATTN_OK)
        st = bwd_run(indptr, indices, sc.lists, row_chunks, sm, Q, K, V, nullptr, nullptr, dO, dQ, dK, dV, N, nnz, H, D,
                     scale, dtype, c, stream);
    pool_free(smb, stream);
    pool_free(sc.base, stream);
    return st;
}

extern "C" gtattn_status gtattn_bwd_plan(const gtattn_plan* plan, const int32_t* indptr, const int32_t* indices,
                                         const void* Q, const void* K, const void* V, const float* O,
                                         const float* stats, const void* dO, float* dQ, float* dK, float* dV, int H,
                                         int D, float scale, gtattn_dtype dtype, cudaStream_t stream) {
    if (!plan) return GTATTN_ERR_INVALID_ARG;
    const int64_t N = plan->N, nnz = plan->nnz;
    GT_TRY(check_bwd(indptr, indices, Q, K, V, dO, dQ, dK, dV, N, nnz, H, D, dtype));
    // O is read as whole float4 rows by the passes
    if ((O == nullptr) != (stats == nullptr) || (reinterpret_cast<uintptr_t>(O) & 15u) ||
        (reinterpret_cast<uintptr_t>(stats) & 3u))
        return GTATTN_ERR_INVALID_ARG;
    if (N == 0) return GTATTN_OK;
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);
    RowChoice c;
    if (!bwd_two_pass(H, D, dtype, Q, K, V, dO, dQ, dK, dV, &c))
        return bwd_fallback(indptr, indices, Q, K, V, dO, dQ, dK, dV, N, H, D, scale, dtype, stream);
    // the plan's destination binning, dense segment included (the forward
    // is recomputed by the row kernels for every row)
    const TaskLists rows{plan->hdr, plan->rows, plan->chunks, plan->longs, plan->opts.chunk_edges, 1};
    const int64_t row_chunks = plan->hdr_host[HdrLayout::kChunks];
    SourceMajor sm;
    const gtattn_plan_opts so = source_opts(plan->opts);
    if (!plan->bwd_pattern) {   // first backward with this plan: the source-major pattern, kept
        void* p = nullptr;
        GT_CUDA(cudaMalloc(&p, source_major_carve(nullptr, N, nnz, so, nullptr)));
        source_major_carve(static_cast<char*>(p), N, nnz, so, &sm);
        const gtattn_status st = source_major_build(indptr, indices, rows, N, nnz, so, sm, stream);
        if (st != GTATTN_OK) {
            cudaStreamSynchronize(stream);
            cudaFree(p);
            return st;
        }
        plan->bwd_pattern = p;
    }
    source_major_carve(static_cast<char*>(plan->bwd_pattern), N, nnz, so, &sm);
    return bwd_run(indptr, indices, rows, row_chunks, sm, Q, K, V, O, stats, dO, dQ, dK, dV, N, nnz, H, D, scale,
                   dtype, c, stream);
}

// The attention block with its projections: q, k, v = X W^T + b (one GEMM
// over the stacked weights, written as three [N, H, D] matrices), the fused
// sparse attention, Y = o Wo^T + bo.
extern "C" gtattn_status gtattn_fwd_proj(const int32_t* indptr, const int32_t* indices, const void* X,
                                         const void* Wqkv, const float* bqkv, const void* Wo, const float* bo,
                                         void* Y, void* qkv, void* attn, int64_t N, int64_t nnz, int F_in, int H,
                                         int D, int F_out, int heads_inner, float scale, gtattn_dtype dtype,
                                         cudaStream_t stream) {
    if (N < 0 || nnz < 0 || N >= (1ll << 31) - 1 || nnz >= (1ll << 31) - 1) return GTATTN_ERR_INVALID_ARG;
    if (F_in < 1 || F_out < 1 || H < 1 || D < 1 || (int64_t)H * D > kMaxHD) return GTATTN_ERR_INVALID_ARG;
    if (dtype != GTATTN_F32 && dtype != GTATTN_BF16 && dtype != GTATTN_BF16_OUT_F32) return GTATTN_ERR_INVALID_ARG;
    if (heads_inner != 0 && heads_inner != 1) return GTATTN_ERR_INVALID_ARG;
    if (!indptr || (nnz > 0 && !indices)) return GTATTN_ERR_INVALID_ARG;
    if (N > 0 && (!X || !Wqkv || !Wo || !Y)) return GTATTN_ERR_INVALID_ARG;
    const bool bf = dtype != GTATTN_F32;
    const size_t esz = bf ? 2 : 4, osz = dtype == GTATTN_BF16 ? 2 : 4;
    const uintptr_t in_al = reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(Wqkv) |
                            reinterpret_cast<uintptr_t>(Wo) | reinterpret_cast<uintptr_t>(qkv) |
                            reinterpret_cast<uintptr_t>(attn);
    const uintptr_t f_al = reinterpret_cast<uintptr_t>(bqkv) | reinterpret_cast<uintptr_t>(bo) |
                           reinterpret_cast<uintptr_t>(indptr) | reinterpret_cast<uintptr_t>(indices);
    if ((in_al & (esz - 1)) || (f_al & 3u) || (reinterpret_cast<uintptr_t>(Y) & (osz - 1)))
        return GTATTN_ERR_INVALID_ARG;
    if (N == 0) return GTATTN_OK;
    GT_DEBUG_CSR(indptr, indices, N, nnz, stream);
    const int HD = H * D;
    const int64_t nhd = N * HD;
    // temporaries: q, k, v and the attention output unless the caller keeps
    // them; the weights in head-major feature order for head-inner features
    size_t off = 0;
    const size_t o_qkv = off; if (!qkv) off = align_up(off + 3 * esz * static_cast<size_t>(nhd));
    const size_t o_att = off; if (!attn) off = align_up(off + esz * static_cast<size_t>(nhd));
    const size_t o_w1 = off, o_b1 = align_up(off + esz * 3 * static_cast<size_t>(HD) * F_in);
    const size_t o_w2 = align_up(o_b1 + 4 * 3 * static_cast<size_t>(HD));
    if (heads_inner) off = align_up(o_w2 + esz * static_cast<size_t>(F_out) * HD);
    void* buf = nullptr;
    if (off > 0) GT_TRY(pool_alloc(&buf, off, stream));
    char* b = static_cast<char*>(buf);
    char* q = qkv ? static_cast<char*>(qkv) : b + o_qkv;
    void* o = attn ? attn : b + o_att;
    const void* W1 = Wqkv;
    const float* b1 = bqkv;
    const void* W2 = Wo;
    gtattn_status st = GTATTN_OK;
    if (heads_inner) {   // SparseMHA's reshape(N, head_dim, num_heads): feature d*H + h is head h, element d
        ProfScope ps(GTATTN_KCAT_GEMM, 2, stream);
        st = launch_permute_rows(Wqkv, b + o_w1, bqkv, bqkv ? reinterpret_cast<float*>(b + o_b1) : nullptr, 3, H, D,
                                 F_in, static_cast<int>(esz), stream);
        if (st == GTATTN_OK) st = launch_permute_cols(Wo, b + o_w2, F_out, H, D, static_cast<int>(esz), stream);
        W1 = b + o_w1;
        b1 = bqkv ? reinterpret_cast<const float*>(b + o_b1) : nullptr;
        W2 = b + o_w2;
    }
    // q, k, v: column c of X W^T goes to matrix c / HD, column c % HD
    if (st == GTATTN_OK) {
        ProfScope ps(GTATTN_KCAT_GEMM, 1, stream);
        const GemmOut o1{q, nhd, HD, HD};
        st = bf && gemm_tc_supported(X, W1, F_in, o1, false)
                 ? launch_gemm_tc(X, W1, b1, N, 3 * HD, F_in, o1, false, stream)
                 : launch_gemm_simt(X, W1, b1, N, 3 * HD, F_in, bf, o1, !bf, stream);
    }
    if (st == GTATTN_OK)
        st = fwd_fused(indptr, indices, q, q + esz * nhd, q + 2 * esz * nhd, nullptr, nullptr, o, N, nnz, H, D, scale,
                       bf ? GTATTN_BF16 : GTATTN_F32, stream);
    if (st == GTATTN_OK) {
        ProfScope ps(GTATTN_KCAT_GEMM, 1, stream);
        const GemmOut o2{Y, 0, F_out, F_out};
        const bool y32 = osz == 4;
        st = bf && gemm_tc_supported(o, W2, HD, o2, y32) ? launch_gemm_tc(o, W2, bo, N, F_out, HD, o2, y32, stream)
                                                          : launch_gemm_simt(o, W2, bo, N, F_out, HD, bf, o2, y32, stream);
    }
    pool_free(buf, stream);
    return st;
}
