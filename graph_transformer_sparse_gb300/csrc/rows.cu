// rows.cu -- the sparse row kernels.
//
// One pass per row computes, for every head h, the logits
// l_e = scale * <q_i, k_j> of the row's entries, their softmax and the
// weighted sum of v_j ("Graph Transformer in a Nutshell", Sparse Multi-head
// Attention: bsddmm -> softmax -> bspmm; "Efficient Sparse Transformer
// implementation with DGL's builtin operators", TransLayer.forward:
// u_dot_v -> edge_softmax -> u_mul_e_sum).  The pages run these as three
// library calls with the per-edge scores in memory; here they are fused:
// logits live in registers, the softmax is an online one (running max m and
// sum s, rescaled by 2^(m_old - m_new) when the max grows), accumulation is
// fp32.  Logits are kept in log2 units (q pre-multiplied by scale*log2(e))
// so every exponential is one ex2.
//
// Lane layout of the vector kernel: a group of G lanes covers one feature row
// of H*D elements, E = 16*VPL/sizeof(T) contiguous elements per lane, so a
// gather of K_j or V_j is G 16-byte-vector loads per lane-group.  lph = D/E
// lanes share a head and reduce their partial dot products with xor
// shuffles.  A warp holds P = 32/G groups; a task assigns them as R rows x S
// edge slots (R*S = P), chosen per degree bucket so short rows share a warp
// and longer rows spread their edges over slots; slots merge their softmax
// states with shuffles at the end.  Rows longer than the split threshold are
// cut into chunks; a chunk writes its (m, s, acc) partial and the combine
// kernel merges them: m* = max m_c, s* = sum s_c 2^(m_c-m*),
// out = sum acc_c 2^(m_c-m*) / s*.
#include "rows.cuh"

#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>
#include <unordered_map>

namespace gt {

constexpr unsigned kFull = 0xffffffffu;

// kSegCopy: rows of exactly one entry, whose output is that neighbour's V
// row (the softmax of one score is 1), taken by the fused kernel without
// reading q or k.
enum SegKind { kSegChunk = 0, kSegRows = 1, kSegCopy = 2 };

struct Seg {
    int first_task;
    int list_begin;
    int count;
    int R, S;
    int kind;
};

constexpr int kMaxSegs = kNumBuckets + 2;
constexpr int kRowBlockMax = 256;   // threads a row-kernel block has at most
constexpr float kLazyMax = 8.f;   // fused row kernel: slack of the running maximum (log2 units)

// Head of feature element el of a node row: [N, H, D] rows are head-major
// (el / D), [N, D, H] rows head-innermost (el % H).
__device__ __forceinline__ int head_of(int el, int D, int H, int ndh) { return ndh ? el % H : el / D; }

// Loads of data read once per call (the bias, and with GT_STREAM_HINTS the
// indices and Q rows) use the streaming cache policy (evict first), so they
// do not push the reused K/V rows out of the L2.
__device__ __forceinline__ float ld_stream(const float* p) { return __ldcs(p); }
__device__ __forceinline__ int ld_stream(const int* p) { return __ldcs(p); }
#ifndef GT_STREAM_HINTS
#define GT_STREAM_HINTS 0
#endif
__device__ __forceinline__ int ld_index(const int* p) {
    if constexpr (GT_STREAM_HINTS) return __ldcs(p);
    else return __ldg(p);
}

// Programmatic dependent launch: the row and combine kernels are launched
// while the kernel before them in the stream (binning, rows) is still
// running, and wait here until it has finished and its writes are visible
// (a no-op for a launch without the attribute).
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Iterations a slot of a row's entries is sized for (more slots per row:
// fewer iterations, more slot merges).
#ifndef GT_SLOT_ITERS
#define GT_SLOT_ITERS 128
#endif

// Builds the task table of a launch in shared memory (one warp).
// P = edge slots per warp; U = edges per slot per loop iteration.
__device__ void build_segments(const TaskLists& L, int P, int U, Seg* segs, int* nseg, int* total,
                               bool copy_deg1 = false) {
    __shared__ int h[HdrLayout::kWords];
    for (int k = threadIdx.x; k < HdrLayout::kWords; k += blockDim.x) h[k] = L.hdr[k];
    __syncthreads();
    if (threadIdx.x == 0) {
        int t = 0, k = 0;
        int nch = h[HdrLayout::kChunks];
        if (nch > 0) { segs[k++] = Seg{t, 0, nch, 1, P, kSegChunk}; t += nch; }
        for (int b = kNumBuckets - 1; b >= 0; --b) {
            int cnt = h[HdrLayout::kCount + b];
            if (cnt == 0) continue;
            int lo = bucket_lo(b);
            if (copy_deg1 && lo == 1 && bucket_lo(b + 1) == 2) {   // the degree-1 bucket
                segs[k++] = Seg{t, h[HdrLayout::kOffset + b], cnt, P, 1, kSegCopy};
                t += (cnt + P - 1) / P;
                continue;
            }
            // slots: enough to cover the row in about GT_SLOT_ITERS (128)
            // iterations, so short rows get one lane group each (4 rows per
            // warp on R-MAT) and walk their entries in order; more slots per
            // row cost slot merges and idle slots on the last iteration
            // (R-MAT: 1.16 ms with one iteration per row, 1.00 ms with 32;
            // with 1024-entry chunks, 0.921 ms at 32, 0.903 at 128, 0.924 at
            // 256, 0.96 at 512)
            int need = (lo + GT_SLOT_ITERS * U - 1) / (GT_SLOT_ITERS * U);
            int S = 1;
            while (S < need && S < P) S <<= 1;
            int R = P / S;
            segs[k++] = Seg{t, h[HdrLayout::kOffset + b], cnt, R, S, kSegRows};
            t += (cnt + R - 1) / R;
        }
        if (L.include_dense) {
            int cnt = h[HdrLayout::kDenseRows];
            if (cnt > 0) { segs[k++] = Seg{t, h[HdrLayout::kDenseSeg], cnt, 1, P, kSegRows}; t += cnt; }
        }
        *nseg = k;
        *total = t;
    }
    __syncthreads();
}

// Block-wide exclusive scan of two counts (every thread of the block calls
// it); *tot_a / *tot_b receive the block's totals.
__device__ __forceinline__ int2 block_scan2(int a, int b, int* tot_a, int* tot_b) {
    __shared__ int wa[kRowBlockMax / 32], wb[kRowBlockMax / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = a, y = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int xo = __shfl_up_sync(0xffffffffu, x, o), yo = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) { x += xo; y += yo; }
    }
    if (lane == 31) { wa[wid] = x; wb[wid] = y; }
    __syncthreads();
    int pa = 0, pb = 0, ta = 0, tb = 0;
    for (int k = 0; k < nw; ++k) {
        if (k < wid) { pa += wa[k]; pb += wb[k]; }
        ta += wa[k];
        tb += wb[k];
    }
    *tot_a = ta;
    *tot_b = tb;
    __syncthreads();   // wa / wb are reused by the next call
    return make_int2(pa + x - a, pb + y - b);
}

// The one-launch path for small graphs: the block's own binning, the same in
// every block.  A first coalesced walk over indptr finds whether any row is
// split (more than long_min entries); only then are the split rows and
// their chunks listed, in row order (rounds of blockDim rows, offsets by
// block scans), into s_longs / s_chunks (counts in s_counts[0..1]).  The
// task table: the chunks, then every row of the graph, R = P rows a task
// with one slot each (a split row is skipped there).
__device__ void build_segments_small(const RowParams& p, int P, Seg* segs, int* nseg, int* total, int2* s_chunks,
                                     int2* s_longs, int* s_counts) {
    const int N = p.N, nt = blockDim.x, chunk = p.lists.chunk_edges;
    auto split = [&](int deg) { return deg > 0 && deg > p.long_min; };
    int any = 0;
    if (!p.small_no_split) {   // (the host knows no row can be split when nnz <= long_min)
        int i0 = 0;
        if ((reinterpret_cast<uintptr_t>(p.indptr) & 15u) == 0) {
            // four rows per 16-byte load (and the next group's first offset),
            // several loads in flight per thread
            const int n4 = N / 4;
            const int4* ip4 = reinterpret_cast<const int4*>(p.indptr);
#pragma unroll 4
            for (int k = threadIdx.x; k < n4; k += nt) {
                const int4 a = __ldg(ip4 + k);
                const int b = __ldg(p.indptr + 4 * k + 4);
                any |= split(a.y - a.x) | split(a.z - a.y) | split(a.w - a.z) | split(b - a.w);
            }
            i0 = 4 * n4;
        }
        for (int i = i0 + threadIdx.x; i < N; i += nt) any |= split(p.indptr[i + 1] - p.indptr[i]);
    }
    any = __syncthreads_or(any);
    int n_long = 0, n_chunks = 0;
    if (any) {
        for (int r0 = 0; r0 < N; r0 += nt) {
            const int i = r0 + threadIdx.x;
            const int beg = i < N ? p.indptr[i] : 0;
            const int deg = i < N ? p.indptr[i + 1] - beg : 0;
            const bool sp = split(deg);
            const int nch = sp ? (deg + chunk - 1) / chunk : 0;
            int tl, tc;
            const int2 ex = block_scan2(sp ? 1 : 0, nch, &tl, &tc);
            if (sp) {
                const int c0 = n_chunks + ex.y;
                s_longs[n_long + ex.x] = make_int2(i, c0);
                for (int c = 0; c < nch; ++c) s_chunks[c0 + c] = make_int2(i, beg + c * chunk);
            }
            n_long += tl;
            n_chunks += tc;
        }
    }
    if (threadIdx.x == 0) {
        s_counts[0] = n_long;
        s_counts[1] = n_chunks;
        int t = 0, k = 0;
        if (n_chunks > 0) { segs[k++] = Seg{t, 0, n_chunks, 1, P, kSegChunk}; t += n_chunks; }
        segs[k++] = Seg{t, 0, N, P, 1, kSegRows};
        t += (N + P - 1) / P;
        *nseg = k;
        *total = t;
    }
    __syncthreads();
}

// After the grid-wide sync of the one-launch path: a warp per split row
// merges its chunks' (m, s, acc) partials in chunk order into the output.
template <typename TO>
__device__ void small_combine(const RowParams& p, const int2* longs, int n_long) {
    const int lane = threadIdx.x & 31;
    const int nw = gridDim.x * (blockDim.x >> 5);
    const int H = p.H, D = p.D, HD = p.HD, chunk = p.lists.chunk_edges;
    TO* O = static_cast<TO*>(p.out);
    for (int li = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); li < n_long; li += nw) {
        const int row = longs[li].x, c0 = longs[li].y;
        const int nch = (p.indptr[row + 1] - p.indptr[row] + chunk - 1) / chunk;
        for (int el = lane; el < HD; el += 32) {
            const int h = p.ndh ? el % H : el / D;
            float M = -INFINITY;
            for (int c = 0; c < nch; ++c) M = fmaxf(M, p.part.m[static_cast<int64_t>(c0 + c) * H + h]);
            const float Mr = M == -INFINITY ? 0.f : M;   // no finite logit in the row: a zero row
            float S = 0.f, v = 0.f;
            for (int c = 0; c < nch; ++c) {
                const int64_t k = static_cast<int64_t>(c0 + c) * H + h;
                const float w = ex2(p.part.m[k] - Mr);
                S += p.part.s[k] * w;
                v += p.part.acc[static_cast<int64_t>(c0 + c) * HD + el] * w;
            }
            store_elem(O, static_cast<int64_t>(row) * p.ld + el, S > 0.f ? v / S : 0.f);
        }
    }
}

// ---------------------------------------------------------------------------
// 16-byte fragments
// ---------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> { static constexpr int kPerVec = 4; };
template <> struct Elem<__nv_bfloat16> { static constexpr int kPerVec = 8; };

template <typename T, int VPL>
struct Frag {
    static constexpr int E = VPL * Elem<T>::kPerVec;
    uint4 v[VPL];
    __device__ __forceinline__ void load(const T* p) {
        const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
        for (int k = 0; k < VPL; ++k) v[k] = __ldg(q + k);
    }
    __device__ __forceinline__ void load_once(const T* p) {   // read once per call (Q rows)
        const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            if constexpr (GT_STREAM_HINTS) v[k] = __ldcs(q + k);
            else v[k] = __ldg(q + k);
        }
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int k = 0; k < VPL; ++k) v[k] = make_uint4(0, 0, 0, 0);
    }
    __device__ __forceinline__ float get(int e) const {   // e compile-time after unrolling
        const uint32_t* w = reinterpret_cast<const uint32_t*>(v);
        if constexpr (sizeof(T) == 4) return __uint_as_float(w[e]);
        else return (e & 1) ? bf16hi(w[e >> 1]) : bf16lo(w[e >> 1]);
    }
};

// (a0, a1) *= c: one f32x2 multiply.
__device__ __forceinline__ void scale2(float& a0, float& a1, float c) {
    asm("{\n\t.reg .b64 rc, ra;\n\t"
        "mov.b64 rc, {%2, %2};\n\tmov.b64 ra, {%0, %1};\n\t"
        "mul.rn.f32x2 ra, ra, rc;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(c));
}

template <typename T, int E>
__device__ __forceinline__ void store_frag(T* p, const float* x) {
    if constexpr (sizeof(T) == 4) {
        float4* q = reinterpret_cast<float4*>(p);
#pragma unroll
        for (int k = 0; k < E / 4; ++k) {
            const float4 v = make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
            if constexpr (GT_STREAM_HINTS) __stcs(q + k, v);
            else q[k] = v;
        }
    } else {
        uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
        for (int k = 0; k < E / 8; ++k) {
            const uint4 v = make_uint4(pack_bf16x2(x[8 * k], x[8 * k + 1]), pack_bf16x2(x[8 * k + 2], x[8 * k + 3]),
                                       pack_bf16x2(x[8 * k + 4], x[8 * k + 5]), pack_bf16x2(x[8 * k + 6], x[8 * k + 7]));
            if constexpr (GT_STREAM_HINTS) __stcs(q + k, v);
            else q[k] = v;
        }
    }
}

// ---------------------------------------------------------------------------
// vector row kernel
// ---------------------------------------------------------------------------
// Tuning knobs (compile time): edges gathered per lane group per loop
// iteration is GT_ROWS_UNROLL / VPL; GT_ROWS_MIN_BLOCKS bounds registers so
// that many blocks of kRowThreads fit on an SM (the kernel is latency-bound:
// more resident warps hide more of the gathers' latency).
#ifndef GT_ROWS_UNROLL
#define GT_ROWS_UNROLL 2
#endif
#ifndef GT_ROWS_MIN_BLOCKS1
#define GT_ROWS_MIN_BLOCKS1 6   // one 16-byte vector per lane (85 registers)
#endif
#ifndef GT_ROWS_MIN_BLOCKS2
#define GT_ROWS_MIN_BLOCKS2 7   // two vectors per lane: 72 registers, 28 warps per SM
#endif
constexpr int kRowThreads = 128;

// Where a task's rows and edges are: one lane group's share of a task.
struct TaskMeta {
    int seg;        // segment of the task table
    int row, beg, end, chunk;
    bool valid;
};

// Blocks of kRowThreads per SM the register budget allows.  Two vectors
// per lane at 72 registers (28 warps) beat 79 registers without spills (24
// warps) by 2-3 % on R-MAT despite a few spilled bytes; fp32 lanes holding
// four vectors (16 values) get 4 blocks' worth so that their operands and
// next-iteration copies stay out of local memory.
template <typename T, int VPL>
constexpr int rows_min_blocks() {
    return VPL == 1 ? GT_ROWS_MIN_BLOCKS1 : VPL == 2 ? GT_ROWS_MIN_BLOCKS2 : 4;
}

// EXT (fused and SDDMM modes): kExtBias -- the logits get p.bias[e*H + h]
// added; kExtValues -- the dot products are multiplied by p.values[e] (the
// weighted adjacency's stored values).
constexpr int kExtBias = 1, kExtValues = 2;
template <typename T, typename TO, int VPL, int MODE, int EXT = 0, bool SMALL = false>
__global__ void __launch_bounds__(kRowThreads, rows_min_blocks<T, VPL>())
k_rows_vec(RowParams p) {
    static_assert(!SMALL || MODE == kFused, "the one-launch path is the fused forward");
    wait_prior_grid();
    constexpr bool BIAS = (EXT & kExtBias) != 0;
    constexpr bool VALS = (EXT & kExtValues) != 0;
    using F = Frag<T, VPL>;
    constexpr int E = F::E;
    constexpr int U = (GT_ROWS_UNROLL / VPL) > 0 ? (GT_ROWS_UNROLL / VPL) : 1;

    __shared__ Seg segs[kMaxSegs];
    __shared__ int s_nseg, s_total;
    __shared__ int s_small[2];            // one-launch path: split rows, chunks
    extern __shared__ int2 small_lists[];   // one-launch path: chunks, then split rows
    const int G = p.G;
    const int P = 32 / G;
    TaskLists L = p.lists;
    if constexpr (SMALL) {
        L.chunks = small_lists;
        L.longs = small_lists + p.small_max_chunks;
        build_segments_small(p, P, segs, &s_nseg, &s_total, small_lists, small_lists + p.small_max_chunks,
                             s_small);
    } else {
        // (rows of one entry are copied unless their statistics are wanted)
        build_segments(p.lists, P, U, segs, &s_nseg, &s_total, MODE == kFused && p.lse == nullptr);
    }

    const int lane = threadIdx.x & 31;
    const int grp = lane / G;
    const int gl = lane - grp * G;
    const int head = gl / p.lph;
    const T* __restrict__ Q = static_cast<const T*>(p.Q);
    const T* __restrict__ K = static_cast<const T*>(p.K);
    const T* __restrict__ V = static_cast<const T*>(p.V);
    TO* __restrict__ O = static_cast<TO*>(p.out);
    const int64_t HD = p.HD;
    const int64_t LD = p.ld;   // row stride of Q, K, V and out (elements; a 32-bit value)
    const int lane_off = gl * E;

    const int warps_total = gridDim.x * (blockDim.x >> 5);
    // task metadata (segment, row, edge range) of task t for this lane group
    auto load_meta = [&](int t, int seg_hint, TaskMeta& m) {
        int seg = seg_hint;
        while (seg + 1 < s_nseg && segs[seg + 1].first_task <= t) ++seg;
        const Seg& sg = segs[seg];
        const int r = grp / sg.S;
        const int pos = (t - sg.first_task) * sg.R + r;
        m.seg = seg;
        m.valid = pos < sg.count;
        m.row = 0;
        m.beg = 0;
        m.end = 0;
        m.chunk = -1;
        if (m.valid) {
            if (sg.kind == kSegChunk) {
                m.chunk = sg.list_begin + pos;
                const int2 c = L.chunks[m.chunk];
                m.row = c.x;
                m.beg = c.y;
                m.end = min(m.beg + L.chunk_edges, p.indptr[m.row + 1]);
            } else {
                if constexpr (SMALL) {
                    m.row = sg.list_begin + pos;   // every row, in index order
                    m.beg = p.indptr[m.row];
                    m.end = p.indptr[m.row + 1];
                    // a split row is walked by its chunks
                    if (m.end - m.beg > 0 && m.end - m.beg > p.long_min) m.valid = false;
                } else {
                    m.row = L.rows[sg.list_begin + pos];
                    m.beg = p.indptr[m.row];
                    m.end = p.indptr[m.row + 1];
                }
            }
        }
    };
    int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    TaskMeta cur, nxt;
    if (t < s_total) load_meta(t, 0, cur);
    for (; t < s_total; t += warps_total, cur = nxt) {
        // the next task's metadata loads are issued now and consumed on the
        // next iteration, off this task's critical path
        const int tn = t + warps_total;
        if (tn < s_total) load_meta(tn, cur.seg, nxt);
        const Seg sg = segs[cur.seg];
        if (MODE == kFused && sg.kind == kSegCopy) {   // uniform over the warp (one task)
            // a row of one entry: its softmax weight is 1, out = V[j]
            if (cur.valid) {
                const int j = ld_index(p.indices + cur.beg);
                F fv;
                fv.load(V + (int64_t)j * LD + lane_off);
                float x[E];
#pragma unroll
                for (int e = 0; e < E; ++e) x[e] = fv.get(e);
                if constexpr (BIAS) {
                    // the weight is 1 for a finite bias, 0 for -inf (the entry
                    // removed: a zero row), NaN for NaN or +inf
                    const float b = __ldg(p.bias + static_cast<int64_t>(cur.beg) * p.H + head);
                    const float wgt = b == -INFINITY ? 0.f : (b - b) + 1.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) x[e] *= wgt;
                }
                store_frag<TO, E>(O + (int64_t)cur.row * LD + lane_off, x);
            }
            continue;
        }
        const int S = sg.S;
        const int r = grp / S;
        const int sl = grp - r * S;
        const bool valid = cur.valid;
        const int row = cur.row, beg = cur.beg, end = cur.end, chunk = cur.chunk;
        const int step = S * U;
        int n_iter = (end - beg + step - 1) / step;
        n_iter = __reduce_max_sync(kFull, n_iter);

        constexpr bool kBf16 = sizeof(T) == 2;
        float q[E];          // fp32 inputs: q pre-scaled
        F fq;                // bf16 inputs: q kept packed, the scale multiplies the dot
        if constexpr (MODE != kSpmm) {
            if (valid) fq.load_once(Q + (int64_t)row * LD + lane_off); else fq.zero();
            if constexpr (!kBf16) {
                const float qs = MODE == kFused ? p.qscale : 1.f;   // SDDMM scales at the store
#pragma unroll
                for (int e = 0; e < E; ++e) q[e] = fq.get(e) * qs;
            }
        }
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        float m = -INFINITY, ssum = 0.f;

        // Two-stage software pipeline over the row's edges: the K/V rows of
        // iteration it+1 and the neighbour indices of iteration it+2 are in
        // flight while iteration it is computed.
        constexpr bool kNeedK = MODE != kSpmm;
        constexpr bool kNeedV = MODE != kSddmm;
        int jn[U];
        bool okc[U];
        F kc[U], vc[U];
        // bias (BIAS): like the indices it comes from DRAM (read once, in CSR
        // order), so it is fetched two iterations ahead: bc for iteration it,
        // bx for it+1
        float bc[U], bx[U];   // (the values (VALS) likewise: ac, ax)
        float ac[U], ax[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = beg + u * S + sl;
            okc[u] = e < end;
            if constexpr (BIAS) {
                bc[u] = okc[u] ? ld_stream(p.bias + static_cast<int64_t>(e) * p.H + head) : 0.f;
                bx[u] = e + step < end ? ld_stream(p.bias + static_cast<int64_t>(e + step) * p.H + head) : 0.f;
            }
            if constexpr (VALS) {
                ac[u] = okc[u] ? ld_stream(p.values + e) : 0.f;
                ax[u] = e + step < end ? ld_stream(p.values + e + step) : 0.f;
            }
            const int j = okc[u] ? ld_index(p.indices + e) : 0;
            if (kNeedK) { if (okc[u]) kc[u].load(K + (int64_t)j * LD + lane_off); else kc[u].zero(); }
            if (kNeedV) { if (okc[u]) vc[u].load(V + (int64_t)j * LD + lane_off); else vc[u].zero(); }
            const int e1 = e + step;
            jn[u] = e1 < end ? ld_index(p.indices + e1) : 0;
        }
        for (int it = 0; it < n_iter; ++it) {
            const int e0 = beg + it * step + sl;
            // issue iteration it+1's gathers and iteration it+2's indices
            bool okn[U];
            F kn[U], vn[U];
            float bn[U], an[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int e1 = e0 + step + u * S;
                okn[u] = e1 < end;
                if constexpr (BIAS) {
                    bn[u] = bx[u];
                    const int e2b = e1 + step;
                    bx[u] = e2b < end ? ld_stream(p.bias + static_cast<int64_t>(e2b) * p.H + head) : 0.f;
                }
                if constexpr (VALS) {
                    an[u] = ax[u];
                    const int e2a = e1 + step;
                    ax[u] = e2a < end ? ld_stream(p.values + e2a) : 0.f;
                }
                if (kNeedK) { if (okn[u]) kn[u].load(K + (int64_t)jn[u] * LD + lane_off); else kn[u].zero(); }
                if (kNeedV) { if (okn[u]) vn[u].load(V + (int64_t)jn[u] * LD + lane_off); else vn[u].zero(); }
                const int e2 = e1 + step;
                jn[u] = e2 < end ? ld_index(p.indices + e2) : 0;
            }
            float l[U];
            if constexpr (kNeedK) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if constexpr (kBf16) {
                        const uint32_t* qw = reinterpret_cast<const uint32_t*>(fq.v);
                        const uint32_t* kw = reinterpret_cast<const uint32_t*>(kc[u].v);
                        float d0 = 0.f, d1 = 0.f;
#pragma unroll
                        for (int w = 0; w < E / 2; w += 2) {
                            d0 = dot2_bf16(qw[w], kw[w], d0);
                            d1 = dot2_bf16(qw[w + 1], kw[w + 1], d1);
                        }
                        l[u] = (d0 + d1) * (MODE == kFused ? p.qscale : 1.f);
                    } else {
                        float d0 = 0.f, d1 = 0.f;
#pragma unroll
                        for (int e = 0; e < E; e += 2) fma2(d0, d1, q[e], q[e + 1], kc[u].get(e), kc[u].get(e + 1));
                        l[u] = d0 + d1;
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
                    for (int o = 1; o < p.lph; o <<= 1) l[u] += __shfl_xor_sync(kFull, l[u], o);
                if constexpr (VALS) {   // weighted adjacency: (q.k) * a_e (scaled or not alike)
#pragma unroll
                    for (int u = 0; u < U; ++u) l[u] *= ac[u];
                }
                if constexpr (BIAS && MODE == kFused) {
#pragma unroll
                    for (int u = 0; u < U; ++u) l[u] = fmaf(bc[u], kLog2e, l[u]);   // logits in log2 units
                }
            }
            if constexpr (MODE == kSddmm) {
                if (gl % p.lph == 0) {
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (okc[u]) p.logits[(int64_t)(e0 + u * S) * p.H + head] = BIAS ? fmaf(l[u], p.qscale, bc[u]) : l[u] * p.qscale;
                }
            } else if constexpr (MODE == kFused) {
                // The running maximum m is raised only when a score exceeds it
                // by more than kLazyMax (log2 units; the weights stay <= 2^kLazyMax),
                // and the rescale of the sum and accumulators is skipped when no
                // lane of the warp raises it -- after a row's first entries,
                // almost always.
                float mx = -INFINITY;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (!okc[u]) l[u] = -INFINITY;
                    mx = fmaxf(mx, l[u]);
                }
                const bool raise = mx > m + kLazyMax;   // false for mx = -inf
                if (__any_sync(kFull, raise)) {
                    const float c = raise ? ex2(m - mx) : 1.f;   // m = -inf: c = 0 (nothing accumulated)
                    if (raise) m = mx;
                    ssum *= c;
#pragma unroll
                    for (int e = 0; e < E; e += 2) scale2(acc[e], acc[e + 1], c);
                }
                const float mref = (m == -INFINITY) ? 0.f : m;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float w = ex2(l[u] - mref);
                    ssum += w;
                    if constexpr (kBf16) {
                        const uint32_t* vw = reinterpret_cast<const uint32_t*>(vc[u].v);
#pragma unroll
                        for (int e = 0; e < E; e += 2) axpy2_bf16(acc[e], acc[e + 1], w, vw[e >> 1]);
                    } else {
#pragma unroll
                        for (int e = 0; e < E; e += 2) fma2(acc[e], acc[e + 1], w, w, vc[u].get(e), vc[u].get(e + 1));
                    }
                }
            } else {   // kSpmm: weights are the given probabilities
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float w = okc[u] ? p.probs[(int64_t)(e0 + u * S) * p.H + head] : 0.f;
                    if constexpr (kBf16) {
                        const uint32_t* vw = reinterpret_cast<const uint32_t*>(vc[u].v);
#pragma unroll
                        for (int e = 0; e < E; e += 2) axpy2_bf16(acc[e], acc[e + 1], w, vw[e >> 1]);
                    } else {
#pragma unroll
                        for (int e = 0; e < E; e += 2) fma2(acc[e], acc[e + 1], w, w, vc[u].get(e), vc[u].get(e + 1));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                okc[u] = okn[u];
                kc[u] = kn[u];
                vc[u] = vn[u];
                if constexpr (BIAS) bc[u] = bn[u];
                if constexpr (VALS) ac[u] = an[u];
            }
        }
        if constexpr (MODE != kSddmm) {
        // merge the S edge slots of each row (lanes G, 2G, ... apart)
        for (int o = G; o < S * G; o <<= 1) {
            if constexpr (MODE == kFused) {
                const float m2 = __shfl_xor_sync(kFull, m, o);
                const float s2 = __shfl_xor_sync(kFull, ssum, o);
                const float M = fmaxf(m, m2);
                const float Mref = (M == -INFINITY) ? 0.f : M;
                const float c1 = ex2(m - Mref), c2 = ex2(m2 - Mref);
                ssum = ssum * c1 + s2 * c2;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float a2 = __shfl_xor_sync(kFull, acc[e], o);
                    acc[e] = acc[e] * c1 + a2 * c2;
                }
                m = M;
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] += __shfl_xor_sync(kFull, acc[e], o);
            }
        }
        if (!valid || sl != 0) continue;
        if (chunk >= 0) {
            float* pa = p.part.acc + (int64_t)chunk * HD + lane_off;
#pragma unroll
            for (int k = 0; k < E / 4; ++k)
                reinterpret_cast<float4*>(pa)[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
            if (MODE == kFused && gl % p.lph == 0) {
                p.part.m[(int64_t)chunk * p.H + head] = m;
                p.part.s[(int64_t)chunk * p.H + head] = ssum;
            }
        } else {
            if constexpr (MODE == kFused) {
                const float inv = ssum > 0.f ? 1.f / ssum : 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = ssum > 0.f ? acc[e] * inv : 0.f;
                // the row's log-sum-exp (log2 units) when the caller asks for it
                if (p.lse && gl % p.lph == 0) p.lse[(int64_t)row * p.H + head] = m + log2f(ssum);
            }
            store_frag<TO, E>(O + (int64_t)row * LD + lane_off, acc);
        }
        }   // MODE != kSddmm
    }
    if constexpr (SMALL) {
        if (s_small[0] > 0) {   // uniform over the grid
            // split rows: every chunk's partial is written once the whole
            // (cooperatively launched) grid arrives here
            cooperative_groups::this_grid().sync();
            small_combine<TO>(p, L.longs, s_small[0]);
        }
    }
}

// ---------------------------------------------------------------------------
// generic row kernel: any H, D with H*D <= 1024 and H <= 256.  One warp per
// task; lane holds elements t = lane + 32k of the feature row; per-head dot
// products are summed from shared memory by one lane per head.
// ---------------------------------------------------------------------------
constexpr int kGenWarps = 4;
constexpr int kGenMaxH = 256;

// KPL: elements of the feature row per lane (ceil(H*D/32) rounded up to 4,
// 8 or 32), so small rows keep few registers per lane.
template <typename T, typename TO, int MODE, int KPL, bool SMALL = false>
__global__ void __launch_bounds__(kGenWarps * 32)
k_rows_generic(RowParams p) {
    static_assert(!SMALL || MODE == kFused, "the one-launch path is the fused forward");
    wait_prior_grid();
    __shared__ Seg segs[kMaxSegs];
    __shared__ int s_nseg, s_total;
    __shared__ float sm_prod[kGenWarps][KPL * 32];
    __shared__ float sm_m[kGenWarps][kGenMaxH];
    __shared__ float sm_s[kGenWarps][kGenMaxH];
    __shared__ float sm_w[kGenWarps][kGenMaxH];
    __shared__ float sm_c[kGenWarps][kGenMaxH];
    __shared__ int s_small[2];              // one-launch path: split rows, chunks
    extern __shared__ int2 small_lists[];   // one-launch path: chunks, then split rows
    TaskLists L = p.lists;
    if constexpr (SMALL) {
        L.chunks = small_lists;
        L.longs = small_lists + p.small_max_chunks;
        build_segments_small(p, 1, segs, &s_nseg, &s_total, small_lists, small_lists + p.small_max_chunks, s_small);
    } else {
        build_segments(p.lists, 1, 1, segs, &s_nseg, &s_total);
    }

    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const T* __restrict__ Q = static_cast<const T*>(p.Q);
    const T* __restrict__ K = static_cast<const T*>(p.K);
    const T* __restrict__ V = static_cast<const T*>(p.V);
    TO* __restrict__ O = static_cast<TO*>(p.out);
    const int H = p.H, D = p.D, HD = p.HD;
    float* prod = sm_prod[wid];
    float* hm = sm_m[wid];
    float* hs = sm_s[wid];
    float* hw = sm_w[wid];
    float* hc = sm_c[wid];

    const int warps_total = gridDim.x * kGenWarps;
    int seg = 0;
    for (int t = blockIdx.x * kGenWarps + wid; t < s_total; t += warps_total) {
        while (seg + 1 < s_nseg && segs[seg + 1].first_task <= t) ++seg;
        const Seg sg = segs[seg];
        const int pos = t - sg.first_task;
        int row, beg, end, chunk = -1;
        if (sg.kind == kSegChunk) {
            chunk = sg.list_begin + pos;
            int2 c = L.chunks[chunk];
            row = c.x;
            beg = c.y;
            end = min(beg + L.chunk_edges, p.indptr[row + 1]);
        } else {
            row = SMALL ? sg.list_begin + pos : L.rows[sg.list_begin + pos];
            beg = p.indptr[row];
            end = p.indptr[row + 1];
            // one-launch path: a split row is walked by its chunks (uniform over the warp)
            if (SMALL && end - beg > 0 && end - beg > p.long_min) continue;
        }
        float q[KPL], acc[KPL];
        const float qs = MODE == kFused ? p.qscale : 1.f;   // SDDMM scales at the store
#pragma unroll
        for (int k = 0; k < KPL; ++k) {
            const int el = lane + 32 * k;
            q[k] = (MODE != kSpmm && el < HD) ? load_elem(Q, (int64_t)row * HD + el) * qs : 0.f;
            acc[k] = 0.f;
        }
        for (int h = lane; h < H; h += 32) { hm[h] = -INFINITY; hs[h] = 0.f; }
        __syncwarp();
        // Rows of few features a lane (KPL <= 8) keep the next entry's K and V
        // values and the index after it in flight while this entry is
        // computed; wider rows load per entry (their registers go to the row).
        constexpr bool kPipe = KPL <= 8;
        constexpr int KP = kPipe ? KPL : 1;
        float kn[KP], vn[KP];
        int64_t jn = 0, jn2 = 0;
        auto fetch = [&](int64_t jj) {
#pragma unroll
            for (int k = 0; k < KP; ++k) {
                const int el = lane + 32 * k;
                kn[k] = (MODE != kSpmm && el < HD) ? load_elem(K, jj * HD + el) : 0.f;
                vn[k] = (MODE != kSddmm && el < HD) ? load_elem(V, jj * HD + el) : 0.f;
            }
        };
        if constexpr (kPipe) {
            if (beg < end) {
                jn = __ldg(p.indices + beg);
                fetch(jn);
            }
            jn2 = beg + 1 < end ? __ldg(p.indices + beg + 1) : 0;
        }
        for (int e = beg; e < end; ++e) {
            int64_t j;
            float kc[KP], vc[KP];
            if constexpr (kPipe) {
                j = jn;
#pragma unroll
                for (int k = 0; k < KP; ++k) { kc[k] = kn[k]; vc[k] = vn[k]; }
                if (e + 1 < end) {   // the next entry's values, the index after it
                    jn = jn2;
                    fetch(jn);
                    jn2 = e + 2 < end ? __ldg(p.indices + e + 2) : 0;
                }
            } else {
                j = __ldg(p.indices + e);
            }
            if constexpr (MODE != kSpmm) {
#pragma unroll
                for (int k = 0; k < KPL; ++k) {
                    const int el = lane + 32 * k;
                    if (el < HD) prod[el] = q[k] * (kPipe ? kc[k < KP ? k : 0] : load_elem(K, j * HD + el));
                }
                __syncwarp();
            }
            for (int h = lane; h < H; h += 32) {
                float l = 0.f;
                if constexpr (MODE != kSpmm) {
                    // eight interleaved partial sums, combined pairwise (error
                    // grows with D/8 instead of D)
                    // head h's D products: contiguous ([N, H, D]) or H apart ([N, D, H])
                    const int st = p.ndh ? H : 1;
                    const float* pr = prod + (p.ndh ? h : h * D);
                    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    int d = 0;
                    for (; d + 8 <= D; d += 8) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) a[k] += pr[(d + k) * st];
                    }
                    for (; d < D; ++d) a[0] += pr[d * st];
                    l = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
                    if (p.values) l *= p.values[e];   // weighted adjacency
                }
                if constexpr (MODE == kSddmm) {
                    p.logits[(int64_t)e * H + h] = p.bias ? fmaf(l, p.qscale, p.bias[(int64_t)e * H + h])
                                                          : l * p.qscale;
                } else if constexpr (MODE == kFused) {
                    if (p.bias) l = fmaf(p.bias[(int64_t)e * H + h], kLog2e, l);   // log2 units
                    const float mo = hm[h];
                    const float mn = fmaxf(mo, l);
                    const float mref = mn == -INFINITY ? 0.f : mn;   // no finite logit yet
                    const float c = ex2(mo - mref);
                    const float w = ex2(l - mref);
                    hs[h] = hs[h] * c + w;
                    hm[h] = mn;
                    hc[h] = c;
                    hw[h] = w;
                } else {
                    hc[h] = 1.f;
                    hw[h] = p.probs[(int64_t)e * H + h];
                }
            }
            __syncwarp();
            if constexpr (MODE != kSddmm) {
#pragma unroll
                for (int k = 0; k < KPL; ++k) {
                    const int el = lane + 32 * k;
                    if (el < HD) {
                        const int h = head_of(el, D, H, p.ndh);
                        acc[k] = acc[k] * hc[h] + hw[h] * (kPipe ? vc[k < KP ? k : 0] : load_elem(V, j * HD + el));
                    }
                }
            }
            __syncwarp();
        }
        if constexpr (MODE == kSddmm) continue;
        if (chunk >= 0) {
#pragma unroll
            for (int k = 0; k < KPL; ++k) {
                const int el = lane + 32 * k;
                if (el < HD) p.part.acc[(int64_t)chunk * HD + el] = acc[k];
            }
            if (MODE == kFused)
                for (int h = lane; h < H; h += 32) {
                    p.part.m[(int64_t)chunk * H + h] = hm[h];
                    p.part.s[(int64_t)chunk * H + h] = hs[h];
                }
        } else {
#pragma unroll
            for (int k = 0; k < KPL; ++k) {
                const int el = lane + 32 * k;
                if (el < HD) {
                    float v = acc[k];
                    if (MODE == kFused) {
                        const float s = hs[head_of(el, D, H, p.ndh)];
                        v = s > 0.f ? v / s : 0.f;
                    }
                    store_elem(O, (int64_t)row * HD + el, v);
                }
            }
            if (MODE == kFused && p.lse)   // the row's log-sum-exp (log2 units)
                for (int h = lane; h < H; h += 32) p.lse[(int64_t)row * H + h] = hm[h] + log2f(hs[h]);
        }
        __syncwarp();
    }
    if constexpr (SMALL) {
        if (s_small[0] > 0) {   // uniform over the grid
            cooperative_groups::this_grid().sync();
            small_combine<TO>(p, L.longs, s_small[0]);
        }
    }
}

// ---------------------------------------------------------------------------
// narrow-head kernel: heads of at most kNarrowMaxD features, fused mode,
// [N, H, D] rows, with the per-entry bias or values of the other kernels
// when given (the molecule configuration of "Graph
// Transformer in a Nutshell": hidden 80 over 8 heads, head width 10, which
// no 16-byte lane split fits).  One lane per head: a row is G lanes (H
// rounded up to a power of two), each holding its head's q, running maximum,
// sum and accumulators, so the dot product and the softmax update are one
// lane's work with no shuffle or shared memory; P = 32 / G rows per warp,
// and rows of many entries get S lane groups (slots) merged at the end.
// PAIR: D even, so a head's features are read two at a time (8-byte fp32,
// 4-byte bf16 loads).
// ---------------------------------------------------------------------------
template <typename T, bool PAIR>
__device__ __forceinline__ void load_head(const T* __restrict__ p, int D, float (&x)[kNarrowMaxD]) {
    if constexpr (PAIR) {
#pragma unroll
        for (int d = 0; d < kNarrowMaxD; d += 2) {
            if (d < D) {
                if constexpr (sizeof(T) == 4) {
                    const float2 v = __ldg(reinterpret_cast<const float2*>(p + d));
                    x[d] = v.x;
                    x[d + 1] = v.y;
                } else {
                    const uint32_t w = __ldg(reinterpret_cast<const unsigned*>(p + d));
                    x[d] = bf16lo(w);
                    x[d + 1] = bf16hi(w);
                }
            } else {
                x[d] = 0.f;
                x[d + 1] = 0.f;
            }
        }
    } else {
#pragma unroll
        for (int d = 0; d < kNarrowMaxD; ++d) x[d] = d < D ? load_elem(p, d) : 0.f;
    }
}

template <typename T, typename TO, bool PAIR, bool SMALL = false>
__global__ void __launch_bounds__(kRowThreads)
k_rows_narrow(RowParams p) {
    wait_prior_grid();
    __shared__ Seg segs[kMaxSegs];
    __shared__ int s_nseg, s_total;
    __shared__ int s_small[2];              // one-launch path: split rows, chunks
    extern __shared__ int2 small_lists[];   // one-launch path: chunks, then split rows
    const int G = p.G;
    const int P = 32 / G;
    TaskLists L = p.lists;
    if constexpr (SMALL) {
        L.chunks = small_lists;
        L.longs = small_lists + p.small_max_chunks;
        build_segments_small(p, P, segs, &s_nseg, &s_total, small_lists, small_lists + p.small_max_chunks, s_small);
    } else {
        // (rows of one entry are copied unless their statistics are wanted)
        build_segments(p.lists, P, 1, segs, &s_nseg, &s_total, p.lse == nullptr);
    }
    const int lane = threadIdx.x & 31;
    const int grp = lane / G;
    const int h = lane - grp * G;           // this lane's head
    const bool on = h < p.H;                // lanes past H (H not a power of two) idle
    const int D = p.D, H = p.H;
    const int64_t HD = p.HD;
    const int off = h * D;
    const T* __restrict__ Q = static_cast<const T*>(p.Q);
    const T* __restrict__ K = static_cast<const T*>(p.K);
    const T* __restrict__ V = static_cast<const T*>(p.V);
    TO* __restrict__ O = static_cast<TO*>(p.out);

    const int warps_total = gridDim.x * (blockDim.x >> 5);
    int seg = 0;
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < s_total; t += warps_total) {
        while (seg + 1 < s_nseg && segs[seg + 1].first_task <= t) ++seg;
        const Seg sg = segs[seg];
        const int S = sg.S;
        const int r = grp / S, sl = grp - r * S;
        const int pos = (t - sg.first_task) * sg.R + r;
        bool valid = pos < sg.count;
        int row = 0, beg = 0, end = 0, chunk = -1;
        if (valid) {
            if (sg.kind == kSegChunk) {
                chunk = sg.list_begin + pos;
                const int2 c = L.chunks[chunk];
                row = c.x;
                beg = c.y;
                end = min(beg + L.chunk_edges, p.indptr[row + 1]);
            } else {
                row = SMALL ? sg.list_begin + pos : L.rows[sg.list_begin + pos];
                beg = p.indptr[row];
                end = p.indptr[row + 1];
                // one-launch path: a split row is walked by its chunks
                if (SMALL && end - beg > 0 && end - beg > p.long_min) valid = false;
            }
        }
        if (sg.kind == kSegCopy) {   // a row of one entry: its softmax weight is 1, out = V[j]
            if (valid && on) {
                float x[kNarrowMaxD];
                load_head<T, PAIR>(V + static_cast<int64_t>(ld_index(p.indices + beg)) * HD + off, D, x);
                // with a bias: weight 1 for a finite bias, 0 for -inf (the
                // entry removed), NaN for NaN or +inf
                float wgt = 1.f;
                if (p.bias) {
                    const float b = __ldg(p.bias + static_cast<int64_t>(beg) * H + h);
                    wgt = b == -INFINITY ? 0.f : (b - b) + 1.f;
                }
#pragma unroll
                for (int d = 0; d < kNarrowMaxD; ++d)
                    if (d < D) store_elem(O, static_cast<int64_t>(row) * HD + off + d, x[d] * wgt);
            }
            continue;
        }
        const bool live = valid && on;
        float q[kNarrowMaxD], acc[kNarrowMaxD];
        if (live) load_head<T, PAIR>(Q + static_cast<int64_t>(row) * HD + off, D, q);
#pragma unroll
        for (int d = 0; d < kNarrowMaxD; ++d) {
            q[d] = live ? q[d] * p.qscale : 0.f;   // logits in log2 units
            acc[d] = 0.f;
        }
        float m = -INFINITY, ssum = 0.f;
        // Two-stage pipeline: the next entry's K and V values and the index
        // after it are in flight while this entry is computed.
        int e = beg + sl;
        float kc[kNarrowMaxD], vc[kNarrowMaxD];
        if (live && e < end) {
            const int64_t j = ld_index(p.indices + e);
            load_head<T, PAIR>(K + j * HD + off, D, kc);
            load_head<T, PAIR>(V + j * HD + off, D, vc);
        }
        int jn = (live && e + S < end) ? ld_index(p.indices + e + S) : 0;
        for (; live && e < end; e += S) {
            const int e1 = e + S;
            float kn[kNarrowMaxD], vn[kNarrowMaxD];
            if (e1 < end) {
                load_head<T, PAIR>(K + static_cast<int64_t>(jn) * HD + off, D, kn);
                load_head<T, PAIR>(V + static_cast<int64_t>(jn) * HD + off, D, vn);
                jn = e1 + S < end ? ld_index(p.indices + e1 + S) : 0;
            }
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int d = 0; d < kNarrowMaxD; d += 2) {
                d0 = fmaf(q[d], kc[d], d0);
                d1 = fmaf(q[d + 1], kc[d + 1], d1);
            }
            float l = d0 + d1;
            if (p.values) l *= ld_stream(p.values + e);   // weighted adjacency
            if (p.bias) l = fmaf(ld_stream(p.bias + static_cast<int64_t>(e) * H + h), kLog2e, l);   // log2 units
            if (l > m) {   // a new maximum: rescale what is accumulated (m = -inf: c = 0)
                const float c = ex2(m - l);
                ssum *= c;
#pragma unroll
                for (int d = 0; d < kNarrowMaxD; ++d) acc[d] *= c;
                m = l;
            }
            const float w = ex2(l - (m == -INFINITY ? 0.f : m));   // (all logits -inf so far: w = 0)
            ssum += w;
#pragma unroll
            for (int d = 0; d < kNarrowMaxD; ++d) acc[d] = fmaf(w, vc[d], acc[d]);
#pragma unroll
            for (int d = 0; d < kNarrowMaxD; ++d) {
                kc[d] = kn[d];
                vc[d] = vn[d];
            }
        }
        // merge the S slots of each row (lane groups G, 2G, ... apart)
        for (int o = G; o < S * G; o <<= 1) {
            const float m2 = __shfl_xor_sync(kFull, m, o);
            const float s2 = __shfl_xor_sync(kFull, ssum, o);
            const float M = fmaxf(m, m2);
            const float Mref = M == -INFINITY ? 0.f : M;
            const float c1 = ex2(m - Mref), c2 = ex2(m2 - Mref);
            ssum = ssum * c1 + s2 * c2;
#pragma unroll
            for (int d = 0; d < kNarrowMaxD; ++d) {
                const float a2 = __shfl_xor_sync(kFull, acc[d], o);
                acc[d] = acc[d] * c1 + a2 * c2;
            }
            m = M;
        }
        if (!live || sl != 0) continue;
        if (chunk >= 0) {
            float* pa = p.part.acc + static_cast<int64_t>(chunk) * HD + off;
#pragma unroll
            for (int d = 0; d < kNarrowMaxD; ++d)
                if (d < D) pa[d] = acc[d];
            p.part.m[static_cast<int64_t>(chunk) * H + h] = m;
            p.part.s[static_cast<int64_t>(chunk) * H + h] = ssum;
        } else {
            const float inv = ssum > 0.f ? 1.f / ssum : 0.f;
#pragma unroll
            for (int d = 0; d < kNarrowMaxD; ++d)
                if (d < D) store_elem(O, static_cast<int64_t>(row) * HD + off + d, ssum > 0.f ? acc[d] * inv : 0.f);
            // the row's log-sum-exp (log2 units) when the caller asks for it
            if (p.lse) p.lse[static_cast<int64_t>(row) * H + h] = m + log2f(ssum);
        }
    }
    if constexpr (SMALL) {
        if (s_small[0] > 0) {   // uniform over the grid
            cooperative_groups::this_grid().sync();
            small_combine<TO>(p, L.longs, s_small[0]);
        }
    }
}

// ---------------------------------------------------------------------------
// combine split-row partials
// ---------------------------------------------------------------------------
// Phase 1, a block per split row of many chunks: the row's chunks are spread
// over groups of threads (a group per head for the statistics, per output
// element for the sums) whose partials meet in shared memory, so a hub row
// of hundreds of chunks costs a few chunk loads per thread.  Phase 2, a warp
// per split row of at most kBigChunks chunks (when H divides 32; else phase 1
// takes every split row).  Binning lists the rows of more chunks first, so
// phase 1 walks only those.
constexpr int kCombThreads = 512;

template <typename TO, int MODE>
__global__ void __launch_bounds__(kCombThreads)
k_combine(RowParams p, int warp_rows) {
    wait_prior_grid();
    __shared__ float sM[kGenMaxH];
    __shared__ float sS[kGenMaxH];
    __shared__ float red[kCombThreads];
    const int n_long = p.lists.hdr[HdrLayout::kLong];
    const int n_big = warp_rows ? p.lists.hdr[HdrLayout::kBig] : n_long;   // phase 1 rows: [0, n_big)
    const int H = p.H, D = p.D, HD = p.HD;
    const int t = threadIdx.x;
    // head groups run one after another had their partials in blocks of
    // their own: each group's rows, its partials and its output columns
    const int groups = p.groups > 0 ? p.groups : 1;
    for (int gi = 0; gi < groups; ++gi) {
    Partials part = p.part;
    part.m += gi * p.gstep_m;
    part.s += gi * p.gstep_m;
    part.acc += gi * p.gstep_acc;
    TO* __restrict__ O = static_cast<TO*>(p.out) + static_cast<int64_t>(gi) * p.gstep_out;
    for (int li = blockIdx.x; li < n_big; li += gridDim.x) {
        const int2 lr = p.lists.longs[li];
        const int row = lr.x, c0 = lr.y;
        const int deg = p.indptr[row + 1] - p.indptr[row];
        const int nch = (deg + p.lists.chunk_edges - 1) / p.lists.chunk_edges;
        if (MODE == kFused) {
            // per head: M = max_c m_c, S = sum_c s_c 2^(m_c - M)
            const int G = kCombThreads / H;   // H <= 256: at least two groups
            const int h = t % H, g = t / H;
            float m = -INFINITY;
            if (g < G)
                for (int c = g; c < nch; c += G) m = fmaxf(m, part.m[(int64_t)(c0 + c) * H + h]);
            red[t] = m;
            __syncthreads();
            if (t < H) {
                float M = -INFINITY;
                for (int k = 0; k < G; ++k) M = fmaxf(M, red[k * H + t]);
                sM[t] = M == -INFINITY ? 0.f : M;   // no finite logit in the row: a zero row
            }
            __syncthreads();
            float sum = 0.f;
            if (g < G) {
                const float M = sM[h];
                for (int c = g; c < nch; c += G) {
                    const int64_t k = (int64_t)(c0 + c) * H + h;
                    sum += part.s[k] * ex2(part.m[k] - M);
                }
            }
            __syncthreads();   // everyone has read red[] for M
            red[t] = sum;
            __syncthreads();
            if (t < H) {
                float S = 0.f;
                for (int k = 0; k < G; ++k) S += red[k * H + t];
                sS[t] = S;
                if (p.lse) p.lse[(int64_t)row * H + t] = sM[t] + log2f(S);   // log-sum-exp, log2 units
            }
            __syncthreads();
        }
        const int Ge = kCombThreads / HD;   // element groups over the chunks
        if (Ge >= 2) {
            const int el = t % HD, g = t / HD;
            const int h = head_of(el, D, H, p.ndh);
            float v = 0.f;
            if (g < Ge) {
                const float M = MODE == kFused ? sM[h] : 0.f;
                // four independent partial sums keep four chunks' loads in flight
                float v4[4] = {0.f, 0.f, 0.f, 0.f};
                int c = g;
                for (; c + 3 * Ge < nch; c += 4 * Ge) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int cu = c + u * Ge;
                        const float a = part.acc[(int64_t)(c0 + cu) * HD + el];
                        v4[u] += MODE == kFused ? a * ex2(part.m[(int64_t)(c0 + cu) * H + h] - M) : a;
                    }
                }
                for (; c < nch; c += Ge) {
                    const float a = part.acc[(int64_t)(c0 + c) * HD + el];
                    v4[0] += MODE == kFused ? a * ex2(part.m[(int64_t)(c0 + c) * H + h] - M) : a;
                }
                v = (v4[0] + v4[1]) + (v4[2] + v4[3]);
            }
            red[t] = v;
            __syncthreads();
            if (t < HD) {
                float tot = 0.f;
                for (int k = 0; k < Ge; ++k) tot += red[k * HD + t];
                if (MODE == kFused) tot = sS[h] > 0.f ? tot / sS[h] : 0.f;
                store_elem(O, (int64_t)row * p.ld + t, tot);
            }
        } else {
            for (int el = t; el < HD; el += kCombThreads) {
                const int h = head_of(el, D, H, p.ndh);
                const float M = MODE == kFused ? sM[h] : 0.f;
                float v = 0.f;
#pragma unroll 4
                for (int c = 0; c < nch; ++c) {
                    const float a = part.acc[(int64_t)(c0 + c) * HD + el];
                    v += MODE == kFused ? a * ex2(part.m[(int64_t)(c0 + c) * H + h] - M) : a;
                }
                if (MODE == kFused) v = sS[h] > 0.f ? v / sS[h] : 0.f;
                store_elem(O, (int64_t)row * p.ld + el, v);
            }
        }
        __syncthreads();
    }
    // phase 2: rows of at most kBigChunks chunks (most of them), a warp
    // per row: lanes over (chunk, head) pairs for the statistics (H divides
    // 32), over output elements for the sums
    if (warp_rows) {
        const int lane = t & 31;
        const int warps = gridDim.x * (blockDim.x >> 5);
        for (int li = n_big + blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); li < n_long; li += warps) {
            const int2 lr = p.lists.longs[li];
            const int row = lr.x, c0 = lr.y;
            const int deg = p.indptr[row + 1] - p.indptr[row];
            const int nch = (deg + p.lists.chunk_edges - 1) / p.lists.chunk_edges;   // <= kBigChunks
            // lane l: head l % H, chunks l / H, l / H + 32 / H, ...; lanes H
            // apart combine, so lane h < H ends with head h's (M, S)
            float M = -INFINITY, S = 0.f;
            if (MODE == kFused) {
                const int h = lane % H, step = 32 / H;
                for (int c = lane / H; c < nch; c += step) M = fmaxf(M, part.m[(int64_t)(c0 + c) * H + h]);
                for (int o = H; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
                if (M == -INFINITY) M = 0.f;   // no finite logit in the row: a zero row
                for (int c = lane / H; c < nch; c += step) {
                    const int64_t k = (int64_t)(c0 + c) * H + h;
                    S += part.s[k] * ex2(part.m[k] - M);
                }
                for (int o = H; o < 32; o <<= 1) S += __shfl_xor_sync(kFull, S, o);
                if (p.lse && lane < H) p.lse[(int64_t)row * H + lane] = M + log2f(S);   // log-sum-exp, log2 units
            }
            for (int el0 = 0; el0 < HD; el0 += 32) {
                const int el = el0 + lane;
                const int h = head_of(min(el, HD - 1), D, H, p.ndh);
                const float Mh = __shfl_sync(kFull, M, h);
                const float Sh = __shfl_sync(kFull, S, h);
                if (el < HD) {
                    // four independent partial sums keep four chunks' loads in flight
                    float v4[4] = {0.f, 0.f, 0.f, 0.f};
                    int c = 0;
                    for (; c + 3 < nch; c += 4) {
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float a = part.acc[(int64_t)(c0 + c + u) * HD + el];
                            v4[u] += MODE == kFused ? a * ex2(part.m[(int64_t)(c0 + c + u) * H + h] - Mh) : a;
                        }
                    }
                    for (; c < nch; ++c) {
                        const float a = part.acc[(int64_t)(c0 + c) * HD + el];
                        v4[0] += MODE == kFused ? a * ex2(part.m[(int64_t)(c0 + c) * H + h] - Mh) : a;
                    }
                    float v = (v4[0] + v4[1]) + (v4[2] + v4[3]);
                    if (MODE == kFused) v = Sh > 0.f ? v / Sh : 0.f;
                    store_elem(O, (int64_t)row * p.ld + el, v);
                }
            }
        }
    }
    }   // head groups
}

// (rows of few chunks: phase 2 of k_combine)
// row: lanes over (chunk, head) pairs for the statistics, over output
// elements for the sums.  Needs H to divide 32; larger rows and other head
// counts go to k_combine.

// ---------------------------------------------------------------------------
// unfused edge softmax
// ---------------------------------------------------------------------------
// p[e,h] = exp(l[e,h] - M_h) / S_h over each row's entries, with accurate
// expf, in three walks per element: the maximum, the sum, the write.
//
// Ordinary rows (the bucketed row list, rows of equal degree side by side):
// a thread per (row, head), so neighbouring threads have the same amount of
// work; the H threads of a row read its logits together (entry-major,
// head-minor), and the second and third walks hit in L1.
__global__ void __launch_bounds__(256)
k_softmax_short(const int* __restrict__ indptr, const int* __restrict__ hdr, const int* __restrict__ rows,
                int H, const float* __restrict__ logits, float* __restrict__ probs) {
    int n_rows = 0;   // length of the bucketed list (the buckets are contiguous)
    for (int b = 0; b < kNumBuckets; ++b)
        n_rows = max(n_rows, hdr[HdrLayout::kOffset + b] + hdr[HdrLayout::kCount + b]);
    const int64_t total = (int64_t)n_rows * H;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int pos = (int)(t / H), h = (int)(t - (int64_t)pos * H);
        const int row = rows[pos];
        const int beg = indptr[row], deg = indptr[row + 1] - beg;
        const float* lr = logits + (int64_t)beg * H + h;
        float* pr = probs + (int64_t)beg * H + h;
        float m = -INFINITY;
        for (int e = 0; e < deg; ++e) m = fmaxf(m, lr[(int64_t)e * H]);
        if (m == -INFINITY) m = 0.f;   // every logit -inf (entries removed): probabilities 0
        float sum = 0.f;
        for (int e = 0; e < deg; ++e) sum += expf(lr[(int64_t)e * H] - m);
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
        for (int e = 0; e < deg; ++e) pr[(int64_t)e * H] = expf(lr[(int64_t)e * H] - m) * inv;
    }
}

// Ordinary rows when H divides 32: a lane group of gs lanes per row (gs a
// power of two and a multiple of H, sized to the widest row of the bucket,
// at most 32), rows of a bucket side by side, 32/gs rows per warp.  A row's
// logits are contiguous (entry-major, head-minor), so element j belongs to
// lane j % gs and head j % H: the group reads the row coalesced and reduces
// each head's maximum and sum over its lanes with xor shuffles.  Rows of at
// most gs elements (most rows of a sparse graph) are held in registers: one
// load and one expf per element; longer rows take three coalesced walks.
struct SmaxSeg {
    int first_task, list_begin, count, gs;
};

__global__ void __launch_bounds__(256)
k_softmax_rows(const int* __restrict__ indptr, const int* __restrict__ hdr, const int* __restrict__ rows,
               int H, const float* __restrict__ logits, float* __restrict__ probs) {
    __shared__ SmaxSeg segs[kNumBuckets];
    __shared__ int s_nseg, s_total;
    if (threadIdx.x == 0) {
        int t = 0, k = 0;
        for (int b = kNumBuckets - 1; b >= 0; --b) {
            const int cnt = hdr[HdrLayout::kCount + b];
            if (cnt == 0) continue;
            const int lb = b - kExactBuckets;
            const int64_t hi = b < kExactBuckets ? b : (lb < kLogBuckets - 1 ? log_bucket_hi(lb) : 0x7fffffff);
            int gs = H;
            while (gs < 32 && gs < hi * H) gs <<= 1;
            segs[k++] = SmaxSeg{t, hdr[HdrLayout::kOffset + b], cnt, gs};
            t += (cnt + 32 / gs - 1) / (32 / gs);
        }
        s_nseg = k;
        s_total = t;
    }
    __syncthreads();
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    int sidx = 0;
    for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < s_total; t += gridDim.x * wpb) {
        while (sidx + 1 < s_nseg && segs[sidx + 1].first_task <= t) ++sidx;
        const SmaxSeg sg = segs[sidx];
        const int gs = sg.gs, grp = lane / gs, lig = lane - grp * gs;
        const int pos = (t - sg.first_task) * (32 / gs) + grp;
        int beg = 0, n = 0;
        if (pos < sg.count) {
            const int row = rows[sg.list_begin + pos];
            beg = indptr[row];
            n = (indptr[row + 1] - beg) * H;
        }
        const float* lr = logits + static_cast<int64_t>(beg) * H;
        float* pr = probs + static_cast<int64_t>(beg) * H;
        const bool inreg = n <= gs;   // the row fits the group: one element per lane
        const float x0 = lig < n ? lr[lig] : -INFINITY;
        float m = x0;
        if (!inreg)
            for (int j = lig + gs; j < n; j += gs) m = fmaxf(m, lr[j]);
        for (int o = H; o < gs; o <<= 1) m = fmaxf(m, __shfl_xor_sync(full, m, o));
        if (m == -INFINITY) m = 0.f;   // every logit -inf (entries removed): probabilities 0
        const float e0 = lig < n ? expf(x0 - m) : 0.f;
        float sum = e0;
        if (!inreg)
            for (int j = lig + gs; j < n; j += gs) sum += expf(lr[j] - m);
        for (int o = H; o < gs; o <<= 1) sum += __shfl_xor_sync(full, sum, o);
        const float inv = sum > 0.f ? 1.f / sum : 0.f;
        if (lig < n) pr[lig] = e0 * inv;
        if (!inreg)
            for (int j = lig + gs; j < n; j += gs) pr[j] = expf(lr[j] - m) * inv;
    }
}

// Split rows' chunks when H divides 32: a warp per chunk, lanes over the
// chunk's contiguous (entry, head) logits (element j: head j % H), heads
// reduced over lanes H apart.  Step 1: the chunk's (M_c, S_c) per head.
__global__ void __launch_bounds__(256)
k_softmax_chunk_stats_w(const int* __restrict__ indptr, const int* __restrict__ hdr, const int2* __restrict__ chunks,
                        int chunk_edges, int H, const float* __restrict__ logits, Partials part) {
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
    const int n_chunks = hdr[HdrLayout::kChunks];
    for (int c = blockIdx.x * wpb + (threadIdx.x >> 5); c < n_chunks; c += gridDim.x * wpb) {
        const int2 ck = chunks[c];
        const int n = (min(ck.y + chunk_edges, indptr[ck.x + 1]) - ck.y) * H;
        const float* lr = logits + static_cast<int64_t>(ck.y) * H;
        float m = -INFINITY;
        for (int j = lane; j < n; j += 32) m = fmaxf(m, lr[j]);
        for (int o = H; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(full, m, o));
        const float mref = m == -INFINITY ? 0.f : m;   // every logit -inf: S_c = 0
        float sum = 0.f;
        for (int j = lane; j < n; j += 32) sum += expf(lr[j] - mref);
        for (int o = H; o < 32; o <<= 1) sum += __shfl_xor_sync(full, sum, o);
        if (lane < H) {
            part.m[static_cast<int64_t>(c) * H + lane] = m;
            part.s[static_cast<int64_t>(c) * H + lane] = sum;
        }
    }
}

// Step 3 (H divides 32), a warp per chunk: p = exp(l - M) / S with the row's
// (M, 1/S) from its first chunk.
__global__ void __launch_bounds__(256)
k_softmax_chunk_write_w(const int* __restrict__ indptr, const int* __restrict__ hdr, const int2* __restrict__ chunks,
                        int chunk_edges, int H, const float* __restrict__ logits, float* __restrict__ probs,
                        Partials part) {
    const int lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
    const int n_chunks = hdr[HdrLayout::kChunks];
    for (int c = blockIdx.x * wpb + (threadIdx.x >> 5); c < n_chunks; c += gridDim.x * wpb) {
        const int2 ck = chunks[c];
        const int rbeg = indptr[ck.x];
        const int n = (min(ck.y + chunk_edges, indptr[ck.x + 1]) - ck.y) * H;
        const int c0 = c - (ck.y - rbeg) / chunk_edges;
        const int h = lane % H;   // the head of every element this lane touches
        const float M = part.m[static_cast<int64_t>(c0) * H + h], inv = part.s[static_cast<int64_t>(c0) * H + h];
        const float* lr = logits + static_cast<int64_t>(ck.y) * H;
        float* pr = probs + static_cast<int64_t>(ck.y) * H;
        for (int j = lane; j < n; j += 32) pr[j] = expf(lr[j] - M) * inv;
    }
}

// Split rows, in their chunks (a thread per (chunk, head)): step 1, each
// chunk's maximum M_c and sum S_c = sum exp(l - M_c) into the partials.
__global__ void __launch_bounds__(256)
k_softmax_chunk_stats(const int* __restrict__ indptr, const int* __restrict__ hdr, const int2* __restrict__ chunks,
                      int chunk_edges, int H, const float* __restrict__ logits, Partials part) {
    const int64_t total = (int64_t)hdr[HdrLayout::kChunks] * H;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(t / H), h = (int)(t - (int64_t)c * H);
        const int2 ck = chunks[c];
        const int beg = ck.y, n = min(ck.y + chunk_edges, indptr[ck.x + 1]) - ck.y;
        const float* lr = logits + (int64_t)beg * H + h;
        float m = -INFINITY;
        for (int e = 0; e < n; ++e) m = fmaxf(m, lr[(int64_t)e * H]);
        const float mref = m == -INFINITY ? 0.f : m;   // every logit -inf: S_c = 0
        float sum = 0.f;
        for (int e = 0; e < n; ++e) sum += expf(lr[(int64_t)e * H] - mref);
        part.m[t] = m;
        part.s[t] = sum;
    }
}

// Step 2, a thread per (split row, head): the row's statistics from its
// chunks' (M = max M_c, S = sum S_c exp(M_c - M)), stored as (M, 1/S) in the
// slot of the row's first chunk.
__global__ void __launch_bounds__(256)
k_softmax_long_merge(const int* __restrict__ indptr, const int* __restrict__ hdr, const int2* __restrict__ longs,
                     int chunk_edges, int H, Partials part) {
    const int64_t total = (int64_t)hdr[HdrLayout::kLong] * H;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int li = (int)(t / H), h = (int)(t - (int64_t)li * H);
        const int2 lg = longs[li];
        const int deg = indptr[lg.x + 1] - indptr[lg.x];
        const int nch = (deg + chunk_edges - 1) / chunk_edges;
        float M = -INFINITY;
        for (int c = 0; c < nch; ++c) M = fmaxf(M, part.m[(int64_t)(lg.y + c) * H + h]);
        if (M == -INFINITY) M = 0.f;   // every logit -inf (entries removed): probabilities 0
        float S = 0.f;
        for (int c = 0; c < nch; ++c) {
            const int64_t k = (int64_t)(lg.y + c) * H + h;
            S += part.s[k] * expf(part.m[k] - M);
        }
        part.m[(int64_t)lg.y * H + h] = M;
        part.s[(int64_t)lg.y * H + h] = S > 0.f ? 1.f / S : 0.f;
    }
}

// Step 3, a thread per (chunk, head): p = exp(l - M) / S with the row's
// (M, 1/S) from its first chunk (a split row's chunks are consecutive).
__global__ void __launch_bounds__(256)
k_softmax_chunk_write(const int* __restrict__ indptr, const int* __restrict__ hdr, const int2* __restrict__ chunks,
                      int chunk_edges, int H, const float* __restrict__ logits, float* __restrict__ probs,
                      Partials part) {
    const int64_t total = (int64_t)hdr[HdrLayout::kChunks] * H;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(t / H), h = (int)(t - (int64_t)c * H);
        const int2 ck = chunks[c];
        const int beg = ck.y, n = min(ck.y + chunk_edges, indptr[ck.x + 1]) - ck.y;
        const int c0 = c - (beg - indptr[ck.x]) / chunk_edges;
        const float M = part.m[(int64_t)c0 * H + h], inv = part.s[(int64_t)c0 * H + h];
        const float* lr = logits + (int64_t)beg * H + h;
        float* pr = probs + (int64_t)beg * H + h;
        for (int e = 0; e < n; ++e) pr[(int64_t)e * H] = expf(lr[(int64_t)e * H] - M) * inv;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

bool choose_row_kernel(int H, int D, gtattn_dtype dt, const void* Q, const void* K, const void* V,
                       const void* out, int force, RowChoice* c) {
    const int esz = dt == GTATTN_F32 ? 4 : 2;   // input element size
    const int HD = H * D;
    const uintptr_t al = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                         reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(out);
    if (force != GTATTN_KERNEL_GENERIC && (al & 15u) == 0) {
        const int per_vec = 16 / esz;
        // Preference: two 16-byte vectors per lane, then one, then four
        // (fp32 only).  Two vectors put twice as many rows in a warp as one
        // (R-MAT, 4 x 32 bf16: 8 lanes and 4 rows per warp instead of 16 and
        // 2), halving the per-row work per warp instruction on graphs of
        // mostly short rows (R-MAT 1.48 -> 1.25 ms); four need too many
        // registers for the K/V pipeline in bf16 (1.52 ms).
        static constexpr int kOrder[3] = {2, 1, 4};
        for (int vpl : kOrder) {
            if (esz == 2 && vpl > 2) continue;
            const int E = vpl * per_vec;
            if (D % E != 0) continue;
            const int lph = D / E;
            const int G = HD / E;
            if (!is_pow2(lph) || !is_pow2(G) || G > 32) continue;
            *c = RowChoice{RowKernel::kVector, vpl, G, lph};
            return true;
        }
    }
    if (force == GTATTN_KERNEL_VECTOR) return false;
    // heads too narrow for a 16-byte lane split: one lane per head
    if ((force == GTATTN_KERNEL_AUTO || force == GTATTN_KERNEL_NARROW) && D <= kNarrowMaxD && H <= 32) {
        int G = 1;
        while (G < H) G <<= 1;
        const bool pair = D % 2 == 0 && (al & static_cast<uintptr_t>(2 * esz - 1)) == 0;
        *c = RowChoice{RowKernel::kNarrow, pair ? 1 : 0, G, 1};
        return true;
    }
    if (force == GTATTN_KERNEL_NARROW) return false;
    if (H > kGenMaxH || HD > kMaxHD) return false;
    *c = RowChoice{RowKernel::kGeneric, 0, 0, 0};
    return true;
}

// Warp tasks of the narrow kernel: P = 32 / G rows per warp, one task per
// chunk, at most one part-filled task per segment.
static int narrow_task_bound(const RowParams& p) {
    if (p.task_bound <= 0) return 0;
    const int P = 32 / p.G;
    const int64_t b = (static_cast<int64_t>(p.N) + P - 1) / P + (p.task_bound - p.N) + kMaxSegs;
    return b < p.task_bound ? static_cast<int>(b) : p.task_bound;
}

// The narrow kernel takes the fused mode on [N, H, D] rows; other calls with
// that choice go to the generic kernel.
static bool narrow_applies(const RowChoice& c, Mode mode, const RowParams& p) {
    return c.kind == RowKernel::kNarrow && mode == kFused && !p.ndh && !(p.bias && p.values);
}

template <typename K>
static int grid_persistent(K kernel, int threads, size_t smem) {
    static std::mutex mu;
    static std::unordered_map<const void*, int> cache;
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(reinterpret_cast<const void*>(kernel));
    if (it != cache.end()) return it->second;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    int grid = per_sm * num_sms();
    cache[reinterpret_cast<const void*>(kernel)] = grid;
    return grid;
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel of the stream finishes (it waits in wait_prior_grid).
template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kernel, int grid, int threads, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The persistent grid, but no more blocks than the tasks can occupy (small
// graphs: a few blocks instead of several per SM).
static int grid_for_tasks(int persistent, int task_bound, int warps_per_block) {
    if (task_bound <= 0) return persistent;
    const int need = (task_bound + warps_per_block - 1) / warps_per_block;
    return need < persistent ? need : persistent;
}

template <typename T, typename TO, int MODE, int EXT = 0>
static gtattn_status launch_vec_t(int vpl, const RowParams& p, cudaStream_t s) {
    auto go = [&](auto kernel) {
        const int grid = grid_for_tasks(grid_persistent(kernel, kRowThreads, 0), p.task_bound, kRowThreads / 32);
        return launch_pdl(kernel, grid, kRowThreads, 0, s, p);
    };
    cudaError_t e;
    switch (vpl) {
        case 1: e = go(k_rows_vec<T, TO, 1, MODE, EXT>); break;
        case 2: e = go(k_rows_vec<T, TO, 2, MODE, EXT>); break;
        case 4:
            if constexpr (sizeof(T) == 4) { e = go(k_rows_vec<T, TO, 4, MODE, EXT>); break; }
            return GTATTN_ERR_UNSUPPORTED;
        default: return GTATTN_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

template <typename T, typename TO>
static gtattn_status launch_rows_t(Mode mode, const RowChoice& c, const RowParams& p, cudaStream_t s) {
    if (narrow_applies(c, mode, p)) {
        auto go = [&](auto kernel) {
            const int grid = grid_for_tasks(grid_persistent(kernel, kRowThreads, 0), narrow_task_bound(p),
                                            kRowThreads / 32);
            return launch_pdl(kernel, grid, kRowThreads, 0, s, p);
        };
        const cudaError_t e = c.vpl ? go(k_rows_narrow<T, TO, true>) : go(k_rows_narrow<T, TO, false>);
        return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
    }
    if (c.kind == RowKernel::kVector) {
        // one of the bias or the values at a time (the entry points take one)
        if (p.bias && p.values) return GTATTN_ERR_UNSUPPORTED;
        switch (mode) {
            case kFused:
                if (p.bias) return launch_vec_t<T, TO, kFused, kExtBias>(c.vpl, p, s);
                if (p.values) return launch_vec_t<T, TO, kFused, kExtValues>(c.vpl, p, s);
                return launch_vec_t<T, TO, kFused>(c.vpl, p, s);
            case kSpmm: return launch_vec_t<T, TO, kSpmm>(c.vpl, p, s);
            case kSddmm:
                if (p.bias) return launch_vec_t<T, TO, kSddmm, kExtBias>(c.vpl, p, s);
                if (p.values) return launch_vec_t<T, TO, kSddmm, kExtValues>(c.vpl, p, s);
                return launch_vec_t<T, TO, kSddmm>(c.vpl, p, s);
        }
        return GTATTN_ERR_UNSUPPORTED;
    }
    auto go = [&](auto kernel) {
        const int grid = grid_for_tasks(grid_persistent(kernel, kGenWarps * 32, 0), p.task_bound, kGenWarps);
        return launch_pdl(kernel, grid, kGenWarps * 32, 0, s, p);
    };
    auto by_kpl = [&](auto kpl4, auto kpl8, auto kpl32) {
        const int kpl = (p.HD + 31) / 32;
        return kpl <= 4 ? go(kpl4) : kpl <= 8 ? go(kpl8) : go(kpl32);
    };
    cudaError_t e;
    switch (mode) {
        case kFused:
            e = by_kpl(k_rows_generic<T, TO, kFused, 4>, k_rows_generic<T, TO, kFused, 8>,
                       k_rows_generic<T, TO, kFused, 32>);
            break;
        case kSpmm:
            e = by_kpl(k_rows_generic<T, TO, kSpmm, 4>, k_rows_generic<T, TO, kSpmm, 8>,
                       k_rows_generic<T, TO, kSpmm, 32>);
            break;
        default:
            e = by_kpl(k_rows_generic<T, TO, kSddmm, 4>, k_rows_generic<T, TO, kSddmm, 8>,
                       k_rows_generic<T, TO, kSddmm, 32>);
            break;
    }
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

// Cooperative launch (every block resident at once, so the grid can sync).
template <typename Kern, typename... Args>
static cudaError_t launch_coop(Kern kernel, int grid, int threads, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Blocks of `kernel` (threads, smem dynamic bytes) resident on the whole GPU
// at once: the bound of a cooperative grid.  Cached per kernel.
template <typename K>
static int coop_grid(K kernel, int threads, size_t smem) {
    static std::mutex mu;
    static std::unordered_map<const void*, int> cache;
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(reinterpret_cast<const void*>(kernel));
    if (it != cache.end()) return it->second;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int grid = per_sm * num_sms();
    cache[reinterpret_cast<const void*>(kernel)] = grid;
    return grid;
}

// The one-launch path's launch: cooperative when a row may be split (the
// grid then synchronises before the combine), else an ordinary launch
// (programmatic dependent launch: it may start while the previous kernel of
// the stream finishes).
template <typename Kern>
static cudaError_t launch_small(Kern kernel, int grid, int threads, size_t smem, cudaStream_t s,
                                const RowParams& p) {
    if (p.small_no_split) return launch_pdl(kernel, grid, threads, smem, s, p);
    return launch_coop(kernel, grid, threads, smem, s, p);
}

template <typename T, typename TO>
static gtattn_status launch_small_t(const RowChoice& c, const RowParams& p, cudaStream_t s) {
    const size_t smem = sizeof(int2) * static_cast<size_t>(p.small_max_chunks + p.small_max_long);
    auto go = [&](auto kernel, int threads) {
        const int grid = grid_for_tasks(coop_grid(kernel, threads, smem), p.task_bound, threads / 32);
        return launch_small(kernel, std::max(grid, 1), threads, smem, s, p);
    };
    cudaError_t e;
    if (narrow_applies(c, kFused, p)) {
        auto go_n = [&](auto kernel) {
            const int grid = grid_for_tasks(coop_grid(kernel, kRowThreads, smem), narrow_task_bound(p),
                                            kRowThreads / 32);
            return launch_small(kernel, std::max(grid, 1), kRowThreads, smem, s, p);
        };
        e = c.vpl ? go_n(k_rows_narrow<T, TO, true, true>) : go_n(k_rows_narrow<T, TO, false, true>);
    } else if (c.kind == RowKernel::kVector) {
        if (p.bias && p.values) return GTATTN_ERR_UNSUPPORTED;
        auto by_ext = [&](auto k0, auto kb, auto kv) {
            return p.bias ? go(kb, kRowThreads) : p.values ? go(kv, kRowThreads) : go(k0, kRowThreads);
        };
        switch (c.vpl) {
            case 1:
                e = by_ext(k_rows_vec<T, TO, 1, kFused, 0, true>, k_rows_vec<T, TO, 1, kFused, kExtBias, true>,
                           k_rows_vec<T, TO, 1, kFused, kExtValues, true>);
                break;
            case 2:
                e = by_ext(k_rows_vec<T, TO, 2, kFused, 0, true>, k_rows_vec<T, TO, 2, kFused, kExtBias, true>,
                           k_rows_vec<T, TO, 2, kFused, kExtValues, true>);
                break;
            case 4:
                if constexpr (sizeof(T) == 4) {
                    e = by_ext(k_rows_vec<T, TO, 4, kFused, 0, true>, k_rows_vec<T, TO, 4, kFused, kExtBias, true>,
                               k_rows_vec<T, TO, 4, kFused, kExtValues, true>);
                    break;
                }
                return GTATTN_ERR_UNSUPPORTED;
            default: return GTATTN_ERR_UNSUPPORTED;
        }
    } else {
        const int kpl = (p.HD + 31) / 32;
        e = kpl <= 4 ? go(k_rows_generic<T, TO, kFused, 4, true>, kGenWarps * 32)
            : kpl <= 8 ? go(k_rows_generic<T, TO, kFused, 8, true>, kGenWarps * 32)
                       : go(k_rows_generic<T, TO, kFused, 32, true>, kGenWarps * 32);
    }
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

gtattn_status launch_rows_small(gtattn_dtype dt, const RowChoice& c, const RowParams& p, cudaStream_t s) {
    switch (dt) {
        case GTATTN_BF16: return launch_small_t<__nv_bfloat16, __nv_bfloat16>(c, p, s);
        case GTATTN_BF16_OUT_F32: return launch_small_t<__nv_bfloat16, float>(c, p, s);
        case GTATTN_F32: return launch_small_t<float, float>(c, p, s);
    }
    return GTATTN_ERR_INVALID_ARG;
}

gtattn_status launch_rows(Mode mode, gtattn_dtype dt, const RowChoice& c, const RowParams& p,
                          cudaStream_t s) {
    switch (dt) {
        case GTATTN_BF16: return launch_rows_t<__nv_bfloat16, __nv_bfloat16>(mode, c, p, s);
        case GTATTN_BF16_OUT_F32: return launch_rows_t<__nv_bfloat16, float>(mode, c, p, s);
        case GTATTN_F32: return launch_rows_t<float, float>(mode, c, p, s);
    }
    return GTATTN_ERR_INVALID_ARG;
}

gtattn_status launch_combine(Mode mode, gtattn_dtype dt, const RowParams& p, cudaStream_t s) {
    // rows of few chunks a warp each (when H divides 32), the others a block each
    const int warp_rows = (32 % p.H == 0) ? 1 : 0;
    auto go = [&](auto kernel) {
        return launch_pdl(kernel, grid_persistent(kernel, kCombThreads, 0), kCombThreads, 0, s, p, warp_rows);
    };
    cudaError_t e;
    if (dt == GTATTN_BF16)
        e = mode == kFused ? go(k_combine<__nv_bfloat16, kFused>) : go(k_combine<__nv_bfloat16, kSpmm>);
    else
        e = mode == kFused ? go(k_combine<float, kFused>) : go(k_combine<float, kSpmm>);
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

gtattn_status launch_edge_softmax(const int* indptr, int N, int H, const TaskLists& L, const Partials& part,
                                  const float* logits, float* probs, cudaStream_t s) {
    if (N == 0) return GTATTN_OK;
    if (32 % H == 0)
        k_softmax_rows<<<grid_persistent(k_softmax_rows, 256, 0), 256, 0, s>>>(indptr, L.hdr, L.rows, H, logits, probs);
    else
        k_softmax_short<<<grid_persistent(k_softmax_short, 256, 0), 256, 0, s>>>(indptr, L.hdr, L.rows, H, logits,
                                                                                  probs);
    if (32 % H == 0)
        k_softmax_chunk_stats_w<<<grid_persistent(k_softmax_chunk_stats_w, 256, 0), 256, 0, s>>>(
            indptr, L.hdr, L.chunks, L.chunk_edges, H, logits, part);
    else
        k_softmax_chunk_stats<<<grid_persistent(k_softmax_chunk_stats, 256, 0), 256, 0, s>>>(
            indptr, L.hdr, L.chunks, L.chunk_edges, H, logits, part);
    k_softmax_long_merge<<<grid_persistent(k_softmax_long_merge, 256, 0), 256, 0, s>>>(
        indptr, L.hdr, L.longs, L.chunk_edges, H, part);
    if (32 % H == 0)
        k_softmax_chunk_write_w<<<grid_persistent(k_softmax_chunk_write_w, 256, 0), 256, 0, s>>>(
            indptr, L.hdr, L.chunks, L.chunk_edges, H, logits, probs, part);
    else
        k_softmax_chunk_write<<<grid_persistent(k_softmax_chunk_write, 256, 0), 256, 0, s>>>(
            indptr, L.hdr, L.chunks, L.chunk_edges, H, logits, probs, part);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
}

}  // namespace gt
