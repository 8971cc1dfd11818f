// dense.cu -- attention over complete blocks on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory, operands staged by TMA).
//
// A complete block (rows r0..r0+n-1 attending to exactly r0..r0+n-1) is
// dense scaled-dot-product attention: out = softmax(scale * Q K^T) V per head
// ("Graph Transformer in a Nutshell", the all-pairs Attn equation;
// "Graph Transformer theory, derivation and implementation", review of
// scaled dot-product attention; a complete graph with self-loops makes the
// sparse definition reduce to it).
//
// A persistent CTA per SM walks work items: two 128-row query tiles (A, B)
// of one block and one head, which share every K/V tile.  Warp roles:
//   warps 0-3 / 4-7   softmax of tile A / B: one warpgroup per tile, each
//                     thread one query row (= TMEM lane) over all 128 key
//                     columns of a tile, held in registers (no exchange
//                     between warps, one TMEM read of S per tile)
//   warp 8            MMA issue: the whole warp runs the loop, one elected
//                     lane issues S_g = Q_g K_j^T (tcgen05.mma M=128 N=128,
//                     fp32 in TMEM) and O_g += P_g V_j (M=128 N=64, P read
//                     from TMEM) once softmax g has written P_g
//   warp 9            TMA: Q tiles (double-buffered across items), K_j and V_j
//                     into a 4-stage ring (128-byte swizzle)
//   warps 10-11       idle; warps 8-11 hand registers to the softmax
//                     warpgroups (setmaxnreg)
// TMEM holds three S/P buffers used in rotation (the next S tile is computed
// while the softmax works on the current one) and O_A, O_B.  The softmax
// takes the row maximum m (log2 units) of an item's first key tile and keeps
// it while later tiles' P sums stay below a limit (P stays small and finite);
// a row whose tile sum goes over takes that tile's exact maximum, and O_g and
// the row sum are rescaled.  It writes P = 2^(s*scale*log2e - m) back over
// S_g as two bf16 terms P_hi = bf16(P), P_lo = bf16(P - P_hi); O_g += P_hi V +
// P_lo V keeps the product at ~16-bit precision on the bf16 tensor path (a
// single bf16 P would cost ~2^-9 relative per weight, outside the accuracy
// bound of the bf16 path).  out = O / l at the end of an item.  Every
// mbarrier wait is bounded: on timeout the CTA records an error code, drains
// (bounded) the copies and MMAs it issued, frees its tensor memory and
// returns.
#include "dense.cuh"
#include "tc.cuh"

#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <mutex>

namespace gt {

namespace {

constexpr int kTile = 128;              // rows per Q / K / V tile
constexpr long long kWaitCycles = kTcWaitCycles;   // drains (and the default bound of the other waits)

// Per head width D (32, 64 or 128).  Tensor memory holds three 128-column
// S/P buffers and O (D columns) for each query tile of an item, so D = 128
// takes one query tile per item; shared memory holds the Q buffers and the
// K/V ring, so D = 128 keeps one Q buffer and three stages (224 KB).  Rows of
// 64 bytes (D = 32) use the 64-byte swizzle; rows of 256 bytes (D = 128) are
// two 128-byte-swizzled 64-column sub-tiles, 16 KB apart.
template <int D>
struct Cfg {
    static_assert(D == 32 || D == 64 || D == 128, "head widths of the dense kernel");
    static constexpr uint32_t kTB = kTile * D * 2;          // one tile, bf16
    static constexpr int kNq = D == 128 ? 1 : 2;            // query tiles per work item
    static constexpr int kQBufs = D == 128 ? 1 : 2;
    static constexpr int kStages = D == 128 ? 3 : 4;        // K/V ring
    static constexpr int kSub = D == 128 ? 2 : 1;           // 64-column sub-tiles of a row
    static constexpr int kBoxX = D == 32 ? 32 : 64;         // TMA box width (elements)
    static constexpr size_t kSmemQ = 0;
    static constexpr size_t kSmemKV = static_cast<size_t>(kQBufs) * kNq * kTB;
    static constexpr size_t kSmemBytes = kSmemKV + static_cast<size_t>(kStages) * 2 * kTB;
    static constexpr size_t kSmemAlloc = kSmemBytes + 1024;
    // descriptor start-address units (16 bytes) between K/V stages and Q tiles
    static constexpr uint64_t kStageUnits = (2 * kTB) >> 4;
    static constexpr uint64_t kQUnits = kTB >> 4;
    static constexpr uint64_t kSubUnits = (kTB / 2) >> 4;   // D = 128: second sub-tile
    static constexpr int kVStep = D == 32 ? 64 : 128;        // units per 16 keys of V (16 rows)
    static constexpr uint32_t kSbo = D == 32 ? 512 : 1024;   // 8-row group stride (bytes)
    static constexpr uint32_t kVLbo = D == 128 ? kTB / 2 : 8192;   // V: stride between 64-column atoms
    static_assert(kSubUnits > 0 && kVStep > 0, "(every instance names its constants)");
};


// Shared-memory descriptor of a 64-byte-swizzled operand (layout type 4):
// start address, leading and stride byte offsets in 16-byte units.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(4) << 61;
    return d;
}
// K-major operand (Q, K: rows of D features) and MN-major operand (V: rows
// of D features read along the keys) descriptors for head width D.
template <int D>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
    if constexpr (D == 32) return smem_desc_sw64(saddr, 16, Cfg<D>::kSbo);
    else return smem_desc_sw128(saddr, 16, Cfg<D>::kSbo);
}
template <int D>
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr) {
    if constexpr (D == 32) return smem_desc_sw64(saddr, Cfg<D>::kVLbo, Cfg<D>::kSbo);
    else return smem_desc_sw128(saddr, Cfg<D>::kVLbo, Cfg<D>::kSbo);
}

// Non-blocking test (never suspends the thread).  The MMA warp issues it
// before a batch of MMAs and reads the answer after the batch, so the test's
// latency overlaps the batch instead of leaving the tensor pipe idle.
__device__ __forceinline__ uint32_t mbar_probe(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok;
}
// Warp vote kept in program order with the surrounding asm (so a probe's
// answer is consumed only where this vote stands).
__device__ __forceinline__ bool warp_any_ordered(uint32_t v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "vote.sync.any.pred q, p, 0xffffffff;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v)
        : "memory");
    return r != 0;
}
// The MMA batches of the dense kernel, each in one asm block issued by one
// elected lane of the converged MMA warp.
// S (+)= Q K^T over K = 64: four K-steps of 32 bytes (descriptor start +2).
__device__ __forceinline__ void mma_s_batch(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\tsetp.ne.b32 p, 0, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %5, %3, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %7, %3, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %9, %3, q;\n\t}"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "l"(a + 2), "l"(b + 2), "l"(a + 4), "l"(b + 4), "l"(a + 6), "l"(b + 6)
        : "memory");
}
// Half a key-tile step of the MMA warp in one asm block (one elected lane):
//   [do_pv] O (+)= P_hi V + P_lo V over 128 keys in eight 16-key steps (P_hi
//           of keys 32c..32c+31 in columns 32c..32c+15, P_lo in 32c+16..
//           32c+31; the V rows of a step start 2048 bytes (128 descriptor
//           units) after the previous step's), commit -> bar_o
//   [do_x]  commit -> bar_x (tracks every MMA issued so far)
//   [do_s]  S = Q K^T over K = 64 in four 16-element steps (descriptor start
//           +2 per step), commit -> bar_s
// The per-step descriptors are formed inside the block from the bases, so
// the MMA warp does little between blocks: the tensor pipe queues only a few
// MMAs ahead, and every gap between blocks risks leaving it idle.
__device__ __forceinline__ void mma_half_step(uint32_t d_o, uint32_t a_p, uint64_t b_v, uint32_t id_o, uint32_t acc,
                                              uint32_t bar_o, uint32_t do_pv, uint32_t bar_x, uint32_t do_x,
                                              uint32_t d_s, uint64_t a_q, uint64_t b_k, uint32_t id_s,
                                              uint32_t bar_s, uint32_t do_s) {
    asm volatile(
        "{\n\t.reg .pred p, q, f, e, pv, px, ps;\n\t"
        ".reg .b64 v1, v2, v3, v4, v5, v6, v7, q2, q4, q6, k2, k4, k6;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, 0, 0;\n\tsetp.ne.b32 f, 0, 0;\n\t"
        "add.s64 v1, %2, 128;\n\tadd.s64 v2, %2, 256;\n\tadd.s64 v3, %2, 384;\n\tadd.s64 v4, %2, 512;\n\t"
        "add.s64 v5, %2, 640;\n\tadd.s64 v6, %2, 768;\n\tadd.s64 v7, %2, 896;\n\t"
        "add.s64 q2, %10, 2;\n\tadd.s64 q4, %10, 4;\n\tadd.s64 q6, %10, 6;\n\t"
        "add.s64 k2, %11, 2;\n\tadd.s64 k4, %11, 4;\n\tadd.s64 k6, %11, 6;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.and.b32 pv, %6, 0, e;\n\tsetp.ne.and.b32 px, %8, 0, e;\n\tsetp.ne.and.b32 ps, %14, 0, e;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+0], %2, %3, p;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+16], %2, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+8], v1, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+24], v1, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+32], v2, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+48], v2, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+40], v3, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+56], v3, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+64], v4, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+80], v4, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+72], v5, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+88], v5, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+96], v6, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+112], v6, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+104], v7, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+120], v7, %3, q;\n\t"
        "@pv tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"
        "@px tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t"
        "@ps tcgen05.mma.cta_group::1.kind::f16 [%9], %10, %11, %12, f;\n\t"
        "@ps tcgen05.mma.cta_group::1.kind::f16 [%9], q2, k2, %12, q;\n\t"
        "@ps tcgen05.mma.cta_group::1.kind::f16 [%9], q4, k4, %12, q;\n\t"
        "@ps tcgen05.mma.cta_group::1.kind::f16 [%9], q6, k6, %12, q;\n\t"
        "@ps tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%13];\n\t}"
        ::"r"(d_o), "r"(a_p), "l"(b_v), "r"(id_o), "r"(acc), "r"(bar_o), "r"(do_pv), "r"(bar_x), "r"(do_x),
          "r"(d_s), "l"(a_q), "l"(b_k), "r"(id_s), "r"(bar_s), "r"(do_s)
        : "memory");
}

// S = Q K^T over K = D for D = 32 (two 16-element steps) or D = 128 (eight:
// four in each 64-column sub-tile), by one elected lane of the converged
// warp; `pred` != 0 to issue (uniform over the warp).
template <int D>
__device__ __forceinline__ void mma_s_batch_d(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t pred) {
    if constexpr (D == 32) {
        asm volatile(
            "{\n\t.reg .pred f, q, e, ps;\n\tsetp.ne.b32 f, 0, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"
            "elect.sync _|e, 0xffffffff;\n\tsetp.ne.and.b32 ps, %4, 0, e;\n\t"
            "@ps tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
            "@ps tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %3, q;\n\t}"
            ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(pred), "l"(a + 2), "l"(b + 2)
            : "memory");
    } else {
        constexpr uint64_t S = Cfg<D>::kSubUnits;
        asm volatile(
            "{\n\t.reg .pred f, q, e, ps;\n\t.reg .b64 a1, a2, a3, a4, a5, a6, a7, b1, b2, b3, b4, b5, b6, b7;\n\t"
            "setp.ne.b32 f, 0, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"
            "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\tadd.s64 a4, %1, %5;\n\t"
            "add.s64 a5, a4, 2;\n\tadd.s64 a6, a4, 4;\n\tadd.s64 a7, a4, 6;\n\t"
            "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\tadd.s64 b4, %2, %5;\n\t"
            "add.s64 b5, b4, 2;\n\tadd.s64 b6, b4, 4;\n\tadd.s64 b7, b4, 6;\n\t"
            "elect.sync _|e, 0xffffffff;\n\tsetp.ne.and.b32 ps, %4, 0, e;\n\t"
            "@ps tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, f;\n\t"
            "@ps tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, q;\n\t"
            "@ps tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, q;\n\t"
            "@ps tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, q;\n\t"
            "@ps tcgen05.mma.cta_group::1.kind::f16 [%0], a4, b4, %3, q;\n\t"
            "@ps tcgen05.mma.cta_group::1.kind::f16 [%0], a5, b5, %3, q;\n\t"
            "@ps tcgen05.mma.cta_group::1.kind::f16 [%0], a6, b6, %3, q;\n\t"
            "@ps tcgen05.mma.cta_group::1.kind::f16 [%0], a7, b7, %3, q;\n\t}"
            ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(pred), "n"(S)
            : "memory");
    }
}
// Commit of everything the elected lane issued so far to an mbarrier, when
// `pred` != 0 (uniform over the warp).
__device__ __forceinline__ void tc_commit_if(uint32_t bar, uint32_t pred) {
    asm volatile(
        "{\n\t.reg .pred e, pc;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.and.b32 pc, %1, 0, e;\n\t"
        "@pc tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        ::"r"(bar), "r"(pred)
        : "memory");
}
// The half key-tile step of mma_half_step for D = 32 or 128: O (+)= P_hi V +
// P_lo V with N = D (V's 16-key steps kVStep units apart), the commits, then
// S over K = D.
template <int D>
__device__ __forceinline__ void mma_half_step_d(uint32_t d_o, uint32_t a_p, uint64_t b_v, uint32_t id_o, uint32_t acc,
                                                uint32_t bar_o, uint32_t do_pv, uint32_t bar_x, uint32_t do_x,
                                                uint32_t d_s, uint64_t a_q, uint64_t b_k, uint32_t id_s,
                                                uint32_t bar_s, uint32_t do_s) {
    constexpr int VS = Cfg<D>::kVStep;
    asm volatile(
        "{\n\t.reg .pred p, q, e, pv, px;\n\t"
        ".reg .b64 v1, v2, v3, v4, v5, v6, v7;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 q, 0, 0;\n\t"
        "add.s64 v1, %2, %9;\n\tadd.s64 v2, %2, %10;\n\tadd.s64 v3, %2, %11;\n\tadd.s64 v4, %2, %12;\n\t"
        "add.s64 v5, %2, %13;\n\tadd.s64 v6, %2, %14;\n\tadd.s64 v7, %2, %15;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.and.b32 pv, %6, 0, e;\n\tsetp.ne.and.b32 px, %8, 0, e;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+0], %2, %3, p;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+16], %2, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+8], v1, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+24], v1, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+32], v2, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+48], v2, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+40], v3, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+56], v3, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+64], v4, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+80], v4, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+72], v5, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+88], v5, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+96], v6, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+112], v6, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+104], v7, %3, q;\n\t"
        "@pv tcgen05.mma.cta_group::1.kind::f16 [%0], [%1+120], v7, %3, q;\n\t"
        "@pv tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"
        "@px tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t}"
        ::"r"(d_o), "r"(a_p), "l"(b_v), "r"(id_o), "r"(acc), "r"(bar_o), "r"(do_pv), "r"(bar_x), "r"(do_x),
          "n"(VS), "n"(2 * VS), "n"(3 * VS), "n"(4 * VS), "n"(5 * VS), "n"(6 * VS), "n"(7 * VS)
        : "memory");
    mma_s_batch_d<D>(d_s, a_q, b_k, id_s, do_s);
    tc_commit_if(bar_s, do_s);
}

struct DenseErr {
    static constexpr int kTimeout = 1;
};

// Warp roles of the CTA (12 warps, three warpgroups).  Two query tiles per
// work item (A: rows q0.., B: rows q0+128..) share every K/V tile.  Each query
// tile has one softmax warpgroup, a thread per query row over all 128 key
// columns:
//   warps 0-3 / 4-7     softmax of tile A / B
//   warp 8              MMA issue (one elected lane of the converged warp)
//   warp 9              TMA loads (one thread)
//   warps 10-11         idle (they complete the third warpgroup, whose
//                       registers move to the softmax warpgroups)
// The grid is persistent (one CTA per SM): each CTA walks work items (a pair
// of query tiles and a head); Q tiles are double-buffered and the K/V ring
// runs on across items, so the next item's loads and first products overlap
// the current item's last softmax and epilogue.
constexpr int kWarps = 12;
constexpr int kThreadsWS = kWarps * 32;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
// Register split (setmaxnreg): the CTA is launched with kRegsLaunch per
// thread; the third warpgroup gives registers up so that each softmax thread
// can hold a whole 128-key row of S.  The split must fit the launch's total.
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoftmax = 208;
constexpr int kRegsOther = 88;
static_assert(kRegsLaunch == 65536 / kThreadsWS / 8 * 8, "the launch bound gives each thread kRegsLaunch");
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsOther <= kRegsLaunch * kThreadsWS, "register split");
// A tile's P sum above this (or not finite) makes the softmax take the exact
// tile maximum and raise its running maximum (P <= 2^12 otherwise).
constexpr float kTileSumLimit = 4096.f;
constexpr int kMaxStages = 4;                     // K/V ring (Cfg<D>::kStages of them used)
constexpr uint32_t kTmemAll = 512;
// TMEM: three S/P buffers (128 columns each) used in rotation by the S tiles
// of the item's query tiles -- S number k (A0, B0, A1, B1, ... within the
// CTA's sequence) lives in buffer k % 3 and its P is written over it -- then
// O_A (and O_B), D columns each.
__host__ __device__ constexpr uint32_t col_buf(int b) { return 128u * static_cast<uint32_t>(b); }
template <int D>
__host__ __device__ constexpr uint32_t col_o(int g) { return 384u + static_cast<uint32_t>(g * D); }
static_assert(384 + 2 * 64 <= 512 && 384 + 2 * 32 <= 512 && 384 + 128 <= 512, "O fits beside the S/P buffers");
// (shared memory: Q buffers x query tiles at 0, then stage s: K at
// kSmemKV + 2 s kTB, V kTB after it)
static_assert((Cfg<64>::kSmemAlloc + 1024) >> 4 < (1u << 14) && (Cfg<128>::kSmemAlloc + 1024) >> 4 < (1u << 14),
              "descriptor start addresses fit 14 bits");
static_assert(Cfg<128>::kSmemAlloc <= 227 * 1024 - 512, "shared memory of the widest heads");
__device__ __forceinline__ int mod3(int x) { return x >= 3 ? x - 3 : x; }   // x < 6
template <int NS>
__device__ __forceinline__ int stage_add(int st, int k) { return (st + k) % NS; }

struct WsBars {
    uint64_t q_full[2], q_empty[2];   // Q buffers (TMA <-> MMA)
    uint64_t kv_full[kMaxStages];
    uint64_t kv_empty[kMaxStages];
    uint64_t s[2][2];    // S tile n of query tile g is in TMEM: barrier s[g][n & 1]
                         // (MMA -> softmax g; two barriers because an S tile
                         // can run two ahead of its softmax)
    uint64_t p[2][2];    // P_g number n written over its S: barrier p[g][n & 1], phase n >> 1
                         // (softmax g -> MMA), 4 warp arrivals.  Two barriers because
                         // the softmax may finish P_g(n+1) before the MMA warp has
                         // waited for P_g(n); P_g(n+2) needs S_g(n+2), which the MMA
                         // warp issues only after PV_g(n).
    uint64_t o[2][2];    // PV_g number n of the CTA is done: barrier o[g][n & 1], phase n >> 1
                         // (MMA -> softmax g, waited at a rescale and the epilogue)
    uint64_t o_free[2];  // softmax g has read O_g in its epilogue (-> MMA), 4 arrivals
    uint64_t drain;
    uint64_t stall;      // never completed: the softmax warps' first wait when a test asks for a stall
};

// Work item w -> (block row, block size, first query row, query tiles) and head.
__device__ __forceinline__ int4 item_of(const int4* items, int w, int H, int* head) {
    *head = w % H;
    return items[w / H];
}

__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\tmov.b64 rc, {%5, %5};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1) {   // d += a
    asm("{\n\t.reg .b64 ra, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rd, {%0, %1};\n\t"
        "add.rn.f32x2 rd, rd, ra;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// 4x4 transpose of 16-byte chunks over the four lanes of a quad: on entry
// lane l of the quad holds chunks 0-3 of its own row; on exit c[k] is chunk l
// of the quad's row k.  The quad then stores one row's four chunks per
// instruction (64 contiguous bytes) instead of four rows' single chunks.
__device__ __forceinline__ void quad_transpose(uint4 (&c)[4], int lane) {
    const bool b0 = lane & 1, b1 = (lane & 2) != 0;
    auto xchg = [](uint4 v, int m) {
        uint4 r;
        r.x = __shfl_xor_sync(0xffffffffu, v.x, m);
        r.y = __shfl_xor_sync(0xffffffffu, v.y, m);
        r.z = __shfl_xor_sync(0xffffffffu, v.z, m);
        r.w = __shfl_xor_sync(0xffffffffu, v.w, m);
        return r;
    };
#pragma unroll
    for (int q = 0; q < 4; q += 2) {   // across lane bit 0: positions (0,1) and (2,3)
        const uint4 r = xchg(b0 ? c[q] : c[q + 1], 1);
        if (b0) c[q] = r; else c[q + 1] = r;
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {      // across lane bit 1: positions (0,2) and (1,3)
        const uint4 r = xchg(b1 ? c[q] : c[q + 2], 2);
        if (b1) c[q] = r; else c[q + 2] = r;
    }
}
// One tile (128 rows of one head) by TMA: one box, or two 64-column boxes
// into the two sub-tiles (D = 128).
template <int D>
__device__ __forceinline__ void tma_tile(unsigned char* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    tma_load_2d(dst, map, x, y, bar);
    if constexpr (Cfg<D>::kSub == 2) tma_load_2d(dst + Cfg<D>::kTB / 2, map, x + 64, y, bar);
}

template <typename TO, int D>
__global__ void __launch_bounds__(kThreadsWS, 1)
k_dense_attn(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const int4* __restrict__ items, int n_work, int H,
             TO* __restrict__ out, int HD, float sl2, int* __restrict__ err, long long wait_limit, int test_stall) {
    using C = Cfg<D>;
    constexpr uint32_t kTileBytes = C::kTB;
    constexpr int kStages = C::kStages;
    constexpr int kQB = C::kQBufs;
    constexpr int kNqMax = C::kNq;
    constexpr uint64_t kStageUnits = C::kStageUnits;
    constexpr uint64_t kQUnits = C::kQUnits;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) WsBars bars;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    auto sQ = [&](int buf, int g) { return smem + C::kSmemQ + (kNqMax * buf + g) * kTileBytes; };
    auto sK = [&](int st) { return smem + C::kSmemKV + st * 2 * kTileBytes; };
    auto sV = [&](int st) { return smem + C::kSmemKV + st * 2 * kTileBytes + kTileBytes; };

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&s_tmem)),
                     "r"(kTmemAll)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        s_abort = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.q_full[b], 1);
            mbar_init(&bars.q_empty[b], 1);
        }
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bars.kv_full[i], 1);
            mbar_init(&bars.kv_empty[i], 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(&bars.s[g][0], 1);
            mbar_init(&bars.s[g][1], 1);
            mbar_init(&bars.p[g][0], 4);
            mbar_init(&bars.p[g][1], 4);
            mbar_init(&bars.o[g][0], 1);
            mbar_init(&bars.o[g][1], 1);
            mbar_init(&bars.o_free[g], 4);
        }
        mbar_init(&bars.drain, 1);
        mbar_init(&bars.stall, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    // The register change is made at the head of each warpgroup's branch, by
    // all four of its warps at the same instruction.
    if (warp >= kMmaWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
    if (warp == kTmaWarp) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            bool ok = true;
            int kv_tile = 0;   // running K/V tile counter over all items of this CTA
            int local = 0;
            int h_next = 0;
            int4 it_next = blockIdx.x < n_work ? item_of(items, blockIdx.x, H, &h_next) : make_int4(0, 0, 0, 0);
            for (int w = blockIdx.x; ok && w < n_work; w += gridDim.x, ++local) {
                const int h = h_next;
                const int4 it = it_next;   // the next item's entry is loaded one item ahead
                if (w + gridDim.x < n_work) it_next = item_of(items, w + gridDim.x, H, &h_next);
                const int r0 = it.x, n = it.y, q0 = it.z, nq = it.w, T = (n + kTile - 1) / kTile, xh = h * D;
                const int qb = local % kQB;
                if (local >= kQB) ok = mbar_wait(&bars.q_empty[qb], ((local / kQB) - 1) & 1, wait_limit);
                if (!ok) break;
                mbar_expect_tx(&bars.q_full[qb], nq * kTileBytes);
                for (int g = 0; g < nq; ++g) tma_tile<D>(sQ(qb, g), &tmQ, xh, q0 + g * kTile, &bars.q_full[qb]);
                for (int j = 0; j < T; ++j, ++kv_tile) {
                    const int st = kv_tile % kStages;
                    if (kv_tile >= kStages) ok = mbar_wait(&bars.kv_empty[st], ((kv_tile / kStages) - 1) & 1, wait_limit);
                    if (!ok) break;
                    mbar_expect_tx(&bars.kv_full[st], 2 * kTileBytes);
                    tma_tile<D>(sK(st), &tmK, xh, r0 + j * kTile, &bars.kv_full[st]);
                    tma_tile<D>(sV(st), &tmV, xh, r0 + j * kTile, &bars.kv_full[st]);
                }
            }
            if (!ok) {
                atomicOr(err, DenseErr::kTimeout);
                atomicExch(&s_abort, 1);
                // drain this thread's copies in flight (bounded): the last use
                // of every stage and of both Q buffers
                for (int st = 0; st < kStages; ++st) {
                    const int uses = kv_tile / kStages + (st < kv_tile % kStages ? 1 : 0);
                    if (uses > 0) mbar_wait(&bars.kv_full[st], (uses - 1) & 1, kWaitCycles / 4);
                }
                for (int b = 0; b < kQB; ++b) {
                    const int uses = (local + kQB - 1 - b) / kQB;
                    if (uses > 0) mbar_wait(&bars.q_full[b], (uses - 1) & 1, kWaitCycles / 4);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        // Order per item (two query tiles): S_A0 S_B0 S_A1, then per key tile j
        // two asm blocks: [PV_Aj, S_B(j+1)] and [PV_Bj, S_A(j+2)].  An S tile is
        // computed one step ahead of its softmax; a buffer is reused only after
        // the PV that read its P (the tensor pipe executes one thread's MMAs in
        // issue order).  The whole warp runs this loop; elect.sync picks the
        // same lane (the lowest) for every batch and commit, so one thread
        // issues them all.  The tensor pipe queues only a few MMAs ahead, so
        // every gap between asm blocks risks leaving it idle: each half step
        // is one block, and the barrier states needed after a block are probed
        // before it (non-blocking) and read after it.
        {
            const uint32_t idS = idesc_bf16(128, 128, 0);
            const uint32_t idO = idesc_bf16(128, D, 1);
            const uint64_t dQ0 = desc_kmajor<D>(su32(sQ(0, 0)));
            const uint64_t dK0 = desc_kmajor<D>(su32(sK(0)));
            const uint64_t dV0 = desc_mnmajor<D>(su32(sV(0)));
            bool ok = true;
            int kv_tile = 0;   // first K/V tile of the current item in the CTA's sequence
            int snum = 0;      // S tiles issued so far (buffer = snum % 3)
            int sg0 = 0, sg1 = 0;   // S tiles issued per query tile (barrier s[g][n & 1])
            int p_cnt0 = 0, p_cnt1 = 0, items0 = 0, items1 = 0;
            int pv0 = 0, pv1 = 0;   // products issued per query tile (barrier o[g][n & 1])
            int local = 0;
            for (int w = blockIdx.x; ok && w < n_work; w += gridDim.x, ++local) {
                int h;
                const int4 it = item_of(items, w, H, &h);
                const int nq = it.w, T = (it.y + kTile - 1) / kTile;
                const int qb = local % kQB;
                const int s0 = snum;   // S number of (g, j) = s0 + nq*j + g
                auto bufk = [&](int g, int j) { return (s0 + nq * j + g) % 3; };
                // S_g(j); the K tile's readiness was established before
                auto issue_s = [&](int g, int j) {
                    const int kt = kv_tile + j;
                    const uint64_t dQ = desc_kmajor<D>(su32(sQ(qb, g)));
                    const uint64_t dK = desc_kmajor<D>(su32(sK(kt % kStages)));
                    if constexpr (D == 64) mma_s_batch(tmem + col_buf(bufk(g, j)), dQ, dK, idS);
                    else mma_s_batch_d<D>(tmem + col_buf(bufk(g, j)), dQ, dK, idS, 1u);
                    int& sn = g == 0 ? sg0 : sg1;
                    tc_commit(&bars.s[g][sn & 1]);
                    ++sn;
                    ++snum;
                };
                auto kv_probe = [&](int j) {
                    const int kt = kv_tile + j;
                    return mbar_probe(&bars.kv_full[kt % kStages], (kt / kStages) & 1);
                };
                auto kv_wait = [&](int j, uint32_t probed) {
                    const int kt = kv_tile + j;
                    if (warp_any_ordered(probed)) return true;
                    return mbar_wait_warp(&bars.kv_full[kt % kStages], (kt / kStages) & 1, wait_limit);
                };
                auto p_probe = [&](int g) {
                    const int pc = g == 0 ? p_cnt0 : p_cnt1;
                    return mbar_probe(&bars.p[g][pc & 1], (pc >> 1) & 1);
                };
                // P_g(j) written (probe answer `probed`, else a blocking wait)
                auto p_wait = [&](int g, uint32_t probed) {
                    int& pc = g == 0 ? p_cnt0 : p_cnt1;
                    const bool r =
                        warp_any_ordered(probed) || mbar_wait_warp(&bars.p[g][pc & 1], (pc >> 1) & 1, wait_limit);
                    ++pc;
                    return r;
                };
                ok = mbar_wait_warp(&bars.q_full[qb], (local / kQB) & 1, wait_limit);
                if (!ok) break;
                // S tiles ahead of the loop: A0 (B0) and A1
                ok = kv_wait(0, 0u);
                if (ok) {
                    tc_fence_after();
                    for (int g = 0; g < nq; ++g) issue_s(g, 0);
                }
                if (ok && T > 1) {
                    ok = kv_wait(1, 0u);
                    tc_fence_after();
                    if (ok) issue_s(0, 1);
                }
                // descriptors: the bases plus a stage's or a Q buffer's offset
                // (the start address field is linear in the byte address)
                const uint64_t dQa = dQ0 + static_cast<uint64_t>(kNqMax * qb) * kQUnits, dQb = dQa + kQUnits;
                int st = kv_tile % kStages;   // stage of K_j, V_j
                int bA = s0 % 3;                    // buffer of S_A(j); S_B(j) is in the next one
                uint32_t pa = p_probe(0);
                for (int j = 0; ok && j < T; ++j, st = stage_add<kStages>(st, 1), bA = mod3(bA + nq)) {
                    // the first product of an item overwrites O_g: the previous
                    // item's epilogue must have read it
                    ok = p_wait(0, pa);
                    if (ok && j == 0 && items0 > 0) ok = mbar_wait_warp(&bars.o_free[0], (items0 - 1) & 1, wait_limit);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t pb = nq > 1 ? p_probe(1) : 0u;
                    const uint32_t kv = j + 2 < T ? kv_probe(j + 2) : 0u;
                    const uint64_t dVj = dV0 + static_cast<uint64_t>(st) * kStageUnits;
                    {   // PV_A(j), then S_B(j+1) into the buffer PV_A(j) has just read
                        const bool sb = nq > 1 && j + 1 < T;
                        const uint64_t dKn = dK0 + static_cast<uint64_t>(stage_add<kStages>(st, 1)) * kStageUnits;
                        if constexpr (D == 64)
                            mma_half_step(tmem + col_o<D>(0), tmem + col_buf(bA), dVj, idO, j > 0 ? 1u : 0u,
                                          su32(&bars.o[0][pv0 & 1]), 1u, 0u, 0u, tmem + col_buf(bA), dQb, dKn, idS,
                                          su32(&bars.s[1][sg1 & 1]), sb ? 1u : 0u);
                        else
                            mma_half_step_d<D>(tmem + col_o<D>(0), tmem + col_buf(bA), dVj, idO, j > 0 ? 1u : 0u,
                                               su32(&bars.o[0][pv0 & 1]), 1u, 0u, 0u, tmem + col_buf(bA), dQb, dKn,
                                               idS, su32(&bars.s[1][sg1 & 1]), sb ? 1u : 0u);
                        ++pv0;
                        if (sb) { ++sg1; ++snum; }
                    }
                    if (j + 2 < T) ok = kv_wait(j + 2, kv);
                    if (ok && nq > 1) {
                        ok = p_wait(1, pb);
                        if (ok && j == 0 && items1 > 0)
                            ok = mbar_wait_warp(&bars.o_free[1], (items1 - 1) & 1, wait_limit);
                    }
                    if (!ok) break;
                    tc_fence_after();
                    pa = p_probe(0);
                    {   // PV_B(j); K_j, V_j free once it (and PV_A(j)) are done; S_A(j+2)
                        // into the buffer of S_B(j) (one query tile: of S_A(j+1)'s successor)
                        const bool sa = j + 2 < T;
                        const int bS = (bA + 2 * nq) % 3;
                        const uint64_t dKn = dK0 + static_cast<uint64_t>(stage_add<kStages>(st, 2)) * kStageUnits;
                        // (O_B's columns exist only when an item holds two query tiles)
                        const uint32_t dOb = tmem + col_o<D>(kNqMax > 1 ? 1 : 0);
                        if constexpr (D == 64)
                            mma_half_step(dOb, tmem + col_buf(mod3(bA + 1)), dVj, idO, j > 0 ? 1u : 0u,
                                          su32(&bars.o[1][pv1 & 1]), nq > 1 ? 1u : 0u, su32(&bars.kv_empty[st]), 1u,
                                          tmem + col_buf(bS), dQa, dKn, idS, su32(&bars.s[0][sg0 & 1]), sa ? 1u : 0u);
                        else
                            mma_half_step_d<D>(dOb, tmem + col_buf(mod3(bA + 1)), dVj, idO, j > 0 ? 1u : 0u,
                                               su32(&bars.o[1][pv1 & 1]), nq > 1 ? 1u : 0u,
                                               su32(&bars.kv_empty[st]), 1u, tmem + col_buf(bS), dQa, dKn, idS,
                                               su32(&bars.s[0][sg0 & 1]), sa ? 1u : 0u);
                        if (nq > 1) ++pv1;
                        if (sa) { ++sg0; ++snum; }
                    }
                }
                if (ok) tc_commit(&bars.q_empty[qb]);        // Q buffer free after this item's products
                ++items0;
                if (nq > 1) ++items1;
                kv_tile += T;
            }
            if (!ok && lane == 0) {
                atomicOr(err, DenseErr::kTimeout);
                atomicExch(&s_abort, 1);
            }
            // drain: everything the elected lane issued has finished before TMEM is freed
            tc_commit(&bars.drain);
            mbar_wait_warp(&bars.drain, 0, kWaitCycles / 4);
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ---------------- softmax warpgroups ----------------
        // One thread per query row (= TMEM lane) and all 128 key columns of a
        // tile: a row's running maximum and sum live in one thread, so the
        // warps of a tile never exchange data and never wait for each other.
        const int g = warp >> 2;                       // query tile
        const int row = (warp & 3) * 32 + lane;        // row of the query tile (= TMEM lane)
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tO = tmem + col_o<D>(g) + lane_base;
        const bool pos = sl2 >= 0.f;
        int s_cnt = 0;      // S tiles of this query tile consumed so far
        int o_cnt = 0;      // PV_g products of finished items
        // Wait for PV_g number n.  Two barriers keep each wait inside the
        // barrier's two-phase window without confirming every product: when
        // the softmax waits for PV_g(n) it has seen S_g complete for a tile
        // whose S was issued after PV_g(n-2) (S_g(j) follows PV_g(j-2) in the
        // MMA order, and the S commit tracks every earlier MMA), so the
        // previous phase of barrier o[g][n & 1] has completed.
        auto o_wait = [&](int n) { return mbar_wait(&bars.o[g][n & 1], (n >> 1) & 1, wait_limit); };
        int snum = 0;   // S tiles of the CTA's sequence before the current item (both query tiles)
        bool failed = false;
        if (test_stall) {
            // tests of the bounded-wait path: a wait on a barrier nothing
            // completes runs out, the CTA is marked aborted, the other warps'
            // waits for this warpgroup's P run out in turn and every role drains
            if (!mbar_wait(&bars.stall, 0, wait_limit)) atomicExch(&s_abort, 1);
            failed = true;
        }
        int h_next = 0;
        int4 it_next = blockIdx.x < n_work ? item_of(items, blockIdx.x, H, &h_next) : make_int4(0, 0, 0, 0);
        for (int w = blockIdx.x; !failed && w < n_work; w += gridDim.x) {
            const int h = h_next;
            const int4 it = it_next;   // the next item's entry is loaded one item ahead
            if (w + gridDim.x < n_work) it_next = item_of(items, w + gridDim.x, H, &h_next);
            const int r0 = it.x, n = it.y, q0 = it.z, nq = it.w, T = (n + kTile - 1) / kTile, xh = h * D;
            const int s0 = snum;
            snum += nq * T;
            if (g >= nq) continue;
            float m_used = -INFINITY, l0 = 0.f, l1 = 0.f;
            for (int j = 0; j < T; ++j) {
                const uint32_t tS = tmem + col_buf((s0 + nq * j + g) % 3) + lane_base;
                // a wait that runs out marks the CTA aborted; the warp leaves
                // its loop (the decision is uniform over the warp)
                const bool bad = !mbar_wait(&bars.s[g][s_cnt & 1], (s_cnt >> 1) & 1, wait_limit);
                ++s_cnt;
                if (bad) atomicExch(&s_abort, 1);
                if (__any_sync(0xffffffffu, bad || *reinterpret_cast<volatile int*>(&s_abort) != 0)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                // the tile's S row, read once: the P pass and (rarely) the
                // maximum work from registers
                uint32_t r[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, r + 32 * c);
                tmem_ld_wait();
                // a block of n keys ends inside its last key tile: the columns
                // past it (another block's keys) become -inf logits (+inf for a
                // negative scale), so their P is 0 and they never set the maximum
                const int n_last = n - (T - 1) * kTile;
                if (j == T - 1 && n_last < kTile) {
                    const uint32_t masked = __float_as_uint(pos ? -INFINITY : INFINITY);
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= n_last) r[c] = masked;
                }
                // the row's largest t = s*scale*log2e over the tile (from its
                // largest s for a positive scale, its smallest for a negative one)
                auto tile_top = [&]() {
                    float ma, mb, mc, md;
                    ma = mb = mc = md = pos ? -INFINITY : INFINITY;
                    if (pos) {
#pragma unroll
                        for (int i = 0; i < 128; i += 8) {
                            ma = max3(ma, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                            mb = max3(mb, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                            mc = max3(mc, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
                            md = max3(md, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
                        }
                        ma = fmaxf(fmaxf(ma, mb), fmaxf(mc, md));
                    } else {
#pragma unroll
                        for (int i = 0; i < 128; i += 8) {
                            ma = min3(ma, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                            mb = min3(mb, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                            mc = min3(mc, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
                            md = min3(md, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
                        }
                        ma = fminf(fminf(ma, mb), fminf(mc, md));
                    }
                    return ma * sl2;
                };
                // P = 2^(t - m) as bf16 hi/lo written over S, 32 keys at a time;
                // (la, lb) = the tile's sum of P
                float la = 0.f, lb = 0.f;
                auto write_p = [&]() {
                    const float nm = -m_used;
                    la = lb = 0.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t* x = r + 32 * c;
                        uint32_t pk[32];
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            float t0, t1;
                            ffma2(t0, t1, __uint_as_float(x[2 * q]), __uint_as_float(x[2 * q + 1]), sl2, nm);
                            const float p0 = ex2(t0), p1 = ex2(t1);
                            fadd2(la, lb, p0, p1);
                            const uint32_t hi = pack2_bf16(p0, p1);
                            // P_lo = bf16(P - P_hi): the differences, exact in fp32, come
                            // from mixed bf16 x bf16 + fp32 FMAs on the packed P_hi halves
                            // (times -1) -- no unpacking of P_hi
                            float d0, d1;
                            asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
                                "fma.rn.f32.bf16 %0, h0, %5, %3;\n\tfma.rn.f32.bf16 %1, h1, %5, %4;\n\t}"
                                : "=f"(d0), "=f"(d1) : "r"(hi), "f"(p0), "f"(p1), "h"((unsigned short)0xBF80));
                            pk[q] = hi;
                            pk[16 + q] = pack2_bf16(d0, d1);
                        }
                        // keys 32c..32c+31: P_hi in columns 32c..32c+15, P_lo in 32c+16..32c+31
                        tmem_st32(tS + 32 * c, pk);
                    }
                };
                // The first tile sets the running maximum m; later tiles use it
                // as it stands, unless a row's tile sum exceeds kTileSumLimit
                // (some P above the limit, or not finite): that row takes the
                // exact maximum of the tile, O_g and its sum are rescaled, and
                // the warp writes the tile's P again.
                if (j == 0) m_used = tile_top();
                write_p();
                if (j > 0) {
                    const bool over = !(la + lb <= kTileSumLimit);
                    if (__any_sync(0xffffffffu, over)) {
                        // O_g may be rescaled only after PV_g(j-1); no later PV_g
                        // can have been issued (it needs this tile's P)
                        if (!o_wait(o_cnt + j - 1)) atomicExch(&s_abort, 1);
                        tc_fence_after();
                        float alpha = 1.f;
                        if (over) {
                            const float mt = fmaxf(tile_top(), m_used);
                            alpha = ex2(m_used - mt);
                            m_used = mt;
                        }
                        l0 *= alpha;
                        l1 *= alpha;
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(tO + 32 * c, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(tO + 32 * c, o);
                        }
                        tmem_st_wait();
                        write_p();
                    }
                }
                l0 += la;
                l1 += lb;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.p[g][(o_cnt + j) & 1]);
            }
            if (failed) break;
            // epilogue: O_g after the item's last product
            const bool bad = !o_wait(o_cnt + T - 1);
            o_cnt += T;
            if (bad) atomicExch(&s_abort, 1);
            if (__any_sync(0xffffffffu, bad)) { failed = true; break; }
            tc_fence_after();
            uint32_t o[D];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + 32 * c, o + 32 * c);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.o_free[g]);
            const float inv = 1.f / (l0 + l1);
            // rows of this lane's quad after each transpose: quad base + k
            // (rows past the block's end, in a ragged last query tile, are
            // computed but not stored)
            const int qrow = q0 + g * kTile + (row & ~3);
            TO* op = out + static_cast<int64_t>(qrow) * HD + xh;
            const int ql = lane & 3;
            const int rows_left = r0 + n - qrow;   // rows k < rows_left of the quad are the block's
            if constexpr (sizeof(TO) == 2) {
#pragma unroll
                for (int gg = 0; gg < D / 32; ++gg) {   // 16-byte chunks 4gg..4gg+3 (columns 32gg..32gg+31)
                    uint4 c[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int e = 32 * gg + 8 * v;
                        c[v] = make_uint4(
                            pack2_bf16(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv),
                            pack2_bf16(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                            pack2_bf16(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                            pack2_bf16(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
                    }
                    quad_transpose(c, lane);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (k < rows_left) reinterpret_cast<uint4*>(op + static_cast<int64_t>(k) * HD)[4 * gg + ql] = c[k];
                }
            } else {
#pragma unroll
                for (int gg = 0; gg < D / 16; ++gg) {   // 16-byte chunks 4gg..4gg+3 (columns 16gg..16gg+15)
                    uint4 c[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int e = 16 * gg + 4 * v;
                        c[v] = make_uint4(__float_as_uint(__uint_as_float(o[e]) * inv),
                                          __float_as_uint(__uint_as_float(o[e + 1]) * inv),
                                          __float_as_uint(__uint_as_float(o[e + 2]) * inv),
                                          __float_as_uint(__uint_as_float(o[e + 3]) * inv));
                    }
                    quad_transpose(c, lane);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (k < rows_left) reinterpret_cast<uint4*>(op + static_cast<int64_t>(k) * HD)[4 * gg + ql] = c[k];
                }
            }
        }
        if (failed) {
            atomicOr(err, DenseErr::kTimeout);
            atomicExch(&s_abort, 1);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemAll) : "memory");
    }
}

// ---- host ------------------------------------------------------------------
// [N, HD] bf16 matrix, boxes of 128 rows: one head of 32 columns with the
// 64-byte swizzle, or 64 columns (a whole head of 64, half of one of 128)
// with the 128-byte swizzle.
template <int D>
bool make_map(CUtensorMap* m, const void* base, int64_t N, int HD) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(HD) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(Cfg<D>::kBoxX), kTile};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The register split of the kernel (setmaxnreg) waits until the registers it
// asks for are free; it is only valid when the CTA was launched with
// kRegsLaunch registers per thread.  Checked once per kernel instance.
template <typename K>
bool regs_fit(K kernel) {
    static std::once_flag once;
    static bool fit = false;
    std::call_once(once, [&] {
        cudaFuncAttributes a{};
        fit = cudaFuncGetAttributes(&a, kernel) == cudaSuccess && a.numRegs == kRegsLaunch &&
              a.maxThreadsPerBlock >= kThreadsWS;
    });
    return fit;
}

}  // namespace

bool dense_supported(int H, int D, gtattn_dtype dt, const void* Q, const void* K, const void* V,
                     const void* out) {
    if (dt != GTATTN_BF16 && dt != GTATTN_BF16_OUT_F32) return false;
    if ((D != 32 && D != 64 && D != 128) || H < 1 || H * D > kMaxHD) return false;
    const uintptr_t al = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                         reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(out);
    if (al & 15u) return false;
    return encode_fn() != nullptr;
}

template <int D>
static gtattn_status launch_dense_d(const int4* tiles, int n_tiles, int64_t N, const void* Q, const void* K,
                                    const void* V, void* out, int H, float scale, gtattn_dtype dt, int* err,
                                    long long wait_limit, int test_stall, cudaStream_t s) {
    const int HD = H * D;
    CUtensorMap mq, mk, mv;
    if (!make_map<D>(&mq, Q, N, HD) || !make_map<D>(&mk, K, N, HD) || !make_map<D>(&mv, V, N, HD))
        return GTATTN_ERR_UNSUPPORTED;
    const float sl2 = scale * kLog2e;
    const int n_work = n_tiles * H;
    const int grid = std::min(n_work, num_sms());
    constexpr int smem = static_cast<int>(Cfg<D>::kSmemAlloc);
    auto go = [&](auto k, auto* o) {
        if (!regs_fit(k)) return GTATTN_ERR_UNSUPPORTED;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess) {
            k<<<grid, kThreadsWS, smem, s>>>(mq, mk, mv, tiles, n_work, H, o, HD, sl2, err, wait_limit, test_stall);
            e = cudaGetLastError();
        }
        return e == cudaSuccess ? GTATTN_OK : cuda_status(e);
    };
    if (dt == GTATTN_BF16) return go(k_dense_attn<__nv_bfloat16, D>, static_cast<__nv_bfloat16*>(out));
    return go(k_dense_attn<float, D>, static_cast<float*>(out));
}

gtattn_status launch_dense(const int4* tiles, const int4* tiles1, int n_tiles, int n_tiles1, int64_t N,
                           const void* Q, const void* K, const void* V, void* out, int H, int D, float scale,
                           gtattn_dtype dt, int* err, long long wait_cycles, int test_stall, cudaStream_t s) {
    const long long wait_limit = wait_cycles > 0 ? wait_cycles : kWaitCycles;
    switch (D) {
        case 32:
            if (n_tiles <= 0) return GTATTN_OK;
            return launch_dense_d<32>(tiles, n_tiles, N, Q, K, V, out, H, scale, dt, err, wait_limit, test_stall, s);
        case 64:
            if (n_tiles <= 0) return GTATTN_OK;
            return launch_dense_d<64>(tiles, n_tiles, N, Q, K, V, out, H, scale, dt, err, wait_limit, test_stall, s);
        case 128:   // one query tile per work item
            if (n_tiles1 <= 0) return GTATTN_OK;
            return launch_dense_d<128>(tiles1, n_tiles1, N, Q, K, V, out, H, scale, dt, err, wait_limit, test_stall,
                                       s);
    }
    return GTATTN_ERR_UNSUPPORTED;
}

}  // namespace gt
