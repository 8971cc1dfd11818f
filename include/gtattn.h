/*
 * gtattn.h -- C ABI of the GB300 sparse multi-head attention library.
 *
 * The operation (per CSR row i and head h):
 *
 *   out[i,h,:] = sum_{e in row i} p[e,h] * V[indices[e],h,:]
 *   p[e,h]     = exp(l[e,h]) / sum_{e' in row i} exp(l[e',h])
 *   l[e,h]     = scale * <Q[i,h,:], K[indices[e],h,:]>
 *
 * i.e. SparseAttn(Q, K, V, A) = softmax((Q K^T) o A / sqrt(d)) V from
 * "Graph Transformer in a Nutshell" (section "Sparse Multi-head Attention",
 * equation SparseAttn and SparseMHA.forward: bsddmm, sparse softmax over the
 * last sparse dimension, bspmm), in the destination-row orientation of
 * "Efficient Sparse Transformer implementation with DGL's builtin
 * operators" (TransLayer.forward: u_dot_v, edge_softmax of e/sqrt(d_qkv),
 * u_mul_e_sum).  The softmax runs over the row's stored entries only
 * (non-edges are excluded, as b_inf = -inf excludes disconnected pairs in
 * "Graph Transformer theory, derivation and implementation", shortest-path
 * bias section).  A row with no entries yields zeros.  Every CSR entry is
 * one edge (duplicates weigh twice).  There is no dropout.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Graph:     CSR by destination.  indptr: int32 [N+1], indptr[0] = 0,
 *            non-decreasing, indptr[N] = nnz.  indices: int32 [nnz], each in
 *            [0, N): row i attends over nodes indices[indptr[i]..indptr[i+1]).
 *            N < 2^31, nnz < 2^31.
 * Features:  Q, K, V, out: [N, H, D] row-major, D innermost, of the types
 *            `dtype` names (fp32, or bf16 as raw 16-bit patterns).  Accumulation
 *            is fp32; a bf16 `out` is rounded to nearest-even.  1 <= H, 1 <= D,
 *            H*D <= 1024.  Pointers must be aligned to their element size.
 *            `out` must not overlap Q, K or V.
 * Memory:    every pointer argument is a DEVICE pointer (cudaMalloc'd or
 *            managed memory) owned by the caller unless noted; the library
 *            never frees caller memory.  Library temporaries come from a
 *            library-owned stream-ordered memory pool (cudaMallocAsync).
 * Streams:   work is enqueued on `stream` (0 = legacy default stream) and the
 *            call returns once it is enqueued, except where noted.
 * Errors:    every call returns a gtattn_status; nothing throws across the
 *            ABI.  Argument checks run on the host before any launch.  CSR
 *            contents are NOT checked on the fast path (use
 *            gtattn_csr_validate); an invalid CSR gives undefined results.
 *            The checking build of the library (compiled with GTATTN_DEBUG:
 *            lib/libgtattn_debug.so) validates the CSR of every call that
 *            takes one on the device first (gtattn_fwd_host: on the host),
 *            synchronously, and returns GTATTN_ERR_BAD_CSR without running
 *            anything else; its one device flag is shared, so calls of the
 *            checking build must not overlap, and it cannot be captured in
 *            a CUDA graph.
 *            GTATTN_ERR_CUDA reports a CUDA runtime error (the last CUDA
 *            error string is available from gtattn_last_error).
 * Threads:   entry points are thread-safe, except that one plan must not be
 *            used by two calls that may run concurrently (it owns a workspace).
 */
#ifndef GTATTN_H
#define GTATTN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GTATTN_OK = 0,
    GTATTN_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misaligned pointer ... */
    GTATTN_ERR_BAD_CSR = 2,       /* gtattn_csr_validate found a malformed CSR */
    GTATTN_ERR_UNSUPPORTED = 3,   /* valid request outside what this build implements */
    GTATTN_ERR_CUDA = 4,          /* a CUDA runtime call failed */
    GTATTN_ERR_NO_MEMORY = 5,     /* a device or host allocation failed */
    GTATTN_ERR_TIMEOUT = 6        /* a bounded device-side wait gave up */
} gtattn_status;

/* Element types: Q, K, V and out share the type, except GTATTN_BF16_OUT_F32
 * (bf16 Q, K, V; fp32 out: the accumulator without the final rounding). */
typedef enum { GTATTN_F32 = 0, GTATTN_BF16 = 1, GTATTN_BF16_OUT_F32 = 2 } gtattn_dtype;

/* Which row kernel a plan uses (tests force each one; AUTO picks the fastest
 * that supports the shape). */
typedef enum {
    GTATTN_KERNEL_AUTO = 0,
    GTATTN_KERNEL_VECTOR = 1,   /* 16-byte gathers, lanes split a feature row */
    GTATTN_KERNEL_GENERIC = 2,  /* any H, D; one warp per row */
    GTATTN_KERNEL_NARROW = 3    /* D <= 16, H <= 32: one lane per head (the fused
                                   forward; the unfused variants run the
                                   generic kernel) */
} gtattn_kernel;

/* Plan-building options.  Zero-initialise and set what you need; a field
 * left at 0 takes its default. */
typedef struct {
    int32_t long_row_min;   /* rows with more entries than this are split into
                               chunks (default 1024; -1: split every non-empty row) */
    int32_t chunk_edges;    /* entries per chunk of a split row (default 1024) */
    int32_t detect_dense;   /* 1: find complete blocks for the dense tensor-core path */
    int32_t kernel;         /* a gtattn_kernel value */
    int32_t wait_cycles;    /* bound of each device-side wait of the dense-block
                               kernel for another warp's data, in SM clock cycles
                               (0: about one second).  A wait that runs out makes
                               the kernel drain what it issued, record
                               device_error and return. */
    int32_t test_stall;     /* tests of that path only: 1 makes the dense-block
                               kernel wait first on a barrier that nothing
                               completes, so every wait runs out and the call's
                               output is not valid */
} gtattn_plan_opts;

/* What a plan found (host copy). */
typedef struct {
    int64_t N, nnz;
    int32_t n_long_rows;     /* rows split into chunks */
    int32_t n_chunks;        /* chunks over all split rows */
    int32_t n_dense_blocks;  /* complete blocks found (detect_dense) */
    int32_t n_dense_rows;    /* rows inside those blocks */
    int32_t n_empty_rows;    /* rows with no entries */
    int32_t max_degree;
    int32_t n_buckets;       /* entries of bucket_rows used */
    int32_t bucket_rows[64]; /* rows per degree bucket (bucket b < 33: degree b) */
    int32_t device_error;    /* nonzero if a bounded device wait of a forward
                                call with this plan gave up since the last
                                gtattn_plan_get_info (1: timeout; the output of
                                that call is not valid) */
} gtattn_plan_info;

typedef struct gtattn_plan gtattn_plan;   /* opaque, library-owned */

/* Human-readable name of a status code (static string). */
const char* gtattn_status_string(gtattn_status s);

/* Text of the last CUDA error seen by this thread ("" if none). */
const char* gtattn_last_error(void);

/*
 * gtattn_csr_build -- degree binning of a CSR graph (the plan).
 * Sorts rows into degree buckets, lists split chunks for long rows and, with
 * opts->detect_dense, finds complete blocks (rows r0..r0+n-1 whose entries are
 * exactly r0..r0+n-1 in order, n >= 128).  Binning is this
 * library's design; the pages define only the operation.
 *   indptr, indices: device CSR as above (not copied: the same arrays must be
 *   passed to the forward calls that use the plan).
 *   opts: may be NULL for defaults.
 *   plan_out: receives a new plan; free it with gtattn_plan_destroy.
 * Synchronises `stream` once (to size the plan).  Errors: INVALID_ARG,
 * NO_MEMORY, CUDA.
 */
gtattn_status gtattn_csr_build(const int32_t* indptr, const int32_t* indices, int64_t N,
                               int64_t nnz, const gtattn_plan_opts* opts,
                               gtattn_plan** plan_out, cudaStream_t stream);

/* Frees a plan (after synchronising the device work that may still use it).
 * NULL is accepted. */
gtattn_status gtattn_plan_destroy(gtattn_plan* plan);

/* Copies the plan's counts to *info (host).  Reads and clears the plan's
 * device error word, so it waits for work already queued that uses the plan. */
gtattn_status gtattn_plan_get_info(const gtattn_plan* plan, gtattn_plan_info* info);

/*
 * gtattn_fwd -- fused sparse MHA forward, no plan: bins the rows on the fly
 * on `stream` (stream-ordered temporaries, no host synchronisation), then
 * runs the fused single-pass row kernels and the split-row combine.  No
 * dense-block path.  Operation and conventions: see the top of this file.
 *   scale: multiplies q.k (normally 1/sqrt(D)).
 * Errors: INVALID_ARG (null pointer with N > 0 / nnz > 0, N or nnz negative
 * or >= 2^31, H or D < 1, H*D > 1024, bad dtype, misaligned pointer),
 * NO_MEMORY, CUDA.
 */
gtattn_status gtattn_fwd(const int32_t* indptr, const int32_t* indices, const void* Q,
                         const void* K, const void* V, void* out, int64_t N, int64_t nnz,
                         int H, int D, float scale, gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_fwd_host -- gtattn_fwd on HOST buffers: the same operation, with
 * the graph and features copied to the device and the output copied back
 * inside the call, all ordered on `stream`.  The copies overlap the
 * computation: K and V are copied first, then the rows are cut into chunks
 * of about equal work whose indptr, indices and Q are copied while earlier
 * chunks are computed, and whose output rows are copied back while later
 * chunks are copied and computed (two library-owned copy streams per device).
 * The pages define no host-buffer call: this one is a convenience of this
 * library for callers whose data lives in host memory.
 *   indptr, indices, Q, K, V: host memory, same layouts as gtattn_fwd; out:
 *   host memory, written when `stream` reaches the end of the call.  Host
 *   buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for the
 *   copies to be asynchronous and at full speed; the caller keeps every host
 *   buffer valid and unchanged until `stream` has passed the call.  indptr is
 *   also read by the host during the call (chunk boundaries).
 *   Device temporaries (about the size of the inputs plus the output) come
 *   from the library's stream-ordered pool and return to it at the end.
 * Errors: those of gtattn_fwd; BAD_CSR when indptr[0] != 0 or
 * indptr[N] != nnz.
 */
gtattn_status gtattn_fwd_host(const int32_t* indptr, const int32_t* indices, const void* Q,
                              const void* K, const void* V, void* out, int64_t N, int64_t nnz,
                              int H, int D, float scale, gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_fwd_ndh -- gtattn_fwd on head-innermost node rows: Q, K, V and out
 * are [N, D, H] (element (h, d) of row i at i*H*D + d*H + h), the layout the
 * SparseMHA of "Graph Transformer in a Nutshell" reshapes its projections to
 * (q.reshape(N, head_dim, num_heads)), so such callers need no transpose.
 * Same arguments, results (up to rounding order) and errors as gtattn_fwd;
 * runs the generic row kernel.
 */
gtattn_status gtattn_fwd_ndh(const int32_t* indptr, const int32_t* indices, const void* Q,
                             const void* K, const void* V, void* out, int64_t N, int64_t nnz,
                             int H, int D, float scale, gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_fwd_plan -- as gtattn_fwd with a prebuilt plan: no binning per
 * call, and complete blocks (if the plan found any) go to the dense
 * tensor-core kernel when dtype is bf16 (or bf16 in, fp32 out), D is 32, 64
 * or 128 and the pointers are 16-byte aligned.  indptr/indices must be
 * the arrays the plan was built from.  Grows the plan's workspace on demand
 * (stream-ordered).
 */
gtattn_status gtattn_fwd_plan(const gtattn_plan* plan, const int32_t* indptr,
                              const int32_t* indices, const void* Q, const void* K,
                              const void* V, void* out, int H, int D, float scale,
                              gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_fwd_plan_stats -- gtattn_fwd_plan that also writes each row's
 * softmax statistic, for a training step whose backward (gtattn_bwd_plan)
 * then skips the forward recompute.
 *   stats: fp32 [N, H], device memory, 4-byte aligned (required):
 *          stats[i, h] = log2 sum_j 2^(scale * log2(e) * q_i.k_j) over row
 *          i's entries, i.e. the natural log-sum-exp of the row's logits
 *          divided by ln 2; -inf for a row without entries.
 *   Other arguments, results and errors: as gtattn_fwd_plan, except that
 *   complete blocks go through the row kernels (the dense-block kernel
 *   writes no statistics).  For the backward, out must be fp32 (dtype F32,
 *   or BF16_OUT_F32 for bf16 inputs).
 */
gtattn_status gtattn_fwd_plan_stats(const gtattn_plan* plan, const int32_t* indptr,
                                    const int32_t* indices, const void* Q, const void* K,
                                    const void* V, void* out, float* stats, int H, int D, float scale,
                                    gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_fwd_probs -- the unfused path: SDDMM (logits), edge softmax
 * (probs), SpMM (out) as three kernel stages with the per-edge values
 * materialised in global memory -- the bsddmm / softmax / bspmm and
 * u_dot_v / edge_softmax / u_mul_e_sum decompositions of the pages.
 *   logits: fp32 [nnz, H] in CSR order, scale * q.k (may be NULL).
 *   probs:  fp32 [nnz, H] in CSR order (may be NULL).
 *   out:    as gtattn_fwd.
 * When logits or probs is NULL the library uses a temporary in its place.
 */
gtattn_status gtattn_fwd_probs(const int32_t* indptr, const int32_t* indices, const void* Q,
                               const void* K, const void* V, void* out, float* logits,
                               float* probs, int64_t N, int64_t nnz, int H, int D,
                               float scale, gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_fwd_bias -- the forward with a per-edge, per-head additive bias on
 * the logits: e = scale * q_i.k_j + bias[e, h] ("Graph Transformer theory,
 * derivation and implementation", section on the shortest-path bias and
 * degree encoding (Graphormer type), spatial encoding: e_ij = q_i.k_j /
 * sqrt(d_k) + b_d(i,j), optionally one bias per head; b = -inf removes the
 * pair).  The caller looks the bias up per CSR entry.
 *   bias:   fp32 [nnz, H] in CSR order, device memory, 4-byte aligned
 *           (required when nnz > 0; entries may be -inf).
 *   logits, probs: as gtattn_fwd_probs; logits include the bias.  When both
 *           are NULL the fused kernels run (no per-edge values in memory),
 *           else the unfused trio.
 *   Other arguments and errors: as gtattn_fwd; INVALID_ARG for a missing or
 *   misaligned bias.
 * A row whose logits are all -inf (every entry removed) gives zeros, like a
 * row without entries, and probabilities 0.
 */
gtattn_status gtattn_fwd_bias(const int32_t* indptr, const int32_t* indices, const void* Q,
                              const void* K, const void* V, const float* bias, void* out,
                              float* logits, float* probs, int64_t N, int64_t nnz, int H, int D,
                              float scale, gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_fwd_weighted -- the forward on a weighted adjacency:
 * SparseAttn(Q, K, V, A) = softmax(((Q K^T) o A) / sqrt(d)) V with
 * A in [0,1] ("Graph Transformer in a Nutshell", section Sparse Multi-head
 * Attention: the Hadamard product with the adjacency matrix's values).
 *   values: fp32 [nnz], A's stored value of each CSR entry (shared by the
 *           heads), device memory, 4-byte aligned (required when nnz > 0).
 *           The logit of entry e is scale * (q.k) * values[e]; the softmax
 *           still runs over the stored entries only (a stored 0 gives logit
 *           0, it does not remove the entry).
 *   logits, probs: as gtattn_fwd_probs (logits include the values); both
 *           NULL: the fused kernels, else the unfused trio.
 *   Other arguments and errors: as gtattn_fwd; INVALID_ARG for missing or
 *   misaligned values.
 */
gtattn_status gtattn_fwd_weighted(const int32_t* indptr, const int32_t* indices, const float* values,
                                  const void* Q, const void* K, const void* V, void* out, float* logits,
                                  float* probs, int64_t N, int64_t nnz, int H, int D, float scale,
                                  gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_bwd -- the backward pass of gtattn_fwd (binary A, no bias): the
 * gradients of L = sum(out * dO) with respect to Q, K and V.  The pages
 * train the block (loss.backward() in the "Graph Transformer in a Nutshell"
 * training loop) without printing a backward; this is the chain rule on the
 * forward's definition: with s = scale q_i.k_j, p the row softmax,
 * dp = dO_i.v_j and ds = p (dp - sum_row p dp):
 *   dQ_i = scale sum_j ds k_j,  dK_j = scale sum_i ds q_i,  dV_j = sum_i p dO_i.
 *   Q, K, V, dO: [N, H, D] in dtype (F32, or BF16 / BF16_OUT_F32 for bf16
 *           inputs), device memory.
 *   dQ, dK, dV: fp32 [N, H, D], device memory, 4-byte aligned; every row
 *           is overwritten (rows without entries get zeros).
 *   H <= 128.  Other arguments: as gtattn_fwd.  Asynchronous on `stream`;
 *   the temporaries (the forward's fp32 output and log-sum-exp, a
 *   source-major copy of the pattern, the split rows' and sources' partial
 *   sums: about 4 N H D + 12 N H + 12 N + 8 nnz bytes plus the binnings and
 *   the partials) come from the library's stream-ordered pool.
 *   indices must lie in [0, N), as for gtattn_fwd (csr_validate checks).
 * Deterministic: the source-major copy lists each source's destination rows
 * in ascending order, every row and source is summed in one fixed order,
 * and the chunks of split rows and sources are added in chunk order, so two
 * calls on the same inputs give the same bits (shapes whose H*D the two
 * passes do not tile -- see below -- fall back to a warp per row with fp32
 * atomics, which is not deterministic).
 */
gtattn_status gtattn_bwd(const int32_t* indptr, const int32_t* indices, const void* Q, const void* K,
                         const void* V, const void* dO, float* dQ, float* dK, float* dV, int64_t N,
                         int64_t nnz, int H, int D, float scale, gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_bwd_plan -- gtattn_bwd with a prebuilt plan, for training on a
 * fixed graph: the plan's destination binning is used as it stands, and the
 * source-major copy of the pattern with its binning (and the rows binned
 * again with the backward's own split thresholds) is built by the first
 * backward call with the plan and kept in it (about 8 N + 4 nnz bytes plus
 * the binnings, freed by gtattn_plan_destroy), so later calls skip it.  Same
 * results, bit for bit, as gtattn_bwd.  indptr/indices must be the arrays
 * the plan was built from.  One plan must not be used by concurrent calls.
 *   O, stats: the fp32 output (16-byte aligned) and statistics that
 *           gtattn_fwd_plan_stats wrote for the same plan, Q, K, V, scale
 *           and (bf16 inputs: BF16_OUT_F32) dtype, or both NULL.  Given,
 *           the backward skips its forward recompute and, with the plan's
 *           default kernel choice, gives the same bits as without them;
 *           NULL, it recomputes both.  One given without the other, or
 *           misaligned: INVALID_ARG.
 */
gtattn_status gtattn_bwd_plan(const gtattn_plan* plan, const int32_t* indptr, const int32_t* indices,
                              const void* Q, const void* K, const void* V, const float* O, const float* stats,
                              const void* dO, float* dQ, float* dK, float* dV, int H, int D, float scale,
                              gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_fwd_noalloc -- gtattn_fwd without any allocation.  The pages have
 * no counterpart: this exists for callers that cannot allocate device memory
 * when they run attention -- code running inside an allocator or memory-pool
 * callback, runtimes that forbid cudaMalloc after start-up (fixed budgets,
 * pre-planned arenas), frameworks that own the whole device heap.
 * Same arguments, operation and argument checks as gtattn_fwd.  Its
 * temporaries live in one fixed 32 MiB device array inside the library
 * (every GPU that loads the library holds it until the process exits); it
 * calls no cudaMalloc/cudaFree or other allocating routine.  Rows with more
 * than 1024 entries are split into chunks of 1024.
 *   Size limit: the call needs, in bytes, about
 *     4*N + 8*(C + L) + 4*C*(H*D + 2*H) (+ a little alignment),
 *   with L = min(N, nnz/1025) and C = nnz/1024 + L; above 32 MiB it returns
 *   GTATTN_ERR_UNSUPPORTED before any GPU work (gtattn_last_error then says
 *   how many bytes were needed).  Example: 2^20 rows, 17.1M entries, 4x32 fits.
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is kept with the id of the
 *   context it was found in: after the device's context is destroyed and
 *   made again (cudaDeviceReset), the next call finds the array anew (and is
 *   again a first call in this sense).
 *   Concurrency: every call shares the one array and leaves its contents
 *   behind (each call re-initialises what it reads), so calls whose GPU work
 *   may overlap -- on different streams, or from different threads -- race
 *   and corrupt each other's results.  Serialise them.
 */
gtattn_status gtattn_fwd_noalloc(const int32_t* indptr, const int32_t* indices, const void* Q,
                                 const void* K, const void* V, void* out, int64_t N, int64_t nnz,
                                 int H, int D, float scale, gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_fwd_proj -- the attention block with its linear projections, as
 * SparseMHA.forward of "Graph Transformer in a Nutshell" (section "Sparse
 * Multi-head Attention": q_proj, k_proj, v_proj, the sparse attention,
 * out_proj; nn.Linear maps with biases) and the attention part of
 * TransLayer.forward of "Efficient Sparse Transformer implementation with
 * DGL's builtin operators" (proj_q, proj_k, proj_v, u_dot_v / edge_softmax /
 * u_mul_e_sum, proj_o; no biases):
 *   q = X Wq^T + bq,  k = X Wk^T + bk,  v = X Wv^T + bv   (H heads of D)
 *   o = SparseAttn(q, k, v, A)                             (as gtattn_fwd)
 *   Y = o Wo^T + bo                                        (o's heads merged)
 *   X:    [N, F_in] node features, of the input type of `dtype` (fp32, or
 *         bf16 for GTATTN_BF16 and GTATTN_BF16_OUT_F32).
 *   Wqkv: [3*H*D, F_in], the weights of the q, k and v maps stacked in that
 *         order (each an nn.Linear weight [out features, in features]), input
 *         type.  bqkv: fp32 [3*H*D] in the same order, or NULL (no biases).
 *   Wo:   [F_out, H*D], input type.  bo: fp32 [F_out] or NULL.
 *   Y:    [N, F_out], the output type of `dtype` (bf16 for GTATTN_BF16, else
 *         fp32).
 *   heads_inner: how projection features map to heads.  0: feature h*D + d
 *         is element d of head h (TransLayer's view(-1, h, d_qkv)); 1:
 *         feature d*H + h is element d of head h (SparseMHA's
 *         reshape(N, head_dim, num_heads)); the out map reads o's features in
 *         the same order.
 *   qkv:  NULL, or [3, N, H, D] (input type, head-major whatever heads_inner
 *         says) receiving q, k, v; attn: NULL, or [N, H, D] receiving o.
 *         When NULL, library temporaries hold them.
 *   scale: multiplies q.k (SparseMHA folds head_dim**-0.5 into q; the
 *         product is the same).
 * q, k, v and o are held in the input type between the stages (bf16 values
 * rounded to nearest even from the fp32 accumulators); every product
 * accumulates in fp32.  bf16 maps with F_in and H*D multiples of 8 (and
 * 16-byte aligned arrays) run on the tensor cores (tcgen05); the others on
 * the CUDA cores.  Pointers are device memory aligned to their element size;
 * library temporaries come from the stream-ordered pool.  Asynchronous on
 * `stream`.  Errors: INVALID_ARG (null pointer, sizes, dtype, heads_inner,
 * alignment), NO_MEMORY, CUDA.  A bounded device wait of the tensor-core
 * maps that gives up is reported by gtattn_device_errors.
 */
gtattn_status gtattn_fwd_proj(const int32_t* indptr, const int32_t* indices, const void* X, const void* Wqkv,
                              const float* bqkv, const void* Wo, const float* bo, void* Y, void* qkv, void* attn,
                              int64_t N, int64_t nnz, int F_in, int H, int D, int F_out, int heads_inner,
                              float scale, gtattn_dtype dtype, cudaStream_t stream);

/*
 * gtattn_device_errors -- error codes recorded on the current device by
 * kernels that have no plan to report into (the tensor-core projections of
 * gtattn_fwd_proj): the bitwise OR since the last reset, 1 = a bounded wait
 * gave up (its results are not valid).  Synchronises the device; with
 * `reset`, clears the record.
 */
gtattn_status gtattn_device_errors(int* code, int reset);

/*
 * gtattn_coo_to_csr -- builds CSR by destination from a COO edge list
 * (src[e] -> dst[e]); within a row, entries are sorted by source and
 * duplicates are kept ("Graph Transformer in a Nutshell" builds A from
 * g.edges() with no values).  indptr: int32 [N+1], indices: int32 [nnz],
 * both caller-allocated.  Edges whose destination is outside [0, N) are
 * dropped (indptr[N] then counts the kept edges); sources are not checked.
 * Uses stream-ordered temporaries.
 */
gtattn_status gtattn_coo_to_csr(const int32_t* src, const int32_t* dst, int64_t nnz, int64_t N,
                                int32_t* indptr, int32_t* indices, cudaStream_t stream);

/*
 * gtattn_csr_validate -- checks indptr[0] == 0, indptr non-decreasing,
 * indptr[N] == nnz and every index in [0, N) on the device.  Synchronous
 * (waits for `stream`).  Returns GTATTN_OK or GTATTN_ERR_BAD_CSR.
 */
gtattn_status gtattn_csr_validate(const int32_t* indptr, const int32_t* indices, int64_t N,
                                  int64_t nnz, cudaStream_t stream);

/*
 * Benchmark instrumentation (not part of the pages' operation).  While
 * enabled, the library brackets each of its kernel launches (or a launch
 * group, for binning) with a pair of CUDA events on the launching stream and
 * counts the launches, by category.  Process-wide and not thread-safe; meant
 * for benchmarks and profiling runs.  gtattn_profile_read synchronises on
 * the recorded events, adds their elapsed times into *out and, with `reset`,
 * clears the record.
 */
typedef enum {
    GTATTN_KCAT_BIN = 0,      /* degree binning (launch group) */
    GTATTN_KCAT_ROWS = 1,     /* row kernels: fused, SDDMM, SpMM modes */
    GTATTN_KCAT_COMBINE = 2,  /* split-row combine */
    GTATTN_KCAT_SOFTMAX = 3,  /* unfused edge softmax */
    GTATTN_KCAT_DENSE = 4,    /* dense-block tensor-core kernel */
    GTATTN_KCAT_GEMM = 5,     /* projections around the attention (and their weight permutations) */
    GTATTN_KCAT_COUNT = 8
} gtattn_kernel_category;

typedef struct {
    int32_t launches[GTATTN_KCAT_COUNT];  /* kernel launches recorded */
    int32_t groups[GTATTN_KCAT_COUNT];    /* event pairs recorded */
    double ms[GTATTN_KCAT_COUNT];         /* summed event-pair durations */
} gtattn_profile;

gtattn_status gtattn_profile_enable(int on);
gtattn_status gtattn_profile_read(gtattn_profile* out, int reset);

#ifdef __cplusplus
}
#endif

#endif /* GTATTN_H */
