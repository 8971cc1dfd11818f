/*
 * oracle.c -- plain fp64 CPU oracle for sparse multi-head attention.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the bench's
 * CPU-baseline leg may call this code.  It shares nothing with the CUDA
 * library: no headers, helpers or constants.
 *
 * What it computes (per CSR row i, per head h):
 *
 *   SparseAttn(Q, K, V, A) = softmax((Q K^T) o A / sqrt(d)) V
 *     -- "Graph Transformer in a Nutshell", section "Sparse Multi-head
 *        Attention", equation SparseAttn; SparseMHA.forward (bsddmm ->
 *        sparse softmax over the last sparse dimension -> bspmm).
 *
 *   e = u_dot_v(g, k, q);  a = edge_softmax(g, e / sqrt(d_qkv));
 *   wv = u_mul_e_sum(g, v, a)
 *     -- "Efficient Sparse Transformer implementation with DGL's builtin
 *        operators", TransLayer.forward.
 *
 *   e_ij = q_i . k_j / sqrt(d_k);  alpha_ij = exp(e_ij) / sum_j' exp(e_ij');
 *   h_i = sum_j alpha_ij v_j
 *     -- "Graph Transformer theory, derivation and implementation"
 *        (グラフTransformerの理論と導出と実装), section "review of scaled
 *        dot-product attention" (スケール付きドット積注意の復習).
 *
 * Readings taken where the pages leave a step open:
 *  - the softmax runs over the stored entries of the row only; non-edges are
 *    excluded (weight 0, i.e. logit -inf as in the same page's shortest-path
 *    bias section, b_inf = -inf), not treated as logit 0;
 *  - A is binary (the spmatrix is built from an edge list with no values)
 *    unless the caller passes its stored values (below);
 *  - row i lists the nodes j it attends to (CSR by destination: node i
 *    aggregates over its in-edges j -> i);
 *  - a row with no entries gives exact zeros;
 *  - every CSR entry is its own edge (duplicates count twice);
 *  - `scale` is an argument (normally 1/sqrt(D)); the logit is
 *    scale * (q . k) in fp64;
 *  - the max is subtracted before exp (does not change the result);
 *  - no dropout (evaluation mode).
 *
 * Optional per-edge additive bias (the Graphormer spatial encoding):
 *   e_ij = q_i . k_j / sqrt(d_k) + b_{d(i,j)}
 *     -- "Graph Transformer theory, derivation and implementation", section
 *        "shortest-path bias and degree encoding (Graphormer type)",
 *        subsection "spatial encoding: shortest-path distance bias" (a
 *        learnable scalar per distance, optionally per head, added to the
 *        logit before the softmax; b_inf = -inf removes a pair).
 *   Reading: the caller supplies the bias already looked up per CSR entry
 *   and head, bias[e*H + h] (float32, promoted to double); it is added to
 *   scale * (q . k).  A row whose logits are all -inf (every entry removed)
 *   gives exact zeros, like a row with no entries, and probabilities 0.
 *
 * Optional weighted adjacency:
 *   SparseAttn(Q, K, V, A) = softmax(((Q K^T) o A) / sqrt(d)) V, A in [0,1]^{NxN}
 *     -- "Graph Transformer in a Nutshell", section "Sparse Multi-head
 *        Attention" (the Hadamard product with A's values).
 *   Reading: values[e] (float32, one per CSR entry, shared by the heads) is
 *   A's stored value; the logit is scale * ((q . k) * values[e]); the
 *   softmax still runs over the stored entries only (a stored 0 gives
 *   logit 0, it does not remove the entry).
 *
 * Projections around the attention (gto_linear, gto_round_store; the
 * composition is in oracle/__init__.py, sparse_mha_proj): Y = X W^T + b for
 * the nn.Linear maps of SparseMHA / TransLayer, and the precision an
 * intermediate is stored in between the stages (float32, or bf16 from the
 * float32 value, ties to even).
 *
 * Arithmetic: inputs are float32 (bf16 inputs arrive as their exact float32
 * widening), every operation is double, the reductions run in index order,
 * exp is the C library's double exp.  Two passes per (row, head): logits and
 * max, then normalised weights and the weighted sum of V.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GTO_OK 0
#define GTO_BAD_CSR -1
#define GTO_BAD_ARG -2
#define GTO_NO_MEMORY -3

/* Check indptr monotone from 0 to nnz and every index in [0, N). */
int gto_check_csr(int64_t N, int64_t nnz, const int32_t* indptr, const int32_t* indices)
{
    if (N < 0 || nnz < 0 || !indptr) return GTO_BAD_ARG;
    if (indptr[0] != 0 || (int64_t)indptr[N] != nnz) return GTO_BAD_CSR;
    for (int64_t i = 0; i < N; ++i)
        if (indptr[i + 1] < indptr[i]) return GTO_BAD_CSR;
    for (int64_t e = 0; e < nnz; ++e)
        if (indices[e] < 0 || (int64_t)indices[e] >= N) return GTO_BAD_CSR;
    return GTO_OK;
}

/*
 * Sparse MHA forward for a list of rows.
 *   Q, K, V : float32 [N, H, D] row-major (D innermost).
 *   rows    : the rows to compute (NULL: rows 0..N-1, then nrows must be N).
 *   out     : double [nrows, H, D], row r of the list at out + r*H*D.
 *   values  : float32 [nnz], A's stored values (weighted A), or NULL (binary A).
 *   bias    : float32 [nnz, H] added to the logits, or NULL for none.
 *   logits, probs : double [nnz, H] indexed by CSR position (may be NULL);
 *             only the entries of the listed rows are written.
 * Returns 0, or a negative code for bad arguments / bad CSR / no memory.
 */
int gto_sparse_mha_rows(int64_t N, int64_t nnz, int32_t H, int32_t D,
                        const int32_t* indptr, const int32_t* indices,
                        const float* Q, const float* K, const float* V, const float* values,
                        const float* bias, double scale,
                        const int64_t* rows, int64_t nrows,
                        double* out, double* logits, double* probs)
{
    if (N < 0 || nnz < 0 || H <= 0 || D <= 0 || nrows < 0 || !indptr || !out) return GTO_BAD_ARG;
    if (!rows && nrows != N) return GTO_BAD_ARG;
    if (nnz > 0 && (!indices || !K || !V)) return GTO_BAD_ARG;
    if (N > 0 && !Q) return GTO_BAD_ARG;
    if (gto_check_csr(N, nnz, indptr, indices) != GTO_OK) return GTO_BAD_CSR;

    int64_t max_deg = 0;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        if (i < 0 || i >= N) return GTO_BAD_ARG;
        int64_t deg = (int64_t)indptr[i + 1] - indptr[i];
        if (deg > max_deg) max_deg = deg;
    }
    double* l = (double*)malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
    double* p = (double*)malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
    if (!l || !p) { free(l); free(p); return GTO_NO_MEMORY; }

    const int64_t HD = (int64_t)H * D;
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        const int64_t beg = indptr[i], end = indptr[i + 1];
        const int64_t deg = end - beg;
        double* o_row = out + r * HD;
        for (int32_t h = 0; h < H; ++h) {
            double* o = o_row + (int64_t)h * D;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            if (deg == 0) continue;                       /* empty row: zeros */
            const float* q = Q + i * HD + (int64_t)h * D;
            /* pass 1: logits l_e = scale * <q_i, k_j> and their max */
            double m = -INFINITY;
            for (int64_t k = 0; k < deg; ++k) {
                const int64_t j = indices[beg + k];
                const float* kj = K + j * HD + (int64_t)h * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += (double)q[d] * (double)kj[d];
                if (values) dot *= (double)values[beg + k];
                l[k] = scale * dot;
                if (bias) l[k] += (double)bias[(beg + k) * H + h];
                if (l[k] > m) m = l[k];
            }
            if (m == -INFINITY) {                         /* every entry removed: zeros */
                if (logits) for (int64_t k = 0; k < deg; ++k) logits[(beg + k) * H + h] = l[k];
                if (probs) for (int64_t k = 0; k < deg; ++k) probs[(beg + k) * H + h] = 0.0;
                continue;
            }
            /* pass 2: softmax weights over the row's stored entries */
            double S = 0.0;
            for (int64_t k = 0; k < deg; ++k) { p[k] = exp(l[k] - m); S += p[k]; }
            for (int64_t k = 0; k < deg; ++k) p[k] /= S;
            /* weighted sum of the neighbours' values */
            for (int64_t k = 0; k < deg; ++k) {
                const int64_t j = indices[beg + k];
                const float* vj = V + j * HD + (int64_t)h * D;
                for (int32_t d = 0; d < D; ++d) o[d] += p[k] * (double)vj[d];
            }
            if (logits) for (int64_t k = 0; k < deg; ++k) logits[(beg + k) * H + h] = l[k];
            if (probs) for (int64_t k = 0; k < deg; ++k) probs[(beg + k) * H + h] = p[k];
        }
    }
    free(l);
    free(p);
    return GTO_OK;
}

/*
 * Dense scaled-dot-product attention, all pairs, per head:
 *   out[i,h,:] = sum_j softmax_j(scale * q_i . k_j) v_j
 * -- "Graph Transformer in a Nutshell", the all-pairs Attn equation, and
 *    "Graph Transformer theory, derivation and implementation", review of
 *    scaled dot-product attention.  Q, K, V float32 [n, H, D]; out double.
 * This is the result a complete graph (with self-loops) must reproduce.
 */
int gto_dense_attention(int64_t n, int32_t H, int32_t D, const float* Q, const float* K,
                        const float* V, double scale, double* out)
{
    if (n < 0 || H <= 0 || D <= 0 || !out) return GTO_BAD_ARG;
    if (n == 0) return GTO_OK;
    if (!Q || !K || !V) return GTO_BAD_ARG;
    double* w = (double*)malloc(sizeof(double) * (size_t)n);
    if (!w) return GTO_NO_MEMORY;
    const int64_t HD = (int64_t)H * D;
    for (int64_t i = 0; i < n; ++i) {
        for (int32_t h = 0; h < H; ++h) {
            const float* q = Q + i * HD + (int64_t)h * D;
            double m = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                const float* kj = K + j * HD + (int64_t)h * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += (double)q[d] * (double)kj[d];
                w[j] = scale * dot;
                if (w[j] > m) m = w[j];
            }
            double S = 0.0;
            for (int64_t j = 0; j < n; ++j) { w[j] = exp(w[j] - m); S += w[j]; }
            double* o = out + i * HD + (int64_t)h * D;
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                const double a = w[j] / S;
                const float* vj = V + j * HD + (int64_t)h * D;
                for (int32_t d = 0; d < D; ++d) o[d] += a * (double)vj[d];
            }
        }
    }
    free(w);
    return GTO_OK;
}

/*
 * Backward pass of the sparse forward (binary A, no bias): the gradients
 * of L = sum_{i,h,d} out[i,h,d] * dO[i,h,d] with respect to Q, K and V.
 * The pages train this block (the molhiv loop of "Graph Transformer in a
 * Nutshell" calls loss.backward() through SparseMHA) but print no backward
 * formula; this is the chain rule applied to the definition above, per row
 * i and head h, with s_e = scale * q_i . k_j and p_e the row softmax:
 *   dp_e  = dO_i . v_j
 *   Dlt   = sum_e p_e dp_e
 *   ds_e  = p_e (dp_e - Dlt)                     (softmax Jacobian)
 *   dQ_i += scale * sum_e ds_e k_j
 *   dK_j += scale * ds_e q_i                     (for each entry e = (i <- j))
 *   dV_j += p_e dO_i
 * Q, K, V, dO float32 [N, H, D]; dQ, dK, dV double [N, H, D], overwritten.
 * Rows without entries contribute nothing.  Every operation is double, the
 * sums run in index order.
 */
int gto_sparse_mha_bwd(int64_t N, int64_t nnz, int32_t H, int32_t D,
                       const int32_t* indptr, const int32_t* indices,
                       const float* Q, const float* K, const float* V, const float* dO, double scale,
                       double* dQ, double* dK, double* dV)
{
    if (N < 0 || nnz < 0 || H <= 0 || D <= 0 || !indptr || !dQ || !dK || !dV) return GTO_BAD_ARG;
    if (nnz > 0 && (!indices || !K || !V)) return GTO_BAD_ARG;
    if (N > 0 && (!Q || !dO)) return GTO_BAD_ARG;
    if (gto_check_csr(N, nnz, indptr, indices) != GTO_OK) return GTO_BAD_CSR;
    const int64_t HD = (int64_t)H * D;
    for (int64_t x = 0; x < N * HD; ++x) { dQ[x] = 0.0; dK[x] = 0.0; dV[x] = 0.0; }
    int64_t max_deg = 0;
    for (int64_t i = 0; i < N; ++i)
        if ((int64_t)indptr[i + 1] - indptr[i] > max_deg) max_deg = (int64_t)indptr[i + 1] - indptr[i];
    double* p = (double*)malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
    double* dp = (double*)malloc(sizeof(double) * (size_t)(max_deg > 0 ? max_deg : 1));
    if (!p || !dp) { free(p); free(dp); return GTO_NO_MEMORY; }
    for (int64_t i = 0; i < N; ++i) {
        const int64_t beg = indptr[i], deg = (int64_t)indptr[i + 1] - beg;
        if (deg == 0) continue;
        for (int32_t h = 0; h < H; ++h) {
            const float* q = Q + i * HD + (int64_t)h * D;
            const float* g = dO + i * HD + (int64_t)h * D;
            /* forward again: logits, their max, softmax weights */
            double m = -INFINITY;
            for (int64_t k = 0; k < deg; ++k) {
                const float* kj = K + (int64_t)indices[beg + k] * HD + (int64_t)h * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += (double)q[d] * (double)kj[d];
                p[k] = scale * dot;
                if (p[k] > m) m = p[k];
            }
            double S = 0.0;
            for (int64_t k = 0; k < deg; ++k) { p[k] = exp(p[k] - m); S += p[k]; }
            for (int64_t k = 0; k < deg; ++k) p[k] /= S;
            /* dp_e = dO_i . v_j and its p-weighted mean */
            double Dlt = 0.0;
            for (int64_t k = 0; k < deg; ++k) {
                const float* vj = V + (int64_t)indices[beg + k] * HD + (int64_t)h * D;
                double dot = 0.0;
                for (int32_t d = 0; d < D; ++d) dot += (double)g[d] * (double)vj[d];
                dp[k] = dot;
                Dlt += p[k] * dot;
            }
            double* dq = dQ + i * HD + (int64_t)h * D;
            for (int64_t k = 0; k < deg; ++k) {
                const int64_t j = indices[beg + k];
                const double ds = p[k] * (dp[k] - Dlt);
                const float* kj = K + j * HD + (int64_t)h * D;
                double* dk = dK + j * HD + (int64_t)h * D;
                double* dv = dV + j * HD + (int64_t)h * D;
                for (int32_t d = 0; d < D; ++d) {
                    dq[d] += scale * ds * (double)kj[d];
                    dk[d] += scale * ds * (double)q[d];
                    dv[d] += p[k] * (double)g[d];
                }
            }
        }
    }
    free(p);
    free(dp);
    return GTO_OK;
}

/*
 * Linear layer: Y = X W^T + b, the nn.Linear maps around the attention --
 * q_proj, k_proj, v_proj and out_proj of SparseMHA ("Graph Transformer in a
 * Nutshell", section "Sparse Multi-head Attention"; nn.Linear keeps a bias)
 * and proj_q, proj_k, proj_v, proj_o of TransLayer ("Efficient Sparse
 * Transformer implementation with DGL's builtin operators"; bias=False).
 * X float32 [M, Kin]; W float32 [Nout, Kin] (nn.Linear's weight: one row per
 * output feature); b float32 [Nout] or NULL (no bias); Y double [M, Nout],
 * overwritten.  Each output is b[n] + sum_k X[m,k] W[n,k] in double, k in
 * index order.
 */
int gto_linear(int64_t M, int32_t Kin, int32_t Nout, const float* X, const float* W, const float* b, double* Y)
{
    if (M < 0 || Kin <= 0 || Nout <= 0 || !Y) return GTO_BAD_ARG;
    if (M == 0) return GTO_OK;
    if (!X || !W) return GTO_BAD_ARG;
    for (int64_t m = 0; m < M; ++m) {
        const float* x = X + m * Kin;
        for (int32_t n = 0; n < Nout; ++n) {
            const float* w = W + (int64_t)n * Kin;
            double acc = 0.0;
            for (int32_t k = 0; k < Kin; ++k) acc += (double)x[k] * (double)w[k];
            Y[m * Nout + n] = (b ? (double)b[n] : 0.0) + acc;
        }
    }
    return GTO_OK;
}

/*
 * Storage precision of intermediate results (the projected Q, K, V and the
 * attention output, which a module keeps in its working type between the
 * layers).  mode 0: the nearest float32 (ties to even, the C conversion
 * under the default rounding mode).  mode 1: that float32, then the nearest
 * bf16 (8 significant bits, ties to even), returned as its float32 value --
 * the two steps of a float32 accumulator stored as bf16.  Infinities and
 * NaNs pass through (a NaN stays a NaN).
 */
int gto_round_store(int64_t n, const double* in, int32_t mode, float* out)
{
    if (n < 0 || (n > 0 && (!in || !out)) || (mode != 0 && mode != 1)) return GTO_BAD_ARG;
    for (int64_t i = 0; i < n; ++i) {
        float f = (float)in[i];
        if (mode == 1 && isfinite(f)) {
            uint32_t u;
            memcpy(&u, &f, sizeof(u));
            const uint32_t low = u & 0xFFFFu;          /* the 16 bits dropped */
            uint32_t hi = u & 0xFFFF0000u;
            const uint32_t lsb = (u >> 16) & 1u;       /* last kept bit: ties go to even */
            if (low > 0x8000u || (low == 0x8000u && lsb)) hi += 0x10000u;   /* may carry into the exponent */
            memcpy(&f, &hi, sizeof(f));
        }
        out[i] = f;
    }
    return GTO_OK;
}
