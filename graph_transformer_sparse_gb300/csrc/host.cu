// host.cu -- gtattn_fwd_host: the plan-less fused forward on host buffers.
//
// The call copies the graph and features to the device, runs the forward and
// copies the output back, overlapping the three: K and V go first (every row
// gathers from all of them), then the rows are cut into chunks of about
// equal work; chunk c's indptr, indices and Q rows are copied on an internal
// host-to-device stream while chunk c-1 is computed on the caller's stream,
// and chunk c's output rows are copied back on an internal device-to-host
// stream while later chunks are copied and computed.  A chunk is computed by
// gtattn_fwd on a view of the device arrays: indptr from the chunk's first
// row (its values stay absolute offsets into indices), Q and out from the
// chunk's first row, K and V whole.
#include "common.cuh"

#include <algorithm>
#include <mutex>
#include <vector>

namespace gt {
namespace {

constexpr int kMaxHostChunks = 8;
constexpr int64_t kEntriesPerChunk = int64_t(1) << 20;   // fewer chunks for small graphs

struct HostStreams {
    cudaStream_t h2d = nullptr, d2h = nullptr;
};

// The two internal copy streams of the current device, created once.
gtattn_status host_streams(HostStreams* out) {
    constexpr int kMaxDev = 64;
    static std::mutex mu;
    static HostStreams streams[kMaxDev];
    int dev = 0;
    GT_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDev) return GTATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> g(mu);
    HostStreams& s = streams[dev];
    if (!s.h2d) {
        GT_CUDA(cudaStreamCreateWithFlags(&s.h2d, cudaStreamNonBlocking));
        cudaError_t e = cudaStreamCreateWithFlags(&s.d2h, cudaStreamNonBlocking);
        if (e != cudaSuccess) {
            cudaStreamDestroy(s.h2d);
            s.h2d = nullptr;
            return cuda_status(e);
        }
    }
    *out = s;
    return GTATTN_OK;
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Row boundaries of `n_chunks` chunks of about equal work (entries plus rows)
// from the host copy of indptr.
std::vector<int64_t> chunk_rows(const int32_t* indptr, int64_t N, int n_chunks) {
    std::vector<int64_t> b(n_chunks + 1, N);
    b[0] = 0;
    const double total = static_cast<double>(indptr[N] - indptr[0]) + static_cast<double>(N);
    int64_t lo = 0;
    for (int c = 1; c < n_chunks; ++c) {
        const double target = total * c / n_chunks;
        int64_t l = lo, h = N;   // first row r with work(r) >= target
        while (l < h) {
            const int64_t m = l + (h - l) / 2;
            if (static_cast<double>(indptr[m] - indptr[0]) + static_cast<double>(m) < target) l = m + 1;
            else h = m;
        }
        b[c] = std::max(l, b[c - 1]);
        lo = b[c];
    }
    return b;
}

}  // namespace
}  // namespace gt

using namespace gt;

extern "C" gtattn_status gtattn_fwd_host(const int32_t* indptr, const int32_t* indices, const void* Q,
                                         const void* K, const void* V, void* out, int64_t N, int64_t nnz,
                                         int H, int D, float scale, gtattn_dtype dtype, cudaStream_t stream) {
    // the argument rules of gtattn_fwd, on host pointers
    if (N < 0 || nnz < 0 || N >= (1ll << 31) - 1 || nnz >= (1ll << 31) - 1) return GTATTN_ERR_INVALID_ARG;
    if (H < 1 || D < 1 || (int64_t)H * D > kMaxHD) return GTATTN_ERR_INVALID_ARG;
    if (dtype != GTATTN_F32 && dtype != GTATTN_BF16 && dtype != GTATTN_BF16_OUT_F32) return GTATTN_ERR_INVALID_ARG;
    if (!indptr || (N > 0 && (!Q || !out)) || (nnz > 0 && (!indices || !K || !V))) return GTATTN_ERR_INVALID_ARG;
    if (N == 0) return GTATTN_OK;
    // indptr is read here on the host (chunk boundaries): check its ends
    if (indptr[0] != 0 || indptr[N] != nnz) return GTATTN_ERR_BAD_CSR;
#ifdef GTATTN_DEBUG
    // the checking build validates the whole CSR, here on the host
    for (int64_t i = 0; i < N; ++i)
        if (indptr[i + 1] < indptr[i]) return GTATTN_ERR_BAD_CSR;
    for (int64_t e = 0; e < nnz; ++e)
        if (indices[e] < 0 || indices[e] >= N) return GTATTN_ERR_BAD_CSR;
#endif

    const size_t esz = dtype == GTATTN_F32 ? 4 : 2;
    const size_t osz = dtype == GTATTN_BF16 ? 2 : 4;
    const size_t HD = static_cast<size_t>(H) * D;
    const size_t b_ip = sizeof(int32_t) * (static_cast<size_t>(N) + 1);
    const size_t b_idx = sizeof(int32_t) * static_cast<size_t>(nnz);
    const size_t b_feat = static_cast<size_t>(N) * HD * esz;
    const size_t b_out = static_cast<size_t>(N) * HD * osz;
    void* base = nullptr;
    GT_TRY(pool_alloc(&base, up256(b_ip) + up256(b_idx) + 3 * up256(b_feat) + up256(b_out), stream));
    char* p = static_cast<char*>(base);
    int32_t* ip_d = reinterpret_cast<int32_t*>(p);
    p += up256(b_ip);
    int32_t* idx_d = reinterpret_cast<int32_t*>(p);
    p += up256(b_idx);
    char* q_d = p;
    p += up256(b_feat);
    char* k_d = p;
    p += up256(b_feat);
    char* v_d = p;
    p += up256(b_feat);
    char* out_d = p;

    HostStreams hs;
    gtattn_status st = host_streams(&hs);
    if (st != GTATTN_OK) {
        pool_free(base, stream);
        return st;
    }
    const int n_chunks = static_cast<int>(
        std::max<int64_t>(1, std::min<int64_t>({kMaxHostChunks, nnz / kEntriesPerChunk, N})));
    const std::vector<int64_t> b = chunk_rows(indptr, N, n_chunks);

    // events: allocation ready, chunk inputs copied, chunk computed, copies joined
    auto ok = [&](cudaError_t e) {
        if (st == GTATTN_OK && e != cudaSuccess) st = cuda_status(e);
        return st == GTATTN_OK;
    };
    std::vector<cudaEvent_t> ev(2 * n_chunks + 3, nullptr);
    for (auto& e : ev)
        if (st == GTATTN_OK) ok(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    cudaEvent_t e_alloc = ev[0], e_h2d_end = ev[2 * n_chunks + 1], e_d2h_end = ev[2 * n_chunks + 2];
    if (st == GTATTN_OK) {
        ok(cudaEventRecord(e_alloc, stream)) && ok(cudaStreamWaitEvent(hs.h2d, e_alloc, 0)) &&
            ok(cudaStreamWaitEvent(hs.d2h, e_alloc, 0));
    }
    if (st == GTATTN_OK && nnz > 0) {
        ok(cudaMemcpyAsync(k_d, K, b_feat, cudaMemcpyHostToDevice, hs.h2d)) &&
            ok(cudaMemcpyAsync(v_d, V, b_feat, cudaMemcpyHostToDevice, hs.h2d));
    }
    for (int c = 0; c < n_chunks && st == GTATTN_OK; ++c) {
        const int64_t r0 = b[c], r1 = b[c + 1];
        const int64_t e0 = indptr[r0], e1 = indptr[r1];
        ok(cudaMemcpyAsync(ip_d + r0, indptr + r0, sizeof(int32_t) * (r1 - r0 + 1), cudaMemcpyHostToDevice,
                           hs.h2d)) &&
            (e1 == e0 || ok(cudaMemcpyAsync(idx_d + e0, indices + e0, sizeof(int32_t) * (e1 - e0),
                                            cudaMemcpyHostToDevice, hs.h2d))) &&
            (r1 == r0 || ok(cudaMemcpyAsync(q_d + r0 * HD * esz, static_cast<const char*>(Q) + r0 * HD * esz,
                                            (r1 - r0) * HD * esz, cudaMemcpyHostToDevice, hs.h2d))) &&
            ok(cudaEventRecord(ev[1 + c], hs.h2d));
    }
    for (int c = 0; c < n_chunks && st == GTATTN_OK; ++c) {
        const int64_t r0 = b[c], r1 = b[c + 1];
        if (!ok(cudaStreamWaitEvent(stream, ev[1 + c], 0))) break;
        if (r1 > r0) {
            st = fwd_view(ip_d + r0, nnz > 0 ? idx_d : nullptr, q_d + r0 * HD * esz, nnz > 0 ? k_d : nullptr,
                            nnz > 0 ? v_d : nullptr, out_d + r0 * HD * osz, r1 - r0, indptr[r1] - indptr[r0], H,
                            D, scale, dtype, N, stream);
            if (st != GTATTN_OK) break;
        }
        ok(cudaEventRecord(ev[1 + n_chunks + c], stream)) &&
            ok(cudaStreamWaitEvent(hs.d2h, ev[1 + n_chunks + c], 0)) &&
            (r1 == r0 || ok(cudaMemcpyAsync(static_cast<char*>(out) + r0 * HD * osz, out_d + r0 * HD * osz,
                                            (r1 - r0) * HD * osz, cudaMemcpyDeviceToHost, hs.d2h)));
    }
    // join: the caller's stream waits for every copy issued, then the
    // temporaries go back to the pool in stream order
    if (e_h2d_end && cudaEventRecord(e_h2d_end, hs.h2d) == cudaSuccess) cudaStreamWaitEvent(stream, e_h2d_end, 0);
    if (e_d2h_end && cudaEventRecord(e_d2h_end, hs.d2h) == cudaSuccess) cudaStreamWaitEvent(stream, e_d2h_end, 0);
    pool_free(base, stream);
    for (auto e : ev)
        if (e) cudaEventDestroy(e);
    return st;
}
