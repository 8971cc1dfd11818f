// plan.cuh -- the plan object and the binning entry points used by api.cu.
#pragma once

#include "common.cuh"

struct gtattn_plan {
    int64_t N = 0, nnz = 0;
    gtattn_plan_opts opts{};
    int device = -1;
    cudaStream_t stream = nullptr;          // stream the plan was built on
    int* hdr = nullptr;                     // device header (HdrLayout words)
    int hdr_host[gt::HdrLayout::kWords] = {};
    int* rows = nullptr;                    // bucketed rows, then the dense segment
    int2* chunks = nullptr;                 // (row, first entry) per chunk
    int2* longs = nullptr;                  // (row, first chunk) per split row
    int2* blocks = nullptr;                 // (first row, size) per dense block
    int4* dense_tiles = nullptr;            // (block row, block size, first query row, query tiles)
    int n_dense_tiles = 0;
    int4* dense_tiles1 = nullptr;           // the same blocks, one query tile per item
    int n_dense_tiles1 = 0;
    int* dense_flag = nullptr;              // 1 for rows inside a dense block
    mutable void* ws = nullptr;             // split-row partials workspace
    mutable size_t ws_bytes = 0;
    mutable void* bwd_pattern = nullptr;    // source-major pattern and source binning (first backward)
};

namespace gt {

// Rows of more than kDefaultLongMin entries are split into kDefaultChunk-
// entry chunks (R-MAT forward: 0.89 ms at 1024 / 1024 against 0.92 at
// 256 / 256: fewer chunk partials to combine, and a task per row of up to
// 1024 entries keeps its lane groups busy).  The backward's source binning
// keeps its own thresholds (kBwdLongMin / kBwdChunk) unless a plan sets
// others.
constexpr int kDefaultLongMin = 1024;
constexpr int kDefaultChunk = 1024;
constexpr int kBwdLongMin = 256;
constexpr int kBwdChunk = 256;

void resolve_opts(const gtattn_plan_opts* in, gtattn_plan_opts* out);
void worst_case_sizes(int64_t N, int64_t nnz, int long_min, int chunk, int64_t* n_long,
                      int64_t* n_chunks);
// Graphs of at most this many rows are binned by a single block in one launch.
constexpr int kBinSmallRows = 4096;
// Bins rows into the given arrays on stream `s` without synchronising:
// zeroes the header, counts, lays out offsets and scatters rows/chunks.
gtattn_status bin_rows(const int* indptr, int N, int long_min, int chunk, const int* dense_flag,
                       int* hdr, int* rows, int2* chunks, int2* longs, cudaStream_t s);
// Kernel launches bin_rows makes for N rows (1 for small graphs, else 3).
int bin_launches(int N, const int* dense_flag);

}  // namespace gt
