// Internal declarations shared by the host side of the library and its kernels.
#pragma once

#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

namespace tide {

// Reduce-scatter kernel geometry: a chunk is the work of one CTA pass, kRsUnroll 16-byte
// bf16 vectors (8 elements) per thread.
constexpr int kRsThreads = 256;
constexpr int kRsUnroll = 2;
constexpr int64_t kRsChunk = int64_t(kRsThreads) * 8 * kRsUnroll;  // 4096 elements
constexpr int kRsCtasPerSm = 2;

// Bulk-copy reduce-scatter geometry: 1 producer warp + kBulkConsumerWarps consumer warps, one CTA
// per SM (16 warps in all), up to kBulkMaxStages shared-memory stages of one rank row of a
// kBulkChunk-element chunk (45 KB).  Measured on GB300 (Llama-3.1-70B layer, R = 8) against 56 KB x 4
// stages with 14 consumer warps: 1.78 against 1.59 TB/s at 16 CTAs, 7.12 against 7.02 at 152.  The
// consumers store a chunk's sums in one burst after its last rank, and the fifth stage keeps the
// copies going meanwhile.
constexpr int kBulkConsumerWarps = 15;
constexpr int kBulkThreads = (kBulkConsumerWarps + 1) * 32;
constexpr int64_t kBulkChunk = 23040;  // 15 warps x 32 threads x 6 groups x 8 elements
constexpr int kBulkMaxStages = 5;       // 5 x 45 KB + the pointer cache fit for R <= 112
constexpr size_t kMaxDynamicSmem = 231424;    // opt-in shared memory per CTA on sm_103 (232448) less 1 KB
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // bound of every device-side wait
constexpr uint64_t kMinTimeoutNs = 1000000ull;         // shortest bound a caller may set (1 ms)

// All-gather placement kernel geometry.
constexpr int kAgThreads = 256;
constexpr int kAgUnroll = 4;
constexpr int64_t kAgChunk = int64_t(kAgThreads) * 8 * kAgUnroll;  // 8192 elements
constexpr int kAgCtasPerSm = 4;

// Bulk-copy placement geometry: lane 0 of warp 0 drives the bulk copies, warps 1..3 copy the chunks
// bulk copies cannot carry; one CTA per SM, kAgBulkStages stages of kAgBulkChunk bf16 (48 KB).
constexpr int kAgBulkThreads = 128;
constexpr int64_t kAgBulkChunk = 24576;
constexpr int kAgBulkStages = 4;
// Default grid of the bulk placement: more CTAs than fit at once (one per SM) measured faster on
// GB300 (6.85 vs 6.66 TB/s on the Llama-3.1-70B layer): late CTAs even out the tail.
constexpr int kAgBulkCtasPerSm = 4;

// One (destination rank d, parameter p) piece of the reduce-scatter output.
struct RsSeg {
    int64_t dst_off;      // o_p: element offset of the piece in shard d
    int64_t src_off;      // d*s_p: element offset of the piece in every rank's gradient of p
    int64_t valid;        // v(d,p)*L_p: elements that are sums; the rest of the piece is padding
    int64_t total;        // s_p
    int64_t chunk_begin;  // index of the piece's first chunk in the flat chunk list
    int32_t d, p;
    int32_t vec;  // the gradient offset allows 16-byte loads and bulk copies (src_off % 8 == 0); the
                  // kernels store with the widest vectors the shard offset allows
    int32_t pad_;
};
static_assert(sizeof(RsSeg) == 56, "RsSeg layout");

// One (source rank r, parameter p) run of valid elements for the all-gather placement.
struct AgSeg {
    int64_t src_off;      // o_p: element offset in shard r
    int64_t dst_off;      // r*s_p: element offset in parameter p
    int64_t len;          // v(r,p)*L_p
    int64_t chunk_begin;  // index of the run's first chunk in the flat chunk list
    int32_t r, p;
    int32_t vec;  // both offsets are multiples of 8 elements
    int32_t pad_;
};
static_assert(sizeof(AgSeg) == 48, "AgSeg layout");

// Group layout (Table 2 of the paper) and the flat work lists built from it.
struct Plan {
    int32_t R = 0, P = 0;
    std::vector<int64_t> rows, row_len, m, s, o;
    int64_t S = 0, U = 0;
    std::vector<RsSeg> rs;
    int64_t rs_chunks = 0;
    std::vector<int32_t> rs_piece;  // index in rs of every chunk's piece
    std::vector<RsSeg> rs_bulk;  // same pieces, chunked for the bulk-copy kernel
    int64_t rs_bulk_chunks = 0;
    std::vector<int32_t> rs_bulk_piece;  // index in rs_bulk of every bulk chunk's piece
    // Summing step over staging slots (tide_reduce_scatter_slots): destination d's P pieces are
    // rs_slots[d*P .. d*P + P), each reading slot r at o_p (one table entry per slot: p field 0)
    // and writing the call's one shard (d field 0); their chunks, counted from 0 for every d, are
    // the same for all destinations (only the valid counts differ).
    std::vector<RsSeg> rs_slots;
    int64_t rs_slot_chunks = 0;          // bulk chunks of one destination
    std::vector<int32_t> rs_slot_piece;  // piece (0..P-1) of each of those chunks
    std::vector<AgSeg> ag;
    int64_t ag_chunks = 0;
    std::vector<int32_t> ag_run;  // index in ag of every chunk's run
    std::vector<AgSeg> ag_bulk;  // same runs, chunked for the bulk-copy placement kernel
    int64_t ag_bulk_chunks = 0;
    int64_t ag_vec_elems = 0;  // valid elements in runs whose offsets allow 16-byte vectors
};

// Returns 0 or a negative TIDE_* status.
int make_layout(int32_t R, int32_t P, const int64_t* rows, const int64_t* row_len, Plan* out);
void make_work_lists(Plan* plan);
// The register-path reduce-scatter pieces of make_work_lists (same pieces, order and chunk
// ranges) written straight into out[d*P + p] without allocating; cap = entries out can hold.
// Returns 0, TIDE_EINVAL or TIDE_ERANGE (the group is invalid, overflows, or needs > cap pieces).
int plan_rs_pieces(int32_t R, int32_t P, const int64_t* rows, const int64_t* row_len, RsSeg* out, size_t cap,
                   int64_t* nchunks);
int64_t valid_rows(int64_t rows_p, int64_t m_p, int64_t d);

// Stores `e` as this host thread's last CUDA error (tide_last_cuda_error) and returns TIDE_ECUDA.
int record_cuda_error(cudaError_t e);

// Kernel launchers (stream-ordered; return the launch status).
// chunk_piece: piece index of every chunk, or nullptr (the kernel then searches the piece list)
cudaError_t launch_reduce_scatter(const RsSeg* segs, int nsegs, const int32_t* chunk_piece, int64_t nchunks,
                                  const uint16_t* const* grads, float* const* shards, int R, int P,
                                  int allow_vec, int ctas, cudaStream_t stream);
// Bulk-copy variant: dynamic shared memory per CTA (stages + the current piece's R pointers), and
// the number of stages used for R ranks.
size_t bulk_smem_bytes(int R, int stages);
int bulk_stages(int R);
cudaError_t launch_reduce_scatter_bulk(const RsSeg* segs, const int32_t* chunk_piece, int64_t nchunks,
                                       const uint16_t* const* grads,
                                       float* const* shards, int R, int P, int allow_vec, int ctas, int* status,
                                       uint64_t timeout_ns, int inject, cudaStream_t stream);
// TMEM-staged variant of the bulk-copy kernel (same tables, same results): the consumers hand
// their sums to Tensor Memory and separate writer warps store them.
cudaError_t launch_reduce_scatter_tmem(const RsSeg* segs, const int32_t* chunk_piece, int64_t nchunks,
                                       const uint16_t* const* grads, float* const* shards, int R, int P,
                                       int allow_vec, int ctas, int* status, uint64_t timeout_ns, int inject,
                                       cudaStream_t stream);
size_t ag_bulk_smem_bytes();
cudaError_t launch_all_gather_bulk(const AgSeg* segs, int nsegs, int64_t nchunks, const uint16_t* const* shards,
                                   uint16_t* const* params, int ctas, int* status, uint64_t timeout_ns,
                                   cudaStream_t stream);
// chunk_run: run index of every chunk, or nullptr (the kernel then searches the run list)
cudaError_t launch_all_gather(const AgSeg* segs, int nsegs, const int32_t* chunk_run, int64_t nchunks,
                              const uint16_t* const* shards, uint16_t* const* params,
                              int allow_vec, int ctas, cudaStream_t stream);

}  // namespace tide
