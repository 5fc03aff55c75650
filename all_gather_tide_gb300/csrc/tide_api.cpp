// C ABI of the library (declared in include/tide.h): argument checks, the group object, the
// per-call pointer-table upload, kernel launches and the copy-engine placement path.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/tide.h"
#include "tide_internal.h"

namespace {

constexpr int kSlots = 4;  // pointer-table ring depth
constexpr int kMaxCeLanes = 8;  // helper streams for copy-engine work
constexpr uint32_t kAllFlags =
    TIDE_FLAG_VEC_STRICT | TIDE_FLAG_CE_STRICT | TIDE_FLAG_CE_2D | TIDE_FLAG_OVERLAP | TIDE_FLAG_CE_1D;

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = int(e);
    return TIDE_ECUDA;
}

#define TIDE_CUDA(call)                                   \
    do {                                                  \
        cudaError_t e_ = (call);                          \
        if (e_ != cudaSuccess) return cuda_fail(e_);      \
    } while (0)

// A copy enqueued on one of the copy-engine lanes: on failure the helper lanes are joined back to
// the caller's stream (so nothing already enqueued on them outlives the call unordered) before the
// error is reported.
#define TIDE_LANE_COPY(lanes, call)                       \
    do {                                                  \
        cudaError_t e_ = (call);                          \
        if (e_ != cudaSuccess) {                          \
            (lanes).end();                                \
            return cuda_fail(e_);                         \
        }                                                 \
    } while (0)

// One entry of the ring of pointer tables.  The host copy is pinned so the upload is a true
// asynchronous copy on the caller's stream; `done` is recorded after the kernel that reads the
// device copy, so the slot is only rewritten once that kernel has finished.
struct Slot {
    std::vector<const void*> content;
    const void** host = nullptr;
    void** dev = nullptr;
    cudaEvent_t done = nullptr;
    cudaStream_t stream = nullptr;
    uint64_t last_use = 0;
    bool valid = false;
    bool pending = false;
};

}  // namespace

int tide::record_cuda_error(cudaError_t e) { return cuda_fail(e); }

struct tide_group {
    tide::Plan plan;
    uint32_t flags = 0;
    int device = 0;
    int sm_count = 0;
    int rs_ctas = 0, ag_ctas = 0;  // 0 = default
    int rs_variant = TIDE_RS_AUTO;
    int ag_variant = TIDE_AG_AUTO;
    uint64_t timeout_ns = tide::kDefaultTimeoutNs;
    uint32_t debug = 0;
    int* d_status = nullptr;  // device status word written by bounded waits that expire
    tide::RsSeg* d_rs = nullptr;
    int32_t* d_rs_piece = nullptr;  // piece index of every register-path chunk
    tide::RsSeg* d_rs_bulk = nullptr;
    int32_t* d_rs_bulk_piece = nullptr;  // piece index of every bulk chunk
    tide::RsSeg* d_rs_slots = nullptr;      // pieces of the summing step over staging slots
    int32_t* d_rs_slot_piece = nullptr;     // piece (0..P-1) of every chunk of one destination
    tide::AgSeg* d_ag_bulk = nullptr;
    tide::AgSeg* d_ag = nullptr;
    int32_t* d_ag_run = nullptr;  // run index of every register-path placement chunk
    size_t slot_cap = 0;
    Slot slots[kSlots];
    uint64_t use_clock = 0;
    int64_t last_ce_copies = 0;
    int32_t last_ce_uniform = 0;
    // copy-engine work is spread over `ce_lanes` streams forked from and joined back to the
    // caller's stream, so several copy engines run at once
    int ce_lanes = kMaxCeLanes;  // measured on GB300: 1-D copies over 8 streams reach ~0.94 x HBM peak
    int ce_bands = 1;  // 2-D copies per parameter (bands of ranks)
    cudaStream_t lane_stream[kMaxCeLanes] = {};
    cudaEvent_t lane_done[kMaxCeLanes] = {};
    cudaEvent_t fork = nullptr;
    std::mutex mu;
};

namespace {

void release(tide_group* g) {
    if (!g) return;
    for (Slot& s : g->slots) {
        if (s.done) {
            cudaEventSynchronize(s.done);
            cudaEventDestroy(s.done);
        }
        if (s.host) cudaFreeHost(s.host);
        if (s.dev) cudaFree(s.dev);
    }
    for (int i = 0; i < kMaxCeLanes; ++i) {
        if (g->lane_stream[i]) {
            cudaStreamSynchronize(g->lane_stream[i]);
            cudaStreamDestroy(g->lane_stream[i]);
        }
        if (g->lane_done[i]) cudaEventDestroy(g->lane_done[i]);
    }
    if (g->fork) cudaEventDestroy(g->fork);
    if (g->d_rs) cudaFree(g->d_rs);
    if (g->d_rs_piece) cudaFree(g->d_rs_piece);
    if (g->d_rs_bulk) cudaFree(g->d_rs_bulk);
    if (g->d_rs_bulk_piece) cudaFree(g->d_rs_bulk_piece);
    if (g->d_rs_slots) cudaFree(g->d_rs_slots);
    if (g->d_rs_slot_piece) cudaFree(g->d_rs_slot_piece);
    if (g->d_ag_bulk) cudaFree(g->d_ag_bulk);
    if (g->d_status) cudaFree(g->d_status);
    if (g->d_ag) cudaFree(g->d_ag);
    if (g->d_ag_run) cudaFree(g->d_ag_run);
    delete g;
}

int check_device(tide_group* g) {
    int dev = -1;
    TIDE_CUDA(cudaGetDevice(&dev));
    return dev == g->device ? TIDE_OK : TIDE_EINVAL;
}

// Uploads `ptrs` into a ring slot (or finds a slot already holding the same table for the
// same stream) and returns its index.  The caller records slots[k].done after its launch.
int upload_table(tide_group* g, const std::vector<const void*>& ptrs, cudaStream_t stream, int* slot) {
    for (int k = 0; k < kSlots; ++k) {
        Slot& s = g->slots[k];
        if (s.valid && s.stream == stream && s.content == ptrs) {
            s.last_use = ++g->use_clock;
            *slot = k;
            return TIDE_OK;
        }
    }
    // victim: an unused slot, else the least recently used one
    int k = -1;
    for (int i = 0; i < kSlots && k < 0; ++i)
        if (!g->slots[i].valid) k = i;
    if (k < 0) {
        k = 0;
        for (int i = 1; i < kSlots; ++i)
            if (g->slots[i].last_use < g->slots[k].last_use) k = i;
    }
    Slot& s = g->slots[k];
    if (s.pending) TIDE_CUDA(cudaEventSynchronize(s.done));
    s.valid = false;
    std::memcpy(s.host, ptrs.data(), ptrs.size() * sizeof(void*));
    TIDE_CUDA(cudaMemcpyAsync(s.dev, s.host, ptrs.size() * sizeof(void*), cudaMemcpyHostToDevice, stream));
    s.content = ptrs;
    s.stream = stream;
    s.valid = true;
    s.last_use = ++g->use_clock;
    *slot = k;
    return TIDE_OK;
}

int finish_slot(tide_group* g, int k, cudaStream_t stream) {
    Slot& s = g->slots[k];
    TIDE_CUDA(cudaEventRecord(s.done, stream));
    s.pending = true;
    return TIDE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A pointer the kernels dereference element by element must be aligned to its element size
// (2 bytes for bf16, 4 for fp32): anything else would be a misaligned access on the device.
bool elem_aligned(const void* p, unsigned bytes) { return (reinterpret_cast<uintptr_t>(p) & (bytes - 1u)) == 0; }

// Stream-ordered fan-out of copy-engine work: lane 0 is the caller's stream; lanes 1.. are helper
// streams that start after everything already enqueued on the caller's stream and that the
// caller's stream waits for at the end.
struct CeLanes {
    tide_group* g;
    cudaStream_t caller;
    int n = 1;
    std::vector<int64_t> load;

    cudaStream_t lane(int i) const { return i == 0 ? caller : g->lane_stream[i]; }

    int begin() {
        n = g->ce_lanes;
        for (int i = 1; i < n; ++i) {
            if (!g->lane_stream[i]) TIDE_CUDA(cudaStreamCreateWithFlags(&g->lane_stream[i], cudaStreamNonBlocking));
            if (!g->lane_done[i]) TIDE_CUDA(cudaEventCreateWithFlags(&g->lane_done[i], cudaEventDisableTiming));
        }
        if (n > 1) {
            if (!g->fork) TIDE_CUDA(cudaEventCreateWithFlags(&g->fork, cudaEventDisableTiming));
            TIDE_CUDA(cudaEventRecord(g->fork, caller));
            for (int i = 1; i < n; ++i) TIDE_CUDA(cudaStreamWaitEvent(g->lane_stream[i], g->fork, 0));
        }
        load.assign(size_t(n), 0);
        return TIDE_OK;
    }
    // the least loaded lane takes the next copy of `bytes`
    cudaStream_t pick(int64_t bytes) {
        int best = 0;
        for (int i = 1; i < n; ++i)
            if (load[i] < load[best]) best = i;
        load[best] += bytes;
        return lane(best);
    }
    int end() {
        for (int i = 1; i < n; ++i) {
            TIDE_CUDA(cudaEventRecord(g->lane_done[i], g->lane_stream[i]));
            TIDE_CUDA(cudaStreamWaitEvent(caller, g->lane_done[i], 0));
        }
        return TIDE_OK;
    }
};

int default_ctas(const tide_group* g, int per_sm) { return std::max(1, g->sm_count * per_sm); }

// CTA budget of a group created with TIDE_FLAG_OVERLAP: about a ninth of the SMs (16 on a 152-SM
// GB300).  Measured on GB300 beside a single-wave cuBLAS bf16 GEMM (4096 x 4096 x 8192, 4-CTA
// clusters, one CTA per SM): up to 16 resident SM-filling CTAs cost it nothing, 20 cost one tile
// round (~16 %).
int overlap_ctas(const tide_group* g) { return std::max(1, g->sm_count / 9); }

bool overlap_mode(const tide_group* g) { return (g->flags & TIDE_FLAG_OVERLAP) != 0; }

// The placement's CTA count when the caller has not set one.
int ag_default_ctas(const tide_group* g, bool bulk) {
    if (overlap_mode(g)) return overlap_ctas(g);
    return default_ctas(g, bulk ? tide::kAgBulkCtasPerSm : tide::kAgCtasPerSm);
}

int rs_default_ctas(const tide_group* g, bool bulk) {
    if (overlap_mode(g)) return overlap_ctas(g);
    return bulk ? g->sm_count : default_ctas(g, tide::kRsCtasPerSm);
}

// The bulk-copy placement needs 16-byte aligned pointers and moves only runs whose offsets are
// 16-byte compatible (the rest go through three warps per CTA).  TIDE_AG_AUTO takes it when at
// least 90 % of the elements can ride bulk copies and either the CTA count is capped below the SM
// count (a bulk CTA moves far more per SM) or the runs are long (>= 1 M elements on average);
// otherwise the register path, whose CTAs copy every run with the widest vectors its alignment
// allows.  Measured on GB300 at the default grid: bulk 6.7-6.8 TB/s against register 6.5 on the
// Llama-3.1-70B layer (12 M-element runs), register 6.7 against bulk 6.5 on the Qwen3 MoE layer
// (0.2 M) and the Wan sweep at R = 64 (0.4 M).
bool ag_uses_bulk(const tide_group* g, bool aligned) {
    if (!aligned || !g->d_ag_bulk || g->ag_variant == TIDE_AG_REGISTER) return false;
    if (g->ag_variant == TIDE_AG_BULK) return true;
    if (g->plan.ag_vec_elems * 10 < g->plan.U * 9) return false;
    const int capped = g->ag_ctas > 0 ? g->ag_ctas : (overlap_mode(g) ? overlap_ctas(g) : 0);
    if (capped > 0 && capped < g->sm_count) return true;
    return g->plan.ag.empty() || g->plan.U >= int64_t(g->plan.ag.size()) * (int64_t(1) << 20);
}

// Bulk-copy kernel unless the register path is asked for; it needs 16-byte aligned gradient
// pointers (the register path's element-wise fallback covers the rest).  Measured on GB300 it is the faster of
// the two at every CTA count, most of all when the count is capped below the SM count.
// Copy-engine form when the caller fixes none (neither TIDE_FLAG_CE_1D nor TIDE_FLAG_CE_2D): the
// host spends one to two microseconds submitting each copy, so the 1-D form (one copy per (rank,
// parameter) run, up to 6.4 TB/s over 8 lanes, 4.5 over one) is host-bound when runs are short,
// while one strided 2-D copy per parameter holds ~3.5 TB/s on every workload measured on GB300.
// The 1-D form wins while runs average >= 4 MiB (Llama-3.1-70B layer, 24 MB runs: 6.5 against
// 3.7 TB/s; 8B layer, 6 MB: 5.0 against 3.6; Wan R = 8, 5.6 MB: 3.7 against 3.5), the 2-D form below
// (Wan R = 16, 2.8 MB runs: 3.5 against 2.5; Qwen3 MoE layer, 0.4 MB: 2.6 against 0.37).  The same
// rule holds over the one lane of TIDE_FLAG_OVERLAP beside a single-wave GEMM: strided copies of
// long runs slow it far more than 1-D copies (70B layer +144 % against +6 %, 8B +24 % against +5 %,
// Wan R = 8 +13 % against +6 %), those of short runs no more (Wan R = 16 / 32 / 64 +2.6 / +1.4 / +2.1 %,
// Qwen3 +1.8 %) while they move up to 4x as much beside it (Qwen3: 0.75 against 0.19 TB/s).
constexpr int64_t kCeLongRunBytes = int64_t(4) << 20;

bool ce_auto_prefers_2d(const tide_group* g) {
    const int64_t runs = int64_t(g->plan.ag.size());
    return runs > 0 && 2 * g->plan.U < runs * kCeLongRunBytes;
}

bool use_bulk(const tide_group* g, bool aligned) {
    if (!aligned || g->plan.rs_bulk.empty() || !g->d_rs_bulk || !g->d_rs_bulk_piece) return false;
    return g->rs_variant != TIDE_RS_REGISTER;
}

// Which bulk-copy kernel: the TMEM-staged one unless TIDE_RS_BULK asks for the original.  Measured
// on GB300 over every workload: at 16 CTAs the staged kernel moves 1-23 % more (70B layer 2.18
// against 1.79 TB/s; Wan R = 64, where the R rows already spread the stores, 2.13 against 2.12), at
// the default grid within +-1.5 % (70B 7.09 against 7.00).
using RsBulkLaunch = cudaError_t (*)(const tide::RsSeg*, const int32_t*, int64_t, const uint16_t* const*,
                                     float* const*, int, int, int, int, int*, uint64_t, int, cudaStream_t);
RsBulkLaunch rs_bulk_launcher(const tide_group* g) {
    return g->rs_variant == TIDE_RS_BULK ? tide::launch_reduce_scatter_bulk : tide::launch_reduce_scatter_tmem;
}

// Entry points return a status, never an exception: an allocation that fails (host vectors of the
// pointer tables and plans) becomes TIDE_ENOMEM, anything else thrown (a mutex error) TIDE_EINVAL.
template <class F>
int no_throw(F&& f) {
    try {
        return f();
    } catch (const std::bad_alloc&) {
        return TIDE_ENOMEM;
    } catch (...) {
        return TIDE_EINVAL;
    }
}

}  // namespace

extern "C" {

int tide_version(void) { return 100; }

const char* tide_strerror(int status) {
    switch (status) {
        case TIDE_OK: return "success";
        case TIDE_EINVAL: return "invalid argument";
        case TIDE_EALIGN: return "pointer not 16-byte aligned (TIDE_FLAG_VEC_STRICT)";
        case TIDE_ELAYOUT: return "shards not at a uniform pitch (TIDE_FLAG_CE_2D | TIDE_FLAG_CE_STRICT)";
        case TIDE_ECUDA: return "CUDA runtime error (see tide_last_cuda_error)";
        case TIDE_ENOMEM: return "out of memory";
        case TIDE_ERANGE: return "size out of range";
        default: return "unknown status";
    }
}

int tide_last_cuda_error(void) { return g_last_cuda_error; }

int tide_plan_layout(int32_t R, int32_t P, const int64_t* rows, const int64_t* row_len, int64_t* m,
                     int64_t* s, int64_t* o, int64_t* S, int64_t* U) {
    return no_throw([&]() -> int {
        if (!m || !s || !o || !S || !U) return TIDE_EINVAL;
        tide::Plan pl;
        const int rc = tide::make_layout(R, P, rows, row_len, &pl);
        if (rc != TIDE_OK) return rc;
        std::copy(pl.m.begin(), pl.m.end(), m);
        std::copy(pl.s.begin(), pl.s.end(), s);
        std::copy(pl.o.begin(), pl.o.end(), o);
        *S = pl.S;
        *U = pl.U;
        return TIDE_OK;
    });
}

int tide_group_create(tide_group_t* out, int32_t R, int32_t P, const int64_t* rows, const int64_t* row_len,
                      uint32_t flags) {
    return no_throw([&]() -> int {
        if (!out) return TIDE_EINVAL;
        *out = nullptr;
        if (flags & ~kAllFlags) return TIDE_EINVAL;
        if ((flags & TIDE_FLAG_CE_1D) && (flags & (TIDE_FLAG_CE_2D | TIDE_FLAG_CE_STRICT))) return TIDE_EINVAL;
        *out = nullptr;
        tide::Plan pl;
        int rc = tide::make_layout(R, P, rows, row_len, &pl);
        if (rc != TIDE_OK) return rc;
        if (int64_t(R) * P > TIDE_MAX_TABLE) return TIDE_ERANGE;
        try {
            tide::make_work_lists(&pl);
        } catch (const std::bad_alloc&) {
            return TIDE_ENOMEM;
        }

        tide_group* g = new (std::nothrow) tide_group();
        if (!g) return TIDE_ENOMEM;
        g->plan = std::move(pl);
        g->flags = flags;
        if (flags & TIDE_FLAG_OVERLAP) g->ce_lanes = 1;
        cudaError_t e = cudaGetDevice(&g->device);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g->sm_count, cudaDevAttrMultiProcessorCount, g->device);
        if (e != cudaSuccess) {
            release(g);
            return cuda_fail(e);
        }
        const auto& rs = g->plan.rs;
        const auto& ag = g->plan.ag;
        e = cudaMalloc(&g->d_rs, std::max<size_t>(1, rs.size()) * sizeof(tide::RsSeg));
        if (e == cudaSuccess) e = cudaMalloc(&g->d_ag, std::max<size_t>(1, ag.size()) * sizeof(tide::AgSeg));
        if (e == cudaSuccess && !rs.empty())
            e = cudaMemcpy(g->d_rs, rs.data(), rs.size() * sizeof(tide::RsSeg), cudaMemcpyHostToDevice);
        const auto& rsp = g->plan.rs_piece;
        if (e == cudaSuccess && !rsp.empty()) {
            e = cudaMalloc(&g->d_rs_piece, rsp.size() * sizeof(int32_t));
            if (e == cudaSuccess)
                e = cudaMemcpy(g->d_rs_piece, rsp.data(), rsp.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
        }
        if (e == cudaSuccess && !ag.empty())
            e = cudaMemcpy(g->d_ag, ag.data(), ag.size() * sizeof(tide::AgSeg), cudaMemcpyHostToDevice);
        const auto& agr = g->plan.ag_run;
        if (e == cudaSuccess && !agr.empty()) {
            e = cudaMalloc(&g->d_ag_run, agr.size() * sizeof(int32_t));
            if (e == cudaSuccess)
                e = cudaMemcpy(g->d_ag_run, agr.data(), agr.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
        }
        const auto& rb = g->plan.rs_bulk;
        if (e == cudaSuccess && !rb.empty()) {
            e = cudaMalloc(&g->d_rs_bulk, rb.size() * sizeof(tide::RsSeg));
            if (e == cudaSuccess)
                e = cudaMemcpy(g->d_rs_bulk, rb.data(), rb.size() * sizeof(tide::RsSeg), cudaMemcpyHostToDevice);
            const auto& rp = g->plan.rs_bulk_piece;
            if (e == cudaSuccess) e = cudaMalloc(&g->d_rs_bulk_piece, rp.size() * sizeof(int32_t));
            if (e == cudaSuccess)
                e = cudaMemcpy(g->d_rs_bulk_piece, rp.data(), rp.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
        }
        const auto& sl = g->plan.rs_slots;
        const auto& slp = g->plan.rs_slot_piece;
        if (e == cudaSuccess && !sl.empty() && !slp.empty()) {
            e = cudaMalloc(&g->d_rs_slots, sl.size() * sizeof(tide::RsSeg));
            if (e == cudaSuccess)
                e = cudaMemcpy(g->d_rs_slots, sl.data(), sl.size() * sizeof(tide::RsSeg), cudaMemcpyHostToDevice);
            if (e == cudaSuccess) e = cudaMalloc(&g->d_rs_slot_piece, slp.size() * sizeof(int32_t));
            if (e == cudaSuccess)
                e = cudaMemcpy(g->d_rs_slot_piece, slp.data(), slp.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
        }
        const auto& ab = g->plan.ag_bulk;
        if (e == cudaSuccess && !ab.empty()) {
            e = cudaMalloc(&g->d_ag_bulk, ab.size() * sizeof(tide::AgSeg));
            if (e == cudaSuccess)
                e = cudaMemcpy(g->d_ag_bulk, ab.data(), ab.size() * sizeof(tide::AgSeg), cudaMemcpyHostToDevice);
        }
        if (e == cudaSuccess) e = cudaMalloc(&g->d_status, sizeof(int));
        if (e == cudaSuccess) e = cudaMemset(g->d_status, 0, sizeof(int));
        // a table holds the R*P gradient pointers + R shard pointers (reduce-scatter) or R + P
        // pointers (all-gather)
        g->slot_cap = size_t(R) * P + R + P;
        for (Slot& s : g->slots) {
            if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void**>(&s.host), g->slot_cap * sizeof(void*), cudaHostAllocDefault);
            if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&s.dev), g->slot_cap * sizeof(void*));
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming);
        }
        if (e != cudaSuccess) {
            release(g);
            return e == cudaErrorMemoryAllocation ? (g_last_cuda_error = int(e), TIDE_ENOMEM) : cuda_fail(e);
        }
        *out = g;
        return TIDE_OK;
    });
}

int tide_group_destroy(tide_group_t g) {
    if (!g) return TIDE_OK;
    release(g);
    return TIDE_OK;
}

int tide_group_shard_elems(tide_group_t g, int64_t* S) {
    if (!g || !S) return TIDE_EINVAL;
    *S = g->plan.S;
    return TIDE_OK;
}

int tide_group_unsharded_elems(tide_group_t g, int64_t* U) {
    if (!g || !U) return TIDE_EINVAL;
    *U = g->plan.U;
    return TIDE_OK;
}

int tide_group_param_layout(tide_group_t g, int32_t p, int64_t* m_p, int64_t* o_p) {
    if (!g || !m_p || !o_p || p < 0 || p >= g->plan.P) return TIDE_EINVAL;
    *m_p = g->plan.m[p];
    *o_p = g->plan.o[p];
    return TIDE_OK;
}

int tide_group_valid_rows(tide_group_t g, int32_t d, int32_t p, int64_t* v) {
    if (!g || !v || p < 0 || p >= g->plan.P || d < 0 || d >= g->plan.R) return TIDE_EINVAL;
    *v = tide::valid_rows(g->plan.rows[p], g->plan.m[p], d);
    return TIDE_OK;
}

int tide_group_set_ctas(tide_group_t g, int32_t rs_ctas, int32_t ag_ctas) {
    if (!g || rs_ctas < 0 || ag_ctas < 0) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    g->rs_ctas = rs_ctas;
    g->ag_ctas = ag_ctas;
    return TIDE_OK;
}

int tide_group_get_ctas(tide_group_t g, int32_t* rs_ctas, int32_t* ag_ctas) {
    if (!g || !rs_ctas || !ag_ctas) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    *rs_ctas = g->rs_ctas ? g->rs_ctas : rs_default_ctas(g, g->rs_variant != TIDE_RS_REGISTER);
    *ag_ctas = g->ag_ctas ? g->ag_ctas : ag_default_ctas(g, ag_uses_bulk(g, true));
    return TIDE_OK;
}

int tide_reduce_scatter(tide_group_t g, const void* const* grads, void* const* shards, void* stream) {
    return no_throw([&]() -> int {
        if (!g || !grads || !shards) return TIDE_EINVAL;
        std::lock_guard<std::mutex> lock(g->mu);
        const int R = g->plan.R, P = g->plan.P;
        std::vector<const void*> table(size_t(R) * P + R);
        bool aligned = true;
        for (size_t i = 0; i < size_t(R) * P; ++i) {
            if (!grads[i] || !elem_aligned(grads[i], 2)) return TIDE_EINVAL;
            table[i] = grads[i];
            aligned &= aligned16(grads[i]);
        }
        // the kernels store the sums with whatever vectors each shard address allows, so only the
        // gradients' alignment decides between the vector paths and the element-wise one
        for (int d = 0; d < R; ++d) {
            if (!shards[d] || !elem_aligned(shards[d], 4)) return TIDE_EINVAL;
            table[size_t(R) * P + d] = shards[d];
        }
        if (!aligned && (g->flags & TIDE_FLAG_VEC_STRICT)) return TIDE_EALIGN;
        int rc = check_device(g);
        if (rc != TIDE_OK) return rc;
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        int k = 0;
        if ((rc = upload_table(g, table, st, &k)) != TIDE_OK) return rc;
        void** dev = g->slots[k].dev;
        const auto* gp = reinterpret_cast<const uint16_t* const*>(dev);
        auto* sp = reinterpret_cast<float* const*>(dev + size_t(R) * P);
        cudaError_t e;
        if (use_bulk(g, aligned)) {
            const int ctas = g->rs_ctas ? g->rs_ctas : rs_default_ctas(g, true);
            auto* launch = rs_bulk_launcher(g);
            e = launch(g->d_rs_bulk, g->d_rs_bulk_piece, g->plan.rs_bulk_chunks, gp, sp, R, P, 1, ctas, g->d_status,
                       g->timeout_ns, (g->debug & TIDE_DEBUG_STALL_PRODUCER) ? 1 : 0, st);
        } else {
            const int ctas = g->rs_ctas ? g->rs_ctas : rs_default_ctas(g, false);
            e = tide::launch_reduce_scatter(g->d_rs, int(g->plan.rs.size()), g->d_rs_piece, g->plan.rs_chunks, gp, sp,
                                            R, P, aligned ? 1 : 0, ctas, st);
        }
        if (e != cudaSuccess) return cuda_fail(e);
        return finish_slot(g, k, st);
    });
}

int tide_reduce_scatter_slots(tide_group_t g, int32_t d, const void* const* slots, void* shard, void* stream) {
    return no_throw([&]() -> int {
        if (!g || !slots || !shard) return TIDE_EINVAL;
        std::lock_guard<std::mutex> lock(g->mu);
        const int R = g->plan.R, P = g->plan.P;
        if (d < 0 || d >= R || !elem_aligned(shard, 4)) return TIDE_EINVAL;
        std::vector<const void*> table(size_t(R) + 1);
        bool aligned = true;
        for (int r = 0; r < R; ++r) {
            if (!slots[r] || !elem_aligned(slots[r], 2)) return TIDE_EINVAL;
            table[size_t(r)] = slots[r];
            aligned &= aligned16(slots[r]);
        }
        table[size_t(R)] = shard;
        if (!aligned && (g->flags & TIDE_FLAG_VEC_STRICT)) return TIDE_EALIGN;
        if (!g->d_rs_slots || !g->d_rs_slot_piece) return TIDE_EINVAL;
        int rc = check_device(g);
        if (rc != TIDE_OK) return rc;
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        int k = 0;
        if ((rc = upload_table(g, table, st, &k)) != TIDE_OK) return rc;
        void** dev = g->slots[k].dev;
        // one table entry per slot and one shard: the pieces carry p = 0 and d = 0
        const auto* gp = reinterpret_cast<const uint16_t* const*>(dev);
        auto* sp = reinterpret_cast<float* const*>(dev + R);
        const int ctas = g->rs_ctas ? g->rs_ctas : rs_default_ctas(g, true);
        auto* launch = rs_bulk_launcher(g);
        cudaError_t e = launch(g->d_rs_slots + size_t(d) * size_t(P), g->d_rs_slot_piece, g->plan.rs_slot_chunks, gp, sp,
                               R, 1, aligned ? 1 : 0, ctas, g->d_status, g->timeout_ns,
                               (g->debug & TIDE_DEBUG_STALL_PRODUCER) ? 1 : 0, st);
        if (e != cudaSuccess) return cuda_fail(e);
        return finish_slot(g, k, st);
    });
}

int tide_all_gather(tide_group_t g, const void* const* shards, void* const* params, void* stream) {
    return no_throw([&]() -> int {
        if (!g || !shards || !params) return TIDE_EINVAL;
        std::lock_guard<std::mutex> lock(g->mu);
        const int R = g->plan.R, P = g->plan.P;
        std::vector<const void*> table(size_t(R) + P);
        bool aligned = true;
        for (int r = 0; r < R; ++r) {
            if (!shards[r] || !elem_aligned(shards[r], 2)) return TIDE_EINVAL;
            table[r] = shards[r];
            aligned &= aligned16(shards[r]);
        }
        for (int p = 0; p < P; ++p) {
            if (!params[p] || !elem_aligned(params[p], 2)) return TIDE_EINVAL;
            table[size_t(R) + p] = params[p];
            aligned &= aligned16(params[p]);
        }
        if (!aligned && (g->flags & TIDE_FLAG_VEC_STRICT)) return TIDE_EALIGN;
        int rc = check_device(g);
        if (rc != TIDE_OK) return rc;
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        int k = 0;
        if ((rc = upload_table(g, table, st, &k)) != TIDE_OK) return rc;
        void** dev = g->slots[k].dev;
        const auto* sp = reinterpret_cast<const uint16_t* const*>(dev);
        auto* pp = reinterpret_cast<uint16_t* const*>(dev + R);
        cudaError_t e;
        if (ag_uses_bulk(g, aligned)) {
            const int ctas = g->ag_ctas ? g->ag_ctas : ag_default_ctas(g, true);
            e = tide::launch_all_gather_bulk(g->d_ag_bulk, int(g->plan.ag_bulk.size()), g->plan.ag_bulk_chunks, sp, pp,
                                             ctas, g->d_status, g->timeout_ns, st);
        } else {
            const int ctas = g->ag_ctas ? g->ag_ctas : ag_default_ctas(g, false);
            e = tide::launch_all_gather(g->d_ag, int(g->plan.ag.size()), g->d_ag_run, g->plan.ag_chunks, sp, pp,
                                        aligned ? 1 : 0, ctas, st);
        }
        if (e != cudaSuccess) return cuda_fail(e);
        return finish_slot(g, k, st);
    });
}

int tide_all_gather_ce(tide_group_t g, const void* const* shards, void* const* params, void* stream) {
    return no_throw([&]() -> int {
        if (!g || !shards || !params) return TIDE_EINVAL;
        std::lock_guard<std::mutex> lock(g->mu);
        const tide::Plan& pl = g->plan;
        const int R = pl.R, P = pl.P;
        for (int r = 0; r < R; ++r)
            if (!shards[r]) return TIDE_EINVAL;
        for (int p = 0; p < P; ++p)
            if (!params[p]) return TIDE_EINVAL;
        // Uniform pitch: shards[r] = shards[0] + r * pitch with pitch >= S*2 bytes.
        const char* base = static_cast<const char*>(shards[0]);
        const int64_t pitch = R > 1 ? static_cast<const char*>(shards[1]) - base : pl.S * 2;
        bool uniform = pitch >= pl.S * 2;
        for (int r = 1; r < R && uniform; ++r) uniform = static_cast<const char*>(shards[r]) == base + int64_t(r) * pitch;
        if (g->flags & TIDE_FLAG_CE_2D) {
            if (!uniform && (g->flags & TIDE_FLAG_CE_STRICT)) return TIDE_ELAYOUT;
        } else if ((g->flags & TIDE_FLAG_CE_1D) || !ce_auto_prefers_2d(g)) {
            uniform = false;  // one 1-D copy per (rank, parameter) run
        }
        int rc = check_device(g);
        if (rc != TIDE_OK) return rc;
        CeLanes lanes{g, static_cast<cudaStream_t>(stream)};
        if ((rc = lanes.begin()) != TIDE_OK) return rc;
        int64_t copies = 0;
        for (int p = 0; p < P; ++p) {
            char* dst = static_cast<char*>(params[p]);
            const int64_t piece_bytes = pl.s[p] * 2;
            if (uniform) {
                // ranks 0 .. f-1 hold full pieces of m_p rows: one 2-D copy per band of ranks (one band
                // by default: the whole parameter in one strided copy), source rows `pitch` apart,
                // destination rows contiguous
                const int64_t f = pl.rows[p] / pl.m[p];
                const int64_t nb = std::min<int64_t>(g->ce_bands, f);
                for (int64_t b = 0; b < nb; ++b) {
                    const int64_t r0 = f * b / nb, r1 = f * (b + 1) / nb;
                    TIDE_LANE_COPY(lanes, cudaMemcpy2DAsync(dst + r0 * piece_bytes, size_t(piece_bytes),
                                                            base + r0 * pitch + pl.o[p] * 2, size_t(pitch),
                                                            size_t(piece_bytes), size_t(r1 - r0), cudaMemcpyDeviceToDevice,
                                                            lanes.pick((r1 - r0) * piece_bytes)));
                    ++copies;
                }
                const int64_t rest = pl.rows[p] - f * pl.m[p];
                if (rest > 0) {
                    const int64_t bytes = rest * pl.row_len[p] * 2;
                    TIDE_LANE_COPY(lanes, cudaMemcpyAsync(dst + f * piece_bytes, base + f * pitch + pl.o[p] * 2,
                                                          size_t(bytes), cudaMemcpyDeviceToDevice, lanes.pick(bytes)));
                    ++copies;
                }
            } else {
                for (int r = 0; r < R; ++r) {
                    const int64_t v = tide::valid_rows(pl.rows[p], pl.m[p], r);
                    if (v == 0) continue;
                    const int64_t bytes = v * pl.row_len[p] * 2;
                    TIDE_LANE_COPY(lanes, cudaMemcpyAsync(dst + r * piece_bytes,
                                                          static_cast<const char*>(shards[r]) + pl.o[p] * 2, size_t(bytes),
                                                          cudaMemcpyDeviceToDevice, lanes.pick(bytes)));
                    ++copies;
                }
            }
        }
        if ((rc = lanes.end()) != TIDE_OK) return rc;
        g->last_ce_copies = copies;
        g->last_ce_uniform = uniform ? 1 : 0;
        return TIDE_OK;
    });
}

int tide_group_set_rs_variant(tide_group_t g, int32_t variant) {
    if (!g || variant < TIDE_RS_AUTO || variant > TIDE_RS_TMEM) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    g->rs_variant = variant;
    return TIDE_OK;
}

int tide_group_rs_kernel(tide_group_t g, int32_t* variant) {
    if (!g || !variant) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    if (!use_bulk(g, true)) *variant = TIDE_RS_REGISTER;
    else *variant = rs_bulk_launcher(g) == tide::launch_reduce_scatter_tmem ? TIDE_RS_TMEM : TIDE_RS_BULK;
    return TIDE_OK;
}

int tide_group_ag_kernel(tide_group_t g, int32_t* variant) {
    if (!g || !variant) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    *variant = ag_uses_bulk(g, true) ? TIDE_AG_BULK : TIDE_AG_REGISTER;
    return TIDE_OK;
}

int tide_group_set_ce_lanes(tide_group_t g, int32_t lanes) {
    if (!g || lanes < 1 || lanes > kMaxCeLanes) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    g->ce_lanes = lanes;
    return TIDE_OK;
}

int tide_group_set_ce_bands(tide_group_t g, int32_t bands) {
    if (!g || bands < 1 || bands > TIDE_MAX_RANKS) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    g->ce_bands = bands;
    return TIDE_OK;
}

int tide_group_set_ag_variant(tide_group_t g, int32_t variant) {
    if (!g || variant < TIDE_AG_AUTO || variant > TIDE_AG_BULK) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    g->ag_variant = variant;
    return TIDE_OK;
}

int tide_group_set_wait_timeout(tide_group_t g, uint64_t timeout_ns) {
    if (!g) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    g->timeout_ns = timeout_ns ? std::max(timeout_ns, tide::kMinTimeoutNs) : tide::kDefaultTimeoutNs;
    return TIDE_OK;
}

int tide_group_set_debug(tide_group_t g, uint32_t flags) {
    if (!g || (flags & ~uint32_t(TIDE_DEBUG_STALL_PRODUCER))) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    g->debug = flags;
    return TIDE_OK;
}

int tide_group_device_status(tide_group_t g, int32_t* status) {
    if (!g || !status) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    int rc = check_device(g);
    if (rc != TIDE_OK) return rc;
    int v = 0;
    TIDE_CUDA(cudaMemcpy(&v, g->d_status, sizeof(int), cudaMemcpyDeviceToHost));
    if (v) TIDE_CUDA(cudaMemset(g->d_status, 0, sizeof(int)));
    *status = v;
    return TIDE_OK;
}

int tide_stage_into_slots(tide_group_t g, const void* const* grads, void* const* slots, int64_t slot_elems,
                          void** staged, void* stream) {
    return no_throw([&]() -> int {
        if (!g || !grads || !slots || !staged) return TIDE_EINVAL;
        std::lock_guard<std::mutex> lock(g->mu);
        const tide::Plan& pl = g->plan;
        const int R = pl.R, P = pl.P;
        if (slot_elems < pl.U) return TIDE_ERANGE;
        for (size_t i = 0; i < size_t(R) * P; ++i)
            if (!grads[i]) return TIDE_EINVAL;
        for (int r = 0; r < R; ++r)
            if (!slots[r]) return TIDE_EINVAL;
        int rc = check_device(g);
        if (rc != TIDE_OK) return rc;
        CeLanes lanes{g, static_cast<cudaStream_t>(stream)};
        if ((rc = lanes.begin()) != TIDE_OK) return rc;
        // parameter p of rank r lands at slot_r + (rows_0*L_0 + ... + rows_{p-1}*L_{p-1}) elements:
        // the unsharded group, packed without padding, 16-byte aligned when every size is a multiple of 8
        int64_t off = 0;
        for (int p = 0; p < P; ++p) {
            const int64_t n = pl.rows[p] * pl.row_len[p];
            for (int r = 0; r < R; ++r) {
                char* dst = static_cast<char*>(slots[r]) + off * 2;
                TIDE_LANE_COPY(lanes, cudaMemcpyAsync(dst, grads[size_t(r) * P + p], size_t(n) * 2,
                                                      cudaMemcpyDeviceToDevice, lanes.pick(n * 2)));
                staged[size_t(r) * P + p] = dst;
            }
            off += n;
        }
        return lanes.end();
    });
}

int tide_stage_slices(tide_group_t g, int32_t d, const void* const* grads, void* const* slots, void* stream) {
    return no_throw([&]() -> int {
        if (!g || !grads || !slots) return TIDE_EINVAL;
        std::lock_guard<std::mutex> lock(g->mu);
        const tide::Plan& pl = g->plan;
        const int R = pl.R, P = pl.P;
        if (d < 0 || d >= R) return TIDE_EINVAL;
        for (size_t i = 0; i < size_t(R) * P; ++i)
            if (!grads[i] || !elem_aligned(grads[i], 2)) return TIDE_EINVAL;
        for (int r = 0; r < R; ++r)
            if (!slots[r] || !elem_aligned(slots[r], 2)) return TIDE_EINVAL;
        int rc = check_device(g);
        if (rc != TIDE_OK) return rc;
        CeLanes lanes{g, static_cast<cudaStream_t>(stream)};
        if ((rc = lanes.begin()) != TIDE_OK) return rc;
        // contributors d+1, ..., R-1, 0, ..., d; within one, parameters in order
        for (int k = 1; k <= R; ++k) {
            const int r = (d + k) % R;
            for (int p = 0; p < P; ++p) {
                const int64_t n = tide::valid_rows(pl.rows[p], pl.m[p], d) * pl.row_len[p];
                if (n == 0) continue;
                const char* src = static_cast<const char*>(grads[size_t(r) * P + p]) + int64_t(d) * pl.s[p] * 2;
                char* dst = static_cast<char*>(slots[r]) + pl.o[p] * 2;
                TIDE_LANE_COPY(lanes, cudaMemcpyAsync(dst, src, size_t(n) * 2, cudaMemcpyDeviceToDevice, lanes.pick(n * 2)));
            }
        }
        return lanes.end();
    });
}

int tide_group_last_ce_copies(tide_group_t g, int64_t* copies, int32_t* uniform_pitch) {
    if (!g || !copies || !uniform_pitch) return TIDE_EINVAL;
    std::lock_guard<std::mutex> lock(g->mu);
    *copies = g->last_ce_copies;
    *uniform_pitch = g->last_ce_uniform;
    return TIDE_OK;
}

}  // extern "C"
