// tide_reduce_scatter_noalloc: the reduce-scatter for callers that must not allocate memory.
//
// The group API keeps its work tables in memory it allocates (cudaMalloc for the piece table and
// the pointer-table ring, cudaHostAlloc for the pinned staging slots).  Some callers cannot do
// that: a framework whose caching allocator has already reserved almost all device memory and
// routes every allocation through itself, or a communication path that runs next to compute and
// cannot afford cudaMalloc/cudaFree, which may synchronise the whole device.  This entry point
// plans the group on the host on every call, straight into a fixed host staging array (no heap
// allocation), and places the kernel's work tables (the piece table and the device pointer table)
// in one fixed array in device memory that the library carries in its image, so no allocation
// routine is called at all.
#include <algorithm>
#include <mutex>
#include <new>

#include "../../include/tide.h"
#include "tide_internal.h"

namespace {

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TIDE_NOALLOC_SCRATCH_BYTES];

// Host image of the tables, written under g_stage_mu and copied to the device array by a
// stream-ordered copy from pageable memory: cudaMemcpyAsync returns only once it has taken the
// bytes, so the next call may rewrite this array as soon as the previous copy call has returned.
alignas(256) unsigned char g_host_stage[TIDE_NOALLOC_SCRATCH_BYTES];
std::mutex g_stage_mu;

constexpr int kMaxDevices = 256;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device
int g_sm_count[kMaxDevices];

// Once per device, with that device current: look up the array's device address.  In host
// code the name g_noalloc_scratch is only a host-side stand-in for the symbol, never an address
// a kernel may use.
cudaError_t setup_device(int dev, void** addr, int* sms) {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_sm_count[dev] = n;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    *sms = g_sm_count[dev];
    return cudaSuccess;
}

constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int reduce_scatter_noalloc(int32_t R, int32_t P, const int64_t* rows, const int64_t* row_len,
                           const void* const* grads, void* const* shards, void* stream) {
    if (!grads || !shards || !rows || !row_len || R < 1 || R > TIDE_MAX_RANKS || P < 1) return TIDE_EINVAL;
    // scratch layout: [piece table, 256-byte aligned][R*P gradient pointers][R shard pointers]
    const size_t npieces = size_t(R) * size_t(P);
    if (npieces > TIDE_NOALLOC_SCRATCH_BYTES / sizeof(tide::RsSeg)) return TIDE_ERANGE;
    const size_t seg_bytes = round_up(npieces * sizeof(tide::RsSeg), 256);
    const size_t need = seg_bytes + (npieces + size_t(R)) * sizeof(void*);
    if (need > TIDE_NOALLOC_SCRATCH_BYTES) return TIDE_ERANGE;

    bool aligned = true;
    for (size_t i = 0; i < npieces; ++i) {
        if (!grads[i] || (reinterpret_cast<uintptr_t>(grads[i]) & 1u)) return TIDE_EINVAL;
        aligned &= (reinterpret_cast<uintptr_t>(grads[i]) & 15u) == 0;
    }
    for (int d = 0; d < R; ++d)  // any fp32 alignment: the kernel picks its store width
        if (!shards[d] || (reinterpret_cast<uintptr_t>(shards[d]) & 3u)) return TIDE_EINVAL;

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tide::record_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return TIDE_EINVAL;
    void* scratch = nullptr;
    int sms = 0;
    if ((e = setup_device(dev, &scratch, &sms)) != cudaSuccess) return tide::record_cuda_error(e);

    std::lock_guard<std::mutex> lock(g_stage_mu);
    auto* segs = reinterpret_cast<tide::RsSeg*>(g_host_stage);
    int64_t nchunks = 0;
    const int rc = tide::plan_rs_pieces(R, P, rows, row_len, segs, npieces, &nchunks);
    if (rc != TIDE_OK) return rc;
    const void** table = reinterpret_cast<const void**>(g_host_stage + seg_bytes);
    std::copy(grads, grads + npieces, table);
    std::copy(shards, shards + R, table + npieces);

    // Stream-ordered: the tables land after every earlier call's kernel on this stream has read
    // its own.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = cudaMemcpyAsync(scratch, g_host_stage, need, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return tide::record_cuda_error(e);
    unsigned char* base = static_cast<unsigned char*>(scratch);
    e = tide::launch_reduce_scatter(reinterpret_cast<const tide::RsSeg*>(base), int(npieces), nullptr, nchunks,
                                    reinterpret_cast<const uint16_t* const*>(base + seg_bytes),
                                    reinterpret_cast<float* const*>(base + seg_bytes + npieces * sizeof(void*)), R,
                                    P, aligned ? 1 : 0, sms * tide::kRsCtasPerSm, st);
    return e == cudaSuccess ? TIDE_OK : tide::record_cuda_error(e);
}

}  // namespace

extern "C" int tide_reduce_scatter_noalloc(int32_t R, int32_t P, const int64_t* rows, const int64_t* row_len,
                                           const void* const* grads, void* const* shards, void* stream) {
    // Nothing here allocates; the only exceptions the host runtime can still raise come from
    // locking a mutex (std::system_error when the system is out of resources).  None may cross
    // the C boundary.
    try {
        return reduce_scatter_noalloc(R, P, rows, row_len, grads, shards, stream);
    } catch (const std::bad_alloc&) {
        return TIDE_ENOMEM;
    } catch (...) {
        return TIDE_ENOMEM;
    }
}
