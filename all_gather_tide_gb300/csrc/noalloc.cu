// tide_reduce_scatter_noalloc: the reduce-scatter for callers that must not allocate memory.
//
// The group API keeps its work tables in memory it allocates (cudaMalloc for the piece table and
// the pointer-table ring, cudaHostAlloc for the pinned staging slots).  Some callers cannot do
// that: a framework whose caching allocator has already reserved almost all device memory and
// routes every allocation through itself, or a communication path that runs next to compute and
// cannot afford cudaMalloc/cudaFree, which may synchronise the whole device.  This entry point
// plans the group on the host on every call and places the kernel's work tables (the piece table
// and the device pointer table) in one fixed array in device memory that the library carries in
// its image, so no allocation routine is called on the device side.
#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/tide.h"
#include "tide_internal.h"

namespace {

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[TIDE_NOALLOC_SCRATCH_BYTES];

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

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" int tide_reduce_scatter_noalloc(int32_t R, int32_t P, const int64_t* rows, const int64_t* row_len,
                                           const void* const* grads, void* const* shards, void* stream) {
    if (!grads || !shards) return TIDE_EINVAL;
    tide::Plan pl;
    int rc = tide::make_layout(R, P, rows, row_len, &pl);
    if (rc != TIDE_OK) return rc;
    // scratch layout: [piece table, 256-byte aligned][R*P gradient pointers][R shard pointers]
    const size_t npieces = size_t(R) * size_t(P);
    const size_t seg_bytes = round_up(npieces * sizeof(tide::RsSeg), 256);
    const size_t need = seg_bytes + (npieces + size_t(R)) * sizeof(void*);
    if (need > TIDE_NOALLOC_SCRATCH_BYTES) return TIDE_ERANGE;
    tide::make_work_lists(&pl);

    bool aligned = true;
    std::vector<unsigned char> staging(need);
    const void** table = reinterpret_cast<const void**>(staging.data() + seg_bytes);
    for (size_t i = 0; i < npieces; ++i) {
        if (!grads[i] || (reinterpret_cast<uintptr_t>(grads[i]) & 1u)) return TIDE_EINVAL;
        table[i] = grads[i];
        aligned &= (reinterpret_cast<uintptr_t>(grads[i]) & 15u) == 0;
    }
    for (int d = 0; d < R; ++d) {
        if (!shards[d] || (reinterpret_cast<uintptr_t>(shards[d]) & 3u)) return TIDE_EINVAL;
        table[npieces + d] = shards[d];  // any fp32 alignment: the kernel picks its store width
    }
    std::copy(reinterpret_cast<const unsigned char*>(pl.rs.data()),
              reinterpret_cast<const unsigned char*>(pl.rs.data() + pl.rs.size()), staging.begin());

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return tide::record_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return TIDE_EINVAL;
    void* scratch = nullptr;
    int sms = 0;
    if ((e = setup_device(dev, &scratch, &sms)) != cudaSuccess) return tide::record_cuda_error(e);

    // Stream-ordered: the tables land after every earlier call's kernel on this stream has read
    // its own.  The copy is from pageable memory, so `staging` may be freed once it returns.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = cudaMemcpyAsync(scratch, staging.data(), need, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return tide::record_cuda_error(e);
    unsigned char* base = static_cast<unsigned char*>(scratch);
    e = tide::launch_reduce_scatter(reinterpret_cast<const tide::RsSeg*>(base), int(pl.rs.size()), nullptr,
                                    pl.rs_chunks,
                                    reinterpret_cast<const uint16_t* const*>(base + seg_bytes),
                                    reinterpret_cast<float* const*>(base + seg_bytes + npieces * sizeof(void*)), R,
                                    P, aligned ? 1 : 0, sms * tide::kRsCtasPerSm, st);
    return e == cudaSuccess ? TIDE_OK : tide::record_cuda_error(e);
}
