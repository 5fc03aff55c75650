// Interference probes (measurement kernels of the interference harness).
//
// Paper: "The Endgame of FSDP Communication" (arXiv 2610.38228).  Fig. 4 measures how a GEMM slows
// as spin kernels keep a growing number of CTAs resident; Table 5 (and Fig. 3) use an SM-id probe:
// CTAs shaped like the GEMM's clusters, each occupying a whole SM, write down the SM number and
// the arrival and departure times, so CTAs displaced past the first wave, and the SMs a collective keeps, can be counted.
// A third probe measures how fast one SM's bulk-copy engine reads as a function of the copy size,
// the fact the bulk-copy reduce-scatter is built around.
//
// Every loop here is bounded by %globaltimer or by the buffer size; nothing waits on another launch.
#include <algorithm>

#include "../../include/tide.h"
#include "tide_internal.h"

namespace tide {
namespace {

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smid() {
    uint32_t s;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
    return s;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Keeps its SM busy for `hold_ns`; thread 0 records (SM id, entry ns, exit ns) when `rec` is set.
// Besides the shared memory the launch gives it, each thread keeps kLive values live, so a
// 1024-thread CTA also claims the whole register file, as a GEMM CTA with 255 registers x 256
// threads does: no other kernel's CTA can share its SM.
constexpr int kLive = 56;
__global__ void __launch_bounds__(1024, 1) hold_kernel(uint64_t hold_ns, uint64_t* rec) {
    extern __shared__ unsigned char pad[];  // sized by the launch to claim shared memory
    const uint64_t t0 = now_ns();
    uint32_t live[kLive];
#pragma unroll
    for (int i = 0; i < kLive; ++i) live[i] = threadIdx.x * (i + 1);
    while (now_ns() - t0 < hold_ns) {
#pragma unroll
        for (int i = 0; i < kLive; ++i) live[i] = live[i] * 1664525u + 1013904223u;
    }
    uint32_t x = 0;
#pragma unroll
    for (int i = 0; i < kLive; ++i) x ^= live[i];
    if (x == 0x9e3779b9u) pad[0] = 1;  // keeps the values live; the store almost never happens
    if (rec && threadIdx.x == 0) {
        const uint64_t cta = blockIdx.x;
        rec[3 * cta + 0] = smid();
        rec[3 * cta + 1] = t0;
        rec[3 * cta + 2] = now_ns();
    }
}

// Reads [buf, buf + bytes) with `copy_bytes` bulk copies through `stages` shared-memory slots;
// thread 0 issues, thread 32 consumes.  XOR of the first word of every copy goes to *out so the
// reads cannot be dropped.  Waits are bounded (error flag in out[1]).
__global__ void bulk_read_kernel(const unsigned char* __restrict__ buf, int64_t bytes, int copy_bytes, int stages,
                                 uint32_t* out) {
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(sm);
    uint64_t* empty = full + stages;
    unsigned char* data = sm + 1024;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&full[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&empty[s])));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int64_t nchunk = bytes / copy_bytes;
    const uint64_t limit = 1000000000ull;  // 1 s per wait
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        const uint64_t t0 = now_ns();
        uint32_t ok = 0;
        while (true) {
            asm volatile(
                "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(ok)
                : "r"(smem_u32(bar)), "r"(parity)
                : "memory");
            if (ok) return true;
            if (now_ns() - t0 > limit) return false;
        }
    };
    if (threadIdx.x == 0) {
        int64_t k = 0;
        for (int64_t c = blockIdx.x; c < nchunk; c += gridDim.x, ++k) {
            const int s = int(k % stages);
            if (!wait(&empty[s], uint32_t(((k / stages) & 1) ^ 1))) {
                atomicOr(&out[1], 1u);
                break;
            }
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&full[s])),
                         "r"(copy_bytes)
                         : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(data + int64_t(s) * copy_bytes)),
                "l"(buf + c * copy_bytes), "r"(copy_bytes), "r"(smem_u32(&full[s]))
                : "memory");
        }
        // every issued copy must land before the CTA exits
        for (int64_t j = k > stages ? k - stages : 0; j < k; ++j)
            if (!wait(&full[j % stages], uint32_t((j / stages) & 1))) atomicOr(&out[1], 2u);
    } else if (threadIdx.x == 32) {
        uint32_t x = 0;
        int64_t k = 0;
        for (int64_t c = blockIdx.x; c < nchunk; c += gridDim.x, ++k) {
            const int s = int(k % stages);
            if (!wait(&full[s], uint32_t((k / stages) & 1))) {
                atomicOr(&out[1], 4u);
                break;
            }
            x ^= *reinterpret_cast<const uint32_t*>(data + int64_t(s) * copy_bytes);
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty[s])) : "memory");
        }
        atomicXor(&out[0], x);
    }
}

}  // namespace
}  // namespace tide

extern "C" {

int tide_probe_hold(int32_t ctas, int32_t threads, int32_t smem_bytes, int32_t cluster_size, uint64_t hold_ns,
                    uint64_t* records, void* stream) {
    if (ctas < 1 || threads < 1 || threads > 1024 || smem_bytes < 0 || cluster_size < 1 || cluster_size > 8 ||
        ctas % cluster_size || hold_ns > 10000000000ull)
        return TIDE_EINVAL;
    cudaError_t e = cudaFuncSetAttribute(tide::hold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         std::max(smem_bytes, 1));
    if (e != cudaSuccess) return tide::record_cuda_error(e);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(ctas));
    cfg.blockDim = dim3(unsigned(threads));
    cfg.dynamicSmemBytes = size_t(std::max(smem_bytes, 1));
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cluster_size);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cluster_size > 1 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, tide::hold_kernel, hold_ns, records);
    return e == cudaSuccess ? TIDE_OK : tide::record_cuda_error(e);
}

int tide_probe_bulk_read(const void* buf, int64_t bytes, int32_t ctas, int32_t copy_bytes, int32_t stages,
                         uint32_t* out, void* stream) {
    if (!buf || !out || bytes < 0 || ctas < 1 || copy_bytes < 16 || copy_bytes % 16 || stages < 2 || stages > 64 ||
        (reinterpret_cast<uintptr_t>(buf) & 15u) || int64_t(copy_bytes) * stages > 200 * 1024)
        return TIDE_EINVAL;
    const int smem = 1024 + copy_bytes * stages;
    cudaError_t e = cudaFuncSetAttribute(tide::bulk_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return tide::record_cuda_error(e);
    tide::bulk_read_kernel<<<ctas, 64, smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const unsigned char*>(buf), bytes, copy_bytes, stages, out);
    e = cudaGetLastError();
    return e == cudaSuccess ? TIDE_OK : tide::record_cuda_error(e);
}

}  // extern "C"
