// Interference probes (measurement kernels of the interference harness).
//
// Paper: "The Endgame of FSDP Communication" (arXiv 2610.38228).  Fig. 4 measures how a GEMM slows
// as spin kernels keep a growing number of CTAs resident; Table 5 (and Fig. 3) use an SM-id probe:
// CTAs shaped like the GEMM's clusters, each occupying a whole SM, write down the SM number and
// the arrival and departure times, so CTAs displaced past the first wave, and the SMs a collective keeps, can be counted.
// A third probe measures how fast one SM's bulk-copy engine reads as a function of the copy size,
// the fact the bulk-copy reduce-scatter is built around; a fourth how many bytes per second one SM
// can bring in at all (bulk copies read out of shared memory, wide register loads, or both at once),
// which bounds any reduce-scatter that may hold only a few SMs.
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

// 32-byte streaming register load (eight 32-bit words).
struct W8 {
    uint32_t w[8];
};
__device__ __forceinline__ void ld32(const unsigned char* p, W8& r) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]), "=r"(r.w[6]),
                   "=r"(r.w[7])
                 : "l"(p));
}

constexpr int kIngestLoads = 8;  // register loads in flight per thread

// Warp 0 lane 0 streams [buf, buf + bulk_bytes) through `stages` slots of `copy_bytes` bulk copies
// (the CTAs' copies a grid stride apart); warps 1..consumers read every 16-byte word of a landed
// slot (`read_all`) or only its first word, then release it; the next `ldg_warps` warps stream
// [ldg, ldg + ldg_bytes) with 32-byte loads, kIngestLoads in flight per thread.  Every wait is
// bounded (1 s): on expiry out[1] gets a flag and the CTA winds down after its copies have landed.
__global__ void __launch_bounds__(512, 1)
ingest_kernel(const unsigned char* __restrict__ buf, int64_t bulk_bytes, const unsigned char* __restrict__ ldg,
              int64_t ldg_bytes, int copy_bytes, int stages, int consumers, int read_all, int ldg_warps,
              uint32_t* out) {
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(sm);
    uint64_t* empty = full + 16;
    unsigned char* data = sm + 256;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&full[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&empty[s])), "r"(consumers));
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    volatile int* abort = &abort_flag;
    const uint64_t limit = 1000000000ull;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        const uint64_t t0 = now_ns();
        uint32_t n = 0, ok = 0;
        while (true) {
            asm volatile(
                "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(ok)
                : "r"(smem_u32(bar)), "r"(parity)
                : "memory");
            if (ok) return true;
            if ((++n & 255) == 0) {
                if (*abort) return false;
                if (now_ns() - t0 > limit) {
                    *abort = 1;
                    atomicOr(&out[1], 1u);
                    return false;
                }
            }
        }
    };
    const int64_t nchunk = bulk_bytes / copy_bytes;
    uint32_t x = 0;
    if (warp == 0) {
        if (lane == 0 && nchunk > 0) {
            int64_t k = 0;
            for (int64_t c = blockIdx.x; c < nchunk; c += gridDim.x, ++k) {
                const int s = int(k % stages);
                if (!wait(&empty[s], uint32_t(((k / stages) & 1) ^ 1))) break;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&full[s])),
                             "r"(copy_bytes)
                             : "memory");
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        smem_u32(data + int64_t(s) * copy_bytes)),
                    "l"(buf + c * copy_bytes), "r"(copy_bytes), "r"(smem_u32(&full[s]))
                    : "memory");
            }
            // every issued copy lands before the CTA exits (bounded)
            const uint64_t t0 = now_ns();
            for (int64_t j = k > stages ? k - stages : 0; j < k; ++j) {
                uint32_t ok = 0;
                while (!ok) {
                    asm volatile(
                        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                        "selp.u32 %0, 1, 0, p;\n\t}"
                        : "=r"(ok)
                        : "r"(smem_u32(&full[j % stages])), "r"(uint32_t((j / stages) & 1))
                        : "memory");
                    if (!ok && now_ns() - t0 > limit) {
                        atomicOr(&out[1], 2u);
                        break;
                    }
                }
            }
        }
    } else if (warp <= consumers) {
        const int ctid = (warp - 1) * 32 + lane;
        const int words = copy_bytes / 16;
        int64_t k = 0;
        for (int64_t c = blockIdx.x; c < nchunk; c += gridDim.x, ++k) {
            const int s = int(k % stages);
            // the warp leaves only as a whole, so its __syncwarp never waits for a lane that left
            if (!__all_sync(0xffffffffu, wait(&full[s], uint32_t((k / stages) & 1)))) break;
            const uint4* row = reinterpret_cast<const uint4*>(data + int64_t(s) * copy_bytes);
            if (read_all) {
                for (int i = ctid; i < words; i += consumers * 32) {
                    const uint4 w = row[i];
                    x ^= w.x ^ w.y ^ w.z ^ w.w;
                }
            } else if (ctid == 0) {
                x ^= row[0].x;
            }
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty[s])) : "memory");
        }
    } else if (warp <= consumers + ldg_warps) {
        const int64_t nthreads = int64_t(gridDim.x) * ldg_warps * 32;
        const int64_t tid = int64_t(blockIdx.x) * ldg_warps * 32 + (warp - consumers - 1) * 32 + lane;
        const int64_t nvec = ldg_bytes / 32;
        for (int64_t v = tid; v < nvec; v += nthreads * kIngestLoads) {
            W8 r[kIngestLoads];
#pragma unroll
            for (int u = 0; u < kIngestLoads; ++u) {
                const int64_t q = v + int64_t(u) * nthreads;
#pragma unroll
                for (int i = 0; i < 8; ++i) r[u].w[i] = 0;
                if (q < nvec) ld32(ldg + q * 32, r[u]);
            }
#pragma unroll
            for (int u = 0; u < kIngestLoads; ++u)
#pragma unroll
                for (int i = 0; i < 8; ++i) x ^= r[u].w[i];
        }
    }
    if (x) atomicXor(&out[0], x);
}


// Reads [buf, buf + bulk_bytes) like ingest_kernel's bulk part (warp 0 lane 0 issues `copy_bytes`
// copies through `stages` slots, `consumers` warps read every 16-byte word of a landed slot) while
// `st_warps` warps write 32-byte vectors into this CTA's share of [st, st + st_bytes), cycling over
// it, until the reads are done (or, with bulk_bytes == 0, for one pass).  out[0] ^= checksum of the
// reads, out[1] |= error flags (1: a wait expired, 2: copies still landing, 4: the writers hit their
// 2 s bound), out[2] += bytes written.  Every loop is bounded by the buffer or by %globaltimer.
__global__ void __launch_bounds__(512, 1)
mixed_kernel(const unsigned char* __restrict__ buf, int64_t bulk_bytes, unsigned char* __restrict__ st,
             int64_t st_bytes, int copy_bytes, int stages, int consumers, int st_warps, int burst_rows, int burst_vecs,
             unsigned long long* out) {
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(sm);
    uint64_t* empty = full + 16;
    unsigned char* data = sm + 256;
    __shared__ int abort_flag;
    __shared__ int reads_done;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&full[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&empty[s])), "r"(consumers));
        }
        abort_flag = 0;
        reads_done = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    volatile int* abort = &abort_flag;
    volatile int* done = &reads_done;
    const uint64_t limit = 1000000000ull;
    auto try_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        return ok != 0;
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        const uint64_t t0 = now_ns();
        uint32_t n = 0;
        while (!try_wait(bar, parity)) {
            if ((++n & 255) == 0) {
                if (*abort) return false;
                if (now_ns() - t0 > limit) {
                    *abort = 1;
                    atomicOr(&out[1], 1ull);
                    return false;
                }
            }
        }
        return true;
    };
    const int64_t nchunk = bulk_bytes / copy_bytes;
    if (warp == 0) {
        if (lane == 0) {
            int64_t k = 0;
            for (int64_t c = blockIdx.x; c < nchunk; c += gridDim.x, ++k) {
                const int s = int(k % stages);
                if (!wait(&empty[s], uint32_t(((k / stages) & 1) ^ 1))) break;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&full[s])),
                             "r"(copy_bytes)
                             : "memory");
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        smem_u32(data + int64_t(s) * copy_bytes)),
                    "l"(buf + c * copy_bytes), "r"(copy_bytes), "r"(smem_u32(&full[s]))
                    : "memory");
            }
            // every issued copy lands before the CTA exits (bounded); then the writers may stop
            const uint64_t t0 = now_ns();
            for (int64_t j = k > stages ? k - stages : 0; j < k; ++j) {
                while (!try_wait(&full[j % stages], uint32_t((j / stages) & 1))) {
                    if (now_ns() - t0 > limit) {
                        atomicOr(&out[1], 2ull);
                        break;
                    }
                }
            }
            *done = 1;
        }
        return;
    }
    if (warp <= consumers) {
        const int ctid = (warp - 1) * 32 + lane;
        const int words = copy_bytes / 16;
        // burst writes: after every `burst_rows` landed copies each reading thread stores
        // `burst_vecs` 32-byte vectors (adjacent threads, adjacent vectors) into this CTA's share of
        // the write region, as a reduce-scatter stores its sums after the last rank's row
        const int64_t per = burst_rows > 0 ? st_bytes / 32 / gridDim.x : 0;
        const int64_t v0 = int64_t(blockIdx.x) * per;
        int64_t cursor = 0, written = 0;
        uint32_t x = 0;
        int64_t k = 0;
        for (int64_t c = blockIdx.x; c < nchunk; c += gridDim.x, ++k) {
            const int s = int(k % stages);
            // the warp leaves only as a whole, so its __syncwarp never waits for a lane that left
            if (!__all_sync(0xffffffffu, wait(&full[s], uint32_t((k / stages) & 1)))) break;
            const uint4* row = reinterpret_cast<const uint4*>(data + int64_t(s) * copy_bytes);
            for (int i = ctid; i < words; i += consumers * 32) {
                const uint4 w = row[i];
                x ^= w.x ^ w.y ^ w.z ^ w.w;
            }
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty[s])) : "memory");
            if (per > 0 && (k + 1) % burst_rows == 0) {
                const float f = __uint_as_float(x | 1u);
                for (int b = 0; b < burst_vecs; ++b) {
                    const int64_t v = (cursor + int64_t(b) * consumers * 32 + ctid) % per;
                    float* p = reinterpret_cast<float*>(st + (v0 + v) * 32);
                    asm volatile("st.global.cs.v8.f32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1};" ::"l"(p), "f"(f)
                                 : "memory");
                }
                cursor = (cursor + int64_t(burst_vecs) * consumers * 32) % per;
                written += int64_t(burst_vecs) * 32;
            }
        }
        if (x) atomicXor(&out[0], (unsigned long long)x);
        if (written) atomicAdd(&out[2], (unsigned long long)written);
        return;
    }
    if (warp <= consumers + st_warps) {
        // this CTA's share of the write region, in 32-byte vectors
        const int64_t nvec = st_bytes / 32;
        const int64_t per = nvec / gridDim.x;
        const int64_t v0 = int64_t(blockIdx.x) * per;
        const int t = (warp - consumers - 1) * 32 + lane, nt = st_warps * 32;
        const uint32_t val = 0x9e3779b9u * uint32_t(blockIdx.x * 1024 + t);
        const uint64_t t0 = now_ns();
        const bool one_pass = bulk_bytes == 0;
        int64_t written = 0, it = 0;
        bool stop = per <= 0;
        while (!stop) {
            for (int64_t v = t; v < per; v += nt) {
                float* p = reinterpret_cast<float*>(st + (v0 + v) * 32);
                const float f = __uint_as_float(val ^ uint32_t(v));
                asm volatile("st.global.cs.v8.f32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1};" ::"l"(p), "f"(f) : "memory");
                written += 32;
                if (!one_pass && (++it & 63) == 0 && *done) {
                    stop = true;
                    break;
                }
            }
            if (one_pass || *done) break;
            if (now_ns() - t0 > 2 * limit) {
                atomicOr(&out[1], 4ull);
                break;
            }
        }
        atomicAdd(&out[2], (unsigned long long)written);
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

int tide_probe_ingest(const void* buf, int64_t bulk_bytes, int64_t ldg_bytes, int32_t ctas, int32_t copy_bytes,
                      int32_t stages, int32_t consumer_warps, int32_t ldg_warps, uint32_t* out, void* stream) {
    const int consumers = consumer_warps > 0 ? consumer_warps : 1;
    if (!buf || !out || bulk_bytes < 0 || ldg_bytes < 0 || ctas < 1 || copy_bytes < 16 || copy_bytes % 16 ||
        stages < 1 || stages > 16 || 256 + int64_t(copy_bytes) * stages > int64_t(tide::kMaxDynamicSmem) || consumer_warps < 0 ||
        ldg_warps < 0 || 1 + consumers + ldg_warps > 16 || (reinterpret_cast<uintptr_t>(buf) & 255u) ||
        ldg_bytes % 32)
        return TIDE_EINVAL;
    const int smem = 256 + copy_bytes * stages;
    cudaError_t e = cudaFuncSetAttribute(tide::ingest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return tide::record_cuda_error(e);
    const auto* base = static_cast<const unsigned char*>(buf);
    const int64_t ldg_off = (bulk_bytes + 255) / 256 * 256;  // the register loads' region follows, 256-byte aligned
    tide::ingest_kernel<<<ctas, 32 * (1 + consumers + ldg_warps), smem, static_cast<cudaStream_t>(stream)>>>(
        base, bulk_bytes, base + ldg_off, ldg_bytes, copy_bytes, stages, consumers, consumer_warps > 0 ? 1 : 0,
        ldg_warps, out);
    e = cudaGetLastError();
    return e == cudaSuccess ? TIDE_OK : tide::record_cuda_error(e);
}

int tide_probe_mixed(const void* buf, int64_t bulk_bytes, void* st_buf, int64_t st_bytes, int32_t ctas,
                     int32_t copy_bytes, int32_t stages, int32_t consumer_warps, int32_t st_warps, int32_t burst_rows,
                     int32_t burst_vecs, uint64_t* out, void* stream) {
    if (burst_rows < 0 || burst_vecs < 0 || (burst_rows > 0 && (!st_buf || st_bytes / 32 < ctas)))
        return TIDE_EINVAL;
    if (!buf || !out || (st_warps > 0 && !st_buf) || bulk_bytes < 0 || st_bytes < 0 || ctas < 1 ||
        copy_bytes < 16 || copy_bytes % 16 || stages < 1 || stages > 16 ||
        256 + int64_t(copy_bytes) * stages > int64_t(tide::kMaxDynamicSmem) || consumer_warps < 1 || st_warps < 0 ||
        1 + consumer_warps + st_warps > 16 || (reinterpret_cast<uintptr_t>(buf) & 255u) ||
        (reinterpret_cast<uintptr_t>(st_buf) & 31u) || st_bytes % 32)
        return TIDE_EINVAL;
    const int smem = 256 + copy_bytes * stages;
    cudaError_t e = cudaFuncSetAttribute(tide::mixed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return tide::record_cuda_error(e);
    tide::mixed_kernel<<<ctas, 32 * (1 + consumer_warps + st_warps), smem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const unsigned char*>(buf), bulk_bytes, static_cast<unsigned char*>(st_buf), st_bytes, copy_bytes,
        stages, consumer_warps, st_warps, burst_rows, burst_vecs, reinterpret_cast<unsigned long long*>(out));
    e = cudaGetLastError();
    return e == cudaSuccess ? TIDE_OK : tide::record_cuda_error(e);
}

}  // extern "C"
