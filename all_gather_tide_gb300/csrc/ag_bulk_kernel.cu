// All-gather placement with bulk asynchronous copies (sm_103a).
//
// Paper: "The Endgame of FSDP Communication" (arXiv 2610.38228).  the paper's all-gather puts shards
// into the parameters' storage with copy engines and no SM work (abstract; Table 1, no SM for the
// all-gather; Fig. 5b, a single strided copy for each parameter).  This kernel is the closest SM-side form: one thread per CTA drives
// the SM's bulk-copy engine, moving each run of valid elements shard_r[o_p ..) -> param_p[r*s_p ..)
// through shared memory (cp.async.bulk global -> shared, then cp.async.bulk shared -> global), so a
// CTA spends almost no issue slots and few CTAs still move a lot of data.
//
// Work: runs of valid elements per (source rank, parameter), cut into kAgBulkChunk-element chunks
// (48 KB); each CTA takes one contiguous range of the flat chunk list, so finding a chunk's run is
// a step of a cursor rather than a search (with many small runs, e.g. hundreds of parameters or 64
// ranks, a search per chunk on the issuing thread halved the bandwidth).  Lane 0 of warp 0 keeps up to
// kAgBulkStages loads in flight: a stage is refilled once the store that last read it has finished
// reading (cp.async.bulk.wait_group.read).  Chunks whose offsets are not 16-byte compatible, and the
// < 8-element tail of a run, are copied with plain loads and stores (warps 1..3 and lane 0).  Padding
// is never read; nothing outside the parameters is written.  Every mbarrier wait is bounded by
// %globaltimer and reports through *status, as in the reduce-scatter kernels.
#include <algorithm>

#include "copy_any.cuh"
#include "tide_internal.h"

namespace tide {
namespace {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, uint64_t timeout_ns, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = globaltimer() + timeout_ns;
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() > deadline) {
            atomicCAS(status, 0, 8);
            return false;
        }
    return true;
}

__device__ __forceinline__ int find_run(const AgSeg* __restrict__ segs, int nsegs, int cur, int64_t c) {
    if (cur + 1 >= nsegs || segs[cur + 1].chunk_begin > c) return cur;
    int lo = cur + 1, hi = nsegs, step = 1;
    for (;;) {
        const int nxt = lo + step;
        if (nxt >= nsegs) break;
        if (segs[nxt].chunk_begin > c) {
            hi = nxt;
            break;
        }
        lo = nxt;
        step <<= 1;
    }
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (segs[mid].chunk_begin <= c) lo = mid; else hi = mid;
    }
    return lo;
}

struct Chunk {
    const uint16_t* src;
    uint16_t* dst;
    int64_t n;     // elements
    int64_t nb;    // leading elements moved by bulk copies (multiple of 8; 0 = plain copy)
};

__device__ __forceinline__ Chunk chunk_of(const AgSeg* __restrict__ segs, int nsegs, int& cur, int64_t c,
                                          const uint16_t* const* __restrict__ shards,
                                          uint16_t* const* __restrict__ params) {
    cur = find_run(segs, nsegs, cur, c);
    const AgSeg sg = segs[cur];
    const int64_t base = (c - sg.chunk_begin) * kAgBulkChunk;
    Chunk k;
    k.n = min(kAgBulkChunk, sg.len - base);
    k.src = shards[sg.r] + sg.src_off + base;
    k.dst = params[sg.p] + sg.dst_off + base;
    k.nb = sg.vec ? (k.n & ~int64_t(7)) : 0;
    return k;
}

__global__ void __launch_bounds__(kAgBulkThreads, 1)
all_gather_bulk_kernel(const AgSeg* __restrict__ segs, int nsegs, int64_t nchunks,
                       const uint16_t* const* __restrict__ shards, uint16_t* const* __restrict__ params, int* status,
                       uint64_t timeout_ns) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    unsigned char* data = smem + 128;
    __shared__ uint16_t* st_dst[kAgBulkStages];
    __shared__ uint32_t st_bytes[kAgBulkStages];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's chunks: [c_begin, c_end)
    const int64_t c_begin = nchunks * blockIdx.x / gridDim.x, c_end = nchunks * (blockIdx.x + 1) / gridDim.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kAgBulkStages; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&full[s])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp > 0) {
        // plain copies of the chunks the bulk copies cannot carry
        const int t = threadIdx.x - 32, nt = kAgBulkThreads - 32;
        int cur = 0;
        for (int64_t c = c_begin; c < c_end; ++c) {
            const Chunk k = chunk_of(segs, nsegs, cur, c, shards, params);
            if (k.nb == 0) copy_bf16_any_alignment<4>(k.dst, k.src, k.n, t, nt);
        }
        return;
    }
    if (lane != 0) return;

    // lane 0 of warp 0: the bulk-copy pipeline
    int cur = 0;
    int64_t c_next = c_begin;  // next chunk of this CTA to examine for loading
    int64_t loaded = 0, stored = 0;
    bool ok = true;
    auto load_next = [&]() -> bool {  // issues the next bulk chunk's load; false when none is left
        while (c_next < c_end) {
            const Chunk k = chunk_of(segs, nsegs, cur, c_next, shards, params);
            ++c_next;
            if (k.nb == 0) continue;  // plain chunk: warps 1..3
            for (int64_t e = k.nb; e < k.n; ++e) k.dst[e] = k.src[e];  // < 8-element tail
            const int s = int(loaded % kAgBulkStages);
            const uint32_t bytes = uint32_t(k.nb * 2);
            st_dst[s] = k.dst;
            st_bytes[s] = bytes;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&full[s])), "r"(bytes)
                         : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(data + int64_t(s) * kAgBulkChunk * 2)),
                "l"(k.src), "r"(bytes), "r"(smem_u32(&full[s]))
                : "memory");
            ++loaded;
            return true;
        }
        return false;
    };
    while (loaded < kAgBulkStages && load_next()) {
    }
    while (stored < loaded) {
        const int s = int(stored % kAgBulkStages);
        if (!wait_bounded(&full[s], uint32_t((stored / kAgBulkStages) & 1), timeout_ns, status)) {
            ok = false;
            break;
        }
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(st_dst[s]),
                     "r"(smem_u32(data + int64_t(s) * kAgBulkChunk * 2)), "r"(st_bytes[s])
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        ++stored;
        // every store but the newest has finished reading its stage: refill up to kAgBulkStages
        // chunks ahead of the oldest stage still being read
        asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        while (loaded < stored - 1 + kAgBulkStages && load_next()) {
        }
    }
    if (!ok) {
        // a load never completed: wait (bounded) for the loads still in flight before leaving
        const uint64_t drain = globaltimer() + 100000000ull;
        for (int64_t j = stored; j < loaded; ++j)
            while (!mbar_try_wait(&full[j % kAgBulkStages], uint32_t((j / kAgBulkStages) & 1)))
                if (globaltimer() > drain) {
                    atomicCAS(status, 0, 4);
                    break;
                }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace

size_t ag_bulk_smem_bytes() { return 128 + size_t(kAgBulkStages) * size_t(kAgBulkChunk) * 2; }

cudaError_t launch_all_gather_bulk(const AgSeg* segs, int nsegs, int64_t nchunks, const uint16_t* const* shards,
                                   uint16_t* const* params, int ctas, int* status, uint64_t timeout_ns,
                                   cudaStream_t stream) {
    if (nchunks <= 0) return cudaSuccess;
    const size_t smem = ag_bulk_smem_bytes();
    cudaError_t e =
        cudaFuncSetAttribute(all_gather_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    const int grid = int(std::min<int64_t>(ctas, nchunks));
    all_gather_bulk_kernel<<<grid, kAgBulkThreads, smem, stream>>>(segs, nsegs, nchunks, shards, params, status,
                                                                  timeout_ns);
    return cudaGetLastError();
}

}  // namespace tide
