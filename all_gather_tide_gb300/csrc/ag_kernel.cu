// All-gather placement kernel (sm_103a).
//
// Paper: "The Endgame of FSDP Communication" (arXiv 2610.38228).  The abstract's TIDE-AG lands
// gathered shards directly in per-parameter storage instead of copying a flat rank-major buffer
// out afterwards (Table 7, the copy-out column); Fig. 5b does it with a single strided copy for each parameter.
// This kernel is the SM form of that placement: for every (source rank r, parameter p) the
// planner emits the run of valid elements, shard_r[o_p, o_p + v(r,p)*L_p) -> param_p[r*s_p, ...),
// cut into chunks of kAgChunk elements; CTAs walk the chunk list with a grid stride.  Each
// thread moves kAgUnroll 16-byte vectors per chunk (all loads first, then all stores); runs whose
// offsets are not 16-byte aligned take the widest vectors their alignment allows.  Padding
// is never read and nothing outside the parameters is written.  Roofline: HBM, 2 bytes read +
// 2 bytes written per valid element.
#include <algorithm>

#include "copy_any.cuh"
#include "tide_internal.h"

namespace tide {
namespace {

__device__ __forceinline__ uint4 ld_stream_v4(const uint16_t* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream_v4(uint16_t* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
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

__global__ void __launch_bounds__(kAgThreads, kAgCtasPerSm)
all_gather_kernel(const AgSeg* __restrict__ segs, int nsegs, const int32_t* __restrict__ chunk_run, int64_t nchunks,
                  const uint16_t* const* __restrict__ shards, uint16_t* const* __restrict__ params,
                  int allow_vec) {
    int cur = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        // the chunk's run: one load from the planner's chunk -> run table (a CTA's chunks are a
        // grid stride apart, many runs apart when runs are short), else a forward search
        cur = chunk_run ? __ldg(&chunk_run[c]) : find_run(segs, nsegs, cur, c);
        const AgSeg sg = segs[cur];
        const int64_t base = (c - sg.chunk_begin) * kAgChunk;
        const int64_t n = min(kAgChunk, sg.len - base);
        const uint16_t* __restrict__ src = shards[sg.r] + sg.src_off + base;
        uint16_t* __restrict__ dst = params[sg.p] + sg.dst_off + base;
        if (allow_vec && sg.vec) {
            uint4 v[kAgUnroll];
#pragma unroll
            for (int u = 0; u < kAgUnroll; ++u) {
                const int64_t e = (int64_t(u) * kAgThreads + threadIdx.x) * 8;
                if (e + 8 <= n) v[u] = ld_stream_v4(src + e);
            }
#pragma unroll
            for (int u = 0; u < kAgUnroll; ++u) {
                const int64_t e = (int64_t(u) * kAgThreads + threadIdx.x) * 8;
                if (e + 8 <= n) {
                    st_stream_v4(dst + e, v[u]);
                } else {
                    for (int64_t k = e; k < n && k < e + 8; ++k) dst[k] = src[k];
                }
            }
        } else {
            copy_bf16_any_alignment<kAgUnroll>(dst, src, n, threadIdx.x, kAgThreads);
        }
    }
}

}  // namespace

cudaError_t launch_all_gather(const AgSeg* segs, int nsegs, const int32_t* chunk_run, int64_t nchunks,
                              const uint16_t* const* shards, uint16_t* const* params,
                              int allow_vec, int ctas, cudaStream_t stream) {
    if (nchunks <= 0) return cudaSuccess;
    const int grid = int(std::min<int64_t>(ctas, nchunks));
    all_gather_kernel<<<grid, kAgThreads, 0, stream>>>(segs, nsegs, chunk_run, nchunks, shards, params, allow_vec);
    return cudaGetLastError();
}

}  // namespace tide
