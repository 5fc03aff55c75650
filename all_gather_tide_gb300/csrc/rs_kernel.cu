// Layout-aware mixed-precision reduce-scatter kernel (sm_103a).
//
// Paper: "The Endgame of FSDP Communication" (arXiv 2610.38228).  The paper's reduce-scatter
// takes each parameter's bf16 gradient where it lies (Table 1, the in-place read row: no
// full-group pack) and sums into fp32 shards (abstract); Fig. 2b step 5 forms the fp32 sums with
// a bounded number of short-lived CTAs.  On one GPU every contributor rank is a buffer in local HBM, so the sum CTAs
// read the R gradients directly, and the landing step is folded into the same pass: each fp32
// result is stored once, at its final address in the destination shard (Fig. 1).
//
// Work decomposition: the planner lists (destination d, parameter p) pieces in shard order and
// cuts each into chunks of kRsChunk elements; a grid of `ctas` CTAs walks the flat chunk list
// with a grid stride.  In a chunk every thread owns kRsUnroll 16-byte output groups of 8
// elements: it issues the 16-byte bf16 loads of up to 8 ranks x kRsUnroll groups back to back
// (memory-level parallelism), widens them exactly (bf16 bits << 16), adds them into fp32 in
// ascending rank order starting from rank 0's value, and writes two 16-byte fp32 stores per
// group (8- or 4-byte stores when the shard offset of the piece is less aligned).  Padding
// elements of the piece are written as +0.0f without any load.  Pieces whose gradient offset
// d*s_p is not a multiple of 8 elements, or gradient pointers that are not 16-byte aligned, take
// an element-wise path.
//
// The data are streamed once: loads bypass L1 (ld.global.nc.L1::no_allocate) and stores are
// marked evict-first (st.global.cs).  Roofline: HBM, R*2 bytes read + 4 bytes written per valid
// output element, 4 bytes written per padding element.
#include <algorithm>

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

__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t* p) {
    unsigned short v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

// Exact bf16 -> fp32 widening of the two elements packed in a 32-bit word (element 2k in the
// low half, 2k+1 in the high half).
__device__ __forceinline__ float lo_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ void add8(float (&acc)[8], const uint4& v, bool first) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float a = lo_f32(w[k]), b = hi_f32(w[k]);
        // __fadd_rn: IEEE round-to-nearest-even, never contracted into an FMA
        acc[2 * k] = first ? a : __fadd_rn(acc[2 * k], a);
        acc[2 * k + 1] = first ? b : __fadd_rn(acc[2 * k + 1], b);
    }
}

// Ascending-rank fp32 sum of one element, element-wise path.
__device__ __forceinline__ float sum_scalar(const uint16_t* const* __restrict__ grads, int R, int P,
                                            int p, int64_t idx) {
    float acc = bf16_f32(ld_stream_u16(grads[p] + idx));
    for (int r = 1; r < R; ++r) acc = __fadd_rn(acc, bf16_f32(ld_stream_u16(grads[int64_t(r) * P + p] + idx)));
    return acc;
}

// Index of the last piece whose chunk_begin <= c, searching forward from `cur` (which already
// satisfies it): gallop, then bisect.  Pieces are sorted by chunk_begin.
__device__ __forceinline__ int find_piece(const RsSeg* __restrict__ segs, int nsegs, int cur, int64_t c) {
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

// Stores 8 fp32 values with the widest stores `sw` (16, 8 or 4 bytes) allows.
__device__ __forceinline__ void store8(float* p, const float (&a)[8], unsigned sw) {
    if (sw == 16u) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(a[0], a[1], a[2], a[3]));
        __stcs(reinterpret_cast<float4*>(p + 4), make_float4(a[4], a[5], a[6], a[7]));
    } else if (sw == 8u) {
#pragma unroll
        for (int k = 0; k < 8; k += 2) __stcs(reinterpret_cast<float2*>(p + k), make_float2(a[k], a[k + 1]));
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) __stcs(p + k, a[k]);
    }
}

__global__ void __launch_bounds__(kRsThreads, kRsCtasPerSm)
reduce_scatter_kernel(const RsSeg* __restrict__ segs, int nsegs, const int32_t* __restrict__ chunk_piece,
                      int64_t nchunks, const uint16_t* const* __restrict__ grads, float* const* __restrict__ shards,
                      int R, int P, int allow_vec) {
    constexpr int kBatch = 8;  // ranks whose loads are in flight together
    int cur = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        // the chunk's piece: from the planner's chunk -> piece table when there is one (one load
        // instead of a search: a CTA's chunks are a grid stride apart, many pieces apart when the
        // pieces are small), else by searching forward from the previous piece
        cur = chunk_piece ? __ldg(&chunk_piece[c]) : find_piece(segs, nsegs, cur, c);
        const RsSeg sg = segs[cur];
        const int64_t base = (c - sg.chunk_begin) * kRsChunk;
        const int64_t n = min(kRsChunk, sg.total - base);                 // elements in this chunk
        const int64_t nvalid = max(int64_t(0), min(n, sg.valid - base));  // of which are sums
        float* __restrict__ dst = shards[sg.d] + sg.dst_off + base;
        const int64_t src = sg.src_off + base;

        if (allow_vec && sg.vec) {
            float acc[kRsUnroll][8];
            bool full[kRsUnroll];
#pragma unroll
            for (int u = 0; u < kRsUnroll; ++u) {
                const int64_t e = (int64_t(u) * kRsThreads + threadIdx.x) * 8;
                full[u] = e + 8 <= nvalid;
            }
            for (int r0 = 0; r0 < R; r0 += kBatch) {
                uint4 v[kRsUnroll][kBatch];
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    if (r0 + j < R) {
                        const uint16_t* g = grads[int64_t(r0 + j) * P + sg.p] + src;
#pragma unroll
                        for (int u = 0; u < kRsUnroll; ++u)
                            if (full[u]) v[u][j] = ld_stream_v4(g + (int64_t(u) * kRsThreads + threadIdx.x) * 8);
                    }
                }
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    if (r0 + j < R) {
#pragma unroll
                        for (int u = 0; u < kRsUnroll; ++u)
                            if (full[u]) add8(acc[u], v[u][j], r0 + j == 0);
                    }
                }
            }
            // the widest stores the shard offset allows (o_p need not be a multiple of 4 elements)
            const unsigned da = unsigned(reinterpret_cast<uintptr_t>(dst) & 15u);
            const unsigned sw = da == 0 ? 16u : (da & 7u) == 0 ? 8u : 4u;
#pragma unroll
            for (int u = 0; u < kRsUnroll; ++u) {
                const int64_t e = (int64_t(u) * kRsThreads + threadIdx.x) * 8;
                if (full[u]) {
                    store8(dst + e, acc[u], sw);
                } else if (e >= nvalid && e + 8 <= n) {
                    const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    store8(dst + e, z, sw);
                } else if (e < n) {
                    // group straddling the end of the valid rows or of the piece
                    for (int k = 0; k < 8 && e + k < n; ++k)
                        dst[e + k] = (e + k < nvalid) ? sum_scalar(grads, R, P, sg.p, src + e + k) : 0.0f;
                }
            }
        } else {
            for (int64_t k = threadIdx.x; k < n; k += kRsThreads)
                dst[k] = (k < nvalid) ? sum_scalar(grads, R, P, sg.p, src + k) : 0.0f;
        }
    }
}

}  // namespace

cudaError_t launch_reduce_scatter(const RsSeg* segs, int nsegs, const int32_t* chunk_piece, int64_t nchunks,
                                  const uint16_t* const* grads, float* const* shards, int R, int P,
                                  int allow_vec, int ctas, cudaStream_t stream) {
    if (nchunks <= 0) return cudaSuccess;
    const int grid = int(std::min<int64_t>(ctas, nchunks));
    reduce_scatter_kernel<<<grid, kRsThreads, 0, stream>>>(segs, nsegs, chunk_piece, nchunks, grads, shards, R, P,
                                                          allow_vec);
    return cudaGetLastError();
}

}  // namespace tide
