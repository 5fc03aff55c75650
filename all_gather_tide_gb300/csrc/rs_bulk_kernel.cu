// Reduce-scatter kernel with bulk asynchronous copies into shared memory (sm_103a).
//
// Paper: "The Endgame of FSDP Communication" (arXiv 2610.38228).  Fig. 2b step 5 and Fig. 6a form
// the fp32 sums in a bounded number of short-lived CTAs fed by bulk (TMA) copies, so that few SMs
// are taken from concurrent compute (Fig. 3, Fig. 4, Table 4).  With few CTAs the register-path
// kernel is limited by the bytes one SM keeps in flight; this variant keeps a deep pipeline of
// bulk copies in flight per SM instead.
//
// The bulk-copy engine of an SM keeps only about four copies in flight, so its bandwidth grows with
// the size of each copy (measured on GB300 at 16 CTAs: about 17 GB/s per SM with 4 KB copies, 68
// with 16 KB, 136 with 32 KB, 190 with 46-72 KB).  The kernel therefore streams one rank's row of a
// chunk per copy: a chunk is kBulkChunk elements of one (destination, parameter) piece, and its R
// rows pass through up to kBulkMaxStages shared-memory stages of kBulkChunk bf16 elements (45 KB),
// rank 0 first.  The fp32 sums of
// the chunk stay in the consumers' registers across the R stages (ascending rank order, starting
// from rank 0's value, exact bf16 -> fp32 widening, __fadd_rn), and are stored once, straight to
// the destination shard (st.global.cs), after the last rank.
//
// One CTA = 1 producer warp (lane 0 issues the copies) + kBulkConsumerWarps consumer warps; one
// CTA per SM.  Per stage the producer waits on the stage's `empty` mbarrier, announces the byte
// count on its `full` mbarrier and issues one cp.async.bulk; consumers wait on `full`, copy their
// slice of the row into registers, release the stage, and then add the slice with mixed-precision
// adds (add.rn.f32.bf16: the bf16 operand widened exactly, the fp32 sum rounded to nearest even; one
// instruction per element).  Elements a bulk copy cannot carry (a piece whose
// offsets are not 16-byte compatible, the < 8-element tail of the valid rows) are read with plain
// loads, and padding is stored as zeros, exactly as in the register-path kernel: the results are
// the same bits.
//
// Every mbarrier wait is bounded by %globaltimer: after `timeout_ns` the waiting thread records
// an error code in *status, all warps stop, the producer waits (again bounded) for the copies it
// has in flight, and the CTA returns.  Nothing traps.
#include <algorithm>

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

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
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

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.  Both addresses 16-byte
// aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// acc0 = fp32(low bf16 of w), acc1 = fp32(high bf16 of w): exact widening.
__device__ __forceinline__ void first_pair(float& acc0, float& acc1, uint32_t w) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.f32.bf16 %0, l;\n\tcvt.f32.bf16 %1, h;\n\t}"
        : "=f"(acc0), "=f"(acc1)
        : "r"(w));
}

// acc0 += low bf16 of w, acc1 += high bf16 of w: mixed-precision adds (the bf16 operand is widened
// exactly, the fp32 sum is rounded to nearest even; no flush to zero).
__device__ __forceinline__ void add_pair(float& acc0, float& acc1, uint32_t w) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(w));
}

// Copies this thread's 8-element groups of one rank row from shared memory into registers (zeros for
// groups past the copied elements, whose sums are never stored).
template <int Groups, int Consumers>
__device__ __forceinline__ void load_row(uint4 (&w)[Groups], const uint4* row, int ctid, bool whole, int64_t nbulk) {
#pragma unroll
    for (int j = 0; j < Groups; ++j) {
        const int g = j * Consumers + ctid;  // 8-element group index in the chunk
        w[j] = (whole || int64_t(g) * 8 + 8 <= nbulk) ? row[g] : make_uint4(0, 0, 0, 0);
    }
}

// Adds (First: widens) one rank row's groups held in registers.
template <bool First, int Groups>
__device__ __forceinline__ void add_row(float (&acc)[Groups][8], const uint4 (&w)[Groups]) {
#pragma unroll
    for (int j = 0; j < Groups; ++j) {
        if (First) {
            first_pair(acc[j][0], acc[j][1], w[j].x);
            first_pair(acc[j][2], acc[j][3], w[j].y);
            first_pair(acc[j][4], acc[j][5], w[j].z);
            first_pair(acc[j][6], acc[j][7], w[j].w);
        } else {
            add_pair(acc[j][0], acc[j][1], w[j].x);
            add_pair(acc[j][2], acc[j][3], w[j].y);
            add_pair(acc[j][4], acc[j][5], w[j].z);
            add_pair(acc[j][6], acc[j][7], w[j].w);
        }
    }
}

__device__ __forceinline__ uint16_t ld_u16(const uint16_t* p) {
    unsigned short v;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ float sum_scalar(const uint16_t* const* __restrict__ grads, int R, int P, int p,
                                            int64_t idx) {
    float acc = bf16_f32(ld_u16(grads[p] + idx));
    for (int r = 1; r < R; ++r) acc = __fadd_rn(acc, bf16_f32(ld_u16(grads[int64_t(r) * P + p] + idx)));
    return acc;
}

// Chunk geometry shared by producer and consumers.
struct ChunkView {
    int64_t n;       // elements in the chunk
    int64_t nvalid;  // of which are sums
    int64_t nbulk;   // leading valid elements delivered by bulk copies (multiple of 8, 0 if none)
    int64_t src;     // element offset of the chunk in every rank's gradient of p
    int64_t dst;     // element offset of the chunk in shard d
    int d, p;
};

constexpr uint64_t kTimerCheckEvery = 256;

// Wait for the phase of `bar` with the given parity, for at most `timeout_ns` from the first
// failed try.  Returns false (after recording `code` in *status and raising the CTA's abort flag)
// when the time runs out, or when another warp of the CTA has aborted.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                             volatile int* abort, int* status, int code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t deadline = globaltimer() + timeout_ns;
    uint64_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (++spins % kTimerCheckEvery == 0) {
            if (*abort) return false;
            if (globaltimer() > deadline) {
                atomicCAS(status, 0, code);
                *abort = 1;
                return false;
            }
        }
    }
    return true;
}

// The piece holding the current chunk, cached across the chunks of one piece: while the chunk stays
// inside the cached piece the cursor costs nothing; when it leaves, one load from the planner's
// chunk -> piece table finds the new piece (the CTAs' chunks are a grid stride apart, so with many
// small pieces a search of the piece list would cost a chain of dependent loads per chunk).
struct PieceCursor {
    int cur = -1;
    int64_t next_begin = 0;  // first chunk after the cached piece
    int64_t dst_off = 0, src_off = 0, valid = 0, total = 0, chunk_begin = 0;
    int d = 0, p = 0, vec = 0;

    // Moves to the piece holding chunk c (chunks only move forward); true when it changed.
    __device__ __forceinline__ bool seek(const RsSeg* __restrict__ segs, const int32_t* __restrict__ chunk_piece,
                                         int64_t c) {
        if (cur >= 0 && c < next_begin) return false;
        cur = __ldg(&chunk_piece[c]);
        const RsSeg* q = segs + cur;
        dst_off = __ldg(&q->dst_off);
        src_off = __ldg(&q->src_off);
        valid = __ldg(&q->valid);
        total = __ldg(&q->total);
        chunk_begin = __ldg(&q->chunk_begin);
        d = __ldg(&q->d);
        p = __ldg(&q->p);
        vec = __ldg(&q->vec);
        next_begin = chunk_begin + (total + kBulkChunk - 1) / kBulkChunk;
        return true;
    }

    __device__ __forceinline__ ChunkView view(int64_t c, int64_t chunk, int allow_vec) const {
        ChunkView v;
        const int64_t base = (c - chunk_begin) * chunk;
        v.n = min(chunk, total - base);
        v.nvalid = max(int64_t(0), min(v.n, valid - base));
        v.nbulk = (allow_vec && vec) ? (v.nvalid & ~int64_t(7)) : 0;
        v.src = src_off + base;
        v.dst = dst_off + base;
        v.d = d;
        v.p = p;
        return v;
    }
};

__device__ __forceinline__ void st_cs_v8(float* p, const float (&a)[8]) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(a[0]), "f"(a[1]),
                 "f"(a[2]), "f"(a[3]), "f"(a[4]), "f"(a[5]), "f"(a[6]), "f"(a[7])
                 : "memory");
}

__global__ void __launch_bounds__(kBulkThreads, 1)
reduce_scatter_bulk_kernel(const RsSeg* __restrict__ segs, const int32_t* __restrict__ chunk_piece, int64_t nchunks,
                           const uint16_t* const* __restrict__ grads, float* const* __restrict__ shards, int R,
                           int P, int allow_vec, int stages, int* status, uint64_t timeout_ns, int inject) {
    constexpr int kConsumers = kBulkConsumerWarps * 32;
    constexpr int kGroups = int(kBulkChunk / 8 / kConsumers);  // 8-element groups per consumer thread
    static_assert(kBulkChunk % (8 * kConsumers) == 0, "chunk must split evenly over the consumers");
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kBulkMaxStages;
    unsigned char* data = smem + 128;  // stage s at data + s * kBulkChunk * 2
    // the R gradient pointers of the producer's current piece
    const uint16_t** gptr = reinterpret_cast<const uint16_t**>(data + int64_t(stages) * kBulkChunk * 2);
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBulkConsumerWarps);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    volatile int* abort = &abort_flag;

    if (warp == kBulkConsumerWarps) {
        // ---------------- producer warp: all lanes track the piece, lane 0 issues ----------------
        PieceCursor pc;
        int64_t it = 0;       // stage uses issued so far (lane 0)
        int s = 0;            // stage of use `it`
        uint32_t phase = 0;   // its phase parity
        for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
            if (pc.seek(segs, chunk_piece, c)) {
                for (int r = lane; r < R; r += 32) gptr[r] = grads[int64_t(r) * P + pc.p];
                __syncwarp();
            }
            const ChunkView v = pc.view(c, kBulkChunk, allow_vec);
            if (v.nbulk == 0) continue;
            int stop = 0;
            if (lane == 0) {
                const uint32_t bytes = uint32_t(v.nbulk * 2);
                for (int r = 0; r < R; ++r) {
                    if (!wait_bounded(&empty[s], phase ^ 1u, timeout_ns, abort, status, 2)) {
                        stop = 1;
                        break;
                    }
                    if (!inject) {  // test hook: never signal the stage
                        mbar_arrive_expect_tx(&full[s], bytes);
                        bulk_g2s(data + int64_t(s) * kBulkChunk * 2, gptr[r] + v.src, bytes, &full[s]);
                    }
                    ++it;
                    if (++s == stages) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
        }
        // Let every copy already issued land before the CTA's shared memory goes away, whether the
        // producer ran out of chunks or stopped early: a consumer wait that expires after the
        // producer issued its last copy must not leave copies writing into freed shared memory.
        // Only the last `stages` stage uses can still be in flight, and each is the newest phase
        // of its stage, so waiting for that phase's parity is exact.
        if (lane == 0 && !inject) {
            const uint64_t drain = globaltimer() + 100000000ull;  // at most 100 ms
            for (int64_t j = max(int64_t(0), it - stages); j < it; ++j) {
                uint64_t* bar = &full[j % stages];
                const uint32_t par = uint32_t((j / stages) & 1);
                bool late = false;
                while (!mbar_try_wait(bar, par)) {
                    if (globaltimer() > drain) {
                        atomicCAS(status, 0, 4);
                        late = true;
                        break;
                    }
                }
                if (late) break;
            }
        }
        return;
    }

    // ---------------- consumer warps ----------------
    const int ctid = threadIdx.x;
    PieceCursor pc;
    float* shard = nullptr;
    int s = 0;
    uint32_t phase = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        if (pc.seek(segs, chunk_piece, c)) shard = shards[pc.d];
        const ChunkView v = pc.view(c, kBulkChunk, allow_vec);
        float* __restrict__ dst = shard + v.dst;
        if (v.nbulk > 0) {
            const bool whole = v.nbulk == kBulkChunk;  // every group of the chunk is carried
            float acc[kGroups][8];
            for (int r = 0; r < R; ++r) {
                // the warp leaves only as a whole (every lane saw the stage land, or none goes on), so
                // the __syncwarp below never waits for a lane that has returned
                if (!__all_sync(0xffffffffu, wait_bounded(&full[s], phase, timeout_ns, abort, status, 1))) return;
                const uint4* row = reinterpret_cast<const uint4*>(data + int64_t(s) * kBulkChunk * 2);
                // release the stage as soon as the warp's slice is in registers, before the adds, so
                // the producer can refill it while the adds run
                uint4 w[kGroups];
                load_row<kGroups, kConsumers>(w, row, ctid, whole, v.nbulk);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                if (r == 0) add_row<true, kGroups>(acc, w);
                else add_row<false, kGroups>(acc, w);
                if (++s == stages) {
                    s = 0;
                    phase ^= 1u;
                }
            }
            // the widest stores the destination allows: the shard offset o_p of a parameter placed
            // after small 1-D parameters need not be a multiple of 4 elements
            const unsigned da = unsigned(reinterpret_cast<uintptr_t>(dst) & 31u);
            const int sw = da == 0 ? 32 : (da & 15u) == 0 ? 16 : (da & 7u) == 0 ? 8 : 4;  // bytes
#pragma unroll
            for (int j = 0; j < kGroups; ++j) {
                const int64_t e = (int64_t(j) * kConsumers + ctid) * 8;
                if (whole || e + 8 <= v.nbulk) {
                    const float* a = acc[j];
                    if (sw == 32) {
                        st_cs_v8(dst + e, acc[j]);
                    } else if (sw == 16) {
                        __stcs(reinterpret_cast<float4*>(dst + e), make_float4(a[0], a[1], a[2], a[3]));
                        __stcs(reinterpret_cast<float4*>(dst + e + 4), make_float4(a[4], a[5], a[6], a[7]));
                    } else if (sw == 8) {
#pragma unroll
                        for (int k = 0; k < 8; k += 2)
                            __stcs(reinterpret_cast<float2*>(dst + e + k), make_float2(a[k], a[k + 1]));
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k) __stcs(dst + e + k, a[k]);
                    }
                }
            }
        }
        // valid elements not carried by the copies, then padding
        for (int64_t e = v.nbulk + ctid; e < v.n; e += kConsumers)
            dst[e] = (e < v.nvalid) ? sum_scalar(grads, R, P, v.p, v.src + e) : 0.0f;
    }
}


// The widest stores a destination address allows (bytes: 32, 16, 8 or 4; shards need only fp32
// alignment) and 8 fp32 sums stored with them, evict-first.
__device__ __forceinline__ int store_width(const float* p) {
    const unsigned da = unsigned(reinterpret_cast<uintptr_t>(p) & 31u);
    return da == 0 ? 32 : (da & 15u) == 0 ? 16 : (da & 7u) == 0 ? 8 : 4;
}

__device__ __forceinline__ void store8(float* p, const float (&a)[8], int sw) {
    if (sw == 32) {
        st_cs_v8(p, a);
    } else if (sw == 16) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(a[0], a[1], a[2], a[3]));
        __stcs(reinterpret_cast<float4*>(p + 4), make_float4(a[4], a[5], a[6], a[7]));
    } else if (sw == 8) {
#pragma unroll
        for (int k = 0; k < 8; k += 2) __stcs(reinterpret_cast<float2*>(p + k), make_float2(a[k], a[k + 1]));
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) __stcs(p + k, a[k]);
    }
}

// ---------------------------------------------------------------------------------------------
// TMEM-staged variant: the same pipeline and the same sums, but the consumers never store to
// global memory.  Measured on GB300 with the read/write probe (16 CTAs): stores issued by the warps
// that read the landed copies cut their reads from ~110 to ~55-67 GB/s per SM, whether issued in
// bursts or spread out, while the same stores from separate warps cost the reads ~5 %.  So here the
// consumers hand each chunk's fp32 sums to Tensor Memory (tcgen05.st, the SM's 256 KB accumulator
// memory, otherwise unused by this kernel; two chunk buffers) and one writer warp per SM
// sub-partition drains them to the shard (tcgen05.ld, then 32-byte stores), and also writes the
// elements the bulk copies do not carry (tails, padding, element-wise pieces).  A warp reaches only
// the TMEM lanes of its own sub-partition (lanes 32 * (warp % 4) ...), so consumer warp w parks
// its sums in lane quarter w % 4 and the writer of that quarter drains them.
//
// Warps 0..14: consumers (6 groups of 8 sums per thread, as in reduce_scatter_bulk_kernel);
// warp 15: producer; warps 16..19: writers of lane quarters 0..3.  640 threads, one CTA per SM.
constexpr int kTmemWriters = 4;
constexpr int kTmemThreads = (kBulkConsumerWarps + 1 + kTmemWriters) * 32;
constexpr int kTmemGroups = int(kBulkChunk / 8 / (kBulkConsumerWarps * 32));  // 6
constexpr uint32_t kTmemCols = 512;                                             // whole TMEM
constexpr uint32_t kTmemBufCols = 4 * kTmemGroups * 8;                          // 4 consumers per quarter
static_assert(2 * kTmemBufCols <= kTmemCols, "two chunk buffers must fit in TMEM");

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&a)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(__float_as_uint(a[0])), "r"(__float_as_uint(a[1])), "r"(__float_as_uint(a[2])),
                 "r"(__float_as_uint(a[3])), "r"(__float_as_uint(a[4])), "r"(__float_as_uint(a[5])),
                 "r"(__float_as_uint(a[6])), "r"(__float_as_uint(a[7]))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&a)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = __uint_as_float(r[k]);
}

__global__ void __launch_bounds__(kTmemThreads, 1)
reduce_scatter_tmem_kernel(const RsSeg* __restrict__ segs, const int32_t* __restrict__ chunk_piece, int64_t nchunks,
                           const uint16_t* const* __restrict__ grads, float* const* __restrict__ shards, int R,
                           int P, int allow_vec, int stages, int* status, uint64_t timeout_ns, int inject) {
    constexpr int kConsumers = kBulkConsumerWarps * 32;
    constexpr int kGroups = kTmemGroups;
    static_assert(kBulkChunk == int64_t(kGroups) * 8 * kConsumers, "chunk must split evenly over the consumers");
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kBulkMaxStages;
    unsigned char* data = smem + 128;
    const uint16_t** gptr = reinterpret_cast<const uint16_t**>(data + int64_t(stages) * kBulkChunk * 2);
    __shared__ int abort_flag;
    __shared__ uint32_t tmem_base;
    __shared__ __align__(8) uint64_t tfull[2];   // a chunk buffer holds the consumers' sums (15 arrivals)
    __shared__ __align__(8) uint64_t tempty[2];  // a chunk buffer has been drained (4 arrivals)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kProducer = kBulkConsumerWarps;
    constexpr int kWriter0 = kBulkConsumerWarps + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kBulkConsumerWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], kBulkConsumerWarps);
            mbar_init(&tempty[b], kTmemWriters);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWriter0) {  // one warp allocates the whole TMEM of this SM (one CTA per SM)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tbase = tmem_base;
    volatile int* abort = &abort_flag;

    if (warp == kProducer) {
        // ---------------- producer: as in reduce_scatter_bulk_kernel ----------------
        PieceCursor pc;
        int64_t it = 0;
        int s = 0;
        uint32_t phase = 0;
        for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
            if (pc.seek(segs, chunk_piece, c)) {
                for (int r = lane; r < R; r += 32) gptr[r] = grads[int64_t(r) * P + pc.p];
                __syncwarp();
            }
            const ChunkView v = pc.view(c, kBulkChunk, allow_vec);
            if (v.nbulk == 0) continue;
            int stop = 0;
            if (lane == 0) {
                const uint32_t bytes = uint32_t(v.nbulk * 2);
                for (int r = 0; r < R; ++r) {
                    if (!wait_bounded(&empty[s], phase ^ 1u, timeout_ns, abort, status, 2)) {
                        stop = 1;
                        break;
                    }
                    if (!inject) {
                        mbar_arrive_expect_tx(&full[s], bytes);
                        bulk_g2s(data + int64_t(s) * kBulkChunk * 2, gptr[r] + v.src, bytes, &full[s]);
                    }
                    ++it;
                    if (++s == stages) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
        }
        if (lane == 0 && !inject) {
            const uint64_t drain = globaltimer() + 100000000ull;
            for (int64_t j = max(int64_t(0), it - stages); j < it; ++j) {
                uint64_t* bar = &full[j % stages];
                const uint32_t par = uint32_t((j / stages) & 1);
                bool late = false;
                while (!mbar_try_wait(bar, par)) {
                    if (globaltimer() > drain) {
                        atomicCAS(status, 0, 4);
                        late = true;
                        break;
                    }
                }
                if (late) break;
            }
        }
    } else if (warp < kProducer) {
        // ---------------- consumers: sums in registers, handed to TMEM per chunk ----------------
        const int ctid = threadIdx.x;
        // this warp's 48 columns in lane quarter warp % 4 (the 32 lanes of its threads)
        const uint32_t tq = tbase + (uint32_t(32 * (warp & 3)) << 16) + uint32_t((warp >> 2) * kGroups * 8);
        PieceCursor pc;
        int s = 0;
        uint32_t phase = 0;
        int64_t nb = 0;  // bulk chunks handed over so far
        bool ok = true;
        for (int64_t c = blockIdx.x; c < nchunks && ok; c += gridDim.x) {
            pc.seek(segs, chunk_piece, c);
            const ChunkView v = pc.view(c, kBulkChunk, allow_vec);
            if (v.nbulk == 0) continue;
            const bool whole = v.nbulk == kBulkChunk;
            float acc[kGroups][8];
            for (int r = 0; r < R; ++r) {
                // every lane waits; the warp goes on only if all of them saw the stage land, so the
                // warp-wide instructions below always run converged
                if (!__all_sync(0xffffffffu, wait_bounded(&full[s], phase, timeout_ns, abort, status, 1))) {
                    ok = false;
                    break;
                }
                const uint4* row = reinterpret_cast<const uint4*>(data + int64_t(s) * kBulkChunk * 2);
                uint4 w[kGroups];
                load_row<kGroups, kConsumers>(w, row, ctid, whole, v.nbulk);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                if (r == 0) add_row<true, kGroups>(acc, w);
                else add_row<false, kGroups>(acc, w);
                if (++s == stages) {
                    s = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            // the chunk buffer must have been drained by all four writers (its use two chunks ago)
            const int b = int(nb & 1);
            if (!__all_sync(0xffffffffu,
                            wait_bounded(&tempty[b], uint32_t(((nb >> 1) & 1) ^ 1), timeout_ns, abort, status, 16)))
                break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t tb = tq + uint32_t(b) * kTmemBufCols;
#pragma unroll
            for (int j = 0; j < kGroups; ++j) tmem_st8(tb + uint32_t(j * 8), acc[j]);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&tfull[b]);
            ++nb;
        }
    } else {
        // ---------------- writers: drain lane quarter q, then the elements copies do not carry ---
        const int q = warp - kWriter0;
        PieceCursor pc;
        float* shard = nullptr;
        int64_t nb = 0;
        for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
            if (pc.seek(segs, chunk_piece, c)) shard = shards[pc.d];
            const ChunkView v = pc.view(c, kBulkChunk, allow_vec);
            float* __restrict__ dst = shard + v.dst;
            if (v.nbulk > 0) {
                const bool whole = v.nbulk == kBulkChunk;
                const int b = int(nb & 1);
                if (!__all_sync(0xffffffffu, wait_bounded(&tfull[b], uint32_t((nb >> 1) & 1), timeout_ns, abort, status, 32)))
                    break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const int sw = store_width(dst);
                const uint32_t tb = tbase + (uint32_t(32 * q) << 16) + uint32_t(b) * kTmemBufCols;
                // consumer warps q, q + 4, q + 8, q + 12 (< 15) park their sums in this quarter
                for (int cw = q; cw < kBulkConsumerWarps; cw += 4) {
                    float a[kGroups][8];
#pragma unroll
                    for (int j = 0; j < kGroups; ++j) tmem_ld8(tb + uint32_t(((cw >> 2) * kGroups + j) * 8), a[j]);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int j = 0; j < kGroups; ++j) {
                        const int64_t e = (int64_t(j) * kConsumers + cw * 32 + lane) * 8;
                        if (whole || e + 8 <= v.nbulk) store8(dst + e, a[j], sw);
                    }
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[b]);
                ++nb;
            }
            // valid elements not carried by the copies, then padding
            for (int64_t e = v.nbulk + q * 32 + lane; e < v.n; e += kTmemWriters * 32)
                dst[e] = (e < v.nvalid) ? sum_scalar(grads, R, P, v.p, v.src + e) : 0.0f;
        }
    }

    // everyone is done with TMEM before the allocating warp frees it
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == kWriter0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols) : "memory");
}

}  // namespace

size_t bulk_smem_bytes(int R, int stages) {
    return 128 + size_t(stages) * size_t(kBulkChunk) * 2 + sizeof(void*) * size_t(R);
}

// The deepest pipeline whose stages and pointer cache fit in one CTA's shared memory.
int bulk_stages(int R) {
    for (int st = kBulkMaxStages; st >= 2; --st)
        if (bulk_smem_bytes(R, st) <= kMaxDynamicSmem) return st;
    return 0;
}

cudaError_t launch_reduce_scatter_bulk(const RsSeg* segs, const int32_t* chunk_piece, int64_t nchunks,
                                       const uint16_t* const* grads,
                                       float* const* shards, int R, int P, int allow_vec, int ctas, int* status,
                                       uint64_t timeout_ns, int inject, cudaStream_t stream) {
    if (nchunks <= 0) return cudaSuccess;
    const int stages = bulk_stages(R);
    if (stages < 2) return cudaErrorInvalidValue;
    const size_t smem = bulk_smem_bytes(R, stages);
    cudaError_t e = cudaFuncSetAttribute(reduce_scatter_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    const int grid = int(std::min<int64_t>(ctas, nchunks));
    reduce_scatter_bulk_kernel<<<grid, kBulkThreads, smem, stream>>>(segs, chunk_piece, nchunks, grads, shards, R, P,
                                                                     allow_vec, stages, status, timeout_ns, inject);
    return cudaGetLastError();
}

cudaError_t launch_reduce_scatter_tmem(const RsSeg* segs, const int32_t* chunk_piece, int64_t nchunks,
                                       const uint16_t* const* grads, float* const* shards, int R, int P,
                                       int allow_vec, int ctas, int* status, uint64_t timeout_ns, int inject,
                                       cudaStream_t stream) {
    if (nchunks <= 0) return cudaSuccess;
    const int stages = bulk_stages(R);
    if (stages < 2) return cudaErrorInvalidValue;
    const size_t smem = bulk_smem_bytes(R, stages);
    cudaError_t e = cudaFuncSetAttribute(reduce_scatter_tmem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    const int grid = int(std::min<int64_t>(ctas, nchunks));
    reduce_scatter_tmem_kernel<<<grid, kTmemThreads, smem, stream>>>(segs, chunk_piece, nchunks, grads, shards, R,
                                                                     P, allow_vec, stages, status, timeout_ns, inject);
    return cudaGetLastError();
}

}  // namespace tide
