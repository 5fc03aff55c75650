// Device helper shared by the placement kernels: a bf16 run copy for any pair of alignments.
#pragma once

#include <cstdint>

namespace tide {

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Read-only load that allocates in L1: the shifted path reads each aligned word twice (as one
// thread's second word and the next thread's first), the second time from L1 (measured: 3.6 ->
// 6.0 TB/s on a Qwen3-shaped group at R = 64 against L1::no_allocate loads).
__device__ __forceinline__ uint4 ld_nc_l1(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// nv vectors of type V, threads t = 0..nt-1, Unroll loads in flight per thread before its stores.
template <typename V, int Unroll>
__device__ __forceinline__ void copy_vectors(V* __restrict__ dst, const V* __restrict__ src, int64_t nv, int t,
                                             int nt) {
    int64_t i = t;
    for (; i + int64_t(Unroll - 1) * nt < nv; i += int64_t(Unroll) * nt) {
        V v[Unroll];
#pragma unroll
        for (int u = 0; u < Unroll; ++u) v[u] = ld_nc(src + i + int64_t(u) * nt);
#pragma unroll
        for (int u = 0; u < Unroll; ++u) dst[i + int64_t(u) * nt] = v[u];
    }
    for (; i < nv; i += nt) dst[i] = ld_nc(src + i);
}

// 16 bytes starting `off` bytes (even, 2..14) into the 32 bytes a:b (little-endian byte order).
__device__ __forceinline__ uint4 bytes_at(const uint4& a, const uint4& b, unsigned off) {
    const uint32_t c[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const unsigned q = off >> 2;  // whole 32-bit words to skip
    uint32_t o[5];
#pragma unroll
    for (int j = 0; j < 5; ++j) o[j] = q == 0 ? c[j] : q == 1 ? c[j + 1] : q == 2 ? c[j + 2] : c[j + 3];
    if (off & 2u) {  // and half a word
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = __funnelshift_r(o[j], o[j + 1], 16);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Copies n bf16 elements src -> dst with threads t = 0..nt-1 for any pair of addresses: a head of
// elements brings dst to a 16-byte boundary; if src is then aligned too, 16-byte vectors follow.
// Otherwise every 16-byte store of dst is assembled from the two aligned 16-byte words of src it
// straddles (the second is also the next thread's first, so it is served from L1); only aligned
// words lying wholly inside the run are read, the rest of the run goes element by element.  Used
// for runs whose offsets rule out the 16-byte fast path (for instance every parameter placed after
// a 1-D parameter of 2 or 4 elements per rank).
template <int Unroll>
__device__ __forceinline__ void copy_bf16_any_alignment(uint16_t* __restrict__ dst, const uint16_t* __restrict__ src,
                                                        int64_t n, int t, int nt) {
    const uintptr_t da = reinterpret_cast<uintptr_t>(dst);
    int64_t head = int64_t(((16u - unsigned(da & 15u)) & 15u) / 2u);  // elements until dst is aligned
    if (head > n) head = n;
    uint16_t* d = dst + head;
    const uint16_t* s = src + head;
    const unsigned s_off = unsigned(reinterpret_cast<uintptr_t>(s) & 15u);  // even: bf16 elements
    int64_t lo = head, hi = head;  // [lo, hi): the elements moved with 16-byte stores
    if (s_off == 0) {
        const int64_t nv = (n - head) / 8;
        copy_vectors<uint4, Unroll>(reinterpret_cast<uint4*>(d), reinterpret_cast<const uint4*>(s), nv, t, nt);
        hi = head + nv * 8;
    } else {
        // output vector i (16 bytes at d + 16 i) = bytes s_off .. s_off+15 of words W_i, W_{i+1}
        // (W_i = the aligned word at s - s_off + 16 i).  W_0 starts before the run and the last
        // word may end after it, so vectors 1 .. iend-1 go this way (W_1 .. W_iend inside the run).
        const uint4* w = reinterpret_cast<const uint4*>(s - s_off / 2u);
        const int64_t run_bytes = (n - head) * 2;
        const int64_t iend = (int64_t(s_off) + run_bytes) / 16 - 1;  // W_{iend} is the last whole word
        if (iend >= 2) {
            lo = head + 8;
            hi = head + 8 * iend;
            uint4* dv = reinterpret_cast<uint4*>(d);
            int64_t i = 1 + t;
            for (; i + int64_t(Unroll - 1) * nt < iend; i += int64_t(Unroll) * nt) {
                uint4 a[Unroll], b[Unroll];
#pragma unroll
                for (int u = 0; u < Unroll; ++u) {
                    a[u] = ld_nc_l1(w + i + int64_t(u) * nt);
                    b[u] = ld_nc_l1(w + i + int64_t(u) * nt + 1);
                }
#pragma unroll
                for (int u = 0; u < Unroll; ++u) dv[i + int64_t(u) * nt] = bytes_at(a[u], b[u], s_off);
            }
            for (; i < iend; i += nt) dv[i] = bytes_at(ld_nc_l1(w + i), ld_nc_l1(w + i + 1), s_off);
        }
    }
    // the rest element by element: [0, lo) and [hi, n)
    for (int64_t k = t; k < lo; k += nt) dst[k] = src[k];
    for (int64_t k = hi + t; k < n; k += nt) dst[k] = src[k];
}

}  // namespace tide
