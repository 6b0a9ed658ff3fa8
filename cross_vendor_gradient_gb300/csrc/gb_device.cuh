// Device-side helpers of libgb: lane layout, streaming vector memory access,
// and the bf16 / OCP fp8 conversions written as inline PTX.
//
// Everything on the hot path is HBM-streaming work (a handful of float32 adds
// per 4-8 bytes moved), so the kernels are built around wide coalesced loads
// and stores, enough bytes in flight per SM, and warp-shuffle block maxima;
// there is no dense contraction and no tensor-core work.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gb.h"

namespace gb {

constexpr int kTile = 256;  // elements per warp tile
constexpr int kWarp = 32;

// ---------------------------------------------------------------- layout
// A warp tile is 256 consecutive elements; lane l owns elements 8l .. 8l+7.
// float32: one 32-byte access per lane (a 1 KiB contiguous warp access);
// bf16: one 16-byte access per lane (512 B per warp); fp8 codes: 8 bytes.
// With codec blocks of 128, lanes 0..15 form block 2t and lanes 16..31
// block 2t+1; with blocks of 256 the whole warp is one block.
__device__ __forceinline__ unsigned lane_elem(int lane, int k) { return (unsigned)(lane * 8 + k); }

// ------------------------------------------ programmatic dependent launch
// Every kernel is launched allowed to start while the kernel before it on the
// stream drains (launch_grid), which hides the gap between back-to-back
// launches.  Before its first global memory access each kernel waits here
// until that kernel has completed and its writes are visible (immediate when
// the previous operation on the stream is not a kernel).  The returned 0 is
// added to the kernel's first index, so every address it touches depends on
// the wait and no load can be scheduled ahead of it.
__device__ __forceinline__ uint32_t wait_prior_grid() {
    uint32_t z;
    asm volatile("griddepcontrol.wait;\n\tmov.u32 %0, 0;" : "=r"(z) : : "memory");
    return z;
}

// ------------------------------------------------------- memory accesses
// Rank buffers are read once per collective: bypass L1 and mark the lines
// evict-first in L2.  Payloads are re-read soon (copy engines, the decode
// kernel), so they are stored and loaded normally.
struct U8x32 { uint32_t w[8]; };

__device__ __forceinline__ U8x32 ld_stream_v8(const void *p) {
    U8x32 r;
    asm("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
          "=r"(r.w[6]), "=r"(r.w[7])
        : "l"(p));
    return r;
}
__device__ __forceinline__ U8x32 ld_v8(const void *p) {
    U8x32 r;
    asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
          "=r"(r.w[6]), "=r"(r.w[7])
        : "l"(p));
    return r;
}
// Coherent (read-write) 32-byte load, for buffers the kernel also writes.
__device__ __forceinline__ U8x32 ld_rw_v8(const void *p) {
    U8x32 r;
    asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
                   "=r"(r.w[6]), "=r"(r.w[7])
                 : "l"(p)
                 : "memory");
    return r;
}
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}
__device__ __forceinline__ uint4 ld_u4(const void *p) {
    uint4 r;
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ld_u2(const void *p) {
    uint2 r;
    asm("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}
__device__ __forceinline__ void st_v8(void *p, const uint32_t w[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void st_stream_v8(void *p, const uint32_t w[8]) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void st_u4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_stream_u4(void *p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_u2(void *p, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// A lane's 8 float32 elements of a rank buffer: one 32-byte access, or,
// when a rank buffer of the launch is only 16-byte aligned (A16), two
// 16-byte accesses at the same addresses (the warp still covers the same
// contiguous 1 KiB).
template <bool A16>
__device__ __forceinline__ U8x32 ld_stream_f32x8(const void *p) {
    if constexpr (A16) {
        const uint4 lo = ld_stream_u4(p), hi = ld_stream_u4((const unsigned char *)p + 16);
        return U8x32{{lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w}};
    } else {
        return ld_stream_v8(p);
    }
}
template <bool A16>
__device__ __forceinline__ void st_stream_f32x8(void *p, const uint32_t w[8]) {
    if constexpr (A16) {
        st_stream_u4(p, make_uint4(w[0], w[1], w[2], w[3]));
        st_stream_u4((unsigned char *)p + 16, make_uint4(w[4], w[5], w[6], w[7]));
    } else {
        st_stream_v8(p, w);
    }
}

// Whether any of the first `count` buffers is 16-byte but not 32-byte
// aligned (host side; rank buffers must be 16-byte aligned).
inline bool any_a16(const void *const *p, int count) {
    for (int i = 0; i < count; ++i)
        if (((uintptr_t)p[i] & 31u) != 0) return true;
    return false;
}

// ------------------------------------------------------------ conversions
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h16) { return __uint_as_float(h16 << 16); }

// Two float32 -> packed bf16x2, round to nearest even (lo in the low half).
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two float32 -> packed OCP fp8x2, round to nearest even, saturating to the
// largest finite value (lo in the low byte).
template <int CODEC>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
    unsigned short r;
    if (CODEC == GB_CODEC_E4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packed fp8x2 (low 16 bits of `pair`) -> two float32 (exact: every E4M3 and
// E5M2 value is a binary16 value, and every binary16 value a binary32 one).
template <int CODEC>
__device__ __forceinline__ void fp8x2_to_f32(uint32_t pair, float &lo, float &hi) {
    uint32_t h2;
    unsigned short p = (unsigned short)pair;
    if (CODEC == GB_CODEC_E4M3)
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(p));
    else
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(p));
    unsigned short l16 = (unsigned short)(h2 & 0xFFFFu), h16 = (unsigned short)(h2 >> 16);
    asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(l16));
    asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(h16));
}

// Largest finite value of the format as M = 0.875 * 2^E.
template <int CODEC> struct Fp8Fmt;
template <> struct Fp8Fmt<GB_CODEC_E4M3> { static constexpr int E = 9; };
template <> struct Fp8Fmt<GB_CODEC_E5M2> { static constexpr int E = 16; };

// Block scale exponent from the bits of the block's largest magnitude m >= 0:
// the smallest k with m * 2^-k <= 0.875 * 2^E, clamped to k >= -126, and 0
// for m == 0.  With m = 1.f * 2^(ef - 127), m * 2^-k <= 0.875 * 2^E holds for
// k = ef - 126 - E exactly when 1.f <= 1.75, i.e. the fraction bits are at
// most 0x600000; otherwise one more power of two is needed.
template <int CODEC>
__device__ __forceinline__ int block_scale_exp(float m) {
    const uint32_t b = __float_as_uint(m);
    if (b == 0u) return 0;
    const int ef = (int)(b >> 23);
    if (ef == 0) return -126;  // subnormal magnitude: clamped
    int k = ef - 126 - Fp8Fmt<CODEC>::E + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return k < -126 ? -126 : k;
}
__device__ __forceinline__ float pow2f(int k) { return __uint_as_float((uint32_t)(127 + k) << 23); }

// ---------------------------------------------------------- payload layout
__host__ __device__ __forceinline__ size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace gb
