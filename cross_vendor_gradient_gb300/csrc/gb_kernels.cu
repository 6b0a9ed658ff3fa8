// CUDA kernels of libgb (sm_103a).
//
//   k_reduce_encode      island reduce + bridge encode, all islands per launch
//   k_decode_bcast       decode + accumulate + (AVG) + broadcast, all islands
//                        per launch (or the reduce_scatter slices)
//   k_decompress_acc     accum (+)= dec(payload), the unfused building block
//   k_copy               exact multi-destination copies (all_gather, broadcast)
//
// The method (gpubridge README, "all_reduce uses reduce-bridge-broadcast" and
// "Bridge compression") fixes what is computed: float32 island sums in
// ascending rank order, a per-block power-of-two scale with round-to-nearest
// -even saturating fp8 codes (or bf16 / raw float32 payloads), decoded terms
// added in float32 in island order.  Every kernel is a warp-per-tile
// streaming kernel: a warp owns 256 consecutive elements (8 per lane), moves
// them with 16-byte coalesced accesses, and for fp8 finds the block maximum
// with warp shuffles, so no shared memory, no atomics and no inter-warp
// ordering enter the arithmetic: the result does not depend on the grid.
#include <atomic>
#include <cuda_runtime.h>

#include "gb_device.cuh"
#include "gb_kernels.cuh"

namespace gb {

static std::atomic<uint64_t> g_launches{0};
uint64_t launches() { return g_launches.load(); }

using bf16 = __nv_bfloat16;

// ------------------------------------------------------ lane loads / stores

// Load this lane's 8 elements of rank buffer `p` in tile `base` as float32.
template <typename T>
__device__ __forceinline__ void load_rank(const void *p, uint64_t base, int lane, uint64_t n,
                                          bool full, float v[8]) {
    if constexpr (sizeof(T) == 4) {
        const float *f = (const float *)p + base;
        if (full) {
            uint4 x = ld_stream_u4(f + 4 * lane);
            uint4 y = ld_stream_u4(f + 128 + 4 * lane);
            v[0] = __uint_as_float(x.x); v[1] = __uint_as_float(x.y);
            v[2] = __uint_as_float(x.z); v[3] = __uint_as_float(x.w);
            v[4] = __uint_as_float(y.x); v[5] = __uint_as_float(y.y);
            v[6] = __uint_as_float(y.z); v[7] = __uint_as_float(y.w);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint64_t j = base + Lay<float>::idx(lane, k);
                v[k] = j < n ? __ldg((const float *)p + j) : 0.0f;
            }
        }
    } else {
        const unsigned short *h = (const unsigned short *)p + base;
        if (full) {
            uint4 x = ld_stream_u4(h + 8 * lane);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(w[i] << 16);
                v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint64_t j = base + Lay<bf16>::idx(lane, k);
                v[k] = j < n ? bf16_bits_to_f32(__ldg((const unsigned short *)p + j)) : 0.0f;
            }
        }
    }
}

// Store this lane's 8 float32 results into a rank buffer of type T (bf16:
// round to nearest even), streaming (the data is not re-read soon).
template <typename T>
__device__ __forceinline__ void store_rank(void *p, uint64_t base, int lane, uint64_t limit,
                                           bool full, const float t[8]) {
    if constexpr (sizeof(T) == 4) {
        float *f = (float *)p + base;
        if (full) {
            st_stream_u4(f + 4 * lane, make_uint4(__float_as_uint(t[0]), __float_as_uint(t[1]),
                                                  __float_as_uint(t[2]), __float_as_uint(t[3])));
            st_stream_u4(f + 128 + 4 * lane,
                         make_uint4(__float_as_uint(t[4]), __float_as_uint(t[5]),
                                    __float_as_uint(t[6]), __float_as_uint(t[7])));
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint64_t j = base + Lay<float>::idx(lane, k);
                if (j < limit) ((float *)p)[j] = t[k];
            }
        }
    } else {
        unsigned short *h = (unsigned short *)p + base;
        if (full) {
            st_stream_u4(h + 8 * lane, make_uint4(cvt_bf16x2(t[0], t[1]), cvt_bf16x2(t[2], t[3]),
                                                  cvt_bf16x2(t[4], t[5]), cvt_bf16x2(t[6], t[7])));
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint64_t j = base + Lay<bf16>::idx(lane, k);
                if (j < limit) ((unsigned short *)p)[j] = (unsigned short)(cvt_bf16x2(t[k], 0.0f) & 0xFFFFu);
            }
        }
    }
}

// ------------------------------------------------------------- the encoder

// Largest magnitude of each lane's block(s), reduced across the lanes of the
// block.  lo covers elements 0..3 of the lane, hi elements 4..7.
template <typename T, int BLOCK>
__device__ __forceinline__ void block_absmax(const float v[8], float &lo, float &hi) {
    float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    float b = fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7])));
    if constexpr (BLOCK == 256) {
        float m = fmaxf(a, b);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        lo = hi = m;
    } else if constexpr (sizeof(T) == 4) {
        // float32 layout, block 128: elements 0..3 of every lane are block
        // 2t, elements 4..7 are block 2t+1; each is a whole-warp maximum
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
            b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, o));
        }
        lo = a;
        hi = b;
    } else {
        // bf16 layout, block 128: lanes 0..15 are block 2t, 16..31 block 2t+1
        float m = fmaxf(a, b);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        lo = hi = m;
    }
}

// Encode this lane's 8 island-sum values into the payload at tile `tile`.
template <typename T, int CODEC, int BLOCK>
__device__ __forceinline__ void encode_store(void *payload, uint64_t scales_off, uint64_t tile,
                                             int lane, uint64_t n, bool full, const float v[8]) {
    const uint64_t base = tile * kTile;
    if constexpr (CODEC == GB_CODEC_NONE) {
        float *o = (float *)payload + base;
        if (full) {
            if constexpr (sizeof(T) == 4) {
                st_u4(o + 4 * lane, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                                               __float_as_uint(v[2]), __float_as_uint(v[3])));
                st_u4(o + 128 + 4 * lane, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]),
                                                     __float_as_uint(v[6]), __float_as_uint(v[7])));
            } else {
                st_u4(o + 8 * lane, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                                               __float_as_uint(v[2]), __float_as_uint(v[3])));
                st_u4(o + 8 * lane + 4, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]),
                                                   __float_as_uint(v[6]), __float_as_uint(v[7])));
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint64_t j = base + Lay<T>::idx(lane, k);
                if (j < n) ((float *)payload)[j] = v[k];
            }
        }
    } else if constexpr (CODEC == GB_CODEC_BF16) {
        unsigned short *o = (unsigned short *)payload + base;
        if (full) {
            const uint32_t c01 = cvt_bf16x2(v[0], v[1]), c23 = cvt_bf16x2(v[2], v[3]);
            const uint32_t c45 = cvt_bf16x2(v[4], v[5]), c67 = cvt_bf16x2(v[6], v[7]);
            if constexpr (sizeof(T) == 4) {
                st_u2(o + 4 * lane, make_uint2(c01, c23));
                st_u2(o + 128 + 4 * lane, make_uint2(c45, c67));
            } else {
                st_u4(o + 8 * lane, make_uint4(c01, c23, c45, c67));
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint64_t j = base + Lay<T>::idx(lane, k);
                if (j < n) ((unsigned short *)payload)[j] = (unsigned short)(cvt_bf16x2(v[k], 0.0f) & 0xFFFFu);
            }
        }
    } else {
        float mlo, mhi;
        block_absmax<T, BLOCK>(v, mlo, mhi);
        const int klo = block_scale_exp<CODEC>(mlo);
        const int khi = block_scale_exp<CODEC>(mhi);
        const float ilo = pow2f(-klo), ihi = pow2f(-khi);
        float y[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) y[k] = __fmul_rn(v[k], ilo);
#pragma unroll
        for (int k = 4; k < 8; ++k) y[k] = __fmul_rn(v[k], ihi);
        unsigned char *o = (unsigned char *)payload + base;
        if (full) {
            const uint32_t w0 = cvt_fp8x2<CODEC>(y[0], y[1]) | (cvt_fp8x2<CODEC>(y[2], y[3]) << 16);
            const uint32_t w1 = cvt_fp8x2<CODEC>(y[4], y[5]) | (cvt_fp8x2<CODEC>(y[6], y[7]) << 16);
            if constexpr (sizeof(T) == 4) {
                st_u1(o + 4 * lane, w0);
                st_u1(o + 128 + 4 * lane, w1);
            } else {
                st_u2(o + 8 * lane, make_uint2(w0, w1));
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                uint64_t j = base + Lay<T>::idx(lane, k);
                if (j < n) ((unsigned char *)payload)[j] = (unsigned char)(cvt_fp8x2<CODEC>(y[k], 0.0f) & 0xFFu);
            }
        }
        // scales: one float32 2^k per block of the tile that exists
        float *sc = (float *)((unsigned char *)payload + scales_off);
        const uint64_t nb = (n + BLOCK - 1) / BLOCK;
        if constexpr (BLOCK == 256) {
            if (lane == 0) sc[tile] = pow2f(klo);
        } else if constexpr (sizeof(T) == 4) {
            if (lane == 0) {
                sc[2 * tile] = pow2f(klo);
                if (2 * tile + 1 < nb) sc[2 * tile + 1] = pow2f(khi);
            }
        } else {
            if (lane == 0) sc[2 * tile] = pow2f(klo);
            if (lane == 16 && 2 * tile + 1 < nb) sc[2 * tile + 1] = pow2f(klo);
        }
    }
}

template <typename T, int CODEC, int BLOCK>
__global__ void __launch_bounds__(256) k_reduce_encode(const __grid_constant__ ReduceEncodeArgs a) {
    const int lane = threadIdx.x & 31;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    const uint64_t items = a.tiles * (uint64_t)a.n_islands;
    for (uint64_t it = warp; it < items; it += nwarps) {
        const int isl = (int)(it / a.tiles);
        const uint64_t tile = it - (uint64_t)isl * a.tiles;
        const uint64_t base = tile * kTile;
        const bool full = base + kTile <= a.n;
        const int r0 = a.first[isl];
        const int K = a.first[isl + 1] - r0;
        float v[8];
        load_rank<T>(a.src[r0], base, lane, a.n, full, v);
        // ascending rank order; four ranks' loads in flight at a time
        for (int q0 = 1; q0 < K; q0 += 4) {
            float w[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (q0 + u < K) load_rank<T>(a.src[r0 + q0 + u], base, lane, a.n, full, w[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (q0 + u < K) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) v[k] = __fadd_rn(v[k], w[u][k]);
                }
        }
        encode_store<T, CODEC, BLOCK>(a.payload[isl], a.scales_off, tile, lane, a.n, full, v);
    }
}

// ------------------------------------------------------------- the decoder

// Decode this lane's 8 elements of a payload; `gbase` is the element index
// (in the full buffer) of the lane layout's element 0.  In the element-wise
// path only elements whose local index (lbase + idx) is below `limit` are
// read; the others decode as 0.
template <typename T, int CODEC, int BLOCK>
__device__ __forceinline__ void decode_lane(const void *payload, uint64_t scales_off, uint64_t gbase,
                                            uint64_t lbase, uint64_t limit, int lane, bool full,
                                            float d[8]) {
    if (full) {
        if constexpr (CODEC == GB_CODEC_NONE) {
            const float *p = (const float *)payload + gbase;
            uint4 x, y;
            if constexpr (sizeof(T) == 4) {
                x = ld_u4(p + 4 * lane);
                y = ld_u4(p + 128 + 4 * lane);
            } else {
                x = ld_u4(p + 8 * lane);
                y = ld_u4(p + 8 * lane + 4);
            }
            d[0] = __uint_as_float(x.x); d[1] = __uint_as_float(x.y);
            d[2] = __uint_as_float(x.z); d[3] = __uint_as_float(x.w);
            d[4] = __uint_as_float(y.x); d[5] = __uint_as_float(y.y);
            d[6] = __uint_as_float(y.z); d[7] = __uint_as_float(y.w);
        } else if constexpr (CODEC == GB_CODEC_BF16) {
            const unsigned short *p = (const unsigned short *)payload + gbase;
            uint32_t w[4];
            if constexpr (sizeof(T) == 4) {
                uint2 x = ld_u2(p + 4 * lane), y = ld_u2(p + 128 + 4 * lane);
                w[0] = x.x; w[1] = x.y; w[2] = y.x; w[3] = y.y;
            } else {
                uint4 x = ld_u4(p + 8 * lane);
                w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                d[2 * i] = __uint_as_float(w[i] << 16);
                d[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else {
            const unsigned char *p = (const unsigned char *)payload + gbase;
            const float *sc = (const float *)((const unsigned char *)payload + scales_off);
            uint32_t w0, w1;
            float s0, s1;
            if constexpr (sizeof(T) == 4) {
                w0 = ld_u1(p + 4 * lane);
                w1 = ld_u1(p + 128 + 4 * lane);
                s0 = __ldg(sc + (gbase + 4 * lane) / BLOCK);
                s1 = __ldg(sc + (gbase + 128 + 4 * lane) / BLOCK);
            } else {
                uint2 x = ld_u2(p + 8 * lane);
                w0 = x.x;
                w1 = x.y;
                s0 = s1 = __ldg(sc + (gbase + 8 * lane) / BLOCK);
            }
            float c[8];
            fp8x2_to_f32<CODEC>(w0 & 0xFFFFu, c[0], c[1]);
            fp8x2_to_f32<CODEC>(w0 >> 16, c[2], c[3]);
            fp8x2_to_f32<CODEC>(w1 & 0xFFFFu, c[4], c[5]);
            fp8x2_to_f32<CODEC>(w1 >> 16, c[6], c[7]);
            // code value * 2^k is exact in float32 (k >= -126 keeps it at or
            // above the subnormal grid)
#pragma unroll
            for (int k = 0; k < 4; ++k) d[k] = __fmul_rn(c[k], s0);
#pragma unroll
            for (int k = 4; k < 8; ++k) d[k] = __fmul_rn(c[k], s1);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint64_t off = Lay<T>::idx(lane, k);
            d[k] = 0.0f;
            if (lbase + off < limit) {
                const uint64_t j = gbase + off;
                if constexpr (CODEC == GB_CODEC_NONE) {
                    d[k] = __ldg((const float *)payload + j);
                } else if constexpr (CODEC == GB_CODEC_BF16) {
                    d[k] = bf16_bits_to_f32(__ldg((const unsigned short *)payload + j));
                } else {
                    const float *sc = (const float *)((const unsigned char *)payload + scales_off);
                    float lo, hi;
                    fp8x2_to_f32<CODEC>(__ldg((const unsigned char *)payload + j), lo, hi);
                    d[k] = __fmul_rn(lo, __ldg(sc + j / BLOCK));
                }
            }
        }
    }
}

template <typename T, int CODEC, int BLOCK>
__global__ void __launch_bounds__(256) k_decode_bcast(const __grid_constant__ DecodeBcastArgs a) {
    const int lane = threadIdx.x & 31;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    const uint64_t units = a.rs ? (uint64_t)a.first[a.n_groups] : (uint64_t)a.n_groups;
    const uint64_t items = a.tiles * units;
    for (uint64_t it = warp; it < items; it += nwarps) {
        const int u = (int)(it / a.tiles);
        const uint64_t tile = it - (uint64_t)u * a.tiles;
        int g, r_lo, r_hi;
        uint64_t gbase, lbase = tile * kTile, limit;
        if (a.rs) {
            g = a.group_of_rank[u];
            r_lo = u;
            r_hi = u + 1;
            gbase = (uint64_t)u * a.m + lbase;
            limit = a.m;
        } else {
            g = u;
            r_lo = a.first[g];
            r_hi = a.first[g + 1];
            gbase = lbase;
            limit = a.n;
        }
        const bool full = a.vec && lbase + kTile <= limit;
        float t[8];
        decode_lane<T, CODEC, BLOCK>(a.payload[g][0], a.scales_off, gbase, lbase, limit, lane, full, t);
        // remaining islands in order, two payloads in flight at a time
        for (int j0 = 1; j0 < a.n_src; j0 += 2) {
            float d[2][8];
#pragma unroll
            for (int q = 0; q < 2; ++q)
                if (j0 + q < a.n_src)
                    decode_lane<T, CODEC, BLOCK>(a.payload[g][j0 + q], a.scales_off, gbase, lbase, limit,
                                                 lane, full, d[q]);
#pragma unroll
            for (int q = 0; q < 2; ++q)
                if (j0 + q < a.n_src) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) t[k] = __fadd_rn(t[k], d[q][k]);
                }
        }
        if (a.avg) {
#pragma unroll
            for (int k = 0; k < 8; ++k) t[k] = __fdiv_rn(t[k], a.world);
        }
        for (int r = r_lo; r < r_hi; ++r) store_rank<T>(a.dst[r], lbase, lane, limit, full, t);
    }
}

template <int CODEC, int BLOCK>
__global__ void __launch_bounds__(256) k_decompress_acc(const __grid_constant__ DecompressAccArgs a) {
    const int lane = threadIdx.x & 31;
    const uint64_t warp = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint64_t nwarps = ((uint64_t)gridDim.x * blockDim.x) >> 5;
    const uint64_t tiles = (a.n + kTile - 1) / kTile;
    for (uint64_t tile = warp; tile < tiles; tile += nwarps) {
        const uint64_t base = tile * kTile;
        const bool full = base + kTile <= a.n;
        float d[8];
        decode_lane<float, CODEC, BLOCK>(a.payload, a.scales_off, base, base, a.n, lane, full, d);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint64_t j = base + Lay<float>::idx(lane, k);
            if (j < a.n) a.accum[j] = a.accumulate ? __fadd_rn(a.accum[j], d[k]) : d[k];
        }
    }
}

__global__ void __launch_bounds__(256) k_copy(const __grid_constant__ CopyArgs a) {
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t nth = (uint64_t)gridDim.x * blockDim.x;
    if (a.vec) {
        const uint64_t chunks = a.bytes / 16;
        const uint64_t total = chunks * (uint64_t)a.n_jobs;
        for (uint64_t c = tid; c < total; c += nth) {
            const int j = (int)(c / chunks);
            const uint64_t off = (c - (uint64_t)j * chunks) * 16;
            const unsigned char *s = a.src[j] + off;
            const uint4 x = ld_stream_u4(s);
            for (int d = a.dst_lo[j]; d < a.dst_hi[j]; ++d) {
                unsigned char *p = a.dst[d] + a.dst_off[j] + off;
                if (p != s) st_stream_u4(p, x);
            }
        }
    } else {
        const uint64_t total = a.bytes * (uint64_t)a.n_jobs;
        for (uint64_t c = tid; c < total; c += nth) {
            const int j = (int)(c / a.bytes);
            const uint64_t off = c - (uint64_t)j * a.bytes;
            const unsigned char *s = a.src[j] + off;
            const unsigned char x = *s;
            for (int d = a.dst_lo[j]; d < a.dst_hi[j]; ++d) {
                unsigned char *p = a.dst[d] + a.dst_off[j] + off;
                if (p != s) *p = x;
            }
        }
    }
}

// ------------------------------------------------------------------ launch

static int sm_count() {
    static int count = 0;
    if (count == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev);
        if (count <= 0) count = 1;
    }
    return count;
}

// One resident wave of 256-thread blocks (or fewer when there is less work);
// the kernels walk their work items with a grid stride.  The occupancy is
// looked up once per kernel instantiation.
template <auto Kern, typename Args>
static cudaError_t launch(uint64_t warp_items, const Args &a, cudaStream_t s) {
    static int per_sm = 0;
    if (per_sm == 0) {
        int v = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, Kern, 256, 0);
        per_sm = v > 0 ? v : 1;
    }
    const uint64_t want = (warp_items + 7) / 8;
    const uint64_t cap = (uint64_t)per_sm * (uint64_t)sm_count();
    const uint64_t g = want < cap ? want : cap;
    Kern<<<(unsigned)(g ? g : 1), 256, 0, s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
}

#define GB_DISPATCH_CODEC(T, KERNEL, ITEMS, ARGS, S)                                           \
    switch (codec) {                                                                           \
    case GB_CODEC_NONE: return launch<KERNEL<T, GB_CODEC_NONE, 256>>(ITEMS, ARGS, S);          \
    case GB_CODEC_BF16: return launch<KERNEL<T, GB_CODEC_BF16, 256>>(ITEMS, ARGS, S);          \
    case GB_CODEC_E4M3:                                                                        \
        return block == 128 ? launch<KERNEL<T, GB_CODEC_E4M3, 128>>(ITEMS, ARGS, S)            \
                            : launch<KERNEL<T, GB_CODEC_E4M3, 256>>(ITEMS, ARGS, S);           \
    case GB_CODEC_E5M2:                                                                        \
        return block == 128 ? launch<KERNEL<T, GB_CODEC_E5M2, 128>>(ITEMS, ARGS, S)            \
                            : launch<KERNEL<T, GB_CODEC_E5M2, 256>>(ITEMS, ARGS, S);           \
    default: return cudaErrorInvalidValue;                                                     \
    }

cudaError_t launch_reduce_encode(const ReduceEncodeArgs &a, int dtype, int codec, int block,
                                 cudaStream_t s) {
    const uint64_t items = a.tiles * (uint64_t)a.n_islands;
    if (dtype == GB_F32) {
        GB_DISPATCH_CODEC(float, k_reduce_encode, items, a, s)
    } else {
        GB_DISPATCH_CODEC(bf16, k_reduce_encode, items, a, s)
    }
}

cudaError_t launch_decode_bcast(const DecodeBcastArgs &a, int dtype, int codec, int block,
                                cudaStream_t s) {
    const uint64_t units = a.rs ? (uint64_t)a.first[a.n_groups] : (uint64_t)a.n_groups;
    const uint64_t items = a.tiles * units;
    if (dtype == GB_F32) {
        GB_DISPATCH_CODEC(float, k_decode_bcast, items, a, s)
    } else {
        GB_DISPATCH_CODEC(bf16, k_decode_bcast, items, a, s)
    }
}

cudaError_t launch_decompress_accumulate(const DecompressAccArgs &a, int codec, int block,
                                         cudaStream_t s) {
    const uint64_t items = (a.n + kTile - 1) / kTile;
    switch (codec) {
    case GB_CODEC_NONE: return launch<k_decompress_acc<GB_CODEC_NONE, 256>>(items, a, s);
    case GB_CODEC_BF16: return launch<k_decompress_acc<GB_CODEC_BF16, 256>>(items, a, s);
    case GB_CODEC_E4M3:
        return block == 128 ? launch<k_decompress_acc<GB_CODEC_E4M3, 128>>(items, a, s)
                            : launch<k_decompress_acc<GB_CODEC_E4M3, 256>>(items, a, s);
    case GB_CODEC_E5M2:
        return block == 128 ? launch<k_decompress_acc<GB_CODEC_E5M2, 128>>(items, a, s)
                            : launch<k_decompress_acc<GB_CODEC_E5M2, 256>>(items, a, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_copy(const CopyArgs &a, cudaStream_t s) {
    const uint64_t units = a.vec ? a.bytes / 16 : a.bytes;
    const uint64_t threads = units * (uint64_t)a.n_jobs;
    return launch<k_copy>((threads + 31) / 32, a, s);
}

}  // namespace gb
