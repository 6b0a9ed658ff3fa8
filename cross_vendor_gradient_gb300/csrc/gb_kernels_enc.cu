// Island reduce + bridge encode (sm_103a).
//
// What is computed (gpubridge README, "all_reduce uses reduce-bridge-
// broadcast" and "Bridge compression"): per island, the float32 sum of its
// rank buffers in ascending rank order, then the island sum encoded for the
// bridge: raw float32, bf16 (nearest even), or OCP fp8 with one power-of-two
// float32 scale per block of 128 / 256 values.
//
// How: one warp per 256-element tile, 8 contiguous elements per lane.  The
// K rank loads of a tile are all issued before the first add (compile-time K
// for islands of 1, 2 or 4 ranks), the fp8 block maximum is a warp-shuffle
// reduction, and the codes leave as one 8-byte store per lane (a 256-byte
// coalesced warp store).  Nothing crosses warps, so the result does not
// depend on the grid.
#include <cuda_runtime.h>

#include "gb_device.cuh"
#include "gb_kernels.cuh"

namespace gb {

using bf16 = __nv_bfloat16;

// This lane's 8 elements of rank buffer `p` in tile `base`, as float32
// (A16: float32 rank buffers only 16-byte aligned).
template <typename T, bool A16>
__device__ __forceinline__ void load_rank(const void *p, uint64_t base, int lane, uint64_t n, bool full,
                                          float v[8]) {
    if constexpr (sizeof(T) == 4) {
        if (full) {
            const U8x32 x = ld_stream_f32x8<A16>((const float *)p + base + 8 * lane);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = __uint_as_float(x.w[k]);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t j = base + lane_elem(lane, k);
                v[k] = j < n ? __ldg((const float *)p + j) : 0.0f;
            }
        }
    } else {
        if (full) {
            const uint4 x = ld_stream_u4((const unsigned short *)p + base + 8 * lane);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(w[i] << 16);
                v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t j = base + lane_elem(lane, k);
                v[k] = j < n ? bf16_bits_to_f32(__ldg((const unsigned short *)p + j)) : 0.0f;
            }
        }
    }
}

// Largest magnitude of the lane's codec block: the whole warp for blocks of
// 256, the lane's half-warp for blocks of 128.
template <int BLOCK>
__device__ __forceinline__ float block_absmax(const float v[8]) {
    float m = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                    fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
#pragma unroll
    for (int o = (BLOCK == 256 ? 16 : 8); o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    return m;
}

// Encode this lane's 8 island-sum values into the payload at tile `tile`.
// With DEC, dec[] receives the decoded value of every code written (the
// value the receiving leaders will add), for error feedback.
template <int CODEC, int BLOCK, bool DEC>
__device__ __forceinline__ void encode_store(unsigned char *payload, uint64_t scales_off, uint32_t tile,
                                             int lane, uint64_t n, bool full, const float v[8], float dec[8]) {
    const uint64_t base = (uint64_t)tile * kTile;
    if constexpr (CODEC == GB_CODEC_NONE) {
        float *o = (float *)payload;
        if (full) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(v[k]);
            st_v8(o + base + 8 * lane, w);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t j = base + lane_elem(lane, k);
                if (j < n) o[j] = v[k];
            }
        }
        if constexpr (DEC) {
#pragma unroll
            for (int k = 0; k < 8; ++k) dec[k] = v[k];
        }
    } else if constexpr (CODEC == GB_CODEC_BF16) {
        unsigned short *o = (unsigned short *)payload;
        const uint32_t c[4] = {cvt_bf16x2(v[0], v[1]), cvt_bf16x2(v[2], v[3]), cvt_bf16x2(v[4], v[5]),
                               cvt_bf16x2(v[6], v[7])};
        if (full) {
            st_u4(o + base + 8 * lane, make_uint4(c[0], c[1], c[2], c[3]));
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t j = base + lane_elem(lane, k);
                if (j < n) o[j] = (unsigned short)((k & 1) ? (c[k >> 1] >> 16) : (c[k >> 1] & 0xFFFFu));
            }
        }
        if constexpr (DEC) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dec[2 * i] = __uint_as_float(c[i] << 16);
                dec[2 * i + 1] = __uint_as_float(c[i] & 0xFFFF0000u);
            }
        }
    } else {
        const int kexp = block_scale_exp<CODEC>(block_absmax<BLOCK>(v));
        const float inv = pow2f(-kexp);
        float y[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = __fmul_rn(v[k], inv);  // exact, or below fp8 half-ulp
        const uint32_t p[4] = {cvt_fp8x2<CODEC>(y[0], y[1]), cvt_fp8x2<CODEC>(y[2], y[3]),
                               cvt_fp8x2<CODEC>(y[4], y[5]), cvt_fp8x2<CODEC>(y[6], y[7])};
        unsigned char *o = payload;
        if (full) {
            st_u2(o + base + 8 * lane, make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16)));
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t j = base + lane_elem(lane, k);
                if (j < n) o[j] = (unsigned char)((k & 1) ? (p[k >> 1] >> 8) : (p[k >> 1] & 0xFFu));
            }
        }
        if constexpr (DEC) {
            const float sc = pow2f(kexp);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float lo, hi;
                fp8x2_to_f32<CODEC>(p[i], lo, hi);
                dec[2 * i] = __fmul_rn(lo, sc);  // exact
                dec[2 * i + 1] = __fmul_rn(hi, sc);
            }
        }
        // one float32 scale 2^k per existing block of the tile
        float *sc = (float *)(payload + scales_off);
        if constexpr (BLOCK == 256) {
            if (lane == 0) sc[tile] = pow2f(kexp);
        } else {
            const uint64_t nb = (n + BLOCK - 1) / BLOCK;
            const uint64_t b = 2 * (uint64_t)tile + (lane >> 4);
            if ((lane & 15) == 0 && b < nb) sc[b] = pow2f(kexp);
        }
    }
}

// The island sum of this lane's 8 elements of the tile at `base` (ascending
// rank order).  KT > 0: exactly KT ranks, all loads issued before the first
// add; KT == 0: K ranks, four ranks' loads in flight at a time.
template <typename T, int KT, bool A16>
__device__ __forceinline__ void island_sum(const ReduceEncodeArgs &a, int r0, int K, uint64_t base, int lane,
                                           bool full, float v[8]) {
    if constexpr (KT > 0) {
        float w[KT][8];
#pragma unroll
        for (int q = 0; q < KT; ++q) load_rank<T, A16>(a.src[r0 + q], base, lane, a.n, full, w[q]);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = w[0][k];
#pragma unroll
        for (int q = 1; q < KT; ++q)
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = __fadd_rn(v[k], w[q][k]);
    } else {
        load_rank<T, A16>(a.src[r0], base, lane, a.n, full, v);
        for (int q0 = 1; q0 < K; q0 += 4) {
            float w[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (q0 + u < K) load_rank<T, A16>(a.src[r0 + q0 + u], base, lane, a.n, full, w[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (q0 + u < K) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) v[k] = __fadd_rn(v[k], w[u][k]);
                }
        }
    }
}

// Tiles a warp takes per step.  bf16 ranks move 16 bytes per lane per tile,
// half of float32's 32, so with a fixed island size a warp takes two
// adjacent tiles and issues all 2 * KT rank loads before the first add: the
// same bytes in flight per warp as float32 (on 8 ranks of bf16 this was the
// difference between 0.78 and 0.9 of the copy peak).
template <typename T, int KT, bool EF>
constexpr int kTilesPerStep = (sizeof(T) == 2 && KT > 0 && !EF) ? 2 : 1;

// KT > 0: every island has KT ranks (loads unrolled); KT == 0: any sizes.
// EF: error feedback -- encode s + r and keep r = (s + r) - dec(codes) in
// the island's residual buffer (float32, n elements).  A16: some float32
// rank buffer is only 16-byte aligned (launched with KT == 0).
template <typename T, int CODEC, int BLOCK, int KT, bool EF, bool A16 = false>
__global__ void __launch_bounds__(256) k_reduce_encode(const __grid_constant__ ReduceEncodeArgs a) {
    const int isl = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int r0 = a.first[isl];
    const int K = KT > 0 ? KT : a.first[isl + 1] - r0;
    const uint32_t wpb = blockDim.x >> 5;
    const uint32_t stride = gridDim.x * wpb;
    const uint64_t n = a.n;
    unsigned char *payload = (unsigned char *)a.payload[isl];
    const uint32_t warp0 = blockIdx.x * wpb + (threadIdx.x >> 5) + wait_prior_grid();
    if constexpr (kTilesPerStep<T, KT, EF> == 2) {
        const uint32_t steps = (a.tiles + 1) / 2;
        for (uint32_t st = warp0; st < steps; st += stride) {
            const uint32_t t0 = 2 * st;
            uint4 raw[2][KT > 0 ? KT : 1];
            bool full[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // every load of both tiles before any add
                const uint64_t base = (uint64_t)(t0 + h) * kTile;
                full[h] = t0 + h < a.tiles && base + kTile <= n;
                if (full[h]) {
#pragma unroll
                    for (int q = 0; q < KT; ++q)
                        raw[h][q] = ld_stream_u4((const unsigned short *)a.src[r0 + q] + base + 8 * lane);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t tile = t0 + h;
                if (tile >= a.tiles) break;
                const uint64_t base = (uint64_t)tile * kTile;
                float v[8];
                if (full[h]) {
#pragma unroll
                    for (int q = 0; q < KT; ++q) {
                        const uint32_t w[4] = {raw[h][q].x, raw[h][q].y, raw[h][q].z, raw[h][q].w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
                            v[2 * i] = q == 0 ? lo : __fadd_rn(v[2 * i], lo);  // ascending rank order
                            v[2 * i + 1] = q == 0 ? hi : __fadd_rn(v[2 * i + 1], hi);
                        }
                    }
                } else {
                    island_sum<T, KT, A16>(a, r0, K, base, lane, false, v);
                }
                encode_store<CODEC, BLOCK, false>(payload, a.scales_off, tile, lane, n, full[h], v, nullptr);
            }
        }
    } else {
        for (uint32_t tile = warp0; tile < a.tiles; tile += stride) {
            const uint64_t base = (uint64_t)tile * kTile;
            const bool full = base + kTile <= n;
            float v[8];
            island_sum<T, KT, A16>(a, r0, K, base, lane, full, v);
            if constexpr (EF) {
                float *res = a.residual[isl];
                float r[8], dec[8];
                if (full) {
                    const U8x32 x = ld_rw_v8(res + base + 8 * lane);
#pragma unroll
                    for (int k = 0; k < 8; ++k) r[k] = __uint_as_float(x.w[k]);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint64_t j = base + lane_elem(lane, k);
                        r[k] = j < n ? res[j] : 0.0f;
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = __fadd_rn(v[k], r[k]);
                encode_store<CODEC, BLOCK, true>(payload, a.scales_off, tile, lane, n, full, v, dec);
                if (full) {
                    uint32_t w[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__fsub_rn(v[k], dec[k]));
                    st_v8(res + base + 8 * lane, w);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint64_t j = base + lane_elem(lane, k);
                        if (j < n) res[j] = __fsub_rn(v[k], dec[k]);
                    }
                }
            } else {
                encode_store<CODEC, BLOCK, false>(payload, a.scales_off, tile, lane, n, full, v, nullptr);
            }
        }
    }
}

template <typename T, int CODEC, int BLOCK, bool EF>
static cudaError_t dispatch_k(const ReduceEncodeArgs &a, cudaStream_t s) {
    int K = a.first[1] - a.first[0];
    for (int i = 1; i < a.n_islands; ++i)
        if (a.first[i + 1] - a.first[i] != K) K = 0;
    const unsigned units = (unsigned)a.n_islands;
    // the grid counts warp steps: tiles, or tile pairs (kTilesPerStep)
    constexpr int P = kTilesPerStep<T, 1, EF>;
    const uint64_t steps = (a.tiles + P - 1) / P;
    if (sizeof(T) == 4 && any_a16(a.src + a.first[0], a.first[a.n_islands] - a.first[0]))
        return launch_grid<k_reduce_encode<T, CODEC, BLOCK, 0, EF, true>>(a.tiles, units, a, s);
    switch (K) {
    case 1: return launch_grid<k_reduce_encode<T, CODEC, BLOCK, 1, EF>>(steps, units, a, s);
    case 2: return launch_grid<k_reduce_encode<T, CODEC, BLOCK, 2, EF>>(steps, units, a, s);
    case 4: return launch_grid<k_reduce_encode<T, CODEC, BLOCK, 4, EF>>(steps, units, a, s);
    default: return launch_grid<k_reduce_encode<T, CODEC, BLOCK, 0, EF>>(a.tiles, units, a, s);
    }
}

template <typename T, int CODEC, int BLOCK>
static cudaError_t dispatch_ef(const ReduceEncodeArgs &a, cudaStream_t s) {
    return a.residual[0] ? dispatch_k<T, CODEC, BLOCK, true>(a, s) : dispatch_k<T, CODEC, BLOCK, false>(a, s);
}

template <typename T>
static cudaError_t dispatch_codec(const ReduceEncodeArgs &a, int codec, int block, cudaStream_t s) {
    switch (codec) {
    case GB_CODEC_NONE: return dispatch_ef<T, GB_CODEC_NONE, 256>(a, s);
    case GB_CODEC_BF16: return dispatch_ef<T, GB_CODEC_BF16, 256>(a, s);
    case GB_CODEC_E4M3:
        return block == 128 ? dispatch_ef<T, GB_CODEC_E4M3, 128>(a, s) : dispatch_ef<T, GB_CODEC_E4M3, 256>(a, s);
    case GB_CODEC_E5M2:
        return block == 128 ? dispatch_ef<T, GB_CODEC_E5M2, 128>(a, s) : dispatch_ef<T, GB_CODEC_E5M2, 256>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_reduce_encode(const ReduceEncodeArgs &a, int dtype, int codec, int block, cudaStream_t s) {
    return dtype == GB_F32 ? dispatch_codec<float>(a, codec, block, s) : dispatch_codec<bf16>(a, codec, block, s);
}

}  // namespace gb
