// Decode + accumulate + broadcast, decompress-accumulate, and exact copies
// (sm_103a).
//
// What is computed (gpubridge README, "Bridge compression" and "all_reduce
// uses reduce-bridge-broadcast"): each leader decodes every island's payload
// (its own included) and adds them in float32 in island order; AVG divides
// once by the world size (API table, all_reduce row); the total, rounded to
// the rank dtype, goes to every rank of the island.
//
// How: the host passes the payloads once, as one output group holding all
// W ranks (every leader would compute the same bits), so each payload is
// read and decoded once.  One warp per 256-element tile per output unit
// (grid y: a group of ranks; reduce_scatter has its own kernel, one grid
// row per rank's slice), 8 contiguous elements per lane; the payloads of a
// tile are all loaded before the first add (compile-time count for 1 or 2
// islands), and for those counts the loads of the warp's next tile are
// issued before the current one is decoded and stored; the result leaves as
// one 32-byte (float32; two 16-byte halves when a rank buffer is only
// 16-byte aligned) or 16-byte (bf16) streaming store per lane per rank.
// The exact copies (all_gather, broadcast) take one grid row per copy job.
#include <atomic>
#include <cuda_runtime.h>

#include "gb_device.cuh"
#include "gb_kernels.cuh"

namespace gb {

using bf16 = __nv_bfloat16;

static std::atomic<uint64_t> g_launches{0};
uint64_t launches() { return g_launches.load(); }
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

int sm_count() {
    static const int count = [] {  // initialised once, thread-safe
        int dev = 0, v = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        return v > 0 ? v : 1;
    }();
    return count;
}

// The raw payload bits of one lane's 8 elements of a full tile: the codes
// and, for fp8, the block scale.  Loading them is split from decoding them
// so that a warp can have the next tile's loads in flight while it decodes
// and stores the current one.
template <int CODEC> struct RawLane;
template <> struct RawLane<GB_CODEC_NONE> { U8x32 x; };
template <> struct RawLane<GB_CODEC_BF16> { uint4 x; };
template <> struct RawLane<GB_CODEC_E4M3> { uint2 x; float s; };
template <> struct RawLane<GB_CODEC_E5M2> { uint2 x; float s; };

template <int CODEC, int BLOCK>
__device__ __forceinline__ void load_raw(const void *payload, uint64_t scales_off, uint64_t gbase, int lane,
                                         RawLane<CODEC> &r) {
    if constexpr (CODEC == GB_CODEC_NONE) {
        r.x = ld_v8((const float *)payload + gbase + 8 * lane);
    } else if constexpr (CODEC == GB_CODEC_BF16) {
        r.x = ld_u4((const unsigned short *)payload + gbase + 8 * lane);
    } else {
        const uint64_t j0 = gbase + 8 * lane;
        r.x = ld_u2((const unsigned char *)payload + j0);
        r.s = __ldg((const float *)((const unsigned char *)payload + scales_off) + j0 / BLOCK);
    }
}

template <int CODEC>
__device__ __forceinline__ void decode_raw(const RawLane<CODEC> &r, float d[8]) {
    if constexpr (CODEC == GB_CODEC_NONE) {
#pragma unroll
        for (int k = 0; k < 8; ++k) d[k] = __uint_as_float(r.x.w[k]);
    } else if constexpr (CODEC == GB_CODEC_BF16) {
        const uint32_t w[4] = {r.x.x, r.x.y, r.x.z, r.x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            d[2 * i] = __uint_as_float(w[i] << 16);
            d[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        float c[8];
        fp8x2_to_f32<CODEC>(r.x.x & 0xFFFFu, c[0], c[1]);
        fp8x2_to_f32<CODEC>(r.x.x >> 16, c[2], c[3]);
        fp8x2_to_f32<CODEC>(r.x.y & 0xFFFFu, c[4], c[5]);
        fp8x2_to_f32<CODEC>(r.x.y >> 16, c[6], c[7]);
        // code value * 2^k is exact in float32: k >= -126 keeps every
        // product on or above the subnormal grid
#pragma unroll
        for (int k = 0; k < 8; ++k) d[k] = __fmul_rn(c[k], r.s);
    }
}

// Decode this lane's 8 elements of a payload.  `gbase` is the index, in the
// full buffer, of the tile's first element; in the element-wise path only
// elements whose index within the output unit (lbase + offset) is below
// `limit` are read, the others decode as 0.
template <int CODEC, int BLOCK>
__device__ __forceinline__ void decode_lane(const void *payload, uint64_t scales_off, uint64_t gbase,
                                            uint64_t lbase, uint64_t limit, int lane, bool full, float d[8]) {
    if (full) {
        RawLane<CODEC> r;
        load_raw<CODEC, BLOCK>(payload, scales_off, gbase, lane, r);
        decode_raw<CODEC>(r, d);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint64_t off = lane_elem(lane, k);
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

// Write this lane's 8 float32 results to a rank buffer of type T (bf16:
// round to nearest even), streaming (A16: float32 rank buffers only
// 16-byte aligned).
template <typename T, bool A16>
__device__ __forceinline__ void store_rank(void *p, uint64_t lbase, int lane, uint64_t limit, bool full,
                                           const float t[8]) {
    if constexpr (sizeof(T) == 4) {
        float *f = (float *)p;
        if (full) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(t[k]);
            st_stream_f32x8<A16>(f + lbase + 8 * lane, w);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t j = lbase + lane_elem(lane, k);
                if (j < limit) f[j] = t[k];
            }
        }
    } else {
        unsigned short *h = (unsigned short *)p;
        if (full) {
            st_stream_u4(h + lbase + 8 * lane, make_uint4(cvt_bf16x2(t[0], t[1]), cvt_bf16x2(t[2], t[3]),
                                                          cvt_bf16x2(t[4], t[5]), cvt_bf16x2(t[6], t[7])));
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t j = lbase + lane_elem(lane, k);
                if (j < limit) h[j] = (unsigned short)(cvt_bf16x2(t[k], 0.0f) & 0xFFFFu);
            }
        }
    }
}

// AVG and the stores of one tile's totals to ranks r_lo .. r_hi - 1.
template <typename T, bool A16>
__device__ __forceinline__ void finish_tile(const DecodeBcastArgs &a, int r_lo, int r_hi, uint64_t lbase, int lane,
                                            uint64_t limit, bool full, float t[8]) {
    if (a.avg) {
        // t / W; for W = 2^e the product with 2^-e is the same correctly
        // rounded quotient (one rounding of the same real number)
        if (a.world_pow2) {
#pragma unroll
            for (int k = 0; k < 8; ++k) t[k] = __fmul_rn(t[k], a.inv_world);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) t[k] = __fdiv_rn(t[k], a.world);
        }
    }
    for (int r = r_lo; r < r_hi; ++r) store_rank<T, A16>(a.dst[r], lbase, lane, limit, full, t);
}

// NS > 0: exactly NS payloads (loads unrolled); NS == 0: a.n_src of them.
// A16: some float32 rank buffer is only 16-byte aligned (launched with
// NS == 0).
template <typename T, int CODEC, int BLOCK, int NS, bool A16 = false>
__global__ void __launch_bounds__(256) k_decode_bcast(const __grid_constant__ DecodeBcastArgs a) {
    const int u = blockIdx.y;
    const int lane = threadIdx.x & 31;
    int g, r_lo, r_hi;
    uint64_t gofs, limit;
    if (a.rs) {
        g = a.group_of_rank[u];
        r_lo = u;
        r_hi = u + 1;
        gofs = a.rs_src[u];
        limit = a.rs_len[u];
    } else {
        g = u;
        r_lo = a.first[g];
        r_hi = a.first[g + 1];
        gofs = 0;
        limit = a.n;
    }
    const int nsrc = NS > 0 ? NS : a.n_src;
    const uint32_t wpb = blockDim.x >> 5;
    const uint32_t stride = gridDim.x * wpb;
    uint32_t tile = blockIdx.x * wpb + (threadIdx.x >> 5) + wait_prior_grid();
    if constexpr (NS > 0) {
        // Full tiles (vector path), software-pipelined: the payload loads of
        // the warp's next tile are in flight while the current one is decoded
        // and stored.  tiles < 2^31 (n < 2^39), so tile + stride never wraps.
        const uint32_t nfull = a.vec ? (uint32_t)(limit / kTile) : 0u;
        RawLane<CODEC> cur[NS];
        if (tile < nfull) {
#pragma unroll
            for (int q = 0; q < NS; ++q)
                load_raw<CODEC, BLOCK>(a.payload[g][q], a.scales_off, gofs + (uint64_t)tile * kTile, lane, cur[q]);
        }
        while (tile < nfull) {
            const uint32_t nxt = tile + stride;
            RawLane<CODEC> nx[NS];
            if (nxt < nfull) {
#pragma unroll
                for (int q = 0; q < NS; ++q)
                    load_raw<CODEC, BLOCK>(a.payload[g][q], a.scales_off, gofs + (uint64_t)nxt * kTile, lane, nx[q]);
            }
            float t[8];
            decode_raw<CODEC>(cur[0], t);
#pragma unroll
            for (int q = 1; q < NS; ++q) {
                float d[8];
                decode_raw<CODEC>(cur[q], d);
#pragma unroll
                for (int k = 0; k < 8; ++k) t[k] = __fadd_rn(t[k], d[k]);  // island order
            }
            finish_tile<T, A16>(a, r_lo, r_hi, (uint64_t)tile * kTile, lane, limit, true, t);
#pragma unroll
            for (int q = 0; q < NS; ++q) cur[q] = nx[q];
            tile = nxt;
        }
    }
    // the rest: every tile when NS == 0, else the ragged last tile (or all
    // tiles when vector accesses are off), element by element
    for (; tile < a.tiles; tile += stride) {
        const uint64_t lbase = (uint64_t)tile * kTile;
        const uint64_t gbase = gofs + lbase;
        const bool full = a.vec && lbase + kTile <= limit;
        float t[8];
        decode_lane<CODEC, BLOCK>(a.payload[g][0], a.scales_off, gbase, lbase, limit, lane, full, t);
        for (int j0 = 1; j0 < nsrc; j0 += 2) {  // two payloads in flight at a time
            float d[2][8];
#pragma unroll
            for (int q = 0; q < 2; ++q)
                if (j0 + q < nsrc)
                    decode_lane<CODEC, BLOCK>(a.payload[g][j0 + q], a.scales_off, gbase, lbase, limit, lane, full,
                                              d[q]);
#pragma unroll
            for (int q = 0; q < 2; ++q)
                if (j0 + q < nsrc) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) t[k] = __fadd_rn(t[k], d[q][k]);
                }
        }
        finish_tile<T, A16>(a, r_lo, r_hi, lbase, lane, limit, full, t);
    }
}

// reduce_scatter's decode (grid y = rank r): rank r's slice only, one
// output per tile.  A warp writes 1 KiB per tile here against 4 KiB in the
// all_reduce decode, so the work per warp is small and the grid holds about
// one tile per warp: the next-tile prefetch of k_decode_bcast buys nothing
// and its registers cost occupancy (40 against 32 per thread, 6 against 8
// resident blocks per SM).  The NS payloads of a full tile are all loaded
// before the first decode.
template <typename T, int CODEC, int BLOCK, int NS, bool A16 = false>
__global__ void __launch_bounds__(256, (NS > 0 && !A16) ? 8 : 1) k_decode_slices(const __grid_constant__ DecodeBcastArgs a) {
    const int u = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int g = a.group_of_rank[u];
    const uint64_t gofs = a.rs_src[u], limit = a.rs_len[u];
    const int nsrc = NS > 0 ? NS : a.n_src;
    const uint32_t wpb = blockDim.x >> 5;
    const uint32_t stride = gridDim.x * wpb;
    const uint32_t nfull = a.vec ? (uint32_t)(limit / kTile) : 0u;
    for (uint32_t tile = blockIdx.x * wpb + (threadIdx.x >> 5) + wait_prior_grid(); tile < a.tiles; tile += stride) {
        const uint64_t lbase = (uint64_t)tile * kTile;
        float t[8];
        if (NS > 0 && tile < nfull) {
            RawLane<CODEC> r[NS > 0 ? NS : 1];
#pragma unroll
            for (int q = 0; q < NS; ++q) load_raw<CODEC, BLOCK>(a.payload[g][q], a.scales_off, gofs + lbase, lane, r[q]);
            decode_raw<CODEC>(r[0], t);
#pragma unroll
            for (int q = 1; q < NS; ++q) {
                float d[8];
                decode_raw<CODEC>(r[q], d);
#pragma unroll
                for (int k = 0; k < 8; ++k) t[k] = __fadd_rn(t[k], d[k]);  // island order
            }
            finish_tile<T, A16>(a, u, u + 1, lbase, lane, limit, true, t);
        } else {
            const bool full = tile < nfull;
            decode_lane<CODEC, BLOCK>(a.payload[g][0], a.scales_off, gofs + lbase, lbase, limit, lane, full, t);
            for (int j = 1; j < nsrc; ++j) {
                float d[8];
                decode_lane<CODEC, BLOCK>(a.payload[g][j], a.scales_off, gofs + lbase, lbase, limit, lane, full, d);
#pragma unroll
                for (int k = 0; k < 8; ++k) t[k] = __fadd_rn(t[k], d[k]);
            }
            finish_tile<T, A16>(a, u, u + 1, lbase, lane, limit, full, t);
        }
    }
}

template <int CODEC, int BLOCK>
__global__ void __launch_bounds__(256) k_decompress_acc(const __grid_constant__ DecompressAccArgs a) {
    const int lane = threadIdx.x & 31;
    const uint32_t wpb = blockDim.x >> 5;
    const uint32_t tiles = (uint32_t)((a.n + kTile - 1) / kTile);
    const uint32_t first = blockIdx.x * wpb + (threadIdx.x >> 5) + wait_prior_grid();
    for (uint32_t tile = first; tile < tiles; tile += gridDim.x * wpb) {
        const uint64_t base = (uint64_t)tile * kTile;
        const bool full = base + kTile <= a.n;
        float d[8];
        decode_lane<CODEC, BLOCK>(a.payload, a.scales_off, base, base, a.n, lane, full, d);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint64_t j = base + lane_elem(lane, k);
            if (j < a.n) a.accum[j] = a.accumulate ? __fadd_rn(a.accum[j], d[k]) : d[k];
        }
    }
}

// Grid row j copies job j.  With vectors (VB = 16 or 32 bytes, when every
// address and the length are multiples of VB) a thread moves 64 bytes per
// step as 64 / VB vectors spaced a grid apart (each warp instruction covers
// 32 * VB contiguous bytes), all loaded before the first store.  32-byte
// vectors halve the store instructions, which otherwise fill the
// load/store queue (ncu: lg_throttle stalls).
template <int VB> struct CopyVec;
template <> struct CopyVec<16> {
    uint4 x;
    __device__ __forceinline__ void ld(const unsigned char *p) { x = ld_stream_u4(p); }
    __device__ __forceinline__ void st(unsigned char *p) const { st_stream_u4(p, x); }
};
template <> struct CopyVec<32> {
    U8x32 x;
    __device__ __forceinline__ void ld(const unsigned char *p) { x = ld_stream_v8(p); }
    __device__ __forceinline__ void st(unsigned char *p) const { st_stream_v8(p, x.w); }
};

template <int VB>
__global__ void __launch_bounds__(256) k_copy(const __grid_constant__ CopyArgs a) {
    const int j = blockIdx.y;
    const unsigned char *s = a.src[j];
    const int d_lo = a.dst_lo[j], d_hi = a.dst_hi[j];
    const uint64_t off = a.dst_off[j];
    const uint64_t nth = (uint64_t)gridDim.x * blockDim.x;
    uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x + wait_prior_grid();
    if constexpr (VB > 0) {
        constexpr int U = 64 / VB;
        const uint64_t chunks = a.bytes / VB;
        for (; t < chunks; t += U * nth) {
            CopyVec<VB> x[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (t + u * nth < chunks) x[u].ld(s + VB * (t + u * nth));
            for (int d = d_lo; d < d_hi; ++d) {
                unsigned char *p = a.dst[d] + off;
                if (p == s) continue;  // the source itself (a leader's received block)
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (t + u * nth < chunks) x[u].st(p + VB * (t + u * nth));
            }
        }
    } else {
        for (; t < a.bytes; t += nth) {
            const unsigned char x = s[t];
            for (int d = d_lo; d < d_hi; ++d) {
                unsigned char *p = a.dst[d] + off;
                if (p != s) p[t] = x;
            }
        }
    }
}

// ------------------------------------------------------------------ launch

template <typename T, int CODEC, int BLOCK>
static cudaError_t dispatch_ns(const DecodeBcastArgs &a, cudaStream_t s) {
    const unsigned units = a.rs ? (unsigned)a.first[a.n_groups] : (unsigned)a.n_groups;
    const bool a16 = sizeof(T) == 4 && any_a16((const void *const *)a.dst, a.first[a.n_groups]);
    if (a.rs) {
        if (a16) return launch_grid<k_decode_slices<T, CODEC, BLOCK, 0, true>>(a.tiles, units, a, s);
        switch (a.n_src) {
        case 1: return launch_grid<k_decode_slices<T, CODEC, BLOCK, 1>>(a.tiles, units, a, s);
        case 2: return launch_grid<k_decode_slices<T, CODEC, BLOCK, 2>>(a.tiles, units, a, s);
        default: return launch_grid<k_decode_slices<T, CODEC, BLOCK, 0>>(a.tiles, units, a, s);
        }
    }
    if (a16) return launch_grid<k_decode_bcast<T, CODEC, BLOCK, 0, true>>(a.tiles, units, a, s);
    switch (a.n_src) {
    case 1: return launch_grid<k_decode_bcast<T, CODEC, BLOCK, 1>>(a.tiles, units, a, s);
    case 2: return launch_grid<k_decode_bcast<T, CODEC, BLOCK, 2>>(a.tiles, units, a, s);
    default: return launch_grid<k_decode_bcast<T, CODEC, BLOCK, 0>>(a.tiles, units, a, s);
    }
}

template <typename T>
static cudaError_t dispatch_codec(const DecodeBcastArgs &a, int codec, int block, cudaStream_t s) {
    switch (codec) {
    case GB_CODEC_NONE: return dispatch_ns<T, GB_CODEC_NONE, 256>(a, s);
    case GB_CODEC_BF16: return dispatch_ns<T, GB_CODEC_BF16, 256>(a, s);
    case GB_CODEC_E4M3:
        return block == 128 ? dispatch_ns<T, GB_CODEC_E4M3, 128>(a, s) : dispatch_ns<T, GB_CODEC_E4M3, 256>(a, s);
    case GB_CODEC_E5M2:
        return block == 128 ? dispatch_ns<T, GB_CODEC_E5M2, 128>(a, s) : dispatch_ns<T, GB_CODEC_E5M2, 256>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_bcast(const DecodeBcastArgs &a, int dtype, int codec, int block, cudaStream_t s) {
    return dtype == GB_F32 ? dispatch_codec<float>(a, codec, block, s) : dispatch_codec<bf16>(a, codec, block, s);
}

cudaError_t launch_decompress_accumulate(const DecompressAccArgs &a, int codec, int block, cudaStream_t s) {
    const uint64_t tiles = (a.n + kTile - 1) / kTile;
    switch (codec) {
    case GB_CODEC_NONE: return launch_grid<k_decompress_acc<GB_CODEC_NONE, 256>>(tiles, 1, a, s);
    case GB_CODEC_BF16: return launch_grid<k_decompress_acc<GB_CODEC_BF16, 256>>(tiles, 1, a, s);
    case GB_CODEC_E4M3:
        return block == 128 ? launch_grid<k_decompress_acc<GB_CODEC_E4M3, 128>>(tiles, 1, a, s)
                            : launch_grid<k_decompress_acc<GB_CODEC_E4M3, 256>>(tiles, 1, a, s);
    case GB_CODEC_E5M2:
        return block == 128 ? launch_grid<k_decompress_acc<GB_CODEC_E5M2, 128>>(tiles, 1, a, s)
                            : launch_grid<k_decompress_acc<GB_CODEC_E5M2, 256>>(tiles, 1, a, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_copy(const CopyArgs &a, cudaStream_t s) {
    // launch_grid counts 8 warps of 32 threads per block, so it is given warps
    bool v32 = a.vec && a.bytes % 32 == 0;
    for (int j = 0; v32 && j < a.n_jobs; ++j) {
        v32 = ((uintptr_t)a.src[j] & 31u) == 0 && a.dst_off[j] % 32 == 0;
        for (int d = a.dst_lo[j]; v32 && d < a.dst_hi[j]; ++d) v32 = ((uintptr_t)a.dst[d] & 31u) == 0;
    }
    // 64 bytes per thread: warps = bytes / (64 * 32)
    if (v32 || a.vec) return (v32 ? launch_grid<k_copy<32>, CopyArgs> : launch_grid<k_copy<16>, CopyArgs>)(
                          (a.bytes + 2047) / 2048, (unsigned)a.n_jobs, a, s);
    return launch_grid<k_copy<0>>((a.bytes + 31) / 32, (unsigned)a.n_jobs, a, s);
}

}  // namespace gb
