// Kernel argument blocks and launchers of libgb (host-visible declarations).
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "gb.h"

namespace gb {

// Fused island reduce + bridge encode over every island at once (grid y =
// island).  Island i's ranks are src[first[i] .. first[i+1]); its payload
// goes to payload[i] (codes at offset 0, fp8 scales at scales_off).
struct ReduceEncodeArgs {
    const void *src[GB_MAX_RANKS];
    void *payload[GB_MAX_ISLANDS];
    float *residual[GB_MAX_ISLANDS];  // error feedback (all null: none)
    int first[GB_MAX_ISLANDS + 1];
    int n_islands;
    uint64_t n;
    uint32_t tiles;       // warp tiles per island = ceil(n / 256)
    uint64_t scales_off;  // byte offset of the fp8 scales in a payload
};

// Fused decode + accumulate + broadcast (grid y = output unit).
// Output group g (one group of all W ranks when the payloads are decoded
// once, see decode_once; an island's ranks for per-leader rows) reads the n_src payloads
// payload[g][0..n_src) (island order), adds their decoded values in float32,
// divides by W for AVG (an exact multiply by 1/W when W is a power of two),
// rounds to the rank dtype and writes the result.
//   all_reduce (rs == 0): unit = group g; every rank buffer
//     dst[first[g] .. first[g+1]) receives the same elements;
//   reduce_scatter (rs == 1): unit = rank r; the unit's rs_len[r] elements
//     start at payload element rs_src[r] and go to dst[r] (the host offsets
//     dst[r] to the slice position they land on); group g =
//     group_of_rank[r].  One chunk of the pipeline covers the parts of the slices that fall
//     inside it.  vec == 0 forces the element-wise path (used when the slice
//     length is not a multiple of 8, which would misalign vector accesses).
struct DecodeBcastArgs {
    void *dst[GB_MAX_RANKS];
    const void *payload[GB_MAX_ISLANDS][GB_MAX_ISLANDS];
    int first[GB_MAX_ISLANDS + 1];
    int group_of_rank[GB_MAX_RANKS];
    int n_groups;
    int n_src;
    int avg;
    int world_pow2;  // W is a power of two
    float world;
    float inv_world;
    uint64_t n;      // elements of the full buffer
    uint64_t scales_off;
    int rs;
    int vec;
    uint64_t rs_src[GB_MAX_RANKS];  // reduce_scatter: first payload element of unit r
    uint64_t rs_len[GB_MAX_RANKS];  // reduce_scatter: elements of unit r (0: none)
    uint32_t tiles;  // all_reduce: tiles per group; reduce_scatter: tiles of the longest unit
};

// One decode for every rank.  Every leader would compute the same total
// from the same payload bits, so on one GPU a single pass over the payloads
// as they crossed the bridge (received[j]: island j's part, as some other
// leader received it; with one island, its own) writes all W ranks.
inline void decode_once(DecodeBcastArgs &da, int W, int I, const void *const *received) {
    da.n_groups = 1;
    da.first[0] = 0;
    da.first[1] = W;
    for (int r = 0; r < W; ++r) da.group_of_rank[r] = 0;
    da.n_src = I;
    for (int j = 0; j < I; ++j) da.payload[0][j] = received[j];
}

// accum = dec(payload) or accum + dec(payload).
struct DecompressAccArgs {
    const void *payload;
    float *accum;
    uint64_t n;
    uint64_t scales_off;
    int accumulate;
};

// Exact copies: job j copies `bytes` from src[j] into dst[d] + dst_off[j]
// for every d in [dst_lo[j], dst_hi[j]), skipping a destination that is the
// source itself.
struct CopyArgs {
    const unsigned char *src[GB_MAX_RANKS];
    uint64_t dst_off[GB_MAX_RANKS];
    int dst_lo[GB_MAX_RANKS];
    int dst_hi[GB_MAX_RANKS];
    unsigned char *dst[GB_MAX_RANKS];
    int n_jobs;
    uint64_t bytes;
    int vec;  // all addresses and `bytes` multiples of 16
};

// Launchers: return the cudaError_t of the launch.  `units` is the grid's y
// extent (islands, or ranks for reduce_scatter).
cudaError_t launch_reduce_encode(const ReduceEncodeArgs &a, int dtype, int codec, int block,
                                 cudaStream_t s);
cudaError_t launch_decode_bcast(const DecodeBcastArgs &a, int dtype, int codec, int block,
                                cudaStream_t s);
cudaError_t launch_decompress_accumulate(const DecompressAccArgs &a, int codec, int block,
                                         cudaStream_t s);
cudaError_t launch_copy(const CopyArgs &a, cudaStream_t s);

// The exact path (MAX / MIN, float16, float64, integers): island fold into
// payload[i] (ReduceEncodeArgs: src, payload, first, n_islands, n), then the
// fold of the payloads into the ranks (DecodeBcastArgs as for decode; vec:
// 16-byte accesses allowed, i.e. for reduce_scatter m is a multiple of
// 16 / sizeof(dtype)).
cudaError_t launch_exact_reduce(const ReduceEncodeArgs &a, int dtype, int op, cudaStream_t s);
cudaError_t launch_exact_combine(const DecodeBcastArgs &a, int dtype, int op, cudaStream_t s);
size_t exact_payload_elem_bytes(int dtype, int op);

uint64_t launches();
void count_launch();
int sm_count();

// 256-thread blocks, one 256-element tile per warp, over `units` grid rows;
// the kernels walk their tiles with a grid stride.  The grid follows the
// work rather than one resident wave: with several waves, blocks that finish
// early are replaced by new ones, so the last tiles are spread over every SM
// instead of leaving the tail to the few warps that hold one tile more (on a
// 25 MiB float32 bucket per rank this took 9 % off the decode kernel and 4 %
// off the encode, back to back).
// It is capped at kMaxWaves resident waves, after which warps loop.  The
// occupancy is looked up once per kernel instantiation.
constexpr uint64_t kMaxWaves = 32;
template <auto Kern, typename Args>
cudaError_t launch_grid(uint64_t tiles_per_unit, unsigned units, const Args &a, cudaStream_t s) {
    static const int per_sm = [] {  // initialised once, thread-safe
        int v = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, Kern, 256, 0);
        return v > 0 ? v : 1;
    }();
    const uint64_t cap = kMaxWaves * (uint64_t)per_sm * (uint64_t)sm_count();
    const uint64_t per_unit_cap = cap / units > 0 ? cap / units : 1;
    const uint64_t want = (tiles_per_unit + 7) / 8;  // 8 warps (tiles) per block
    const uint64_t gx = want < per_unit_cap ? want : per_unit_cap;
    // programmatic dependent launch: the grid may be scheduled while the
    // previous kernel on the stream drains; the kernel itself waits for that
    // kernel's completion before touching memory (wait_prior_grid)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(gx ? gx : 1), units);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, Kern, a);
    count_launch();
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear it: the caller reports e
        return e;
    }
    return cudaGetLastError();
}

}  // namespace gb
