// gb_all_reduce_noalloc: the reduce-bridge-broadcast all_reduce without any
// memory allocation, for callers that must not allocate.
//
// Who needs it: code that runs where a cudaMalloc / cudaHostAlloc is not an
// option -- a gradient hook inside a training step whose framework has
// already reserved nearly all device memory in its own caching allocator (a
// cudaMalloc there can fail, and the cudaFree that growing staging implies
// waits for the whole device), or a host process that must not pin more
// memory.  gb_all_reduce grows context-owned device and pinned staging on
// demand; this variant instead uses
//   - one file-scope __device__ array of GB_NOALLOC_DEVICE_BYTES for the
//     payloads (own + received), present on every GPU that loads the
//     library until the process exits, and
//   - one file-scope host array of GB_NOALLOC_HOST_BYTES for the bridge
//     slots, in ordinary pageable memory (the copies are then synchronous
//     for the host, like the pageable default of the pages' bridge).
// It produces the same bits as gb_all_reduce (same kernels, same payload
// layout per island, same island order).
#include <mutex>

#include "gb_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_scratch[GB_NOALLOC_DEVICE_BYTES];
alignas(256) static unsigned char g_host_slots[GB_NOALLOC_HOST_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per
// device).  In host code `g_scratch` only names a host-side shadow symbol,
// so the kernels must be given this address, never &g_scratch.
gb_status scratch_address(int dev, unsigned char **out) {
    if (dev < 0 || dev >= kMaxDevices) return GB_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return GB_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = (unsigned char *)g_scratch_addr[dev];
    return GB_OK;
}

// The host slots hold I payload slots and the device array I * I: the
// device bound keeps I * slot <= GB_NOALLOC_DEVICE_BYTES / I, within the host
// array for every I >= 2, so one size check covers both.
static_assert(2ull * GB_NOALLOC_HOST_BYTES >= GB_NOALLOC_DEVICE_BYTES, "host slots smaller than the device bound");

}  // namespace

extern "C" gb_status gb_all_reduce_noalloc(gb_ctx *ctx, void *const *rank_bufs, size_t n,
                                           gb_dtype dtype, gb_op op, gb_codec codec, int block,
                                           gb_stream stream) {
    // ---- validation: the checks of gb_all_reduce (arguments first, the
    // device after them), restricted to the codec path, plus the size limit
    using namespace gbrt;
    GB_TRY(check_ctx(ctx));
    GB_TRY(check_codec_dtype(ctx, dtype));
    if (op != GB_SUM && op != GB_AVG) return set_msg(ctx, GB_ERR_UNSUPPORTED_OP, "noalloc all_reduce takes SUM / AVG");
    GB_TRY(check_codec(ctx, codec, block));
    GB_TRY(check_n(ctx, n));
    const int I = ctx->I, W = ctx->W;
    GB_TRY(check_rank_bufs(ctx, (const void *const *)rank_bufs, W, "rank_bufs"));
    if (n == 0) return GB_OK;
    const int eff = I == 1 ? GB_CODEC_NONE : (int)codec;
    const int blk = is_fp8(eff) ? block : 256;
    const size_t P = payload_bytes(eff, blk, n);
    const size_t slot = round_up(P, 256);
    // own payloads (I slots), then each leader's received payloads (I - 1 slots each)
    if (slot > GB_NOALLOC_DEVICE_BYTES / ((size_t)I * I))
        return set_msg(ctx, GB_ERR_TOO_LARGE, "%d x %d payload slots of %zu bytes exceed the fixed %u bytes", I, I,
                       slot, (unsigned)GB_NOALLOC_DEVICE_BYTES);

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_msg(ctx, GB_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    }
    dev = seen_device(ctx, dev);
    if (ctx->device >= 0 && dev != ctx->device)
        return set_msg(ctx, GB_ERR_INVALID_ARG, "context is bound to device %d, current device is %d", ctx->device,
                       dev);
    unsigned char *scratch = nullptr;
    if (scratch_address(dev, &scratch) != GB_OK)
        return set_msg(ctx, GB_ERR_CUDA, "cudaGetSymbolAddress of the fixed staging array failed");
    cudaStream_t s = (cudaStream_t)stream;

    // ---- island reduce + encode into the own-payload slots
    gb::ReduceEncodeArgs ra;
    memset(&ra, 0, sizeof ra);
    for (int r = 0; r < W; ++r) ra.src[r] = rank_bufs[r];
    for (int i = 0; i < I; ++i) ra.payload[i] = scratch + (size_t)i * slot;
    for (int i = 0; i <= I; ++i) ra.first[i] = ctx->first[i];
    ra.n_islands = I;
    ra.n = n;
    ra.tiles = (uint32_t)((n + gb::kTile - 1) / gb::kTile);
    ra.scales_off = is_fp8(eff) ? round_up(n, 16) : P;
    if (gb::launch_reduce_encode(ra, dtype, eff, blk, s) != cudaSuccess) return GB_ERR_CUDA;

    // ---- bridge hop through the host slots: own slots out, others' in
    unsigned char *inbox = scratch + (size_t)I * slot;
    if (I > 1) {
        if (cudaMemcpyAsync(g_host_slots, scratch, (size_t)(I - 1) * slot + P, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess)
            return GB_ERR_BRIDGE;
        for (int g = 0; g < I; ++g) {
            unsigned char *mine = inbox + (size_t)g * (I - 1) * slot;
            if (g > 0 && cudaMemcpyAsync(mine, g_host_slots, (size_t)(g - 1) * slot + P,
                                         cudaMemcpyHostToDevice, s) != cudaSuccess)
                return GB_ERR_BRIDGE;
            if (g < I - 1 && cudaMemcpyAsync(mine + (size_t)g * slot, g_host_slots + (size_t)(g + 1) * slot,
                                             (size_t)(I - g - 2) * slot + P, cudaMemcpyHostToDevice,
                                             s) != cudaSuccess)
                return GB_ERR_BRIDGE;
        }
    }

    // ---- decode + accumulate (island order) + broadcast to every rank
    gb::DecodeBcastArgs da;
    memset(&da, 0, sizeof da);
    for (int r = 0; r < W; ++r) {
        da.dst[r] = rank_bufs[r];
        da.group_of_rank[r] = ctx->island_of[r];
    }
    const void *received[GB_MAX_ISLANDS];
    for (int j = 0; j < I; ++j) {
        const int g = (j + 1) % I;  // the leader whose received copy of island j is read
        received[j] = I == 1 ? (const void *)scratch
                             : (const void *)(inbox + ((size_t)g * (I - 1) + (j < g ? j : j - 1)) * slot);
    }
    gb::decode_once(da, W, I, received);
    da.avg = op == GB_AVG;
    da.world = (float)W;
    da.world_pow2 = (W & (W - 1)) == 0;
    da.inv_world = 1.0f / (float)W;
    da.n = n;
    da.scales_off = ra.scales_off;
    da.rs = 0;
    da.vec = 1;
    da.tiles = ra.tiles;
    if (gb::launch_decode_bcast(da, dtype, eff, blk, s) != cudaSuccess) return GB_ERR_CUDA;
    return GB_OK;
}
