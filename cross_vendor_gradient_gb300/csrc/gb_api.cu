// Host side of libgb: contexts, argument validation, staging buffers, the
// bridge hop through pinned host memory, and the collectives composed from
// the kernels in gb_kernels.cu.  Declarations and contracts: include/gb.h.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include <cuda_runtime.h>

#include "gb.h"
#include "gb_device.cuh"
#include "gb_kernels.cuh"

using gb::round_up;

struct gb_ctx {
    int I = 0, W = 0;
    int size[GB_MAX_ISLANDS] = {};
    int first[GB_MAX_ISLANDS + 1] = {};
    int island_of[GB_MAX_RANKS] = {};
    int device = -1;
    gb_status sticky = GB_OK;
    char msg[256] = {};
    int inject = 0;
    // device staging: I own-payload slots, then I x I inbox slots
    unsigned char *d_stage = nullptr;
    size_t d_stage_bytes = 0;
    // pinned host staging: the bridge slots
    unsigned char *h_stage = nullptr;
    size_t h_stage_bytes = 0;
    // device copies of host rank buffers (gb_all_reduce_host)
    unsigned char *d_ranks = nullptr;
    size_t d_ranks_bytes = 0;
    // ordering of staging reuse across calls
    cudaEvent_t done = nullptr;
    bool done_recorded = false;
    cudaStream_t last_stream = nullptr;
    // phase timing (observer marks): a ring of `tcap` records of 4 events
    int tcap = 0;
    cudaEvent_t *tev = nullptr;
    long long tcount = 0;   // collectives recorded so far
    bool ev_bridge = false;
};

namespace {

constexpr uint64_t kMaxElems = 1ull << 38;

gb_status set_msg(gb_ctx *c, gb_status s, const char *fmt, ...) {
    if (c) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(c->msg, sizeof c->msg, fmt, ap);
        va_end(ap);
    }
    return s;
}

// A failure after validation: the context becomes failed for good.
gb_status fail(gb_ctx *c, gb_status s, const char *what, cudaError_t e = cudaSuccess) {
    c->sticky = s;
    if (e != cudaSuccess)
        snprintf(c->msg, sizeof c->msg, "%s: %s", what, cudaGetErrorString(e));
    else
        snprintf(c->msg, sizeof c->msg, "%s", what);
    return s;
}

size_t elem_bytes(gb_dtype d) { return d == GB_F32 ? 4 : 2; }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

gb_status check_ctx(gb_ctx *c) {
    if (!c) return GB_ERR_INVALID_ARG;
    if (c->sticky != GB_OK) return GB_ERR_CONTEXT_FAILED;
    return GB_OK;
}

gb_status check_dtype(gb_ctx *c, int d) {
    if (d != GB_F32 && d != GB_BF16) return set_msg(c, GB_ERR_UNSUPPORTED_DTYPE, "dtype %d", d);
    return GB_OK;
}

gb_status check_op(gb_ctx *c, int op) {
    if (op != GB_SUM && op != GB_AVG) return set_msg(c, GB_ERR_UNSUPPORTED_OP, "op %d", op);
    return GB_OK;
}

bool codec_ok(int codec, int block) {
    switch (codec) {
    case GB_CODEC_NONE:
    case GB_CODEC_BF16: return true;
    case GB_CODEC_E4M3:
    case GB_CODEC_E5M2: return block == 128 || block == 256;
    default: return false;
    }
}

gb_status check_codec(gb_ctx *c, int codec, int block) {
    if (!codec_ok(codec, block))
        return set_msg(c, GB_ERR_UNSUPPORTED_CODEC, "codec %d block %d", codec, block);
    return GB_OK;
}

gb_status check_n(gb_ctx *c, size_t n) {
    if ((uint64_t)n > kMaxElems) return set_msg(c, GB_ERR_INVALID_ARG, "n = %zu too large", n);
    return GB_OK;
}

gb_status check_dev_bufs(gb_ctx *c, const void *const *bufs, int count, const char *name) {
    if (!bufs) return set_msg(c, GB_ERR_INVALID_ARG, "%s is NULL", name);
    for (int r = 0; r < count; ++r) {
        if (!bufs[r]) return set_msg(c, GB_ERR_INVALID_ARG, "%s[%d] is NULL", name, r);
        if (!aligned16(bufs[r])) return set_msg(c, GB_ERR_MISALIGNED, "%s[%d] not 16-byte aligned", name, r);
    }
    return GB_OK;
}

gb_status check_dev_ptr(gb_ctx *c, const void *p, const char *name) {
    if (!p) return set_msg(c, GB_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(p)) return set_msg(c, GB_ERR_MISALIGNED, "%s not 16-byte aligned", name);
    return GB_OK;
}

#define GB_TRY(expr)                         \
    do {                                     \
        gb_status _s = (expr);               \
        if (_s != GB_OK) return _s;          \
    } while (0)

// Bind the context to the current device on first use.
gb_status bind(gb_ctx *c) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_msg(c, GB_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    }
    if (c->device < 0) {
        if ((e = cudaEventCreateWithFlags(&c->done, cudaEventDisableTiming)) != cudaSuccess)
            return fail(c, GB_ERR_CUDA, "cudaEventCreate", e);
        c->device = dev;
    } else if (dev != c->device) {
        return set_msg(c, GB_ERR_INVALID_ARG, "context is bound to device %d, current device is %d",
                       c->device, dev);
    }
    return GB_OK;
}

// The previous call's use of the staging buffers precedes this one.
gb_status begin(gb_ctx *c, cudaStream_t s) {
    if (c->done_recorded && c->last_stream != s) {
        cudaError_t e = cudaStreamWaitEvent(s, c->done, 0);
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaStreamWaitEvent", e);
    }
    return GB_OK;
}

gb_status end(gb_ctx *c, cudaStream_t s) {
    cudaError_t e = cudaEventRecord(c->done, s);
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaEventRecord", e);
    c->done_recorded = true;
    c->last_stream = s;
    return GB_OK;
}

gb_status mark(gb_ctx *c, int i, cudaStream_t s) {
    if (c->tcap <= 0) return GB_OK;
    cudaEvent_t &ev = c->tev[(size_t)(c->tcount % c->tcap) * 4 + i];
    cudaError_t e = cudaSuccess;
    if (!ev && (e = cudaEventCreate(&ev)) != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaEventCreate", e);
    if ((e = cudaEventRecord(ev, s)) != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaEventRecord", e);
    if (i == 3) ++c->tcount;
    return GB_OK;
}

void free_marks(gb_ctx *c) {
    if (c->tev) {
        for (int i = 0; i < 4 * c->tcap; ++i)
            if (c->tev[i]) cudaEventDestroy(c->tev[i]);
        delete[] c->tev;
    }
    c->tev = nullptr;
    c->tcap = 0;
    c->tcount = 0;
}

gb_status grow_device(gb_ctx *c, unsigned char **buf, size_t *have, size_t need) {
    if (need <= *have) return GB_OK;
    if (c->inject == GB_INJECT_ALLOC) {
        c->inject = 0;
        return fail(c, GB_ERR_ALLOC, "device staging allocation failed (injected)");
    }
    if (*buf) {
        cudaFree(*buf);  // waits for the device
        *buf = nullptr;
        *have = 0;
    }
    const size_t bytes = round_up(need, 2u << 20);
    cudaError_t e = cudaMalloc((void **)buf, bytes);
    if (e != cudaSuccess) {
        *buf = nullptr;
        return fail(c, GB_ERR_ALLOC, "cudaMalloc of device staging", e);
    }
    *have = bytes;
    return GB_OK;
}

gb_status grow_host(gb_ctx *c, size_t need) {
    if (need <= c->h_stage_bytes) return GB_OK;
    if (c->inject == GB_INJECT_ALLOC) {
        c->inject = 0;
        return fail(c, GB_ERR_ALLOC, "pinned staging allocation failed (injected)");
    }
    if (c->h_stage) {
        cudaFreeHost(c->h_stage);  // waits for the device
        c->h_stage = nullptr;
        c->h_stage_bytes = 0;
    }
    const size_t bytes = round_up(need, 2u << 20);
    cudaError_t e = cudaHostAlloc((void **)&c->h_stage, bytes, cudaHostAllocDefault);
    if (e != cudaSuccess) {
        c->h_stage = nullptr;
        return fail(c, GB_ERR_ALLOC, "cudaHostAlloc of the bridge slots", e);
    }
    c->h_stage_bytes = bytes;
    return GB_OK;
}

size_t payload_bytes(int codec, int block, size_t n) {
    switch (codec) {
    case GB_CODEC_NONE: return 4 * n;
    case GB_CODEC_BF16: return 2 * n;
    case GB_CODEC_E4M3:
    case GB_CODEC_E5M2: return round_up(n, 16) + 4 * ((n + block - 1) / block);
    default: return 0;
    }
}

size_t scales_offset(int codec, size_t n) {
    return (codec == GB_CODEC_E4M3 || codec == GB_CODEC_E5M2) ? round_up(n, 16) : payload_bytes(codec, 256, n);
}

// Staging needed by a reduce-bridge-broadcast over n elements.
void rbb_staging(const gb_ctx *c, size_t n, int codec, int block, size_t *dev, size_t *host,
                 size_t *slot) {
    const int eff = c->I == 1 ? GB_CODEC_NONE : codec;
    *slot = round_up(payload_bytes(eff, block, n), 256);
    *dev = (size_t)(c->I + (c->I > 1 ? c->I * c->I : 0)) * *slot;
    *host = c->I > 1 ? (size_t)c->I * *slot : 0;
}

gb_status check_launch(gb_ctx *c, cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, what, e);
    return GB_OK;
}

gb_status copy_async(gb_ctx *c, void *dst, const void *src, size_t bytes, cudaMemcpyKind kind,
                     cudaStream_t s) {
    if (bytes == 0) return GB_OK;
    cudaError_t e = cudaMemcpyAsync(dst, src, bytes, kind, s);
    if (e != cudaSuccess) return fail(c, GB_ERR_BRIDGE, "bridge copy", e);
    return GB_OK;
}

// The bridge hop of reduce-bridge-broadcast: every island's payload (slot i
// of the device outbox) goes to pinned host slot i; every leader i receives
// the other islands' slots into its inbox.  All on the caller's stream.
gb_status bridge_exchange(gb_ctx *c, size_t P, size_t slot, cudaStream_t s) {
    const int I = c->I;
    if (c->inject == GB_INJECT_BRIDGE) {
        c->inject = 0;
        return fail(c, GB_ERR_BRIDGE, "bridge hop failed (injected)");
    }
    unsigned char *outbox = c->d_stage;
    unsigned char *inbox = c->d_stage + (size_t)I * slot;
    // leaders -> host (the own-payload slots are contiguous: one copy)
    GB_TRY(copy_async(c, c->h_stage, outbox, (size_t)(I - 1) * slot + P, cudaMemcpyDeviceToHost, s));
    // host -> every leader, the slots of the other islands
    for (int i = 0; i < I; ++i) {
        unsigned char *mine = inbox + (size_t)i * I * slot;
        if (i > 0)
            GB_TRY(copy_async(c, mine, c->h_stage, (size_t)(i - 1) * slot + P, cudaMemcpyHostToDevice, s));
        if (i < I - 1)
            GB_TRY(copy_async(c, mine + (size_t)(i + 1) * slot, c->h_stage + (size_t)(i + 1) * slot,
                              (size_t)(I - i - 2) * slot + P, cudaMemcpyHostToDevice, s));
    }
    return GB_OK;
}

// Reduce-bridge-broadcast over W rank buffers `in` (n elements).  rs == 0:
// the total goes to out[r] (all n elements; out may equal in).  rs == 1:
// out[r] receives slice r (n / W elements).
gb_status run_rbb(gb_ctx *c, const void *const *in, void *const *out, size_t n, gb_dtype dtype,
                  gb_op op, gb_codec codec, int block, cudaStream_t s, int rs) {
    const int I = c->I;
    const int eff = I == 1 ? GB_CODEC_NONE : (int)codec;
    const int blk = (eff == GB_CODEC_E4M3 || eff == GB_CODEC_E5M2) ? block : 256;
    size_t dev, host, slot;
    rbb_staging(c, n, eff, blk, &dev, &host, &slot);
    const size_t P = payload_bytes(eff, blk, n);
    GB_TRY(grow_device(c, &c->d_stage, &c->d_stage_bytes, dev));
    if (host) GB_TRY(grow_host(c, host));
    GB_TRY(begin(c, s));
    GB_TRY(mark(c, 0, s));

    gb::ReduceEncodeArgs ra;
    memset(&ra, 0, sizeof ra);
    for (int r = 0; r < c->W; ++r) ra.src[r] = in[r];
    for (int i = 0; i < I; ++i) ra.payload[i] = c->d_stage + (size_t)i * slot;
    for (int i = 0; i <= I; ++i) ra.first[i] = c->first[i];
    ra.n_islands = I;
    ra.n = n;
    ra.tiles = (n + gb::kTile - 1) / gb::kTile;
    ra.scales_off = scales_offset(eff, n);
    GB_TRY(check_launch(c, gb::launch_reduce_encode(ra, dtype, eff, blk, s), "island reduce + encode"));
    GB_TRY(mark(c, 1, s));

    if (I > 1) GB_TRY(bridge_exchange(c, P, slot, s));
    c->ev_bridge = I > 1;
    GB_TRY(mark(c, 2, s));

    gb::DecodeBcastArgs da;
    memset(&da, 0, sizeof da);
    for (int r = 0; r < c->W; ++r) {
        da.dst[r] = out[r];
        da.group_of_rank[r] = c->island_of[r];
    }
    unsigned char *inbox = c->d_stage + (size_t)I * slot;
    for (int g = 0; g < I; ++g)
        for (int j = 0; j < I; ++j)
            da.payload[g][j] = (j == g) ? (const void *)(c->d_stage + (size_t)j * slot)
                                        : (const void *)(inbox + ((size_t)g * I + j) * slot);
    for (int i = 0; i <= I; ++i) da.first[i] = c->first[i];
    da.n_groups = I;
    da.n_src = I;
    da.avg = op == GB_AVG;
    da.world = (float)c->W;
    da.n = n;
    da.scales_off = scales_offset(eff, n);
    if (rs) {
        da.rs = 1;
        da.m = n / (size_t)c->W;
        da.vec = (da.m % 8) == 0;
        da.tiles = (da.m + gb::kTile - 1) / gb::kTile;
    } else {
        da.rs = 0;
        da.vec = 1;
        da.m = 0;
        da.tiles = (n + gb::kTile - 1) / gb::kTile;
    }
    if (da.tiles > 0)
        GB_TRY(check_launch(c, gb::launch_decode_bcast(da, dtype, eff, blk, s), "decode + broadcast"));
    GB_TRY(mark(c, 3, s));
    return end(c, s);
}

gb_status check_collective(gb_ctx *c, size_t n, int dtype, int op, int codec, int block) {
    GB_TRY(check_dtype(c, dtype));
    GB_TRY(check_op(c, op));
    GB_TRY(check_codec(c, codec, block));
    GB_TRY(check_n(c, n));
    return GB_OK;
}

}  // namespace

extern "C" {

gb_status gb_create(gb_ctx **out, int n_islands, const int *island_sizes) {
    if (!out || !island_sizes || n_islands < 1 || n_islands > GB_MAX_ISLANDS) return GB_ERR_INVALID_ARG;
    int W = 0;
    for (int i = 0; i < n_islands; ++i) {
        if (island_sizes[i] < 1) return GB_ERR_INVALID_ARG;
        W += island_sizes[i];
        if (W > GB_MAX_RANKS) return GB_ERR_INVALID_ARG;
    }
    gb_ctx *c = new (std::nothrow) gb_ctx();
    if (!c) return GB_ERR_ALLOC;
    c->I = n_islands;
    c->W = W;
    int r = 0;
    for (int i = 0; i < n_islands; ++i) {
        c->size[i] = island_sizes[i];
        c->first[i] = r;
        for (int q = 0; q < island_sizes[i]; ++q) c->island_of[r + q] = i;
        r += island_sizes[i];
    }
    c->first[n_islands] = W;
    *out = c;
    return GB_OK;
}

gb_status gb_destroy(gb_ctx *c) {
    if (!c) return GB_OK;
    if (c->device >= 0) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (cur != c->device) cudaSetDevice(c->device);
        if (c->done_recorded) cudaEventSynchronize(c->done);
        if (c->d_stage) cudaFree(c->d_stage);
        if (c->d_ranks) cudaFree(c->d_ranks);
        if (c->h_stage) cudaFreeHost(c->h_stage);
        if (c->done) cudaEventDestroy(c->done);
        free_marks(c);
        if (cur >= 0 && cur != c->device) cudaSetDevice(cur);
    }
    delete c;
    return GB_OK;
}

int gb_world_size(const gb_ctx *c) { return c ? c->W : -1; }
int gb_n_islands(const gb_ctx *c) { return c ? c->I : -1; }
int gb_island_size(const gb_ctx *c, int i) { return (c && i >= 0 && i < c->I) ? c->size[i] : -1; }
int gb_island_first_rank(const gb_ctx *c, int i) { return (c && i >= 0 && i < c->I) ? c->first[i] : -1; }
int gb_island_of_rank(const gb_ctx *c, int r) { return (c && r >= 0 && r < c->W) ? c->island_of[r] : -1; }

gb_status gb_context_status(const gb_ctx *c) { return c ? c->sticky : GB_ERR_INVALID_ARG; }
const char *gb_last_error_message(const gb_ctx *c) { return c ? c->msg : "NULL context"; }

const char *gb_status_string(gb_status s) {
    switch (s) {
    case GB_OK: return "GB_OK";
    case GB_ERR_INVALID_ARG: return "GB_ERR_INVALID_ARG";
    case GB_ERR_UNSUPPORTED_DTYPE: return "GB_ERR_UNSUPPORTED_DTYPE";
    case GB_ERR_UNSUPPORTED_OP: return "GB_ERR_UNSUPPORTED_OP";
    case GB_ERR_UNSUPPORTED_CODEC: return "GB_ERR_UNSUPPORTED_CODEC";
    case GB_ERR_MISALIGNED: return "GB_ERR_MISALIGNED";
    case GB_ERR_ALLOC: return "GB_ERR_ALLOC";
    case GB_ERR_CUDA: return "GB_ERR_CUDA";
    case GB_ERR_BRIDGE: return "GB_ERR_BRIDGE";
    case GB_ERR_CONTEXT_FAILED: return "GB_ERR_CONTEXT_FAILED";
    case GB_ERR_NO_DEVICE: return "GB_ERR_NO_DEVICE";
    case GB_ERR_TOO_LARGE: return "GB_ERR_TOO_LARGE";
    default: return "GB_ERR_UNKNOWN";
    }
}

size_t gb_payload_bytes(gb_codec codec, int block, size_t n) {
    if (!codec_ok(codec, block)) return 0;
    return payload_bytes(codec, block, n);
}

size_t gb_payload_scales_offset(gb_codec codec, int block, size_t n) {
    if (!codec_ok(codec, block)) return 0;
    return scales_offset(codec, n);
}

gb_status gb_reserve(gb_ctx *c, size_t n, gb_dtype dtype, gb_codec codec, int block) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_dtype(c, dtype));
    GB_TRY(check_codec(c, codec, block));
    GB_TRY(check_n(c, n));
    GB_TRY(bind(c));
    size_t dev, host, slot;
    rbb_staging(c, n, codec, block, &dev, &host, &slot);
    const size_t ag_host = (size_t)c->W * n * elem_bytes(dtype);
    GB_TRY(grow_device(c, &c->d_stage, &c->d_stage_bytes, dev));
    GB_TRY(grow_host(c, host > ag_host ? host : ag_host));
    return GB_OK;
}

gb_status gb_island_reduce(gb_ctx *c, int island, const void *const *rank_bufs, size_t n,
                           gb_dtype dtype, float *island_sum, gb_stream stream) {
    GB_TRY(check_ctx(c));
    if (island < 0 || island >= c->I) return set_msg(c, GB_ERR_INVALID_ARG, "island %d", island);
    const int K = c->size[island];
    GB_TRY(check_dtype(c, dtype));
    GB_TRY(check_n(c, n));
    GB_TRY(check_dev_bufs(c, rank_bufs, K, "rank_bufs"));
    GB_TRY(check_dev_ptr(c, island_sum, "island_sum"));
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    cudaStream_t s = (cudaStream_t)stream;
    gb::ReduceEncodeArgs ra;
    memset(&ra, 0, sizeof ra);
    for (int q = 0; q < K; ++q) ra.src[q] = rank_bufs[q];
    ra.payload[0] = island_sum;
    ra.first[0] = 0;
    ra.first[1] = K;
    ra.n_islands = 1;
    ra.n = n;
    ra.tiles = (n + gb::kTile - 1) / gb::kTile;
    ra.scales_off = 0;
    return check_launch(c, gb::launch_reduce_encode(ra, dtype, GB_CODEC_NONE, 256, s), "island reduce");
}

gb_status gb_bridge_compress(gb_ctx *c, const float *island_sum, size_t n, gb_codec codec, int block,
                             void *payload, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_codec(c, codec, block));
    GB_TRY(check_n(c, n));
    GB_TRY(check_dev_ptr(c, island_sum, "island_sum"));
    GB_TRY(check_dev_ptr(c, payload, "payload"));
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    const int blk = (codec == GB_CODEC_E4M3 || codec == GB_CODEC_E5M2) ? block : 256;
    gb::ReduceEncodeArgs ra;
    memset(&ra, 0, sizeof ra);
    ra.src[0] = island_sum;
    ra.payload[0] = payload;
    ra.first[0] = 0;
    ra.first[1] = 1;
    ra.n_islands = 1;
    ra.n = n;
    ra.tiles = (n + gb::kTile - 1) / gb::kTile;
    ra.scales_off = scales_offset(codec, n);
    return check_launch(c, gb::launch_reduce_encode(ra, GB_F32, codec, blk, (cudaStream_t)stream),
                        "bridge compress");
}

gb_status gb_bridge_decompress_accumulate(gb_ctx *c, const void *payload, size_t n, gb_codec codec,
                                          int block, float *accum, int accumulate, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_codec(c, codec, block));
    GB_TRY(check_n(c, n));
    GB_TRY(check_dev_ptr(c, payload, "payload"));
    GB_TRY(check_dev_ptr(c, accum, "accum"));
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    const int blk = (codec == GB_CODEC_E4M3 || codec == GB_CODEC_E5M2) ? block : 256;
    gb::DecompressAccArgs a;
    a.payload = payload;
    a.accum = accum;
    a.n = n;
    a.scales_off = scales_offset(codec, n);
    a.accumulate = accumulate ? 1 : 0;
    return check_launch(c, gb::launch_decompress_accumulate(a, codec, blk, (cudaStream_t)stream),
                        "bridge decompress");
}

gb_status gb_island_broadcast(gb_ctx *c, int island, const float *total, size_t n, gb_op op,
                              void *const *rank_bufs, gb_dtype dtype, gb_stream stream) {
    GB_TRY(check_ctx(c));
    if (island < 0 || island >= c->I) return set_msg(c, GB_ERR_INVALID_ARG, "island %d", island);
    const int K = c->size[island];
    GB_TRY(check_dtype(c, dtype));
    GB_TRY(check_op(c, op));
    GB_TRY(check_n(c, n));
    GB_TRY(check_dev_ptr(c, total, "total"));
    GB_TRY(check_dev_bufs(c, (const void *const *)rank_bufs, K, "rank_bufs"));
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    gb::DecodeBcastArgs da;
    memset(&da, 0, sizeof da);
    for (int q = 0; q < K; ++q) da.dst[q] = rank_bufs[q];
    da.payload[0][0] = total;
    da.first[0] = 0;
    da.first[1] = K;
    da.n_groups = 1;
    da.n_src = 1;
    da.avg = op == GB_AVG;
    da.world = (float)c->W;
    da.n = n;
    da.scales_off = 0;
    da.rs = 0;
    da.vec = 1;
    da.tiles = (n + gb::kTile - 1) / gb::kTile;
    return check_launch(c, gb::launch_decode_bcast(da, dtype, GB_CODEC_NONE, 256, (cudaStream_t)stream),
                        "island broadcast");
}

gb_status gb_all_reduce(gb_ctx *c, void *const *rank_bufs, size_t n, gb_dtype dtype, gb_op op,
                        gb_codec codec, int block, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_collective(c, n, dtype, op, codec, block));
    GB_TRY(check_dev_bufs(c, (const void *const *)rank_bufs, c->W, "rank_bufs"));
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    return run_rbb(c, (const void *const *)rank_bufs, rank_bufs, n, dtype, op, codec, block,
                   (cudaStream_t)stream, 0);
}

gb_status gb_reduce_scatter(gb_ctx *c, const void *const *in, void *const *out, size_t n_in,
                            gb_dtype dtype, gb_op op, gb_codec codec, int block, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_collective(c, n_in, dtype, op, codec, block));
    GB_TRY(check_dev_bufs(c, in, c->W, "in"));
    GB_TRY(check_dev_bufs(c, (const void *const *)out, c->W, "out"));
    if (n_in % (size_t)c->W)
        return set_msg(c, GB_ERR_INVALID_ARG, "n_in = %zu is not a multiple of W = %d", n_in, c->W);
    if (n_in == 0) return GB_OK;
    GB_TRY(bind(c));
    return run_rbb(c, in, out, n_in, dtype, op, codec, block, (cudaStream_t)stream, 1);
}

gb_status gb_all_gather(gb_ctx *c, const void *const *in, void *const *out, size_t n_in,
                        gb_dtype dtype, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_dtype(c, dtype));
    GB_TRY(check_n(c, n_in));
    GB_TRY(check_dev_bufs(c, in, c->W, "in"));
    GB_TRY(check_dev_bufs(c, (const void *const *)out, c->W, "out"));
    if (n_in == 0) return GB_OK;
    GB_TRY(bind(c));
    cudaStream_t s = (cudaStream_t)stream;
    const int W = c->W, I = c->I;
    const size_t mb = n_in * elem_bytes(dtype);
    if (I > 1) GB_TRY(grow_host(c, (size_t)W * mb));
    GB_TRY(begin(c, s));
    GB_TRY(mark(c, 0, s));
    GB_TRY(mark(c, 1, s));
    if (I > 1) {
        if (c->inject == GB_INJECT_BRIDGE) {
            c->inject = 0;
            return fail(c, GB_ERR_BRIDGE, "bridge hop failed (injected)");
        }
        // every rank's block goes to the host slots ...
        for (int q = 0; q < W; ++q)
            GB_TRY(copy_async(c, c->h_stage + (size_t)q * mb, in[q], mb, cudaMemcpyDeviceToHost, s));
        // ... and each leader receives the other islands' blocks in place
        for (int i = 0; i < I; ++i) {
            unsigned char *lead = (unsigned char *)out[c->first[i]];
            const size_t lo = (size_t)c->first[i] * mb, hi = (size_t)c->first[i + 1] * mb;
            GB_TRY(copy_async(c, lead, c->h_stage, lo, cudaMemcpyHostToDevice, s));
            GB_TRY(copy_async(c, lead + hi, c->h_stage + hi, (size_t)W * mb - hi, cudaMemcpyHostToDevice, s));
        }
    }
    c->ev_bridge = I > 1;
    GB_TRY(mark(c, 2, s));
    // each island: own ranks' blocks from the inputs, the others from the
    // leader's received copy, into every rank of the island
    for (int i = 0; i < I; ++i) {
        gb::CopyArgs a;
        memset(&a, 0, sizeof a);
        const unsigned char *lead = (const unsigned char *)out[c->first[i]];
        a.n_jobs = W;
        a.bytes = mb;
        a.vec = (mb % 16) == 0;
        for (int q = 0; q < W; ++q) {
            const bool own = c->island_of[q] == i;
            a.src[q] = own ? (const unsigned char *)in[q] : lead + (size_t)q * mb;
            a.dst_off[q] = (size_t)q * mb;
            a.dst_lo[q] = 0;
            a.dst_hi[q] = c->size[i];
        }
        for (int k = 0; k < c->size[i]; ++k) a.dst[k] = (unsigned char *)out[c->first[i] + k];
        GB_TRY(check_launch(c, gb::launch_copy(a, s), "all_gather copy"));
    }
    GB_TRY(mark(c, 3, s));
    return end(c, s);
}

gb_status gb_broadcast(gb_ctx *c, void *const *rank_bufs, size_t n, gb_dtype dtype, int src,
                       gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_dtype(c, dtype));
    GB_TRY(check_n(c, n));
    GB_TRY(check_dev_bufs(c, (const void *const *)rank_bufs, c->W, "rank_bufs"));
    if (src < 0 || src >= c->W) return set_msg(c, GB_ERR_INVALID_ARG, "src %d", src);
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    cudaStream_t s = (cudaStream_t)stream;
    const int I = c->I;
    const int si = c->island_of[src];
    const size_t nb = n * elem_bytes(dtype);
    if (I > 1) GB_TRY(grow_host(c, nb));
    GB_TRY(begin(c, s));
    GB_TRY(mark(c, 0, s));
    GB_TRY(mark(c, 1, s));
    if (I > 1) {
        if (c->inject == GB_INJECT_BRIDGE) {
            c->inject = 0;
            return fail(c, GB_ERR_BRIDGE, "bridge hop failed (injected)");
        }
        // src's island leader sends over the bridge (the bytes are src's);
        // every other leader receives in place
        GB_TRY(copy_async(c, c->h_stage, rank_bufs[src], nb, cudaMemcpyDeviceToHost, s));
        for (int i = 0; i < I; ++i)
            if (i != si)
                GB_TRY(copy_async(c, rank_bufs[c->first[i]], c->h_stage, nb, cudaMemcpyHostToDevice, s));
    }
    c->ev_bridge = I > 1;
    GB_TRY(mark(c, 2, s));
    // each island: its source (src, or the leader that received) -> its ranks
    gb::CopyArgs a;
    memset(&a, 0, sizeof a);
    a.n_jobs = I;
    a.bytes = nb;
    a.vec = (nb % 16) == 0;
    for (int r = 0; r < c->W; ++r) a.dst[r] = (unsigned char *)rank_bufs[r];
    for (int i = 0; i < I; ++i) {
        a.src[i] = (const unsigned char *)rank_bufs[i == si ? src : c->first[i]];
        a.dst_off[i] = 0;
        a.dst_lo[i] = c->first[i];
        a.dst_hi[i] = c->first[i + 1];
    }
    GB_TRY(check_launch(c, gb::launch_copy(a, s), "broadcast copy"));
    GB_TRY(mark(c, 3, s));
    return end(c, s);
}

gb_status gb_all_reduce_host(gb_ctx *c, void *const *host_bufs, size_t n, gb_dtype dtype, gb_op op,
                             gb_codec codec, int block, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_collective(c, n, dtype, op, codec, block));
    if (!host_bufs) return set_msg(c, GB_ERR_INVALID_ARG, "host_bufs is NULL");
    for (int r = 0; r < c->W; ++r)
        if (!host_bufs[r]) return set_msg(c, GB_ERR_INVALID_ARG, "host_bufs[%d] is NULL", r);
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    cudaStream_t s = (cudaStream_t)stream;
    const size_t nb = n * elem_bytes(dtype);
    const size_t stride = round_up(nb, 256);
    GB_TRY(grow_device(c, &c->d_ranks, &c->d_ranks_bytes, (size_t)c->W * stride));
    GB_TRY(begin(c, s));
    void *dev[GB_MAX_RANKS];
    for (int r = 0; r < c->W; ++r) {
        dev[r] = c->d_ranks + (size_t)r * stride;
        cudaError_t e = cudaMemcpyAsync(dev[r], host_bufs[r], nb, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "host -> device staging", e);
    }
    GB_TRY(run_rbb(c, (const void *const *)dev, dev, n, dtype, op, codec, block, s, 0));
    for (int r = 0; r < c->W; ++r) {
        cudaError_t e = cudaMemcpyAsync(host_bufs[r], dev[r], nb, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "device -> host copy back", e);
    }
    return end(c, s);
}

gb_status gb_bucket_plan(const size_t *numel, int n_tensors, size_t elem_bytes_, size_t cap_bytes,
                         size_t pad_elems, int *bucket_of, size_t *offset, size_t *bucket_numel,
                         int max_buckets, int *n_buckets) {
    if (n_tensors < 0 || !n_buckets || elem_bytes_ == 0 || max_buckets < 0) return GB_ERR_INVALID_ARG;
    if (n_tensors > 0 && (!numel || !bucket_of || !offset || !bucket_numel)) return GB_ERR_INVALID_ARG;
    int nb = 0;
    size_t cur = 0;
    for (int t = 0; t < n_tensors; ++t) {
        const bool open_new = nb == 0 || (cur > 0 && (cur + numel[t]) * elem_bytes_ > cap_bytes);
        if (open_new) {
            if (nb > 0) bucket_numel[nb - 1] = cur;
            if (nb == max_buckets) return GB_ERR_INVALID_ARG;
            ++nb;
            cur = 0;
        }
        bucket_of[t] = nb - 1;
        offset[t] = cur;
        cur += numel[t];
    }
    if (nb > 0) bucket_numel[nb - 1] = cur;
    if (pad_elems > 1)
        for (int b = 0; b < nb; ++b) bucket_numel[b] = round_up(bucket_numel[b], pad_elems);
    *n_buckets = nb;
    return GB_OK;
}

gb_status gb_all_reduce_buckets(gb_ctx *c, int n_buckets, void *const *bucket_bufs,
                                const size_t *bucket_numel, gb_dtype dtype, gb_op op, gb_codec codec,
                                int block, gb_stream stream) {
    GB_TRY(check_ctx(c));
    if (n_buckets < 0 || (n_buckets > 0 && (!bucket_bufs || !bucket_numel)))
        return set_msg(c, GB_ERR_INVALID_ARG, "bucket arrays");
    GB_TRY(check_collective(c, 0, dtype, op, codec, block));
    for (int b = 0; b < n_buckets; ++b) {
        GB_TRY(check_n(c, bucket_numel[b]));
        GB_TRY(check_dev_bufs(c, (const void *const *)(bucket_bufs + (size_t)b * c->W), c->W, "bucket_bufs"));
    }
    for (int b = 0; b < n_buckets; ++b)
        GB_TRY(gb_all_reduce(c, bucket_bufs + (size_t)b * c->W, bucket_numel[b], dtype, op, codec, block,
                             stream));
    return GB_OK;
}

gb_status gb_set_phase_timing(gb_ctx *c, int capacity) {
    if (!c || capacity < 0 || capacity > (1 << 20)) return GB_ERR_INVALID_ARG;
    if (c->tev && c->done_recorded) cudaEventSynchronize(c->done);
    free_marks(c);
    if (capacity > 0) {
        c->tev = new (std::nothrow) cudaEvent_t[(size_t)capacity * 4]();
        if (!c->tev) return set_msg(c, GB_ERR_ALLOC, "phase timing records");
        c->tcap = capacity;
    }
    return GB_OK;
}

gb_status gb_phase_times(gb_ctx *c, int age, float *ms) {
    if (!c || !ms) return GB_ERR_INVALID_ARG;
    for (int i = 0; i < GB_N_PHASES; ++i) ms[i] = 0.0f;
    if (age < 0 || age >= c->tcap || age >= c->tcount)
        return set_msg(c, GB_ERR_INVALID_ARG, "no timed collective %d calls back", age);
    const cudaEvent_t *ev = c->tev + (size_t)((c->tcount - 1 - age) % c->tcap) * 4;
    cudaError_t e = cudaEventSynchronize(ev[3]);
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaEventSynchronize", e);
    for (int i = 0; i < GB_N_PHASES; ++i) {
        e = cudaEventElapsedTime(&ms[i], ev[i], ev[i + 1]);
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaEventElapsedTime", e);
    }
    return GB_OK;
}

gb_status gb_last_phase_times(gb_ctx *c, float *ms) { return gb_phase_times(c, 0, ms); }

gb_status gb_debug_inject(gb_ctx *c, int what) {
    if (!c || (what != 0 && what != GB_INJECT_BRIDGE && what != GB_INJECT_ALLOC)) return GB_ERR_INVALID_ARG;
    c->inject = what;
    return GB_OK;
}

uint64_t gb_kernel_launch_count(void) { return gb::launches(); }

}  // extern "C"
