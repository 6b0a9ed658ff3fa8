// Host runtime of libgb: argument validation, context binding, staging
// buffers, timing marks, and the pipelines that compose the kernels with the
// bridge hop through pinned host memory.  The C entry points are in
// gb_api.cu; the contracts in include/gb.h.
#include <cmath>

#include "gb_internal.cuh"

namespace gbrt {


gb_status set_msg(gb_ctx *c, gb_status s, const char *fmt, ...) {
    if (c) {
        if (s != GB_OK) c->last = s;
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(c->msg, sizeof c->msg, fmt, ap);
        va_end(ap);
    }
    return s;
}

// A failure after validation: the context becomes failed for good.
gb_status fail(gb_ctx *c, gb_status s, const char *what, cudaError_t e) {
    c->sticky = s;
    c->last = s;
    if (e != cudaSuccess)
        snprintf(c->msg, sizeof c->msg, "%s: %s", what, cudaGetErrorString(e));
    else
        snprintf(c->msg, sizeof c->msg, "%s", what);
    return s;
}

size_t elem_bytes(gb_dtype d) {
    switch (d) {
    case GB_F32: case GB_I32: return 4;
    case GB_BF16: case GB_F16: return 2;
    case GB_F64: case GB_I64: return 8;
    default: return 1;
    }
}

bool is_float_dtype(int d) { return d == GB_F32 || d == GB_BF16 || d == GB_F16 || d == GB_F64; }

// MAX / MIN, and every dtype but float32 / bfloat16, take the exact path.
bool is_exact(int dtype, int op) { return op == GB_MAX || op == GB_MIN || (dtype != GB_F32 && dtype != GB_BF16); }

// Payloads, island sums, accumulators and residuals: the kernels move their
// float32 data with 32-byte vector accesses.
bool aligned32(const void *p) { return ((uintptr_t)p & 31u) == 0; }

gb_status check_ctx(gb_ctx *c) {
    if (!c) return GB_ERR_INVALID_ARG;
    if (c->sticky != GB_OK) return c->last = GB_ERR_CONTEXT_FAILED;  // the message keeps the cause
    return GB_OK;
}

gb_status check_dtype(gb_ctx *c, int d) {
    if (d < GB_F32 || d > GB_I64) return set_msg(c, GB_ERR_UNSUPPORTED_DTYPE, "dtype %d", d);
    return GB_OK;
}

// The codec path's phase-level calls take float32 / bfloat16 only.
gb_status check_codec_dtype(gb_ctx *c, int d) {
    if (d != GB_F32 && d != GB_BF16) return set_msg(c, GB_ERR_UNSUPPORTED_DTYPE, "dtype %d on the codec path", d);
    return GB_OK;
}

gb_status check_op(gb_ctx *c, int op) {
    if (op < GB_SUM || op > GB_MIN) return set_msg(c, GB_ERR_UNSUPPORTED_OP, "op %d", op);
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
        if (!aligned32(bufs[r])) return set_msg(c, GB_ERR_MISALIGNED, "%s[%d] not 32-byte aligned", name, r);
    }
    return GB_OK;
}

// Rank buffers (the collectives' inputs and outputs): 16-byte aligned.  The
// kernels move float32 rank data with 32-byte accesses when every rank
// buffer of a launch is 32-byte aligned, else with two 16-byte accesses.
gb_status check_rank_bufs(gb_ctx *c, const void *const *bufs, int count, const char *name) {
    if (!bufs) return set_msg(c, GB_ERR_INVALID_ARG, "%s is NULL", name);
    for (int r = 0; r < count; ++r) {
        if (!bufs[r]) return set_msg(c, GB_ERR_INVALID_ARG, "%s[%d] is NULL", name, r);
        if (((uintptr_t)bufs[r] & 15u) != 0)
            return set_msg(c, GB_ERR_MISALIGNED, "%s[%d] not 16-byte aligned", name, r);
    }
    return GB_OK;
}

gb_status check_dev_ptr(gb_ctx *c, const void *p, const char *name) {
    if (!p) return set_msg(c, GB_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned32(p)) return set_msg(c, GB_ERR_MISALIGNED, "%s not 32-byte aligned", name);
    return GB_OK;
}


// The current device `dev` as this call sees it: GB_INJECT_OTHER_DEVICE
// makes one call of a bound context see another device (a test of the
// mismatch refusal that needs no second GPU); unbound, the injection is
// dropped.
int seen_device(gb_ctx *c, int dev) {
    if (c->inject != GB_INJECT_OTHER_DEVICE) return dev;
    c->inject = 0;
    return c->device >= 0 ? c->device + 1 : dev;
}

// Bind the context to the current device on first use (creates its streams
// and events there).
gb_status bind(gb_ctx *c) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_msg(c, GB_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    }
    dev = seen_device(c, dev);
    if (c->device < 0) {
        if ((e = cudaEventCreateWithFlags(&c->done, cudaEventDisableTiming)) != cudaSuccess)
            return fail(c, GB_ERR_CUDA, "cudaEventCreate", e);
        cudaStream_t *streams[4] = {&c->sd, &c->sh, &c->scap, &c->sg};
        for (cudaStream_t *st : streams)
            if ((e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking)) != cudaSuccess)
                return fail(c, GB_ERR_CUDA, "cudaStreamCreate", e);
        for (int i = 0; i < kMaxChunks; ++i) {
            cudaEvent_t *evs[5] = {&c->ev_k1[i], &c->ev_d2h[i], &c->ev_h2d[i], &c->ev_in[i], &c->ev_k2[i]};
            for (cudaEvent_t *ev : evs)
                if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess)
                    return fail(c, GB_ERR_CUDA, "cudaEventCreate", e);
        }
        if ((e = cudaEventCreateWithFlags(&c->ev_join_d, cudaEventDisableTiming)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&c->ev_join_h, cudaEventDisableTiming)) != cudaSuccess)
            return fail(c, GB_ERR_CUDA, "cudaEventCreate", e);
        for (int i = 0; i < GB_MAX_RANKS; ++i)
            if ((e = cudaEventCreateWithFlags(&c->ev_ag[i], cudaEventDisableTiming)) != cudaSuccess)
                return fail(c, GB_ERR_CUDA, "cudaEventCreate", e);
        for (int i = 0; i < kMarks; ++i)
            if ((e = cudaEventCreate(&c->cap_mark[i])) != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaEventCreate", e);
        int mp = 0;
        if (cudaDeviceGetAttribute(&mp, cudaDevAttrMaxPitch, dev) == cudaSuccess && mp > 0) c->max_pitch = (size_t)mp;
        cudaGetLastError();
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


gb_status ring_event(gb_ctx *c, long long slot, int idx, cudaEvent_t *out) {
    cudaEvent_t &ev = c->tev[(size_t)slot * kMarks + idx];
    if (!ev) {
        cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaEventCreate", e);
    }
    *out = ev;
    return GB_OK;
}

gb_status mark(gb_ctx *c, int mode, int idx, cudaStream_t s) {
    if (mode == kMarkOff) return GB_OK;
    cudaEvent_t ev;
    unsigned flags = cudaEventRecordDefault;
    if (mode == kMarkCapture) {
        ev = c->cap_mark[idx];
        flags = cudaEventRecordExternal;
    } else {
        GB_TRY(ring_event(c, c->tcount % c->tcap, idx, &ev));
    }
    cudaError_t e = cudaEventRecordWithFlags(ev, s, flags);
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaEventRecord", e);
    return GB_OK;
}

// The marks of one collective are complete: remember its shape, advance.
void commit_marks(gb_ctx *c, int n_decode, bool bridge) {
    if (c->tcap <= 0) return;
    const long long slot = c->tcount % c->tcap;
    c->tnk2[slot] = n_decode;
    c->tbridge[slot] = bridge ? 1 : 0;
    ++c->tcount;
}

void free_marks(gb_ctx *c) {
    if (c->tev) {
        for (size_t i = 0; i < (size_t)c->tcap * kMarks; ++i)
            if (c->tev[i]) cudaEventDestroy(c->tev[i]);
        delete[] c->tev;
    }
    delete[] c->tnk2;
    delete[] c->tbridge;
    c->tev = nullptr;
    c->tnk2 = nullptr;
    c->tbridge = nullptr;
    c->tcap = 0;
    c->tcount = 0;
}

void drop_graphs(gb_ctx *c) {
    for (int i = 0; i < c->n_graphs; ++i) {
        if (c->graphs[i].exec) cudaGraphExecDestroy(c->graphs[i].exec);
        if (c->graphs[i].graph) cudaGraphDestroy(c->graphs[i].graph);
        c->graphs[i] = GraphEntry();
    }
    c->n_graphs = 0;
    for (auto &bg : c->bucket_graphs) {
        if (bg.exec) cudaGraphExecDestroy(bg.exec);
        if (bg.graph) cudaGraphDestroy(bg.graph);
    }
    c->bucket_graphs.clear();
}

gb_status grow_device(gb_ctx *c, unsigned char **buf, size_t *have, size_t need) {
    if (need <= *have) return GB_OK;
    if (c->inject == GB_INJECT_ALLOC) {
        c->inject = 0;
        return fail(c, GB_ERR_ALLOC, "device staging allocation failed (injected)");
    }
    if (*buf) {
        if (buf == &c->d_stage) drop_graphs(c);
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
        drop_graphs(c);
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


bool is_fp8(int codec) { return codec == GB_CODEC_E4M3 || codec == GB_CODEC_E5M2; }

size_t part_bytes(const Plan &p, uint64_t m) {
    size_t b = round_up(m * p.cb, 16);
    if (is_fp8(p.eff)) b += 4 * ((m + p.blk - 1) / p.blk);
    return b;
}

// The stride of a chunk's I parts inside its I-part staging region (I x
// p.part bytes): the chunk's own part rounded to 256 bytes, so that the one
// copy that moves several parts carries no padding when the chunk is shorter
// than the plan's longest (a bucket set's smaller buckets, a short last
// chunk).  Copying the full part stride had moved up to 15 % more bytes over
// the host link on the 1.1B bucket set.
size_t chunk_stride(const Plan &p, uint64_t m) { return round_up(part_bytes(p, m), 256); }

Plan make_plan(const gb_ctx *c, uint64_t n, gb_dtype dtype, gb_op op, gb_codec codec, int block, int rs,
               bool sharded_ok, size_t chunk_bytes, bool balance, uint64_t chunk_elems) {
    // chunk_bytes == 0: the single-buffer all_reduce's or reduce_scatter's
    // chunk, derived from the pipeline chunk and grown with the payload
    const bool grow = chunk_bytes == 0;
    if (chunk_bytes == 0) chunk_bytes = c->chunk_bytes;
    Plan p;
    p.I = c->I;
    p.W = c->W;
    p.n = n;
    p.dtype = dtype;
    p.op = op;
    p.rs = rs;
    p.eff = (c->I == 1 || is_exact(dtype, op)) ? GB_CODEC_NONE : (int)codec;
    p.blk = is_fp8(p.eff) ? block : 256;
    p.eb = elem_bytes(dtype);
    // payload bytes per element: the codec's, or the exact path's (the dtype,
    // or float32 sums of 16-bit floats)
    p.cb = is_exact(dtype, op) ? gb::exact_payload_elem_bytes(dtype, op)
                               : p.eff == GB_CODEC_NONE ? 4 : p.eff == GB_CODEC_BF16 ? 2 : 1;
    p.chunk = n;
    int k = c->I > 1 ? c->size[0] : 1;  // sharded-bridge: k = the smallest island's size
    for (int i = 1; i < c->I; ++i)
        if (c->size[i] < k) k = c->size[i];
    if (sharded_ok && !rs && c->sharded && c->I > 1 && k > 1) {
        // k segments of ceil(n / k) elements rounded up to whole tiles (so
        // whole codec blocks), one per bridge link
        const uint64_t seg = round_up((n + (uint64_t)k - 1) / (uint64_t)k, gb::kTile);
        if (seg < n) p.chunk = seg;
    } else if (c->I > 1 && chunk_bytes > 0) {
        // chunk_bytes of one island's payload per chunk
        const double per_elem = (double)p.cb + (is_fp8(p.eff) ? 4.0 / p.blk : 0.0);
        // The pipeline's fill and drain (the first chunk's device -> host copy
        // and the last one's host -> device copy, each alone on the link)
        // grow with the chunk; the copies' fixed costs grow with the chunk
        // count.  Their sum is least at a count proportional to sqrt(P), so
        // above kChunkGrowRef chunks' worth of one island's payload P the
        // all_reduce chunk grows as sqrt(P / (kChunkGrowRef * chunk_bytes)).
        // On GB300 this matched the best fixed chunk of 2 .. 16 MiB measured
        // at 16 .. 256 MiB per rank for every codec (64 MiB uncompressed:
        // 947 us against 1099 us with 2 MiB chunks).  reduce_scatter's
        // decodes write only the slices, so its drain is shorter: it takes
        // that chunk less half the pipeline chunk, at least half of it (the
        // half chunk up to 3 chunks of payload; on the 25 MiB float32 E4M3
        // bucket 147 us against 152 us with whole chunks; at 256 MiB E4M3 991
        // us against 1107 us with half chunks).
        double cbytes = (double)chunk_bytes;
        const double P = per_elem * (double)n;
        if (grow) {
            const double s_ar = P > kChunkGrowRef * cbytes ? cbytes * sqrt(P / (kChunkGrowRef * cbytes)) : cbytes;
            const double half = cbytes / (double)kRsChunkDiv;
            cbytes = !rs ? s_ar : s_ar - half > half ? s_ar - half : half;
        }
        uint64_t ch = (chunk_elems ? chunk_elems : (uint64_t)(cbytes / per_elem)) / gb::kTile * gb::kTile;
        if (ch < (uint64_t)gb::kTile) ch = gb::kTile;
        const uint64_t min_ch = round_up((n + kMaxChunks - 1) / kMaxChunks, gb::kTile);
        if (ch < min_ch) ch = min_ch;
        if (balance && ch < n) {
            // as many chunks as chunk_bytes needs, of equal size (whole tiles):
            // no short remainder chunk whose copies would cost their fixed
            // overhead for a sliver of data
            const uint64_t cnt = (n + ch - 1) / ch;
            ch = round_up((n + cnt - 1) / cnt, gb::kTile);
        }
        if (ch < n) p.chunk = ch;
    }
    p.C = (int)((n + p.chunk - 1) / p.chunk);
    for (int ch = 0; ch <= p.C; ++ch) p.off[ch] = (uint64_t)ch * p.chunk < n ? (uint64_t)ch * p.chunk : n;
    if (sharded_ok && !rs && c->sharded && c->I > 1 && k > 1) p.links = p.C < kMaxLinks ? p.C : kMaxLinks;
    p.part = round_up(part_bytes(p, p.chunk), 256);
    // received parts: two islands share one mirror of the host slots (leader
    // 1 holds island 0's part, leader 0 island 1's); more islands keep one
    // I-part region per leader
    const int recv = p.I == 1 ? 0 : p.I == 2 ? 2 : p.I * p.I;
    p.dev_bytes = (size_t)(p.I + recv) * p.C * p.part;
    p.host_bytes = p.I > 1 ? (size_t)p.I * p.C * p.part : 0;
    return p;
}

gb_status check_launch(gb_ctx *c, cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, what, e);
    return GB_OK;
}

// The two kernels of a plan: the codec path's, or the exact path's (MAX /
// MIN, exact dtypes).
gb_status launch_encode(gb_ctx *c, const Plan &p, const gb::ReduceEncodeArgs &ra, cudaStream_t s) {
    if (is_exact(p.dtype, p.op)) return check_launch(c, gb::launch_exact_reduce(ra, p.dtype, p.op, s), "island fold");
    return check_launch(c, gb::launch_reduce_encode(ra, p.dtype, p.eff, p.blk, s), "island reduce + encode");
}

gb_status launch_decode(gb_ctx *c, const Plan &p, const gb::DecodeBcastArgs &da, cudaStream_t s) {
    if (is_exact(p.dtype, p.op))
        return check_launch(c, gb::launch_exact_combine(da, p.dtype, p.op, s), "fold + broadcast");
    return check_launch(c, gb::launch_decode_bcast(da, p.dtype, p.eff, p.blk, s), "decode + broadcast");
}

// Vector accesses move 8 elements per lane (codec kernels) or 16 bytes per
// thread (exact kernels); a reduce_scatter slice length must be a multiple.
uint64_t vec_elems(const Plan &p) { return is_exact(p.dtype, p.op) ? 16 / p.eb : 8; }

gb_status copy_async(gb_ctx *c, void *dst, const void *src, size_t bytes, cudaMemcpyKind kind,
                     cudaStream_t s) {
    if (bytes == 0) return GB_OK;
    cudaError_t e = cudaMemcpyAsync(dst, src, bytes, kind, s);
    if (e != cudaSuccess) return fail(c, GB_ERR_BRIDGE, "bridge copy", e);
    return GB_OK;
}

gb_status wait_on(gb_ctx *c, cudaStream_t s, cudaEvent_t ev) {
    cudaError_t e = cudaStreamWaitEvent(s, ev, 0);
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaStreamWaitEvent", e);
    return GB_OK;
}

gb_status record(gb_ctx *c, cudaEvent_t ev, cudaStream_t s) {
    cudaError_t e = cudaEventRecord(ev, s);
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaEventRecord", e);
    return GB_OK;
}

// Enqueue one reduce-bridge-broadcast.  Kernels run on s.  With multi (and
// more than one island) the bridge copies run on the context's copy streams
// so that, chunk by chunk, encode, device -> host, host -> device and
// decode overlap: chunk c's copies wait for its encode, and its decode waits
// for its copies.  Staging (see Plan): own parts outbox(c, i), host slots
// host(c, j), leader g's received parts inbox(g, c, j).
gb_status enqueue_rbb(gb_ctx *c, const Plan &p, const void *const *in, void *const *out,
                      float *const *res, cudaStream_t s, int markmode, bool multi) {
    const int I = p.I;
    auto stride = [&](int ch) {
        uint64_t e0, m;
        chunk_range(p, ch, &e0, &m);
        return chunk_stride(p, m);
    };
    auto outbox = [&](int ch, int i) { return c->d_stage + (size_t)ch * I * p.part + (size_t)i * stride(ch); };
    // leader g's received copy of island j's part of chunk ch (j != g)
    auto inbox = [&](int g, int ch, int j) {
        unsigned char *base = c->d_stage + (size_t)I * p.C * p.part;
        if (I == 2) return base + (size_t)ch * I * p.part + (size_t)j * stride(ch);  // mirror of the host slots
        return base + ((size_t)g * p.C + ch) * I * p.part + (size_t)j * stride(ch);
    };
    auto host = [&](int ch, int j) { return c->h_stage + (size_t)ch * I * p.part + (size_t)j * stride(ch); };
    multi = multi && I > 1 && p.C > 1;

    // 1. island reduce + encode, chunk by chunk
    GB_TRY(mark(c, markmode, 0, s));
    for (int ch = 0; ch < p.C; ++ch) {
        uint64_t e0, m;
        chunk_range(p, ch, &e0, &m);
        gb::ReduceEncodeArgs ra;
        memset(&ra, 0, sizeof ra);
        for (int r = 0; r < p.W; ++r) ra.src[r] = (const unsigned char *)in[r] + e0 * p.eb;
        for (int i = 0; i < I; ++i) ra.payload[i] = outbox(ch, i);
        for (int i = 0; res && I > 1 && i < I; ++i) ra.residual[i] = res[i] + e0;  // no bridge: no feedback
        for (int i = 0; i <= I; ++i) ra.first[i] = c->first[i];
        ra.n_islands = I;
        ra.n = m;
        ra.tiles = (uint32_t)((m + gb::kTile - 1) / gb::kTile);
        ra.scales_off = is_fp8(p.eff) ? round_up(m * p.cb, 16) : 0;
        GB_TRY(launch_encode(c, p, ra, s));
        if (multi) GB_TRY(record(c, c->ev_k1[ch], s));
    }
    GB_TRY(mark(c, markmode, 1, s));

    // 2. the bridge hop: own parts to the host slots, others' parts to every leader
    if (I > 1) {
        if (c->inject == GB_INJECT_BRIDGE) {
            c->inject = 0;
            return fail(c, GB_ERR_BRIDGE, "bridge hop failed (injected)");
        }
        // chunk ch's copies run on link ch % links (sharded-bridge: one
        // segment per link; otherwise one link for every chunk)
        auto link_d = [&](int ch) { const int l = ch % p.links; return l ? c->lsd[l] : c->sd; };
        auto link_h = [&](int ch) { const int l = ch % p.links; return l ? c->lsh[l] : c->sh; };
        cudaStream_t D = s, H = s;
        for (int ch = 0; ch < p.C; ++ch) {
            uint64_t e0, m;
            chunk_range(p, ch, &e0, &m);
            const size_t pb = part_bytes(p, m), st = chunk_stride(p, m);
            if (multi) {
                D = link_d(ch);
                H = link_h(ch);
            }
            if (multi) GB_TRY(wait_on(c, D, c->ev_k1[ch]));
            if (ch == 0) GB_TRY(mark(c, markmode, 2, D));
            GB_TRY(copy_async(c, host(ch, 0), outbox(ch, 0), (size_t)(I - 1) * st + pb, cudaMemcpyDeviceToHost, D));
            if (multi) {
                GB_TRY(record(c, c->ev_d2h[ch], D));
                GB_TRY(wait_on(c, H, c->ev_d2h[ch]));
            }
            if (I == 2) {  // island 0's part to leader 1, island 1's part to leader 0: one copy
                GB_TRY(copy_async(c, inbox(1, ch, 0), host(ch, 0), st + pb, cudaMemcpyHostToDevice, H));
            } else {
                for (int g = 0; g < I; ++g) {
                    if (g > 0)
                        GB_TRY(copy_async(c, inbox(g, ch, 0), host(ch, 0), (size_t)(g - 1) * st + pb,
                                          cudaMemcpyHostToDevice, H));
                    if (g < I - 1)
                        GB_TRY(copy_async(c, inbox(g, ch, g + 1), host(ch, g + 1),
                                          (size_t)(I - g - 2) * st + pb, cudaMemcpyHostToDevice, H));
                }
            }
            if (multi) GB_TRY(record(c, c->ev_h2d[ch], H));
        }
        if (multi && p.links > 1 && markmode != kMarkOff) {
            // the bridge ends when every link's last copy has landed
            H = link_h(0);
            for (int l = 1; l < p.links && l < p.C; ++l) {
                const int last = l + (p.C - 1 - l) / p.links * p.links;
                GB_TRY(wait_on(c, H, c->ev_h2d[last]));
            }
        }
        GB_TRY(mark(c, markmode, 3, H));
    }

    // 3. decode + accumulate + broadcast, chunk by chunk
    for (int ch = 0; ch < p.C; ++ch) {
        uint64_t e0, m;
        chunk_range(p, ch, &e0, &m);
        if (multi) GB_TRY(wait_on(c, s, c->ev_h2d[ch]));
        GB_TRY(mark(c, markmode, 4 + 2 * ch, s));
        gb::DecodeBcastArgs da;
        memset(&da, 0, sizeof da);
        for (int r = 0; r < p.W; ++r) {
            da.dst[r] = (unsigned char *)out[r] + (p.rs ? 0 : e0 * p.eb);
            da.group_of_rank[r] = c->island_of[r];
        }
        uint64_t rs_max = 0;
        if (p.rs) {  // the parts of the slices that fall inside this chunk
            const uint64_t ms = p.n / (uint64_t)p.W;
            for (int r = 0; r < p.W; ++r) {
                const uint64_t s0 = (uint64_t)r * ms;
                const uint64_t lo = e0 > s0 ? e0 : s0;
                const uint64_t hi = (e0 + m) < (s0 + ms) ? (e0 + m) : (s0 + ms);
                if (hi > lo) {
                    da.rs_src[r] = lo - e0;
                    da.rs_len[r] = hi - lo;
                    da.dst[r] = (unsigned char *)out[r] + (lo - s0) * p.eb;
                    if (hi - lo > rs_max) rs_max = hi - lo;
                }
            }
        }
        const void *received[GB_MAX_ISLANDS];
        for (int j = 0; j < I; ++j)
            received[j] = I == 1 ? (const void *)outbox(ch, 0) : (const void *)inbox((j + 1) % I, ch, j);
        gb::decode_once(da, p.W, I, received);
        da.avg = p.op == GB_AVG;
        da.world = (float)p.W;
        da.world_pow2 = (p.W & (p.W - 1)) == 0;
        da.inv_world = 1.0f / (float)p.W;
        da.n = m;
        da.scales_off = is_fp8(p.eff) ? round_up(m * p.cb, 16) : 0;
        if (p.rs) {
            da.rs = 1;
            da.vec = ((p.n / (uint64_t)p.W) % vec_elems(p)) == 0;
            da.tiles = (uint32_t)((rs_max + gb::kTile - 1) / gb::kTile);
        } else {
            da.rs = 0;
            da.vec = 1;
            da.tiles = (uint32_t)((m + gb::kTile - 1) / gb::kTile);
        }
        if (da.tiles > 0) GB_TRY(launch_decode(c, p, da, s));
        GB_TRY(mark(c, markmode, 5 + 2 * ch, s));
    }
    if (multi) {  // the copy streams' last work precedes the end of the call
        GB_TRY(record(c, c->ev_join_d, c->sd));
        GB_TRY(record(c, c->ev_join_h, c->sh));
        GB_TRY(wait_on(c, s, c->ev_join_d));
        GB_TRY(wait_on(c, s, c->ev_join_h));
        for (int l = 1; l < p.links; ++l) {
            GB_TRY(record(c, c->ev_ljd[l], c->lsd[l]));
            GB_TRY(record(c, c->ev_ljh[l], c->lsh[l]));
            GB_TRY(wait_on(c, s, c->ev_ljd[l]));
            GB_TRY(wait_on(c, s, c->ev_ljh[l]));
        }
    }
    return GB_OK;
}

// Copy stream pairs 1 .. L - 1 of the sharded-bridge policy, created on
// first use (link 0 is the pipelined policy's pair).
gb_status ensure_links(gb_ctx *c, int L) {
    for (int l = 1; l < L && l < kMaxLinks; ++l) {
        // each handle on its own, so that a failure part way leaves nothing
        // half made for a later call to use
        cudaError_t e = cudaSuccess;
        if (!c->lsd[l]) e = cudaStreamCreateWithFlags(&c->lsd[l], cudaStreamNonBlocking);
        if (e == cudaSuccess && !c->lsh[l]) e = cudaStreamCreateWithFlags(&c->lsh[l], cudaStreamNonBlocking);
        if (e == cudaSuccess && !c->ev_ljd[l]) e = cudaEventCreateWithFlags(&c->ev_ljd[l], cudaEventDisableTiming);
        if (e == cudaSuccess && !c->ev_ljh[l]) e = cudaEventCreateWithFlags(&c->ev_ljh[l], cudaEventDisableTiming);
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "bridge link streams", e);
    }
    return GB_OK;
}

// Staging of the host rank buffers.  Every cudaMemcpyAsync pays a fixed
// cost of a few microseconds on its copy stream, and the host-buffer
// pipeline would issue W of them per chunk in each direction; when the
// buffers are the rows of one host allocation (hpitch > 0) a single 2D copy
// moves every rank's part.  (Equal spacing alone is not enough: separate
// pinned allocations can lie at equal distances, and the runtime refuses a
// 2D copy that spans several allocations.)
// Bytes [off, off + bytes) of every rank buffer between the host buffers and
// the context's rank copies, in the direction `kind`.
gb_status stage_ranks(gb_ctx *c, void *const *host, void *const *dev, size_t dpitch, size_t hpitch, size_t off,
                      size_t bytes, cudaMemcpyKind kind, cudaStream_t s) {
    if (bytes == 0) return GB_OK;
    const bool in = kind == cudaMemcpyHostToDevice;
    const char *what = in ? "host -> device staging" : "device -> host copy back";
    if (hpitch) {
        unsigned char *d0 = (unsigned char *)dev[0] + off, *h0 = (unsigned char *)host[0] + off;
        cudaError_t e = in ? cudaMemcpy2DAsync(d0, dpitch, h0, hpitch, bytes, (size_t)c->W, kind, s)
                           : cudaMemcpy2DAsync(h0, hpitch, d0, dpitch, bytes, (size_t)c->W, kind, s);
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, what, e);
        return GB_OK;
    }
    for (int r = 0; r < c->W; ++r) {
        unsigned char *d = (unsigned char *)dev[r] + off, *h = (unsigned char *)host[r] + off;
        cudaError_t e = in ? cudaMemcpyAsync(d, h, bytes, kind, s) : cudaMemcpyAsync(h, d, bytes, kind, s);
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, what, e);
    }
    return GB_OK;
}

// gb_all_reduce_host, pipelined: chunk c of every host rank buffer goes to
// the device (copy stream H), is encoded (s), its payload crosses the
// bridge (D, then H), is decoded into the device rank chunks (s) and copied
// back to the host buffers (D).  Issued one chunk ahead so that both copy
// directions stay busy: H carries in(0), in(1), bridge-in(0), in(2), ...; D
// carries bridge-out(0), bridge-out(1), out(0), bridge-out(2), out(1), ...
gb_status enqueue_host_pipeline(gb_ctx *c, const Plan &p, void *const *host, void *const *dev, size_t dpitch,
                                size_t hpitch, cudaStream_t s) {
    const int I = p.I, W = p.W;
    auto range = [&](int ch, uint64_t *e0, uint64_t *m) { chunk_range(p, ch, e0, m); };
    auto stride = [&](int ch) {
        uint64_t e0, m;
        range(ch, &e0, &m);
        return chunk_stride(p, m);
    };
    auto outbox = [&](int ch, int i) { return c->d_stage + (size_t)ch * I * p.part + (size_t)i * stride(ch); };
    auto inbox = [&](int g, int ch, int j) {
        unsigned char *base = c->d_stage + (size_t)I * p.C * p.part;
        if (I == 2) return base + (size_t)ch * I * p.part + (size_t)j * stride(ch);
        return base + ((size_t)g * p.C + ch) * I * p.part + (size_t)j * stride(ch);
    };
    auto hslot = [&](int ch, int j) { return c->h_stage + (size_t)ch * I * p.part + (size_t)j * stride(ch); };
    cudaStream_t D = c->sd, H = c->sh;
    if (c->inject == GB_INJECT_BRIDGE) {
        c->inject = 0;
        return fail(c, GB_ERR_BRIDGE, "bridge hop failed (injected)");
    }
    GB_TRY(record(c, c->ev_join_d, s));  // the copy streams start after the caller's prior work
    GB_TRY(wait_on(c, H, c->ev_join_d));
    GB_TRY(wait_on(c, D, c->ev_join_d));
    auto issue_front = [&](int ch) -> gb_status {  // in(ch), encode(ch), bridge-out(ch)
        uint64_t e0, m;
        range(ch, &e0, &m);
        GB_TRY(stage_ranks(c, host, dev, dpitch, hpitch, e0 * p.eb, m * p.eb, cudaMemcpyHostToDevice, H));
        GB_TRY(record(c, c->ev_in[ch], H));
        GB_TRY(wait_on(c, s, c->ev_in[ch]));
        gb::ReduceEncodeArgs ra;
        memset(&ra, 0, sizeof ra);
        for (int r = 0; r < W; ++r) ra.src[r] = (const unsigned char *)dev[r] + e0 * p.eb;
        for (int i = 0; i < I; ++i) ra.payload[i] = outbox(ch, i);
        for (int i = 0; i <= I; ++i) ra.first[i] = c->first[i];
        ra.n_islands = I;
        ra.n = m;
        ra.tiles = (uint32_t)((m + gb::kTile - 1) / gb::kTile);
        ra.scales_off = is_fp8(p.eff) ? round_up(m * p.cb, 16) : 0;
        GB_TRY(launch_encode(c, p, ra, s));
        GB_TRY(record(c, c->ev_k1[ch], s));
        if (I > 1) {
            GB_TRY(wait_on(c, D, c->ev_k1[ch]));
            GB_TRY(copy_async(c, hslot(ch, 0), outbox(ch, 0), (size_t)(I - 1) * stride(ch) + part_bytes(p, m),
                              cudaMemcpyDeviceToHost, D));
            GB_TRY(record(c, c->ev_d2h[ch], D));
        }
        return GB_OK;
    };
    auto issue_back = [&](int ch) -> gb_status {  // bridge-in(ch), decode(ch), out(ch)
        uint64_t e0, m;
        range(ch, &e0, &m);
        const size_t pb = part_bytes(p, m), st = chunk_stride(p, m);
        if (I > 1) {
            GB_TRY(wait_on(c, H, c->ev_d2h[ch]));
            if (I == 2) {
                GB_TRY(copy_async(c, inbox(1, ch, 0), hslot(ch, 0), st + pb, cudaMemcpyHostToDevice, H));
            } else {
                for (int g = 0; g < I; ++g) {
                    if (g > 0)
                        GB_TRY(copy_async(c, inbox(g, ch, 0), hslot(ch, 0), (size_t)(g - 1) * st + pb,
                                          cudaMemcpyHostToDevice, H));
                    if (g < I - 1)
                        GB_TRY(copy_async(c, inbox(g, ch, g + 1), hslot(ch, g + 1), (size_t)(I - g - 2) * st + pb,
                                          cudaMemcpyHostToDevice, H));
                }
            }
            GB_TRY(record(c, c->ev_h2d[ch], H));
            GB_TRY(wait_on(c, s, c->ev_h2d[ch]));
        }
        gb::DecodeBcastArgs da;
        memset(&da, 0, sizeof da);
        for (int r = 0; r < W; ++r) {
            da.dst[r] = (unsigned char *)dev[r] + e0 * p.eb;
            da.group_of_rank[r] = c->island_of[r];
        }
        const void *received[GB_MAX_ISLANDS];
        for (int j = 0; j < I; ++j)
            received[j] = I == 1 ? (const void *)outbox(ch, 0) : (const void *)inbox((j + 1) % I, ch, j);
        gb::decode_once(da, W, I, received);
        da.avg = p.op == GB_AVG;
        da.world = (float)W;
        da.world_pow2 = (W & (W - 1)) == 0;
        da.inv_world = 1.0f / (float)W;
        da.n = m;
        da.scales_off = is_fp8(p.eff) ? round_up(m * p.cb, 16) : 0;
        da.vec = 1;
        da.tiles = (uint32_t)((m + gb::kTile - 1) / gb::kTile);
        GB_TRY(launch_decode(c, p, da, s));
        GB_TRY(record(c, c->ev_k2[ch], s));
        GB_TRY(wait_on(c, D, c->ev_k2[ch]));
        GB_TRY(stage_ranks(c, host, dev, dpitch, hpitch, e0 * p.eb, m * p.eb, cudaMemcpyDeviceToHost, D));
        return GB_OK;
    };
    GB_TRY(issue_front(0));
    for (int ch = 0; ch < p.C; ++ch) {
        if (ch + 1 < p.C) GB_TRY(issue_front(ch + 1));
        GB_TRY(issue_back(ch));
    }
    GB_TRY(record(c, c->ev_join_d, D));
    GB_TRY(record(c, c->ev_join_h, H));
    GB_TRY(wait_on(c, s, c->ev_join_d));
    GB_TRY(wait_on(c, s, c->ev_join_h));
    return GB_OK;
}


// A bucket set as one pipeline over every bucket's chunks.  Chunk i's
// encode, bridge hop and decode use staging slot i % R (an R-slot ring), and
// chunks are issued R - 1 ahead (encode + device -> host of chunk i + R - 1
// before host -> device + decode of chunk i), so both copy streams always
// have their next copy queued and the bridge of one bucket overlaps the
// kernels of the next.  The ring is safe because on the kernel stream
// encode(i + R - 1) follows decode(i - 1), which waited for every copy of
// chunk i - 1, the slot's previous user.  Three slots took the 1.1B set from
// 19.2 to 15.8 ms against two; four gained nothing more.
// in / out: nb x W rank buffers, bucket-major.  rs == 0: all_reduce (out
// may equal in); rs == 1: reduce_scatter, out[b * W + r] receives slice r of
// bucket b (numel[b] / W elements).  res: error feedback, nb x I residuals.
gb_status enqueue_buckets(gb_ctx *c, const Plan &p, const std::vector<WorkChunk> &work, const void *const *in,
                          void *const *out, const size_t *numel, int rs, float *const *res, cudaStream_t s) {
    const int I = p.I, W = p.W;
    constexpr int R = kBucketSlots;
    // slot `slot` holds the parts of one chunk of m elements at its own stride
    auto outbox = [&](int slot, int i, uint64_t m) {
        return c->d_stage + (size_t)slot * I * p.part + (size_t)i * chunk_stride(p, m);
    };
    auto inbox = [&](int g, int slot, int j, uint64_t m) {
        unsigned char *base = c->d_stage + (size_t)I * R * p.part;
        if (I == 2) return base + (size_t)slot * I * p.part + (size_t)j * chunk_stride(p, m);
        return base + ((size_t)g * R + slot) * I * p.part + (size_t)j * chunk_stride(p, m);
    };
    auto hslot = [&](int slot, int j, uint64_t m) {
        return c->h_stage + (size_t)slot * I * p.part + (size_t)j * chunk_stride(p, m);
    };
    if (c->inject == GB_INJECT_BRIDGE) {
        c->inject = 0;
        return fail(c, GB_ERR_BRIDGE, "bridge hop failed (injected)");
    }
    cudaStream_t D = c->sd, H = c->sh;
    const int N = (int)work.size();
    auto front = [&](int i) -> gb_status {
        const WorkChunk &w = work[i];
        const int slot = i % R, ev = i % kMaxChunks;
        gb::ReduceEncodeArgs ra;
        memset(&ra, 0, sizeof ra);
        for (int r = 0; r < W; ++r) ra.src[r] = (const unsigned char *)in[(size_t)w.b * W + r] + w.e0 * p.eb;
        for (int q = 0; res && q < I; ++q) ra.residual[q] = res[(size_t)w.b * I + q] + w.e0;  // error feedback
        for (int q = 0; q < I; ++q) ra.payload[q] = outbox(slot, q, w.m);
        for (int q = 0; q <= I; ++q) ra.first[q] = c->first[q];
        ra.n_islands = I;
        ra.n = w.m;
        ra.tiles = (uint32_t)((w.m + gb::kTile - 1) / gb::kTile);
        ra.scales_off = is_fp8(p.eff) ? round_up(w.m * p.cb, 16) : 0;
        GB_TRY(launch_encode(c, p, ra, s));
        GB_TRY(record(c, c->ev_k1[ev], s));
        GB_TRY(wait_on(c, D, c->ev_k1[ev]));
        GB_TRY(copy_async(c, hslot(slot, 0, w.m), outbox(slot, 0, w.m),
                          (size_t)(I - 1) * chunk_stride(p, w.m) + part_bytes(p, w.m), cudaMemcpyDeviceToHost, D));
        GB_TRY(record(c, c->ev_d2h[ev], D));
        return GB_OK;
    };
    auto back = [&](int i) -> gb_status {
        const WorkChunk &w = work[i];
        const int slot = i % R, ev = i % kMaxChunks;
        const size_t pb = part_bytes(p, w.m), st = chunk_stride(p, w.m);
        GB_TRY(wait_on(c, H, c->ev_d2h[ev]));
        if (I == 2) {
            GB_TRY(copy_async(c, inbox(1, slot, 0, w.m), hslot(slot, 0, w.m), st + pb, cudaMemcpyHostToDevice, H));
        } else {
            for (int g = 0; g < I; ++g) {
                if (g > 0)
                    GB_TRY(copy_async(c, inbox(g, slot, 0, w.m), hslot(slot, 0, w.m), (size_t)(g - 1) * st + pb,
                                      cudaMemcpyHostToDevice, H));
                if (g < I - 1)
                    GB_TRY(copy_async(c, inbox(g, slot, g + 1, w.m), hslot(slot, g + 1, w.m),
                                      (size_t)(I - g - 2) * st + pb, cudaMemcpyHostToDevice, H));
            }
        }
        GB_TRY(record(c, c->ev_h2d[ev], H));
        GB_TRY(wait_on(c, s, c->ev_h2d[ev]));
        gb::DecodeBcastArgs da;
        memset(&da, 0, sizeof da);
        uint64_t rs_max = 0;
        for (int r = 0; r < W; ++r) da.dst[r] = (unsigned char *)out[(size_t)w.b * W + r] + w.e0 * p.eb;
        if (rs) {  // the parts of bucket b's slices that fall inside this chunk
            const uint64_t ms = numel[w.b] / (uint64_t)W;
            for (int r = 0; r < W; ++r) {
                const uint64_t s0 = (uint64_t)r * ms;
                const uint64_t lo = w.e0 > s0 ? w.e0 : s0;
                const uint64_t hi = (w.e0 + w.m) < (s0 + ms) ? (w.e0 + w.m) : (s0 + ms);
                da.dst[r] = out[(size_t)w.b * W + r];
                if (hi > lo) {
                    da.rs_src[r] = lo - w.e0;
                    da.rs_len[r] = hi - lo;
                    da.dst[r] = (unsigned char *)out[(size_t)w.b * W + r] + (lo - s0) * p.eb;
                    if (hi - lo > rs_max) rs_max = hi - lo;
                }
            }
        }
        const void *received[GB_MAX_ISLANDS];
        for (int j = 0; j < I; ++j)
            received[j] = I == 1 ? (const void *)outbox(slot, 0, w.m) : (const void *)inbox((j + 1) % I, slot, j, w.m);
        gb::decode_once(da, W, I, received);
        da.avg = p.op == GB_AVG;
        da.world = (float)W;
        da.world_pow2 = (W & (W - 1)) == 0;
        da.inv_world = 1.0f / (float)W;
        da.n = w.m;
        da.scales_off = is_fp8(p.eff) ? round_up(w.m * p.cb, 16) : 0;
        if (rs) {
            da.rs = 1;
            da.vec = ((numel[w.b] / (uint64_t)W) % vec_elems(p)) == 0;
            da.tiles = (uint32_t)((rs_max + gb::kTile - 1) / gb::kTile);
        } else {
            da.vec = 1;
            da.tiles = (uint32_t)((w.m + gb::kTile - 1) / gb::kTile);
        }
        if (da.tiles > 0)
            GB_TRY(launch_decode(c, p, da, s));
        return GB_OK;
    };
    // chunks are issued R - 1 ahead: chunk i + R - 1's encode and device ->
    // host copy are queued before chunk i's host -> device copy and decode,
    // so each copy stream always has the next copy waiting (its slot was
    // last used by chunk i - 1, whose decode is already queued before it)
    constexpr int ahead = R - 1;
    for (int k = 0; k < ahead && k < N; ++k) GB_TRY(front(k));
    for (int i = 0; i < N; ++i) {
        if (i + ahead < N) GB_TRY(front(i + ahead));
        GB_TRY(back(i));
    }
    GB_TRY(record(c, c->ev_join_d, D));
    GB_TRY(record(c, c->ev_join_h, H));
    GB_TRY(wait_on(c, s, c->ev_join_d));
    GB_TRY(wait_on(c, s, c->ev_join_h));
    return GB_OK;
}

// A whole gradient set as one CUDA graph: the first call with a key runs
// `enqueue` directly (loading modules, sizing grids) and remembers the key;
// the second captures it on the context's private stream; later calls
// replay it.  Up to 8 sets are cached (least recently used out).  `kernels`
// is the number of kernel launches one replay makes.
gb_status run_set_graph(gb_ctx *c, const std::vector<uint64_t> &key, int kernels,
                        const std::function<gb_status(cudaStream_t)> &enqueue, cudaStream_t s) {
    gb_ctx::BucketGraph *bg = nullptr;
    for (auto &g : c->bucket_graphs)
        if (g.key == key) bg = &g;
    if (!bg) {  // first time: run directly, remember the shape
        if (c->bucket_graphs.size() >= 8) {
            size_t lru = 0;
            for (size_t i = 1; i < c->bucket_graphs.size(); ++i)
                if (c->bucket_graphs[i].last_use < c->bucket_graphs[lru].last_use) lru = i;
            if (c->bucket_graphs[lru].exec) cudaGraphExecDestroy(c->bucket_graphs[lru].exec);
            if (c->bucket_graphs[lru].graph) cudaGraphDestroy(c->bucket_graphs[lru].graph);
            c->bucket_graphs.erase(c->bucket_graphs.begin() + lru);
        }
        c->bucket_graphs.emplace_back();
        c->bucket_graphs.back().key = key;
        c->bucket_graphs.back().last_use = ++c->clock;
        GB_TRY(enqueue(s));
        return end(c, s);
    }
    bg->last_use = ++c->clock;
    if (!bg->exec) {
        cudaError_t e = cudaStreamBeginCapture(c->scap, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaStreamBeginCapture", e);
        gb_status st = enqueue(c->scap);
        cudaGraph_t g = nullptr;
        e = cudaStreamEndCapture(c->scap, &g);
        if (st != GB_OK) {
            if (g) cudaGraphDestroy(g);
            return st;
        }
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaStreamEndCapture", e);
        cudaGraphExec_t x = nullptr;
        if ((e = cudaGraphInstantiate(&x, g, 0)) != cudaSuccess) {
            cudaGraphDestroy(g);
            return fail(c, GB_ERR_CUDA, "cudaGraphInstantiate", e);
        }
        bg->graph = g;
        bg->exec = x;
        bg->kernels = kernels;
    }
    cudaError_t e = cudaGraphLaunch(bg->exec, s);
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaGraphLaunch", e);
    for (int k = 0; k < bg->kernels; ++k) gb::count_launch();
    return end(c, s);
}

gb_status run_buckets(gb_ctx *c, int nb, const void *const *in, void *const *out, const size_t *numel,
                      gb_dtype dtype, gb_op op, gb_codec codec, int block, int rs, float *const *res,
                      cudaStream_t s) {
    // the chunk shape of the largest bucket fixes the slot size.  Chunks are
    // kBucketChunkScale x the pipeline chunk: across a gradient set the
    // pipeline fills once, so larger copies only save per-chunk cost (two
    // copies, two launches and their event waits).  On GB300 12 MiB, which
    // leaves most buckets of both bf16 sets (GPT-2 small, the 1.1B
    // Llama-style set) in one chunk, beat 6 MiB by 4-5 % and tied 16-24 MiB
    size_t nmax = 0;
    for (int b = 0; b < nb; ++b) nmax = numel[b] > nmax ? numel[b] : nmax;
    Plan p = make_plan(c, nmax, dtype, op, codec, block, 0, false, kBucketChunkScale * c->chunk_bytes, false);
    // each bucket in balanced chunks of whole tiles, none larger than the
    // plan's chunk (so a bucket never ends in a sliver of a chunk)
    std::vector<WorkChunk> work;
    for (int b = 0; b < nb; ++b) {
        const uint64_t k = (numel[b] + p.chunk - 1) / p.chunk;
        const uint64_t ch = k ? round_up((numel[b] + k - 1) / k, gb::kTile) : p.chunk;
        const uint64_t cb = ch < p.chunk ? ch : p.chunk;
        for (uint64_t e0 = 0; e0 < numel[b]; e0 += cb)
            work.push_back({b, e0, (numel[b] - e0) < cb ? (numel[b] - e0) : cb});
    }
    const size_t recv = c->I == 2 ? 2 : (size_t)c->I * c->I;
    GB_TRY(grow_device(c, &c->d_stage, &c->d_stage_bytes, (size_t)(c->I + recv) * kBucketSlots * p.part));
    GB_TRY(grow_host(c, (size_t)c->I * kBucketSlots * p.part));
    GB_TRY(begin(c, s));
    if (!c->use_graphs) {
        GB_TRY(enqueue_buckets(c, p, work, in, out, numel, rs, res, s));
        return end(c, s);
    }
    std::vector<uint64_t> key = {1, (uint64_t)nb, (uint64_t)dtype, (uint64_t)op, (uint64_t)p.eff, (uint64_t)p.blk,
                                 (uint64_t)p.chunk, (uint64_t)(uintptr_t)c->d_stage, (uint64_t)(uintptr_t)c->h_stage,
                                 (uint64_t)rs};
    for (int b = 0; b < nb; ++b) {
        key.push_back(numel[b]);
        for (int r = 0; r < c->W; ++r) {
            key.push_back((uint64_t)(uintptr_t)in[(size_t)b * c->W + r]);
            key.push_back((uint64_t)(uintptr_t)out[(size_t)b * c->W + r]);
        }
        for (int q = 0; res && q < c->I; ++q) key.push_back((uint64_t)(uintptr_t)res[(size_t)b * c->I + q]);
    }
    key.push_back(res ? 1 : 0);
    return run_set_graph(c, key, 2 * (int)work.size(),
                         [&](cudaStream_t st) { return enqueue_buckets(c, p, work, in, out, numel, rs, res, st); }, s);
}

// Capture one pipelined all_reduce on the context's capture stream and
// instantiate it.  The stand-in mark events become event-record nodes.
gb_status capture_rbb(gb_ctx *c, const Plan &p, const void *const *in, float *const *res, bool timed,
                      GraphEntry *ge) {
    cudaError_t e = cudaStreamBeginCapture(c->scap, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaStreamBeginCapture", e);
    gb_status st = enqueue_rbb(c, p, in, (void *const *)in, res, c->scap, timed ? kMarkCapture : kMarkOff, true);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(c->scap, &g);
    if (st != GB_OK) {
        if (g) cudaGraphDestroy(g);
        return st;
    }
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaStreamEndCapture", e);
    cudaGraphExec_t x = nullptr;
    if ((e = cudaGraphInstantiate(&x, g, 0)) != cudaSuccess) {
        cudaGraphDestroy(g);
        return fail(c, GB_ERR_CUDA, "cudaGraphInstantiate", e);
    }
    ge->graph = g;
    ge->exec = x;
    ge->n_marks = 0;
    if (timed) {
        size_t count = 0;
        cudaGraphGetNodes(g, nullptr, &count);
        cudaGraphNode_t *nodes = new (std::nothrow) cudaGraphNode_t[count ? count : 1];
        if (!nodes) return fail(c, GB_ERR_ALLOC, "graph node list");
        cudaGraphGetNodes(g, nodes, &count);
        for (size_t i = 0; i < count; ++i) {
            cudaGraphNodeType t;
            cudaEvent_t ev;
            if (cudaGraphNodeGetType(nodes[i], &t) != cudaSuccess || t != cudaGraphNodeTypeEventRecord) continue;
            if (cudaGraphEventRecordNodeGetEvent(nodes[i], &ev) != cudaSuccess) continue;
            for (int k = 0; k < kMarks; ++k)
                if (c->cap_mark[k] == ev) {
                    ge->mark_node[k] = nodes[i];
                    ++ge->n_marks;
                }
        }
        delete[] nodes;
    }
    return GB_OK;
}

GraphEntry *find_graph(gb_ctx *c, const GraphKey &k) {
    for (int i = 0; i < c->n_graphs; ++i)
        if (memcmp(&c->graphs[i].key, &k, sizeof k) == 0) return &c->graphs[i];
    return nullptr;
}

GraphEntry *new_graph_slot(gb_ctx *c) {
    if (c->n_graphs < kMaxGraphs) return &c->graphs[c->n_graphs++];
    int lru = 0;
    for (int i = 1; i < c->n_graphs; ++i)
        if (c->graphs[i].last_use < c->graphs[lru].last_use) lru = i;
    GraphEntry &g = c->graphs[lru];
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.graph) cudaGraphDestroy(g.graph);
    g = GraphEntry();
    return &g;
}

// all_gather of every bucket as one pipeline (bucket b: W inputs of
// numel_in[b] elements, W outputs of W * numel_in[b]).  For bucket b, one
// copy kernel on the context's gather stream first gathers each island's
// rank blocks into its leader's output (gather(b)); groups of consecutive
// blocks of one island (whole islands, up to kBucketChunkScale pipeline
// chunks) then go device -> host from there through host slot b % 2 in one
// copy each on stream D, and each group on to every other leader on stream
// H as soon as it has landed; once bucket b has landed, one copy kernel per
// island spreads the leader's W blocks to the island's other ranks
// (spread(b), on s) while the next buckets' blocks are on the link.  Every
// copy carries a fixed cost of a few microseconds on its stream, so
// gathering first moves the same bytes in one device -> host copy per group
// instead of one per rank block.  The gathers depend on nothing but the
// caller's prior work, so on their own stream they run ahead of the copies
// instead of waiting behind spreads.  A slot is written again only after the
// host -> device copies that read it.
gb_status enqueue_ag_buckets(gb_ctx *c, int nb, const void *const *in, void *const *out, const size_t *numel_in,
                             size_t eb, size_t slot_bytes, cudaStream_t s) {
    const int W = c->W, I = c->I;
    cudaStream_t D = c->sd, H = c->sh, G = c->sg;
    if (c->inject == GB_INJECT_BRIDGE) {
        c->inject = 0;
        return fail(c, GB_ERR_BRIDGE, "bridge hop failed (injected)");
    }
    GB_TRY(record(c, c->ev_join_d, s));  // the other streams start after the caller's prior work
    GB_TRY(wait_on(c, D, c->ev_join_d));
    GB_TRY(wait_on(c, H, c->ev_join_d));
    GB_TRY(wait_on(c, G, c->ev_join_d));
    int ng = 0;
    auto front = [&](int b, int slot, bool reuse) -> gb_status {  // gather(b), then its groups' copies
        const size_t mb = numel_in[b] * eb;
        unsigned char *host = c->h_stage + (size_t)slot * slot_bytes;
        const void *const *bin = in + (size_t)b * W;
        void *const *bout = out + (size_t)b * W;
        gb::CopyArgs a;
        memset(&a, 0, sizeof a);
        a.n_jobs = W;
        a.bytes = mb;
        a.vec = (mb % 16) == 0;
        for (int i = 0; i < I; ++i) a.dst[i] = (unsigned char *)bout[c->first[i]];
        for (int q = 0; q < W; ++q) {
            a.src[q] = (const unsigned char *)bin[q];
            a.dst_off[q] = (size_t)q * mb;
            a.dst_lo[q] = c->island_of[q];
            a.dst_hi[q] = c->island_of[q] + 1;
        }
        GB_TRY(check_launch(c, gb::launch_copy(a, G), "all_gather gather"));
        cudaEvent_t gathered = c->ev_ag[ng++ % GB_MAX_RANKS];
        GB_TRY(record(c, gathered, G));
        GB_TRY(wait_on(c, D, gathered));
        if (reuse) GB_TRY(wait_on(c, D, c->ev_in[slot]));  // the slot's last reader has finished
        const size_t target = kBucketChunkScale * c->chunk_bytes;
        const size_t per_s = mb >= target ? 1 : target / mb;
        const int per = per_s > (size_t)W ? W : (int)per_s;
        for (int i = 0; i < I; ++i) {
            const unsigned char *lead_i = (const unsigned char *)bout[c->first[i]];
            for (int q0 = c->first[i]; q0 < c->first[i + 1]; q0 += per) {
                const int q1 = (q0 + per) < c->first[i + 1] ? (q0 + per) : c->first[i + 1];
                GB_TRY(copy_async(c, host + (size_t)q0 * mb, lead_i + (size_t)q0 * mb, (size_t)(q1 - q0) * mb,
                                  cudaMemcpyDeviceToHost, D));
                cudaEvent_t ev = c->ev_ag[ng++ % GB_MAX_RANKS];
                GB_TRY(record(c, ev, D));
                GB_TRY(wait_on(c, H, ev));
                for (int g = 0; g < I; ++g) {
                    if (g == i) continue;
                    unsigned char *lead = (unsigned char *)bout[c->first[g]];
                    GB_TRY(copy_async(c, lead + (size_t)q0 * mb, host + (size_t)q0 * mb, (size_t)(q1 - q0) * mb,
                                      cudaMemcpyHostToDevice, H));
                }
            }
        }
        GB_TRY(record(c, c->ev_in[slot], H));  // bucket b has landed; slot free again
        return GB_OK;
    };
    auto back = [&](int b, int slot) -> gb_status {  // spread(b)
        const size_t mb = numel_in[b] * eb;
        void *const *bout = out + (size_t)b * W;
        GB_TRY(wait_on(c, s, c->ev_in[slot]));
        for (int i = 0; i < I; ++i) {
            if (c->size[i] < 2) continue;  // the leader already holds every block
            gb::CopyArgs a;
            memset(&a, 0, sizeof a);
            a.n_jobs = 1;
            a.bytes = (size_t)W * mb;
            a.vec = (mb % 16) == 0;
            a.src[0] = (const unsigned char *)bout[c->first[i]];
            a.dst_off[0] = 0;
            a.dst_lo[0] = 0;
            a.dst_hi[0] = c->size[i] - 1;
            for (int k = 1; k < c->size[i]; ++k) a.dst[k - 1] = (unsigned char *)bout[c->first[i] + k];
            GB_TRY(check_launch(c, gb::launch_copy(a, s), "all_gather spread"));
        }
        return GB_OK;
    };
    // spread(b) is enqueued after front(b + 1) and before front(b + 2), which
    // records the next landing in the same slot's event
    int prev = -1, prev_slot = 0, done = 0;
    for (int b = 0; b < nb; ++b) {
        if (numel_in[b] == 0) continue;
        const int slot = done % 2;
        GB_TRY(front(b, slot, done >= 2));
        if (prev >= 0) GB_TRY(back(prev, prev_slot));
        prev = b;
        prev_slot = slot;
        ++done;
    }
    if (prev >= 0) GB_TRY(back(prev, prev_slot));
    cudaEvent_t g_end = c->ev_ag[ng++ % GB_MAX_RANKS];
    GB_TRY(record(c, g_end, G));
    GB_TRY(record(c, c->ev_join_d, D));
    GB_TRY(record(c, c->ev_join_h, H));
    GB_TRY(wait_on(c, s, c->ev_join_d));
    GB_TRY(wait_on(c, s, c->ev_join_h));
    GB_TRY(wait_on(c, s, g_end));
    return GB_OK;
}

// Reduce-bridge-broadcast over W rank buffers `in` (n elements).  rs == 0:
// the total goes to out[r] (all n elements; out may equal in).  rs == 1:
// out[r] receives slice r (n / W elements).  A pipelined in-place
// all_reduce runs as a CUDA graph captured on the second call with the same
// buffers and shape (the first runs directly) and replayed afterwards.
gb_status run_rbb(gb_ctx *c, const void *const *in, void *const *out, size_t n, gb_dtype dtype,
                  gb_op op, gb_codec codec, int block, cudaStream_t s, int rs, float *const *res) {
    // the chunk follows the payload; reduce_scatter's is shorter (make_plan)
    const Plan p = make_plan(c, n, dtype, op, codec, block, rs, true);
    GB_TRY(ensure_links(c, p.links));
    GB_TRY(grow_device(c, &c->d_stage, &c->d_stage_bytes, p.dev_bytes));
    if (p.host_bytes) GB_TRY(grow_host(c, p.host_bytes));
    GB_TRY(begin(c, s));
    const bool timed = c->tcap > 0;
    const bool graphable = !rs && p.C > 1 && c->use_graphs && (const void *)in == (const void *)out;
    if (!graphable) {
        GB_TRY(enqueue_rbb(c, p, in, out, res, s, timed ? kMarkDirect : kMarkOff, p.C > 1));
        commit_marks(c, p.C, p.I > 1);
        return end(c, s);
    }
    GraphKey k;
    memset(&k, 0, sizeof k);
    for (int r = 0; r < c->W; ++r) k.in[r] = in[r];
    for (int i = 0; res && i < c->I; ++i) k.res[i] = res[i];
    k.n = n;
    k.chunk = p.chunk;
    k.dtype = dtype;
    k.op = op;
    k.codec = p.eff;
    k.block = p.blk;
    k.timed = timed;
    k.links = p.links;
    k.d_stage = c->d_stage;
    k.h_stage = c->h_stage;
    GraphEntry *ge = find_graph(c, k);
    if (!ge) {  // first time: run directly (loads modules, sizes grids), remember the shape
        ge = new_graph_slot(c);
        ge->key = k;
        ge->last_use = ++c->clock;
        GB_TRY(enqueue_rbb(c, p, in, out, res, s, timed ? kMarkDirect : kMarkOff, true));
        commit_marks(c, p.C, true);
        return end(c, s);
    }
    ge->last_use = ++c->clock;
    if (!ge->exec) GB_TRY(capture_rbb(c, p, in, res, timed, ge));
    if (timed) {
        const long long slot = c->tcount % c->tcap;
        for (int idx = 0; idx < kMarks; ++idx) {
            if (!ge->mark_node[idx]) continue;
            cudaEvent_t ev;
            GB_TRY(ring_event(c, slot, idx, &ev));
            cudaError_t e = cudaGraphExecEventRecordNodeSetEvent(ge->exec, ge->mark_node[idx], ev);
            if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaGraphExecEventRecordNodeSetEvent", e);
        }
    }
    cudaError_t e = cudaGraphLaunch(ge->exec, s);
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaGraphLaunch", e);
    for (int k = 0; k < 2 * p.C; ++k) gb::count_launch();  // the graph's kernel nodes
    commit_marks(c, p.C, true);
    return end(c, s);
}

gb_status check_collective(gb_ctx *c, size_t n, int dtype, int op, int codec, int block) {
    GB_TRY(check_dtype(c, dtype));
    GB_TRY(check_op(c, op));
    GB_TRY(check_codec(c, codec, block));
    GB_TRY(check_n(c, n));
    if (op == GB_AVG && !is_float_dtype(dtype))
        return set_msg(c, GB_ERR_UNSUPPORTED_OP, "AVG needs a floating dtype");
    if ((dtype == GB_F16 || dtype == GB_F64) && (op == GB_SUM || op == GB_AVG) && codec != GB_CODEC_NONE)
        return set_msg(c, GB_ERR_UNSUPPORTED_CODEC, "float16 / float64 are not compressed");
    return GB_OK;
}

}  // namespace gbrt
