// The C entry points of libgb (include/gb.h): argument checks, then the
// runtime's pipelines (gb_runtime.cu).
#include "gb_internal.cuh"

using namespace gbrt;


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
        drop_graphs(c);
        free_marks(c);
        cudaStream_t streams[4] = {c->sd, c->sh, c->scap, c->sg};
        for (cudaStream_t st : streams)
            if (st) cudaStreamDestroy(st);
        for (int i = 0; i < kMaxChunks; ++i) {
            cudaEvent_t evs[5] = {c->ev_k1[i], c->ev_d2h[i], c->ev_h2d[i], c->ev_in[i], c->ev_k2[i]};
            for (cudaEvent_t ev : evs)
                if (ev) cudaEventDestroy(ev);
        }
        if (c->ev_join_d) cudaEventDestroy(c->ev_join_d);
        if (c->ev_join_h) cudaEventDestroy(c->ev_join_h);
        for (int i = 0; i < GB_MAX_RANKS; ++i)
            if (c->ev_ag[i]) cudaEventDestroy(c->ev_ag[i]);
        for (int l = 1; l < kMaxLinks; ++l) {
            if (c->lsd[l]) cudaStreamDestroy(c->lsd[l]);
            if (c->lsh[l]) cudaStreamDestroy(c->lsh[l]);
            if (c->ev_ljd[l]) cudaEventDestroy(c->ev_ljd[l]);
            if (c->ev_ljh[l]) cudaEventDestroy(c->ev_ljh[l]);
        }
        for (int i = 0; i < kMarks; ++i)
            if (c->cap_mark[i]) cudaEventDestroy(c->cap_mark[i]);
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
gb_status gb_last_error(const gb_ctx *c) { return c ? c->last : GB_ERR_INVALID_ARG; }

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
    const Plan ar = make_plan(c, n, dtype, GB_SUM, codec, block, 0, true);
    const Plan rs = make_plan(c, n, dtype, GB_SUM, codec, block, 1, false);
    const size_t ag_host = (size_t)c->W * n * elem_bytes(dtype);
    size_t dev = ar.dev_bytes > rs.dev_bytes ? ar.dev_bytes : rs.dev_bytes;
    size_t host = ar.host_bytes > rs.host_bytes ? ar.host_bytes : rs.host_bytes;
    const size_t ex_part = round_up(n * gb::exact_payload_elem_bytes(dtype, GB_SUM), 256);
    const size_t ex_dev = (size_t)(c->I + (c->I == 1 ? 0 : c->I == 2 ? 2 : c->I * c->I)) * ex_part;
    if (ex_dev > dev) dev = ex_dev;
    if (c->I > 1 && (size_t)c->I * ex_part > host) host = (size_t)c->I * ex_part;
    if (ag_host > host) host = ag_host;
    GB_TRY(grow_device(c, &c->d_stage, &c->d_stage_bytes, dev));
    GB_TRY(grow_host(c, host));
    return GB_OK;
}

gb_status gb_set_pipeline(gb_ctx *c, size_t chunk_bytes, int use_graphs) {
    if (!c) return GB_ERR_INVALID_ARG;
    if (c->device >= 0 && c->done_recorded) cudaEventSynchronize(c->done);
    drop_graphs(c);
    c->chunk_bytes = chunk_bytes;
    c->use_graphs = use_graphs ? 1 : 0;
    return GB_OK;
}

gb_status gb_set_sharded_bridge(gb_ctx *c, int on) {
    if (!c) return GB_ERR_INVALID_ARG;
    if (c->device >= 0 && c->done_recorded) cudaEventSynchronize(c->done);
    drop_graphs(c);
    c->sharded = on ? 1 : 0;
    return GB_OK;
}

gb_status gb_island_reduce(gb_ctx *c, int island, const void *const *rank_bufs, size_t n,
                           gb_dtype dtype, float *island_sum, gb_stream stream) {
    GB_TRY(check_ctx(c));
    if (island < 0 || island >= c->I) return set_msg(c, GB_ERR_INVALID_ARG, "island %d", island);
    const int K = c->size[island];
    GB_TRY(check_codec_dtype(c, dtype));
    GB_TRY(check_n(c, n));
    GB_TRY(check_rank_bufs(c, rank_bufs, K, "rank_bufs"));
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
    ra.tiles = (uint32_t)((n + gb::kTile - 1) / gb::kTile);
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
    ra.tiles = (uint32_t)((n + gb::kTile - 1) / gb::kTile);
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
    GB_TRY(check_codec_dtype(c, dtype));
    if (op != GB_SUM && op != GB_AVG) return set_msg(c, GB_ERR_UNSUPPORTED_OP, "island broadcast takes SUM / AVG");
    GB_TRY(check_n(c, n));
    GB_TRY(check_dev_ptr(c, total, "total"));
    GB_TRY(check_rank_bufs(c, (const void *const *)rank_bufs, K, "rank_bufs"));
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
    da.world_pow2 = (c->W & (c->W - 1)) == 0;
    da.inv_world = 1.0f / (float)c->W;
    da.n = n;
    da.scales_off = 0;
    da.rs = 0;
    da.vec = 1;
    da.tiles = (uint32_t)((n + gb::kTile - 1) / gb::kTile);
    return check_launch(c, gb::launch_decode_bcast(da, dtype, GB_CODEC_NONE, 256, (cudaStream_t)stream),
                        "island broadcast");
}

// gb_island_reduce_compress with (res != NULL) or without error feedback.
static gb_status island_reduce_compress(gb_ctx *c, const void *const *rank_bufs, float *const *res, size_t n,
                                        gb_dtype dtype, gb_codec codec, int block, void *const *payloads,
                                        gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_codec_dtype(c, dtype));
    GB_TRY(check_codec(c, codec, block));
    GB_TRY(check_n(c, n));
    GB_TRY(check_rank_bufs(c, rank_bufs, c->W, "rank_bufs"));
    GB_TRY(check_dev_bufs(c, (const void *const *)payloads, c->I, "payloads"));
    if (res) GB_TRY(check_dev_bufs(c, (const void *const *)res, c->I, "residuals"));
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    const int blk = is_fp8(codec) ? block : 256;
    gb::ReduceEncodeArgs ra;
    memset(&ra, 0, sizeof ra);
    for (int r = 0; r < c->W; ++r) ra.src[r] = rank_bufs[r];
    for (int i = 0; i < c->I; ++i) ra.payload[i] = payloads[i];
    for (int i = 0; res && i < c->I; ++i) ra.residual[i] = res[i];
    for (int i = 0; i <= c->I; ++i) ra.first[i] = c->first[i];
    ra.n_islands = c->I;
    ra.n = n;
    ra.tiles = (uint32_t)((n + gb::kTile - 1) / gb::kTile);
    ra.scales_off = scales_offset(codec, n);
    return check_launch(c, gb::launch_reduce_encode(ra, dtype, codec, blk, (cudaStream_t)stream),
                        "island reduce + compress");
}

gb_status gb_island_reduce_compress(gb_ctx *c, const void *const *rank_bufs, size_t n, gb_dtype dtype,
                                    gb_codec codec, int block, void *const *payloads, gb_stream stream) {
    return island_reduce_compress(c, rank_bufs, nullptr, n, dtype, codec, block, payloads, stream);
}

gb_status gb_island_reduce_compress_ef(gb_ctx *c, const void *const *rank_bufs, float *const *residuals, size_t n,
                                       gb_dtype dtype, gb_codec codec, int block, void *const *payloads,
                                       gb_stream stream) {
    if (c && !residuals) return set_msg(c, GB_ERR_INVALID_ARG, "residuals is NULL");
    return island_reduce_compress(c, rank_bufs, residuals, n, dtype, codec, block, payloads, stream);
}

// The second half of the fused pair: decode (or fold) the payloads, add them
// in island order, divide for AVG, and write every rank (rs == 0) or rank
// r's slice of n / W elements (rs == 1).
static gb_status decompress_to_ranks(gb_ctx *c, const void *const *payloads, size_t n, gb_dtype dtype, gb_op op,
                                     gb_codec codec, int block, void *const *dst, int rs, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_collective(c, n, dtype, op, codec, block));
    GB_TRY(check_dev_bufs(c, payloads, c->I * c->I, "payloads"));
    GB_TRY(check_rank_bufs(c, (const void *const *)dst, c->W, rs ? "out" : "rank_bufs"));
    if (rs && n % (size_t)c->W)
        return set_msg(c, GB_ERR_INVALID_ARG, "n = %zu is not a multiple of W = %d", n, c->W);
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    const bool exact = is_exact(dtype, op);
    const int blk = is_fp8(codec) ? block : 256;
    gb::DecodeBcastArgs da;
    memset(&da, 0, sizeof da);
    for (int r = 0; r < c->W; ++r) {
        da.dst[r] = dst[r];
        da.group_of_rank[r] = c->island_of[r];
    }
    bool same_rows = true;  // every leader holds the same pointers: decode once
    for (int g = 1; g < c->I && same_rows; ++g)
        for (int j = 0; j < c->I; ++j) same_rows = same_rows && payloads[g * c->I + j] == payloads[j];
    if (same_rows) {
        gb::decode_once(da, c->W, c->I, payloads);
    } else {
        for (int g = 0; g < c->I; ++g)
            for (int j = 0; j < c->I; ++j) da.payload[g][j] = payloads[g * c->I + j];
        for (int i = 0; i <= c->I; ++i) da.first[i] = c->first[i];
        da.n_groups = c->I;
        da.n_src = c->I;
    }
    if (rs) {  // grid unit r (first[n_groups] = W of them): rank r's slice, from row group_of_rank[r]
        const uint64_t m = n / (uint64_t)c->W;
        for (int r = 0; r < c->W; ++r) {
            da.rs_src[r] = (uint64_t)r * m;
            da.rs_len[r] = m;
        }
        da.rs = 1;
        const uint64_t ve = exact ? 16 / elem_bytes(dtype) : 8;
        da.vec = (m % ve) == 0;
        da.tiles = (uint32_t)((m + gb::kTile - 1) / gb::kTile);
    } else {
        da.rs = 0;
        da.vec = 1;
        da.tiles = (uint32_t)((n + gb::kTile - 1) / gb::kTile);
    }
    da.avg = op == GB_AVG;
    da.world = (float)c->W;
    da.world_pow2 = (c->W & (c->W - 1)) == 0;
    da.inv_world = 1.0f / (float)c->W;
    da.n = n;
    da.scales_off = exact ? 0 : scales_offset(codec, n);
    cudaStream_t s = (cudaStream_t)stream;
    if (exact) return check_launch(c, gb::launch_exact_combine(da, dtype, op, s), "fold + broadcast");
    return check_launch(c, gb::launch_decode_bcast(da, dtype, codec, blk, s), "decompress + island broadcast");
}

gb_status gb_decompress_island_broadcast(gb_ctx *c, const void *const *payloads, size_t n, gb_dtype dtype,
                                         gb_op op, gb_codec codec, int block, void *const *rank_bufs,
                                         gb_stream stream) {
    return decompress_to_ranks(c, payloads, n, dtype, op, codec, block, rank_bufs, 0, stream);
}

gb_status gb_decompress_scatter(gb_ctx *c, const void *const *payloads, size_t n, gb_dtype dtype, gb_op op,
                                gb_codec codec, int block, void *const *out, gb_stream stream) {
    return decompress_to_ranks(c, payloads, n, dtype, op, codec, block, out, 1, stream);
}

size_t gb_island_payload_bytes(gb_dtype dtype, gb_op op, gb_codec codec, int block, size_t n) {
    if (dtype < GB_F32 || dtype > GB_I64 || op < GB_SUM || op > GB_MIN || !codec_ok(codec, block)) return 0;
    if (op == GB_AVG && !is_float_dtype(dtype)) return 0;
    if ((dtype == GB_F16 || dtype == GB_F64) && (op == GB_SUM || op == GB_AVG) && codec != GB_CODEC_NONE) return 0;
    if (is_exact(dtype, op)) return n * gb::exact_payload_elem_bytes(dtype, op);
    return payload_bytes(codec, block, n);
}

gb_status gb_island_reduce_compress_op(gb_ctx *c, const void *const *rank_bufs, size_t n, gb_dtype dtype,
                                       gb_op op, gb_codec codec, int block, void *const *payloads,
                                       gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_collective(c, n, dtype, op, codec, block));
    if (!is_exact(dtype, op))
        return island_reduce_compress(c, rank_bufs, nullptr, n, dtype, codec, block, payloads, stream);
    GB_TRY(check_rank_bufs(c, rank_bufs, c->W, "rank_bufs"));
    GB_TRY(check_dev_bufs(c, (const void *const *)payloads, c->I, "payloads"));
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    gb::ReduceEncodeArgs ra;
    memset(&ra, 0, sizeof ra);
    for (int r = 0; r < c->W; ++r) ra.src[r] = rank_bufs[r];
    for (int i = 0; i < c->I; ++i) ra.payload[i] = payloads[i];
    for (int i = 0; i <= c->I; ++i) ra.first[i] = c->first[i];
    ra.n_islands = c->I;
    ra.n = n;
    ra.tiles = (uint32_t)((n + gb::kTile - 1) / gb::kTile);
    return check_launch(c, gb::launch_exact_reduce(ra, dtype, op, (cudaStream_t)stream), "island fold");
}

gb_status gb_all_reduce(gb_ctx *c, void *const *rank_bufs, size_t n, gb_dtype dtype, gb_op op,
                        gb_codec codec, int block, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_collective(c, n, dtype, op, codec, block));
    GB_TRY(check_rank_bufs(c, (const void *const *)rank_bufs, c->W, "rank_bufs"));
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    return run_rbb(c, (const void *const *)rank_bufs, rank_bufs, n, dtype, op, codec, block,
                   (cudaStream_t)stream, 0);
}

gb_status gb_all_reduce_ef(gb_ctx *c, void *const *rank_bufs, float *const *residuals, size_t n, gb_dtype dtype,
                           gb_op op, gb_codec codec, int block, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_collective(c, n, dtype, op, codec, block));
    if (is_exact(dtype, op))
        return set_msg(c, GB_ERR_UNSUPPORTED_OP, "error feedback applies to float32 / bfloat16 SUM / AVG");
    GB_TRY(check_rank_bufs(c, (const void *const *)rank_bufs, c->W, "rank_bufs"));
    GB_TRY(check_dev_bufs(c, (const void *const *)residuals, c->I, "residuals"));
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    return run_rbb(c, (const void *const *)rank_bufs, rank_bufs, n, dtype, op, codec, block, (cudaStream_t)stream,
                   0, residuals);
}

gb_status gb_reduce_scatter(gb_ctx *c, const void *const *in, void *const *out, size_t n_in,
                            gb_dtype dtype, gb_op op, gb_codec codec, int block, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_collective(c, n_in, dtype, op, codec, block));
    GB_TRY(check_rank_bufs(c, in, c->W, "in"));
    GB_TRY(check_rank_bufs(c, (const void *const *)out, c->W, "out"));
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
    GB_TRY(check_rank_bufs(c, in, c->W, "in"));
    GB_TRY(check_rank_bufs(c, (const void *const *)out, c->W, "out"));
    if (n_in == 0) return GB_OK;
    GB_TRY(bind(c));
    cudaStream_t s = (cudaStream_t)stream;
    const int W = c->W, I = c->I;
    const size_t mb = n_in * elem_bytes(dtype);
    if (I > 1) {  // one island touches no staging: nothing to order against other calls
        GB_TRY(grow_host(c, (size_t)W * mb));
        GB_TRY(begin(c, s));
    }
    const int mm = c->tcap > 0 ? kMarkDirect : kMarkOff;
    GB_TRY(mark(c, mm, 0, s));
    GB_TRY(mark(c, mm, 1, s));
    if (I > 1) {
        if (c->inject == GB_INJECT_BRIDGE) {
            c->inject = 0;
            return fail(c, GB_ERR_BRIDGE, "bridge hop failed (injected)");
        }
        GB_TRY(mark(c, mm, 2, s));
        if (c->chunk_bytes == 0) {
            // one hop on the caller's stream: every rank's block goes to the
            // host slots, then each leader receives the other islands' blocks
            for (int q = 0; q < W; ++q)
                GB_TRY(copy_async(c, c->h_stage + (size_t)q * mb, in[q], mb, cudaMemcpyDeviceToHost, s));
            for (int i = 0; i < I; ++i) {
                unsigned char *lead = (unsigned char *)out[c->first[i]];
                const size_t lo = (size_t)c->first[i] * mb, hi = (size_t)c->first[i + 1] * mb;
                GB_TRY(copy_async(c, lead, c->h_stage, lo, cudaMemcpyHostToDevice, s));
                GB_TRY(copy_async(c, lead + hi, c->h_stage + hi, (size_t)W * mb - hi, cudaMemcpyHostToDevice, s));
            }
        } else {
            // pipelined: groups of consecutive ranks of one island (about
            // chunk_bytes each) go to the host on copy stream D; as soon as
            // a group has landed, stream H carries it to every other leader
            const size_t per_s = mb >= c->chunk_bytes ? 1 : c->chunk_bytes / mb;
            const int per = per_s > (size_t)W ? W : (int)per_s;
            cudaStream_t D = c->sd, H = c->sh;
            GB_TRY(record(c, c->ev_join_d, s));  // the copy streams start after the caller's prior work
            GB_TRY(wait_on(c, D, c->ev_join_d));
            GB_TRY(wait_on(c, H, c->ev_join_d));
            int ng = 0;
            for (int i = 0; i < I; ++i) {
                for (int q0 = c->first[i]; q0 < c->first[i + 1]; q0 += per) {
                    const int q1 = (q0 + per) < c->first[i + 1] ? (q0 + per) : c->first[i + 1];
                    for (int q = q0; q < q1; ++q)
                        GB_TRY(copy_async(c, c->h_stage + (size_t)q * mb, in[q], mb, cudaMemcpyDeviceToHost, D));
                    GB_TRY(record(c, c->ev_ag[ng], D));
                    GB_TRY(wait_on(c, H, c->ev_ag[ng]));
                    ++ng;
                    for (int g = 0; g < I; ++g) {
                        if (g == i) continue;
                        unsigned char *lead = (unsigned char *)out[c->first[g]];
                        GB_TRY(copy_async(c, lead + (size_t)q0 * mb, c->h_stage + (size_t)q0 * mb,
                                          (size_t)(q1 - q0) * mb, cudaMemcpyHostToDevice, H));
                    }
                }
            }
            GB_TRY(record(c, c->ev_join_d, D));
            GB_TRY(record(c, c->ev_join_h, H));
            GB_TRY(wait_on(c, s, c->ev_join_d));
            GB_TRY(wait_on(c, s, c->ev_join_h));
        }
        GB_TRY(mark(c, mm, 3, s));
    }
    GB_TRY(mark(c, mm, 4, s));
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
    GB_TRY(mark(c, mm, 5, s));
    commit_marks(c, 1, I > 1);
    return I > 1 ? end(c, s) : GB_OK;
}

gb_status gb_broadcast(gb_ctx *c, void *const *rank_bufs, size_t n, gb_dtype dtype, int src,
                       gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_dtype(c, dtype));
    GB_TRY(check_n(c, n));
    GB_TRY(check_rank_bufs(c, (const void *const *)rank_bufs, c->W, "rank_bufs"));
    if (src < 0 || src >= c->W) return set_msg(c, GB_ERR_INVALID_ARG, "src %d", src);
    if (n == 0) return GB_OK;
    GB_TRY(bind(c));
    cudaStream_t s = (cudaStream_t)stream;
    const int I = c->I;
    const int si = c->island_of[src];
    const size_t nb = n * elem_bytes(dtype);
    if (I > 1) {  // one island touches no staging: nothing to order against other calls
        GB_TRY(grow_host(c, nb));
        GB_TRY(begin(c, s));
    }
    const int mm = c->tcap > 0 ? kMarkDirect : kMarkOff;
    GB_TRY(mark(c, mm, 0, s));
    GB_TRY(mark(c, mm, 1, s));
    if (I > 1) {
        if (c->inject == GB_INJECT_BRIDGE) {
            c->inject = 0;
            return fail(c, GB_ERR_BRIDGE, "bridge hop failed (injected)");
        }
        GB_TRY(mark(c, mm, 2, s));
        // src's island leader sends over the bridge (the bytes are src's);
        // every other leader receives in place
        if (c->chunk_bytes == 0 || nb <= kBcastPieceScale * c->chunk_bytes) {
            GB_TRY(copy_async(c, c->h_stage, rank_bufs[src], nb, cudaMemcpyDeviceToHost, s));
            for (int i = 0; i < I; ++i)
                if (i != si)
                    GB_TRY(copy_async(c, rank_bufs[c->first[i]], c->h_stage, nb, cudaMemcpyHostToDevice, s));
        } else {
            // pipelined: equal pieces of up to kBcastPieceScale x chunk_bytes
            // (at most GB_MAX_RANKS of them) go to the host on copy stream D;
            // as soon as one has landed, stream H carries it on to every other
            // leader.  Every piece is two plain copies, so larger pieces pay
            // (on GB300, 25 MiB: 237 us with 8 MiB pieces, 256 us with 2 MiB)
            size_t piece = round_up((nb + GB_MAX_RANKS - 1) / GB_MAX_RANKS, 256);
            if (piece < kBcastPieceScale * c->chunk_bytes) piece = kBcastPieceScale * c->chunk_bytes;
            const size_t pieces = (nb + piece - 1) / piece;
            piece = round_up((nb + pieces - 1) / pieces, 256);
            cudaStream_t D = c->sd, H = c->sh;
            GB_TRY(record(c, c->ev_join_d, s));  // the copy streams start after the caller's prior work
            GB_TRY(wait_on(c, D, c->ev_join_d));
            GB_TRY(wait_on(c, H, c->ev_join_d));
            int k = 0;
            for (size_t off = 0; off < nb; off += piece, ++k) {
                const size_t len = (nb - off) < piece ? (nb - off) : piece;
                GB_TRY(copy_async(c, c->h_stage + off, (const unsigned char *)rank_bufs[src] + off, len,
                                  cudaMemcpyDeviceToHost, D));
                GB_TRY(record(c, c->ev_ag[k], D));
                GB_TRY(wait_on(c, H, c->ev_ag[k]));
                for (int i = 0; i < I; ++i)
                    if (i != si)
                        GB_TRY(copy_async(c, (unsigned char *)rank_bufs[c->first[i]] + off, c->h_stage + off, len,
                                          cudaMemcpyHostToDevice, H));
            }
            GB_TRY(record(c, c->ev_join_d, D));
            GB_TRY(record(c, c->ev_join_h, H));
            GB_TRY(wait_on(c, s, c->ev_join_d));
            GB_TRY(wait_on(c, s, c->ev_join_h));
        }
        GB_TRY(mark(c, mm, 3, s));
    }
    GB_TRY(mark(c, mm, 4, s));
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
    GB_TRY(mark(c, mm, 5, s));
    commit_marks(c, 1, I > 1);
    return I > 1 ? end(c, s) : GB_OK;
}

// The body of gb_all_reduce_host and gb_all_reduce_host_rows, after their
// argument checks.  row_pitch > 0: the host buffers are the rows of one host
// allocation, row_pitch bytes apart, staged with 2D copies when the device
// takes both pitches.
static gb_status host_all_reduce(gb_ctx *c, void *const *host_bufs, size_t row_pitch, size_t n, gb_dtype dtype,
                                 gb_op op, gb_codec codec, int block, gb_stream stream) {
    GB_TRY(bind(c));
    cudaStream_t s = (cudaStream_t)stream;
    const size_t nb = n * elem_bytes(dtype);
    const size_t stride = round_up(nb, 256);
    GB_TRY(grow_device(c, &c->d_ranks, &c->d_ranks_bytes, (size_t)c->W * stride));
    void *dev[GB_MAX_RANKS];
    for (int r = 0; r < c->W; ++r) dev[r] = c->d_ranks + (size_t)r * stride;
    const size_t hpitch = row_pitch && row_pitch <= c->max_pitch && stride <= c->max_pitch ? row_pitch : 0;
    // Every chunk here also carries W rank buffers' worth of staging in and
    // out, which outweighs its payload, so a chunk is sized by that staging:
    // the elements whose W rank slices total kHostStageScale pipeline chunks
    // (16 MiB at the default).  On GB300 this kept the 25 MiB float32 E4M3
    // step (951 against 951 us with chunks of 1 MiB of payload, the earlier
    // rule) and took 64 MiB uncompressed from 2940 to 2792 us.  The chunks
    // are not balanced: a short last chunk shortens the drain of the copy
    // back to the host (25.2-25.7 GB/s, against 24.8-25.0 balanced).
    const uint64_t stage_elems = (uint64_t)(kHostStageScale * c->chunk_bytes) / ((uint64_t)c->W * elem_bytes(dtype));
    const Plan p = make_plan(c, n, dtype, op, codec, block, 0, false, c->chunk_bytes, false,
                             stage_elems > 0 ? stage_elems : 1);
    if (p.C > 1 && c->tcap == 0) {
        // pipelined: staging in, bridge and copy-back overlap chunk by chunk
        GB_TRY(grow_device(c, &c->d_stage, &c->d_stage_bytes, p.dev_bytes));
        GB_TRY(grow_host(c, p.host_bytes));
        GB_TRY(begin(c, s));
        if (!c->use_graphs) {
            GB_TRY(enqueue_host_pipeline(c, p, host_bufs, dev, stride, hpitch, s));
            return end(c, s);
        }
        GraphKey k;
        memset(&k, 0, sizeof k);
        for (int r = 0; r < c->W; ++r) {
            k.in[r] = dev[r];
            k.host[r] = host_bufs[r];
        }
        k.n = n;
        k.chunk = p.chunk;
        k.host_pitch = hpitch;
        k.dtype = dtype;
        k.op = op;
        k.codec = p.eff;
        k.block = p.blk;
        k.d_stage = c->d_stage;
        k.h_stage = c->h_stage;
        GraphEntry *ge = find_graph(c, k);
        if (!ge) {  // first time: run directly, remember the shape
            ge = new_graph_slot(c);
            ge->key = k;
            ge->last_use = ++c->clock;
            GB_TRY(enqueue_host_pipeline(c, p, host_bufs, dev, stride, hpitch, s));
            return end(c, s);
        }
        ge->last_use = ++c->clock;
        if (!ge->exec) {
            cudaError_t e = cudaStreamBeginCapture(c->scap, cudaStreamCaptureModeThreadLocal);
            if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaStreamBeginCapture", e);
            gb_status st = enqueue_host_pipeline(c, p, host_bufs, dev, stride, hpitch, c->scap);
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
        }
        cudaError_t e = cudaGraphLaunch(ge->exec, s);
        if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaGraphLaunch", e);
        for (int k2 = 0; k2 < 2 * p.C; ++k2) gb::count_launch();
        return end(c, s);
    }
    GB_TRY(begin(c, s));
    GB_TRY(stage_ranks(c, host_bufs, dev, stride, hpitch, 0, nb, cudaMemcpyHostToDevice, s));
    GB_TRY(run_rbb(c, (const void *const *)dev, dev, n, dtype, op, codec, block, s, 0));
    GB_TRY(stage_ranks(c, host_bufs, dev, stride, hpitch, 0, nb, cudaMemcpyDeviceToHost, s));
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
    return host_all_reduce(c, host_bufs, 0, n, dtype, op, codec, block, stream);
}

gb_status gb_all_reduce_host_rows(gb_ctx *c, void *host, size_t pitch, size_t n, gb_dtype dtype, gb_op op,
                                  gb_codec codec, int block, gb_stream stream) {
    GB_TRY(check_ctx(c));
    GB_TRY(check_collective(c, n, dtype, op, codec, block));
    if (!host) return set_msg(c, GB_ERR_INVALID_ARG, "host is NULL");
    if (n == 0) return GB_OK;
    const size_t nb = n * elem_bytes(dtype);
    if (c->W > 1 && pitch < nb)
        return set_msg(c, GB_ERR_INVALID_ARG, "pitch %zu is below a row's %zu bytes: the rows would overlap", pitch,
                       nb);
    if (c->W > 1 && pitch > (UINTPTR_MAX - (uintptr_t)host) / (size_t)(c->W - 1))
        return set_msg(c, GB_ERR_INVALID_ARG, "pitch %zu puts the last row past the end of the address space",
                       pitch);
    void *rows[GB_MAX_RANKS];
    for (int r = 0; r < c->W; ++r) rows[r] = (unsigned char *)host + (size_t)r * pitch;
    return host_all_reduce(c, rows, c->W > 1 ? pitch : 0, n, dtype, op, codec, block, stream);
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

// gb_all_reduce_buckets with (res != NULL) or without error feedback.
static gb_status all_reduce_buckets(gb_ctx *c, int n_buckets, void *const *bucket_bufs, float *const *res,
                                    const size_t *bucket_numel, gb_dtype dtype, gb_op op, gb_codec codec,
                                    int block, gb_stream stream) {
    GB_TRY(check_ctx(c));
    if (n_buckets < 0 || (n_buckets > 0 && (!bucket_bufs || !bucket_numel)))
        return set_msg(c, GB_ERR_INVALID_ARG, "bucket arrays");
    GB_TRY(check_collective(c, 0, dtype, op, codec, block));
    if (res && is_exact(dtype, op))
        return set_msg(c, GB_ERR_UNSUPPORTED_OP, "error feedback applies to float32 / bfloat16 SUM / AVG");
    for (int b = 0; b < n_buckets; ++b) {
        GB_TRY(check_n(c, bucket_numel[b]));
        if (bucket_numel[b] == 0) continue;  // an empty bucket's pointers are never used
        GB_TRY(check_rank_bufs(c, (const void *const *)(bucket_bufs + (size_t)b * c->W), c->W, "bucket_bufs"));
        if (res)
            GB_TRY(check_dev_bufs(c, (const void *const *)(res + (size_t)b * c->I), c->I, "residuals"));
    }
    size_t total = 0;
    for (int b = 0; b < n_buckets; ++b) total += bucket_numel[b];
    if (total == 0) return GB_OK;
    if (c->I > 1 && c->chunk_bytes > 0 && c->tcap == 0 && !c->sharded) {
        GB_TRY(bind(c));
        return run_buckets(c, n_buckets, (const void *const *)bucket_bufs, bucket_bufs, bucket_numel, dtype, op,
                           codec, block, 0, res, (cudaStream_t)stream);
    }
    for (int b = 0; b < n_buckets; ++b) {
        if (bucket_numel[b] == 0) continue;
        if (res)
            GB_TRY(gb_all_reduce_ef(c, bucket_bufs + (size_t)b * c->W, res + (size_t)b * c->I, bucket_numel[b], dtype,
                                    op, codec, block, stream));
        else
            GB_TRY(gb_all_reduce(c, bucket_bufs + (size_t)b * c->W, bucket_numel[b], dtype, op, codec, block, stream));
    }
    return GB_OK;
}

gb_status gb_all_reduce_buckets(gb_ctx *c, int n_buckets, void *const *bucket_bufs, const size_t *bucket_numel,
                                gb_dtype dtype, gb_op op, gb_codec codec, int block, gb_stream stream) {
    return all_reduce_buckets(c, n_buckets, bucket_bufs, nullptr, bucket_numel, dtype, op, codec, block, stream);
}

gb_status gb_all_reduce_buckets_ef(gb_ctx *c, int n_buckets, void *const *bucket_bufs, float *const *residuals,
                                   const size_t *bucket_numel, gb_dtype dtype, gb_op op, gb_codec codec, int block,
                                   gb_stream stream) {
    if (c && n_buckets > 0 && !residuals) return set_msg(c, GB_ERR_INVALID_ARG, "residuals is NULL");
    return all_reduce_buckets(c, n_buckets, bucket_bufs, residuals, bucket_numel, dtype, op, codec, block, stream);
}

gb_status gb_reduce_scatter_buckets(gb_ctx *c, int n_buckets, const void *const *in_bufs, void *const *out_bufs,
                                    const size_t *bucket_numel, gb_dtype dtype, gb_op op, gb_codec codec, int block,
                                    gb_stream stream) {
    GB_TRY(check_ctx(c));
    if (n_buckets < 0 || (n_buckets > 0 && (!in_bufs || !out_bufs || !bucket_numel)))
        return set_msg(c, GB_ERR_INVALID_ARG, "bucket arrays");
    GB_TRY(check_collective(c, 0, dtype, op, codec, block));
    size_t total = 0;
    for (int b = 0; b < n_buckets; ++b) {
        GB_TRY(check_n(c, bucket_numel[b]));
        if (bucket_numel[b] == 0) continue;  // an empty bucket's pointers are never used
        if (bucket_numel[b] % (size_t)c->W)
            return set_msg(c, GB_ERR_INVALID_ARG, "bucket %d: %zu elements is not a multiple of W = %d", b,
                           bucket_numel[b], c->W);
        GB_TRY(check_rank_bufs(c, in_bufs + (size_t)b * c->W, c->W, "in_bufs"));
        GB_TRY(check_rank_bufs(c, (const void *const *)(out_bufs + (size_t)b * c->W), c->W, "out_bufs"));
        total += bucket_numel[b];
    }
    if (total == 0) return GB_OK;
    if (c->I > 1 && c->chunk_bytes > 0 && c->tcap == 0) {
        GB_TRY(bind(c));
        return run_buckets(c, n_buckets, in_bufs, out_bufs, bucket_numel, dtype, op, codec, block, 1, nullptr,
                           (cudaStream_t)stream);
    }
    for (int b = 0; b < n_buckets; ++b)
        if (bucket_numel[b] > 0)
            GB_TRY(gb_reduce_scatter(c, in_bufs + (size_t)b * c->W, out_bufs + (size_t)b * c->W, bucket_numel[b],
                                     dtype, op, codec, block, stream));
    return GB_OK;
}

gb_status gb_all_gather_buckets(gb_ctx *c, int n_buckets, const void *const *in_bufs, void *const *out_bufs,
                                const size_t *bucket_numel_in, gb_dtype dtype, gb_stream stream) {
    GB_TRY(check_ctx(c));
    if (n_buckets < 0 || (n_buckets > 0 && (!in_bufs || !out_bufs || !bucket_numel_in)))
        return set_msg(c, GB_ERR_INVALID_ARG, "bucket arrays");
    GB_TRY(check_dtype(c, dtype));
    size_t total = 0, mb_max = 0;
    for (int b = 0; b < n_buckets; ++b) {
        GB_TRY(check_n(c, bucket_numel_in[b]));
        GB_TRY(check_n(c, bucket_numel_in[b] * (size_t)c->W));
        if (bucket_numel_in[b] == 0) continue;
        GB_TRY(check_rank_bufs(c, in_bufs + (size_t)b * c->W, c->W, "in_bufs"));
        GB_TRY(check_rank_bufs(c, (const void *const *)(out_bufs + (size_t)b * c->W), c->W, "out_bufs"));
        total += bucket_numel_in[b];
        const size_t mb = bucket_numel_in[b] * elem_bytes(dtype);
        if (mb > mb_max) mb_max = mb;
    }
    if (total == 0) return GB_OK;
    if (c->I > 1 && c->chunk_bytes > 0 && c->tcap == 0) {
        GB_TRY(bind(c));
        cudaStream_t s = (cudaStream_t)stream;
        const size_t slot_bytes = round_up((size_t)c->W * mb_max, 256);
        GB_TRY(grow_host(c, 2 * slot_bytes));
        GB_TRY(begin(c, s));
        const size_t eb = elem_bytes(dtype);
        int nonempty = 0;
        for (int b = 0; b < n_buckets; ++b) nonempty += bucket_numel_in[b] > 0;
        auto enqueue = [&](cudaStream_t st) {
            return enqueue_ag_buckets(c, n_buckets, in_bufs, out_bufs, bucket_numel_in, eb, slot_bytes, st);
        };
        if (!c->use_graphs) {
            GB_TRY(enqueue(s));
            return end(c, s);
        }
        std::vector<uint64_t> key = {2, (uint64_t)n_buckets, (uint64_t)dtype, (uint64_t)c->chunk_bytes,
                                     (uint64_t)(uintptr_t)c->h_stage};
        for (int b = 0; b < n_buckets; ++b) {
            key.push_back(bucket_numel_in[b]);
            for (int r = 0; r < c->W; ++r) {
                key.push_back((uint64_t)(uintptr_t)in_bufs[(size_t)b * c->W + r]);
                key.push_back((uint64_t)(uintptr_t)out_bufs[(size_t)b * c->W + r]);
            }
        }
        int spreads = 0;  // per bucket: one gather, one spread per island of two or more ranks
        for (int i = 0; i < c->I; ++i) spreads += c->size[i] > 1;
        return run_set_graph(c, key, nonempty * (1 + spreads), enqueue, s);
    }
    for (int b = 0; b < n_buckets; ++b)
        if (bucket_numel_in[b] > 0)
            GB_TRY(gb_all_gather(c, in_bufs + (size_t)b * c->W, out_bufs + (size_t)b * c->W, bucket_numel_in[b],
                                 dtype, stream));
    return GB_OK;
}

gb_status gb_set_phase_timing(gb_ctx *c, int capacity) {
    if (!c || capacity < 0 || capacity > (1 << 20)) return GB_ERR_INVALID_ARG;
    if (c->tev && c->done_recorded) cudaEventSynchronize(c->done);
    drop_graphs(c);
    free_marks(c);
    if (capacity > 0) {
        c->tev = new (std::nothrow) cudaEvent_t[(size_t)capacity * kMarks]();
        c->tnk2 = new (std::nothrow) int[capacity]();
        c->tbridge = new (std::nothrow) unsigned char[capacity]();
        if (!c->tev || !c->tnk2 || !c->tbridge) {
            free_marks(c);
            return set_msg(c, GB_ERR_ALLOC, "phase timing records");
        }
        c->tcap = capacity;
    }
    return GB_OK;
}

gb_status gb_phase_times(gb_ctx *c, int age, float *ms) {
    if (!c || !ms) return GB_ERR_INVALID_ARG;
    for (int i = 0; i < GB_N_PHASES; ++i) ms[i] = 0.0f;
    if (age < 0 || age >= c->tcap || age >= c->tcount)
        return set_msg(c, GB_ERR_INVALID_ARG, "no timed collective %d calls back", age);
    const long long slot = (c->tcount - 1 - age) % c->tcap;
    const cudaEvent_t *ev = c->tev + (size_t)slot * kMarks;
    const int nd = c->tnk2[slot];
    cudaError_t e = cudaEventSynchronize(ev[5 + 2 * (nd - 1)]);
    if (e != cudaSuccess) return fail(c, GB_ERR_CUDA, "cudaEventSynchronize", e);
    float t = 0.0f;
    if ((e = cudaEventElapsedTime(&ms[0], ev[0], ev[1])) != cudaSuccess)
        return fail(c, GB_ERR_CUDA, "cudaEventElapsedTime", e);
    if (c->tbridge[slot] && (e = cudaEventElapsedTime(&ms[1], ev[2], ev[3])) != cudaSuccess)
        return fail(c, GB_ERR_CUDA, "cudaEventElapsedTime", e);
    for (int j = 0; j < nd; ++j) {
        if ((e = cudaEventElapsedTime(&t, ev[4 + 2 * j], ev[5 + 2 * j])) != cudaSuccess)
            return fail(c, GB_ERR_CUDA, "cudaEventElapsedTime", e);
        ms[2] += t;
    }
    return GB_OK;
}

gb_status gb_last_phase_times(gb_ctx *c, float *ms) { return gb_phase_times(c, 0, ms); }

gb_status gb_debug_inject(gb_ctx *c, int what) {
    if (!c || (what != 0 && what != GB_INJECT_BRIDGE && what != GB_INJECT_ALLOC && what != GB_INJECT_OTHER_DEVICE))
        return GB_ERR_INVALID_ARG;
    c->inject = what;
    return GB_OK;
}

uint64_t gb_kernel_launch_count(void) { return gb::launches(); }

}  // extern "C"
