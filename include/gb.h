/*
 * gb.h - C ABI of libgb: the reduce-bridge-broadcast gradient all_reduce of
 * gpubridge, for simulated ranks that all live on one GB300 GPU.
 *
 * Model (gpubridge README, island / bridge paragraph and "all_reduce uses
 * reduce-bridge-broadcast"): W ranks form I islands; island i is the
 * contiguous block of global ranks [first_i, first_i + K_i), its leader is
 * its lowest rank.  An all_reduce
 *   1. sums each island's rank buffers onto the leader (float32, ascending
 *      rank order),
 *   2. encodes the island sum for the bridge (codec none / bf16 / fp8),
 *   3. moves the payloads between leaders through pinned host memory
 *      (device -> host -> device copies on the caller's stream),
 *   4. decodes every island's payload and adds them in float32, in island
 *      order (AVG then divides once by W),
 *   5. writes the total, rounded to the rank dtype, to every rank buffer.
 * Each simulated rank's buffer is a separate device allocation owned by the
 * caller.  Steps 1+2 and 4+5 run as one fused kernel each.
 *
 * Conventions for every call below:
 *   - Pointers named *_bufs / rank_bufs / in / out are arrays of W (or K_i)
 *     DEVICE pointers, in global rank order, each 16-byte aligned (the
 *     all_reduce alignment rule of the torch-mojo-backend page,
 *     "Distributed training", Limitations), so that a gradient view
 *     inside a bucket may start at any multiple of 16 bytes.  The kernels
 *     move float32 rank data with 32-byte accesses when every rank buffer of
 *     a launch is 32-byte aligned, else with two 16-byte accesses.  Every
 *     other device buffer argument (payloads, island sums, accumulators,
 *     totals, error-feedback residuals) must be 32-byte aligned (cudaMalloc
 *     and torch allocations are).  GB_ERR_MISALIGNED otherwise.  The caller
 *     owns them.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call validates all of its arguments first and returns an error with
 *     nothing enqueued; otherwise it enqueues its work on `stream` and returns
 *     without waiting for it (stream order, as torch.distributed's NCCL
 *     collectives: gpubridge README, "Stream semantics").  Inputs must not be
 *     written, and outputs not read, before that work completes.  The
 *     kernels are programmatic dependent launches: one may be scheduled
 *     while the kernel before it on the stream drains, but it touches no
 *     memory until that kernel has completed, so plain stream order holds
 *     for the caller's own kernels on both sides.
 *   - n = 0 is a valid no-op.
 *   - A context owns its pinned host slots and device staging buffers.  They
 *     grow to the largest call made so far and are released by gb_destroy
 *     (gpubridge README, "Pinned staging").  Growing frees and re-allocates,
 *     which waits for the device; gb_reserve grows ahead of time.
 *   - Calls on one context are ordered: each call waits (on the device) for
 *     the previous call's use of the staging buffers, even on another stream.
 *     Use one context per thread if calls come from several host threads.
 *   - Sticky failure (gpubridge README, "Async collectives": after a failed
 *     collective every later one refuses to start): if anything fails after
 *     work was enqueued (a CUDA error, an allocation failure, an injected
 *     bridge fault), the call returns that error and every later call on the
 *     context returns GB_ERR_CONTEXT_FAILED.  Argument errors are not sticky.
 */
#ifndef GB_H
#define GB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef void *gb_stream;

typedef enum {
    GB_OK = 0,
    GB_ERR_INVALID_ARG = 1,       /* null pointer, bad layout, bad size, bad rank index   */
    GB_ERR_UNSUPPORTED_DTYPE = 2, /* not a gb_dtype, or a dtype the call does not take    */
    GB_ERR_UNSUPPORTED_OP = 3,    /* not a gb_op, AVG on integers, or an op the call does */
                                  /* not take (MAX / MIN where only SUM / AVG apply)      */
    GB_ERR_UNSUPPORTED_CODEC = 4, /* unknown codec, fp8 block not 128 / 256, or a codec   */
                                  /* on float16 / float64 SUM / AVG                       */
    GB_ERR_MISALIGNED = 5,        /* a rank buffer not 16-byte aligned, or another device */
                                  /* buffer not 32-byte aligned                           */
    GB_ERR_ALLOC = 6,             /* pinned or device staging allocation failed (sticky)  */
    GB_ERR_CUDA = 7,              /* a CUDA runtime call failed (sticky)                  */
    GB_ERR_BRIDGE = 8,            /* the bridge hop failed (sticky)                       */
    GB_ERR_CONTEXT_FAILED = 9,    /* an earlier call on this context failed               */
    GB_ERR_NO_DEVICE = 10,        /* no CUDA device is usable                             */
    GB_ERR_TOO_LARGE = 11         /* exceeds the fixed buffers of gb_all_reduce_noalloc   */
} gb_status;

/* Rank-buffer element types (gpubridge README: float16, bfloat16, float32,
 * float64, int8, uint8, int32, int64; bool is excluded).  float32 and
 * bfloat16 SUM / AVG take the codec path; everything else (MAX / MIN, and
 * the other dtypes) takes the exact path: no compression, float16 /
 * bfloat16 fold in float32 and round once, float64 folds in float64,
 * integer SUM wraps modulo 2^bits. */
typedef enum {
    GB_F32 = 0,
    GB_BF16 = 1,
    GB_F16 = 2,
    GB_F64 = 3,
    GB_I8 = 4,
    GB_U8 = 5,
    GB_I32 = 6,
    GB_I64 = 7
} gb_dtype;

/* gpubridge README, API table, all_reduce row: SUM; AVG = the SUM divided
 * by the world size, identically on every rank (floating dtypes only,
 * GB_ERR_UNSUPPORTED_OP otherwise); MAX and MIN (among equal values, +0 and
 * -0, the lower rank's value is kept; NaN inputs are outside the contract).
 * PRODUCT is not supported.  Compression applies to float32 / bfloat16 SUM
 * and AVG only: MAX / MIN and integer dtypes stay exact whatever the codec
 * argument (the README's rule), and float16 / float64 SUM / AVG accept
 * GB_CODEC_NONE only (GB_ERR_UNSUPPORTED_CODEC otherwise). */
typedef enum { GB_SUM = 0, GB_AVG = 1, GB_MAX = 2, GB_MIN = 3 } gb_op;

/* gpubridge README, "Bridge compression".
 *   GB_CODEC_NONE: the payload is the float32 island sum (4n bytes).
 *   GB_CODEC_BF16: bf16 of the island sum, rounded to nearest even (2n bytes).
 *   GB_CODEC_E4M3 / GB_CODEC_E5M2: OCP 8-bit floats with one power-of-two
 *     float32 scale per `block` elements (block 128 or 256; blocks start at
 *     element 0, the last may be short).  For a block with largest magnitude
 *     m, the scale is 2^k, k the smallest integer with m * 2^-k <= the
 *     format's largest finite value (448 / 57344), clamped to k >= -126; k = 0
 *     for an all-zero block.  code = round-to-nearest-even(x * 2^-k) with
 *     saturation; decoded value = code value * 2^k (exact).
 * Compression applies only where there is a bridge (two or more islands);
 * with one island the codec argument is ignored (gpubridge README: a
 * single-vendor job has no bridge), and broadcast / all_gather never
 * compress. */
typedef enum {
    GB_CODEC_NONE = 0,
    GB_CODEC_BF16 = 1,
    GB_CODEC_E4M3 = 2,
    GB_CODEC_E5M2 = 3
} gb_codec;

#define GB_MAX_RANKS 64
#define GB_MAX_ISLANDS 8

typedef struct gb_ctx gb_ctx;

/* ---------------------------------------------------------------- context */

/* Create a context for W = sum(island_sizes[0..n_islands)) simulated ranks in
 * n_islands contiguous islands (1 <= n_islands <= GB_MAX_ISLANDS, every size
 * >= 1, W <= GB_MAX_RANKS).  Makes no CUDA call: the device is the current
 * CUDA device at the first call that enqueues work, and stays bound.
 * Errors: GB_ERR_INVALID_ARG (nothing allocated, *out untouched),
 * GB_ERR_ALLOC (host memory). */
gb_status gb_create(gb_ctx **out, int n_islands, const int *island_sizes);

/* Wait for the context's outstanding work, free its pinned and device
 * staging, free the context.  NULL is a no-op. */
gb_status gb_destroy(gb_ctx *ctx);

/* Topology queries (gpubridge README, Topology: islands, ranks, leaders).
 * Return -1 for a NULL context or an index out of range. */
int gb_world_size(const gb_ctx *ctx);
int gb_n_islands(const gb_ctx *ctx);
int gb_island_size(const gb_ctx *ctx, int island);
int gb_island_first_rank(const gb_ctx *ctx, int island); /* = the island's leader */
int gb_island_of_rank(const gb_ctx *ctx, int rank);

/* Grow the context's staging so that the single-buffer collectives
 * (gb_all_reduce, gb_all_reduce_ef, gb_reduce_scatter, gb_all_gather,
 * gb_broadcast) on up to n elements of `dtype` with `codec` / `block`, under
 * the policy set when it is called, need no further allocation.  The
 * bucket-set calls and gb_all_reduce_host may still grow it.  Enqueues
 * nothing. */
gb_status gb_reserve(gb_ctx *ctx, size_t n, gb_dtype dtype, gb_codec codec, int block);

/* Collective policy of gb_all_reduce and gb_all_reduce_host when there are
 * two or more islands (gpubridge README, policy table):
 *   chunk_bytes == 0: reduce-bridge-broadcast, one bridge hop for the whole
 *     buffer on the caller's stream;
 *   chunk_bytes > 0 (default 2 MiB, measured best on GB300 for 25 MiB
 *     buckets; the README's policy defaults to 4M): pipelined-
 *     reduce-bridge-broadcast.  The leaders' bridge step is cut into the
 *     fewest chunks of at most about S bytes of one island's payload P,
 *     of equal size (whole 256-element tiles, at least one tile, at most 32
 *     chunks per call), where for gb_all_reduce and gb_all_reduce_ef
 *     S = chunk_bytes while P <= 3 * chunk_bytes and
 *     S = chunk_bytes * sqrt(P / (3 * chunk_bytes)) above (the fill and
 *     drain of the pipeline grow with the chunk, the copies' fixed costs
 *     with the chunk count); chunk c's device ->
 *     host copy, chunk c-1's host -> device copy and the kernels of other
 *     chunks overlap on the context's two copy streams, ordered with CUDA
 *     events.  Chunks are whole codec blocks, so the result is the same
 *     bits.
 *   use_graphs != 0 (default): a pipelined call is captured into a CUDA
 *     graph the second time the same buffers and shape are seen, and
 *     replayed from then on (one launch instead of a few dozen).
 * reduce_scatter follows the same policy with chunks of at most
 * max(chunk_bytes / 2, S - chunk_bytes / 2) (its chunks' decodes write only
 * the parts of the slices they cover, so its drain is shorter).
 * all_gather with chunk_bytes > 0 moves groups of whole rank blocks of
 * about chunk_bytes: one group's host -> device copies overlap the next
 * group's device -> host copies.  broadcast with chunk_bytes > 0 moves the
 * source the same way in equal pieces of up to 4 x chunk_bytes (at most 64
 * pieces; one hop up to that size).  Waits for the context's outstanding
 * work. */
gb_status gb_set_pipeline(gb_ctx *ctx, size_t chunk_bytes, int use_graphs);

/* The sharded-bridge policy of gb_all_reduce and gb_all_reduce_ef (gpubridge
 * README, policy table, sharded-bridge row), on (on != 0) or off (default).
 * k = the size of the smallest island.  Each island's sum is cut into k
 * segments of ceil(n / k) elements rounded up to whole 256-element tiles
 * (whole codec blocks; trailing segments may be short or absent); rank j of
 * every island encodes segment j of its island sum, all_reduces it with the
 * other islands over its own bridge link (a pinned host slot and a pair of
 * copy streams; segment j uses link j mod 8), and every island gathers the
 * segments into all its ranks.  The result is the same bits as
 * reduce-bridge-broadcast.  With one island, or an island of one rank
 * (k == 1), the call falls back to the gb_set_pipeline policy.  use_graphs of
 * gb_set_pipeline applies.  gb_all_reduce_host, gb_reduce_scatter and, while
 * this policy is on, gb_all_reduce_buckets bucket by bucket keep one link.
 * Waits for the context's outstanding work. */
gb_status gb_set_sharded_bridge(gb_ctx *ctx, int on);

/* gb_context_status: the context's sticky status (GB_OK until a call fails
 * after enqueueing; then that failure, for good).  gb_last_error: the status
 * of the most recent call on this context that failed, sticky or not (an
 * argument error included), GB_OK if none has; a later successful call does
 * not clear it; calls refused by a failed context set it to
 * GB_ERR_CONTEXT_FAILED.  gb_last_error_message: a one-line description of
 * the last error (for a failed context, of the failure that caused it).
 * With a NULL context the first two return GB_ERR_INVALID_ARG. */
gb_status gb_context_status(const gb_ctx *ctx);
gb_status gb_last_error(const gb_ctx *ctx);
const char *gb_last_error_message(const gb_ctx *ctx);
const char *gb_status_string(gb_status status);

/* --------------------------------------------------------------- payloads */

/* Bytes of one island's bridge payload for n elements.  Layout: codes first
 * (n float32 for none, n bf16 for bf16, n bytes for fp8), then for fp8 the
 * ceil(n / block) float32 scales, starting at gb_payload_scales_offset (the
 * code bytes rounded up to 16).  Returns 0 for an unknown codec or block. */
size_t gb_payload_bytes(gb_codec codec, int block, size_t n);
size_t gb_payload_scales_offset(gb_codec codec, int block, size_t n);

/* -------------------------------------------------- phase-level building
 * blocks (gpubridge README, observer phases: island-reduce, compress,
 * bridge, decompress, island-broadcast).  Composing them as
 *   island_reduce -> bridge_compress -> (caller moves payloads) ->
 *   bridge_decompress_accumulate (island 0 with accumulate = 0, then islands
 *   1..I-1 with accumulate = 1) -> island_broadcast
 * gives bit for bit what gb_all_reduce gives. */

/* island_sum[j] = ((x_0[j] + x_1[j]) + ...) + x_{K-1}[j] in float32, over the
 * K = gb_island_size(ctx, island) buffers of `rank_bufs` (that island's
 * ranks, in rank order, 16-byte aligned).  island_sum: n float32, device,
 * 32-byte aligned, must not overlap the inputs. */
gb_status gb_island_reduce(gb_ctx *ctx, int island, const void *const *rank_bufs, size_t n,
                           gb_dtype dtype, float *island_sum, gb_stream stream);

/* Encode n float32 values (device) into `payload` (device, 32-byte aligned,
 * gb_payload_bytes(codec, block, n) bytes, laid out as described above).
 * block is ignored for none / bf16.  The phase-level calls cover the codec
 * path: float32 / bfloat16 rank buffers, SUM / AVG. */
gb_status gb_bridge_compress(gb_ctx *ctx, const float *island_sum, size_t n, gb_codec codec,
                             int block, void *payload, gb_stream stream);

/* accum[j] = dec(payload)[j] (accumulate == 0) or accum[j] + dec(payload)[j]
 * (accumulate != 0), float32, round to nearest even.  accum: n float32,
 * device, 32-byte aligned. */
gb_status gb_bridge_decompress_accumulate(gb_ctx *ctx, const void *payload, size_t n,
                                          gb_codec codec, int block, float *accum, int accumulate,
                                          gb_stream stream);

/* Write total[j] (SUM) or total[j] / W (AVG, float32 division), rounded to
 * `dtype` (nearest even for bf16), into the K = gb_island_size(ctx, island)
 * buffers of `rank_bufs`. */
gb_status gb_island_broadcast(gb_ctx *ctx, int island, const float *total, size_t n, gb_op op,
                              void *const *rank_bufs, gb_dtype dtype, gb_stream stream);

/* The two fused halves of reduce-bridge-broadcast, for a caller that moves
 * the payloads over a bridge of its own (gpubridge README, "all_reduce uses
 * reduce-bridge-broadcast": island reduce, the leaders' bridge step, island
 * broadcast; "Bridge compression": leaders compress before the bridge and
 * decompress after it).
 *
 * gb_island_reduce_compress: for every island i, payloads[i] receives the
 * encoding of s_i, the float32 sum of the island's ranks in ascending order,
 * with `codec` and `block`, in the layout of gb_payload_bytes (codes, then
 * the fp8 scales at gb_payload_scales_offset).  The codec is applied as
 * given, with one island too (gb_all_reduce skips it there: no bridge).
 * rank_bufs: W device buffers of n elements, 16-byte aligned, read only.
 * payloads: I device buffers of gb_payload_bytes(codec, block, n) bytes,
 * 32-byte aligned, owned by the caller.  dtype F32 or BF16.  One kernel
 * launch for all islands, stream-ordered on `stream`.
 *
 * gb_decompress_island_broadcast: payloads holds I * I device pointers,
 * row g being what leader g holds after the bridge: payloads[g * I + j] is
 * island j's payload (its own for j == g), and the same pointer may appear
 * in several rows.  Every rank of island g receives
 * t = dec(payloads[g * I + 0]) + ... + dec(payloads[g * I + I - 1]) in
 * float32, island order, divided by W for AVG (float32 division), rounded to
 * dtype (nearest even for bf16).  With the payloads of
 * gb_island_reduce_compress, carried bit for bit, this is what gb_all_reduce
 * writes.  op SUM or AVG.  One kernel launch.
 *
 * Errors as for gb_all_reduce; n == 0 is a no-op.  Neither call allocates. */
gb_status gb_island_reduce_compress(gb_ctx *ctx, const void *const *rank_bufs, size_t n, gb_dtype dtype,
                                    gb_codec codec, int block, void *const *payloads, gb_stream stream);
/* gb_island_reduce_compress with error feedback: island i encodes
 * s_i + residuals[i] and sets residuals[i] = (s_i + residuals[i]) -
 * dec(payload_i), as gb_all_reduce_ef does (float32, n elements per island,
 * device, 32-byte aligned, owned by the caller). */
gb_status gb_island_reduce_compress_ef(gb_ctx *ctx, const void *const *rank_bufs, float *const *residuals, size_t n,
                                       gb_dtype dtype, gb_codec codec, int block, void *const *payloads,
                                       gb_stream stream);
/* The second half, decode + accumulate + broadcast (described with
 * gb_island_reduce_compress above).  It also takes the exact path's
 * payloads (the dtypes and ops of gb_island_reduce_compress_op; codec as
 * for gb_all_reduce): every rank of island g receives the fold of
 * payloads[g * I + 0 .. I - 1] in island order (AVG divided by W), rounded
 * to dtype. */
gb_status gb_decompress_island_broadcast(gb_ctx *ctx, const void *const *payloads, size_t n, gb_dtype dtype,
                                         gb_op op, gb_codec codec, int block, void *const *rank_bufs,
                                         gb_stream stream);

/* The fused halves for every dtype and op gb_all_reduce takes (gpubridge
 * README, API table, all_reduce row and the supported dtypes; "Bridge
 * compression": MAX / MIN and integer dtypes stay exact).
 *
 * gb_island_payload_bytes: bytes of one island's payload for n elements --
 * gb_payload_bytes(codec, block, n) on the codec path (float32 / bfloat16
 * SUM / AVG); otherwise the exact path's island fold: n elements of the
 * dtype, or n float32 sums for float16 / bfloat16 SUM / AVG.  0 for a
 * combination gb_all_reduce refuses.
 *
 * gb_island_reduce_compress_op: gb_island_reduce_compress with an op.  On
 * the codec path it is that call; otherwise payloads[i] receives the fold
 * of island i's ranks in ascending rank order (MAX / MIN: among equal values
 * the lower rank's is kept; integer SUM wraps; float16 / bfloat16 sums in
 * float32, float64 in float64), the codec ignored (float16 / float64 SUM /
 * AVG take GB_CODEC_NONE only).  payloads: I device buffers of
 * gb_island_payload_bytes bytes, 32-byte aligned.  One kernel launch.
 *
 * gb_decompress_scatter: reduce_scatter's second half (API table,
 * reduce_scatter_tensor row): out[r] (n / W elements, device, 16-byte
 * aligned, not overlapping the payloads) receives elements
 * [r * n / W, (r + 1) * n / W) of what gb_decompress_island_broadcast would
 * write into every rank from the same payloads (payloads: I * I pointers as
 * there).  n must be a multiple of W.  One kernel launch.
 *
 * Errors as for gb_all_reduce / gb_reduce_scatter; n == 0 is a no-op.
 * Neither call allocates. */
size_t gb_island_payload_bytes(gb_dtype dtype, gb_op op, gb_codec codec, int block, size_t n);
gb_status gb_island_reduce_compress_op(gb_ctx *ctx, const void *const *rank_bufs, size_t n, gb_dtype dtype,
                                       gb_op op, gb_codec codec, int block, void *const *payloads,
                                       gb_stream stream);
gb_status gb_decompress_scatter(gb_ctx *ctx, const void *const *payloads, size_t n, gb_dtype dtype, gb_op op,
                                gb_codec codec, int block, void *const *out, gb_stream stream);

/* ------------------------------------------------------------ collectives */

/* In-place all_reduce of W rank buffers of n elements (gpubridge README, API
 * table, all_reduce row, and "all_reduce uses reduce-bridge-broadcast").
 * Every rank buffer ends with the same bits. */
gb_status gb_all_reduce(gb_ctx *ctx, void *const *rank_bufs, size_t n, gb_dtype dtype, gb_op op,
                        gb_codec codec, int block, gb_stream stream);

/* gb_all_reduce with error feedback (gpubridge README, "Bridge
 * compression": each bridge member keeps an error-feedback residual per
 * buffer, so rounding error carries into the next step instead of
 * accumulating).  residuals: I device float32 arrays of n elements, one per
 * island, owned by the caller, zero before the first call and kept (with
 * the rank buffers' shape) from call to call of the same gradient buffer.
 * Each leader encodes s_i + r_i and sets r_i = (s_i + r_i) - dec(payload_i)
 * (float32); the rest is gb_all_reduce.  With one island there is no bridge
 * and the residuals are left unchanged.  Saving and restoring the residual
 * arrays checkpoints and resumes the feedback state.  float32 / bfloat16
 * SUM / AVG only (the exact path has nothing to feed back):
 * GB_ERR_UNSUPPORTED_OP otherwise. */
gb_status gb_all_reduce_ef(gb_ctx *ctx, void *const *rank_bufs, float *const *residuals, size_t n,
                           gb_dtype dtype, gb_op op, gb_codec codec, int block, gb_stream stream);

/* reduce_scatter (API table, reduce_scatter_tensor row): out_r (n_in / W
 * elements) receives elements [r * n_in / W, (r + 1) * n_in / W) of what
 * gb_all_reduce would compute on `in`; the island sums are encoded whole,
 * with the same codec blocks as gb_all_reduce.  n_in must be a multiple of W.
 * `in` is not modified; out buffers must not overlap the inputs. */
gb_status gb_reduce_scatter(gb_ctx *ctx, const void *const *in, void *const *out, size_t n_in,
                            gb_dtype dtype, gb_op op, gb_codec codec, int block,
                            gb_stream stream);

/* all_gather (API table, all_gather_into_tensor row): out_r (W * n_in
 * elements) = in_0 | in_1 | ... | in_{W-1}, exact, for every r.  Data from
 * another island crosses the bridge (pinned host slots) uncompressed. */
gb_status gb_all_gather(gb_ctx *ctx, const void *const *in, void *const *out, size_t n_in,
                        gb_dtype dtype, gb_stream stream);

/* broadcast (API table, broadcast row; three hops: src -> its island, its
 * leader -> the other leaders over the bridge, each leader -> its island):
 * every rank buffer receives rank src's n elements, exact, in place. */
gb_status gb_broadcast(gb_ctx *ctx, void *const *rank_bufs, size_t n, gb_dtype dtype, int src,
                       gb_stream stream);

/* gb_all_reduce for W HOST buffers (pinned, for asynchronous copies): the
 * buffers are staged onto the GPU in context-owned device buffers, reduced
 * there and copied back (gpubridge README, torch.distributed backend, CPU
 * tensors: staged onto the rank's GPU, carried by the same topology and
 * copied back).  Under the pipelined policy (no phase marks kept) the
 * staging, the bridge hop and the copy-back run chunk by chunk (every chunk
 * carries the rank buffers in and out, so a chunk is the elements whose W
 * rank slices total 8 x chunk_bytes, whole 256-element tiles, at most 32
 * chunks) on the context's copy streams so that both directions of the
 * host link stay busy, replayed as a CUDA graph from the second call with
 * the same buffers; otherwise staging, all_reduce and copy-back run in
 * sequence.  Host buffers need no alignment; they must not be touched until
 * `stream` has completed the call. */
gb_status gb_all_reduce_host(gb_ctx *ctx, void *const *host_bufs, size_t n, gb_dtype dtype,
                             gb_op op, gb_codec codec, int block, gb_stream stream);

/* gb_all_reduce_host for W host rank buffers that are the rows of ONE host
 * allocation: rank r's n elements start at host + r * pitch bytes, as in a
 * pinned [W, n] tensor (pitch >= n * element bytes when W > 1; ignored when
 * W == 1).  Same semantics, ordering and results as gb_all_reduce_host.
 * The staging and the copy-back move every rank's chunk with one 2D copy
 * (cudaMemcpy2DAsync) per chunk and direction instead of W copies, each of
 * which costs a few microseconds of fixed time on its copy stream.  The rows
 * must lie in one allocation: the CUDA runtime refuses a 2D copy across
 * separate ones (even at equal spacing), which fails the call and the
 * context with GB_ERR_CUDA.  A pitch beyond the device's 2D copy limit
 * (cudaDevAttrMaxPitch) is staged row by row instead.  Errors as
 * gb_all_reduce_host, plus GB_ERR_INVALID_ARG for a NULL host, pitch
 * < n * element bytes (rows that would overlap) or rows past the end of the
 * address space. */
gb_status gb_all_reduce_host_rows(gb_ctx *ctx, void *host, size_t pitch, size_t n, gb_dtype dtype,
                                  gb_op op, gb_codec codec, int block, gb_stream stream);

/* ------------------------------------------------------ gradient buckets */

/* Greedy bucket plan (gpubridge README, DDP comm hook: one all_reduce per
 * DDP gradient bucket): walk n_tensors tensors of numel[t] elements of
 * elem_bytes in the given order; append each to the open bucket unless the
 * bucket already holds elements and the tensor would take it past cap_bytes,
 * in which case a new bucket opens (a tensor larger than the cap sits
 * alone).  Tensors are packed without gaps: tensor t is elements
 * [offset[t], offset[t] + numel[t]) of bucket bucket_of[t].  Each bucket's
 * element count is rounded up to a multiple of pad_elems (0 or 1: none).
 * Host-only; makes no CUDA call.  GB_ERR_INVALID_ARG if more than
 * max_buckets would be needed. */
gb_status gb_bucket_plan(const size_t *numel, int n_tensors, size_t elem_bytes, size_t cap_bytes,
                         size_t pad_elems, int *bucket_of, size_t *offset, size_t *bucket_numel,
                         int max_buckets, int *n_buckets);

/* All_reduce of every bucket, in bucket order: each bucket gets the bits
 * gb_all_reduce would give it.  bucket_bufs holds n_buckets * W device
 * pointers, bucket-major (bucket b, rank r at [b * W + r]); bucket b has
 * bucket_numel[b] elements.  The tensors of the plan are views into these
 * flat buffers, so nothing is copied in or out.  Under the pipelined policy
 * (two or more islands, no phase marks kept) the buckets run as one
 * pipeline of chunks (each bucket cut evenly into chunks of at most
 * 6 x chunk_bytes of payload: the pipeline fills once per set, so larger
 * copies pay) on a three-slot staging ring, the bridge of one bucket
 * overlapping the kernels of the next, captured as one
 * CUDA graph for the whole set from the second call with the same buffers
 * (one launch per gradient sync); otherwise one gb_all_reduce per bucket.
 * Empty buckets are allowed (nothing to do; their pointers may be NULL). */
gb_status gb_all_reduce_buckets(gb_ctx *ctx, int n_buckets, void *const *bucket_bufs,
                                const size_t *bucket_numel, gb_dtype dtype, gb_op op,
                                gb_codec codec, int block, gb_stream stream);

/* gb_all_reduce_buckets with error feedback (as gb_all_reduce_ef, per
 * bucket): residuals holds n_buckets * I device float32 arrays, bucket-major
 * (bucket b, island i at [b * I + i]), of bucket_numel[b] elements each,
 * owned by the caller, zero before the first call and kept from step to
 * step.  float32 / bfloat16 SUM / AVG only.  Same policy, pipeline and graph
 * as gb_all_reduce_buckets; with one island the residuals are unchanged. */
gb_status gb_all_reduce_buckets_ef(gb_ctx *ctx, int n_buckets, void *const *bucket_bufs, float *const *residuals,
                                   const size_t *bucket_numel, gb_dtype dtype, gb_op op, gb_codec codec, int block,
                                   gb_stream stream);

/* reduce_scatter of every bucket (the gradient sets of a sharded data
 * parallel step): out_bufs[b * W + r] receives slice r (bucket_numel[b] / W
 * elements) of what gb_all_reduce would compute on bucket b's inputs
 * in_bufs[b * W + 0 .. W - 1] (in bucket order; the island sums are encoded
 * whole, with the all_reduce codec blocks).  bucket_numel[b] must be a
 * multiple of W; inputs are not modified; outputs must not overlap inputs.
 * Under the pipelined policy (two or more islands, no phase marks kept)
 * the buckets run as one pipeline of chunks, as in gb_all_reduce_buckets,
 * captured as one CUDA graph per set from the
 * second call with the same buffers; otherwise one gb_reduce_scatter per
 * bucket.  Empty buckets are allowed (their pointers may be NULL). */
gb_status gb_reduce_scatter_buckets(gb_ctx *ctx, int n_buckets, const void *const *in_bufs, void *const *out_bufs,
                                    const size_t *bucket_numel, gb_dtype dtype, gb_op op, gb_codec codec,
                                    int block, gb_stream stream);

/* all_gather of every bucket, exact: out_bufs[b * W + r] (W *
 * bucket_numel_in[b] elements) receives in_bufs[b * W + 0], ...,
 * in_bufs[b * W + W - 1] concatenated, for every r.  Under the pipelined
 * policy (two or more islands, no phase marks kept) the buckets run as one
 * pipeline: a copy kernel on the context's gather stream gathers each
 * island's blocks of a bucket into its leader's output, from where they
 * cross the bridge in groups of whole islands (of up to 6 x chunk_bytes)
 * through two alternating host slots, one copy per group and direction;
 * the kernels that spread each leader's blocks to its island overlap the
 * next buckets' copies; captured as one CUDA graph per
 * set from the second call with the same buffers.  Otherwise one
 * gb_all_gather per bucket.  Empty buckets are allowed (pointers may be
 * NULL).  Inputs must not overlap outputs. */
gb_status gb_all_gather_buckets(gb_ctx *ctx, int n_buckets, const void *const *in_bufs, void *const *out_bufs,
                                const size_t *bucket_numel_in, gb_dtype dtype, gb_stream stream);

/* --------------------------------------------------------- phase timing */

/* gpubridge README, "Observing collectives": timing marks per phase, taken
 * with CUDA events on GPUs, never synchronising the call.  With capacity > 0
 * every collective records CUDA events around its phases and the marks of
 * the last `capacity` collectives are kept; 0 turns the marks off.  Changing
 * the capacity waits for the context's outstanding work.  Phases:
 *   0: the island reduce + compress kernels (their launches run back to
 *      back on the caller's stream; the window covers all of them),
 *   1: the bridge hop, from the first device -> host copy's start to the
 *      last host -> device copy's end (0 without a bridge),
 *   2: the decompress + broadcast kernels (all_reduce / reduce_scatter) or
 *      the copy kernels (all_gather / broadcast), the sum of their own
 *      durations.
 * With the pipelined policy the phases overlap in time. */
#define GB_N_PHASES 3
gb_status gb_set_phase_timing(gb_ctx *ctx, int capacity);

/* Milliseconds of each phase of the collective `age` calls back (0 = the
 * most recent one that recorded marks); waits for its events.  A phase that
 * collective did not have reads 0.  GB_ERR_INVALID_ARG if no such record. */
gb_status gb_phase_times(gb_ctx *ctx, int age, float *ms /* [GB_N_PHASES] */);
gb_status gb_last_phase_times(gb_ctx *ctx, float *ms /* [GB_N_PHASES] */);

/* ------------------------------------------------------------ test hooks */

/* Fault injection for tests, all on the host, none touching the GPU:
 *   GB_INJECT_BRIDGE: the next bridge hop fails before it enqueues its
 *     copies (the call returns GB_ERR_BRIDGE, no rank buffer is written,
 *     the context becomes failed);
 *   GB_INJECT_ALLOC: the next staging allocation fails (GB_ERR_ALLOC, the
 *     context becomes failed);
 *   GB_INJECT_OTHER_DEVICE: the next call of a context already bound to a
 *     device sees a current device other than that one, as a caller that
 *     switched devices would (GB_ERR_INVALID_ARG with nothing enqueued; not
 *     sticky).  Without a bound device it has no effect and is dropped. */
#define GB_INJECT_BRIDGE 1
#define GB_INJECT_ALLOC 2
#define GB_INJECT_OTHER_DEVICE 3
gb_status gb_debug_inject(gb_ctx *ctx, int what);

/* ------------------------------------------- all_reduce without allocation
 * No counterpart on the gpubridge page: an addition of this library.
 *
 * For callers that cannot allocate memory at the point where they sync
 * gradients: for example a hook running inside a training step whose
 * framework has already reserved almost all device memory in its own caching
 * allocator (a cudaMalloc there can fail, and freeing staging to grow it
 * waits for the whole device), or a process that must not pin more host
 * memory.  gb_all_reduce grows context-owned device and pinned host staging
 * on demand; gb_all_reduce_noalloc computes the same bits without any
 * allocation:
 *   - its payload staging is one fixed device array of
 *     GB_NOALLOC_DEVICE_BYTES, defined in the library, which every GPU that
 *     loads the library holds until the process exits;
 *   - its bridge slots are one fixed host array of GB_NOALLOC_HOST_BYTES in
 *     ordinary pageable memory, so the device -> host copy blocks the
 *     calling thread until the first kernel and the copy have finished.
 * Limits: with I islands and P = gb_payload_bytes(codec, block, n) (the
 * float32 sum, 4n, when I == 1), I * I * round_up(P, 256) must fit the
 * device array; larger calls return GB_ERR_TOO_LARGE with nothing enqueued.
 * (The host array holds I * round_up(P, 256), which that bound already keeps
 * within GB_NOALLOC_HOST_BYTES for every I >= 2.)  It covers the codec path
 * only (float32 / bfloat16 rank buffers, SUM / AVG); the other arguments are
 * checked as in gb_all_reduce, the device included: a context already bound
 * to a device (by an earlier call of another entry point) refuses a call
 * made with another device current (GB_ERR_INVALID_ARG), and an unbound
 * context takes the current device without being bound by this call.
 * Sharing: every call in the process uses the same two arrays, which keep
 * the last call's contents; nothing in them needs to start at zero (each
 * call reads only what it wrote).  Calls that overlap on the GPU -- from
 * several host threads, or on several streams without ordering between
 * them -- race on the arrays; order them.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.
 * The context supplies only the island layout: this call neither uses the
 * context's staging nor marks it failed; a failed context is refused. */
#define GB_NOALLOC_DEVICE_BYTES (64u << 20)
#define GB_NOALLOC_HOST_BYTES (32u << 20)
gb_status gb_all_reduce_noalloc(gb_ctx *ctx, void *const *rank_bufs, size_t n, gb_dtype dtype,
                                gb_op op, gb_codec codec, int block, gb_stream stream);

/* Number of kernels this library has launched in this process. */
uint64_t gb_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GB_H */
