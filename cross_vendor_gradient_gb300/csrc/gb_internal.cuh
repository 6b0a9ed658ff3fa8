// Internal declarations of libgb's host runtime, shared by gb_runtime.cu
// (validation, staging, the pipelines) and gb_api.cu (the C entry points).
// Not installed; the public contract is include/gb.h.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <new>
#include <vector>

#include <cuda_runtime.h>

#include "gb.h"
#include "gb_device.cuh"
#include "gb_kernels.cuh"

namespace gbrt {
constexpr int kMaxChunks = 32;
// timing marks of one collective: 0 start, 1 end of island reduce + encode,
// 2 bridge start, 3 bridge end, then decode start / end per chunk
constexpr int kMarks = 4 + 2 * kMaxChunks;
constexpr int kMaxGraphs = 16;
// sharded-bridge: copy stream pairs ("bridge links"); segment j uses link j % kMaxLinks
constexpr int kMaxLinks = 8;
constexpr double kChunkGrowRef = 3.0;    // single-buffer all_reduce: the chunk grows beyond 3 chunks of payload
constexpr size_t kBucketChunkScale = 6;  // gb_all_reduce_buckets: chunk = 6 x the pipeline chunk
constexpr int kBucketSlots = 3;          // gb_all_reduce_buckets: staging ring slots (chunks in flight)
constexpr size_t kHostStageScale = 8;    // gb_all_reduce_host: a chunk stages 8 x the pipeline chunk of rank data
constexpr size_t kRsChunkDiv = 2;        // gb_reduce_scatter: chunk = the all_reduce chunk - the pipeline chunk / 2, >= chunk / 2
constexpr size_t kBcastPieceScale = 4;   // gb_broadcast: pieces of up to 4 x the pipeline chunk
constexpr uint64_t kMaxElems = 1ull << 38;
}  // namespace gbrt

// Identity of a captured all_reduce (every value its graph bakes in).
struct GraphKey {
    const void *in[GB_MAX_RANKS];
    const void *host[GB_MAX_RANKS];  // gb_all_reduce_host: the host rank buffers
    const void *res[GB_MAX_ISLANDS];
    uint64_t n, chunk;
    uint64_t host_pitch;  // gb_all_reduce_host_rows: 2D staging copies at this host pitch
    int dtype, op, codec, block, timed, links;
    const void *d_stage, *h_stage;
};

struct GraphEntry {
    GraphKey key;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;  // null: seen once, not captured yet
    cudaGraphNode_t mark_node[gbrt::kMarks] = {};
    int n_marks = 0;
    uint64_t last_use = 0;
};

struct gb_ctx {
    int I = 0, W = 0;
    int size[GB_MAX_ISLANDS] = {};
    int first[GB_MAX_ISLANDS + 1] = {};
    int island_of[GB_MAX_RANKS] = {};
    int device = -1;
    gb_status sticky = GB_OK;
    gb_status last = GB_OK;  // the most recent failed call's status, sticky or not
    char msg[256] = {};
    int inject = 0;
    // device staging, chunk-major: C x I own-payload parts, then I leaders x
    // C x I received parts
    unsigned char *d_stage = nullptr;
    size_t d_stage_bytes = 0;
    // pinned host staging: the bridge slots, C x I parts
    unsigned char *h_stage = nullptr;
    size_t h_stage_bytes = 0;
    // device copies of host rank buffers (gb_all_reduce_host)
    unsigned char *d_ranks = nullptr;
    size_t d_ranks_bytes = 0;
    size_t max_pitch = 0;  // cudaDevAttrMaxPitch of the bound device (2D copies)
    // ordering of staging reuse across calls
    cudaEvent_t done = nullptr;
    bool done_recorded = false;
    cudaStream_t last_stream = nullptr;
    // pipelined-reduce-bridge-broadcast: chunk size, copy streams, events
    size_t chunk_bytes = 2u << 20;
    int use_graphs = 1;
    cudaStream_t sd = nullptr, sh = nullptr, scap = nullptr;
    cudaStream_t sg = nullptr;  // gb_all_gather_buckets: the gather kernels, ahead of the copies
    cudaEvent_t ev_k1[gbrt::kMaxChunks] = {}, ev_d2h[gbrt::kMaxChunks] = {}, ev_h2d[gbrt::kMaxChunks] = {};
    cudaEvent_t ev_in[gbrt::kMaxChunks] = {}, ev_k2[gbrt::kMaxChunks] = {};  // host-buffer pipeline
    cudaEvent_t ev_join_d = nullptr, ev_join_h = nullptr;
    cudaEvent_t ev_ag[GB_MAX_RANKS] = {};  // all_gather: one per group of rank blocks
    // sharded-bridge policy: links 1 .. gbrt::kMaxLinks - 1 (link 0 is sd / sh),
    // created on first use, with their join events
    int sharded = 0;
    cudaStream_t lsd[gbrt::kMaxLinks] = {}, lsh[gbrt::kMaxLinks] = {};
    cudaEvent_t ev_ljd[gbrt::kMaxLinks] = {}, ev_ljh[gbrt::kMaxLinks] = {};
    cudaEvent_t cap_mark[gbrt::kMarks] = {};  // stand-ins recorded while capturing
    GraphEntry graphs[gbrt::kMaxGraphs];
    int n_graphs = 0;
    uint64_t clock = 0;
    // gb_all_reduce_buckets: whole gradient sets captured as one graph each
    struct BucketGraph {
        std::vector<uint64_t> key;
        cudaGraph_t graph = nullptr;
        cudaGraphExec_t exec = nullptr;  // null: seen once
        uint64_t last_use = 0;
        int kernels = 0;
    };
    std::vector<BucketGraph> bucket_graphs;
    // phase timing (observer marks): a ring of `tcap` records of gbrt::kMarks events
    int tcap = 0;
    cudaEvent_t *tev = nullptr;
    int *tnk2 = nullptr;
    unsigned char *tbridge = nullptr;
    long long tcount = 0;  // collectives recorded so far
};

#define GB_TRY(expr)                         \
    do {                                     \
        gb_status _s = (expr);               \
        if (_s != GB_OK) return _s;          \
    } while (0)

namespace gbrt {

using gb::round_up;

// Timing marks.  mode 0: off; 1: record the ring slot's event (direct
// launches); 2: record the stand-in event as an event-record node of a graph
// being captured (re-pointed at the ring slot's event before each launch).
enum { kMarkOff = 0, kMarkDirect = 1, kMarkCapture = 2 };

// Shape of one reduce-bridge-broadcast: the element range is cut into C
// chunks of whole 256-element tiles (so whole codec blocks); every chunk's
// payload parts have a fixed stride `part`.  C == 1 is the plain policy.
// chunk_range gives chunk ch's first element and length.
struct Plan {
    int I = 0, W = 0;
    uint64_t n = 0;
    gb_dtype dtype = GB_F32;
    gb_op op = GB_SUM;
    int eff = GB_CODEC_NONE, blk = 256, rs = 0;
    size_t eb = 4, cb = 4;
    uint64_t chunk = 0;  // the longest chunk (the part stride holds it)
    int C = 1;
    uint64_t off[kMaxChunks + 1] = {};  // chunk ch is elements [off[ch], off[ch + 1])
    int links = 1;  // copy stream pairs the chunks' bridge copies are spread over
    size_t part = 0;
    size_t dev_bytes = 0, host_bytes = 0;
};

inline void chunk_range(const Plan &p, int ch, uint64_t *e0, uint64_t *m) {
    *e0 = p.off[ch];
    *m = p.off[ch + 1] - p.off[ch];
}

// One chunk of a bucket set's pipeline (enqueue_buckets): bucket b,
// elements [e0, e0 + m).
struct WorkChunk {
    int b;
    uint64_t e0, m;
};

gb_status set_msg(gb_ctx *c, gb_status s, const char *fmt, ...);
gb_status fail(gb_ctx *c, gb_status s, const char *what, cudaError_t e = cudaSuccess);
size_t elem_bytes(gb_dtype d);
bool is_float_dtype(int d);
bool is_exact(int dtype, int op);
bool aligned32(const void *p);
gb_status check_ctx(gb_ctx *c);
gb_status check_dtype(gb_ctx *c, int d);
gb_status check_codec_dtype(gb_ctx *c, int d);
gb_status check_op(gb_ctx *c, int op);
bool codec_ok(int codec, int block);
gb_status check_codec(gb_ctx *c, int codec, int block);
gb_status check_n(gb_ctx *c, size_t n);
gb_status check_dev_bufs(gb_ctx *c, const void *const *bufs, int count, const char *name);
gb_status check_rank_bufs(gb_ctx *c, const void *const *bufs, int count, const char *name);
gb_status check_dev_ptr(gb_ctx *c, const void *p, const char *name);
int seen_device(gb_ctx *c, int dev);
gb_status bind(gb_ctx *c);
gb_status begin(gb_ctx *c, cudaStream_t s);
gb_status end(gb_ctx *c, cudaStream_t s);
gb_status ring_event(gb_ctx *c, long long slot, int idx, cudaEvent_t *out);
gb_status mark(gb_ctx *c, int mode, int idx, cudaStream_t s);
void commit_marks(gb_ctx *c, int n_decode, bool bridge);
void free_marks(gb_ctx *c);
void drop_graphs(gb_ctx *c);
gb_status grow_device(gb_ctx *c, unsigned char **buf, size_t *have, size_t need);
gb_status grow_host(gb_ctx *c, size_t need);
size_t payload_bytes(int codec, int block, size_t n);
size_t scales_offset(int codec, size_t n);
bool is_fp8(int codec);
size_t part_bytes(const Plan &p, uint64_t m);
size_t chunk_stride(const Plan &p, uint64_t m);  // a chunk's part stride in its staging region
// balance: cut n into equal chunks of whole tiles (no short remainder);
// the bucket pipeline balances per bucket itself and passes false.
// chunk_elems > 0: chunks of that many elements (rounded down to whole tiles)
// instead of a payload size.
Plan make_plan(const gb_ctx *c, uint64_t n, gb_dtype dtype, gb_op op, gb_codec codec, int block, int rs,
               bool sharded_ok = false, size_t chunk_bytes = 0, bool balance = true, uint64_t chunk_elems = 0);
gb_status check_launch(gb_ctx *c, cudaError_t e, const char *what);
gb_status launch_encode(gb_ctx *c, const Plan &p, const gb::ReduceEncodeArgs &ra, cudaStream_t s);
gb_status launch_decode(gb_ctx *c, const Plan &p, const gb::DecodeBcastArgs &da, cudaStream_t s);
uint64_t vec_elems(const Plan &p);
gb_status copy_async(gb_ctx *c, void *dst, const void *src, size_t bytes, cudaMemcpyKind kind,
                     cudaStream_t s);
gb_status wait_on(gb_ctx *c, cudaStream_t s, cudaEvent_t ev);
gb_status record(gb_ctx *c, cudaEvent_t ev, cudaStream_t s);
gb_status enqueue_rbb(gb_ctx *c, const Plan &p, const void *const *in, void *const *out,
                      float *const *res, cudaStream_t s, int markmode, bool multi);
gb_status ensure_links(gb_ctx *c, int L);
// Rank staging of gb_all_reduce_host(_rows): `dev` is the context's rank
// copies at `dpitch` bytes apart; hpitch > 0 says that the host buffers are
// the rows of one host allocation, hpitch bytes apart: one 2D copy moves
// every rank's bytes [off, off + bytes).
gb_status stage_ranks(gb_ctx *c, void *const *host, void *const *dev, size_t dpitch, size_t hpitch, size_t off,
                      size_t bytes, cudaMemcpyKind kind, cudaStream_t s);
gb_status enqueue_host_pipeline(gb_ctx *c, const Plan &p, void *const *host, void *const *dev, size_t dpitch,
                                size_t hpitch, cudaStream_t s);
gb_status enqueue_buckets(gb_ctx *c, const Plan &p, const std::vector<WorkChunk> &work, const void *const *in,
                          void *const *out, const size_t *numel, int rs, float *const *res, cudaStream_t s);
gb_status run_set_graph(gb_ctx *c, const std::vector<uint64_t> &key, int kernels,
                        const std::function<gb_status(cudaStream_t)> &enqueue, cudaStream_t s);
gb_status run_buckets(gb_ctx *c, int nb, const void *const *in, void *const *out, const size_t *numel,
                      gb_dtype dtype, gb_op op, gb_codec codec, int block, int rs, float *const *res,
                      cudaStream_t s);
gb_status capture_rbb(gb_ctx *c, const Plan &p, const void *const *in, float *const *res, bool timed,
                      GraphEntry *ge);
GraphEntry *find_graph(gb_ctx *c, const GraphKey &k);
GraphEntry *new_graph_slot(gb_ctx *c);
gb_status enqueue_ag_buckets(gb_ctx *c, int nb, const void *const *in, void *const *out, const size_t *numel_in,
                             size_t eb, size_t slot_bytes, cudaStream_t s);
gb_status run_rbb(gb_ctx *c, const void *const *in, void *const *out, size_t n, gb_dtype dtype,
                  gb_op op, gb_codec codec, int block, cudaStream_t s, int rs, float *const *res = nullptr);
gb_status check_collective(gb_ctx *c, size_t n, int dtype, int op, int codec, int block);

}  // namespace gbrt
