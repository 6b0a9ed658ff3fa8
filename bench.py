"""Benchmark of the reduce-bridge-broadcast gradient all_reduce on one GB300.

Bucketed workloads (--workload c4, c5): a step is the all_reduce of a whole
GPT-2 small or 1.1B Llama-style bf16 gradient set in 25 MiB buckets through
gb_all_reduce_buckets; c5 adds reduce_scatter then all_gather of every bucket.

Default workload: 4 simulated ranks as 2 islands of 2, one 25 MiB float32
DDP bucket per rank (n = 6,553,600), values N(0, 1e-3) with 1% of them x100,
op AVG, bridge codec fp8 E4M3 with a power-of-two scale per 256 values.

A step is one gb_all_reduce of that bucket: fused island reduce + encode
kernel, bridge hop (device -> pinned host -> device copies), fused decode +
accumulate + broadcast kernel.  Before every timed step the rank buffers are
restored from a pristine device copy and L2 is flushed by writing a 512 MiB
buffer and then reading a separate 256 MiB one (so no dirty line is left to
be written back during the step); neither is inside the step's CUDA events.

Reported: algorithm GB/s (bytes of one rank buffer / step time, summed over
replicas), the dominant kernel's HBM roofline fraction from live CUDA event
durations (each kernel launched back to back over input sets cycled so that
none is in L2, in steady state; the per-kernel durations inside a step, with
a CUDA event around every phase, are reported beside it), the bridge hop
against measured pinned copy bandwidth, the same metric end to end through
gb_all_reduce_host with pinned host buffers, the oracle timed on the host
cores (``--impl reference`` times only the oracle), and, on one GPU, the
metric's curve: the 4 KiB .. 256 MiB payload sweep x codec as a compact
`sweep` object.  Multi-GPU: one independent replica per GPU (the path has no
exchange between GPUs), max time over ranks.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "all_reduce algorithm GB/s and % of GB300 HBM roofline vs payload size, per codec"
FLUSH_BYTES = 512 << 20
L2_BYTES = 129 << 20  # GB300 L2 (nominal 129 MB)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["gb", "reference"], default="gb")
    p.add_argument("--workload", default="c2")
    p.add_argument("--codec", default=None)
    p.add_argument("--block", type=int, default=None, help="fp8 scale block override (128 or 256)")
    p.add_argument("--dtype", default=None, help="rank dtype override (f32 bf16 f16 f64 i8 u8 i32 i64)")
    p.add_argument("--op", default=None, help="op override (sum avg max min)")
    p.add_argument("--n", type=int, default=None, help="override elements per rank")
    p.add_argument("--islands", default=None, help="override the island sizes, e.g. 4,4 (single-buffer workloads)")
    p.add_argument("--chunk-kib", type=int, default=None,
                   help="pipelined bridge chunk (KiB of one island's payload); 0 = one hop per call")
    p.add_argument("--no-graphs", action="store_true")
    p.add_argument("--sharded", action="store_true", help="sharded-bridge policy for the timed step")
    p.add_argument("--ef", action="store_true",
                   help="error feedback: the step is gb_all_reduce_ef (gb_all_reduce_buckets_ef for c4 / c5)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--roofline-only", action="store_true",
                   help="only the per-kernel timed regions (kernels inside one-hop steps, and back to "
                        "back); for profiling")
    p.add_argument("--sweep", action="store_true", help="payload sweep rows only (one JSON line each)")
    p.add_argument("--no-sweep", action="store_true",
                   help="leave the payload sweep out of the default bench line")
    p.add_argument("--collective", default="all_reduce",
                   choices=["all_reduce", "reduce_scatter", "all_gather", "broadcast"],
                   help="the collective one step runs (all_reduce: the default bench line)")
    return p.parse_args()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------ distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value, device=None):
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (read only)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "gb_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.6)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for nm, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------- CPU baseline

def cpu_baseline(w, xs, codec, budget_s=10.0):
    """The oracle as it stands, single-threaded, on full steps of the
    workload (repeated until the budget is spent, at least once)."""
    import oracle
    n = xs[0].size
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.all_reduce(xs, w.island_sizes, w.op, codec, w.block)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    per = el / reps
    return {"value": n * w.elem_bytes / per / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%d full steps of the workload (%d ranks x %d elements), %.1f s" % (
                reps, len(xs), n, el),
            "host_cores_available": len(os.sched_getaffinity(0))}


# -------------------------------------------------------------- GPU leg

def alg_bytes(W, I, n, b, P):
    """Algorithmic HBM bytes of the two kernels for one all_reduce:
    reduce+encode reads W*n*b and writes I*P; decode+broadcast reads the I
    payloads once (I*P) and writes W*n*b."""
    return W * n * b + I * P, I * P + W * n * b


def dataclasses_replace_f32(w):
    """The workload drawn as float32 (the draw's own type)."""
    import dataclasses
    return dataclasses.replace(w, dtype="f32")


def stream_set_count(set_bytes):
    """Input sets cycled by kernel_stream: together at least 4 x L2 when a
    set is large (at least 5, at most 8 GiB in all), else 16 sets."""
    return max(5, min(-(-(4 * L2_BYTES) // set_bytes), 16 if set_bytes * 16 < 4 * L2_BYTES else 1 << 30,
                      (8 << 30) // set_bytes))


def make_sets(pristine, I, P, S, ef=False):
    """S distinct input sets (copies of the rank buffers), output buffers,
    payloads of P bytes per island and, with error feedback, residuals."""
    import torch
    n = pristine[0].numel()
    dev = pristine[0].device
    return {"S": S,
            "ins": [[p.clone() for p in pristine] for _ in range(S)],
            "outs": [[torch.empty_like(p) for p in pristine] for _ in range(S)],
            "pays": [[torch.empty(P, dtype=torch.uint8, device=dev) for _ in range(I)] for _ in range(S)],
            "res": [[torch.zeros(n, dtype=torch.float32, device=dev) for _ in range(I)] for _ in range(S)]
            if ef else None}


def b2b_ms(stream, clean, warm, batches, S, launch):
    """Back-to-back launches, in steady state.  launch(q) enqueues one launch
    on input set q.  Each batch starts from a clean L2 (a 256 MiB read) after
    a ~0.4 ms GPU spin, so the host has queued the whole batch before its
    first event.  A CUDA event between two launches takes away the second
    one's programmatic early start, so the events sit after launch 0 and
    after the batch's last launch, and two batch lengths are timed: S
    launches (S - 1 after the first event) and 2 launches (1 after it).
    Their difference is S - 2 launches of a long run of back-to-back
    launches, without the start-up gap that follows the first event.
    Returns milliseconds per launch: (steady, with the gap) where `with the
    gap` is the long batch's window divided by S - 1."""
    import torch
    ea = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(batches)]
    with torch.cuda.stream(stream):
        for it in range(warm + batches):
            e = ea[it - warm] if it >= warm else None
            for count, (i0, i1) in ((S, (0, 1)), (2, (2, 3))):
                clean.amax()
                torch.cuda._sleep(800_000)
                for q in range(count):
                    launch(q)
                    if e and q == 0:
                        e[i0].record(stream)
                if e:
                    e[i1].record(stream)
    torch.cuda.synchronize()
    long_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in ea]))
    short_ms = float(np.mean([e[2].elapsed_time(e[3]) for e in ea]))
    return (long_ms - short_ms) / (S - 2), long_ms / (S - 1)


def kernel_stream(ctx, pristine, I, P, codec, block, op, stream, clean, warm, batches,
                  names=("k_reduce_encode", "k_decode_bcast"), ef=False, sets=None, scatter=False):
    """Timed region 3: each kernel launched back to back (b2b_ms), as the
    fused halves of the path (gb_island_reduce_compress_op, then
    gb_decompress_island_broadcast, or gb_decompress_scatter for
    reduce_scatter), with the same grid as in a step.  S distinct input
    sets, outputs and payloads (together at least 4 x L2 when a set is
    large, else 16 sets) are cycled, so no launch finds its inputs in L2:
    the decode batch starts after the payloads have been evicted, as
    payloads landed by the bridge's copies are read from HBM in a step.
    Every timed launch also writes back what its predecessor left dirty in
    L2: the steady state of a stream of buckets.  Returns per-launch
    milliseconds of both kernels.  ef: the encode carries error feedback
    (gb_island_reduce_compress_ef, one float32 residual per island and
    set).  sets: prebuilt make_sets() buffers (their payloads at least P
    bytes), reused across calls.  The op selects the codec path or the exact
    path (MAX / MIN, other dtypes)."""
    import torch
    W = len(pristine)
    n = pristine[0].numel()
    b = pristine[0].element_size()
    set_bytes = W * n * b + I * P + (I * n * 4 if ef else 0)
    if sets is None:
        sets = make_sets(pristine, I, P, stream_set_count(set_bytes), ef)
    S = sets["S"]
    ins, outs, pays, res = sets["ins"], sets["outs"], sets["pays"], sets["res"]
    if scatter:
        outs = [[o[: n // W] for o in row] for row in outs]
    # every leader's row holds the same I payloads: the call decodes them
    # once and writes all ranks, as the decode in a step does
    rows = [[pays[q][j] for g in range(I) for j in range(I)] for q in range(S)]

    def enc(q):
        if ef:
            ctx.island_reduce_compress_ef(ins[q], res[q], codec, block, pays[q], stream=stream)
        else:
            ctx.island_reduce_compress_op(ins[q], op, codec, block, pays[q], stream=stream)

    def dec(q):
        if scatter:
            ctx.decompress_scatter(rows[q], n, op, codec, block, outs[q], stream=stream)
        else:
            ctx.decompress_island_broadcast(rows[q], op, codec, block, outs[q], stream=stream)

    t1, g1 = b2b_ms(stream, clean, warm, batches, S, enc)
    t2, g2 = b2b_ms(stream, clean, warm, batches, S, dec)  # the payloads were written by the encodes
    return {"sets": S, "timed_launches_per_batch": S - 2, "batches": batches, "set_bytes": set_bytes,
            names[0]: t1, names[1]: t2, "with_first_gap": {names[0]: g1, names[1]: g2}}


def pinned_link(dev, stream, big=256 << 20):
    """Pinned copy bandwidth (the bridge's roofline): the best of five
    256 MiB cudaMemcpyAsync copies each way, CUDA events on the stream."""
    import torch
    hbuf = torch.empty(big, dtype=torch.uint8, pin_memory=True)
    dbuf = torch.empty(big, dtype=torch.uint8, device=dev)
    link = {}
    with torch.cuda.stream(stream):
        for name, (dst, src) in (("d2h_gbs", (hbuf, dbuf)), ("h2d_gbs", (dbuf, hbuf))):
            best = 0.0
            for _ in range(5):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dst.copy_(src, non_blocking=True)
                e1.record(stream)
                e1.synchronize()
                best = max(best, big / (e0.elapsed_time(e1) * 1e-3) / 1e9)
            link[name] = best
    return link


def run_gb(args, world, rank, local, pg):
    import torch
    from cross_vendor_gradient_gb300 import Context, kernel_launch_count, payload_bytes
    from cross_vendor_gradient_gb300 import workloads as wl
    from cross_vendor_gradient_gb300 import build as gbuild

    gbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = wl.WORKLOADS[args.workload]
    if args.dtype or args.op or args.islands or args.block:
        import dataclasses
        w = dataclasses.replace(w, dtype=args.dtype or w.dtype, op=args.op or w.op,
                                island_sizes=tuple(int(v) for v in args.islands.split(",")) if args.islands
                                else w.island_sizes, block=args.block or w.block)
    exact = w.op in ("max", "min") or w.dtype not in ("f32", "bf16")
    codec = "none" if exact else (args.codec or w.codecs[0])
    n = args.n or w.n
    W, I = w.world_size, len(w.island_sizes)
    xs = wl.host_rank_inputs(dataclasses_replace_f32(w), n=n)
    xs = [wl.as_dtype(x, w.dtype) for x in xs]
    b = xs[0].itemsize
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "f64": torch.float64,
           "i8": torch.int8, "u8": torch.uint8, "i32": torch.int32, "i64": torch.int64}[w.dtype]

    def dev_tensor(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(x).to(dev)

    pristine = [dev_tensor(x) for x in xs]
    bufs = [p.clone() for p in pristine]
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean = torch.zeros(FLUSH_BYTES // 8, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    K, Wm = args.steps, args.warmup
    ctx = Context(w.island_sizes)
    chunk_bytes = 2 << 20 if args.chunk_kib is None else args.chunk_kib << 10
    ctx.reserve(n, tdt, codec, w.block)

    link = pinned_link(dev, stream)

    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ef = args.ef and not exact and I > 1
    res = [torch.zeros(n, dtype=torch.float32, device=dev) for _ in range(I)] if ef else None

    def step(i, timed):
        for r in range(W):
            bufs[r].copy_(pristine[r], non_blocking=True)
        flush.zero_()   # L2 flush: write 512 MiB ...
        clean.amax()    # ... then read 256 MiB, so the lines left in L2 are clean
        if timed:
            ev0[i].record(stream)
        if ef:  # the residuals carry from step to step, as in training
            ctx.all_reduce_ef(bufs, res, w.op, codec, w.block, stream=stream)
        else:
            ctx.all_reduce(bufs, w.op, codec, w.block, stream=stream)
        if timed:
            ev1[i].record(stream)

    # ---- timed region 1: the step as a user runs it (pipelined policy, graph
    # replay, no phase marks: a CUDA event between kernels drains the stream)
    launches, clk, t_wall, ms, host_us = 0, None, 0.0, None, None
    if not args.roofline_only:
        ctx.set_pipeline(chunk_bytes, not args.no_graphs)
        ctx.set_sharded_bridge(args.sharded)
        with torch.cuda.stream(stream):
            for i in range(Wm):
                step(i, False)
        torch.cuda.synchronize()
        clocks = ClockSampler(local)
        clocks.start()
        barrier(pg)
        torch.cuda.synchronize()
        l0 = kernel_launch_count()
        t_wall = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(K):
                step(i, True)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        barrier(pg)
        launches = kernel_launch_count() - l0
        clk = clocks.stop()
        step_ms = [ev0[i].elapsed_time(ev1[i]) for i in range(K)]
        ms = max_over_ranks(pg, float(np.mean(step_ms)), dev if pg is not None else None)
        if not ef:
            host_us = host_call_us(ctx, bufs, pristine, w.op, codec, w.block, stream)

    # ---- timed region 2: per-kernel durations for the roofline.  One full
    # launch of each kernel per step (one bridge hop per call), CUDA events
    # around every phase on the launching stream.
    Kr = args.steps if args.roofline_only else min(K, 500)
    ctx.set_pipeline(0, False)
    ctx.set_sharded_bridge(False)
    # the same one-hop steps without phase marks first: the difference is
    # what the marks' CUDA events cost the step
    with torch.cuda.stream(stream):
        for i in range(Wm):
            step(i, False)
        for i in range(Kr):
            step(i, True)
    torch.cuda.synchronize()
    nomark_ms = float(np.mean([ev0[i].elapsed_time(ev1[i]) for i in range(Kr)]))
    ctx.set_phase_timing(Kr)
    with torch.cuda.stream(stream):
        for i in range(Wm):
            step(i, False)
        torch.cuda.synchronize()
        for i in range(Kr):
            step(i, True)
    torch.cuda.synchronize()
    plain_ms = float(np.mean([ev0[i].elapsed_time(ev1[i]) for i in range(Kr)]))
    if ms is None:
        ms = plain_ms
    phases = np.array([ctx.phase_times(Kr - 1 - i) for i in range(Kr)])  # oldest first
    ctx.set_phase_timing(0)
    ctx.set_pipeline(chunk_bytes, not args.no_graphs)

    if exact:
        pe = 4 if (w.dtype in ("bf16", "f16") and w.op in ("sum", "avg")) else b
        P = pe * n
        names = ("k_exact_reduce", "k_exact_combine")
    else:
        P = payload_bytes(codec, w.block, n) if I > 1 else 4 * n
        names = ("k_reduce_encode", "k_decode_bcast")
    k1_ms, bridge_ms, k2_ms = (float(np.mean(phases[:, j])) for j in range(3))
    k1_bytes, k2_bytes = alg_bytes(W, I, n, b, P)
    if ef:  # the encode also reads and writes every island's float32 residual
        k1_bytes += 2 * I * n * 4
    peak, peak_kind = measured_peaks()

    # ---- timed region 3: each kernel back to back (see kernel_stream)
    ks = None
    if I > 1:  # the codec path's kernels, or the exact path's (MAX / MIN, other dtypes)
        ks = kernel_stream(ctx, pristine, I, P, codec, w.block, w.op, stream, clean, Wm, max(3, min(Kr, 50)),
                           names, ef=ef)
        S, set_bytes = ks["sets"], ks["set_bytes"]
    if ks:
        r1, r2 = ks[names[0]], ks[names[1]]
        region = ("timed region 3: each kernel launched back to back over %d input sets (%.0f MB each, "
                  "distinct, from a clean L2); CUDA events after the first and the last launch of batches of "
                  "%d and of 2 launches, the difference over %d launches"
                  % (S, set_bytes / 1e6, S, S - 2))
    else:
        r1, r2 = k1_ms, k2_ms
        region = "timed region 2: one bridge hop per call, CUDA events around each phase"
    dom = (names[0], k1_bytes, r1) if r1 >= r2 else (names[1], k2_bytes, r2)
    achieved = dom[1] / (dom[2] * 1e-3) / 1e9
    link_bytes = I * P + I * (I - 1) * P
    link_peak = min(link["d2h_gbs"], link["h2d_gbs"])

    # end to end through the host-buffer entry point (pinned host buffers)
    # The W host rank buffers are the rows of one pinned [W, n] tensor (staged
    # with 2D copies by gb_all_reduce_host_rows); the same step on W separate
    # pinned tensors (gb_all_reduce_host, one copy per rank) is reported beside.
    e2e_ms, sep_ms, Ke = float("nan"), float("nan"), 0
    if not args.roofline_only:
        rows = torch.from_numpy(np.stack(xs) if xs[0].dtype == np.float32 else np.stack(xs).view(np.int16))
        rows = rows.pin_memory()
        if xs[0].dtype != np.float32:
            rows = rows.view(torch.bfloat16)
        host = [torch.from_numpy(x.copy()).pin_memory() if x.dtype == np.float32 else
                torch.from_numpy(x.view(np.int16).copy()).pin_memory().view(torch.bfloat16) for x in xs]
        Ke = max(10, min(200, K // 10))

        def e2e_mean(bufs):
            e_ms = []
            with torch.cuda.stream(stream):
                for i in range(3 + Ke):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    ctx.all_reduce_host(bufs, w.op, codec, w.block, stream=stream)
                    e1.record(stream)
                    e1.synchronize()
                    if i >= 3:
                        e_ms.append(e0.elapsed_time(e1))
            return float(np.mean(e_ms))
        e2e_ms = max_over_ranks(pg, e2e_mean(rows), dev if pg is not None else None)
        sep_ms = max_over_ranks(pg, e2e_mean(host), dev if pg is not None else None)
    ctx.close()

    # the metric's curve: the payload sweep, on the default line at N = 1
    sweep = None
    if (not args.roofline_only and not args.no_sweep and world == 1 and args.workload == "c2"
            and not (args.dtype or args.op or args.islands or args.block or args.n or args.codec or args.ef
                     or args.sharded or args.no_graphs or args.chunk_kib is not None)):
        del pristine, bufs
        torch.cuda.empty_cache()
        t0 = time.perf_counter()
        rows = sweep_rows(args, dev, stream, flush, clean, link_peak, max_steps=min(K, 20))
        sweep = sweep_line_object(rows, peak, peak_kind, link_peak, time.perf_counter() - t0)

    value = world * n * b / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded PCG64 per rank; no dataset)",
        "config": {"workload": "%s: %d simulated ranks as islands %s, one %.0f MiB %s buffer per rank "
                               "(n=%d), %s, op %s, codec %s block %d" % (
                                   w.key, W, list(w.island_sizes), n * b / 2 ** 20, w.dtype, n, w.dist,
                                   w.op, codec, w.block),
                   "ranks": W, "islands": list(w.island_sizes), "n": n, "codec": codec, "block": w.block,
                   "op": w.op, "error_feedback": bool(ef),
                   "policy": (("sharded-bridge, %d links%s" % (
                       min(w.island_sizes), ", CUDA graph replay" if not args.no_graphs else ""))
                              if args.sharded and min(w.island_sizes) > 1 else
                              ("pipelined-reduce-bridge-broadcast, equal payload chunks of at most %d KiB x "
                               "max(1, sqrt(P / (3 x %d KiB))) for one island's payload P%s" % (
                                  chunk_bytes >> 10, chunk_bytes >> 10,
                                  ", CUDA graph replay" if not args.no_graphs else ""))
                              if chunk_bytes else "reduce-bridge-broadcast"),
                   "l2": "flushed before every timed step (512 MiB write, then a 256 MiB "
                                     "read so that no dirty line is left); inputs restored from a device "
                                     "copy outside the timed events",
                   "parallelism": "replicas x%d" % world},
        "roofline": {"bound": "hbm", "kernel": dom[0], "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "alg_bytes_per_launch": dom[1], "avg_launch_ms": dom[2], "traffic": None,
                     "region": region,
                     "bytes_from": ("HBM, all of them: the inputs of every timed launch (rank buffers, or the "
                                    "payloads the encode batch wrote) are read after a clean L2; ncu with the "
                                    "cache control off found the decode's DRAM reads at 100.2 % of its payload "
                                    "bytes; written lines still dirty in L2 when a launch ends are written back "
                                    "during the next one") if ks else "one-hop steps: payloads may hit L2"},
        **({"kernels_stream_ms": ks,
            "kernels_stream_hbm_frac": {names[0]: k1_bytes / (ks[names[0]] * 1e-3) / 1e9 / peak,
                                        names[1]: k2_bytes / (ks[names[1]] * 1e-3) / 1e9 / peak}}
           if ks else {}),
        "kernels_ms": {names[0]: k1_ms, "bridge_hop": bridge_ms, names[1]: k2_ms,
                       "region": "timed region 2: one bridge hop per call, CUDA events around each phase",
                       "step_ms_with_marks": plain_ms, "step_ms_without_marks": nomark_ms,
                       "marks_cost_ms": plain_ms - nomark_ms},
        "kernels_hbm_frac": {names[0]: k1_bytes / (k1_ms * 1e-3) / 1e9 / peak,
                             names[1]: k2_bytes / (k2_ms * 1e-3) / 1e9 / peak},
        "bridge": {"bytes_per_step": link_bytes, "ms": bridge_ms,
                   "achieved_gbs": link_bytes / (bridge_ms * 1e-3) / 1e9 if bridge_ms > 0 else None,
                   "pinned_copy_gbs": link, "frac": (link_bytes / (bridge_ms * 1e-3) / 1e9) / link_peak
                   if bridge_ms > 0 else None},
        "e2e": {"value": world * n * b / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "steps": Ke, "h2d_bytes_per_step": W * n * b, "d2h_bytes_per_step": W * n * b,
                "api": "gb_all_reduce_host_rows (the W pinned host rank buffers as the rows of one [W, n] tensor)",
                "separate_buffers": {"ms_per_step": sep_ms, "value": world * n * b / (sep_ms * 1e-3) / 1e9,
                                     "api": "gb_all_reduce_host (W separate pinned host tensors)"}},
        "gpu_launches": int(launches),
        "timed_wall_s": t_wall,
        "clocks": clk,
        **({"host_call_us": host_us} if host_us else {}),
        **({"sweep": sweep} if sweep else {}),
    }
    return line, w, xs, codec


def host_call_us(ctx, bufs, pristine, op, codec, block, stream, calls=200):
    """Host wall time of one all_reduce call: the library's own work per call
    (argument checks, plan and graph lookup, the enqueue) through a ctypes
    call with prepared arguments, and the same call through the tensor-level
    Context.  The queue is drained every 20 calls, outside the timed calls,
    so that no call waits for queue space.  The rank buffers are restored
    between calls, also outside the timed calls."""
    import torch
    from cross_vendor_gradient_gb300 import binding as B
    from cross_vendor_gradient_gb300.api import _codec, _dtype, _op
    arr = B._ptrs([t.data_ptr() for t in bufs])
    args = (ctx.handle, arr, bufs[0].numel(), _dtype(bufs), _op(op), _codec(codec), block, stream.cuda_stream)
    fn = B.lib().gb_all_reduce
    out = {}
    for name, call in (("library", lambda: fn(*args)),
                       ("python_api", lambda: ctx.all_reduce(bufs, op, codec, block, stream=stream))):
        torch.cuda.synchronize()
        t = []
        for k in range(calls):
            if k % 20 == 0:
                torch.cuda.synchronize()  # keep the queue short: no call waits for queue space
            with torch.cuda.stream(stream):
                for b, p0 in zip(bufs, pristine):
                    b.copy_(p0, non_blocking=True)
            t0 = time.perf_counter()
            st = call()
            t.append(time.perf_counter() - t0)
            if name == "library" and st != 0:
                raise RuntimeError("gb_all_reduce failed: %d" % st)
        torch.cuda.synchronize()
        out[name + "_median_us"] = statistics.median(t) * 1e6
    out["calls"] = calls
    out["what"] = ("host wall time per gb_all_reduce call (enqueue of the graph-replayed pipelined step; "
                   "the device work runs after): a ctypes call with prepared arguments, and "
                   "Context.all_reduce")
    return out


KERNEL_SOURCES = ("gb_kernels_enc.cu", "gb_kernels_dec.cu", "gb_kernels_exact.cu", "gb_device.cuh", "gb_kernels.cuh")


def _code_only(text):
    """C++ source without its comments and blank lines: what the compiler sees."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_sha():
    """sha256[:16] over the kernel sources' code, comments left out (the key
    of a recorded capture: a comment edit does not change what was profiled)."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "cross_vendor_gradient_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel):
    """DRAM bytes per launch recorded by an ncu capture of the current kernel
    sources, or None (profiles/dram_traffic.txt, 'key=value' lines)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha()
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kv = dict(x.split("=", 1) for x in line.split() if "=" in x)
        if kv.get("kernel") == kernel and kv.get("src_sha") == sha:
            return float(kv["dram_bytes_per_launch_full_size"])
    return None


def run_buckets_bench(args, world, rank, local, pg):
    """Bucketed workloads (c4: GPT-2 small, c5: 1.1B Llama-style): one step is
    the all_reduce of the whole bf16 gradient set, fused into 25 MiB DDP
    buckets, through gb_all_reduce_buckets (one pipeline, one graph)."""
    import torch
    from cross_vendor_gradient_gb300 import Context, bucket_plan, kernel_launch_count, payload_bytes
    from cross_vendor_gradient_gb300 import workloads as wl
    from cross_vendor_gradient_gb300 import build as gbuild

    gbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = wl.WORKLOADS[args.workload]
    codec = args.codec or w.codecs[0]
    W, I = w.world_size, len(w.island_sizes)
    numels = [wl.numel(sh) for sh in w.tensors]
    rs_ag = args.workload == "c5"  # this set is also reduce_scattered then all_gathered
    # reduce_scatter slices of whole 8-element vectors: buckets padded to 8 * W elements
    _, _, bn = bucket_plan(numels, w.elem_bytes, wl.BUCKET_CAP_BYTES, 8 * W if rs_ag else 1)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    pristine = [[wl.draw_device(w.dist, nb, wl.bucket_seed(w.cid, bi, r), dev, tdt) for r in range(W)]
                for bi, nb in enumerate(bn)]
    bufs = [[x.clone() for x in row] for row in pristine]
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean = torch.zeros(FLUSH_BYTES // 8, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    K, Wm = args.steps, max(3, args.warmup)
    ctx = Context(w.island_sizes)
    chunk_bytes = 2 << 20 if args.chunk_kib is None else args.chunk_kib << 10
    ctx.set_pipeline(chunk_bytes, not args.no_graphs)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ef = args.ef
    res = [[torch.zeros(nb, dtype=torch.float32, device=dev) for _ in range(I)] for nb in bn] if ef else None

    def step(i, timed, per_bucket=False):
        for row_p, row_b in zip(pristine, bufs):
            for x, y in zip(row_p, row_b):
                y.copy_(x, non_blocking=True)
        flush.zero_()
        clean.amax()
        if timed:
            ev0[i].record(stream)
        if per_bucket:
            for bi, row in enumerate(bufs):
                if ef:
                    ctx.all_reduce_ef(row, res[bi], w.op, codec, w.block, stream=stream)
                else:
                    ctx.all_reduce(row, w.op, codec, w.block, stream=stream)
        elif ef:  # the residuals carry from step to step, as in training
            ctx.all_reduce_buckets_ef(bufs, res, w.op, codec, w.block, stream=stream)
        else:
            ctx.all_reduce_buckets(bufs, w.op, codec, w.block, stream=stream)
        if timed:
            ev1[i].record(stream)

    with torch.cuda.stream(stream):
        for i in range(Wm):
            step(i, False)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(pg)
    torch.cuda.synchronize()
    l0 = kernel_launch_count()
    with torch.cuda.stream(stream):
        for i in range(K):
            step(i, True)
    torch.cuda.synchronize()
    barrier(pg)
    launches = kernel_launch_count() - l0
    clk = clocks.stop()
    ms = max_over_ranks(pg, float(np.mean([ev0[i].elapsed_time(ev1[i]) for i in range(K)])),
                        dev if pg is not None else None)
    rs_line = None
    if rs_ag:
        # reduce_scatter then all_gather of every bucket, same ranks, same buffers
        slices = [[torch.empty(nb // W, dtype=tdt, device=dev) for _ in range(W)] for nb in bn]
        Ks = max(2, min(K, 5))

        def step_rs(i, timed, sets):
            for row_p, row_b in zip(pristine, bufs):
                for x, y in zip(row_p, row_b):
                    y.copy_(x, non_blocking=True)
            flush.zero_()
            clean.amax()
            if timed:
                ev0[i].record(stream)
            if sets:  # the whole set per call: one pipeline, one graph each
                ctx.reduce_scatter_buckets(bufs, slices, w.op, codec, w.block, stream=stream)
                ctx.all_gather_buckets(slices, bufs, stream=stream)
            else:
                for row, sl in zip(bufs, slices):
                    ctx.reduce_scatter(row, sl, w.op, codec, w.block, stream=stream)
                    ctx.all_gather(sl, row, stream=stream)
            if timed:
                ev1[i].record(stream)

        ms_rs = {}
        for sets in (True, False):
            with torch.cuda.stream(stream):
                for i in range(Wm):
                    step_rs(i, False, sets)
                for i in range(Ks):
                    step_rs(i, True, sets)
            torch.cuda.synchronize()
            ms_rs[sets] = float(np.mean([ev0[i].elapsed_time(ev1[i]) for i in range(Ks)]))
        per = sum(bn) * w.elem_bytes
        rs_line = {"what": "gb_reduce_scatter_buckets then gb_all_gather_buckets of the whole set (one pipeline "
                           "and one graph each, payload chunks of at most 6 x %d KiB; all_gather in groups of "
                           "whole rank blocks)" % (chunk_bytes >> 10),
                   "ms_per_step": ms_rs[True], "value": per / (ms_rs[True] * 1e-3) / 1e9, "unit": "GB/s",
                   "steps": Ks,
                   "per_bucket_calls_ms_per_step": ms_rs[False]}
        del slices
    # roofline region: one hop per bucket, phase marks around every kernel
    Kr = max(2, min(K, 5))
    ctx.set_pipeline(0, False)
    ctx.set_phase_timing(Kr * len(bn))
    with torch.cuda.stream(stream):
        step(0, False, per_bucket=True)
        torch.cuda.synchronize()
        for i in range(Kr):
            step(i, True, per_bucket=True)
    torch.cuda.synchronize()
    ph = np.array([ctx.phase_times(a) for a in range(Kr * len(bn))])  # newest first
    ctx.set_phase_timing(0)
    # timed region 3 on the set's largest bucket within the 25 MiB cap (the
    # shape most of the set's kernels have): each kernel back to back
    b = w.elem_bytes
    bi = max((i for i, nb in enumerate(bn) if nb * b <= wl.BUCKET_CAP_BYTES), key=lambda i: bn[i])
    Pb = payload_bytes(codec, w.block, bn[bi])
    ks = kernel_stream(ctx, pristine[bi], I, Pb, codec, w.block, w.op, stream, clean, 2, 5, ef=ef)
    ctx.close()
    kb1, kb2 = alg_bytes(W, I, bn[bi], b, Pb)
    if ef:
        kb1 += 2 * I * bn[bi] * 4
    per_rank = sum(bn) * b
    bytes1 = bytes2 = 0
    for nb in bn:
        P = payload_bytes(codec, w.block, nb)
        x1, x2 = alg_bytes(W, I, nb, b, P)
        if ef:  # the encode also reads and writes every island's float32 residual
            x1 += 2 * I * nb * 4
        bytes1 += x1
        bytes2 += x2
    t1 = float(np.sum(ph[:, 0])) / Kr
    t2 = float(np.sum(ph[:, 2])) / Kr
    peak, peak_kind = measured_peaks()
    s1, s2 = ks["k_reduce_encode"], ks["k_decode_bcast"]
    dom = ("k_reduce_encode", kb1, s1) if s1 >= s2 else ("k_decode_bcast", kb2, s2)
    achieved = dom[1] / (dom[2] * 1e-3) / 1e9
    return {
        "metric": METRIC, "value": world * per_rank / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded torch generators on the device)",
        "config": {"workload": "%s: %d simulated ranks as islands %s, %d-tensor %s gradient set (%d values) in %d "
                               "buckets of <= 25 MiB, %s, op %s, codec %s block %d" % (
                                   w.key, W, list(w.island_sizes), len(numels), w.dtype, sum(numels), len(bn),
                                   w.dist, w.op, codec, w.block),
                   "buckets": len(bn), "values_per_rank": sum(bn),
                   "error_feedback": bool(ef),
                   "policy": "one pipeline over all buckets (payload chunks of at most 6 x %d KiB, each bucket "
                             "cut evenly), one CUDA graph per step" % (chunk_bytes >> 10),
                   "l2": "flushed before every timed step (512 MiB write, then a 256 MiB read)"},
        "roofline": {"bound": "hbm", "kernel": dom[0], "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": achieved / peak, "alg_bytes_per_launch": dom[1],
                     "avg_launch_ms": dom[2], "traffic": None,
                     "region": "timed region 3 on bucket %d (%d values per rank, the largest within the 25 MiB "
                               "cap): each kernel back to back over %d input sets, steady state"
                               % (bi, bn[bi], ks["sets"])},
        "kernels_stream_ms": ks,
        "kernels_in_step": {"k_reduce_encode_ms_per_step": t1, "k_decode_bcast_ms_per_step": t2,
                            "k_reduce_encode_hbm_frac": bytes1 / (t1 * 1e-3) / 1e9 / peak,
                            "k_decode_bcast_hbm_frac": bytes2 / (t2 * 1e-3) / 1e9 / peak,
                            "region": "one hop per bucket over the whole set, CUDA events around each kernel"},
        "gpu_launches": int(launches), "clocks": clk,
        **({"rs_ag": rs_line} if rs_line else {}),
    }


SWEEP_COLUMNS = ["bytes_per_rank", "codec", "steps", "ms_per_step", "algbw_gbs", "encode_frac", "decode_frac",
                 "encode_frac_in_step", "decode_frac_in_step", "bridge_gbs", "bridge_frac", "floor_ms",
                 "ms_median"]


def op_floor_ms(ctx, bufs, I, P, codec, block, op, stream, flush, clean, reps=100):
    """The sum of a one-chunk step's operations, each timed on its own on the
    device (CUDA events around it, L2 flushed before it as before a step,
    after a spin so the host is ahead): the encode launch, the bridge's
    device -> host and host -> device copies of the step's sizes, the decode
    launch; minus one event pair per extra measurement (each one carries the
    cost of its own two events).  Host buffers are pinned.  Returns (floor,
    parts) in milliseconds."""
    import torch
    dev = bufs[0].device
    nbytes = I * P
    hb = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    db = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    pays = [torch.empty(P, dtype=torch.uint8, device=dev) for _ in range(I)]
    rows = [pays[j] for g in range(I) for j in range(I)]

    def each(fn):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        with torch.cuda.stream(stream):
            fn()
            torch.cuda.synchronize()
            torch.cuda._sleep(20_000_000)
            for a, b in evs:
                flush.zero_()
                clean.amax()
                a.record(stream)
                fn()
                b.record(stream)
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in evs]))

    parts = {"events": each(lambda: None),
             "encode": each(lambda: ctx.island_reduce_compress(bufs, codec, block, pays, stream=stream)),
             "copies": each(lambda: (hb.copy_(db, non_blocking=True), db.copy_(hb, non_blocking=True))),
             "decode": each(lambda: ctx.decompress_island_broadcast(rows, op, codec, block, bufs, stream=stream))}
    return parts["encode"] + parts["copies"] + parts["decode"] - 2 * parts["events"], parts


def sweep_rows(args, dev, stream, flush, clean, link_peak, max_steps, emit=None):
    """The payload sweep (workload c3): 4 KiB .. 256 MiB of float32 per rank
    at 2 islands x 2 ranks, U(-1, 1), SUM, codecs none / bf16 / e4m3.  Per
    row: the step as a user runs it (pipelined policy, graph replay, no phase
    marks; L2 flushed before each timed step) for the algorithm GB/s; each
    kernel back to back over distinct input sets (kernel_stream) for the HBM
    roofline fractions; one-hop steps with phase marks for the kernels inside
    a step and the bridge against pinned copy bandwidth; and, up to 1 MiB,
    the sum of the step's operations timed one by one (op_floor_ms).  Rank
    buffers are drawn on the device (torch.Generator seeded per rank).
    Returns compact rows (SWEEP_COLUMNS); emit(row_dict) gets each row's
    details as it is measured."""
    import torch
    from cross_vendor_gradient_gb300 import Context, payload_bytes
    from cross_vendor_gradient_gb300 import workloads as wl
    w = wl.WORKLOADS["c3"]
    W, I = w.world_size, len(w.island_sizes)
    peak, peak_kind = measured_peaks()
    codecs = [args.codec] if args.codec else list(w.codecs)
    chunk = 2 << 20 if args.chunk_kib is None else args.chunk_kib << 10
    rows = []
    for lg in wl.SWEEP_LOG2:
        n = 1 << lg
        pristine = [wl.draw_device(w.dist, n, wl.seed_of(w.cid, r), dev, torch.float32) for r in range(W)]
        bufs = [p.clone() for p in pristine]
        # up to 1 MiB a step is a few tens of microseconds: 50 of them, for the comparison with the floor
        K = 50 if n * 4 <= (1 << 20) else max(10, min(max_steps, int(4e9 // (n * 4 * W))))
        Pmax = max(payload_bytes(c, w.block, n) for c in codecs)
        sets = make_sets(pristine, I, Pmax, stream_set_count(W * n * 4 + I * Pmax))
        for codec in codecs:
            ctx = Context(w.island_sizes)
            ctx.reserve(n, torch.float32, codec, w.block)
            ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
            ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
            Kt = K  # timed steps of the user-facing step

            def steps(count, timed):
                with torch.cuda.stream(stream):
                    for i in range(count):
                        for r in range(W):
                            bufs[r].copy_(pristine[r], non_blocking=True)
                        flush.zero_()
                        clean.amax()
                        if timed:
                            ev0[i].record(stream)
                        ctx.all_reduce(bufs, w.op, codec, w.block, stream=stream)
                        if timed:
                            ev1[i].record(stream)
                torch.cuda.synchronize()
                return float(np.mean([ev0[i].elapsed_time(ev1[i]) for i in range(count)])) if timed else 0.0

            ctx.set_pipeline(chunk, True)
            steps(3, False)
            if n * 4 >= (16 << 20):
                # the large rows (the >= 16 MiB the kernels' target applies to): at least 100 ms of timed
                # steps, counted from one more (replayed, timed) warm-up step
                one = steps(1, True)
                Kt = max(K, min(1000, int(math.ceil(100.0 / max(one, 1e-3)))))
                ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(Kt)]
                ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(Kt)]
            ms = steps(Kt, True)
            ms_median = float(np.median([ev0[i].elapsed_time(ev1[i]) for i in range(Kt)]))
            ctx.set_pipeline(0, False)
            ctx.set_phase_timing(K)
            steps(2, False)
            plain = steps(K, True)
            ph = np.array([ctx.phase_times(a) for a in range(K)])
            ctx.set_phase_timing(0)
            k1, br, k2 = (float(np.mean(ph[:, j])) for j in range(3))
            P = payload_bytes(codec, w.block, n)
            b1, b2 = alg_bytes(W, I, n, 4, P)
            ks = kernel_stream(ctx, pristine, I, P, codec, w.block, w.op, stream, clean, 1,
                               max(3, min(10, int(2e9 // (n * 4 * W)))), sets=sets)
            floor = parts = None
            if n * 4 <= (1 << 20):
                floor, parts = op_floor_ms(ctx, bufs, I, P, codec, w.block, w.op, stream, flush, clean)
            ctx.close()
            s1, s2 = ks["k_reduce_encode"], ks["k_decode_bcast"]
            link_bytes = I * P + I * (I - 1) * P
            bridge = link_bytes / (br * 1e-3) / 1e9 if br > 0 else None
            row = [4 * n, codec, Kt, ms, 4 * n / (ms * 1e-3) / 1e9, b1 / (s1 * 1e-3) / 1e9 / peak,
                   b2 / (s2 * 1e-3) / 1e9 / peak, b1 / (k1 * 1e-3) / 1e9 / peak, b2 / (k2 * 1e-3) / 1e9 / peak,
                   bridge, bridge / link_peak if bridge else None, floor, ms_median]
            rows.append([float('%.6g' % v) if isinstance(v, float) else v for v in row])
            if emit:
                emit({"metric": METRIC, "sweep_row": True, "workload": "c3", "codec": codec, "n": n,
                      "bytes_per_rank": 4 * n, "value": row[4], "unit": "GB/s", "ms_per_step": ms, "steps": Kt,
                      "one_hop_ms_per_step": plain,
                      "hbm_frac": {"k_reduce_encode": row[5], "k_decode_bcast": row[6], "peak_gbs": peak,
                                   "peak_kind": peak_kind,
                                   "region": "each kernel back to back over %d distinct input sets" % ks["sets"]},
                      "kernels_stream_ms": {"k_reduce_encode": s1, "k_decode_bcast": s2},
                      "in_step_hbm_frac": {"k_reduce_encode": row[7], "k_decode_bcast": row[8]},
                      "kernels_ms": {"k_reduce_encode": k1, "bridge_hop": br, "k_decode_bcast": k2},
                      "bridge_gbs": bridge, "bridge_frac": row[10],
                      **({"floor_ms": floor, "floor_parts_ms": parts} if floor is not None else {})})
        del pristine, bufs, sets
        torch.cuda.empty_cache()
    return rows


def sweep_line_object(rows, peak, peak_kind, link_peak, wall_s):
    """The sweep as one compact object of the bench line."""
    return {"workload": "c3: 4 simulated ranks as islands [2, 2], float32 U(-1, 1) per rank, SUM, "
                        "4 KiB .. 256 MiB per rank in powers of two, codecs none / bf16 / e4m3 block 256",
            "columns": SWEEP_COLUMNS, "rows": rows,
            "notes": {"ms_per_step": "the step as a user runs it (pipelined policy, CUDA graph replay), L2 flushed "
                                     "before each timed step, CUDA events around the step",
                      "algbw_gbs": "bytes of one rank buffer / step time",
                      "encode_frac, decode_frac": "algorithmic HBM bytes / back-to-back launch time / %.1f GB/s "
                                                  "(%s HBM copy peak)" % (peak, peak_kind),
                      "*_in_step": "the same kernels inside one-hop steps with CUDA events around each phase",
                      "bridge_gbs, bridge_frac": "one-hop device->host + host->device bytes / bridge time, and "
                                                 "its fraction of min(D2H, H2D) pinned copy bandwidth %.1f GB/s"
                                                 % link_peak,
                      "floor_ms": "rows up to 1 MiB: encode + copies + decode, each timed alone after an L2 "
                                  "flush (median of 100), minus the extra event pairs",
                      "ms_median": "the median step, beside the mean ms_per_step"},
            "wall_s": wall_s}


def run_reference(args, world, rank, pg):
    """The oracle, as it stands, on the host cores: each step is one oracle
    all_reduce of a bounded sample (a prefix of every rank buffer) of the
    workload, sized so that warmup + steps take about two minutes."""
    import oracle
    from cross_vendor_gradient_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    codec = args.codec or w.codecs[0]
    n_full = args.n or w.n
    xs_full = wl.host_rank_inputs(w, n=n_full)
    probe = min(n_full, 1 << 16)
    t0 = time.perf_counter()
    oracle.all_reduce([x[:probe] for x in xs_full], w.island_sizes, w.op, codec, w.block)
    rate = probe / max(time.perf_counter() - t0, 1e-6)  # elements per second per step
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(min(n_full, max(256, rate * budget)) // 256 * 256) or min(n_full, 256)
    xs = [np.ascontiguousarray(x[:n]) for x in xs_full]
    for _ in range(args.warmup):
        oracle.all_reduce(xs, w.island_sizes, w.op, codec, w.block)
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.all_reduce(xs, w.island_sizes, w.op, codec, w.block)
        t.append(time.perf_counter() - t0)
    ms = 1e3 * float(np.mean(t))
    value = n * w.elem_bytes / (ms * 1e-3) / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded PCG64 per rank; no dataset)",
        "config": {"workload": "%s: %d simulated ranks as islands %s, %s, op %s, codec %s block %d; "
                               "each step a prefix of %d of the %d elements per rank" % (
                                   w.key, w.world_size, list(w.island_sizes), w.dtype, w.op, codec,
                                   w.block, n, n_full),
                   "ranks": w.world_size, "islands": list(w.island_sizes), "n": n, "codec": codec,
                   "block": w.block, "op": w.op, "parallelism": "host, single thread"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "prefix of %d elements of each of the %d rank buffers per step" % (
                             n, w.world_size),
                         "host_cores_available": len(os.sched_getaffinity(0))},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_collective(args, world, rank, local, pg):
    """reduce_scatter, all_gather or broadcast on the default workload's
    ranks and buffer size: one step is one call of the collective.
    reduce_scatter: n elements per rank in, n / W out (the codec applies);
    all_gather: n / W in, n out (exact); broadcast: n in place from rank 0
    (exact).  value = n * b / step time (bytes of one full rank buffer).  The
    kernels' HBM fractions come from their launches back to back (the
    roofline; timed region 3) and from one-hop calls with phase marks, with
    the algorithmic bytes of each collective: reduce_scatter encode
    W*n*b + I*P, decode I*P + n*b; all_gather copy W*m*b read + W*W*m*b
    written (m = n / W); broadcast copy n*b read + (W - 1)*n*b written."""
    import torch
    from cross_vendor_gradient_gb300 import Context, kernel_launch_count, payload_bytes
    from cross_vendor_gradient_gb300 import workloads as wl
    from cross_vendor_gradient_gb300 import build as gbuild

    gbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = wl.WORKLOADS[args.workload]
    coll = args.collective
    codec = (args.codec or w.codecs[0]) if coll == "reduce_scatter" else "none"
    W, I = w.world_size, len(w.island_sizes)
    n = (args.n or w.n) // W * W
    m = n // W
    xs = wl.host_rank_inputs(dataclasses_replace_f32(w), n=n)
    pristine = [torch.from_numpy(x).to(dev) for x in xs]
    if coll == "all_gather":
        pristine = [p[:m].clone() for p in pristine]
    ins = [p.clone() for p in pristine]
    outs = ([torch.empty(m, dtype=torch.float32, device=dev) for _ in range(W)] if coll == "reduce_scatter" else
            [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(W)] if coll == "all_gather" else None)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean = torch.zeros(FLUSH_BYTES // 8, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    K, Wm = args.steps, max(3, args.warmup)
    ctx = Context(w.island_sizes)
    chunk_bytes = 2 << 20 if args.chunk_kib is None else args.chunk_kib << 10
    b = 4

    def call():
        if coll == "reduce_scatter":
            ctx.reduce_scatter(ins, outs, w.op, codec, w.block, stream=stream)
        elif coll == "all_gather":
            ctx.all_gather(ins, outs, stream=stream)
        else:
            ctx.broadcast(ins, 0, stream=stream)

    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]

    def steps(count, timed):
        with torch.cuda.stream(stream):
            for i in range(count):
                for x, y in zip(pristine, ins):
                    y.copy_(x, non_blocking=True)
                flush.zero_()
                clean.amax()
                if timed:
                    ev0[i].record(stream)
                call()
                if timed:
                    ev1[i].record(stream)
        torch.cuda.synchronize()
        return float(np.mean([ev0[i].elapsed_time(ev1[i]) for i in range(count)])) if timed else 0.0

    ms, launches, clk = None, 0, None
    if not args.roofline_only:  # timed region 1: the call as a user makes it
        ctx.set_pipeline(chunk_bytes, not args.no_graphs)
        steps(Wm, False)
        clocks = ClockSampler(local)
        clocks.start()
        barrier(pg)
        l0 = kernel_launch_count()
        ms = steps(K, True)
        launches = kernel_launch_count() - l0
        barrier(pg)
        clk = clocks.stop()
        ms = max_over_ranks(pg, ms, dev if pg is not None else None)
    Kr = min(K, 200)
    ctx.set_pipeline(0, False)
    ctx.set_phase_timing(Kr)
    steps(3, False)
    one_hop = steps(Kr, True)
    if ms is None:
        ms = one_hop
    ph = np.array([ctx.phase_times(a) for a in range(Kr)])
    ctx.set_phase_timing(0)
    k1, br, k2 = (float(np.mean(ph[:, j])) for j in range(3))
    P = payload_bytes(codec, w.block, n) if coll == "reduce_scatter" else m * b
    if coll == "reduce_scatter":
        kern = [("k_reduce_encode", W * n * b + I * P, k1), ("k_decode_slices", I * P + n * b, k2)]
        link = I * P + I * (I - 1) * P
    elif coll == "all_gather":
        kern = [("k_copy", W * m * b + W * W * m * b, k2)]
        link = W * m * b + (I - 1) * W * m * b
    else:
        kern = [("k_copy", n * b + (W - 1) * n * b, k2)]
        link = n * b + (I - 1) * n * b

    # ---- timed region 3: the collective's kernels back to back.
    # reduce_scatter: the fused halves (encode, then the slice decode);
    # all_gather / broadcast: the copy kernel alone, as the whole call of a
    # one-island context over the same W ranks (no bridge, nothing else
    # launched), algorithmic bytes W*m*b + W*W*m*b and n*b + (W-1)*n*b.
    Kb = max(3, min(K, 20))
    if coll == "reduce_scatter":
        ks = kernel_stream(ctx, pristine, I, P, codec, w.block, w.op, stream, clean, 1, Kb,
                           ("k_reduce_encode", "k_decode_slices"), scatter=True)
        b2b = [(k, nb, ks[k]) for k, nb, _ in kern]
        sets_used = ks["sets"]
    else:
        one = Context((W,))
        set_bytes = (W * m * b + W * n * b) if coll == "all_gather" else W * n * b
        S = stream_set_count(set_bytes)
        srcs = [[p.clone() for p in pristine] for _ in range(S)]
        dsts = [[torch.empty(n, dtype=torch.float32, device=dev) for _ in range(W)] for _ in range(S)] \
            if coll == "all_gather" else None

        def launch(q):
            if coll == "all_gather":
                one.all_gather(srcs[q], dsts[q], stream=stream)
            else:
                one.broadcast(srcs[q], 0, stream=stream)

        t, _ = b2b_ms(stream, clean, 1, Kb, S, launch)
        one.close()
        b2b = [("k_copy (one island of %d ranks)" % W, kern[0][1], t)]
        sets_used = S
        del srcs, dsts
    ctx.close()
    peak, peak_kind = measured_peaks()
    dom = max(b2b, key=lambda t: t[2])
    achieved = dom[1] / (dom[2] * 1e-3) / 1e9
    return {
        "metric": "%s algorithm GB/s and %% of GB300 HBM roofline" % coll, "value": world * n * b / (ms * 1e-3) / 1e9,
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded PCG64 per rank; no dataset)",
        "config": {"workload": "%s: %d simulated ranks as islands %s, %s of one %.0f MiB f32 buffer per rank "
                               "(n=%d), %s%s" % (w.key, W, list(w.island_sizes), coll, n * b / 2 ** 20, n, w.dist,
                                                 (", op %s, codec %s block %d" % (w.op, codec, w.block))
                                                 if coll == "reduce_scatter" else ", exact"),
                   "policy": {"reduce_scatter": "pipelined, equal payload chunks of at most max(%d KiB, S - %d KiB), "
                                                "S = %d KiB x max(1, sqrt(P / (3 x %d KiB))) for one island's "
                                                "payload P" % (chunk_bytes >> 11, chunk_bytes >> 11,
                                                               chunk_bytes >> 10, chunk_bytes >> 10),
                              "all_gather": "pipelined, groups of whole rank blocks of about %d KiB" % (
                                  chunk_bytes >> 10),
                              "broadcast": "pipelined, equal pieces of up to %d KiB" % (chunk_bytes >> 8)}[coll]
                   if chunk_bytes else "one bridge hop",
                   "l2": "flushed before every timed step (512 MiB write, then a 256 MiB read)"},
        "roofline": {"bound": "hbm", "kernel": dom[0], "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": achieved / peak, "alg_bytes_per_launch": dom[1],
                     "avg_launch_ms": dom[2], "traffic": None,
                     "region": "timed region 3: back to back over %d distinct input sets from a clean L2"
                               % sets_used},
        "kernels_stream": [{"kernel": k, "alg_bytes": nb, "ms": t, "hbm_frac": nb / (t * 1e-3) / 1e9 / peak}
                           for k, nb, t in b2b],
        "kernels": [{"kernel": k, "alg_bytes": nb, "ms": t, "hbm_frac": nb / (t * 1e-3) / 1e9 / peak,
                     "region": "one bridge hop per call, CUDA events around each phase"}
                    for k, nb, t in kern],
        "bridge": {"bytes_per_step": link, "ms": br, "achieved_gbs": link / (br * 1e-3) / 1e9 if br > 0 else None},
        "one_hop_ms_per_step": one_hop, "gpu_launches": int(launches), "clocks": clk,
        "e2e": None, "e2e_note": "no host-buffer entry point for this collective",
    }


def main():
    args = parse()
    world, rank, local, pg = dist_setup(args)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank, pg)), flush=True)
        if pg is not None:
            pg.destroy_process_group()
        return
    if args.sweep:
        if rank == 0:
            import torch
            from cross_vendor_gradient_gb300 import build as gbuild
            gbuild.build()
            torch.cuda.set_device(local)
            dev = torch.device("cuda", local)
            stream = torch.cuda.Stream(device=dev)
            flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
            clean = torch.zeros(FLUSH_BYTES // 8, dtype=torch.float32, device=dev)
            link = pinned_link(dev, stream)
            sweep_rows(args, dev, stream, flush, clean, min(link["d2h_gbs"], link["h2d_gbs"]), args.steps,
                       emit=lambda d: print(json.dumps(d), flush=True))
        if pg is not None:
            pg.destroy_process_group()
        return
    from cross_vendor_gradient_gb300 import workloads as _wl
    if _wl.WORKLOADS[args.workload].tensors:
        line = run_buckets_bench(args, world, rank, local, pg)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if pg is not None:
            pg.destroy_process_group()
        return
    if args.collective != "all_reduce":
        line = run_collective(args, world, rank, local, pg)
        if rank == 0:
            print(json.dumps(line), flush=True)
        if pg is not None:
            pg.destroy_process_group()
        return
    line, w, xs, codec = run_gb(args, world, rank, local, pg)
    # the recorded capture is of the kernel without error feedback
    line["roofline"]["traffic"] = None if args.ef else traffic_from_profiles(line["roofline"]["kernel"])
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, xs, codec)
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
