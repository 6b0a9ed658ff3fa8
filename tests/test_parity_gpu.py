"""CUDA path vs the oracle, element by element and bit for bit, through the
C ABI, at sizes that span several warp tiles and codec blocks and end in a
ragged tail, for every codec, layout, rank dtype and op."""
import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context, payload_bytes, payload_scales_offset
from cross_vendor_gradient_gb300 import binding as B
from cross_vendor_gradient_gb300 import workloads as wl
from tests.gpu_util import assert_bits_equal, to_dev, to_host

pytestmark = pytest.mark.gpu

CODECS = [("none", 256), ("bf16", 256), ("e4m3", 256), ("e4m3", 128), ("e5m2", 128), ("e5m2", 256)]
LAYOUTS = [(1,), (1, 1), (2, 2), (1, 3), (4, 4), (2, 1, 3), (8,), (1, 1, 1, 1, 1, 1, 1, 1)]
SIZES = [1, 7, 8, 255, 256, 257, 1000, 4096 + 13, 65536 + 200]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def inputs(sizes, n, dtype="f32", dist="normal_1e-3_outliers", cid=11):
    w = wl.Workload("t", cid, tuple(sizes), dtype, dist, "sum", ())
    return wl.host_rank_inputs(w, n=n)


@pytest.mark.parametrize("codec,block", CODECS)
@pytest.mark.parametrize("sizes", LAYOUTS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_reduce_matches_oracle(codec, block, sizes, dtype):
    with Context(sizes) as ctx:
        for n in SIZES:
            for op in ("sum", "avg"):
                xs = inputs(sizes, n, dtype, cid=n % 97)
                bufs = [to_dev(x) for x in xs]
                ctx.all_reduce(bufs, op, codec, block)
                want = orc.all_reduce(xs, sizes, op, codec, block)
                torch.cuda.synchronize()
                for r, b in enumerate(bufs):
                    assert_bits_equal(to_host(b), want[r], "%s/%d %s n=%d %s rank %d" % (
                        codec, block, sizes, n, op, r))


@pytest.mark.parametrize("dist", ["uniform_pm1", "student_t3_1e-3", "normal_1e-3_zero_blocks", "integers"])
@pytest.mark.parametrize("codec,block", CODECS)
def test_all_reduce_distributions(dist, codec, block):
    sizes = (2, 2)
    n = 128 * 1000 + 77
    xs = inputs(sizes, n, "f32", dist, cid=5)
    with Context(sizes) as ctx:
        bufs = [to_dev(x) for x in xs]
        ctx.all_reduce(bufs, "sum", codec, block)
        want = orc.all_reduce(xs, sizes, "sum", codec, block)
        torch.cuda.synchronize()
        for r, b in enumerate(bufs):
            assert_bits_equal(to_host(b), want[r], "%s %s rank %d" % (dist, codec, r))


def test_special_blocks():
    """Zero, signed-zero, subnormal, huge and mixed-binade blocks."""
    B_ = 256
    n = B_ * 12 + 5
    rng = np.random.default_rng(3)
    base = rng.standard_normal(n).astype(np.float32)
    x0 = base.copy()
    x1 = (-base).copy()                      # block 0 cancels to exact zeros
    x0[B_:2 * B_] = -0.0
    x1[B_:2 * B_] = -0.0                     # all -0.0: sum -0.0
    x0[2 * B_:3 * B_] *= np.float32(1e-39)   # subnormal sums
    x1[2 * B_:3 * B_] = 0
    x0[3 * B_:4 * B_] *= np.float32(1e37)    # near the top of float32
    x1[3 * B_:4 * B_] = 0
    x0[4 * B_:5 * B_] = np.float32(448.0)
    x1[4 * B_:5 * B_] = np.float32(0.0)      # absmax exactly M
    x0[5 * B_] = np.float32(448.0 * 2.0 ** 10 * (1 + 2.0 ** -20))  # just above M * 2^10
    x0[6 * B_:7 * B_] = np.exp2(rng.integers(-60, 60, B_)).astype(np.float32)  # mixed binades
    xs = [x0, x1]
    x1[:B_] = -x0[:B_]
    for codec, block in CODECS:
        with Context((1, 1)) as ctx:
            bufs = [to_dev(x) for x in xs]
            ctx.all_reduce(bufs, "sum", codec, block)
            want = orc.all_reduce(xs, (1, 1), "sum", codec, block)
            torch.cuda.synchronize()
            for r, b in enumerate(bufs):
                assert_bits_equal(to_host(b), want[r], "special %s/%d rank %d" % (codec, block, r))


@pytest.mark.parametrize("codec,block", CODECS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_phase_blocks_match_oracle_and_compose_to_all_reduce(codec, block, dtype):
    """island_reduce, bridge_compress, bridge_decompress_accumulate and
    island_broadcast each match the oracle's step bit for bit, and their
    composition equals the fused all_reduce."""
    sizes = (2, 3)
    n = 3000 + 11
    xs = inputs(sizes, n, dtype, cid=23)
    _, mid = orc.rbb_total(xs, sizes, "avg", codec, block, intermediates=True)
    with Context(sizes) as ctx:
        bufs = [to_dev(x) for x in xs]
        first = [0, 2]
        payloads = []
        for i, K in enumerate(sizes):
            s = torch.empty(n, dtype=torch.float32, device="cuda")
            ctx.island_reduce(i, bufs[first[i]:first[i] + K], s)
            torch.cuda.synchronize()
            assert_bits_equal(to_host(s), mid["island_sums"][i], "island sum %d" % i)
            P = payload_bytes(codec, block, n)
            p = torch.empty(P, dtype=torch.uint8, device="cuda")
            ctx.bridge_compress(s, codec, block, p)
            torch.cuda.synchronize()
            ph = to_host(p)
            cd = orc.code_dtype(codec)
            cb = np.dtype(cd).itemsize
            assert_bits_equal(ph[:n * cb].view(cd), mid["codes"][i], "codes %d" % i)
            if codec in ("e4m3", "e5m2"):
                off = payload_scales_offset(codec, block, n)
                nb = orc.n_blocks(n, block)
                assert_bits_equal(ph[off:off + 4 * nb].view(np.float32), mid["scales"][i], "scales %d" % i)
                dec = orc.decode(mid["codes"][i], mid["scales"][i], codec, block)
            else:
                dec = orc.decode(mid["codes"][i], np.zeros(0, np.float32), codec, block)
            one = torch.empty(n, dtype=torch.float32, device="cuda")
            ctx.bridge_decompress_accumulate(p, n, codec, block, one, False)
            torch.cuda.synchronize()
            assert_bits_equal(to_host(one), dec, "decode %d" % i)
            payloads.append(p)
        total = torch.empty(n, dtype=torch.float32, device="cuda")
        for i, p in enumerate(payloads):
            ctx.bridge_decompress_accumulate(p, n, codec, block, total, i > 0)
        outs = [torch.empty_like(b) for b in bufs]
        for i, K in enumerate(sizes):
            ctx.island_broadcast(i, total, "avg", outs[first[i]:first[i] + K])
        ctx.all_reduce(bufs, "avg", codec, block)
        want = orc.all_reduce(xs, sizes, "avg", codec, block)
        torch.cuda.synchronize()
        for r in range(sum(sizes)):
            assert_bits_equal(to_host(outs[r]), want[r], "composed rank %d" % r)
            assert_bits_equal(to_host(bufs[r]), want[r], "fused rank %d" % r)


@pytest.mark.parametrize("codec,block", CODECS)
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (4, 4), (1, 2), (3,), (2, 1, 1)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_and_all_gather(codec, block, sizes, dtype):
    W = sum(sizes)
    with Context(sizes) as ctx:
        for m in (1, 5, 8, 300, 4096, 4099):  # slice lengths: 8 | m uses vector accesses
            n = W * m
            xs = inputs(sizes, n, dtype, cid=m % 13)
            ins = [to_dev(x) for x in xs]
            outs = [torch.empty(m, dtype=ins[0].dtype, device="cuda") for _ in range(W)]
            ctx.reduce_scatter(ins, outs, "avg", codec, block)
            want = orc.reduce_scatter(xs, sizes, "avg", codec, block)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(outs[r]), want[r], "RS %s m=%d rank %d" % (sizes, m, r))
                assert_bits_equal(to_host(ins[r]), xs[r], "RS input untouched %d" % r)
            gathered = [torch.empty(n, dtype=ins[0].dtype, device="cuda") for _ in range(W)]
            ctx.all_gather(outs, gathered)
            ar = orc.all_reduce(xs, sizes, "avg", codec, block)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(gathered[r]), ar[r], "RS then AG == AR rank %d" % r)


@pytest.mark.parametrize("sizes", [(1,), (1, 1), (2, 2), (1, 3), (3, 2, 1)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_gather_and_broadcast_exact(sizes, dtype):
    W = sum(sizes)
    with Context(sizes) as ctx:
        for m in (1, 3, 8, 1001, 4096):
            xs = inputs(sizes, m, dtype, cid=m % 7)
            ins = [to_dev(x) for x in xs]
            outs = [torch.empty(W * m, dtype=ins[0].dtype, device="cuda") for _ in range(W)]
            ctx.all_gather(ins, outs)
            want = orc.all_gather(xs)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(outs[r]), want[r], "AG m=%d rank %d" % (m, r))
            for src in range(W):
                bufs = [to_dev(x) for x in xs]
                ctx.broadcast(bufs, src)
                want = orc.broadcast(xs, src)
                torch.cuda.synchronize()
                for r in range(W):
                    assert_bits_equal(to_host(bufs[r]), want[r], "bcast src %d rank %d" % (src, r))


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)])
def test_all_reduce_host_buffers(codec, block):
    sizes = (2, 2)
    n = 70000 + 3
    xs = inputs(sizes, n, "f32", cid=31)
    with Context(sizes) as ctx:
        host = [torch.from_numpy(x.copy()).pin_memory() for x in xs]
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            ctx.all_reduce_host(host, "avg", codec, block)
        s.synchronize()
        want = orc.all_reduce(xs, sizes, "avg", codec, block)
        for r in range(4):
            assert_bits_equal(host[r].numpy(), want[r], "host rank %d" % r)


def test_bucketed_all_reduce_small_model():
    """A scaled-down gradient set (a handful of tensors of mixed sizes) with
    a small cap so that it spans several buckets, bf16 ranks, e5m2/128."""
    sizes = (2, 2)
    W = 4
    shapes = [(300, 7), (64,), (33, 33), (5,), (1000,), (128, 9), (2,)]
    numels = [wl.numel(s) for s in shapes]
    bo, off, bn = orc.bucket_plan(numels, 2, 4096, 8)
    assert len(bn) >= 3
    with Context(sizes) as ctx:
        buckets, hosts = [], []
        for b, nb_ in enumerate(bn):
            xs = inputs(sizes, int(nb_), "bf16", cid=40 + b)
            hosts.append(xs)
            buckets.append([to_dev(x) for x in xs])
        ctx.all_reduce_buckets(buckets, "sum", "e5m2", 128)
        torch.cuda.synchronize()
        for b in range(len(bn)):
            want = orc.all_reduce(hosts[b], sizes, "sum", "e5m2", 128)
            for r in range(W):
                assert_bits_equal(to_host(buckets[b][r]), want[r], "bucket %d rank %d" % (b, r))


def test_other_stream_and_phase_timing():
    sizes = (2, 2)
    n = 1 << 20
    xs = inputs(sizes, n, "f32", cid=77)
    with Context(sizes) as ctx:
        ctx.set_phase_timing(4)
        s = torch.cuda.Stream()
        bufs = [to_dev(x) for x in xs]
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            ctx.all_reduce(bufs, "sum", "e4m3", 256)
        ms = ctx.last_phase_times()
        s.synchronize()
        assert all(v > 0 for v in ms), ms
        want = orc.all_reduce(xs, sizes, "sum", "e4m3", 256)
        for r in range(4):
            assert_bits_equal(to_host(bufs[r]), want[r], "stream rank %d" % r)
        # a second call on the default stream is ordered after the first
        ctx.all_reduce(bufs, "sum", "none", 256)
        torch.cuda.synchronize()
        want2 = orc.all_reduce(want, sizes, "sum", "none", 256)
        assert_bits_equal(to_host(bufs[0]), want2[0], "second call")


def test_empty_inputs_are_noops():
    with Context((2, 2)) as ctx:
        bufs = [torch.zeros(16, device="cuda") for _ in range(4)]
        st = B.gb_all_reduce(ctx.handle, [b.data_ptr() for b in bufs], 0, 0, 0, 2, 256, 0)
        assert st == B.GB_OK
        st = B.gb_reduce_scatter(ctx.handle, [b.data_ptr() for b in bufs], [b.data_ptr() for b in bufs],
                                 0, 0, 0, 0, 256, 0)
        assert st == B.GB_OK


@pytest.mark.parametrize("codec,block", CODECS)
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (4, 4), (2, 1, 3), (1, 1, 1, 1, 1, 1, 1, 1)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pipelined_all_reduce_matches_oracle(codec, block, sizes, dtype):
    """The pipelined policy (chunked bridge on copy streams, replayed as a
    CUDA graph) gives the oracle's bits: three calls on the same buffers
    (direct, captured, replayed), several chunk sizes, ragged tails, and a
    size that needs more than the 32-chunk cap."""
    W = sum(sizes)
    with Context(sizes) as ctx:
        for chunk_bytes, n in ((1024, 5000), (4096, 256 * 37 + 5), (65536, 300_007), (1024, 40_000), (300, 70_001)):
            ctx.set_pipeline(chunk_bytes, True)
            xs = inputs(sizes, n, dtype, cid=n % 89)
            want = orc.all_reduce(xs, sizes, "avg", codec, block)
            bufs = [to_dev(x) for x in xs]
            src = [to_dev(x) for x in xs]
            for call in range(3):
                for b, s_ in zip(bufs, src):
                    b.copy_(s_)
                ctx.all_reduce(bufs, "avg", codec, block)
                torch.cuda.synchronize()
                for r in range(W):
                    assert_bits_equal(to_host(bufs[r]), want[r], "pipelined chunk=%d n=%d call %d rank %d" % (
                        chunk_bytes, n, call, r))
        ctx.set_pipeline(0, False)
        xs = inputs(sizes, 9999, dtype, cid=3)
        bufs = [to_dev(x) for x in xs]
        ctx.all_reduce(bufs, "sum", codec, block)
        want = orc.all_reduce(xs, sizes, "sum", codec, block)
        torch.cuda.synchronize()
        for r in range(W):
            assert_bits_equal(to_host(bufs[r]), want[r], "plain policy rank %d" % r)


def test_pipelined_graph_replay_timing_and_streams():
    """Phase marks are recorded for direct, captured and replayed calls, and
    a replay on another stream is ordered after the previous call."""
    sizes = (2, 2)
    n = 1 << 21
    xs = inputs(sizes, n, "f32", cid=91)
    want = orc.all_reduce(xs, sizes, "sum", "e4m3", 256)
    with Context(sizes) as ctx:
        ctx.set_pipeline(1 << 20, True)
        ctx.set_phase_timing(8)
        bufs = [to_dev(x) for x in xs]
        src = [to_dev(x) for x in xs]
        s2 = torch.cuda.Stream()
        for call in range(4):
            stream = s2 if call % 2 else torch.cuda.current_stream()
            with torch.cuda.stream(stream):
                for b, s_ in zip(bufs, src):
                    b.copy_(s_)
                ctx.all_reduce(bufs, "sum", "e4m3", 256)
            stream.synchronize()
            ms = ctx.last_phase_times()
            assert ms[0] > 0 and ms[1] > 0 and ms[2] > 0, (call, ms)
            for r in range(4):
                assert_bits_equal(to_host(bufs[r]), want[r], "call %d rank %d" % (call, r))
        assert len([ctx.phase_times(a) for a in range(4)]) == 4


@pytest.mark.parametrize("codec,block", CODECS)
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (2, 1, 3), (3,)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [0, 1024])
def test_error_feedback_matches_oracle_over_steps(codec, block, sizes, dtype, chunk):
    """gb_all_reduce_ef: outputs and residuals equal the oracle's bit for bit
    over consecutive steps on the same buffers (direct, captured, replayed)."""
    W, I = sum(sizes), len(sizes)
    n = 256 * 23 + 9
    with Context(sizes) as ctx:
        ctx.set_pipeline(chunk, True)
        res_h = [np.zeros(n, np.float32) for _ in range(I)]
        res_d = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(I)]
        bufs = [torch.empty(n, dtype=torch.float32 if dtype == "f32" else torch.bfloat16, device="cuda")
                for _ in range(W)]
        for step in range(4):
            xs = inputs(sizes, n, dtype, cid=200 + step)
            for b, x in zip(bufs, xs):
                b.copy_(to_dev(x))
            ctx.all_reduce_ef(bufs, res_d, "avg", codec, block)
            want = orc.all_reduce_ef(xs, sizes, res_h, "avg", codec, block)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(bufs[r]), want[r], "EF step %d rank %d" % (step, r))
            for i in range(I):
                assert_bits_equal(to_host(res_d[i]), res_h[i], "EF step %d residual %d" % (step, i))


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)])
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (2, 1, 3)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_reduce_host_pipelined(codec, block, sizes, dtype):
    """gb_all_reduce_host under the pipelined policy (staging, bridge and
    copy-back chunk by chunk): the oracle's bits on three calls with the same
    host buffers (direct, captured, replayed)."""
    W = sum(sizes)
    n = 256 * 97 + 5
    xs = inputs(sizes, n, dtype, cid=61)
    want = orc.all_reduce(xs, sizes, "avg", codec, block)
    with Context(sizes) as ctx:
        ctx.set_pipeline(2048, True)
        host = [torch.from_numpy(x.view(np.int16) if dtype == "bf16" else x).clone().pin_memory() for x in xs]
        if dtype == "bf16":
            host = [h.view(torch.bfloat16) for h in host]
        for call in range(3):
            for h, x in zip(host, xs):
                h.copy_(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if dtype == "bf16"
                        else torch.from_numpy(x))
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                ctx.all_reduce_host(host, "avg", codec, block)
            s.synchronize()
            for r in range(W):
                got = host[r].view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else host[r].numpy()
                assert_bits_equal(got, want[r], "host pipelined call %d rank %d" % (call, r))


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)])
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (4, 4), (2, 1, 3)])
def test_bucket_pipeline_matches_oracle(codec, block, sizes):
    """gb_all_reduce_buckets as one pipeline over all buckets' chunks (three-slot
    staging ring, one CUDA graph for the set): every bucket gets the
    oracle's bits, on three calls with the same buffers."""
    W = sum(sizes)
    numels = [5000, 0, 257, 40_000, 1, 9000, 31_337]
    with Context(sizes) as ctx:
        ctx.set_pipeline(4096, True)  # several chunks per bucket
        hosts = [inputs(sizes, n, "bf16", cid=300 + b) if n else [np.zeros(0, np.uint16)] * W
                 for b, n in enumerate(numels)]
        bufs = [[torch.empty(max(n, 1), dtype=torch.bfloat16, device="cuda")[:n] for _ in range(W)] for n in numels]
        wants = [orc.all_reduce(h, sizes, "sum", codec, block) if n else None for h, n in zip(hosts, numels)]
        for call in range(3):
            for b, n in enumerate(numels):
                for r in range(W):
                    if n:
                        bufs[b][r].copy_(to_dev(hosts[b][r]))
            ctx.all_reduce_buckets(bufs, "sum", codec, block)
            torch.cuda.synchronize()
            for b, n in enumerate(numels):
                for r in range(W):
                    if n:
                        assert_bits_equal(to_host(bufs[b][r]), wants[b][r], "call %d bucket %d rank %d" % (call, b, r))


@pytest.mark.parametrize("codec,block", CODECS)
@pytest.mark.parametrize("sizes", [(1,), (3,), (1, 1), (2, 2), (2, 1, 3), (1, 1, 1, 1, 1, 1, 1, 1)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_halves_match_oracle(codec, block, sizes, dtype):
    """island_reduce_compress writes every island's payload as the oracle
    encodes its island sum (codes and scales bit for bit); after a plain copy
    of the payloads, decompress_island_broadcast writes the oracle's total to
    every rank, which for two or more islands is the fused all_reduce."""
    W, I = sum(sizes), len(sizes)
    first = np.concatenate([[0], np.cumsum(sizes)]).astype(int)
    with Context(sizes) as ctx:
        for n in (1, 255, 256 * 9 + 17, 40000):
            for op in ("sum", "avg"):
                xs = inputs(sizes, n, dtype, cid=31 + n % 13)
                bufs = [to_dev(x) for x in xs]
                P = payload_bytes(codec, block, n)
                pay = [torch.empty(P, dtype=torch.uint8, device="cuda") for _ in range(I)]
                ctx.island_reduce_compress(bufs, codec, block, pay)
                # the caller's own bridge: every leader receives its own copy
                # of every other island's payload (row g, island order)
                rows = [pay[j] if j == g else pay[j].clone() for g in range(I) for j in range(I)]
                # (the shared-set form, I payloads, for AVG)
                ctx.decompress_island_broadcast(rows if op == "sum" else pay, op, codec, block, bufs)
                torch.cuda.synchronize()
                cd = orc.code_dtype(codec)
                cb = np.dtype(cd).itemsize
                enc = []
                for i in range(I):
                    s = orc.island_sum(xs[first[i]:first[i + 1]])
                    codes, scales = orc.encode(s, codec, block)
                    ph = to_host(pay[i])
                    assert_bits_equal(ph[:n * cb].view(cd), codes, "codes island %d n=%d" % (i, n))
                    if scales.size:
                        off = payload_scales_offset(codec, block, n)
                        assert_bits_equal(ph[off:off + 4 * scales.size].view(np.float32), scales,
                                          "scales island %d n=%d" % (i, n))
                    enc.append((codes, scales))
                t = orc.bridge_total(enc, codec, block, op, W)
                want = t if dtype == "f32" else orc.f32_to_bf16_array(t)
                for r in range(W):
                    assert_bits_equal(to_host(bufs[r]), want, "%s %s n=%d %s rank %d" % (
                        codec, sizes, n, op, r))
                if I > 1:
                    ref = orc.all_reduce(xs, sizes, op, codec, block)
                    assert_bits_equal(to_host(bufs[0]), ref[0], "equals all_reduce n=%d" % n)


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e4m3", 128),
                                         ("e5m2", 128)])
@pytest.mark.parametrize("sizes", [(2, 2), (4, 4), (3, 5), (2, 3, 4), (8, 8), (1, 3), (6,)])
@pytest.mark.parametrize("graphs", [True, False])
def test_sharded_bridge_matches_oracle(codec, block, sizes, graphs):
    """sharded-bridge policy: k = smallest island size segments, each over its
    own link; bit-identical to the oracle's sharded all_reduce (and so to
    reduce-bridge-broadcast), direct, captured and replayed."""
    W = sum(sizes)
    with Context(sizes) as ctx:
        ctx.set_pipeline(2 << 20, graphs)
        ctx.set_sharded_bridge(True)
        for n in (1, 255, 257, 5000, 40000):
            for dtype in ("f32", "bf16"):
                for op in ("sum", "avg"):
                    xs = inputs(sizes, n, dtype, cid=50 + n % 11)
                    want = orc.all_reduce_sharded(xs, sizes, op, codec, block)
                    bufs = [to_dev(x) for x in xs]
                    pristine = [b.clone() for b in bufs]
                    for call in range(3):  # direct, then captured, then replayed
                        for b, p in zip(bufs, pristine):
                            b.copy_(p)
                        ctx.all_reduce(bufs, op, codec, block)
                        torch.cuda.synchronize()
                        for r in range(W):
                            assert_bits_equal(to_host(bufs[r]), want[r], "%s %s n=%d %s %s call %d rank %d" % (
                                codec, sizes, n, dtype, op, call, r))


def test_sharded_bridge_timing_ef_and_other_calls():
    """Phase marks span every link; error feedback and the calls that keep
    one link (reduce_scatter, host buffers, buckets) stay bit-exact."""
    sizes, codec, block, n = (4, 4), "e4m3", 256, 70000
    W = sum(sizes)
    with Context(sizes) as ctx:
        ctx.set_sharded_bridge(True)
        ctx.set_phase_timing(4)
        xs = inputs(sizes, n, "f32", cid=61)
        for _ in range(2):
            bufs = [to_dev(x) for x in xs]
            ctx.all_reduce(bufs, "sum", codec, block)
        torch.cuda.synchronize()
        k1, br, k2 = ctx.phase_times(0)
        assert k1 > 0 and br > 0 and k2 > 0
        want = orc.all_reduce(xs, sizes, "sum", codec, block)
        for r in range(W):
            assert_bits_equal(to_host(bufs[r]), want[r], "timed rank %d" % r)
        ctx.set_phase_timing(0)
        # error feedback over three steps
        res_h = [np.zeros(n, np.float32) for _ in sizes]
        res_d = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in sizes]
        for step in range(3):
            xs = inputs(sizes, n, "f32", cid=70 + step)
            bufs = [to_dev(x) for x in xs]
            ctx.all_reduce_ef(bufs, res_d, "avg", codec, block)
            want = orc.all_reduce_ef(xs, sizes, res_h, "avg", codec, block)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(bufs[r]), want[r], "ef step %d rank %d" % (step, r))
            for i in range(len(sizes)):
                assert_bits_equal(to_host(res_d[i]), res_h[i], "ef residual %d" % i)
        # reduce_scatter and host buffers
        nr = 8 * 1000
        xs = inputs(sizes, nr, "f32", cid=81)
        outs = [torch.empty(nr // W, dtype=torch.float32, device="cuda") for _ in range(W)]
        ctx.reduce_scatter([to_dev(x) for x in xs], outs, "sum", codec, block)
        want = orc.reduce_scatter(xs, sizes, "sum", codec, block)
        host = [torch.from_numpy(x.copy()).pin_memory() for x in xs]
        ctx.all_reduce_host(host, "sum", codec, block)
        torch.cuda.synchronize()
        want_ar = orc.all_reduce(xs, sizes, "sum", codec, block)
        for r in range(W):
            assert_bits_equal(to_host(outs[r]), want[r], "rs rank %d" % r)
            assert_bits_equal(host[r].numpy(), want_ar[r], "host rank %d" % r)
        # bucketed, bucket by bucket under this policy
        numels = [5000, 0, 257, 40000]
        sets = [inputs(sizes, max(m, 1), "f32", cid=90 + b)[:W] for b, m in enumerate(numels)]
        buckets = [[to_dev(x[:m]) for x in xs_b] for xs_b, m in zip(sets, numels)]
        ctx.all_reduce_buckets(buckets, "sum", codec, block)
        torch.cuda.synchronize()
        for b, m in enumerate(numels):
            if m == 0:
                continue
            want = orc.all_reduce([x[:m] for x in sets[b]], sizes, "sum", codec, block)
            for r in range(W):
                assert_bits_equal(to_host(buckets[b][r]), want[r], "bucket %d rank %d" % (b, r))


@pytest.mark.parametrize("codec,block", CODECS)
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (4, 4), (2, 1, 3), (3,)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [1024, 6000])
def test_pipelined_reduce_scatter_and_all_gather(codec, block, sizes, dtype, chunk):
    """With small pipeline chunks, reduce_scatter's chunk decodes write the
    parts of the slices they cover (slices straddle chunk boundaries) and
    all_gather moves rank-block groups on the copy streams; both stay
    bit-identical to the oracle."""
    W = sum(sizes)
    with Context(sizes) as ctx:
        ctx.set_pipeline(chunk)
        for m in (1, 5, 8, 300, 4096, 4099, 20000):
            n = W * m
            xs = inputs(sizes, n, dtype, cid=17 + m % 13)
            ins = [to_dev(x) for x in xs]
            outs = [torch.empty(m, dtype=ins[0].dtype, device="cuda") for _ in range(W)]
            ctx.reduce_scatter(ins, outs, "avg", codec, block)
            want = orc.reduce_scatter(xs, sizes, "avg", codec, block)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(outs[r]), want[r], "RS %s m=%d rank %d" % (sizes, m, r))
                assert_bits_equal(to_host(ins[r]), xs[r], "RS input untouched %d" % r)
            gathered = [torch.empty(n, dtype=ins[0].dtype, device="cuda") for _ in range(W)]
            ctx.all_gather(outs, gathered)
            ar = orc.all_reduce(xs, sizes, "avg", codec, block)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(gathered[r]), ar[r], "RS then AG == AR m=%d rank %d" % (m, r))


@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (2, 1, 3), (4,)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pipelined_broadcast_is_exact(sizes, dtype):
    """With small pipeline chunks the broadcast's bridge hop moves the source
    in pieces; every rank still ends with the source's bits."""
    W = sum(sizes)
    with Context(sizes) as ctx:
        ctx.set_pipeline(1024)
        for n in (1, 255, 300, 4099, 70001):
            for src in sorted({0, W - 1, W // 2}):
                xs = inputs(sizes, n, dtype, cid=91 + n % 7)
                bufs = [to_dev(x) for x in xs]
                ctx.broadcast(bufs, src)
                want = orc.broadcast(xs, src)
                torch.cuda.synchronize()
                for r in range(W):
                    assert_bits_equal(to_host(bufs[r]), want[r], "bcast %s n=%d src=%d rank %d" % (sizes, n, src, r))


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)])
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (4, 4), (2, 1, 3), (3,)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bucket_sets_reduce_scatter_then_all_gather(codec, block, sizes, dtype):
    """gb_reduce_scatter_buckets and gb_all_gather_buckets (one pipeline, one
    graph per set): every bucket's slices are the oracle's reduce_scatter,
    and the gathered buffers its all_reduce; empty buckets are skipped;
    direct, captured and replayed calls agree."""
    W = sum(sizes)
    slices = [500, 0, 1, 3000, 64, 7919]  # elements per rank slice, per bucket
    with Context(sizes) as ctx:
        ctx.set_pipeline(4096)
        for op in ("sum", "avg"):
            xs = [inputs(sizes, max(m, 1) * W, dtype, cid=120 + b) for b, m in enumerate(slices)]
            ins = [[to_dev(x[:m * W]) for x in row] for row, m in zip(xs, slices)]
            for call in range(3):
                outs = [[torch.full((m,), 7.0, device="cuda").to(ins[0][0].dtype) for _ in range(W)] for m in slices]
                ctx.reduce_scatter_buckets(ins, outs, op, codec, block)
                gathered = [[torch.empty(m * W, dtype=ins[0][0].dtype, device="cuda") for _ in range(W)]
                            for m in slices]
                ctx.all_gather_buckets(outs, gathered)
                torch.cuda.synchronize()
                for b, m in enumerate(slices):
                    if m == 0:
                        continue
                    part = [x[:m * W] for x in xs[b]]
                    want_rs = orc.reduce_scatter(part, sizes, op, codec, block)
                    want_ar = orc.all_reduce(part, sizes, op, codec, block)
                    for r in range(W):
                        assert_bits_equal(to_host(outs[b][r]), want_rs[r], "RS bucket %d rank %d call %d" % (b, r, call))
                        assert_bits_equal(to_host(gathered[b][r]), want_ar[r], "AG bucket %d rank %d call %d" % (b, r, call))
                        assert_bits_equal(to_host(ins[b][r]), part[r], "inputs untouched")


def test_bucket_sets_exact_and_plain_paths():
    """MAX and the plain policy take the per-bucket loop and agree with the
    oracle too."""
    sizes = (2, 2)
    W = 4
    slices = [100, 0, 257]
    with Context(sizes) as ctx:
        for chunk, op in ((0, "sum"), (2 << 20, "max")):
            ctx.set_pipeline(chunk)
            xs = [inputs(sizes, max(m, 1) * W, "f32", cid=140 + b) for b, m in enumerate(slices)]
            ins = [[to_dev(x[:m * W]) for x in row] for row, m in zip(xs, slices)]
            outs = [[torch.empty(m, device="cuda") for _ in range(W)] for m in slices]
            ctx.reduce_scatter_buckets(ins, outs, op, "none", 256)
            gathered = [[torch.empty(m * W, device="cuda") for _ in range(W)] for m in slices]
            ctx.all_gather_buckets(outs, gathered)
            torch.cuda.synchronize()
            for b, m in enumerate(slices):
                if m == 0:
                    continue
                part = [x[:m * W] for x in xs[b]]
                want_rs = orc.reduce_scatter(part, sizes, op, "none", 256)
                want_ar = orc.all_reduce(part, sizes, op, "none", 256)
                for r in range(W):
                    assert_bits_equal(to_host(outs[b][r]), want_rs[r], "RS %s bucket %d rank %d" % (op, b, r))
                    assert_bits_equal(to_host(gathered[b][r]), want_ar[r], "AG %s bucket %d rank %d" % (op, b, r))


def test_two_contexts_on_two_threads_and_streams():
    """Two contexts, each driven by its own host thread on its own stream,
    run pipelined all_reduces, bucket sets and reduce_scatters at the same
    time; every result matches the oracle (no state is shared between
    contexts)."""
    import threading
    jobs = [((2, 2), "e4m3", 256, 31), ((1, 3), "bf16", 256, 32)]
    errors = []

    def work(sizes, codec, block, cid):
        try:
            W = sum(sizes)
            stream = torch.cuda.Stream()
            with Context(sizes) as ctx:
                ctx.set_pipeline(4096)
                for rep in range(4):
                    n = 20000 + 256 * rep
                    xs = inputs(sizes, n, "f32", cid=cid + rep)
                    with torch.cuda.stream(stream):
                        bufs = [to_dev(x) for x in xs]
                        ctx.all_reduce(bufs, "sum", codec, block, stream=stream)
                        outs = [torch.empty(n // W, device="cuda") for _ in range(W)]
                        ins = [to_dev(x[:n // W * W]) for x in xs]
                        ctx.reduce_scatter(ins, outs, "avg", codec, block, stream=stream)
                    stream.synchronize()
                    want = orc.all_reduce(xs, sizes, "sum", codec, block)
                    want_rs = orc.reduce_scatter([x[:n // W * W] for x in xs], sizes, "avg", codec, block)
                    for r in range(W):
                        assert_bits_equal(to_host(bufs[r]), want[r], "thread %s rank %d" % (sizes, r))
                        assert_bits_equal(to_host(outs[r]), want_rs[r], "thread %s RS rank %d" % (sizes, r))
        except BaseException as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=j) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        raise errors[0]


@pytest.mark.parametrize("codec,block", [("bf16", 256), ("e4m3", 256), ("e5m2", 128)])
@pytest.mark.parametrize("sizes", [(2, 2), (2, 1, 3), (3,)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bucket_set_error_feedback_over_steps(codec, block, sizes, dtype):
    """gb_all_reduce_buckets_ef (one pipeline, one graph per set) equals the
    oracle's all_reduce_ef bucket by bucket over several steps, outputs and
    every island's residual bit for bit."""
    I = len(sizes)
    numels = [3000, 0, 257, 20000]
    with Context(sizes) as ctx:
        ctx.set_pipeline(4096)
        res_h = [[np.zeros(m, np.float32) for _ in range(I)] for m in numels]
        res_d = [[torch.zeros(m, dtype=torch.float32, device="cuda") for _ in range(I)] for m in numels]
        for step in range(4):
            xs = [inputs(sizes, max(m, 1), dtype, cid=160 + 10 * step + b) for b, m in enumerate(numels)]
            bufs = [[to_dev(x[:m]) for x in row] for row, m in zip(xs, numels)]
            ctx.all_reduce_buckets_ef(bufs, res_d, "avg", codec, block)
            torch.cuda.synchronize()
            for b, m in enumerate(numels):
                if m == 0:
                    continue
                want = orc.all_reduce_ef([x[:m] for x in xs[b]], sizes, res_h[b], "avg", codec, block)
                for r in range(sum(sizes)):
                    assert_bits_equal(to_host(bufs[b][r]), want[r], "EF set step %d bucket %d rank %d" % (step, b, r))
                for i in range(I):
                    assert_bits_equal(to_host(res_d[b][i]), res_h[b][i], "EF set residual step %d bucket %d" % (step, b))


@pytest.mark.parametrize("codec,block", [("bf16", 256), ("e4m3", 256), ("e5m2", 128), ("none", 256)])
@pytest.mark.parametrize("sizes", [(2, 2), (1, 3), (2, 1, 3)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_encode_half_with_error_feedback(codec, block, sizes, dtype):
    """gb_island_reduce_compress_ef writes the oracle's error-feedback
    encoding of every island sum and updates the residuals bit for bit,
    over several steps."""
    W, I = sum(sizes), len(sizes)
    first = np.concatenate([[0], np.cumsum(sizes)]).astype(int)
    n = 256 * 7 + 33
    with Context(sizes) as ctx:
        res_h = [np.zeros(n, np.float32) for _ in range(I)]
        res_d = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(I)]
        P = payload_bytes(codec, block, n)
        cd = orc.code_dtype(codec)
        cb = np.dtype(cd).itemsize
        for step in range(3):
            xs = inputs(sizes, n, dtype, cid=180 + step)
            pay = [torch.empty(P, dtype=torch.uint8, device="cuda") for _ in range(I)]
            ctx.island_reduce_compress_ef([to_dev(x) for x in xs], res_d, codec, block, pay)
            torch.cuda.synchronize()
            for i in range(I):
                s = orc.island_sum(xs[first[i]:first[i + 1]])
                codes, scales = orc.encode_ef(s, res_h[i], codec, block)
                ph = to_host(pay[i])
                assert_bits_equal(ph[:n * cb].view(cd), codes, "EF codes step %d island %d" % (step, i))
                if scales.size:
                    off = payload_scales_offset(codec, block, n)
                    assert_bits_equal(ph[off:off + 4 * scales.size].view(np.float32), scales, "EF scales")
                assert_bits_equal(to_host(res_d[i]), res_h[i], "EF residual step %d island %d" % (step, i))
