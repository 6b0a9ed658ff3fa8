"""The largest layouts the library accepts: 64 simulated ranks (the rank
limit) in 8 islands (the island limit), even and uneven, and 64 ranks in one
island.  Every collective, bit for bit against the oracle, with ragged sizes,
many pipeline chunks and a guard canary after every output."""
import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context
from cross_vendor_gradient_gb300 import binding as B
from cross_vendor_gradient_gb300 import workloads as wl
from tests.gpu_util import assert_bits_equal, to_dev, to_host

pytestmark = pytest.mark.gpu

MAX_LAYOUTS = [(8,) * 8, (1, 57, 1, 1, 1, 1, 1, 1), (64,)]
CODECS = [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)]
TORCH = {"f32": torch.float32, "bf16": torch.bfloat16}
GUARD = 64


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def test_limits_are_the_header_values():
    assert B.GB_MAX_RANKS == 64 and B.GB_MAX_ISLANDS == 8
    for sizes in MAX_LAYOUTS:
        assert sum(sizes) == B.GB_MAX_RANKS and len(sizes) <= B.GB_MAX_ISLANDS


def inputs(sizes, n, dtype="f32", cid=11):
    w = wl.Workload("t", cid, tuple(sizes), dtype, "normal_1e-3_outliers", "sum", ())
    return wl.host_rank_inputs(w, n=n)


def guarded(x: np.ndarray, dtype):
    """A device copy of x followed by GUARD canary elements; returns (raw, view)."""
    raw = torch.full((x.size + GUARD,), 7, dtype=TORCH[dtype], device="cuda")
    view = raw[:x.size]
    view.copy_(to_dev(x))
    return raw, view


def check_guard(raw, n, what):
    tail = raw[n:].float().cpu()
    assert bool((tail == 7).all()), "write past the end: " + what


@pytest.mark.parametrize("codec,block", CODECS)
@pytest.mark.parametrize("sizes", MAX_LAYOUTS, ids=["8x8", "1-57-1x6", "64"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [2 << 20, 1024])  # 1 KiB: the chunk cap of the pipeline
def test_all_reduce_max_ranks(codec, block, sizes, dtype, chunk):
    with Context(sizes) as ctx:
        ctx.set_pipeline(chunk)
        for n in (7, 4096 + 13, 65536 + 200):
            for op in ("sum", "avg"):
                xs = inputs(sizes, n, dtype, cid=n % 89)
                bufs = [guarded(x, dtype) for x in xs]
                ctx.all_reduce([v for _, v in bufs], op, codec, block)
                want = orc.all_reduce(xs, sizes, op, codec, block)
                torch.cuda.synchronize()
                for r, (raw, v) in enumerate(bufs):
                    what = "%s/%d %s n=%d %s rank %d" % (codec, block, sizes, n, op, r)
                    assert_bits_equal(to_host(v), want[r], what)
                    check_guard(raw, n, what)


@pytest.mark.parametrize("codec,block", [("none", 256), ("e4m3", 256)])
@pytest.mark.parametrize("sizes", MAX_LAYOUTS[:2], ids=["8x8", "1-57-1x6"])
def test_reduce_scatter_all_gather_max_ranks(codec, block, sizes):
    W = sum(sizes)
    with Context(sizes) as ctx:
        ctx.set_pipeline(4096)
        for m in (1, 8, 13, 300):
            n = W * m
            xs = inputs(sizes, n, "f32", cid=m)
            ins = [to_dev(x) for x in xs]
            outs = [guarded(np.zeros(m, np.float32), "f32") for _ in range(W)]
            ctx.reduce_scatter(ins, [v for _, v in outs], "avg", codec, block)
            want = orc.reduce_scatter(xs, sizes, "avg", codec, block)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(outs[r][1]), want[r], "RS m=%d rank %d" % (m, r))
                check_guard(outs[r][0], m, "RS m=%d rank %d" % (m, r))
            gathered = [guarded(np.zeros(n, np.float32), "f32") for _ in range(W)]
            ctx.all_gather([v for _, v in outs], [v for _, v in gathered])
            ar = orc.all_reduce(xs, sizes, "avg", codec, block)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(gathered[r][1]), ar[r], "RS then AG == AR m=%d rank %d" % (m, r))
                check_guard(gathered[r][0], n, "AG m=%d rank %d" % (m, r))


@pytest.mark.parametrize("sizes", MAX_LAYOUTS, ids=["8x8", "1-57-1x6", "64"])
def test_broadcast_max_ranks(sizes):
    W = sum(sizes)
    n = 4096 + 5
    xs = inputs(sizes, n, "bf16", cid=3)
    with Context(sizes) as ctx:
        for src in (0, 1, 31, W - 1):
            bufs = [guarded(x, "bf16") for x in xs]
            ctx.broadcast([v for _, v in bufs], src)
            want = orc.broadcast(xs, src)
            torch.cuda.synchronize()
            for r, (raw, v) in enumerate(bufs):
                assert_bits_equal(to_host(v), want[r], "bcast src %d rank %d" % (src, r))
                check_guard(raw, n, "bcast src %d rank %d" % (src, r))


@pytest.mark.parametrize("sizes", MAX_LAYOUTS, ids=["8x8", "1-57-1x6", "64"])
def test_exact_ops_max_ranks(sizes):
    """MAX over float32 and SUM over int32 (wrapping) through all_reduce,
    MIN over int8 through reduce_scatter."""
    W = sum(sizes)
    rng = np.random.default_rng(17)
    n = 1000 * W + 3 * W
    with Context(sizes) as ctx:
        ctx.set_pipeline(2048)
        cases = [("max", (rng.standard_normal((W, n)) * 10).astype(np.float32), torch.float32),
                 ("sum", rng.integers(-2**31, 2**31 - 1, (W, n), dtype=np.int32, endpoint=True), torch.int32)]
        for op, xs, tdt in cases:
            xs = list(xs)
            bufs = [torch.from_numpy(x.copy()).to("cuda") for x in xs]
            ctx.all_reduce(bufs, op)
            want = orc.all_reduce(xs, sizes, op)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(bufs[r]), want[r], "%s rank %d" % (op, r))
        xs = list(rng.integers(-128, 127, (W, n), dtype=np.int8, endpoint=True))
        ins = [torch.from_numpy(x.copy()).to("cuda") for x in xs]
        outs = [torch.empty(n // W, dtype=torch.int8, device="cuda") for _ in range(W)]
        ctx.reduce_scatter(ins, outs, "min")
        want = orc.reduce_scatter(xs, sizes, "min")
        torch.cuda.synchronize()
        for r in range(W):
            assert_bits_equal(to_host(outs[r]), want[r], "RS min rank %d" % r)


def test_host_buffers_max_ranks():
    sizes = (8,) * 8
    n = 20000 + 3
    xs = inputs(sizes, n, "f32", cid=41)
    with Context(sizes) as ctx:
        host = [torch.from_numpy(x.copy()).pin_memory() for x in xs]
        ctx.all_reduce_host(host, "avg", "e4m3", 256)
        torch.cuda.synchronize()
        want = orc.all_reduce(xs, sizes, "avg", "e4m3", 256)
        for r in range(64):
            assert_bits_equal(host[r].numpy(), want[r], "host rank %d" % r)


@pytest.mark.parametrize("sizes", MAX_LAYOUTS[:2], ids=["8x8", "1-57-1x6"])
def test_bucket_sets_max_ranks(sizes):
    """gb_all_reduce_buckets, then the reduce_scatter / all_gather bucket
    sets, on buckets padded to a multiple of W (and one empty bucket)."""
    W = sum(sizes)
    numels = [W * 3, 0, W * 700 + 0, W * 41]
    with Context(sizes) as ctx:
        ctx.set_pipeline(4096, True)
        hosts = [inputs(sizes, n, "bf16", cid=500 + b) if n else [np.zeros(0, np.uint16)] * W
                 for b, n in enumerate(numels)]
        bufs = [[torch.empty(max(n, 1), dtype=torch.bfloat16, device="cuda")[:n] for _ in range(W)]
                for n in numels]
        for b, n in enumerate(numels):
            for r in range(W):
                if n:
                    bufs[b][r].copy_(to_dev(hosts[b][r]))
        ctx.all_reduce_buckets(bufs, "sum", "e4m3", 256)
        torch.cuda.synchronize()
        for b, n in enumerate(numels):
            if not n:
                continue
            want = orc.all_reduce(hosts[b], sizes, "sum", "e4m3", 256)
            for r in range(W):
                assert_bits_equal(to_host(bufs[b][r]), want[r], "AR bucket %d rank %d" % (b, r))
        ins = [[to_dev(h) for h in hosts[b]] if n else [torch.empty(0, dtype=torch.bfloat16, device="cuda")] * W
               for b, n in enumerate(numels)]
        outs = [[torch.empty(n // W, dtype=torch.bfloat16, device="cuda") for _ in range(W)] for n in numels]
        ctx.reduce_scatter_buckets(ins, outs, "avg", "bf16", 256)
        gathered = [[torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(W)] for n in numels]
        ctx.all_gather_buckets(outs, gathered)
        torch.cuda.synchronize()
        for b, n in enumerate(numels):
            if not n:
                continue
            rs = orc.reduce_scatter(hosts[b], sizes, "avg", "bf16", 256)
            ar = orc.all_reduce(hosts[b], sizes, "avg", "bf16", 256)
            for r in range(W):
                assert_bits_equal(to_host(outs[b][r]), rs[r], "RS bucket %d rank %d" % (b, r))
                assert_bits_equal(to_host(gathered[b][r]), ar[r], "AG bucket %d rank %d" % (b, r))
