"""The fused halves for every dtype and op, and reduce_scatter's second half,
against the oracle bit for bit through the C ABI: gb_island_reduce_compress_op
(the codec path's encode or the exact path's island fold),
gb_decompress_island_broadcast on the exact path's payloads, and
gb_decompress_scatter on both paths, with ragged sizes and guard canaries
after every output."""
import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context, island_payload_bytes, payload_bytes, payload_scales_offset
from cross_vendor_gradient_gb300 import binding as B
from cross_vendor_gradient_gb300 import workloads as wl
from tests.gpu_util import assert_bits_equal, to_dev, to_host

pytestmark = pytest.mark.gpu

DTYPES = [np.float32, "bf16", np.float16, np.float64, np.int8, np.uint8, np.int32, np.int64]
TORCH = {np.float32: torch.float32, "bf16": torch.bfloat16, np.float16: torch.float16, np.float64: torch.float64,
         np.int8: torch.int8, np.uint8: torch.uint8, np.int32: torch.int32, np.int64: torch.int64}
GUARD = 256
SENTINEL = 0x5A


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def draw(dt, n, seed):
    rng = np.random.default_rng(seed)
    if dt == "bf16":
        return wl.to_bf16_bits((rng.standard_normal(n) * 10).astype(np.float32))
    if np.issubdtype(dt, np.integer):
        info = np.iinfo(dt)
        return rng.integers(info.min, info.max, n, dtype=dt, endpoint=True)
    x = (rng.standard_normal(n) * 10).astype(dt)
    x[rng.integers(0, n, max(1, n // 50))] = 0
    return x


def exact_ops(dt):
    """The ops that take the exact path for this dtype."""
    if dt in (np.float32, "bf16"):
        return ["max", "min"]
    return ["sum", "max", "min"] + (["avg"] if np.issubdtype(dt, np.floating) else [])


class Guarded:
    """count elements of tdt between two sentinel guards."""

    def __init__(self, count, tdt):
        es = torch.empty(0, dtype=tdt).element_size()
        self.nbytes = count * es
        self.raw = torch.full((2 * GUARD + self.nbytes,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(tdt)

    def intact(self):
        return bool(torch.all(self.raw[:GUARD] == SENTINEL)) and bool(torch.all(self.raw[GUARD + self.nbytes:]
                                                                               == SENTINEL))


def dev_inputs(xs, tdt):
    out = []
    for x in xs:
        g = Guarded(x.size, tdt)
        g.t.copy_(to_dev(x))
        out.append(g)
    return out


@pytest.mark.parametrize("dt", DTYPES, ids=str)
@pytest.mark.parametrize("sizes", [(1,), (2, 2), (2, 1, 3), (1, 1, 1, 1, 1, 1, 1, 1)])
def test_exact_halves_compose_to_all_reduce(dt, sizes):
    """The exact path's fold (every island's payload) and combine + broadcast,
    with a caller-moved bridge (each leader holds its own copies), give every
    rank the oracle's all_reduce, and write nothing outside the buffers."""
    W, I = sum(sizes), len(sizes)
    tdt = TORCH[dt]
    with Context(sizes) as ctx:
        for n in (1, 15, 16, 17, 1000, 70_001):
            for op in exact_ops(dt):
                xs = [draw(dt, n, 100 * n + r) for r in range(W)]
                ranks = dev_inputs(xs, tdt)
                P = island_payload_bytes(tdt, op, "none", 256, n)
                assert P > 0
                pays = [Guarded(P, torch.uint8) for _ in range(I)]
                ctx.island_reduce_compress_op([g.t for g in ranks], op, "none", 256, [p.t for p in pays])
                rows = [pays[j].t if j == g else pays[j].t.clone() for g in range(I) for j in range(I)]
                ctx.decompress_island_broadcast(rows, op, "none", 256, [g.t for g in ranks])
                torch.cuda.synchronize()
                want = orc.all_reduce(xs, sizes, op, "none", 256)
                for r in range(W):
                    assert_bits_equal(to_host(ranks[r].t), want[r], "%s %s n=%d %s rank %d" % (dt, sizes, n, op, r))
                for g in ranks + pays:
                    assert g.intact(), (dt, sizes, n, op)


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_op_encode_half_is_the_codec_encode(codec, block, dtype):
    """On the codec path gb_island_reduce_compress_op writes the bytes of
    gb_island_reduce_compress."""
    sizes = (2, 1, 3)
    w = wl.Workload("h", 41, sizes, dtype, "normal_1e-3_outliers", "sum", ())
    with Context(sizes) as ctx:
        for n in (1, 257, 40_003):
            xs = wl.host_rank_inputs(w, n=n)
            bufs = [to_dev(x) for x in xs]
            P = payload_bytes(codec, block, n)
            assert island_payload_bytes(bufs[0].dtype, "avg", codec, block, n) == P
            a = [torch.zeros(P, dtype=torch.uint8, device="cuda") for _ in sizes]
            b = [torch.ones(P, dtype=torch.uint8, device="cuda") for _ in sizes]
            ctx.island_reduce_compress(bufs, codec, block, a)
            ctx.island_reduce_compress_op(bufs, "avg", codec, block, b)
            torch.cuda.synchronize()
            # the written bytes: the codes, then the fp8 scales (padding between them is not written)
            cb = {"none": 4, "bf16": 2}.get(codec, 1)
            off = payload_scales_offset(codec, block, n)
            spans = [(0, n * cb)] + ([(off, P)] if codec in ("e4m3", "e5m2") else [])
            for i in range(len(sizes)):
                for lo, hi in spans:
                    assert_bits_equal(to_host(b[i])[lo:hi], to_host(a[i])[lo:hi], "%s n=%d island %d" % (codec, n, i))


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e4m3", 128),
                                         ("e5m2", 128)])
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (2, 1, 3), (4, 4)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decompress_scatter_is_reduce_scatter(codec, block, sizes, dtype):
    """Encode, a caller-moved bridge, then gb_decompress_scatter: rank r holds
    slice r of the oracle's reduce_scatter, bit for bit, and nothing outside
    its slice buffer is written.  Slices of a multiple of 8 elements take the
    vector path, the others the element-wise one."""
    W, I = sum(sizes), len(sizes)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    w = wl.Workload("h", 43, sizes, dtype, "normal_1e-3_outliers", "sum", ())
    with Context(sizes) as ctx:
        for m in (1, 7, 8, 33, 256, 1000, 8192 + 8):
            n = m * W
            xs = wl.host_rank_inputs(w, n=n)
            bufs = [to_dev(x) for x in xs]
            P = payload_bytes(codec, block, n)
            pays = [torch.empty(P, dtype=torch.uint8, device="cuda") for _ in range(I)]
            for op in ("sum", "avg"):
                ctx.island_reduce_compress(bufs, codec, block, pays)
                rows = [pays[j] if j == g else pays[j].clone() for g in range(I) for j in range(I)]
                outs = [Guarded(m, tdt) for _ in range(W)]
                ctx.decompress_scatter(rows, n, op, codec, block, [o.t for o in outs])
                torch.cuda.synchronize()
                want = orc.reduce_scatter(xs, sizes, op, codec, block)
                for r in range(W):
                    assert_bits_equal(to_host(outs[r].t), want[r], "%s %s m=%d %s rank %d" % (
                        codec, sizes, m, op, r))
                    assert outs[r].intact(), (codec, sizes, m, op, r)


@pytest.mark.parametrize("dt", DTYPES, ids=str)
@pytest.mark.parametrize("sizes", [(2, 2), (1, 3), (2, 1, 3)])
def test_exact_decompress_scatter_is_reduce_scatter(dt, sizes):
    W, I = sum(sizes), len(sizes)
    tdt = TORCH[dt]
    with Context(sizes) as ctx:
        for m in (1, 15, 16, 17, 4096 + 3):
            n = m * W
            for op in exact_ops(dt):
                xs = [draw(dt, n, 7 * n + r) for r in range(W)]
                ranks = dev_inputs(xs, tdt)
                P = island_payload_bytes(tdt, op, "none", 256, n)
                pays = [torch.empty(P, dtype=torch.uint8, device="cuda") for _ in range(I)]
                ctx.island_reduce_compress_op([g.t for g in ranks], op, "none", 256, pays)
                outs = [Guarded(m, tdt) for _ in range(W)]
                ctx.decompress_scatter(pays, n, op, "none", 256, [o.t for o in outs])
                torch.cuda.synchronize()
                want = orc.reduce_scatter(xs, sizes, op, "none", 256)
                for r in range(W):
                    assert_bits_equal(to_host(outs[r].t), want[r], "%s %s m=%d %s rank %d" % (dt, sizes, m, op, r))
                    assert outs[r].intact(), (dt, sizes, m, op, r)


def test_halves_refuse_what_all_reduce_refuses():
    with Context((2, 2)) as ctx:
        t = [torch.zeros(64, dtype=torch.int32, device="cuda") for _ in range(4)]
        p = [torch.zeros(256, dtype=torch.uint8, device="cuda") for _ in range(2)]
        for call in (lambda: ctx.island_reduce_compress_op(t, "avg", "none", 256, p),
                     lambda: ctx.decompress_scatter(p, 64, "avg", "none", 256, t),
                     lambda: ctx.decompress_island_broadcast(p, "avg", "none", 256, t)):
            with pytest.raises(Exception) as e:
                call()
            assert e.value.status == B.GB_ERR_UNSUPPORTED_OP
        with pytest.raises(Exception) as e:  # n not a multiple of W
            ctx.decompress_scatter(p, 63, "sum", "none", 256, t)
        assert e.value.status == B.GB_ERR_INVALID_ARG
        h = [torch.zeros(64, dtype=torch.float16, device="cuda") for _ in range(4)]
        with pytest.raises(Exception) as e:
            ctx.island_reduce_compress_op(h, "sum", "e4m3", 256, p)
        assert e.value.status == B.GB_ERR_UNSUPPORTED_CODEC
        assert island_payload_bytes(torch.int32, "avg", "none", 256, 10) == 0
        assert island_payload_bytes(torch.float16, "sum", "bf16", 256, 10) == 0
        assert island_payload_bytes(torch.float16, "sum", "none", 256, 10) == 40
        assert island_payload_bytes(torch.int8, "max", "e4m3", 256, 10) == 10
