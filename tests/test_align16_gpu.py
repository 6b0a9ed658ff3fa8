"""Rank buffers that are 16-byte but not 32-byte aligned (for example a
float32 gradient view at an odd multiple of 4 elements inside a bucket):
every collective takes them and gives the oracle's bits, and nothing outside
the views is written.  Views sit at byte offset 16 (or, for some ranks, 32 or
48) inside larger allocations whose bytes around the view hold a sentinel."""
import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context, payload_bytes
from cross_vendor_gradient_gb300 import binding as B
from cross_vendor_gradient_gb300 import workloads as wl
from tests.gpu_util import assert_bits_equal, to_dev, to_host

pytestmark = pytest.mark.gpu
GUARD = 256
SENTINEL = 0xC3
CODECS = [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


class View:
    """count elements of tdt at byte offset `off` (16, 32 or 48) after a
    256-byte-aligned guard region, with a guard after it."""

    def __init__(self, count, tdt, off=16):
        es = torch.empty(0, dtype=tdt).element_size()
        self.nbytes = count * es
        self.lo = GUARD + off
        self.raw = torch.full((self.lo + self.nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[self.lo:self.lo + self.nbytes].view(tdt)
        assert self.t.data_ptr() % 16 == 0 and (self.t.data_ptr() % 32 != 0) == (off % 32 != 0)

    def intact(self):
        return bool(torch.all(self.raw[:self.lo] == SENTINEL)) and bool(torch.all(self.raw[self.lo + self.nbytes:]
                                                                                  == SENTINEL))


def views(xs, tdt, offs):
    out = []
    for x, off in zip(xs, offs):
        v = View(x.size, tdt, off)
        v.t.copy_(to_dev(x))
        out.append(v)
    return out


def offsets(W, mixed):
    # every rank at 16 mod 32, or a mix of 16-, 32- and 48-byte offsets
    return [(16, 32, 48)[r % 3] if mixed else 16 for r in range(W)]


@pytest.mark.parametrize("codec,block", CODECS)
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (2, 1, 3), (4,)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mixed", [False, True])
def test_all_reduce_and_reduce_scatter_on_16_byte_views(codec, block, sizes, dtype, mixed):
    W = sum(sizes)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    w = wl.Workload("a16", 61, sizes, dtype, "normal_1e-3_outliers", "sum", ())
    with Context(sizes) as ctx:
        for chunk in (0, 4096):  # one hop, and many pipeline chunks (graph replay on the second call)
            ctx.set_pipeline(chunk, True)
            for n in (1, 255, 257, 8 * W * 129, 40_000 * W + 8 * W):
                xs = wl.host_rank_inputs(w, n=n)
                ranks = views(xs, tdt, offsets(W, mixed))
                for op in ("sum", "avg"):
                    want = orc.all_reduce(xs, sizes, op, codec, block)
                    for call in range(2):  # the same buffers twice: the second call replays a graph
                        for v, x in zip(ranks, xs):
                            v.t.copy_(to_dev(x))
                        ctx.all_reduce([v.t for v in ranks], op, codec, block)
                        torch.cuda.synchronize()
                        for r in range(W):
                            assert_bits_equal(to_host(ranks[r].t), want[r], "AR %s %s n=%d %s rank %d call %d" % (
                                codec, sizes, n, op, r, call))
                            assert ranks[r].intact(), ("AR", codec, sizes, n, r)
                if n % W == 0:
                    m = n // W
                    ranks = views(xs, tdt, offsets(W, mixed))
                    outs = [View(m, tdt, off) for off in offsets(W, not mixed)]
                    ctx.reduce_scatter([v.t for v in ranks], [o.t for o in outs], "sum", codec, block)
                    torch.cuda.synchronize()
                    want = orc.reduce_scatter(xs, sizes, "sum", codec, block)
                    for r in range(W):
                        assert_bits_equal(to_host(outs[r].t), want[r], "RS %s %s n=%d rank %d" % (
                            codec, sizes, n, r))
                        assert outs[r].intact() and ranks[r].intact(), ("RS", codec, sizes, n, r)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("sizes", [(2, 2), (2, 1, 3)])
def test_gather_broadcast_halves_and_feedback_on_16_byte_views(dtype, sizes):
    W, I = sum(sizes), len(sizes)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    w = wl.Workload("a16", 62, sizes, dtype, "normal_1e-3_outliers", "sum", ())
    with Context(sizes) as ctx:
        for n in (3, 1000, 65_536 + 24):
            xs = wl.host_rank_inputs(w, n=n)
            # all_gather: 16-byte inputs and outputs
            ins = views(xs, tdt, offsets(W, True))
            outs = [View(W * n, tdt, 16) for _ in range(W)]
            ctx.all_gather([v.t for v in ins], [o.t for o in outs])
            # broadcast from the last rank
            bc = views(xs, tdt, offsets(W, False))
            ctx.broadcast([v.t for v in bc], W - 1)
            # the fused halves
            ranks = views(xs, tdt, offsets(W, False))
            P = payload_bytes("e4m3", 256, n)
            pays = [torch.empty(P, dtype=torch.uint8, device="cuda") for _ in range(I)]
            ctx.island_reduce_compress([v.t for v in ranks], "e4m3", 256, pays)
            ctx.decompress_island_broadcast(pays, "avg", "e4m3", 256, [v.t for v in ranks])
            # error feedback (residuals stay 32-byte aligned)
            efr = views(xs, tdt, offsets(W, True))
            res = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(I)]
            ctx.all_reduce_ef([v.t for v in efr], res, "sum", "e5m2", 128)
            torch.cuda.synchronize()
            gat = orc.all_gather(xs)
            for r in range(W):
                assert_bits_equal(to_host(outs[r].t), gat[r], "AG n=%d rank %d" % (n, r))
                assert_bits_equal(to_host(bc[r].t), xs[W - 1], "BC n=%d rank %d" % (n, r))
            want = orc.all_reduce(xs, sizes, "avg", "e4m3", 256)
            res_want = [np.zeros(n, np.float32) for _ in range(I)]
            want_ef = orc.all_reduce_ef(xs, sizes, res_want, "sum", "e5m2", 128)  # updates res_want
            for r in range(W):
                assert_bits_equal(to_host(ranks[r].t), want[r], "halves n=%d rank %d" % (n, r))
                assert_bits_equal(to_host(efr[r].t), want_ef[r], "EF n=%d rank %d" % (n, r))
            for i in range(I):
                assert_bits_equal(to_host(res[i]), res_want[i], "EF residual n=%d island %d" % (n, i))
            for v in ins + outs + bc + ranks + efr:
                assert v.intact(), (dtype, sizes, n)


@pytest.mark.parametrize("codec,block", CODECS)
def test_bucket_set_of_16_byte_views(codec, block):
    """A bucket set whose rank views start 16 bytes into their allocations,
    through the bucket pipeline and its graph replay."""
    sizes = (2, 2)
    W = 4
    numels = [1000, 3, 257 * 8 + 4, 70_000]
    w = wl.Workload("a16", 63, sizes, "f32", "normal_1e-3_outliers", "sum", ())
    with Context(sizes) as ctx:
        ctx.set_pipeline(8192, True)
        xs = [wl.host_rank_inputs(w, n=n) for n in numels]
        wants = [orc.all_reduce(x, sizes, "sum", codec, block) for x in xs]
        for mixed in (False, True):
            bk = [views(x, torch.float32, offsets(W, mixed)) for x in xs]
            for call in range(2):  # the same buffers twice: the second call replays the set's graph
                for row, x in zip(bk, xs):
                    for v, xr in zip(row, x):
                        v.t.copy_(to_dev(xr))
                ctx.all_reduce_buckets([[v.t for v in row] for row in bk], "sum", codec, block)
                torch.cuda.synchronize()
                for b, row in enumerate(bk):
                    for r in range(W):
                        assert_bits_equal(to_host(row[r].t), wants[b][r], "bucket %d rank %d call %d" % (b, r, call))
                        assert row[r].intact(), (codec, b, r, call)


def test_eight_byte_views_are_refused():
    with Context((2, 2)) as ctx:
        raw = [torch.zeros(1024 + 8, dtype=torch.float32, device="cuda") for _ in range(4)]
        bad = [r[2:2 + 1024] for r in raw]  # 8 bytes in: not 16-byte aligned
        with pytest.raises(Exception) as e:
            ctx.all_reduce(bad, "sum", "e4m3", 256)
        assert e.value.status == B.GB_ERR_MISALIGNED
        assert "16-byte" in B.gb_last_error_message(ctx.handle)
        assert ctx.status() == B.GB_OK
