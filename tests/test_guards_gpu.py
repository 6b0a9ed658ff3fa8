"""Out-of-bounds write checks (compute-sanitizer is not available on this
pool): every output buffer sits inside a larger allocation whose guard
regions before and after it hold a sentinel pattern; after each call the
guards must be intact.  Ragged sizes, every entry point that writes."""
import numpy as np
import pytest
import torch

from cross_vendor_gradient_gb300 import Context, payload_bytes
from cross_vendor_gradient_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
GUARD = 512  # bytes on each side (keeps the buffer 32-byte aligned)
SENTINEL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


class Guarded:
    """A device buffer of `count` elements of `dtype` between two guards."""

    def __init__(self, count, dtype):
        es = torch.empty(0, dtype=dtype).element_size()
        self.nbytes = count * es
        self.raw = torch.full((GUARD * 2 + self.nbytes,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype)

    def intact(self):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool(torch.all(head == SENTINEL)) and bool(torch.all(tail == SENTINEL))


def fill(g, seed):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    g.t.copy_(torch.randn(g.t.numel(), generator=gen, device="cuda").to(g.t.dtype))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (1, 2, 1), (3,)])
def test_collectives_stay_in_bounds(dtype, sizes):
    W = sum(sizes)
    with Context(sizes) as ctx:
        for n in (1, 7, 255, 257, 1000, 8 * W * 37 + W):
            n -= n % W if n >= W else 0
            n = max(n, W)
            for codec, block in (("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)):
                for chunk in (0, 1024):
                    ctx.set_pipeline(chunk, True)
                    bufs = [Guarded(n, dtype) for _ in range(W)]
                    for r, g in enumerate(bufs):
                        fill(g, r)
                    ctx.all_reduce([g.t for g in bufs], "avg", codec, block)
                    ctx.all_reduce([g.t for g in bufs], "sum", codec, block)  # second call (graph path)
                    outs = [Guarded(n // W, dtype) for _ in range(W)]
                    ctx.reduce_scatter([g.t for g in bufs], [o.t for o in outs], "sum", codec, block)
                    gath = [Guarded(n, dtype) for _ in range(W)]
                    ctx.all_gather([o.t for o in outs], [g.t for g in gath])
                    ctx.broadcast([g.t for g in bufs], W - 1)
                    torch.cuda.synchronize()
                    for g in bufs + outs + gath:
                        assert g.intact(), (sizes, n, codec, chunk)


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)])
def test_phase_blocks_stay_in_bounds(codec, block):
    sizes = (2, 1)
    with Context(sizes) as ctx:
        for n in (1, 9, 129, 257, 5001):
            ranks = [Guarded(n, torch.bfloat16) for _ in range(3)]
            for r, g in enumerate(ranks):
                fill(g, 10 + r)
            s = Guarded(n, torch.float32)
            ctx.island_reduce(0, [g.t for g in ranks[:2]], s.t)
            p = Guarded(payload_bytes(codec, block, n), torch.uint8)
            ctx.bridge_compress(s.t, codec, block, p.t)
            acc = Guarded(n, torch.float32)
            ctx.bridge_decompress_accumulate(p.t, n, codec, block, acc.t, False)
            ctx.bridge_decompress_accumulate(p.t, n, codec, block, acc.t, True)
            ctx.island_broadcast(0, acc.t, "avg", [g.t for g in ranks[:2]])
            torch.cuda.synchronize()
            for g in ranks + [s, p, acc]:
                assert g.intact(), (codec, n)


def test_host_entry_point_leaves_host_guards():
    sizes = (2, 2)
    n = 100_003
    with Context(sizes) as ctx:
        raw = [torch.full((n + 64,), 7.0).pin_memory() for _ in range(4)]
        host = [r[32:32 + n] for r in raw]
        for h in host:
            h.copy_(torch.randn(n))
        ctx.all_reduce_host(host, "sum", "e4m3", 256)
        torch.cuda.synchronize()
        for r in raw:
            assert torch.all(r[:32] == 7.0) and torch.all(r[32 + n:] == 7.0)


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)])
@pytest.mark.parametrize("sizes", [(2, 2), (2, 1, 3)])
def test_newer_entry_points_stay_in_bounds(codec, block, sizes):
    """The fused halves, the sharded-bridge policy, the bucket pipeline and
    error feedback write nothing outside their buffers."""
    W, I = sum(sizes), len(sizes)
    with Context(sizes) as ctx:
        ctx.set_pipeline(1024, True)
        for n in (1, 9, 257, 5001, 40003):
            ranks = [Guarded(n, torch.float32) for _ in range(W)]
            for r, g in enumerate(ranks):
                fill(g, 20 + r)
            pays = [Guarded(payload_bytes(codec, block, n), torch.uint8) for _ in range(I)]
            ctx.island_reduce_compress([g.t for g in ranks], codec, block, [p.t for p in pays])
            efres = [Guarded(n, torch.float32) for _ in range(I)]
            for g in efres:
                g.t.zero_()
            ctx.island_reduce_compress_ef([g.t for g in ranks], [g.t for g in efres], codec, block, [p.t for p in pays])
            ctx.decompress_island_broadcast([p.t for p in pays], "avg", codec, block, [g.t for g in ranks])
            ctx.set_sharded_bridge(True)
            for _ in range(2):
                ctx.all_reduce([g.t for g in ranks], "sum", codec, block)
            res = [Guarded(n, torch.float32) for _ in range(I)]
            for g in res:
                g.t.zero_()
            ctx.all_reduce_ef([g.t for g in ranks], [g.t for g in res], "sum", codec, block)
            ctx.set_sharded_bridge(False)
            numels = [n, 3, n // 2 + 1]
            buckets = [[Guarded(m, torch.bfloat16) for _ in range(W)] for m in numels]
            for b, row in enumerate(buckets):
                for r, g in enumerate(row):
                    fill(g, 100 * b + r)
            for _ in range(2):
                ctx.all_reduce_buckets([[g.t for g in row] for row in buckets], "sum", codec, block)
            torch.cuda.synchronize()
            for g in ranks + pays + res + efres + [g for row in buckets for g in row]:
                assert g.intact(), (codec, sizes, n)
