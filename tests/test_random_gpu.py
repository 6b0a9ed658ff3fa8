"""Seeded random cases against the oracle, bit for bit: random island layouts,
lengths, dtypes, ops, codecs, pipeline chunk sizes and rank-view offsets (16
or 32 bytes into the allocation), through all_reduce (twice on the same
buffers: the second replays a graph where the policy captures one; every
third case under the sharded-bridge policy), reduce_scatter, all_gather,
broadcast, the host-buffer all_reduce (rows of one pinned block or separate
pinned tensors), and the same inputs as a bucket set of three through the
bucket all_reduce and reduce_scatter then all_gather of the set.  Each case is
reproducible from its index."""
import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context
from cross_vendor_gradient_gb300 import workloads as wl
from tests.gpu_util import assert_bits_equal, to_dev, to_host

pytestmark = pytest.mark.gpu

TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "f64": torch.float64,
         "i8": torch.int8, "u8": torch.uint8, "i32": torch.int32, "i64": torch.int64}
CODECS = [("none", 256), ("bf16", 256), ("e4m3", 256), ("e4m3", 128), ("e5m2", 128), ("e5m2", 256)]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def case(seed):
    rng = np.random.default_rng(10_000 + seed)
    I = int(rng.integers(1, 5))
    sizes = tuple(int(v) for v in rng.integers(1, 5, I))
    W = sum(sizes)
    if seed % 2 == 0:  # the codec path: float32 / bfloat16 SUM / AVG
        dtype = str(rng.choice(["f32", "bf16"]))
        op = str(rng.choice(["sum", "avg"]))
        codec, block = CODECS[int(rng.integers(0, len(CODECS)))]
    else:  # the exact path
        dtype = str(rng.choice(list(TORCH)))
        ops = (["max", "min"] if dtype in ("f32", "bf16") else
               ["sum", "max", "min"] + (["avg"] if dtype in ("f16", "f64") else []))
        op = str(rng.choice(ops))
        codec, block = "none", 256
    m = int(rng.integers(1, 20_000))
    n = m * W
    chunk = int(rng.choice([0, 1024, 4096, 65536, 2 << 20]))
    offs = [int(rng.choice([16, 32])) for _ in range(W)]
    return sizes, dtype, op, codec, block, n, chunk, offs


def draw(dtype, n, seed):
    rng = np.random.default_rng(seed)
    if dtype == "f32":
        return (rng.standard_normal(n) * 1e-2).astype(np.float32)
    if dtype == "bf16":
        return wl.to_bf16_bits((rng.standard_normal(n) * 1e-2).astype(np.float32))
    if dtype in ("f16", "f64"):
        return (rng.standard_normal(n) * 10).astype(np.float16 if dtype == "f16" else np.float64)
    npdt = {"i8": np.int8, "u8": np.uint8, "i32": np.int32, "i64": np.int64}[dtype]
    info = np.iinfo(npdt)
    return rng.integers(info.min, info.max, n, dtype=npdt, endpoint=True)


class View:
    def __init__(self, count, tdt, off):
        es = torch.empty(0, dtype=tdt).element_size()
        self.nbytes, self.lo = count * es, 256 + off
        self.raw = torch.full((self.lo + self.nbytes + 256,), 0x3C, dtype=torch.uint8, device="cuda")
        self.t = self.raw[self.lo:self.lo + self.nbytes].view(tdt)

    def intact(self):
        return bool(torch.all(self.raw[:self.lo] == 0x3C)) and bool(torch.all(self.raw[self.lo + self.nbytes:] == 0x3C))


@pytest.mark.parametrize("seed", range(150))
def test_random_case_matches_oracle(seed):
    sizes, dtype, op, codec, block, n, chunk, offs = case(seed)
    W = sum(sizes)
    tdt = TORCH[dtype]
    xs = [draw(dtype, n, 100 * seed + r) for r in range(W)]
    what = "seed %d: %s %s %s %s/%d n=%d chunk=%d" % (seed, sizes, dtype, op, codec, block, n, chunk)
    with Context(sizes) as ctx:
        ctx.set_pipeline(chunk, True)
        ctx.set_sharded_bridge(seed % 3 == 0)  # every third case under the sharded-bridge policy
        ranks = [View(n, tdt, o) for o in offs]
        want = orc.all_reduce(xs, sizes, op, codec, block)
        for call in range(2):
            for v, x in zip(ranks, xs):
                v.t.copy_(to_dev(x))
            ctx.all_reduce([v.t for v in ranks], op, codec, block)
            torch.cuda.synchronize()
            for r in range(W):
                assert_bits_equal(to_host(ranks[r].t), want[r], "AR %s call %d rank %d" % (what, call, r))
        # reduce_scatter then all_gather over the same ranks
        m = n // W
        ins = [View(n, tdt, o) for o in offs]
        outs = [View(m, tdt, o) for o in reversed(offs)]
        for v, x in zip(ins, xs):
            v.t.copy_(to_dev(x))
        ctx.reduce_scatter([v.t for v in ins], [o.t for o in outs], op, codec, block)
        torch.cuda.synchronize()
        want = orc.reduce_scatter(xs, sizes, op, codec, block)
        for r in range(W):
            assert_bits_equal(to_host(outs[r].t), want[r], "RS %s rank %d" % (what, r))
        gat = [View(n, tdt, o) for o in offs]
        ctx.all_gather([o.t for o in outs], [g.t for g in gat])
        torch.cuda.synchronize()
        want_ag = orc.all_gather([to_host(o.t) for o in outs])
        for r in range(W):
            assert_bits_equal(to_host(gat[r].t), want_ag[r], "AG %s rank %d" % (what, r))
        src = seed % W
        bc = [View(n, tdt, o) for o in offs]
        for v, x in zip(bc, xs):
            v.t.copy_(to_dev(x))
        ctx.broadcast([v.t for v in bc], src)
        torch.cuda.synchronize()
        for r in range(W):
            assert_bits_equal(to_host(bc[r].t), xs[src], "BC %s rank %d" % (what, r))
        for v in ranks + bc:
            assert v.intact(), what
        # the host-buffer entry points: the ranks as rows of one pinned [W, n] block (even seeds, the rows
        # entry point with its 2D staging copies) or as separate pinned tensors (odd seeds)
        want = orc.all_reduce(xs, sizes, op, codec, block)
        hx = [torch.from_numpy(x.view(np.int16) if dtype == "bf16" else x) for x in xs]
        if seed % 2 == 0:
            blk = torch.stack(hx).pin_memory()
            host = [blk[r] for r in range(W)]
        else:
            host = [h.clone().pin_memory() for h in hx]
        if dtype == "bf16":
            host = [h.view(torch.bfloat16) for h in host]
        ctx.all_reduce_host(host, op, codec, block)
        torch.cuda.synchronize()
        for r in range(W):
            got = host[r].view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else host[r].numpy()
            assert_bits_equal(got, want[r], "host %s rank %d" % (what, r))
        # the same inputs as a bucket set of three (bucket sizes multiples of W for reduce_scatter)
        if n >= 3 * W:  # (the sharded policy, where on, stays on: bucket sets keep one link under it)
            cut = [0, (n // 3) // W * W, (2 * n // 3) // W * W, n]
            xb = [[x[cut[b]:cut[b + 1]].copy() for x in xs] for b in range(3)]
            bk = [[View(cut[b + 1] - cut[b], tdt, o) for o in offs] for b in range(3)]
            for row, xr in zip(bk, xb):
                for v, x in zip(row, xr):
                    v.t.copy_(to_dev(x))
            ctx.all_reduce_buckets([[v.t for v in row] for row in bk], op, codec, block)
            torch.cuda.synchronize()
            for b in range(3):
                want = orc.all_reduce(xb[b], sizes, op, codec, block)
                for r in range(W):
                    assert_bits_equal(to_host(bk[b][r].t), want[r], "buckets %s bucket %d rank %d" % (what, b, r))
                    assert bk[b][r].intact(), what
            rs = [[View((cut[b + 1] - cut[b]) // W, tdt, o) for o in offs] for b in range(3)]
            for row, xr in zip(bk, xb):
                for v, x in zip(row, xr):
                    v.t.copy_(to_dev(x))
            ctx.reduce_scatter_buckets([[v.t for v in row] for row in bk], [[v.t for v in row] for row in rs], op,
                                       codec, block)
            ctx.all_gather_buckets([[v.t for v in row] for row in rs], [[v.t for v in row] for row in bk])
            torch.cuda.synchronize()
            for b in range(3):
                want = orc.all_reduce(xb[b], sizes, op, codec, block)  # RS then AG equals AR
                for r in range(W):
                    assert_bits_equal(to_host(bk[b][r].t), want[r], "RS+AG buckets %s bucket %d rank %d" % (
                        what, b, r))
                    assert bk[b][r].intact() and rs[b][r].intact(), what  # nothing written around the views
