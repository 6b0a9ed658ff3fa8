"""Tiny cases by brute force, GPU against the oracle bit for bit: every
split of W = 1, 2, 3, 4 and 8 ranks into contiguous islands, every buffer
length 1 .. 300, every codec and op.

The 300 lengths run as one bucket set per call: each rank holds one flat
buffer with the buckets at 32-byte aligned offsets and a canary gap after
each, so one call exercises all ragged tails and every gap must keep its
bits.  The set runs as the bucket pipeline (more than one island), as
per-bucket calls of the plain policy, and with a 1 KiB pipeline chunk.
Separate loops cover one all_reduce call per length, and reduce_scatter
then all_gather over every length that W divides."""
import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context
from cross_vendor_gradient_gb300 import workloads as wl
from tests.gpu_util import assert_bits_equal, to_dev, to_host

pytestmark = pytest.mark.gpu

LENGTHS = list(range(1, 301))
CODECS = [("none", 256), ("bf16", 256), ("e4m3", 256), ("e4m3", 128), ("e5m2", 128), ("e5m2", 256)]
CANARY = {"f32": np.float32(-3.5), "bf16": np.uint16(0x7F7F)}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def compositions(W):
    """Every tuple of positive island sizes summing to W, in order."""
    if W == 0:
        return [()]
    return [(k,) + rest for k in range(1, W + 1) for rest in compositions(W - k)]


def test_compositions_count():
    for W in (1, 2, 3, 4, 8):
        c = compositions(W)
        assert len(c) == 2 ** (W - 1) and len(set(c)) == len(c) and all(sum(s) == W for s in c)


def carve(lengths, elem_bytes):
    """Offsets of each bucket in a flat rank buffer: 32-byte aligned, with
    at least one 32-byte canary gap after every bucket."""
    a = 32 // elem_bytes
    offs, pos = [], 0
    for n in lengths:
        offs.append(pos)
        pos += -(-n // a) * a + a
    return offs, pos


def draw(rng, n, dtype):
    x = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    if n > 4:
        x[rng.integers(0, n, max(1, n // 40))] *= np.float32(100.0)  # outliers
        x[rng.integers(0, n, max(1, n // 40))] = 0.0
    return wl.to_bf16_bits(x) if dtype == "bf16" else x


def flat_inputs(sizes, lengths, dtype, seed):
    W = sum(sizes)
    eb = 2 if dtype == "bf16" else 4
    offs, total = carve(lengths, eb)
    rng = np.random.default_rng(seed)
    flats = []
    for _ in range(W):
        f = np.full(total, CANARY[dtype])
        for o, n in zip(offs, lengths):
            f[o:o + n] = draw(rng, n, dtype)
        flats.append(f)
    return offs, flats


def run_set(ctx, sizes, lengths, dtype, op, codec, block, seed):
    W = sum(sizes)
    offs, flats = flat_inputs(sizes, lengths, dtype, seed)
    dev = [to_dev(f) for f in flats]
    bufs = [[dev[r][o:o + n] for r in range(W)] for o, n in zip(offs, lengths)]
    ctx.all_reduce_buckets(bufs, op, codec, block)
    want = [f.copy() for f in flats]
    for o, n in zip(offs, lengths):
        outs = orc.all_reduce([f[o:o + n] for f in flats], sizes, op, codec, block)
        for r in range(W):
            want[r][o:o + n] = outs[r]
    torch.cuda.synchronize()
    for r in range(W):
        assert_bits_equal(to_host(dev[r]), want[r], "%s %s %s %s/%d rank %d" % (sizes, dtype, op, codec, block, r))


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["set", "plain", "chunk1k"])
def test_all_reduce_every_split_and_length(W, dtype, mode):
    for li, sizes in enumerate(compositions(W)):
        with Context(sizes) as ctx:
            if mode == "plain":
                ctx.set_pipeline(0)
            elif mode == "chunk1k":
                ctx.set_pipeline(1024)
            for ci, (codec, block) in enumerate(CODECS):
                for op in ("sum", "avg"):
                    run_set(ctx, sizes, LENGTHS, dtype, op, codec, block, seed=1000 * W + 100 * li + 10 * ci)


@pytest.mark.parametrize("part", range(4))
def test_all_reduce_every_split_of_eight(part):
    """The 128 island splits of 8 ranks, a quarter per test, float32."""
    splits = compositions(8)[part::4]
    for li, sizes in enumerate(splits):
        with Context(sizes) as ctx:
            for ci, (codec, block) in enumerate([("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)]):
                for op in ("sum", "avg"):
                    run_set(ctx, sizes, LENGTHS, "f32", op, codec, block, seed=8000 + 37 * li + ci + part)


@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (1, 3), (2, 1, 1)])
@pytest.mark.parametrize("codec,block", [("none", 256), ("e4m3", 256), ("e5m2", 128)])
def test_all_reduce_one_call_per_length(sizes, codec, block):
    """gb_all_reduce itself (pipelined policy, graph capture on repeats) for
    every length, each buffer followed by a canary gap."""
    W = sum(sizes)
    with Context(sizes) as ctx:
        for n in LENGTHS:
            offs, flats = flat_inputs(sizes, [n], "f32", seed=n)
            dev = [to_dev(f) for f in flats]
            ctx.all_reduce([d[:n] for d in dev], "avg", codec, block)
            outs = orc.all_reduce([f[:n] for f in flats], sizes, "avg", codec, block)
            torch.cuda.synchronize()
            for r in range(W):
                want = flats[r].copy()
                want[:n] = outs[r]
                assert_bits_equal(to_host(dev[r]), want, "%s n=%d rank %d" % (sizes, n, r))


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_all_gather_every_split_and_length(W, dtype):
    """Bucket sets of every length 1 .. 300 that W divides: reduce_scatter
    matches the oracle's slices, and all_gather of them its all_reduce."""
    lengths = [n for n in LENGTHS if n % W == 0]
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    for li, sizes in enumerate(compositions(W)):
        with Context(sizes) as ctx:
            for ci, (codec, block) in enumerate(CODECS):
                op = ("sum", "avg")[ci % 2]
                offs, flats = flat_inputs(sizes, lengths, dtype, seed=2000 * W + 100 * li + ci)
                dev = [to_dev(f) for f in flats]
                ins = [[dev[r][o:o + n] for r in range(W)] for o, n in zip(offs, lengths)]
                outs = [[torch.empty(n // W, dtype=tdt, device="cuda") for _ in range(W)] for n in lengths]
                ctx.reduce_scatter_buckets(ins, outs, op, codec, block)
                gathered = [[torch.empty(n, dtype=tdt, device="cuda") for _ in range(W)] for n in lengths]
                ctx.all_gather_buckets(outs, gathered)
                torch.cuda.synchronize()
                for b, (o, n) in enumerate(zip(offs, lengths)):
                    part = [f[o:o + n] for f in flats]
                    rs = orc.reduce_scatter(part, sizes, op, codec, block)
                    ar = orc.all_reduce(part, sizes, op, codec, block)
                    for r in range(W):
                        what = "%s %s/%d n=%d rank %d" % (sizes, codec, block, n, r)
                        assert_bits_equal(to_host(outs[b][r]), rs[r], "RS " + what)
                        assert_bits_equal(to_host(gathered[b][r]), ar[r], "AG " + what)
                for r in range(W):
                    assert_bits_equal(to_host(dev[r]), flats[r], "inputs untouched rank %d" % r)
