"""Stream order with back-to-back launches and no host synchronisation in
between.  Every kernel of the library may be scheduled while the previous
kernel on the stream drains (programmatic dependent launch) and waits for
it before touching memory; these tests chain dependent work so that a
read or write that slipped ahead of that wait would change bits:
the library's kernels after its own (an accumulator carried from launch to
launch), after and before torch kernels on the same stream (inputs written,
results read and overwritten), and through the captured graphs of
repeated calls."""
import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context, payload_bytes, payload_scales_offset
from cross_vendor_gradient_gb300 import workloads as wl
from tests.gpu_util import assert_bits_equal, to_dev, to_host

pytestmark = pytest.mark.gpu

CODECS = [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def packed_payload(s, codec, block):
    """The oracle's encoding of s, laid out as a bridge payload: codes, then
    the float32 scales at the payload's scale offset."""
    n = s.size
    codes, scales = orc.encode(s, codec, block)
    buf = np.zeros(payload_bytes(codec, block, n), np.uint8)
    cb = codes.view(np.uint8)
    buf[:cb.size] = cb
    if scales.size:
        off = payload_scales_offset(codec, block, n)
        buf[off:off + 4 * scales.size] = scales.view(np.uint8)
    return (codes, scales), buf


@pytest.mark.parametrize("codec,block", CODECS)
def test_accumulator_chain(codec, block):
    """Twelve decompress-accumulate launches into one accumulator: each one
    reads what the previous launch wrote."""
    n = (1 << 20) + 13
    rng = np.random.default_rng(7)
    sums = [(rng.standard_normal(n) * 10.0 ** rng.integers(-3, 3)).astype(np.float32) for _ in range(12)]
    packed = [packed_payload(s, codec, block) for s in sums]
    pay = [torch.from_numpy(b).to("cuda") for _, b in packed]
    want = orc.bridge_total([p for p, _ in packed], codec, block, "sum", 1)
    with Context((1,)) as ctx:
        total = torch.empty(n, dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        for i, p in enumerate(pay):
            ctx.bridge_decompress_accumulate(p, n, codec, block, total, i > 0)
        torch.cuda.synchronize()
        assert_bits_equal(to_host(total), want, "accumulated over 12 launches")


@pytest.mark.parametrize("codec,block", CODECS)
@pytest.mark.parametrize("chunk", [2 << 20, 0])  # pipelined (graph replay from the third call) and plain
def test_torch_kernels_around_all_reduce(codec, block, chunk):
    """Per iteration on one stream: torch writes the inputs (an elementwise
    kernel), a torch kernel reads them, all_reduce runs in place, torch reads
    the result and then overwrites the buffers again.  Two input sets
    alternate, so a stale read or an early write changes the bits."""
    sizes = (2, 2)
    W = 4
    n = 3 * (1 << 20) + 77
    sets = []
    for k in range(2):
        w = wl.Workload("t", 60 + k, sizes, "f32", "normal_1e-3_outliers", "avg", ())
        sets.append(wl.host_rank_inputs(w, n=n))
    wants = [orc.all_reduce(xs, sizes, "avg", codec, block) for xs in sets]
    src = [[to_dev(x) for x in xs] for xs in sets]
    iters = 8
    with Context(sizes) as ctx:
        ctx.set_pipeline(chunk)
        bufs = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(W)]
        snaps, results = [], []
        torch.cuda.synchronize()
        for it in range(iters):
            k = it % 2
            for r in range(W):
                torch.mul(src[k][r], 1.0, out=bufs[r])          # kernel: write the inputs
            snaps.append([b * 1.0 for b in bufs])              # kernel: read them
            ctx.all_reduce(bufs, "avg", codec, block)
            results.append([b * 1.0 for b in bufs])            # kernel: read the result
            for r in range(W):
                bufs[r].fill_(float("nan"))                    # kernel: overwrite
        torch.cuda.synchronize()
        for it in range(iters):
            k = it % 2
            for r in range(W):
                assert_bits_equal(to_host(snaps[it][r]), sets[k][r], "inputs read before, iter %d rank %d" % (it, r))
                assert_bits_equal(to_host(results[it][r]), wants[k][r], "result iter %d rank %d" % (it, r))


@pytest.mark.parametrize("codec,block", CODECS)
def test_fused_halves_back_to_back(codec, block):
    """island_reduce_compress straight into decompress_island_broadcast, and
    the next call's encode straight after the previous decode, which
    rewrites the buffers the next encode reads."""
    sizes = (2, 3)
    W = 5
    n = (1 << 20) + 300
    w = wl.Workload("t", 71, sizes, "f32", "normal_1e-3_outliers", "sum", ())
    xs = wl.host_rank_inputs(w, n=n)
    # the sum of the sum: rank buffers carry the previous total into the next round
    want = [xs]
    for _ in range(4):
        want.append(orc.all_reduce(want[-1], sizes, "sum", codec, block))
    P = payload_bytes(codec, block, n)
    with Context(sizes) as ctx:
        bufs = [to_dev(x) for x in xs]
        pay = [torch.empty(P, dtype=torch.uint8, device="cuda") for _ in sizes]
        torch.cuda.synchronize()
        for _ in range(4):
            ctx.island_reduce_compress(bufs, codec, block, pay)
            ctx.decompress_island_broadcast(pay, "sum", codec, block, bufs)
        torch.cuda.synchronize()
        for r in range(W):
            assert_bits_equal(to_host(bufs[r]), want[-1][r], "after 4 rounds, rank %d" % r)
