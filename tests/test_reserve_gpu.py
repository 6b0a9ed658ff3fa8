"""gb_reserve's promise: after reserving n elements of a dtype and codec,
the single-buffer collectives on up to n elements allocate nothing.  An
injected allocation failure is armed after the reserve; any staging growth
would trip it (GB_ERR_ALLOC, sticky), so every call must succeed and leave
the injection pending.  The results are checked against the oracle too."""
import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context
from cross_vendor_gradient_gb300 import binding as B
from cross_vendor_gradient_gb300 import workloads as wl
from tests.gpu_util import assert_bits_equal, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def inputs(sizes, n, dtype, cid):
    w = wl.Workload("t", cid, tuple(sizes), dtype, "normal_1e-3_outliers", "sum", ())
    return wl.host_rank_inputs(w, n=n)


@pytest.mark.parametrize("sizes", [(2, 2), (2, 1, 3)])
@pytest.mark.parametrize("codec,block,dtype", [("e4m3", 256, "f32"), ("bf16", 256, "bf16"), ("none", 256, "f32"),
                                               ("e5m2", 128, "bf16")])
@pytest.mark.parametrize("chunk", [2 << 20, 4096, 0])
def test_no_allocation_after_reserve(sizes, codec, block, dtype, chunk):
    W = sum(sizes)
    n = 3 * (1 << 20) + 4 * W  # a multiple of W: reduce_scatter takes it whole
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    with Context(sizes) as ctx:
        ctx.set_pipeline(chunk)
        ctx.reserve(n, tdt, codec, block)
        ctx.debug_inject(B.GB_INJECT_ALLOC)
        for m in (n, n - 7 * W, 1000 * W, W):
            xs = inputs(sizes, m, dtype, cid=m % 89)
            bufs = [to_dev(x) for x in xs]
            ctx.all_reduce(bufs, "avg", codec, block)
            want = orc.all_reduce(xs, sizes, "avg", codec, block)
            ins = [to_dev(x) for x in xs]
            outs = [torch.empty(m // W, dtype=tdt, device="cuda") for _ in range(W)]
            ctx.reduce_scatter(ins, outs, "sum", codec, block)
            want_rs = orc.reduce_scatter(xs, sizes, "sum", codec, block)
            gathered = [torch.empty(m, dtype=tdt, device="cuda") for _ in range(W)]
            ctx.all_gather([x[:m // W] for x in ins], gathered)
            want_ag = orc.all_gather([x[:m // W] for x in xs])
            bc = [to_dev(x) for x in xs]
            ctx.broadcast(bc, W - 1)
            torch.cuda.synchronize()
            assert ctx.status() == B.GB_OK
            for r in range(W):
                assert_bits_equal(to_host(bufs[r]), want[r], "all_reduce m=%d rank %d" % (m, r))
                assert_bits_equal(to_host(outs[r]), want_rs[r], "reduce_scatter m=%d rank %d" % (m, r))
                assert_bits_equal(to_host(gathered[r]), want_ag[r], "all_gather m=%d rank %d" % (m, r))
                assert_bits_equal(to_host(bc[r]), xs[W - 1], "broadcast m=%d rank %d" % (m, r))
        # the injection is still armed: nothing grew.  Clear it.
        ctx.debug_inject(0)
        assert ctx.status() == B.GB_OK


def test_growth_trips_the_injection():
    """The converse, so the test above can fail: a call past the reserve
    must grow the staging and hits the armed failure."""
    sizes = (2, 2)
    with Context(sizes) as ctx:
        ctx.reserve(4096, torch.float32, "e4m3", 256)
        ctx.debug_inject(B.GB_INJECT_ALLOC)
        xs = inputs(sizes, 64 << 20, "f32", cid=3)
        bufs = [to_dev(x) for x in xs]
        with pytest.raises(Exception):
            ctx.all_reduce(bufs, "sum", "e4m3", 256)
        assert ctx.status() == B.GB_ERR_ALLOC
