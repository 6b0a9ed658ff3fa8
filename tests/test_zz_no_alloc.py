"""gb_all_reduce_noalloc, the all_reduce for callers that cannot allocate
memory when they sync gradients (its staging lives in fixed arrays inside
the library), against gb_all_reduce through the C ABI: the same bits on two
calls in a row (different sizes and codecs, so stale contents of the shared
arrays would show), and a clear refusal beyond the fixed size.

Kept in a file of its own, named to be collected last."""
import numpy as np
import pytest
import torch

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


def _inputs(sizes, n, dtype, cid):
    w = wl.Workload("noalloc", cid, tuple(sizes), dtype, "normal_1e-3_outliers", "sum", ())
    return wl.host_rank_inputs(w, n=n)


CODES = {"none": B.GB_CODEC_NONE, "bf16": B.GB_CODEC_BF16, "e4m3": B.GB_CODEC_E4M3, "e5m2": B.GB_CODEC_E5M2}


@pytest.mark.parametrize("sizes", [(2, 2), (1, 1), (1, 2, 1), (3,)])
def test_noalloc_matches_all_reduce_on_consecutive_calls(sizes):
    calls = [(6_553_600, "f32", B.GB_AVG, "e4m3", 256),   # a 25 MiB float32 bucket
             (100_003, "bf16", B.GB_SUM, "e5m2", 128),    # smaller, ragged: stale bytes would show
             (300_001, "f32", B.GB_SUM, "bf16", 256)]
    with Context(sizes) as ctx:
        for i, (n, dtype, op, codec, block) in enumerate(calls):
            xs = _inputs(sizes, n, dtype, 70 + i)
            ref = [to_dev(x) for x in xs]
            got = [to_dev(x) for x in xs]
            dt = B.GB_F32 if dtype == "f32" else B.GB_BF16
            st = B.gb_all_reduce(ctx.handle, [t.data_ptr() for t in ref], n, dt, op, CODES[codec], block,
                                 torch.cuda.current_stream().cuda_stream)
            assert st == B.GB_OK
            st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in got], n, dt, op, CODES[codec],
                                         block, torch.cuda.current_stream().cuda_stream)
            assert st == B.GB_OK, B.gb_status_string(st)
            torch.cuda.synchronize()
            for r in range(len(xs)):
                assert_bits_equal(to_host(got[r]), to_host(ref[r]), "call %d rank %d" % (i, r))


def test_noalloc_refuses_beyond_its_fixed_size():
    with Context((2, 2)) as ctx:
        n = B.GB_NOALLOC_DEVICE_BYTES // 16 + 1024  # 4 slots of 4n bytes no longer fit (codec none)
        bufs = [torch.ones(n, device="cuda") for _ in range(4)]
        st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in bufs], n, B.GB_F32, B.GB_SUM,
                                     B.GB_CODEC_NONE, 256, 0)
        assert st == B.GB_ERR_TOO_LARGE
        torch.cuda.synchronize()
        assert np.all(to_host(bufs[0]) == 1.0)
        # the same size fits compressed (about n bytes per payload)
        st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in bufs], n, B.GB_F32, B.GB_SUM,
                                     B.GB_CODEC_E4M3, 256, 0)
        assert st == B.GB_OK
        torch.cuda.synchronize()
        assert np.all(to_host(bufs[3]) == 4.0)
        assert ctx.status() == B.GB_OK
