"""gb_all_reduce_host_rows: host rank buffers that are the rows of one host
allocation, staged with one 2D copy per chunk and direction.  Bit for bit
against the oracle and against gb_all_reduce_host on the same rows, under
the pipelined policy (direct, captured, replayed) and the plain one, with
padded rows whose gaps must stay untouched, and its argument refusals."""
import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context
from cross_vendor_gradient_gb300 import binding as B
from cross_vendor_gradient_gb300 import workloads as wl
from tests.gpu_util import assert_bits_equal

pytestmark = pytest.mark.gpu

GUARD = -7.25


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def inputs(sizes, n, dtype, cid):
    w = wl.Workload("t", cid, tuple(sizes), dtype, "normal_1e-3_outliers", "sum", ())
    return wl.host_rank_inputs(w, n=n)


def rows_tensor(xs, dtype, pad):
    """One pinned [W, n + 2 * pad] tensor holding rank r in row r at column
    pad, the columns around it filled with GUARD; returns (block, rows)."""
    W, n = len(xs), xs[0].size
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    blk = torch.full((W, n + 2 * pad), GUARD, dtype=tdt).pin_memory()
    for r, x in enumerate(xs):
        src = torch.from_numpy(x) if dtype == "f32" else torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
        blk[r, pad:pad + n].copy_(src)
    return blk, [blk[r, pad:pad + n] for r in range(W)]


def host_bits(t):
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def refill(rows, xs, dtype):
    for h, x in zip(rows, xs):
        h.copy_(torch.from_numpy(x) if dtype == "f32" else torch.from_numpy(x.view(np.int16)).view(torch.bfloat16))


def guards_intact(blk, pad, n):
    if pad == 0:
        return True
    g = blk.float()
    return bool(torch.all(g[:, :pad] == GUARD)) and bool(torch.all(g[:, pad + n:] == GUARD))


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)])
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (2, 1, 3), (4, 4)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("pad", [0, 40])
def test_rows_pipelined_match_the_oracle(codec, block, sizes, dtype, pad):
    """Many small chunks: every chunk's staging and copy-back is one 2D copy.
    Three calls with the same rows (direct, captured, replayed)."""
    W = sum(sizes)
    n = 256 * 97 + 5
    xs = inputs(sizes, n, dtype, 71)
    want = orc.all_reduce(xs, sizes, "avg", codec, block)
    blk, rows = rows_tensor(xs, dtype, pad)
    eb = rows[0].element_size()
    with Context(sizes) as ctx:
        ctx.set_pipeline(2048, True)
        for call in range(3):
            refill(rows, xs, dtype)
            s = torch.cuda.Stream()
            st = B.gb_all_reduce_host_rows(ctx.handle, rows[0].data_ptr(), (n + 2 * pad) * eb, n,
                                           B.GB_F32 if dtype == "f32" else B.GB_BF16, B.GB_AVG,
                                           {"none": 0, "bf16": 1, "e4m3": 2, "e5m2": 3}[codec], block, s.cuda_stream)
            assert st == B.GB_OK, B.gb_status_string(st)
            s.synchronize()
            for r in range(W):
                assert_bits_equal(host_bits(rows[r]), want[r], "rows call %d rank %d" % (call, r))
            assert guards_intact(blk, pad, n), "a 2D copy wrote between the rows"


@pytest.mark.parametrize("codec,block", [("none", 256), ("e4m3", 256)])
@pytest.mark.parametrize("chunk", [0, 1 << 21])
def test_rows_and_pointer_entry_points_agree(codec, block, chunk):
    """The same rows through gb_all_reduce_host (W pointers, one copy per
    rank) and gb_all_reduce_host_rows, under the plain policy (chunk 0: one
    staging copy for the whole buffer) and the default pipelined one: the
    same bits, and the oracle's."""
    sizes = (2, 2)
    n = 3 * 65536 + 77
    xs = inputs(sizes, n, "f32", 72)
    want = orc.all_reduce(xs, sizes, "sum", codec, block)
    blk_a, rows_a = rows_tensor(xs, "f32", 8)
    blk_b, rows_b = rows_tensor(xs, "f32", 8)
    with Context(sizes) as ctx:
        ctx.set_pipeline(chunk, True)
        for call in range(2):
            refill(rows_a, xs, "f32")
            refill(rows_b, xs, "f32")
            ctx.all_reduce_host(rows_a, "sum", codec, block)  # rows of one storage: the rows entry point
            st = B.gb_all_reduce_host(ctx.handle, [t.data_ptr() for t in rows_b], n, B.GB_F32, B.GB_SUM,
                                      {"none": 0, "e4m3": 2}[codec], block,
                                      torch.cuda.current_stream().cuda_stream)
            assert st == B.GB_OK
            torch.cuda.synchronize()
            for r in range(4):
                assert_bits_equal(rows_a[r].numpy(), want[r], "rows call %d rank %d" % (call, r))
                assert_bits_equal(rows_b[r].numpy(), want[r], "pointers call %d rank %d" % (call, r))
            assert guards_intact(blk_a, 8, n) and guards_intact(blk_b, 8, n)


def test_a_2d_host_tensor_through_the_python_api():
    """Context.all_reduce_host takes a [W, n] host tensor as the W ranks."""
    sizes = (1, 2)
    n = 10_000 + 3
    xs = inputs(sizes, n, "f32", 73)
    want = orc.all_reduce(xs, sizes, "avg", "bf16", 256)
    blk = torch.from_numpy(np.stack(xs)).pin_memory()
    with Context(sizes) as ctx:
        ctx.all_reduce_host(blk, "avg", "bf16", 256)
        torch.cuda.synchronize()
    for r in range(3):
        assert_bits_equal(blk[r].numpy(), want[r], "rank %d" % r)


def test_rows_refusals_write_nothing():
    """Rows that would overlap (pitch below a row's bytes) and a NULL base
    are refused before anything is enqueued, and the context stays usable;
    n = 0 is a no-op; with one rank the pitch is ignored."""
    sizes = (2, 2)
    n = 4096 + 8
    xs = inputs(sizes, n, "f32", 74)
    blk, rows = rows_tensor(xs, "f32", 0)
    with Context(sizes) as ctx:
        launches = B.gb_kernel_launch_count()
        st = B.gb_all_reduce_host_rows(ctx.handle, rows[0].data_ptr(), n * 4 - 4, n, B.GB_F32, B.GB_SUM, 0, 256, 0)
        assert st == B.GB_ERR_INVALID_ARG
        st = B.gb_all_reduce_host_rows(ctx.handle, None, n * 4, n, B.GB_F32, B.GB_SUM, 0, 256, 0)
        assert st == B.GB_ERR_INVALID_ARG
        st = B.gb_all_reduce_host_rows(ctx.handle, rows[0].data_ptr(), n * 4, 0, B.GB_F32, B.GB_SUM, 0, 256, 0)
        assert st == B.GB_OK
        assert B.gb_kernel_launch_count() == launches
        torch.cuda.synchronize()
        for r in range(4):
            assert_bits_equal(rows[r].numpy(), xs[r], "refused call wrote rank %d" % r)
        assert ctx.status() == B.GB_OK
        ctx.all_reduce_host(rows, "sum", "none", 256)
        torch.cuda.synchronize()
        want = orc.all_reduce(xs, sizes, "sum", "none", 256)
        for r in range(4):
            assert_bits_equal(rows[r].numpy(), want[r], "rank %d after the refusals" % r)
    x1 = inputs((1,), n, "f32", 75)
    h = torch.from_numpy(x1[0].copy()).pin_memory()
    with Context((1,)) as ctx:
        st = B.gb_all_reduce_host_rows(ctx.handle, h.data_ptr(), 0, n, B.GB_F32, B.GB_SUM, 0, 256, 0)
        assert st == B.GB_OK
        torch.cuda.synchronize()
    assert_bits_equal(h.numpy(), x1[0], "one rank: identity")
