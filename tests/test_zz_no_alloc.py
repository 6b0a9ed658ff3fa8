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


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("sizes", [(1,), (3,), (2, 2), (1, 2, 1)])
def test_noalloc_matches_the_oracle(dtype, sizes):
    """Every codec against the oracle directly, bit for bit: one rank, one
    island, two and three islands, ragged lengths (a short last fp8 block
    and a partial warp tile)."""
    import oracle
    dt = B.GB_F32 if dtype == "f32" else B.GB_BF16
    with Context(sizes) as ctx:
        for i, n in enumerate((1, 255, 1000, 65_537)):
            xs = _inputs(sizes, n, dtype, 80 + i)
            for codec, block in (("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128)):
                for op, opn in ((B.GB_SUM, "sum"), (B.GB_AVG, "avg")):
                    got = [to_dev(x) for x in xs]
                    st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in got], n, dt, op,
                                                 CODES[codec], block, torch.cuda.current_stream().cuda_stream)
                    assert st == B.GB_OK, B.gb_status_string(st)
                    torch.cuda.synchronize()
                    want = oracle.all_reduce(xs, sizes, opn, codec, block)
                    for r in range(len(xs)):
                        assert_bits_equal(to_host(got[r]), want[r], "%s n=%d %s %s rank %d" % (
                            sizes, n, codec, opn, r))


GUARD = 512
SENTINEL = 0xA5


def _guarded(n, tdtype):
    es = torch.empty(0, dtype=tdtype).element_size()
    raw = torch.full((2 * GUARD + n * es,), SENTINEL, dtype=torch.uint8, device="cuda")
    return raw, raw[GUARD:GUARD + n * es].view(tdtype)


@pytest.mark.parametrize("sizes,n,codec,block", [
    ((1, 1, 1, 1, 1, 1, 1, 1), 1_032_191, "e4m3", 256),  # 8 islands: 64 slots of 1 MiB fill the array
    ((1, 1, 1, 1, 1, 1, 1, 1), 1_001, "e5m2", 128),
    ((2, 1, 3), 40_003, "bf16", 256),
    ((4,), 5_001, "none", 256),
])
def test_noalloc_stays_in_bounds(sizes, n, codec, block):
    """Guard canaries before and after every rank buffer survive two calls,
    including the largest island count with slots that fill the device
    array, and the results equal gb_all_reduce's."""
    W = sum(sizes)
    with Context(sizes) as ctx:
        for call in range(2):
            g = [_guarded(n, torch.float32) for _ in range(W)]
            ref = []
            for r, (raw, t) in enumerate(g):
                gen = torch.Generator(device="cuda")
                gen.manual_seed(1000 * call + r)
                t.copy_(torch.randn(n, generator=gen, device="cuda"))
                ref.append(t.clone())
            st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for _, t in g], n, B.GB_F32, B.GB_SUM,
                                         CODES[codec], block, torch.cuda.current_stream().cuda_stream)
            assert st == B.GB_OK, B.gb_status_string(st)
            ctx.all_reduce(ref, "sum", codec, block)
            torch.cuda.synchronize()
            for r, (raw, t) in enumerate(g):
                assert bool(torch.all(raw[:GUARD] == SENTINEL)) and bool(torch.all(raw[-GUARD:] == SENTINEL)), r
                assert_bits_equal(to_host(t), to_host(ref[r]), "call %d rank %d" % (call, r))


def test_noalloc_refuses_a_device_other_than_the_bound_one():
    """A context bound to a device refuses a call made while another device
    is current, before anything is enqueued (simulated on one GPU with the
    host-side GB_INJECT_OTHER_DEVICE hook)."""
    n = 4096
    with Context((2, 2)) as ctx:
        bufs = [torch.full((n,), float(r + 1), device="cuda") for r in range(4)]
        ctx.all_reduce(bufs, "sum", "e4m3", 256)  # binds the context to this device
        torch.cuda.synchronize()
        before = [to_host(t).copy() for t in bufs]
        launches = B.gb_kernel_launch_count()
        assert B.gb_debug_inject(ctx.handle, B.GB_INJECT_OTHER_DEVICE) == B.GB_OK
        st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in bufs], n, B.GB_F32, B.GB_SUM,
                                     B.GB_CODEC_E4M3, 256, 0)
        assert st == B.GB_ERR_INVALID_ARG
        assert B.gb_kernel_launch_count() == launches
        torch.cuda.synchronize()
        for r in range(4):
            assert_bits_equal(to_host(bufs[r]), before[r], "rank %d" % r)
        assert ctx.status() == B.GB_OK  # an argument error, not sticky
        st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in bufs], n, B.GB_F32, B.GB_SUM,
                                     B.GB_CODEC_NONE, 256, 0)
        assert st == B.GB_OK
        torch.cuda.synchronize()
        assert np.all(to_host(bufs[0]) == 40.0)


def test_noalloc_size_limits():
    """The limit is I * I payload slots in the fixed device array: a
    three-island call one tile below it runs and matches gb_all_reduce bit
    for bit, one tile more is refused with nothing written, and a huge n is
    refused before any access."""
    sizes = (1, 1, 1)
    # e4m3 / 256: P = 260 * k bytes for n = 256 * k; 9 * round_up(P, 256) <= 64 MiB holds up to k = 28678
    n_fit = 256 * 28_678
    with Context(sizes) as ctx:
        xs = _inputs(sizes, n_fit + 256, "f32", 90)
        got = [to_dev(x[:n_fit]) for x in xs]
        ref = [to_dev(x[:n_fit]) for x in xs]
        st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in got], n_fit, B.GB_F32, B.GB_SUM,
                                     B.GB_CODEC_E4M3, 256, 0)
        assert st == B.GB_OK, B.gb_status_string(st)
        ctx.all_reduce(ref, "sum", "e4m3", 256)
        torch.cuda.synchronize()
        for r in range(3):
            assert_bits_equal(to_host(got[r]), to_host(ref[r]), "rank %d" % r)
        over = [to_dev(x) for x in xs]
        launches = B.gb_kernel_launch_count()
        st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in over], n_fit + 256, B.GB_F32, B.GB_SUM,
                                     B.GB_CODEC_E4M3, 256, 0)
        assert st == B.GB_ERR_TOO_LARGE
        # n far beyond the rank buffers: refused from the sizes alone, nothing read or written
        st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in over], 1 << 30, B.GB_F32, B.GB_SUM,
                                     B.GB_CODEC_E4M3, 256, 0)
        assert st == B.GB_ERR_TOO_LARGE
        st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in over], 1 << 39, B.GB_F32, B.GB_SUM,
                                     B.GB_CODEC_E4M3, 256, 0)
        assert st == B.GB_ERR_INVALID_ARG
        assert B.gb_kernel_launch_count() == launches
        torch.cuda.synchronize()
        for r in range(3):
            assert_bits_equal(to_host(over[r]), xs[r], "refused call wrote rank %d" % r)


def test_noalloc_takes_16_byte_views():
    """Rank buffers that start 16 bytes into their allocations (views inside
    a flat bucket): the same bits as gb_all_reduce on the same views, and
    the bytes around each view untouched."""
    sizes, n = (2, 2), 65_536 + 24
    xs = _inputs(sizes, n, "f32", 95)
    with Context(sizes) as ctx:
        raws, views, refs = [], [], []
        for x in xs:
            raw = torch.full((n + 16,), -7.0, device="cuda")
            v = raw[4:4 + n]  # 16 bytes in
            assert v.data_ptr() % 32 == 16
            v.copy_(to_dev(x))
            raws.append(raw)
            views.append(v)
            refs.append(to_dev(x))
        st = B.gb_all_reduce_noalloc(ctx.handle, [t.data_ptr() for t in views], n, B.GB_F32, B.GB_AVG,
                                     B.GB_CODEC_E4M3, 256, torch.cuda.current_stream().cuda_stream)
        assert st == B.GB_OK, B.gb_status_string(st)
        ctx.all_reduce(refs, "avg", "e4m3", 256)
        torch.cuda.synchronize()
        for r in range(4):
            assert_bits_equal(to_host(views[r]), to_host(refs[r]), "rank %d" % r)
            assert bool(torch.all(raws[r][:4] == -7.0)) and bool(torch.all(raws[r][4 + n:] == -7.0)), r
