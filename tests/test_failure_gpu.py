"""Failure handling on the GPU path, injected on the host only: a failed
bridge hop or staging allocation writes no rank buffer and makes the context
refuse every later call (sticky failure); argument errors are not sticky."""
import numpy as np
import pytest
import torch

from cross_vendor_gradient_gb300 import Context, GbError
from cross_vendor_gradient_gb300 import binding as B
from tests.gpu_util import to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _bufs(W, n, seed=0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return [torch.randn(n, device="cuda", generator=g) for _ in range(W)]


@pytest.mark.parametrize("call", ["all_reduce", "reduce_scatter", "all_gather", "broadcast"])
def test_injected_bridge_fault_is_sticky_and_writes_nothing(call):
    ctx = Context((2, 2))
    n = 4096
    bufs = _bufs(4, n, 1)
    before = [to_host(b).copy() for b in bufs]
    outs = [torch.full((n * 4 if call == "all_gather" else n // 4,), 7.0, device="cuda") for _ in range(4)]
    outs_before = [to_host(o).copy() for o in outs]
    ctx.debug_inject(B.GB_INJECT_BRIDGE)
    with pytest.raises(GbError) as e:
        if call == "all_reduce":
            ctx.all_reduce(bufs, "sum", "e4m3", 256)
        elif call == "reduce_scatter":
            ctx.reduce_scatter(bufs, outs, "sum", "bf16", 256)
        elif call == "all_gather":
            ctx.all_gather(bufs, outs)
        else:
            ctx.broadcast(bufs, 3)
    assert e.value.status == B.GB_ERR_BRIDGE
    torch.cuda.synchronize()
    for r in range(4):
        assert np.array_equal(to_host(bufs[r]), before[r])
        assert np.array_equal(to_host(outs[r]), outs_before[r])
    assert ctx.status() == B.GB_ERR_BRIDGE
    assert B.gb_last_error(ctx.handle) == B.GB_ERR_BRIDGE
    with pytest.raises(GbError) as e2:
        ctx.all_reduce(bufs, "sum", "none", 256)
    assert e2.value.status == B.GB_ERR_CONTEXT_FAILED
    assert B.gb_last_error(ctx.handle) == B.GB_ERR_CONTEXT_FAILED
    assert "injected" in B.gb_last_error_message(ctx.handle)  # the cause is kept
    with pytest.raises(GbError) as e3:
        ctx.island_reduce(0, bufs[:2], torch.empty(n, device="cuda"))
    assert e3.value.status == B.GB_ERR_CONTEXT_FAILED
    ctx.close()
    # a fresh context works
    with Context((2, 2)) as ok:
        ok.all_reduce(bufs, "sum", "none", 256)
        torch.cuda.synchronize()


def test_injected_alloc_failure_is_sticky():
    ctx = Context((1, 1))
    bufs = _bufs(2, 1000, 2)
    before = [to_host(b).copy() for b in bufs]
    ctx.debug_inject(B.GB_INJECT_ALLOC)
    with pytest.raises(GbError) as e:
        ctx.all_reduce(bufs, "avg", "bf16", 256)
    assert e.value.status == B.GB_ERR_ALLOC
    torch.cuda.synchronize()
    for r in range(2):
        assert np.array_equal(to_host(bufs[r]), before[r])
    with pytest.raises(GbError) as e2:
        ctx.broadcast(bufs, 0)
    assert e2.value.status == B.GB_ERR_CONTEXT_FAILED
    ctx.close()


def test_argument_errors_are_not_sticky_on_a_live_context():
    with Context((2, 2)) as ctx:
        bufs = _bufs(4, 512, 3)
        st = B.gb_all_reduce(ctx.handle, [b.data_ptr() + 4 for b in bufs], 100, 0, 0, 0, 256, 0)
        assert st == B.GB_ERR_MISALIGNED
        st = B.gb_all_reduce(ctx.handle, [b.data_ptr() for b in bufs], 512, 0, 0, 2, 100, 0)
        assert st == B.GB_ERR_UNSUPPORTED_CODEC
        assert ctx.status() == B.GB_OK
        ctx.all_reduce(bufs, "sum", "e4m3", 128)
        torch.cuda.synchronize()


def test_context_bound_to_its_device_and_destroy_waits():
    ctx = Context((1, 2))
    bufs = _bufs(3, 1 << 20, 4)
    ctx.all_reduce(bufs, "sum", "e5m2", 128)
    ctx.close()  # waits for the work, frees staging
    torch.cuda.synchronize()
    a = to_host(bufs[0])
    assert np.array_equal(a, to_host(bufs[2]))


@pytest.mark.parametrize("call", ["all_reduce", "reduce_scatter", "all_gather", "broadcast", "halves"])
def test_a_foreign_device_is_refused_before_anything_runs(call):
    """A context bound to a device refuses a call made while another device
    is current (simulated on one GPU with GB_INJECT_OTHER_DEVICE): an
    argument error, nothing launched or written, the context still usable."""
    ctx = Context((2, 2))
    n = 4096
    bufs = _bufs(4, n, 3)
    ctx.all_reduce([b.clone() for b in bufs], "sum", "none", 256)  # binds the context
    torch.cuda.synchronize()
    before = [to_host(b).copy() for b in bufs]
    outs = [torch.full((n * 4 if call == "all_gather" else n // 4,), 7.0, device="cuda") for _ in range(4)]
    pays = [torch.zeros(2 * n, dtype=torch.uint8, device="cuda") for _ in range(2)]  # >= the E4M3 payload
    launches = B.gb_kernel_launch_count()
    ctx.debug_inject(B.GB_INJECT_OTHER_DEVICE)
    with pytest.raises(GbError) as e:
        if call == "all_reduce":
            ctx.all_reduce(bufs, "sum", "e4m3", 256)
        elif call == "reduce_scatter":
            ctx.reduce_scatter(bufs, outs, "sum", "bf16", 256)
        elif call == "all_gather":
            ctx.all_gather(bufs, outs)
        elif call == "broadcast":
            ctx.broadcast(bufs, 3)
        else:
            ctx.island_reduce_compress(bufs, "e4m3", 256, pays)
    assert e.value.status == B.GB_ERR_INVALID_ARG
    assert "device" in B.gb_last_error_message(ctx.handle)
    assert B.gb_kernel_launch_count() == launches
    torch.cuda.synchronize()
    for r in range(4):
        assert np.array_equal(to_host(bufs[r]), before[r])
    assert ctx.status() == B.GB_OK
    ctx.all_reduce(bufs, "sum", "none", 256)  # the next call runs
    torch.cuda.synchronize()
    ctx.close()
