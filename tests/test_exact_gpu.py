"""The exact path on the GPU: MAX / MIN for every dtype and SUM / AVG for
float16, float64 and the integers, bit for bit against the oracle, through
all_reduce, reduce_scatter and all_gather, ragged sizes, with a guard
canary after every output."""
import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context
from tests.gpu_util import assert_bits_equal, to_dev, to_host

pytestmark = pytest.mark.gpu

DTYPES = [np.float32, "bf16", np.float16, np.float64, np.int8, np.uint8, np.int32, np.int64]
TORCH = {np.float32: torch.float32, "bf16": torch.bfloat16, np.float16: torch.float16, np.float64: torch.float64,
         np.int8: torch.int8, np.uint8: torch.uint8, np.int32: torch.int32, np.int64: torch.int64}


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def draw(dt, n, seed):
    rng = np.random.default_rng(seed)
    if dt == "bf16":
        from cross_vendor_gradient_gb300 import workloads as wl
        return wl.to_bf16_bits((rng.standard_normal(n) * 10).astype(np.float32))
    if np.issubdtype(dt, np.integer):
        info = np.iinfo(dt)
        x = rng.integers(info.min, info.max, n, dtype=dt, endpoint=True)
        return x
    x = (rng.standard_normal(n) * 10).astype(dt)
    x[rng.integers(0, n, max(1, n // 50))] = 0  # zeros (and, after negation, -0) appear
    return x


def ops_for(dt):
    return ["sum", "max", "min"] + (["avg"] if dt == "bf16" or np.issubdtype(dt, np.floating) else [])


def guarded(n, tdt):
    raw = torch.full((n + 64,), 0, dtype=tdt, device="cuda")
    return raw, raw[:n]


@pytest.mark.parametrize("dt", DTYPES, ids=str)
@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (2, 1, 3), (3,)])
@pytest.mark.parametrize("chunk", [2 << 20, 1024])  # 1 KiB: many pipeline chunks, slices straddling them
def test_exact_collectives_match_oracle(dt, sizes, chunk):
    W = sum(sizes)
    with Context(sizes) as ctx:
        ctx.set_pipeline(chunk)
        for n in (1, 15, 16, 17, 1000, 4096 * W + 3 * W, 70_001):
            n -= n % W if n >= W else 0
            n = max(n, W)
            for op in ops_for(dt):
                if dt in (np.float32, "bf16") and op in ("sum", "avg"):
                    continue  # the codec path, covered elsewhere
                xs = [draw(dt, n, 17 * r + n % 7) for r in range(W)]
                if dt not in ("bf16",) and not np.issubdtype(dt, np.integer):
                    xs[1][:5] = -xs[0][:5]  # +0 / -0 ties
                ins = [to_dev(x) for x in xs]
                raws, outs = zip(*[guarded(n, ins[0].dtype) for _ in range(W)])
                for o, i in zip(outs, ins):
                    o.copy_(i)
                # MAX / MIN and integers ignore the codec; float16 / float64 sums accept none only
                ignored = op in ("max", "min") or dt == "bf16" or np.issubdtype(dt, np.integer)
                ctx.all_reduce(list(outs), op, "e4m3" if ignored else "none", 256)
                want = orc.all_reduce(xs, sizes, op)
                torch.cuda.synchronize()
                for r in range(W):
                    assert_bits_equal(to_host(outs[r]), want[r], "%s %s %s n=%d rank %d" % (dt, op, sizes, n, r))
                    assert torch.all(raws[r][n:] == 0)
                rs_raw, rs_out = zip(*[guarded(n // W, ins[0].dtype) for _ in range(W)])
                ctx.reduce_scatter(ins, list(rs_out), op, "none", 256)
                want_rs = orc.reduce_scatter(xs, sizes, op)
                torch.cuda.synchronize()
                for r in range(W):
                    assert_bits_equal(to_host(rs_out[r]), want_rs[r], "RS %s %s n=%d rank %d" % (dt, op, n, r))
                    assert torch.all(rs_raw[r][n // W:] == 0)
                ag = [torch.empty(n, dtype=ins[0].dtype, device="cuda") for _ in range(W)]
                ctx.all_gather(list(rs_out), ag)
                torch.cuda.synchronize()
                for r in range(W):
                    assert_bits_equal(to_host(ag[r]), want[r], "RS then AG %s %s rank %d" % (dt, op, r))


def test_exact_path_refusals():
    from cross_vendor_gradient_gb300 import GbError
    from cross_vendor_gradient_gb300 import binding as B
    with Context((1, 1)) as ctx:
        ints = [torch.zeros(64, dtype=torch.int32, device="cuda") for _ in range(2)]
        with pytest.raises(GbError) as e:
            ctx.all_reduce(ints, "avg")
        assert e.value.status == B.GB_ERR_UNSUPPORTED_OP
        f64 = [torch.zeros(64, dtype=torch.float64, device="cuda") for _ in range(2)]
        with pytest.raises(GbError) as e:
            ctx.all_reduce(f64, "sum", "bf16")
        assert e.value.status == B.GB_ERR_UNSUPPORTED_CODEC
        ctx.all_reduce(f64, "sum", "none")
        torch.cuda.synchronize()
        assert ctx.status() == B.GB_OK


@pytest.mark.parametrize("dt", [np.float16, np.float64, np.int8, np.uint8, np.int32, np.int64, np.float32], ids=str)
@pytest.mark.parametrize("sizes", [(2, 2), (2, 1, 3)])
def test_exact_bucket_sets_and_host_buffers(dt, sizes):
    """The exact path through the bucket pipelines (all_reduce and
    reduce_scatter sets, one graph per set) and the host-buffer pipeline,
    bit for bit against the oracle."""
    W = sum(sizes)
    numels = [1000 * W, 0, 37 * W, 5000 * W]
    with Context(sizes) as ctx:
        ctx.set_pipeline(4096)
        for op in (["sum", "max"] if dt != np.float32 else ["max", "min"]):
            for call in range(2):  # direct, then captured
                xs = [[draw(dt, max(m, 1), 300 + 17 * r + b)[:m] for r in range(W)] for b, m in enumerate(numels)]
                bufs = [[to_dev(x) for x in row] for row in xs]
                ctx.all_reduce_buckets(bufs, op, "none", 256)
                outs = [[torch.empty(m // W, dtype=TORCH[dt], device="cuda") for _ in range(W)] for m in numels]
                ins = [[to_dev(x) for x in row] for row in xs]
                ctx.reduce_scatter_buckets(ins, outs, op, "none", 256)
                torch.cuda.synchronize()
                for b, m in enumerate(numels):
                    if m == 0:
                        continue
                    want = orc.all_reduce(xs[b], sizes, op)
                    want_rs = orc.reduce_scatter(xs[b], sizes, op)
                    for r in range(W):
                        assert_bits_equal(to_host(bufs[b][r]), want[r], "%s %s bucket %d rank %d" % (dt, op, b, r))
                        assert_bits_equal(to_host(outs[b][r]), want_rs[r], "RS %s %s bucket %d rank %d" % (dt, op, b, r))
            n = 7000 * W + 3
            xs = [draw(dt, n, 400 + r) for r in range(W)]
            host = [torch.from_numpy(x.copy()).pin_memory() for x in xs]
            ctx.all_reduce_host(host, op, "none", 256)
            torch.cuda.synchronize()
            want = orc.all_reduce(xs, sizes, op)
            for r in range(W):
                assert_bits_equal(host[r].numpy(), want[r], "host %s %s rank %d" % (dt, op, r))
