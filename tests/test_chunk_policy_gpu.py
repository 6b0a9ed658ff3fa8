"""The pipelined policy's chunk count, as gb_set_pipeline documents it: the
all_reduce chunk S = chunk_bytes * max(1, sqrt(P / (3 * chunk_bytes))) of
one island's payload P, reduce_scatter's max(chunk_bytes / 2, S -
chunk_bytes / 2), both cut into the fewest equal chunks of whole 256-element
tiles (at most 32).  A call launches one encode and one decode per chunk,
so the library's launch counter shows the count.  The results themselves do
not depend on the chunks (the parity tests check them at every size)."""
import math

import pytest
import torch

from cross_vendor_gradient_gb300 import Context, kernel_launch_count

pytestmark = pytest.mark.gpu

TILE = 256
CHUNK = 2 << 20


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def round_up(x, m):
    return (x + m - 1) // m * m


def expected_chunks(n, code_bytes, block, rs):
    per = code_bytes + (4.0 / block if block else 0.0)
    P = per * n
    s_ar = CHUNK * math.sqrt(P / (3 * CHUNK)) if P > 3 * CHUNK else float(CHUNK)
    half = CHUNK / 2
    S = s_ar if not rs else (s_ar - half if s_ar - half > half else half)
    ch = max(int(S / per) // TILE * TILE, TILE)
    ch = max(ch, round_up((n + 31) // 32, TILE))
    if ch >= n:
        return 1
    cnt = (n + ch - 1) // ch
    ch = round_up((n + cnt - 1) // cnt, TILE)
    return (n + ch - 1) // ch


CASES = [  # (elements per rank, codec, code bytes, fp8 block)
    (1 << 20, "e4m3", 1, 256),
    (1 << 22, "none", 4, 0),
    (1 << 22, "bf16", 2, 0),
    (6_553_600, "e4m3", 1, 256),  # the 25 MiB bucket: four chunks, seven for reduce_scatter
    (1 << 24, "none", 4, 0),
    (1 << 24, "bf16", 2, 0),
    (1 << 24, "e4m3", 1, 256),
    (1 << 26, "none", 4, 0),
    (1 << 26, "e4m3", 1, 256),
]


@pytest.mark.parametrize("n,codec,cb,block", CASES)
def test_chunk_counts_follow_the_documented_rule(n, codec, cb, block):
    W = 4
    bufs = [torch.ones(n, device="cuda") for _ in range(W)]
    outs = [torch.empty(n // W, device="cuda") for _ in range(W)]
    with Context((2, 2)) as ctx:
        k0 = kernel_launch_count()
        ctx.all_reduce(bufs, "sum", codec, block or 256)
        k1 = kernel_launch_count()
        ctx.reduce_scatter(bufs, outs, "sum", codec, block or 256)
        k2 = kernel_launch_count()
        torch.cuda.synchronize()
    assert k1 - k0 == 2 * expected_chunks(n, cb, block, False), (n, codec)
    assert k2 - k1 == 2 * expected_chunks(n, cb, block, True), (n, codec)
    if n == 6_553_600:
        assert expected_chunks(n, cb, block, False) == 4 and expected_chunks(n, cb, block, True) == 7
