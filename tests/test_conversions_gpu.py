"""The device conversions against the oracle's encoders, over every float32
bit pattern that the codec can meet:
  - fp8 (E4M3, E5M2): every pattern with |y| <= the largest finite value,
    fed through gb_bridge_compress in blocks whose largest element is that
    value, so the block scale is 2^0 and the code is the conversion itself;
  - bf16: every non-NaN pattern;
  - the block scale rule over absmax values at and around every power-of-two
    boundary, subnormals and the float32 extremes;
  - decode of every 8-bit code at several scales.
The oracle side runs in a spawn-started process pool (one chunk per task)."""
import multiprocessing as mp

import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import Context, payload_bytes, payload_scales_offset
from tests.gpu_util import assert_bits_equal, to_dev, to_host

pytestmark = pytest.mark.gpu

CHUNK = 1 << 25
MAXBITS = {"e4m3": 0x43E00000, "e5m2": 0x47600000}  # 448.0, 57344.0


def _oracle_fp8(args):
    lo, hi, fmt = args
    pats = np.arange(lo, hi, dtype=np.uint64).astype(np.uint32)
    return orc.fp8_encode_f32_array(pats.view(np.float32), fmt)


def _oracle_bf16(args):
    lo, hi = args
    pats = np.arange(lo, hi, dtype=np.uint64).astype(np.uint32)
    x = pats.view(np.float32)
    return orc.f32_to_bf16_array(x)


@pytest.fixture(scope="module")
def pool():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ctx = mp.get_context("spawn")
    with ctx.Pool(processes=max(1, min(16, mp.cpu_count()))) as p:
        yield p


def _ranges(lo, hi):
    return [(a, min(a + CHUNK, hi)) for a in range(lo, hi, CHUNK)]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_conversion_every_pattern(fmt, pool):
    M = np.float32(orc.fp8_max(fmt))
    B = 256
    per_block = B - 1
    top = MAXBITS[fmt] + 1
    ranges = []
    for sign in (0, 0x80000000):
        ranges += [(a + sign, b + sign) for a, b in _ranges(0, top)]
    results = pool.imap(_oracle_fp8, [(a, b, fmt) for a, b in ranges])
    with Context((1, 1)) as ctx:
        for (a, b), want in zip(ranges, results):
            pats = np.arange(a, b, dtype=np.uint64).astype(np.uint32)
            cnt = pats.size
            nblk = -(-cnt // per_block)
            s = np.zeros(nblk * B, np.float32)
            grid = s.reshape(nblk, B)  # a view of s
            grid[:, 0] = M  # pins the scale to 2^0
            body = np.zeros(nblk * per_block, np.float32)
            body[:cnt] = pats.view(np.float32)
            grid[:, 1:] = body.reshape(nblk, per_block)
            sd = to_dev(s)
            n = s.size
            p = torch.empty(payload_bytes(fmt, B, n), dtype=torch.uint8, device="cuda")
            ctx.bridge_compress(sd, fmt, B, p)
            ph = to_host(p)
            off = payload_scales_offset(fmt, B, n)
            assert np.all(ph[off:off + 4 * nblk].view(np.float32) == 1.0)
            codes = ph[:n].reshape(nblk, B)[:, 1:].reshape(-1)[:cnt]
            assert_bits_equal(codes, want, "%s patterns [0x%x, 0x%x)" % (fmt, a, b))


def test_bf16_conversion_every_pattern(pool):
    ranges = _ranges(0, 1 << 32)
    results = pool.imap(_oracle_bf16, ranges)
    with Context((1, 1)) as ctx:
        for (a, b), want in zip(ranges, results):
            pats = np.arange(a, b, dtype=np.uint64).astype(np.uint32)
            x = pats.view(np.float32)
            keep = ~np.isnan(x)
            sd = to_dev(x)
            p = torch.empty(payload_bytes("bf16", 256, x.size), dtype=torch.uint8, device="cuda")
            ctx.bridge_compress(sd, "bf16", 256, p)
            got = to_host(p).view(np.uint16)
            assert_bits_equal(got[keep], want[keep], "bf16 patterns [0x%x, 0x%x)" % (a, b))
            # NaN stays NaN
            nan_out = got[~keep].astype(np.uint32) << 16
            assert np.all(np.isnan(nan_out.view(np.float32)))


@pytest.mark.parametrize("fmt,B", [("e4m3", 256), ("e4m3", 128), ("e5m2", 128), ("e5m2", 256)])
def test_block_scale_rule(fmt, B):
    M = orc.fp8_max(fmt)
    vals = [0.0, float(np.finfo(np.float32).max), float(np.finfo(np.float32).tiny), 1e-45, 2.0 ** -140]
    for j in range(-160, 128):
        v = np.float32(M * 2.0 ** j) if M * 2.0 ** j < 3.4e38 else None
        if v is None:
            continue
        vals += [float(v), float(np.nextafter(v, np.float32(np.inf))), float(np.nextafter(v, np.float32(0)))]
    rng = np.random.default_rng(1)
    vals += list(np.exp2(rng.uniform(-149, 127, 4000)).astype(np.float32).astype(float))
    vals = np.array(vals, np.float32)
    nblk = vals.size
    s = np.zeros(nblk * B, np.float32)
    s.reshape(nblk, B)[:, 7] = vals
    s.reshape(nblk, B)[:, 9] = -vals / 3
    codes_w, scales_w = orc.encode(s, fmt, B)
    with Context((1, 1)) as ctx:
        p = torch.empty(payload_bytes(fmt, B, s.size), dtype=torch.uint8, device="cuda")
        ctx.bridge_compress(to_dev(s), fmt, B, p)
        ph = to_host(p)
    off = payload_scales_offset(fmt, B, s.size)
    assert_bits_equal(ph[off:off + 4 * nblk].view(np.float32), scales_w, "scales")
    assert_bits_equal(ph[:s.size], codes_w, "codes")


@pytest.mark.parametrize("fmt,B", [("e4m3", 256), ("e5m2", 128)])
def test_decode_every_code(fmt, B):
    ks = [-126, -100, -9, 0, 1, 17, 100, 120]
    n = 256 * len(ks) * (B // 128 if B > 128 else 1)
    codes = np.tile(np.arange(256, dtype=np.uint8), n // 256)
    finite = np.array([np.isfinite(orc.fp8_value(int(c), fmt)) for c in range(256)])
    codes = np.where(finite[codes], codes, 0).astype(np.uint8)
    nb = orc.n_blocks(n, B)
    scales = np.array([2.0 ** ks[b % len(ks)] for b in range(nb)], np.float32)
    want = orc.decode(codes, scales, fmt, B)
    P = payload_bytes(fmt, B, n)
    off = payload_scales_offset(fmt, B, n)
    buf = np.zeros(P, np.uint8)
    buf[:n] = codes
    buf[off:off + 4 * nb] = scales.view(np.uint8)
    with Context((1, 1)) as ctx:
        acc = torch.empty(n, dtype=torch.float32, device="cuda")
        ctx.bridge_decompress_accumulate(to_dev(buf), n, fmt, B, acc, False)
        got = to_host(acc)
    assert_bits_equal(got, want, "decode")
