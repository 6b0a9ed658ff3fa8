"""Pins of the CPU oracle against facts fixed outside it: the worked example
and the size ratios printed on the gpubridge README, the OCP 8-bit float
tables, torch's CPU conversions (library routines), closed forms, exact
integer arithmetic, error bounds against fp64 / rational sums, exhaustive
search, and the identities of the collectives.

No GPU.  Each pin is chosen so that a plausible slip in the oracle (a dropped
term, a transposed operand, a wrong rounding direction, a wrong exponent
offset) fails at least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as orc
from tests.conftest import read_golden
from cross_vendor_gradient_gb300 import workloads as wl

U = 2.0 ** -24  # unit roundoff of binary32


# ------------------------------------------------------------ worked example

def _demo():
    rows = read_golden("demo_four_ranks.txt")
    sizes = [int(v) for v in rows[0][1:]]
    n = int(rows[1][1])
    inputs = [np.array([float(v) for v in r[2:]], np.float32) for r in rows if r[0] == "input"]
    expected = np.array([float(v) for v in rows[-1][1:]], np.float32)
    assert all(x.size == n for x in inputs)
    return sizes, inputs, expected


@pytest.mark.parametrize("codec", ["none", "bf16", "e4m3", "e5m2"])
def test_demo_four_ranks_sum(codec):
    sizes, inputs, expected = _demo()
    outs = orc.all_reduce(inputs, sizes, "sum", codec, 256)
    for o in outs:
        assert np.array_equal(o, expected)


def test_demo_four_ranks_avg_and_bf16_buffers():
    sizes, inputs, expected = _demo()
    outs = orc.all_reduce(inputs, sizes, "avg", "e4m3", 256)
    for o in outs:
        assert np.array_equal(o, expected / 4)
    bf = [wl.to_bf16_bits(x) for x in inputs]
    outs = orc.all_reduce(bf, sizes, "sum", "bf16")
    for o in outs:
        assert np.array_equal(orc.bf16_bits_to_f32_array(o), expected)


def test_codec_size_ratios():
    rows = dict((r[0], r[1]) for r in read_golden("codec_sizes.txt"))
    B = int(rows["fp8_e4m3_block"])
    for nblocks in (1, 7, 1000):
        n = nblocks * B
        codes, scales = orc.encode(np.ones(n, np.float32), "e4m3", B)
        payload = codes.nbytes + scales.nbytes
        assert round(4 * n / payload, 1) == float(rows["fp8_ratio_one_decimal"])
        codes, _ = orc.encode(np.ones(n, np.float32), "bf16")
        assert 4 * n / codes.nbytes == float(rows["bf16_ratio"])


# ----------------------------------------------------------------- OCP fp8

def test_fp8_table_values():
    for fmt, code, val in read_golden("ofp8_values.txt"):
        v = orc.fp8_value(int(code, 16), fmt)
        if val == "nan":
            assert math.isnan(v), (fmt, code)
        elif val.endswith("inf"):
            assert v == float(val), (fmt, code)
        else:
            assert v == float(val), (fmt, code, v)
    assert orc.fp8_max("e4m3") == 448.0 and orc.fp8_max("e5m2") == 57344.0


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_values_monotone_and_symmetric(fmt):
    finite = [c for c in range(128) if math.isfinite(orc.fp8_value(c, fmt))]
    vals = [orc.fp8_value(c, fmt) for c in finite]
    assert finite == list(range(len(finite)))  # finite codes are a prefix
    assert all(b > a for a, b in zip(vals, vals[1:]))
    for c in finite:
        neg = orc.fp8_value(c | 0x80, fmt)
        assert neg == -vals[c] and math.copysign(1.0, neg) == -1.0
    # 126 positive finite non-zero E4M3 codes, 123 for E5M2
    assert len(finite) - 1 == (126 if fmt == "e4m3" else 123)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_encode_roundtrip_every_code(fmt):
    for c in range(256):
        v = orc.fp8_value(c, fmt)
        if math.isfinite(v):
            assert orc.fp8_encode(v, fmt) == c


def _fp8_probe_points(fmt):
    """Every grid value, every midpoint, and the neighbours of each midpoint
    in float32, both signs, up to the largest finite value."""
    vals = sorted({abs(orc.fp8_value(c, fmt)) for c in range(128)
                   if math.isfinite(orc.fp8_value(c, fmt))})
    pts = []
    for a, b in zip(vals, vals[1:]):
        mid = np.float32((a + b) / 2)  # exact: few significant bits
        pts += [a, b, mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(np.inf))]
    pts = np.array(pts, np.float32)
    return np.concatenate([pts, -pts])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_encode_matches_exhaustive_search(fmt):
    rng = np.random.default_rng(7)
    M = orc.fp8_max(fmt)
    rand = (rng.uniform(-1, 1, 3000) * np.exp2(rng.uniform(-20, math.log2(M) + 0.5, 3000)))
    pts = np.concatenate([_fp8_probe_points(fmt), rand.astype(np.float32),
                          np.array([M * 1.01, -M * 5, 1e30, -np.inf, np.inf], np.float32)])
    for y in pts:
        assert orc.fp8_encode(float(y), fmt) == orc.fp8_encode_bruteforce(float(y), fmt), y


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_fp8_encode_matches_torch_cast_in_range(fmt, tdt):
    """torch's CPU float8 casts round to nearest even; inside [-M, M] they
    must agree with the oracle exactly (outside, torch does not saturate)."""
    M = orc.fp8_max(fmt)
    rng = np.random.default_rng(11)
    rand = rng.uniform(-1, 1, 400_000) * np.exp2(rng.uniform(-30, math.log2(M), 400_000))
    y = np.concatenate([_fp8_probe_points(fmt), rand.astype(np.float32)])
    y = y[np.abs(y) <= M]
    ours = orc.fp8_encode_f32_array(y, fmt)
    ref = torch.from_numpy(y).to(tdt).view(torch.uint8).numpy()
    # torch writes -0.0 for tiny negatives as 0x80 as well; compare every byte
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------------- bf16

def test_bf16_matches_torch_cast():
    """Strided sweep of all 2^32 binary32 patterns plus every bf16 midpoint
    and its neighbours, against torch's CPU round-to-nearest-even cast."""
    stride = 4099  # odd, co-prime with 2^32: reaches every low-bit pattern
    bits = (np.arange(0, 1 << 32, stride, dtype=np.uint64)).astype(np.uint32)
    hi = np.arange(0, 1 << 16, dtype=np.uint32) << 16
    mids = hi | 0x8000
    extra = np.concatenate([mids, mids - 1, mids + 1, hi | 0x7FFF, hi | 0x0001])
    bits = np.concatenate([bits, extra.astype(np.uint32)])
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    ours = orc.f32_to_bf16_array(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_roundtrip_and_bound():
    rng = np.random.default_rng(3)
    h = rng.integers(0, 1 << 16, 20000).astype(np.uint16)
    x = orc.bf16_bits_to_f32_array(h)
    keep = np.isfinite(x)
    assert np.array_equal(orc.f32_to_bf16_array(x[keep]), h[keep])
    y = (rng.standard_normal(20000) * np.exp2(rng.uniform(-100, 100, 20000))).astype(np.float32)
    back = orc.bf16_bits_to_f32_array(orc.f32_to_bf16_array(y))
    assert np.all(np.abs(back.astype(np.float64) - y) <= 2.0 ** -8 * np.abs(y.astype(np.float64)))


# ------------------------------------------------------------- scale rule

def _k_by_search(m, M):
    """Smallest k with m * 2^-k <= M (exact rational search), clamped."""
    if m == 0:
        return 0
    m = Fraction(float(m))
    k = -300
    while m * Fraction(2) ** (-k) > M:
        k += 1
    return max(k, -126)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_block_scale_exponent(fmt):
    M = orc.fp8_max(fmt)
    f32 = np.float32
    cases = [0.0, float(np.finfo(np.float32).max), float(np.finfo(np.float32).tiny),
             1e-45, 2.0 ** -140]
    for j in range(-130, 118):
        v = f32(M * 2.0 ** j) if M * 2.0 ** j < 3.4e38 else None
        if v is None or v == 0:
            continue
        cases += [float(v), float(np.nextafter(v, f32(np.inf))), float(np.nextafter(v, f32(0)))]
        if f32(v) != 0 and abs(math.log2(M) + j) < 126:
            assert orc.block_scale_exponent(float(v), fmt) == max(j, -126)
    rng = np.random.default_rng(5)
    cases += list((np.exp2(rng.uniform(-149, 127, 3000))).astype(np.float32).astype(float))
    for m in cases:
        k = orc.block_scale_exponent(m, fmt)
        assert k == _k_by_search(f32(m), M), (m, k)
    assert orc.block_scale_exponent(float(np.finfo(np.float32).max), "e4m3") == 120
    assert orc.block_scale_exponent(float(np.finfo(np.float32).max), "e5m2") == 113


@pytest.mark.parametrize("fmt,B", [("e4m3", 256), ("e5m2", 128)])
def test_fp8_blocks_of_grid_values_roundtrip(fmt, B):
    """Blocks built as code values * 2^k whose largest magnitude lies in
    (M/2, M] encode back to the same codes and to scale 2^k."""
    M = orc.fp8_max(fmt)
    finite = [c for c in range(128) if math.isfinite(orc.fp8_value(c, fmt))]
    tops = [c for c in finite if M / 2 < orc.fp8_value(c, fmt) <= M]
    rng = np.random.default_rng(9)
    for k in (-126, -20, -3, 0, 5, 60):
        for top in tops:
            codes = rng.choice(finite, B) | (rng.integers(0, 2, B) << 7)
            codes[rng.integers(0, B)] = top | (rng.integers(0, 2) << 7)
            s = np.array([orc.fp8_value(int(c), fmt) * 2.0 ** k for c in codes], np.float32)
            got_codes, got_scales = orc.encode(s, fmt, B)
            # a -0.0 code may come back as +0.0 only if the value is +0: values keep sign
            assert np.array_equal(got_codes, codes.astype(np.uint8)), (k, top)
            assert got_scales[0] == np.float32(2.0 ** k)


@pytest.mark.parametrize("fmt,B,c", [("e4m3", 256, 2.0 ** -4), ("e5m2", 128, 2.0 ** -3)])
def test_fp8_error_bound_per_block(fmt, B, c):
    """Decode(encode(s)) stays within c * absmax of its block (about one
    significant digit relative to the block's largest value for E4M3)."""
    rng = np.random.default_rng(13)
    n = B * 300 + 77
    s = (rng.standard_normal(n) * np.exp2(rng.integers(-60, 60, n))).astype(np.float32)
    s[:B] = 0.0
    s[B:2 * B] = rng.standard_normal(B).astype(np.float32) * np.float32(1e-40)  # subnormal block
    codes, scales = orc.encode(s, fmt, B)
    back = orc.decode(codes, scales, fmt, B).astype(np.float64)
    for b in range(orc.n_blocks(n, B)):
        blk = s[b * B:(b + 1) * B].astype(np.float64)
        err = np.abs(back[b * B:(b + 1) * B] - blk)
        assert np.all(err <= c * np.max(np.abs(blk))), b
    assert np.array_equal(codes[:B], np.zeros(B, np.uint8)) and scales[0] == 1.0


def test_fp8_signed_zero_and_saturation():
    assert orc.fp8_encode(-0.0, "e4m3") == 0x80 and orc.fp8_encode(0.0, "e4m3") == 0x00
    assert orc.fp8_encode(1e9, "e4m3") == 0x7E and orc.fp8_encode(-np.inf, "e4m3") == 0xFE
    assert orc.fp8_encode(1e9, "e5m2") == 0x7B and orc.fp8_encode(np.inf, "e5m2") == 0x7B
    # tiny values round to signed zero
    assert orc.fp8_encode(2.0 ** -11, "e4m3") == 0x00 and orc.fp8_encode(-2.0 ** -10, "e4m3") == 0x80
    assert orc.fp8_encode(2.0 ** -10 * 1.0000001, "e4m3") == 0x01


# ----------------------------------------------------------- island sums

def test_island_sum_order_is_ascending_rank():
    """1 + 2^-24 rounds back to 1 (tie to even); adding a second 2^-24 again
    gives 1.  The reverse order gives 1 + 2^-23."""
    a = np.array([1.0], np.float32)
    b = np.array([2.0 ** -24], np.float32)
    assert orc.island_sum([a, b, b])[0] == np.float32(1.0)
    assert orc.island_sum([b, b, a])[0] == np.float32(1.0 + 2.0 ** -23)


def test_island_sum_integers_exact():
    rng = np.random.default_rng(17)
    for K in (1, 2, 3, 4, 8):
        xs = [rng.integers(-2 ** 20, 2 ** 20, 5000).astype(np.float32) for _ in range(K)]
        exact = np.sum([x.astype(np.int64) for x in xs], axis=0)
        assert np.array_equal(orc.island_sum(xs).astype(np.int64), exact)


def test_island_sum_recursive_bound():
    rng = np.random.default_rng(19)
    for K in (2, 3, 5, 8):
        xs = [(rng.standard_normal(20000) * np.exp2(rng.integers(-10, 10, 20000))).astype(np.float32)
              for _ in range(K)]
        s = orc.island_sum(xs).astype(np.float64)
        exact = np.sum([x.astype(np.float64) for x in xs], axis=0)  # exact for these magnitudes
        absum = np.sum([np.abs(x.astype(np.float64)) for x in xs], axis=0)
        assert np.all(np.abs(s - exact) <= (K - 1) * U * absum)


def test_bf16_inputs_widen_exactly():
    rng = np.random.default_rng(23)
    h = [wl.to_bf16_bits(rng.integers(-100, 100, 3000).astype(np.float32)) for _ in range(4)]
    exact = np.sum([orc.bf16_bits_to_f32_array(x).astype(np.int64) for x in h], axis=0)
    assert np.array_equal(orc.island_sum(h).astype(np.int64), exact)


# --------------------------------------------------------------- collectives

LAYOUTS = [(1,), (2,), (1, 1), (2, 2), (1, 2), (3, 1), (1, 1, 1), (4, 4), (2, 3, 3), (8,)]


@pytest.mark.parametrize("sizes", LAYOUTS)
def test_one_world_integer_sum_exact_uncompressed(sizes):
    rng = np.random.default_rng(29)
    W = sum(sizes)
    xs = [rng.integers(-1000, 1000, 777).astype(np.float32) for _ in range(W)]
    exact = np.sum([x.astype(np.int64) for x in xs], axis=0)
    for o in orc.all_reduce(xs, sizes, "sum", "none"):
        assert np.array_equal(o.astype(np.int64), exact)


@pytest.mark.parametrize("codec", ["none", "bf16", "e4m3", "e5m2"])
def test_one_rank_is_identity(codec):
    rng = np.random.default_rng(31)
    x = (rng.standard_normal(1000) * 3).astype(np.float32)
    for op in ("sum", "avg"):
        (o,) = orc.all_reduce([x], (1,), op, codec)
        assert np.array_equal(o.view(np.uint32), x.view(np.uint32))
    h = wl.to_bf16_bits(x)
    (o,) = orc.all_reduce([h], (1,), "sum", codec)
    assert np.array_equal(o, h)


@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (1, 2), (3,), (2, 3, 3)])
@pytest.mark.parametrize("codec", ["none", "e4m3"])
def test_avg_is_sum_divided_by_world_size(sizes, codec):
    """AVG is the SUM divided by W: the float32 result is the quotient
    rounded to nearest, checked with exact rationals."""
    rng = np.random.default_rng(37)
    W = sum(sizes)
    xs = [rng.standard_normal(500).astype(np.float32) for _ in range(W)]
    s = orc.all_reduce(xs, sizes, "sum", codec)[0]
    a = orc.all_reduce(xs, sizes, "avg", codec)[0]
    for sj, aj in zip(s, a):
        q = Fraction(float(sj)) / W
        lo = np.nextafter(aj, np.float32(-np.inf))
        hi = np.nextafter(aj, np.float32(np.inf))
        assert abs(Fraction(float(aj)) - q) <= abs(Fraction(float(lo)) - q)
        assert abs(Fraction(float(aj)) - q) <= abs(Fraction(float(hi)) - q)
    if W in (2, 4, 8):
        assert np.array_equal(a, s / np.float32(W))  # power of two: exact scaling


@pytest.mark.parametrize("sizes", [(1, 1), (2, 2), (4, 4), (1, 3), (2, 1, 1)])
@pytest.mark.parametrize("codec", ["none", "bf16", "e4m3", "e5m2"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_then_all_gather_is_all_reduce(sizes, codec, dtype):
    rng = np.random.default_rng(41)
    W = sum(sizes)
    n = W * 300
    xs = [rng.standard_normal(n).astype(np.float32) for _ in range(W)]
    if dtype == "bf16":
        xs = [wl.to_bf16_bits(x) for x in xs]
    ar = orc.all_reduce(xs, sizes, "avg", codec, 128)
    rs = orc.reduce_scatter(xs, sizes, "avg", codec, 128)
    ag = orc.all_gather(rs)
    for r in range(W):
        assert np.array_equal(ag[r], ar[r])
        assert np.array_equal(ar[r], ar[0])


def test_broadcast_and_all_gather_are_exact_copies():
    rng = np.random.default_rng(43)
    xs = [rng.standard_normal(33).astype(np.float32) for _ in range(5)]
    for src in range(5):
        for o in orc.broadcast(xs, src):
            assert np.array_equal(o.view(np.uint32), xs[src].view(np.uint32))
    ag = orc.all_gather(xs)
    cat = np.concatenate(xs)
    for o in ag:
        assert np.array_equal(o.view(np.uint32), cat.view(np.uint32))


def test_every_island_term_is_decoded():
    """Every island, its own included, contributes dec(enc(s_i)): with two
    one-rank islands the e4m3 total equals the sum of the two decoded sums,
    and differs from leader 0 adding its exact sum."""
    x0 = np.array([1.0 + 2.0 ** -10] + [0.0] * 255, np.float32)
    x1 = np.array([1.0] + [0.0] * 255, np.float32)
    t = orc.all_reduce([x0, x1], (1, 1), "sum", "e4m3")[0]
    assert t[0] == np.float32(2.0)  # 1 + 2^-10 encodes to 1.0 in E4M3
    assert x0[0] + x1[0] != t[0]


@pytest.mark.parametrize("fmt,B,c", [("e4m3", 256, 2.0 ** -4), ("e5m2", 128, 2.0 ** -3),
                                     ("bf16", 256, None), ("none", 256, 0.0)])
def test_end_to_end_bound_against_exact_sum(fmt, B, c):
    """Compressed all_reduce within the codec bound of the exact (fp64) sum:
    |t - exact| <= sum_i c * absmax_block(s_i) + (W + I) u (sum|x| + sum_i |dec_i|)."""
    rng = np.random.default_rng(47)
    sizes = (2, 2)
    W, I = 4, 2
    n = B * 40 + 19
    xs = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(W)]
    xs[1][rng.permutation(n)[: n // 100]] *= 100
    t, mid = orc.rbb_total(xs, sizes, "sum", fmt, B, intermediates=True)
    exact = np.sum([x.astype(np.float64) for x in xs], axis=0)
    absx = np.sum([np.abs(x.astype(np.float64)) for x in xs], axis=0)
    bound = np.zeros(n)
    absdec = np.zeros(n)
    for i in range(I):
        s = mid["island_sums"][i].astype(np.float64)
        dec = orc.decode(mid["codes"][i], mid["scales"][i], fmt, B).astype(np.float64)
        absdec += np.abs(dec)
        if fmt == "bf16":
            bound += 2.0 ** -8 * np.abs(s)
        elif c:
            for b in range(orc.n_blocks(n, B)):
                bound[b * B:(b + 1) * B] += c * np.max(np.abs(s[b * B:(b + 1) * B]))
    bound += (W + I) * U * (absx + absdec)
    assert np.all(np.abs(t.astype(np.float64) - exact) <= bound)
    if fmt == "none":
        assert np.all(np.abs(t.astype(np.float64) - exact) <= (W - 1) * U * absx)


def test_tiny_cases_brute_force():
    """Every layout of 1..8 ranks into contiguous islands (up to 3) and
    sizes 1..300: all outputs bit-identical, integer data exact when
    uncompressed, RS then AG equal to AR when n divides."""
    rng = np.random.default_rng(53)
    layouts = [(1,), (1, 1), (2,), (1, 2), (2, 1), (3,), (2, 2), (1, 1, 2), (4,), (1, 3),
               (3, 1), (2, 2, 4), (4, 4), (8,), (1, 1, 1), (3, 3, 2)]
    ns = [1, 2, 3, 7, 8, 9, 31, 127, 128, 129, 255, 256, 257, 300]
    for sizes in layouts:
        W = sum(sizes)
        for n in ns:
            ints = [rng.integers(-50, 50, n).astype(np.float32) for _ in range(W)]
            exact = np.sum([x.astype(np.int64) for x in ints], axis=0)
            for o in orc.all_reduce(ints, sizes, "sum", "none"):
                assert np.array_equal(o.astype(np.int64), exact)
            for codec in ("bf16", "e4m3", "e5m2"):
                xs = [rng.standard_normal(n).astype(np.float32) for _ in range(W)]
                outs = orc.all_reduce(xs, sizes, "sum", codec, 128)
                assert all(np.array_equal(o, outs[0]) for o in outs)
                if n % W == 0:
                    ag = orc.all_gather(orc.reduce_scatter(xs, sizes, "sum", codec, 128))
                    assert np.array_equal(ag[0], outs[0])


# --------------------------------------------------------------- bucket plan

def _check_greedy(numels, elem_bytes, cap, bucket_of, offset, bucket_numel, pad=1):
    numels = [int(v) for v in numels]
    T = len(numels)
    nb = len(bucket_numel)
    assert list(bucket_of) == sorted(bucket_of) and bucket_of[0] == 0 and bucket_of[-1] == nb - 1
    for b in range(nb):
        members = [t for t in range(T) if bucket_of[t] == b]
        assert members, "empty bucket"
        used = sum(numels[t] for t in members)
        pos = 0
        for t in members:
            assert offset[t] == pos
            pos += numels[t]
        assert int(bucket_numel[b]) == -(-used // pad) * pad
        if len(members) > 1:
            assert used * elem_bytes <= cap
        if b + 1 < nb:  # greedy: the next tensor did not fit
            nxt = members[-1] + 1
            assert (used + numels[nxt]) * elem_bytes > cap


def test_bucket_plan_gpt2_and_llama():
    for shapes, eb in ((wl.gpt2_small_shapes(), 2), (wl.llama_1b_shapes(), 2)):
        numels = [wl.numel(s) for s in shapes]
        bo, off, bn = orc.bucket_plan(numels, eb, wl.BUCKET_CAP_BYTES, 1)
        _check_greedy(numels, eb, wl.BUCKET_CAP_BYTES, bo, off, bn)
        assert int(np.sum(bn)) == sum(numels)
    numels = [wl.numel(s) for s in wl.gpt2_small_shapes()]
    assert sum(numels) == 124_439_808
    bo, off, bn = orc.bucket_plan(numels, 2, wl.BUCKET_CAP_BYTES, 1)
    assert bo[0] == 0 and bo[1] == 1 and int(bn[0]) == 50257 * 768  # wte alone
    assert sum(wl.numel(s) for s in wl.llama_1b_shapes()) == 1_100_048_384


def test_bucket_plan_small_cases_and_padding():
    rng = np.random.default_rng(59)
    for _ in range(200):
        T = int(rng.integers(1, 30))
        numels = rng.integers(1, 5000, T)
        cap = int(rng.integers(1, 20000))
        pad = int(rng.choice([1, 2, 8, 256]))
        bo, off, bn = orc.bucket_plan(numels, 4, cap, pad)
        _check_greedy(numels, 4, cap, bo, off, bn, pad)


# ------------------------------------------------------------- error feedback

def _grid_data(rng, n, W):
    """Values on a 2^-12 grid in [-1, 1]: every float32 operation of the
    error-feedback step is then exact (dec values sit on a grid no coarser
    than 2^-16, s + r spans fewer than 24 bits, and s' - dec(enc(s')) is
    exact by Sterbenz's lemma or because dec is 0)."""
    return [(rng.integers(-4096, 4097, n) / 4096.0).astype(np.float32) for _ in range(W)]


@pytest.mark.parametrize("codec,block", [("e4m3", 256), ("e5m2", 128), ("bf16", 256)])
def test_error_feedback_telescopes_exactly(codec, block):
    """sum_t dec(p_t) = sum_t s_t + r_0 - r_T per element, exactly (the
    residual carries every rounding error into the next step)."""
    rng = np.random.default_rng(71)
    n, T = 3 * block + 17, 6
    r = np.zeros(n, np.float32)
    r0 = r.copy()
    sum_dec = np.zeros(n, dtype=object)
    sum_s = np.zeros(n, dtype=object)
    for _ in range(T):
        s = _grid_data(rng, n, 1)[0] * np.float32(3.0)
        codes, scales = orc.encode_ef(s, r, codec, block)
        dec = orc.decode(codes, scales, codec, block)
        sum_dec += np.array([Fraction(float(v)) for v in dec], dtype=object)
        sum_s += np.array([Fraction(float(v)) for v in s], dtype=object)
    rhs = sum_s + np.array([Fraction(float(v)) for v in r0], dtype=object) - \
        np.array([Fraction(float(v)) for v in r], dtype=object)
    assert all(a == b for a, b in zip(sum_dec, rhs))


@pytest.mark.parametrize("codec,block,c", [("e4m3", 256, 2.0 ** -4), ("e5m2", 128, 2.0 ** -3)])
def test_error_feedback_residual_bound(codec, block, c):
    rng = np.random.default_rng(73)
    n = 5 * block + 3
    r = np.zeros(n, np.float32)
    for _ in range(4):
        s = (rng.standard_normal(n) * np.exp2(rng.integers(-20, 5, n))).astype(np.float32)
        sp = (s + r).astype(np.float32)
        orc.encode_ef(s, r, codec, block)
        for b in range(orc.n_blocks(n, block)):
            blk = slice(b * block, (b + 1) * block)
            assert np.all(np.abs(r[blk].astype(np.float64)) <= c * np.max(np.abs(sp[blk].astype(np.float64))))


def test_error_feedback_none_codec_is_plain_all_reduce():
    rng = np.random.default_rng(79)
    sizes = (2, 1, 1)
    xs = [rng.standard_normal(1000).astype(np.float32) for _ in range(4)]
    res = [np.zeros(1000, np.float32) for _ in range(3)]
    outs = orc.all_reduce_ef(xs, sizes, res, "avg", "none")
    want = orc.all_reduce(xs, sizes, "avg", "none")
    for o, w_ in zip(outs, want):
        assert np.array_equal(o.view(np.uint32), w_.view(np.uint32))
    assert all(not np.any(r) for r in res)


def test_error_feedback_error_does_not_accumulate():
    """Over many steps the summed compressed totals stay within the final
    residuals (plus float32 rounding) of the summed exact totals; without
    error feedback the gap grows with the number of steps."""
    rng = np.random.default_rng(83)
    sizes, n, T = (1, 1), 512, 64
    res = [np.zeros(n, np.float32) for _ in range(2)]
    acc_ef = np.zeros(n)
    acc_plain = np.zeros(n)
    acc_exact = np.zeros(n)
    base = rng.standard_normal(n).astype(np.float32)
    for _ in range(T):
        xs = [(base + rng.standard_normal(n).astype(np.float32) * np.float32(1e-3)) for _ in range(2)]
        acc_exact += xs[0].astype(np.float64) + xs[1].astype(np.float64)
        acc_ef += orc.all_reduce_ef(xs, sizes, res, "sum", "e4m3", 256)[0]
        acc_plain += orc.all_reduce(xs, sizes, "sum", "e4m3", 256)[0]
    gap_ef = np.abs(acc_ef - acc_exact)
    bound = np.abs(res[0].astype(np.float64)) + np.abs(res[1].astype(np.float64)) + T * 4 * U * np.abs(acc_exact / T) * 4
    assert np.all(gap_ef <= bound + 1e-6)
    assert np.max(np.abs(acc_plain - acc_exact)) > 4 * np.max(gap_ef)


# ------------------------------------------------ exact path: MAX/MIN, dtypes

INT_DTS = [np.int8, np.uint8, np.int32, np.int64]


def test_f16_conversions_match_numpy():
    """float32 -> float16 rounding against numpy's correctly rounded cast
    (strided sweep of all patterns plus every float16 midpoint and its
    neighbours); float16 -> float32 widening over all 65536 patterns."""
    bits = np.arange(0, 1 << 32, 8191, dtype=np.uint64).astype(np.uint32)
    h = np.arange(0, 1 << 16, dtype=np.uint32)
    f = h.astype(np.uint16).view(np.float16).astype(np.float32)
    ok = np.isfinite(f)
    mids = ((f[ok][:-1].astype(np.float64) + f[ok][1:].astype(np.float64)) / 2).astype(np.float32)
    x = np.concatenate([bits.view(np.float32), mids, np.nextafter(mids, np.float32(np.inf)),
                        np.nextafter(mids, np.float32(-np.inf))])
    x = x[~np.isnan(x)]
    with np.errstate(over="ignore"):  # values past float16's range round to infinity, as intended
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(orc.f32_to_f16_array(x), ref)
    for hv in range(0, 1 << 16, 7):
        want = np.uint16(hv).view(np.float16).astype(np.float32)
        got = orc.f16_to_f32(hv)
        assert (np.isnan(want) and np.isnan(got)) or got == want


@pytest.mark.parametrize("dt", INT_DTS)
@pytest.mark.parametrize("sizes", [(1, 1), (2, 3), (4, 4), (3,)])
def test_integer_sum_wraps_modulo(dt, sizes):
    rng = np.random.default_rng(101)
    info = np.iinfo(dt)
    W = sum(sizes)
    xs = [rng.integers(info.min, info.max, 257, dtype=dt, endpoint=True) for _ in range(W)]
    xs[0][:3] = [info.max, info.min, info.max]
    bits = np.dtype(dt).itemsize * 8
    exact = [sum(int(x[j]) for x in xs) for j in range(257)]
    want = np.array([((v % (1 << bits)) if info.min == 0 else ((v + (1 << (bits - 1))) % (1 << bits) - (1 << (bits - 1))))
                     for v in exact], dtype=dt)
    for o in orc.all_reduce(xs, sizes, "sum"):
        assert np.array_equal(o, want)


@pytest.mark.parametrize("dt", [np.float32, np.float64, np.float16, np.int8, np.uint8, np.int32, np.int64])
@pytest.mark.parametrize("op,ref", [("max", np.max), ("min", np.min)])
def test_max_min_match_numpy(dt, op, ref):
    rng = np.random.default_rng(103)
    W = 5
    if np.issubdtype(dt, np.integer):
        info = np.iinfo(dt)
        xs = [rng.integers(info.min, info.max, 500, dtype=dt, endpoint=True) for _ in range(W)]
    else:
        xs = [(rng.standard_normal(500) * 100 + 1.0).astype(dt) for _ in range(W)]  # no zeros
    want = ref(np.stack(xs), axis=0)
    for sizes in ((2, 3), (5,), (1, 1, 1, 1, 1)):
        for o in orc.all_reduce(xs, sizes, op):
            assert np.array_equal(o, want)
    bf = [wl.to_bf16_bits(x.astype(np.float32)) for x in xs] if not np.issubdtype(dt, np.integer) else None
    if bf is not None and dt == np.float32:
        want_bf = orc.bf16_bits_to_f32_array(np.stack(bf)).max(axis=0) if op == "max" else \
            orc.bf16_bits_to_f32_array(np.stack(bf)).min(axis=0)
        assert np.array_equal(orc.bf16_bits_to_f32_array(orc.all_reduce(bf, (2, 3), op)[0]), want_bf)


def test_max_min_ties_keep_the_lower_rank():
    a = np.array([-0.0, 0.0, -0.0], np.float32)
    b = np.array([0.0, -0.0, -0.0], np.float32)
    for op in ("max", "min"):
        o = orc.all_reduce([a, b], (1, 1), op)[0]
        assert np.array_equal(np.signbit(o), np.signbit(a))
        o = orc.all_reduce([b, a], (2,), op)[0]
        assert np.array_equal(np.signbit(o), np.signbit(b))


@pytest.mark.parametrize("dt", [np.float64, np.float16])
def test_float64_and_float16_sums(dt):
    rng = np.random.default_rng(107)
    sizes = (2, 2)
    lim = 400 if dt == np.float16 else 2 ** 40
    xs = [rng.integers(-lim, lim, 777).astype(dt) for _ in range(4)]
    exact = np.sum([x.astype(np.int64) for x in xs], axis=0)
    for o in orc.all_reduce(xs, sizes, "sum"):
        assert np.array_equal(o.astype(np.int64), exact)
    # AVG: the float32 (float16) or float64 quotient, rounded once to the dtype
    xs = [rng.standard_normal(300).astype(dt) for _ in range(4)]
    s = orc.all_reduce(xs, sizes, "sum")[0]
    a = orc.all_reduce(xs, sizes, "avg")[0]
    if dt == np.float64:
        assert np.array_equal(a, s / 4.0)
        ex = np.array([sum(Fraction(float(x[j])) for x in xs) for j in range(300)], dtype=object)
        absx = np.sum([np.abs(x) for x in xs], axis=0)
        assert all(abs(Fraction(float(s[j])) - ex[j]) <= 3 * 2.0 ** -53 * absx[j] for j in range(300))
    else:
        s32 = orc.island_sum([x.astype(np.float32) for x in xs[:2]]) + orc.island_sum(
            [x.astype(np.float32) for x in xs[2:]])
        assert np.array_equal(a, (s32 / np.float32(4)).astype(np.float16))


@pytest.mark.parametrize("dt", [np.float64, np.float16, np.int32, np.uint8])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_exact_rs_then_ag_is_ar(dt, op):
    rng = np.random.default_rng(109)
    sizes = (2, 1, 1)
    xs = [(rng.standard_normal(400) * 50).astype(dt) for _ in range(4)]
    ag = orc.all_gather(orc.reduce_scatter(xs, sizes, op))
    ar = orc.all_reduce(xs, sizes, op)
    assert all(np.array_equal(g, r) for g, r in zip(ag, ar))


def test_avg_refused_on_integers():
    with pytest.raises(ValueError):
        orc.all_reduce([np.zeros(4, np.int32)] * 2, (1, 1), "avg")


def _f16_double_rounding_cases(rng, want, count=40):
    """Random float16 triples (a, b, c) where float32 arithmetic followed by
    one rounding to float16 differs from rounding the exact value once."""
    found = []
    while len(found) < count:
        h = rng.integers(0, 1 << 16, (4096, 3)).astype(np.uint16)
        v = h.view(np.float16).astype(np.float64)
        ok = np.all(np.isfinite(v), axis=1)
        for a, b, c in v[ok]:
            exact = (a + b) + c  # exact in float64 for float16 inputs
            f32 = (np.float32(a) + np.float32(b)) + np.float32(c)
            with np.errstate(over="ignore"):  # sums past float16's range round to infinity
                h32, hx = np.float16(f32), np.float16(exact)
            if want == "sum" and h32 != hx and np.isfinite(h32):
                found.append((a, b, c))
            if want == "avg":
                q32 = np.float32(f32) / np.float32(3)
                if np.float16(q32) != np.float16(exact / 3) and np.isfinite(np.float16(q32)):
                    found.append((a, b, c))
    return np.array(found[:count])


@pytest.mark.parametrize("op", ["sum", "avg"])
def test_float16_accumulates_and_divides_in_float32(op):
    """float16 buffers: the sum (and the AVG quotient) is formed in float32
    and rounded once to float16, not formed exactly."""
    rng = np.random.default_rng(113)
    cases = _f16_double_rounding_cases(rng, op)
    xs = [cases[:, q].astype(np.float16) for q in range(3)]
    f32 = (xs[0].astype(np.float32) + xs[1].astype(np.float32)) + xs[2].astype(np.float32)
    want = (f32 if op == "sum" else f32 / np.float32(3)).astype(np.float16)
    for o in orc.all_reduce(xs, (3,), op):
        assert np.array_equal(o.view(np.uint16), want.view(np.uint16))


# ------------------------------------------------------------ sharded bridge
# gpubridge README, policy table, sharded-bridge row: k = smallest island size;
# island reduce_scatter onto k ranks, rank j of every island all_reduces
# segment j over its own link, island all_gather.

@pytest.mark.parametrize("sizes,n,seg", [((2, 2), 1000, 512), ((4, 4), 6_553_600, 1_638_400),
                                         ((3, 5), 1, 256), ((2, 3, 4), 513, 512), ((4, 2), 4097, 2304),
                                         ((1, 3), 700, 700), ((4,), 900, 900)])
def test_sharded_segment_length_is_the_reading(sizes, n, seg):
    xs = [np.zeros(n, np.float32) for _ in range(sum(sizes))]
    _, got = orc.all_reduce_sharded(xs, sizes, with_segment=True)
    assert got == seg


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e4m3", 128),
                                         ("e5m2", 128), ("e5m2", 256)])
@pytest.mark.parametrize("sizes", [(2, 2), (3, 2), (4, 4), (2, 3, 4), (1, 3), (5,)])
def test_sharded_equals_reduce_bridge_broadcast(codec, block, sizes):
    """Codec blocks are local and every segment starts on a block boundary,
    so cutting the tensor into segments changes no bit: the sharded result
    equals reduce-bridge-broadcast for every codec, op, dtype and length,
    short and empty trailing segments included."""
    W = sum(sizes)
    for n in (1, 255, 256, 257, 600, 3 * 256 + 5, 5000):
        for dtype in ("f32", "bf16"):
            w = wl.Workload("t", 40 + n % 7, tuple(sizes), dtype, "normal_1e-3_outliers", "sum", ())
            xs = wl.host_rank_inputs(w, n=n)
            for op in ("sum", "avg"):
                got = orc.all_reduce_sharded(xs, sizes, op, codec, block)
                want = orc.all_reduce(xs, sizes, op, codec, block)
                for r in range(W):
                    assert np.array_equal(got[r].view(np.uint8), want[r].view(np.uint8)), (n, dtype, op, r)


@pytest.mark.parametrize("sizes", [(2, 2), (3, 4), (2, 2, 2)])
@pytest.mark.parametrize("op", ["sum", "avg"])
def test_sharded_integer_sums_are_exact(sizes, op):
    """Integer-valued float32 inputs below 2^24 in magnitude: every segment's
    uncompressed sum is the exact integer sum, and AVG its one correctly
    rounded quotient by W, independent of where the segments fall."""
    W = sum(sizes)
    rng = np.random.default_rng(77)
    n = 2000
    xs = [rng.integers(-1000, 1001, n).astype(np.float32) for _ in range(W)]
    exact = np.sum(np.stack(xs).astype(np.float64), axis=0)
    want = exact if op == "sum" else exact / W
    got = orc.all_reduce_sharded(xs, sizes, op, "none", 256)
    for r in range(W):
        assert np.array_equal(got[r], want.astype(np.float32)), r


# ------------------------------------------------------------ C self-test

def test_oracle_c_selftest():
    """oracle/selftest.c checks the oracle from C, with no Python in between:
    the README's four-rank demo for every codec, the codec size ratios and the
    OFP8 table values (the golden fixtures), and the block-scale rule's
    closed forms."""
    import os
    import subprocess
    from oracle import build as ob
    ob.build()
    golden = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    out = subprocess.run([ob.SELFTEST] + [os.path.join(golden, f) for f in
                                          ("demo_four_ranks.txt", "codec_sizes.txt", "ofp8_values.txt")],
                         capture_output=True, text=True, timeout=60)
    lines = out.stdout.strip().splitlines()
    assert out.returncode == 0 and not [l for l in lines if not l.startswith("ok ")], out.stdout + out.stderr
    assert len(lines) == 16
