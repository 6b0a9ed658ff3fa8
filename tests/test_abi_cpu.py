"""The C ABI without a GPU: the library loads, exports every entry point that
include/gb.h declares, its host-only logic (payload sizes, bucket plan)
matches the oracle, and argument validation answers before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as orc
from cross_vendor_gradient_gb300 import binding as B
from cross_vendor_gradient_gb300 import build as gbuild
from cross_vendor_gradient_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    gbuild.build()


def _declared():
    text = open(os.path.join(ROOT, "include", "gb.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gb_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported_and_bound():
    names = _declared()
    assert len(names) >= 28
    L = ctypes.CDLL(B.LIB_PATH)
    for name in names:
        assert hasattr(L, name), name
        assert name in B.SIGNATURES, "binding lacks %s" % name
        assert hasattr(B, name), "binding function %s" % name
    assert set(B.SIGNATURES) == set(names)


def test_status_strings():
    for s in range(12):
        assert B.gb_status_string(s).startswith("GB_")
    assert B.gb_status_string(B.GB_OK) == "GB_OK"


@pytest.mark.parametrize("codec,block", [("none", 256), ("bf16", 256), ("e4m3", 256), ("e5m2", 128),
                                         ("e4m3", 128)])
def test_payload_bytes_hold_the_oracle_payload(codec, block):
    cid = {"none": 0, "bf16": 1, "e4m3": 2, "e5m2": 3}[codec]
    for n in (1, 7, 255, 256, 257, 1000, 6_553_600):
        s = np.zeros(min(n, 4096), np.float32)
        codes, scales = orc.encode(s, codec, block)
        per = codes.itemsize
        nsc = orc.n_blocks(n, block) if codec in ("e4m3", "e5m2") else 0
        P = B.gb_payload_bytes(cid, block, n)
        off = B.gb_payload_scales_offset(cid, block, n)
        assert off >= n * per and off % 16 == 0 or nsc == 0
        assert P == (off + 4 * nsc if nsc else n * per)
    assert B.gb_payload_bytes(2, 64, 100) == 0 and B.gb_payload_bytes(9, 256, 100) == 0


def test_fp8_payload_ratio_is_the_pages_3_9():
    n = 256 * 25600
    assert round(4 * n / B.gb_payload_bytes(B.GB_CODEC_E4M3, 256, n), 1) == 3.9
    assert 4 * n / B.gb_payload_bytes(B.GB_CODEC_BF16, 256, n) == 2.0


def test_bucket_plan_matches_oracle():
    rng = np.random.default_rng(61)
    cases = [([wl.numel(s) for s in wl.gpt2_small_shapes()], 2, wl.BUCKET_CAP_BYTES, 1),
             ([wl.numel(s) for s in wl.llama_1b_shapes()], 2, wl.BUCKET_CAP_BYTES, 64)]
    for _ in range(100):
        T = int(rng.integers(1, 40))
        cases.append((list(rng.integers(0, 3000, T)), int(rng.choice([2, 4])), int(rng.integers(1, 9000)),
                      int(rng.choice([1, 8, 64]))))
    for numels, eb, cap, pad in cases:
        st, bo, off, bn = B.gb_bucket_plan(numels, eb, cap, pad)
        assert st == B.GB_OK
        obo, ooff, obn = orc.bucket_plan(numels, eb, cap, pad)
        assert bo == list(obo) and off == [int(v) for v in ooff] and bn == [int(v) for v in obn]
    st, *_ = B.gb_bucket_plan([10, 10, 10], 4, 40, 1, max_buckets=2)
    assert st == B.GB_ERR_INVALID_ARG


def test_gpt2_and_llama_bucket_counts():
    st, bo, off, bn = B.gb_bucket_plan([wl.numel(s) for s in wl.gpt2_small_shapes()], 2, wl.BUCKET_CAP_BYTES)
    assert st == 0 and len(bn) == 9 and bn[0] == 50257 * 768
    st, bo, off, bn = B.gb_bucket_plan([wl.numel(s) for s in wl.llama_1b_shapes()], 2, wl.BUCKET_CAP_BYTES)
    assert st == 0 and len(bn) == 90


def test_create_validation_and_topology():
    assert B.gb_create([])[0] == B.GB_ERR_INVALID_ARG
    assert B.gb_create([2, 0])[0] == B.GB_ERR_INVALID_ARG
    assert B.gb_create([1] * 9)[0] == B.GB_ERR_INVALID_ARG
    assert B.gb_create([40, 30])[0] == B.GB_ERR_INVALID_ARG
    st, ctx = B.gb_create([2, 3, 1])
    assert st == B.GB_OK and ctx
    try:
        assert B.gb_world_size(ctx) == 6 and B.gb_n_islands(ctx) == 3
        assert [B.gb_island_first_rank(ctx, i) for i in range(3)] == [0, 2, 5]
        assert [B.gb_island_of_rank(ctx, r) for r in range(6)] == [0, 0, 1, 1, 1, 2]
        assert B.gb_island_size(ctx, 1) == 3 and B.gb_island_size(ctx, 3) == -1
        assert B.gb_context_status(ctx) == B.GB_OK
        assert B.gb_last_error(ctx) == B.GB_OK
    finally:
        assert B.gb_destroy(ctx) == B.GB_OK


def test_argument_errors_need_no_device():
    """Every malformed call is refused before any CUDA call; fake pointers
    are never dereferenced."""
    st, ctx = B.gb_create([2, 2])
    fake = [0x10000 * (r + 1) for r in range(4)]
    try:
        assert B.gb_all_reduce(0, fake, 10, 0, 0, 0, 256) == B.GB_ERR_INVALID_ARG
        assert B.gb_all_reduce(ctx, fake, 10, 9, 0, 0, 256) == B.GB_ERR_UNSUPPORTED_DTYPE
        assert B.gb_all_reduce(ctx, fake, 10, 0, 5, 0, 256) == B.GB_ERR_UNSUPPORTED_OP
        assert B.gb_all_reduce(ctx, fake, 10, B.GB_I32, B.GB_AVG, 0, 256) == B.GB_ERR_UNSUPPORTED_OP
        assert B.gb_all_reduce(ctx, fake, 10, B.GB_F64, B.GB_SUM, 2, 256) == B.GB_ERR_UNSUPPORTED_CODEC
        assert B.gb_island_reduce(ctx, 0, fake, 10, B.GB_F64, fake[0]) == B.GB_ERR_UNSUPPORTED_DTYPE
        assert B.gb_island_broadcast(ctx, 0, fake[0], 10, B.GB_MAX, fake, B.GB_F32) == B.GB_ERR_UNSUPPORTED_OP
        assert B.gb_all_reduce(ctx, fake, 10, 0, 0, 2, 64) == B.GB_ERR_UNSUPPORTED_CODEC
        assert B.gb_all_reduce(ctx, fake, 10, 0, 0, 5, 256) == B.GB_ERR_UNSUPPORTED_CODEC
        assert B.gb_all_reduce(ctx, fake[:3] + [0], 10, 0, 0, 0, 256) == B.GB_ERR_INVALID_ARG
        assert B.gb_all_reduce(ctx, fake[:3] + [0x10008], 10, 0, 0, 0, 256) == B.GB_ERR_MISALIGNED
        assert B.gb_all_reduce(ctx, fake[:3] + [0x10004], 10, 1, 0, 0, 256) == B.GB_ERR_MISALIGNED
        assert "16-byte" in B.gb_last_error_message(ctx)
        assert B.gb_reduce_scatter(ctx, fake, fake, 10, 0, 0, 0, 256) == B.GB_ERR_INVALID_ARG  # 10 % 4
        assert B.gb_broadcast(ctx, fake, 10, 0, 4) == B.GB_ERR_INVALID_ARG
        assert B.gb_island_reduce(ctx, 2, fake, 10, 0, fake[0]) == B.GB_ERR_INVALID_ARG
        assert B.gb_island_reduce(ctx, 0, fake, 10, 0, fake[0] + 4) == B.GB_ERR_MISALIGNED
        assert B.gb_all_reduce(ctx, fake, 1 << 39, 0, 0, 0, 256) == B.GB_ERR_INVALID_ARG
        # the fused halves
        pl = [0x40000, 0x50000]
        assert B.gb_island_reduce_compress(ctx, fake, 10, B.GB_F64, 2, 256, pl) == B.GB_ERR_UNSUPPORTED_DTYPE
        assert B.gb_island_reduce_compress(ctx, fake, 10, 0, 2, 64, pl) == B.GB_ERR_UNSUPPORTED_CODEC
        assert B.gb_island_reduce_compress(ctx, fake, 10, 0, 2, 256, [pl[0], 0]) == B.GB_ERR_INVALID_ARG
        assert B.gb_island_reduce_compress(ctx, fake, 10, 0, 2, 256, [pl[0], pl[1] + 16]) == B.GB_ERR_MISALIGNED
        pl4 = pl + pl[::-1]  # every leader's row
        assert B.gb_decompress_island_broadcast(ctx, pl4, 10, B.GB_I32, B.GB_AVG, 0, 256, fake) == \
            B.GB_ERR_UNSUPPORTED_OP
        assert B.gb_decompress_island_broadcast(ctx, pl4, 10, B.GB_F16, B.GB_SUM, 2, 256, fake) == \
            B.GB_ERR_UNSUPPORTED_CODEC
        # the halves for every dtype and op, and reduce_scatter's second half
        assert B.gb_island_reduce_compress_op(ctx, fake, 10, B.GB_I8, B.GB_AVG, 0, 256, pl) == B.GB_ERR_UNSUPPORTED_OP
        assert B.gb_island_reduce_compress_op(ctx, fake, 10, 9, 0, 0, 256, pl) == B.GB_ERR_UNSUPPORTED_DTYPE
        assert B.gb_island_reduce_compress_op(ctx, fake, 10, B.GB_F64, B.GB_AVG, 1, 256, pl) == \
            B.GB_ERR_UNSUPPORTED_CODEC
        assert B.gb_island_reduce_compress_op(ctx, fake, 10, B.GB_I32, B.GB_MAX, 0, 256, [pl[0], 0]) == \
            B.GB_ERR_INVALID_ARG
        assert B.gb_island_reduce_compress_op(ctx, fake, 0, B.GB_I32, B.GB_MAX, 0, 256, pl) == B.GB_OK
        assert B.gb_decompress_scatter(ctx, pl4, 10, 0, 0, 2, 256, fake) == B.GB_ERR_INVALID_ARG  # 10 % 4
        assert B.gb_decompress_scatter(ctx, pl4, 12, B.GB_U8, B.GB_AVG, 0, 256, fake) == B.GB_ERR_UNSUPPORTED_OP
        assert B.gb_decompress_scatter(ctx, pl4, 12, 0, 0, 2, 256, fake[:3] + [0x10008]) == B.GB_ERR_MISALIGNED
        assert B.gb_decompress_scatter(ctx, pl4, 0, 0, 0, 2, 256, fake) == B.GB_OK
        assert B.gb_island_payload_bytes(B.GB_F32, B.GB_SUM, 2, 256, 1024) == B.gb_payload_bytes(2, 256, 1024)
        assert B.gb_island_payload_bytes(B.GB_BF16, B.GB_MAX, 2, 256, 1024) == 2048
        assert B.gb_island_payload_bytes(B.GB_F16, B.GB_AVG, 0, 256, 1024) == 4096
        assert B.gb_island_payload_bytes(B.GB_I64, B.GB_SUM, 0, 256, 3) == 24
        assert B.gb_island_payload_bytes(B.GB_I64, B.GB_AVG, 0, 256, 3) == 0
        assert B.gb_island_payload_bytes(B.GB_F32, B.GB_SUM, 2, 64, 3) == 0
        assert B.gb_decompress_island_broadcast(ctx, pl4, 10, 0, 0, 7, 256, fake) == B.GB_ERR_UNSUPPORTED_CODEC
        assert B.gb_decompress_island_broadcast(ctx, pl4, 10, 0, 0, 2, 256, fake[:3] + [0]) == B.GB_ERR_INVALID_ARG
        assert B.gb_decompress_island_broadcast(ctx, pl4[:3] + [0], 10, 0, 0, 2, 256, fake) == B.GB_ERR_INVALID_ARG
        assert B.gb_island_reduce_compress(ctx, fake, 0, 0, 2, 256, pl) == B.GB_OK
        assert B.gb_decompress_island_broadcast(ctx, pl4, 0, 1, 1, 3, 128, fake) == B.GB_OK
        assert B.gb_all_reduce_ef(ctx, fake, fake[:2], 16, 0, B.GB_MAX, 0, 256) == B.GB_ERR_UNSUPPORTED_OP
        # bucket sets
        assert B.gb_all_reduce_buckets_ef(ctx, fake, fake[:2], [16], 0, B.GB_MAX, 0, 256) == B.GB_ERR_UNSUPPORTED_OP
        assert B.gb_all_reduce_buckets_ef(ctx, fake, [0x40000, 0], [16], 0, 0, 2, 256) == B.GB_ERR_INVALID_ARG
        assert B.gb_reduce_scatter_buckets(ctx, fake, fake, [10], 0, 0, 2, 256) == B.GB_ERR_INVALID_ARG  # 10 % 4
        assert B.gb_reduce_scatter_buckets(ctx, fake[:3] + [0], fake, [8], 0, 0, 2, 256) == B.GB_ERR_INVALID_ARG
        assert B.gb_reduce_scatter_buckets(ctx, fake, fake, [8], 0, 0, 2, 64) == B.GB_ERR_UNSUPPORTED_CODEC
        assert B.gb_all_gather_buckets(ctx, fake, fake, [8], 9) == B.GB_ERR_UNSUPPORTED_DTYPE
        assert B.gb_all_gather_buckets(ctx, fake, fake[:3] + [0x10008], [8], 0) == B.GB_ERR_MISALIGNED
        assert B.gb_reduce_scatter_buckets(ctx, [0] * 8, [0] * 8, [0, 0], 0, 0, 2, 256) == B.GB_OK  # empty
        assert B.gb_all_gather_buckets(ctx, [0] * 4, [0] * 4, [0], 1) == B.GB_OK
        # n == 0 is a valid no-op, answered without a device
        assert B.gb_all_reduce(ctx, fake, 0, 0, 0, 2, 256) == B.GB_OK
        assert B.gb_all_gather(ctx, fake, fake, 0, 1) == B.GB_OK
        # none of these is sticky; the last one is remembered
        assert B.gb_context_status(ctx) == B.GB_OK
        assert B.gb_last_error(ctx) == B.GB_ERR_MISALIGNED  # the last refused call: the misaligned bucket set
        assert B.gb_debug_inject(ctx, 77) == B.GB_ERR_INVALID_ARG
        # the fixed-buffer all_reduce checks its arguments the same way, before any device call
        na = B.gb_all_reduce_noalloc
        assert na(0, fake, 10, 0, 0, 0, 256) == B.GB_ERR_INVALID_ARG
        assert na(ctx, fake, 10, B.GB_F64, 0, 0, 256) == B.GB_ERR_UNSUPPORTED_DTYPE
        assert na(ctx, fake, 10, 0, B.GB_MAX, 0, 256) == B.GB_ERR_UNSUPPORTED_OP
        assert na(ctx, fake, 10, 0, 0, 2, 64) == B.GB_ERR_UNSUPPORTED_CODEC
        assert na(ctx, fake[:3] + [0], 10, 0, 0, 0, 256) == B.GB_ERR_INVALID_ARG
        assert na(ctx, fake[:3] + [0x10008], 10, 0, 0, 0, 256) == B.GB_ERR_MISALIGNED
        assert na(ctx, fake, 1 << 39, 0, 0, 0, 256) == B.GB_ERR_INVALID_ARG
        # 2 x 2 slots of 4n bytes beyond the fixed array: refused from the sizes alone
        assert na(ctx, fake, B.GB_NOALLOC_DEVICE_BYTES // 16 + 256, 0, 0, 0, 256) == B.GB_ERR_TOO_LARGE
        assert "exceed" in B.gb_last_error_message(ctx)
        assert na(ctx, fake, 0, 0, 0, 2, 256) == B.GB_OK
        # the device-mismatch hook is accepted; on an unbound context it is dropped
        assert B.gb_debug_inject(ctx, B.GB_INJECT_OTHER_DEVICE) == B.GB_OK
        assert B.gb_debug_inject(ctx, 0) == B.GB_OK
        assert B.gb_context_status(ctx) == B.GB_OK
    finally:
        B.gb_destroy(ctx)


def test_no_device_is_reported_not_sticky():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    st, ctx = B.gb_create([1, 1])
    fake = [0x10000, 0x20000]
    try:
        assert B.gb_all_reduce(ctx, fake, 16, 0, 0, 0, 256) == B.GB_ERR_NO_DEVICE
        assert B.gb_context_status(ctx) == B.GB_OK
        assert "device" in B.gb_last_error_message(ctx)
    finally:
        B.gb_destroy(ctx)


def test_plain_c_caller(tmp_path):
    """include/gb.h is a C99 header: a C program built against it alone links
    libgb.so and gets the host-only answers (topology, payload sizes,
    argument errors before any CUDA call, the bucket plan)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    exe = str(tmp_path / "c_abi_host")
    libdir = os.path.dirname(B.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_host.c"),
                    "-L", libdir, "-lgb", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    got = dict(line.split(" ", 1) for line in out.strip().splitlines())
    assert got["create"] == "0" and got["destroy"] == "0"
    assert got["world"] == "6" and got["islands"] == "3"
    assert got["first2"] == "5" and got["island_of4"] == "1"
    assert int(got["payload_e4m3"]) == B.gb_payload_bytes(B.GB_CODEC_E4M3, 256, 6553600) == 6656000
    assert int(got["payload_bf16"]) == 2000
    assert int(got["scales_off"]) == B.gb_payload_scales_offset(B.GB_CODEC_E5M2, 128, 1001)
    assert got["null_bufs"] == str(B.GB_ERR_INVALID_ARG) and got["sticky"] == "0"
    assert got["status_string"] == "GB_ERR_MISALIGNED"
    _, _, bn = orc.bucket_plan([600, 500, 1200, 10, 990], 4, 4000, 1)
    assert got["plan"].split() == ["0", str(len(bn))] + [str(int(v)) for v in bn]


def test_host_rows_detection():
    """Context.all_reduce_host takes the rows entry point only for equally
    spaced, ascending rows of one storage at least a row apart."""
    import torch
    from cross_vendor_gradient_gb300.api import _row_pitch
    blk = torch.zeros((4, 1000))
    assert _row_pitch(list(blk.unbind(0))) == 4000
    padded = torch.zeros((4, 1040))
    assert _row_pitch([padded[r, 20:1020] for r in range(4)]) == 4160
    assert _row_pitch([blk[r] for r in (3, 2, 1, 0)]) is None  # descending
    assert _row_pitch([blk[r] for r in (0, 1, 3, 2)]) is None  # not equally spaced
    assert _row_pitch([torch.zeros(1000) for _ in range(4)]) is None  # separate storages
    assert _row_pitch([blk[0]]) is None  # one rank: the pointer entry point
    flat = torch.zeros(4000)
    assert _row_pitch([flat[r * 900:r * 900 + 1000] for r in range(4)]) is None  # overlapping rows
