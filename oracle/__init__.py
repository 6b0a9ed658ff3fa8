"""Oracle for the reduce-bridge-broadcast gradient all_reduce (Python side).

TEST INFRASTRUCTURE ONLY.  A thin ctypes wrapper over ``oracle.c``: plain,
slow, single-threaded CPU code that states what the collectives compute.  It
shares no code with the CUDA library; only ``tests/``, the smoke check and the
benchmark's CPU-baseline / reference legs may import it.

Conventions: float32 buffers are ``np.float32`` arrays; bfloat16 buffers are
``np.uint16`` arrays holding the bf16 bit patterns.  Islands are contiguous
blocks of global ranks, given by their sizes.
"""
import ctypes
import os

import numpy as np

from . import build as _build

DT_F32, DT_BF16, DT_F16, DT_F64, DT_I8, DT_U8, DT_I32, DT_I64 = 0, 1, 2, 3, 4, 5, 6, 7
OP_SUM, OP_AVG, OP_MAX, OP_MIN = 0, 1, 2, 3
CODEC_NONE, CODEC_BF16, CODEC_E4M3, CODEC_E5M2 = 0, 1, 2, 3

CODECS = {"none": CODEC_NONE, "bf16": CODEC_BF16, "e4m3": CODEC_E4M3, "e5m2": CODEC_E5M2}
OPS = {"sum": OP_SUM, "avg": OP_AVG, "max": OP_MAX, "min": OP_MIN}
# numpy dtype of a rank buffer -> oracle dtype id (bf16 buffers are uint16 bit patterns)
_NP_DT = {np.dtype(np.float32): DT_F32, np.dtype(np.uint16): DT_BF16, np.dtype(np.float16): DT_F16,
          np.dtype(np.float64): DT_F64, np.dtype(np.int8): DT_I8, np.dtype(np.uint8): DT_U8,
          np.dtype(np.int32): DT_I32, np.dtype(np.int64): DT_I64}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        c_size = ctypes.c_size_t
        vp = ctypes.c_void_p
        L.orc_bf16_to_f32.restype = ctypes.c_float
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f32_to_bf16.restype = ctypes.c_uint16
        L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
        L.orc_fp8_max.restype = ctypes.c_double
        L.orc_fp8_max.argtypes = [ctypes.c_int]
        L.orc_fp8_value.restype = ctypes.c_double
        L.orc_fp8_value.argtypes = [ctypes.c_uint8, ctypes.c_int]
        L.orc_fp8_encode.restype = ctypes.c_uint8
        L.orc_fp8_encode.argtypes = [ctypes.c_double, ctypes.c_int]
        L.orc_fp8_encode_bruteforce.restype = ctypes.c_uint8
        L.orc_fp8_encode_bruteforce.argtypes = [ctypes.c_double, ctypes.c_int]
        L.orc_block_scale_exponent.restype = ctypes.c_int
        L.orc_block_scale_exponent.argtypes = [ctypes.c_float, ctypes.c_int]
        L.orc_island_sum.restype = None
        L.orc_island_sum.argtypes = [ctypes.c_int, vp, ctypes.c_int, c_size, vp]
        L.orc_n_blocks.restype = c_size
        L.orc_n_blocks.argtypes = [c_size, ctypes.c_int]
        L.orc_encode.restype = None
        L.orc_encode.argtypes = [vp, c_size, ctypes.c_int, ctypes.c_int, vp, vp]
        L.orc_decode.restype = None
        L.orc_decode.argtypes = [vp, vp, c_size, ctypes.c_int, ctypes.c_int, vp]
        L.orc_bridge_total.restype = None
        L.orc_bridge_total.argtypes = [ctypes.c_int, vp, vp, c_size, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, vp]
        L.orc_rbb_total.restype = ctypes.c_int
        L.orc_rbb_total.argtypes = [ctypes.c_int, vp, vp, c_size, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]
        for name in ("orc_all_reduce", "orc_reduce_scatter"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_int, vp, vp, vp, c_size, ctypes.c_int, ctypes.c_int,
                          ctypes.c_int, ctypes.c_int]
        L.orc_all_gather.restype = None
        L.orc_all_gather.argtypes = [ctypes.c_int, vp, vp, c_size]
        L.orc_broadcast.restype = None
        L.orc_broadcast.argtypes = [ctypes.c_int, vp, vp, c_size, ctypes.c_int]
        L.orc_bucket_plan.restype = ctypes.c_int
        L.orc_bucket_plan.argtypes = [vp, ctypes.c_int, c_size, c_size, c_size, vp, vp, vp,
                                      ctypes.c_int]
        L.orc_encode_ef.restype = None
        L.orc_encode_ef.argtypes = [vp, c_size, ctypes.c_int, ctypes.c_int, vp, vp, vp]
        L.orc_all_reduce_ef.restype = ctypes.c_int
        L.orc_all_reduce_ef.argtypes = [ctypes.c_int, vp, vp, vp, c_size, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, vp]
        for name in ("orc_all_reduce_exact", "orc_reduce_scatter_exact"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.c_int, vp, vp, vp, c_size, ctypes.c_int, ctypes.c_int]
        L.orc_all_reduce_sharded.restype = ctypes.c_int
        L.orc_all_reduce_sharded.argtypes = [ctypes.c_int, vp, vp, vp, c_size, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, vp]
        L.orc_f16_to_f32.restype = ctypes.c_float
        L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f32_to_f16.restype = ctypes.c_uint16
        L.orc_f32_to_f16.argtypes = [ctypes.c_float]
        L.orc_f32_to_f16_array.restype = None
        L.orc_f32_to_f16_array.argtypes = [vp, c_size, vp]
        L.orc_fp8_encode_f32_array.restype = None
        L.orc_fp8_encode_f32_array.argtypes = [vp, c_size, ctypes.c_int, vp]
        L.orc_f32_to_bf16_array.restype = None
        L.orc_f32_to_bf16_array.argtypes = [vp, c_size, vp]
        _lib = L
    return _lib


# ---------------------------------------------------------------- helpers ---

def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _ptr_array(arrays):
    arr = (ctypes.c_void_p * max(1, len(arrays)))(*[a.ctypes.data for a in arrays])
    return ctypes.cast(arr, ctypes.c_void_p), arr


def _dtype_id(a: np.ndarray) -> int:
    if a.dtype in _NP_DT:
        return _NP_DT[a.dtype]
    raise TypeError("unsupported rank buffer dtype %s" % a.dtype)


def _codec_id(codec) -> int:
    return CODECS[codec] if isinstance(codec, str) else int(codec)


def _op_id(op) -> int:
    return OPS[op] if isinstance(op, str) else int(op)


def code_dtype(codec) -> np.dtype:
    c = _codec_id(codec)
    return {CODEC_NONE: np.float32, CODEC_BF16: np.uint16}.get(c, np.uint8)


def n_blocks(n: int, block: int) -> int:
    return (n + block - 1) // block


# ------------------------------------------------------------ conversions ---

def bf16_to_f32(h: int) -> float:
    return lib().orc_bf16_to_f32(int(h))


def f32_to_bf16(x: float) -> int:
    return lib().orc_f32_to_bf16(float(x))


def f32_to_bf16_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16_array(_ptr(x), x.size, _ptr(out))
    return out


def bf16_bits_to_f32_array(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 patterns (a 16-bit shift)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f16_to_f32(h: int) -> float:
    return lib().orc_f16_to_f32(int(h))


def f32_to_f16_array(x: np.ndarray) -> np.ndarray:
    """float16 bit patterns (uint16) of float32 inputs, nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_f16_array(_ptr(x), x.size, _ptr(out))
    return out


def fp8_max(codec) -> float:
    return lib().orc_fp8_max(_codec_id(codec))


def fp8_value(code: int, codec) -> float:
    return lib().orc_fp8_value(int(code), _codec_id(codec))


def fp8_encode(y: float, codec) -> int:
    return lib().orc_fp8_encode(float(y), _codec_id(codec))


def fp8_encode_bruteforce(y: float, codec) -> int:
    return lib().orc_fp8_encode_bruteforce(float(y), _codec_id(codec))


def fp8_encode_f32_array(y: np.ndarray, codec) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, np.uint8)
    lib().orc_fp8_encode_f32_array(_ptr(y), y.size, _codec_id(codec), _ptr(out))
    return out


def block_scale_exponent(absmax: float, codec) -> int:
    return lib().orc_block_scale_exponent(float(absmax), _codec_id(codec))


# ---------------------------------------------------------- collective steps

def island_sum(ranks) -> np.ndarray:
    """Float32 island sum of the given rank buffers, in the order given."""
    ranks = [np.ascontiguousarray(r) for r in ranks]
    n = ranks[0].size
    dt = _dtype_id(ranks[0])
    s = np.empty(n, np.float32)
    p, _keep = _ptr_array(ranks)
    lib().orc_island_sum(len(ranks), p, dt, n, _ptr(s))
    return s


def encode(s: np.ndarray, codec, block: int = 256):
    """Bridge payload of an island sum: (codes, scales).  scales is an empty
    float32 array for the none and bf16 codecs."""
    s = np.ascontiguousarray(s, dtype=np.float32)
    c = _codec_id(codec)
    n = s.size
    codes = np.empty(n, code_dtype(c))
    nb = n_blocks(n, block) if c in (CODEC_E4M3, CODEC_E5M2) else 0
    scales = np.empty(nb, np.float32)
    lib().orc_encode(_ptr(s), n, c, block, _ptr(codes), _ptr(scales))
    return codes, scales


def decode(codes: np.ndarray, scales: np.ndarray, codec, block: int = 256) -> np.ndarray:
    c = _codec_id(codec)
    codes = np.ascontiguousarray(codes, dtype=code_dtype(c))
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    out = np.empty(codes.size, np.float32)
    lib().orc_decode(_ptr(codes), _ptr(scales), codes.size, c, block, _ptr(out))
    return out


def bridge_total(payloads, codec, block: int, op, world_size: int) -> np.ndarray:
    """Decode-and-add of I payloads [(codes, scales), ...] in island order,
    then the AVG division."""
    c = _codec_id(codec)
    codes = [np.ascontiguousarray(p[0], dtype=code_dtype(c)) for p in payloads]
    scales = [np.ascontiguousarray(p[1], dtype=np.float32) for p in payloads]
    scales = [s if s.size else np.zeros(1, np.float32) for s in scales]
    n = codes[0].size
    t = np.empty(n, np.float32)
    pc, _k1 = _ptr_array(codes)
    ps, _k2 = _ptr_array(scales)
    lib().orc_bridge_total(len(codes), pc, ps, n, c, block, _op_id(op), world_size, _ptr(t))
    return t


def rbb_total(ranks, island_sizes, op="sum", codec="none", block: int = 256, intermediates=False):
    """Float32 total of reduce-bridge-broadcast (after AVG), optionally with
    the island sums, codes and scales of every island."""
    ranks = [np.ascontiguousarray(r) for r in ranks]
    sizes = np.asarray(island_sizes, dtype=np.int32)
    assert int(sizes.sum()) == len(ranks)
    I = len(sizes)
    n = ranks[0].size
    c = _codec_id(codec)
    eff = CODEC_NONE if I == 1 else c
    t = np.empty(n, np.float32)
    sums = np.empty((I, n), np.float32)
    codes = np.empty((I, n), code_dtype(eff))
    nb = n_blocks(n, block) if eff in (CODEC_E4M3, CODEC_E5M2) else 0
    scales = np.empty((I, max(nb, 0)), np.float32)
    p, _keep = _ptr_array(ranks)
    rc = lib().orc_rbb_total(I, _ptr(sizes), p, n, _dtype_id(ranks[0]), _op_id(op), c, block,
                             _ptr(t), _ptr(sums), _ptr(codes), _ptr(scales) if nb else None)
    if rc:
        raise MemoryError("oracle allocation failed")
    if intermediates:
        return t, {"island_sums": sums, "codes": codes, "scales": scales, "codec": eff}
    return t


def _exact(ranks, op) -> bool:
    """MAX / MIN and the float16, float64 and integer dtypes take the exact
    path (no codec: it stays exact or is not offered)."""
    return _op_id(op) in (OP_MAX, OP_MIN) or _dtype_id(ranks[0]) not in (DT_F32, DT_BF16)


def _exact_call(name, ranks, island_sizes, op, out_elems):
    sizes = np.asarray(island_sizes, dtype=np.int32)
    outs = [np.empty(out_elems, ranks[0].dtype) for _ in ranks]
    pi, _k1 = _ptr_array(ranks)
    po, _k2 = _ptr_array(outs)
    rc = getattr(lib(), name)(len(sizes), _ptr(sizes), pi, po, ranks[0].size, _dtype_id(ranks[0]), _op_id(op))
    if rc:
        raise ValueError("oracle %s refused (%d): AVG needs a float dtype, RS needs n %% W == 0" % (name, rc))
    return outs


def all_reduce(ranks, island_sizes, op="sum", codec="none", block: int = 256):
    """Outputs of every rank (new arrays, rank dtype)."""
    ranks = [np.ascontiguousarray(r) for r in ranks]
    if _exact(ranks, op):
        return _exact_call("orc_all_reduce_exact", ranks, island_sizes, op, ranks[0].size)
    sizes = np.asarray(island_sizes, dtype=np.int32)
    outs = [np.empty_like(r) for r in ranks]
    pi, _k1 = _ptr_array(ranks)
    po, _k2 = _ptr_array(outs)
    rc = lib().orc_all_reduce(len(sizes), _ptr(sizes), pi, po, ranks[0].size, _dtype_id(ranks[0]),
                              _op_id(op), _codec_id(codec), block)
    if rc:
        raise RuntimeError("oracle all_reduce failed (%d)" % rc)
    return outs


def reduce_scatter(ranks, island_sizes, op="sum", codec="none", block: int = 256):
    ranks = [np.ascontiguousarray(r) for r in ranks]
    sizes = np.asarray(island_sizes, dtype=np.int32)
    W = len(ranks)
    n = ranks[0].size
    if n % W:
        raise ValueError("reduce_scatter needs n divisible by the world size")
    if _exact(ranks, op):
        return _exact_call("orc_reduce_scatter_exact", ranks, island_sizes, op, n // W)
    outs = [np.empty(n // W, ranks[0].dtype) for _ in ranks]
    pi, _k1 = _ptr_array(ranks)
    po, _k2 = _ptr_array(outs)
    rc = lib().orc_reduce_scatter(len(sizes), _ptr(sizes), pi, po, n, _dtype_id(ranks[0]),
                                  _op_id(op), _codec_id(codec), block)
    if rc:
        raise RuntimeError("oracle reduce_scatter failed (%d)" % rc)
    return outs


def all_gather(ranks):
    ranks = [np.ascontiguousarray(r) for r in ranks]
    W = len(ranks)
    outs = [np.empty(W * ranks[0].size, ranks[0].dtype) for _ in ranks]
    pi, _k1 = _ptr_array(ranks)
    po, _k2 = _ptr_array(outs)
    lib().orc_all_gather(W, pi, po, ranks[0].nbytes)
    return outs


def broadcast(ranks, src: int):
    ranks = [np.ascontiguousarray(r) for r in ranks]
    outs = [np.empty_like(r) for r in ranks]
    pi, _k1 = _ptr_array(ranks)
    po, _k2 = _ptr_array(outs)
    lib().orc_broadcast(len(ranks), pi, po, ranks[0].nbytes, int(src))
    return outs


def bucket_plan(numels, elem_bytes: int, cap_bytes: int = 25 * 1024 * 1024, pad_elems: int = 1):
    """(bucket_of[t], offset[t], bucket_numel[b]) of the greedy bucket plan."""
    numels = np.ascontiguousarray(numels, dtype=np.uint64)
    T = numels.size
    bucket_of = np.empty(max(T, 1), np.int32)
    offset = np.empty(max(T, 1), np.uint64)
    bucket_numel = np.empty(max(T, 1), np.uint64)
    nb = lib().orc_bucket_plan(_ptr(numels), T, elem_bytes, cap_bytes, pad_elems, _ptr(bucket_of),
                               _ptr(offset), _ptr(bucket_numel), max(T, 1))
    if nb < 0:
        raise RuntimeError("bucket plan overflow")
    return bucket_of[:T], offset[:T], bucket_numel[:nb]


# ------------------------------------------------------------ error feedback

def encode_ef(s: np.ndarray, residual: np.ndarray, codec, block: int = 256):
    """Encode s + residual; `residual` (float32, updated in place) becomes
    (s + residual) - dec(codes).  Returns (codes, scales)."""
    s = np.ascontiguousarray(s, dtype=np.float32)
    assert residual.dtype == np.float32 and residual.flags.c_contiguous and residual.size == s.size
    c = _codec_id(codec)
    n = s.size
    codes = np.empty(n, code_dtype(c))
    nb = n_blocks(n, block) if c in (CODEC_E4M3, CODEC_E5M2) else 0
    scales = np.empty(max(nb, 1), np.float32)
    lib().orc_encode_ef(_ptr(s), n, c, block, _ptr(residual), _ptr(codes), _ptr(scales))
    return codes, scales[:nb]


def all_reduce_ef(ranks, island_sizes, residuals, op="sum", codec="none", block: int = 256):
    """all_reduce with one error-feedback residual per island (float32 arrays
    of n, updated in place).  Returns the outputs of every rank."""
    ranks = [np.ascontiguousarray(r) for r in ranks]
    sizes = np.asarray(island_sizes, dtype=np.int32)
    assert len(residuals) == len(sizes)
    for r in residuals:
        assert r.dtype == np.float32 and r.flags.c_contiguous and r.size == ranks[0].size
    outs = [np.empty_like(r) for r in ranks]
    pi, _k1 = _ptr_array(ranks)
    po, _k2 = _ptr_array(outs)
    pr, _k3 = _ptr_array(residuals)
    rc = lib().orc_all_reduce_ef(len(sizes), _ptr(sizes), pi, po, ranks[0].size, _dtype_id(ranks[0]),
                                 _op_id(op), _codec_id(codec), block, pr)
    if rc:
        raise RuntimeError("oracle all_reduce_ef failed (%d)" % rc)
    return outs


# ------------------------------------------------------------ sharded bridge

def all_reduce_sharded(ranks, island_sizes, op="sum", codec="none", block: int = 256, with_segment=False):
    """all_reduce under the sharded-bridge policy: k = smallest island size
    segments of ceil(n / k) rounded up to 256 elements, each all_reduced over
    its own link, then all_gathered.  Returns the outputs of every rank (and
    the segment length with with_segment)."""
    ranks = [np.ascontiguousarray(r) for r in ranks]
    sizes = np.asarray(island_sizes, dtype=np.int32)
    outs = [np.empty_like(r) for r in ranks]
    pi, _k1 = _ptr_array(ranks)
    po, _k2 = _ptr_array(outs)
    seg = np.zeros(1, np.uint64)
    rc = lib().orc_all_reduce_sharded(len(sizes), _ptr(sizes), pi, po, ranks[0].size, _dtype_id(ranks[0]),
                                      _op_id(op), _codec_id(codec), block, _ptr(seg))
    if rc:
        raise RuntimeError("oracle all_reduce_sharded failed (%d)" % rc)
    return (outs, int(seg[0])) if with_segment else outs
