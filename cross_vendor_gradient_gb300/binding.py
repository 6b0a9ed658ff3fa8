"""ctypes binding of libgb: one Python function per C entry point, same name,
argument marshalling only (pointers and sizes are Python ints, arrays are
Python sequences).  Every function returns the raw ``gb_status`` integer.

All computation happens in libgb's CUDA kernels; if the library is missing
this module raises on import of the library instead of falling back.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgb.so")

# gb_status
GB_OK = 0
GB_ERR_INVALID_ARG = 1
GB_ERR_UNSUPPORTED_DTYPE = 2
GB_ERR_UNSUPPORTED_OP = 3
GB_ERR_UNSUPPORTED_CODEC = 4
GB_ERR_MISALIGNED = 5
GB_ERR_ALLOC = 6
GB_ERR_CUDA = 7
GB_ERR_BRIDGE = 8
GB_ERR_CONTEXT_FAILED = 9
GB_ERR_NO_DEVICE = 10
GB_ERR_TOO_LARGE = 11
# gb_dtype / gb_op / gb_codec
GB_F32, GB_BF16, GB_F16, GB_F64, GB_I8, GB_U8, GB_I32, GB_I64 = 0, 1, 2, 3, 4, 5, 6, 7
GB_SUM, GB_AVG, GB_MAX, GB_MIN = 0, 1, 2, 3
GB_CODEC_NONE, GB_CODEC_BF16, GB_CODEC_E4M3, GB_CODEC_E5M2 = 0, 1, 2, 3
GB_MAX_RANKS = 64
GB_MAX_ISLANDS = 8
GB_N_PHASES = 3
GB_INJECT_BRIDGE = 1
GB_INJECT_ALLOC = 2
GB_INJECT_OTHER_DEVICE = 3
GB_NOALLOC_DEVICE_BYTES = 64 << 20
GB_NOALLOC_HOST_BYTES = 32 << 20

_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_i = ctypes.c_int
_P = ctypes.POINTER

# name -> (restype, argtypes)
SIGNATURES = {
    "gb_create": (_i, [_P(_vp), _i, _P(_i)]),
    "gb_destroy": (_i, [_vp]),
    "gb_world_size": (_i, [_vp]),
    "gb_n_islands": (_i, [_vp]),
    "gb_island_size": (_i, [_vp, _i]),
    "gb_island_first_rank": (_i, [_vp, _i]),
    "gb_island_of_rank": (_i, [_vp, _i]),
    "gb_reserve": (_i, [_vp, _sz, _i, _i, _i]),
    "gb_set_pipeline": (_i, [_vp, _sz, _i]),
    "gb_context_status": (_i, [_vp]),
    "gb_last_error": (_i, [_vp]),
    "gb_last_error_message": (ctypes.c_char_p, [_vp]),
    "gb_status_string": (ctypes.c_char_p, [_i]),
    "gb_payload_bytes": (_sz, [_i, _i, _sz]),
    "gb_payload_scales_offset": (_sz, [_i, _i, _sz]),
    "gb_island_reduce": (_i, [_vp, _i, _P(_vp), _sz, _i, _vp, _vp]),
    "gb_bridge_compress": (_i, [_vp, _vp, _sz, _i, _i, _vp, _vp]),
    "gb_bridge_decompress_accumulate": (_i, [_vp, _vp, _sz, _i, _i, _vp, _i, _vp]),
    "gb_island_broadcast": (_i, [_vp, _i, _vp, _sz, _i, _P(_vp), _i, _vp]),
    "gb_set_sharded_bridge": (_i, [_vp, _i]),
    "gb_island_reduce_compress": (_i, [_vp, _P(_vp), _sz, _i, _i, _i, _P(_vp), _vp]),
    "gb_island_reduce_compress_ef": (_i, [_vp, _P(_vp), _P(_vp), _sz, _i, _i, _i, _P(_vp), _vp]),
    "gb_decompress_island_broadcast": (_i, [_vp, _P(_vp), _sz, _i, _i, _i, _i, _P(_vp), _vp]),
    "gb_island_payload_bytes": (_sz, [_i, _i, _i, _i, _sz]),
    "gb_island_reduce_compress_op": (_i, [_vp, _P(_vp), _sz, _i, _i, _i, _i, _P(_vp), _vp]),
    "gb_decompress_scatter": (_i, [_vp, _P(_vp), _sz, _i, _i, _i, _i, _P(_vp), _vp]),
    "gb_all_reduce": (_i, [_vp, _P(_vp), _sz, _i, _i, _i, _i, _vp]),
    "gb_all_reduce_ef": (_i, [_vp, _P(_vp), _P(_vp), _sz, _i, _i, _i, _i, _vp]),
    "gb_reduce_scatter": (_i, [_vp, _P(_vp), _P(_vp), _sz, _i, _i, _i, _i, _vp]),
    "gb_all_gather": (_i, [_vp, _P(_vp), _P(_vp), _sz, _i, _vp]),
    "gb_broadcast": (_i, [_vp, _P(_vp), _sz, _i, _i, _vp]),
    "gb_all_reduce_host": (_i, [_vp, _P(_vp), _sz, _i, _i, _i, _i, _vp]),
    "gb_all_reduce_host_rows": (_i, [_vp, _vp, _sz, _sz, _i, _i, _i, _i, _vp]),
    "gb_bucket_plan": (_i, [_P(_sz), _i, _sz, _sz, _sz, _P(_i), _P(_sz), _P(_sz), _i, _P(_i)]),
    "gb_all_reduce_buckets": (_i, [_vp, _i, _P(_vp), _P(_sz), _i, _i, _i, _i, _vp]),
    "gb_all_reduce_buckets_ef": (_i, [_vp, _i, _P(_vp), _P(_vp), _P(_sz), _i, _i, _i, _i, _vp]),
    "gb_reduce_scatter_buckets": (_i, [_vp, _i, _P(_vp), _P(_vp), _P(_sz), _i, _i, _i, _i, _vp]),
    "gb_all_gather_buckets": (_i, [_vp, _i, _P(_vp), _P(_vp), _P(_sz), _i, _vp]),
    "gb_set_phase_timing": (_i, [_vp, _i]),
    "gb_phase_times": (_i, [_vp, _i, _P(ctypes.c_float)]),
    "gb_last_phase_times": (_i, [_vp, _P(ctypes.c_float)]),
    "gb_debug_inject": (_i, [_vp, _i]),
    "gb_all_reduce_noalloc": (_i, [_vp, _P(_vp), _sz, _i, _i, _i, _i, _vp]),
    "gb_kernel_launch_count": (ctypes.c_uint64, []),
}

_lib = None


def lib():
    """The loaded libgb (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libgb.so is not built (expected at %s); build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` or "
                "`python -m cross_vendor_gradient_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptrs(seq):
    arr = (_vp * max(1, len(seq)))(*[int(p) if p is not None else None for p in seq])
    return arr


def _sizes(seq):
    return (_sz * max(1, len(seq)))(*[int(v) for v in seq])


# ------------------------------------------------------------ entry points

def gb_create(island_sizes):
    """Returns (status, ctx_handle_int)."""
    h = _vp()
    arr = (_i * max(1, len(island_sizes)))(*[int(v) for v in island_sizes])
    st = lib().gb_create(ctypes.byref(h), len(island_sizes), arr)
    return st, (h.value or 0)


def gb_destroy(ctx):
    return lib().gb_destroy(ctx)


def gb_world_size(ctx):
    return lib().gb_world_size(ctx)


def gb_n_islands(ctx):
    return lib().gb_n_islands(ctx)


def gb_island_size(ctx, island):
    return lib().gb_island_size(ctx, island)


def gb_island_first_rank(ctx, island):
    return lib().gb_island_first_rank(ctx, island)


def gb_island_of_rank(ctx, rank):
    return lib().gb_island_of_rank(ctx, rank)


def gb_reserve(ctx, n, dtype, codec, block):
    return lib().gb_reserve(ctx, n, dtype, codec, block)


def gb_set_pipeline(ctx, chunk_bytes, use_graphs=1):
    return lib().gb_set_pipeline(ctx, int(chunk_bytes), 1 if use_graphs else 0)


def gb_context_status(ctx):
    return lib().gb_context_status(ctx)


def gb_last_error(ctx):
    return lib().gb_last_error(ctx)


def gb_last_error_message(ctx):
    m = lib().gb_last_error_message(ctx)
    return m.decode() if m else ""


def gb_status_string(status):
    return lib().gb_status_string(status).decode()


def gb_payload_bytes(codec, block, n):
    return lib().gb_payload_bytes(codec, block, n)


def gb_payload_scales_offset(codec, block, n):
    return lib().gb_payload_scales_offset(codec, block, n)


def gb_island_reduce(ctx, island, rank_bufs, n, dtype, island_sum, stream=0):
    return lib().gb_island_reduce(ctx, island, _ptrs(rank_bufs), n, dtype, island_sum, stream)


def gb_bridge_compress(ctx, island_sum, n, codec, block, payload, stream=0):
    return lib().gb_bridge_compress(ctx, island_sum, n, codec, block, payload, stream)


def gb_bridge_decompress_accumulate(ctx, payload, n, codec, block, accum, accumulate, stream=0):
    return lib().gb_bridge_decompress_accumulate(ctx, payload, n, codec, block, accum,
                                                 1 if accumulate else 0, stream)


def gb_island_broadcast(ctx, island, total, n, op, rank_bufs, dtype, stream=0):
    return lib().gb_island_broadcast(ctx, island, total, n, op, _ptrs(rank_bufs), dtype, stream)


def gb_set_sharded_bridge(ctx, on):
    return lib().gb_set_sharded_bridge(ctx, 1 if on else 0)


def gb_island_reduce_compress(ctx, rank_bufs, n, dtype, codec, block, payloads, stream=0):
    return lib().gb_island_reduce_compress(ctx, _ptrs(rank_bufs), n, dtype, codec, block, _ptrs(payloads),
                                           stream)


def gb_island_reduce_compress_ef(ctx, rank_bufs, residuals, n, dtype, codec, block, payloads, stream=0):
    return lib().gb_island_reduce_compress_ef(ctx, _ptrs(rank_bufs), _ptrs(residuals), n, dtype, codec, block,
                                              _ptrs(payloads), stream)


def gb_decompress_island_broadcast(ctx, payloads, n, dtype, op, codec, block, rank_bufs, stream=0):
    return lib().gb_decompress_island_broadcast(ctx, _ptrs(payloads), n, dtype, op, codec, block,
                                                _ptrs(rank_bufs), stream)


def gb_island_payload_bytes(dtype, op, codec, block, n):
    return lib().gb_island_payload_bytes(dtype, op, codec, block, n)


def gb_island_reduce_compress_op(ctx, rank_bufs, n, dtype, op, codec, block, payloads, stream=0):
    return lib().gb_island_reduce_compress_op(ctx, _ptrs(rank_bufs), n, dtype, op, codec, block, _ptrs(payloads),
                                              stream)


def gb_decompress_scatter(ctx, payloads, n, dtype, op, codec, block, out, stream=0):
    return lib().gb_decompress_scatter(ctx, _ptrs(payloads), n, dtype, op, codec, block, _ptrs(out), stream)


def gb_all_reduce(ctx, rank_bufs, n, dtype, op, codec, block, stream=0):
    return lib().gb_all_reduce(ctx, _ptrs(rank_bufs), n, dtype, op, codec, block, stream)


def gb_all_reduce_ef(ctx, rank_bufs, residuals, n, dtype, op, codec, block, stream=0):
    return lib().gb_all_reduce_ef(ctx, _ptrs(rank_bufs), _ptrs(residuals), n, dtype, op, codec, block, stream)


def gb_reduce_scatter(ctx, inp, out, n_in, dtype, op, codec, block, stream=0):
    return lib().gb_reduce_scatter(ctx, _ptrs(inp), _ptrs(out), n_in, dtype, op, codec, block, stream)


def gb_all_gather(ctx, inp, out, n_in, dtype, stream=0):
    return lib().gb_all_gather(ctx, _ptrs(inp), _ptrs(out), n_in, dtype, stream)


def gb_broadcast(ctx, rank_bufs, n, dtype, src, stream=0):
    return lib().gb_broadcast(ctx, _ptrs(rank_bufs), n, dtype, src, stream)


def gb_all_reduce_host(ctx, host_bufs, n, dtype, op, codec, block, stream=0):
    return lib().gb_all_reduce_host(ctx, _ptrs(host_bufs), n, dtype, op, codec, block, stream)


def gb_all_reduce_host_rows(ctx, host, pitch, n, dtype, op, codec, block, stream=0):
    return lib().gb_all_reduce_host_rows(ctx, host, pitch, n, dtype, op, codec, block, stream)


def gb_bucket_plan(numel, elem_bytes, cap_bytes, pad_elems=1, max_buckets=None):
    """Returns (status, bucket_of list, offset list, bucket_numel list)."""
    T = len(numel)
    mb = T if max_buckets is None else max_buckets
    bo = (_i * max(1, T))()
    off = (_sz * max(1, T))()
    bn = (_sz * max(1, mb))()
    nb = _i(0)
    st = lib().gb_bucket_plan(_sizes(numel), T, elem_bytes, cap_bytes, pad_elems, bo, off, bn, mb,
                              ctypes.byref(nb))
    return st, list(bo[:T]), list(off[:T]), list(bn[:nb.value])


def gb_all_reduce_buckets(ctx, bucket_bufs, bucket_numel, dtype, op, codec, block, stream=0):
    """bucket_bufs: flat list of n_buckets * W device pointers, bucket-major."""
    nb = len(bucket_numel)
    return lib().gb_all_reduce_buckets(ctx, nb, _ptrs(bucket_bufs), _sizes(bucket_numel), dtype, op,
                                       codec, block, stream)


def gb_all_reduce_buckets_ef(ctx, bucket_bufs, residuals, bucket_numel, dtype, op, codec, block, stream=0):
    """residuals: flat list of n_buckets * I float32 device pointers, bucket-major."""
    nb = len(bucket_numel)
    return lib().gb_all_reduce_buckets_ef(ctx, nb, _ptrs(bucket_bufs), _ptrs(residuals), _sizes(bucket_numel),
                                          dtype, op, codec, block, stream)


def gb_reduce_scatter_buckets(ctx, in_bufs, out_bufs, bucket_numel, dtype, op, codec, block, stream=0):
    """in_bufs / out_bufs: flat lists of n_buckets * W device pointers, bucket-major."""
    nb = len(bucket_numel)
    return lib().gb_reduce_scatter_buckets(ctx, nb, _ptrs(in_bufs), _ptrs(out_bufs), _sizes(bucket_numel), dtype,
                                           op, codec, block, stream)


def gb_all_gather_buckets(ctx, in_bufs, out_bufs, bucket_numel_in, dtype, stream=0):
    nb = len(bucket_numel_in)
    return lib().gb_all_gather_buckets(ctx, nb, _ptrs(in_bufs), _ptrs(out_bufs), _sizes(bucket_numel_in), dtype,
                                       stream)


def gb_set_phase_timing(ctx, capacity):
    return lib().gb_set_phase_timing(ctx, int(capacity))


def gb_phase_times(ctx, age):
    """Returns (status, [ms per phase])."""
    ms = (ctypes.c_float * GB_N_PHASES)()
    st = lib().gb_phase_times(ctx, age, ms)
    return st, list(ms)


def gb_last_phase_times(ctx):
    """Returns (status, [ms per phase])."""
    ms = (ctypes.c_float * GB_N_PHASES)()
    st = lib().gb_last_phase_times(ctx, ms)
    return st, list(ms)


def gb_debug_inject(ctx, what):
    return lib().gb_debug_inject(ctx, what)


def gb_all_reduce_noalloc(ctx, rank_bufs, n, dtype, op, codec, block, stream=0):
    return lib().gb_all_reduce_noalloc(ctx, _ptrs(rank_bufs), n, dtype, op, codec, block, stream)


def gb_kernel_launch_count():
    return lib().gb_kernel_launch_count()
