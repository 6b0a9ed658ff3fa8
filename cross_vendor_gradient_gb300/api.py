"""Tensor-level interface over libgb.

torch supplies device memory and the current CUDA stream; every computation
runs in libgb's kernels (there is no CPU or PyTorch fallback).  Each method
marshals tensors to pointers, calls the C entry point of the same name on the
current stream and raises ``GbError`` on a non-OK status.
"""
import torch

from . import binding as B

_DTYPES = {torch.float32: B.GB_F32, torch.bfloat16: B.GB_BF16, torch.float16: B.GB_F16,
           torch.float64: B.GB_F64, torch.int8: B.GB_I8, torch.uint8: B.GB_U8, torch.int32: B.GB_I32,
           torch.int64: B.GB_I64}
CODECS = {"none": B.GB_CODEC_NONE, "bf16": B.GB_CODEC_BF16, "e4m3": B.GB_CODEC_E4M3,
          "e5m2": B.GB_CODEC_E5M2}
OPS = {"sum": B.GB_SUM, "avg": B.GB_AVG, "max": B.GB_MAX, "min": B.GB_MIN}


class GbError(RuntimeError):
    def __init__(self, status, message=""):
        self.status = status
        super().__init__("%s%s" % (B.gb_status_string(status), (": " + message) if message else ""))


def _codec(c):
    return CODECS[c] if isinstance(c, str) else int(c)


def _op(o):
    return OPS[o] if isinstance(o, str) else int(o)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype(tensors):
    dt = tensors[0].dtype
    if dt not in _DTYPES:
        raise GbError(B.GB_ERR_UNSUPPORTED_DTYPE, str(dt))
    for t in tensors:
        if t.dtype != dt or not t.is_contiguous() or t.device != tensors[0].device:
            raise GbError(B.GB_ERR_INVALID_ARG, "tensors must share dtype and device and be contiguous")
    return _DTYPES[dt]


def _row_pitch(tensors):
    """The byte distance between consecutive tensors when all of them lie in
    one storage (one host allocation) at equal, ascending spacing of at
    least one tensor's bytes; else None."""
    if len(tensors) < 2:
        return None
    base = tensors[0].untyped_storage().data_ptr()
    if any(t.untyped_storage().data_ptr() != base for t in tensors[1:]):
        return None
    nb = tensors[0].numel() * tensors[0].element_size()
    pitch = tensors[1].data_ptr() - tensors[0].data_ptr()
    if pitch < nb or any(t.data_ptr() != tensors[0].data_ptr() + r * pitch for r, t in enumerate(tensors)):
        return None
    return pitch


def payload_bytes(codec, block, n):
    return B.gb_payload_bytes(_codec(codec), block, n)


def island_payload_bytes(dtype, op, codec, block, n):
    """Bytes of one island's payload for any dtype and op (the exact path's
    fold, or the codec's payload)."""
    dt = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return B.gb_island_payload_bytes(dt, _op(op), _codec(codec), block, n)


def payload_scales_offset(codec, block, n):
    return B.gb_payload_scales_offset(_codec(codec), block, n)


def bucket_plan(numels, elem_bytes, cap_bytes=25 * 1024 * 1024, pad_elems=1):
    st, bo, off, bn = B.gb_bucket_plan(list(numels), elem_bytes, cap_bytes, pad_elems)
    if st != B.GB_OK:
        raise GbError(st, "bucket plan")
    return bo, off, bn


def kernel_launch_count():
    return B.gb_kernel_launch_count()


class Context:
    """W simulated ranks in contiguous islands on the current CUDA device."""

    def __init__(self, island_sizes):
        st, h = B.gb_create(list(island_sizes))
        if st != B.GB_OK:
            raise GbError(st, "gb_create(%s)" % (list(island_sizes),))
        self.handle = h
        self.island_sizes = tuple(int(v) for v in island_sizes)
        self.world_size = B.gb_world_size(h)

    def close(self):
        if self.handle:
            B.gb_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def _check(self, st):
        if st != B.GB_OK:
            raise GbError(st, B.gb_last_error_message(self.handle))

    # ------------------------------------------------------------ topology
    def island_first_rank(self, i):
        return B.gb_island_first_rank(self.handle, i)

    def island_of_rank(self, r):
        return B.gb_island_of_rank(self.handle, r)

    def status(self):
        return B.gb_context_status(self.handle)

    def set_pipeline(self, chunk_bytes, use_graphs=True):
        """chunk_bytes > 0: pipelined bridge in chunks of about that many bytes
        of one island's payload (default 2 MiB); 0: one bridge hop per call."""
        self._check(B.gb_set_pipeline(self.handle, chunk_bytes, use_graphs))

    def set_sharded_bridge(self, on=True):
        """Sharded-bridge policy for all_reduce: k = smallest island size
        segments, each over its own bridge link (same bits)."""
        self._check(B.gb_set_sharded_bridge(self.handle, on))

    def reserve(self, n, dtype=torch.float32, codec="none", block=256):
        self._check(B.gb_reserve(self.handle, n, _DTYPES[dtype], _codec(codec), block))

    # ---------------------------------------------------------- collectives
    def all_reduce(self, tensors, op="sum", codec="none", block=256, stream=None):
        dt = _dtype(tensors)
        self._check(B.gb_all_reduce(self.handle, [t.data_ptr() for t in tensors], tensors[0].numel(), dt,
                                    _op(op), _codec(codec), block, _stream(stream)))

    def all_reduce_ef(self, tensors, residuals, op="sum", codec="none", block=256, stream=None):
        """all_reduce with error feedback; residuals: one float32 tensor of the
        buffers' size per island, zero before the first step, kept across steps."""
        dt = _dtype(tensors)
        for r in residuals:
            if r.dtype != torch.float32 or not r.is_contiguous() or r.numel() != tensors[0].numel():
                raise GbError(B.GB_ERR_INVALID_ARG, "residuals: contiguous float32 of the buffers' size")
        self._check(B.gb_all_reduce_ef(self.handle, [t.data_ptr() for t in tensors], [r.data_ptr() for r in residuals],
                                       tensors[0].numel(), dt, _op(op), _codec(codec), block, _stream(stream)))

    def reduce_scatter(self, inputs, outputs, op="sum", codec="none", block=256, stream=None):
        dt = _dtype(list(inputs) + list(outputs))
        self._check(B.gb_reduce_scatter(self.handle, [t.data_ptr() for t in inputs],
                                        [t.data_ptr() for t in outputs], inputs[0].numel(), dt, _op(op),
                                        _codec(codec), block, _stream(stream)))

    def all_gather(self, inputs, outputs, stream=None):
        dt = _dtype(list(inputs) + list(outputs))
        self._check(B.gb_all_gather(self.handle, [t.data_ptr() for t in inputs],
                                    [t.data_ptr() for t in outputs], inputs[0].numel(), dt,
                                    _stream(stream)))

    def broadcast(self, tensors, src, stream=None):
        dt = _dtype(tensors)
        self._check(B.gb_broadcast(self.handle, [t.data_ptr() for t in tensors], tensors[0].numel(), dt,
                                   src, _stream(stream)))

    def all_reduce_host(self, host_tensors, op="sum", codec="none", block=256, stream=None):
        """host_tensors: W host tensors (pinned for asynchronous copies), or
        one [W, n] host tensor whose rows are the ranks.  Rows of one
        storage at equal, ascending spacing go through
        gb_all_reduce_host_rows (2D staging copies); anything else through
        gb_all_reduce_host."""
        if isinstance(host_tensors, torch.Tensor):
            if host_tensors.dim() != 2:
                raise GbError(B.GB_ERR_INVALID_ARG, "a host tensor of ranks must be [W, n]")
            host_tensors = list(host_tensors.unbind(0))
        if any(t.device.type != "cpu" for t in host_tensors):
            raise GbError(B.GB_ERR_INVALID_ARG, "all_reduce_host takes host (CPU) tensors; use all_reduce for CUDA tensors")
        dt = _dtype(host_tensors)
        n = host_tensors[0].numel()
        pitch = _row_pitch(host_tensors)
        if pitch is not None:
            self._check(B.gb_all_reduce_host_rows(self.handle, host_tensors[0].data_ptr(), pitch, n, dt, _op(op),
                                                  _codec(codec), block, _stream(stream)))
            return
        self._check(B.gb_all_reduce_host(self.handle, [t.data_ptr() for t in host_tensors], n, dt, _op(op),
                                         _codec(codec), block, _stream(stream)))

    def all_reduce_buckets(self, buckets, op="sum", codec="none", block=256, stream=None):
        """buckets: list of per-bucket lists of W flat tensors."""
        flat = [t for b in buckets for t in b]
        dt = _dtype(flat)
        self._check(B.gb_all_reduce_buckets(self.handle, [t.data_ptr() for t in flat],
                                            [b[0].numel() for b in buckets], dt, _op(op), _codec(codec),
                                            block, _stream(stream)))

    def all_reduce_buckets_ef(self, buckets, residuals, op="sum", codec="none", block=256, stream=None):
        """buckets[b]: W flat tensors; residuals[b]: I float32 tensors of the
        bucket's length (zero at the start, kept across steps)."""
        flat = [t for b in buckets for t in b]
        res = [r for b in residuals for r in b]
        for r in res:
            if r.dtype != torch.float32 or not r.is_contiguous():
                raise GbError(B.GB_ERR_INVALID_ARG, "residuals must be contiguous float32 tensors")
        dt = _dtype(flat)
        self._check(B.gb_all_reduce_buckets_ef(self.handle, [t.data_ptr() for t in flat], [r.data_ptr() for r in res],
                                               [b[0].numel() for b in buckets], dt, _op(op), _codec(codec), block,
                                               _stream(stream)))

    def reduce_scatter_buckets(self, in_buckets, out_buckets, op="sum", codec="none", block=256, stream=None):
        """in_buckets[b]: W flat tensors of bucket b; out_buckets[b]: W
        tensors of numel / W elements."""
        ins = [t for b in in_buckets for t in b]
        outs = [t for b in out_buckets for t in b]
        dt = _dtype(ins)
        self._check(B.gb_reduce_scatter_buckets(self.handle, [t.data_ptr() for t in ins],
                                                [t.data_ptr() for t in outs], [b[0].numel() for b in in_buckets],
                                                dt, _op(op), _codec(codec), block, _stream(stream)))

    def all_gather_buckets(self, in_buckets, out_buckets, stream=None):
        """in_buckets[b]: W tensors of m_b elements; out_buckets[b]: W
        tensors of W * m_b elements."""
        ins = [t for b in in_buckets for t in b]
        outs = [t for b in out_buckets for t in b]
        dt = _dtype(ins)
        self._check(B.gb_all_gather_buckets(self.handle, [t.data_ptr() for t in ins], [t.data_ptr() for t in outs],
                                            [b[0].numel() for b in in_buckets], dt, _stream(stream)))

    # ------------------------------------------------------- phase blocks
    def island_reduce(self, island, tensors, island_sum, stream=None):
        dt = _dtype(tensors)
        self._check(B.gb_island_reduce(self.handle, island, [t.data_ptr() for t in tensors],
                                       tensors[0].numel(), dt, island_sum.data_ptr(), _stream(stream)))

    def bridge_compress(self, island_sum, codec, block, payload, stream=None):
        self._check(B.gb_bridge_compress(self.handle, island_sum.data_ptr(), island_sum.numel(),
                                         _codec(codec), block, payload.data_ptr(), _stream(stream)))

    def bridge_decompress_accumulate(self, payload, n, codec, block, accum, accumulate, stream=None):
        self._check(B.gb_bridge_decompress_accumulate(self.handle, payload.data_ptr(), n, _codec(codec),
                                                      block, accum.data_ptr(), accumulate,
                                                      _stream(stream)))

    def island_broadcast(self, island, total, op, tensors, stream=None):
        dt = _dtype(tensors)
        self._check(B.gb_island_broadcast(self.handle, island, total.data_ptr(), total.numel(), _op(op),
                                          [t.data_ptr() for t in tensors], dt, _stream(stream)))

    def island_reduce_compress(self, tensors, codec, block, payloads, stream=None):
        """Fused island reduce + encode of every island: payloads[i] (uint8
        device tensors of payload_bytes(codec, block, n) bytes) receive the
        encoded island sums."""
        dt = _dtype(tensors)
        self._check(B.gb_island_reduce_compress(self.handle, [t.data_ptr() for t in tensors],
                                                tensors[0].numel(), dt, _codec(codec), block,
                                                [p.data_ptr() for p in payloads], _stream(stream)))

    def island_reduce_compress_ef(self, tensors, residuals, codec, block, payloads, stream=None):
        """island_reduce_compress with error feedback: residuals are I
        float32 tensors of n elements (updated in place)."""
        dt = _dtype(tensors)
        self._check(B.gb_island_reduce_compress_ef(self.handle, [t.data_ptr() for t in tensors],
                                                   [r.data_ptr() for r in residuals], tensors[0].numel(), dt,
                                                   _codec(codec), block, [p.data_ptr() for p in payloads],
                                                   _stream(stream)))

    def decompress_island_broadcast(self, payloads, op, codec, block, tensors, stream=None):
        """Fused decode of every island's payload + accumulate + broadcast
        into all rank tensors.  payloads: I tensors (every leader holds the
        same ones) or I * I (row g: what leader g holds, island order)."""
        dt = _dtype(tensors)
        I = len(self.island_sizes)
        if len(payloads) == I and I > 1:  # one shared set: every leader's row
            payloads = [p for _ in range(I) for p in payloads]
        self._check(B.gb_decompress_island_broadcast(self.handle, [p.data_ptr() for p in payloads],
                                                     tensors[0].numel(), dt, _op(op), _codec(codec), block,
                                                     [t.data_ptr() for t in tensors], _stream(stream)))

    def island_reduce_compress_op(self, tensors, op, codec, block, payloads, stream=None):
        """The first fused half for every dtype and op: the codec path's
        encode, or the exact path's island fold (payloads of
        island_payload_bytes bytes)."""
        dt = _dtype(tensors)
        self._check(B.gb_island_reduce_compress_op(self.handle, [t.data_ptr() for t in tensors],
                                                   tensors[0].numel(), dt, _op(op), _codec(codec), block,
                                                   [p.data_ptr() for p in payloads], _stream(stream)))

    def decompress_scatter(self, payloads, n, op, codec, block, outputs, stream=None):
        """reduce_scatter's second half: outputs[r] (n / W elements) receives
        slice r of the decoded total.  payloads: I tensors (every leader holds
        the same ones) or I * I."""
        dt = _dtype(outputs)
        I = len(self.island_sizes)
        if len(payloads) == I and I > 1:
            payloads = [p for _ in range(I) for p in payloads]
        self._check(B.gb_decompress_scatter(self.handle, [p.data_ptr() for p in payloads], n, dt, _op(op),
                                            _codec(codec), block, [t.data_ptr() for t in outputs],
                                            _stream(stream)))

    # -------------------------------------------------------------- timing
    def set_phase_timing(self, capacity):
        """capacity > 0: keep the phase marks of the last `capacity` calls."""
        self._check(B.gb_set_phase_timing(self.handle, int(capacity)))

    def phase_times(self, age):
        st, ms = B.gb_phase_times(self.handle, age)
        self._check(st)
        return ms

    def last_phase_times(self):
        st, ms = B.gb_last_phase_times(self.handle)
        self._check(st)
        return ms

    def debug_inject(self, what):
        self._check(B.gb_debug_inject(self.handle, what))
