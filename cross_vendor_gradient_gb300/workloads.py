"""Seeded synthetic workloads: rank counts, island layouts, gradient shapes and
value distributions.

This module holds no arithmetic of the collectives (no sums, no codecs, no
bucket planning): it only describes the workloads and draws their inputs, so
that the CUDA path and the oracle can be fed the same bytes.

Seeds: rank r of workload c draws from ``numpy.random.PCG64(1000 * c + r)``
(host: the small workloads and the oracle-checked sizes) or from a
``torch.Generator`` seeded the same way on the target device (the payload
sweep, and large buffers, generated where they are used); bucket b of a
bucketed workload draws on the device with seed bucket_seed(c, b, r).
"""
from dataclasses import dataclass, field

import numpy as np

MiB = 1024 * 1024
BUCKET_CAP_BYTES = 25 * MiB  # torch DDP's default bucket cap


@dataclass(frozen=True)
class Workload:
    key: str                 # short name
    cid: int                 # seed base: rank r uses seed 1000 * cid + r
    island_sizes: tuple      # contiguous islands of simulated ranks
    dtype: str               # rank-buffer element type: f32 bf16 f16 f64 i8 u8 i32 i64
    dist: str                # value distribution, see draw_host / draw_device
    op: str                  # "sum", "avg", "max" or "min"
    codecs: tuple            # bridge codecs exercised
    block: int = 256         # fp8 scale block
    n: int = 0               # elements per rank buffer (single-buffer workloads)
    tensors: tuple = field(default=())  # gradient tensor shapes (bucketed workloads)

    @property
    def world_size(self) -> int:
        return sum(self.island_sizes)

    @property
    def elem_bytes(self) -> int:
        return {"f32": 4, "bf16": 2, "f16": 2, "f64": 8, "i8": 1, "u8": 1, "i32": 4, "i64": 8}[self.dtype]


def gpt2_small_shapes():
    """Per-tensor gradient shapes of GPT-2 small (12 layers, d = 768,
    vocabulary 50257, 1024 positions): 148 tensors, 124,439,808 values."""
    d, v, ctx, ff = 768, 50257, 1024, 3072
    shapes = [(v, d), (ctx, d)]
    for _ in range(12):
        shapes += [(d,), (d,), (d, 3 * d), (3 * d,), (d, d), (d,), (d,), (d,), (d, ff), (ff,),
                   (ff, d), (d,)]
    shapes += [(d,), (d,)]
    return tuple(shapes)


def llama_1b_shapes():
    """Per-tensor gradient shapes of a 1.1B Llama-style model (22 layers,
    d = 2048, ffn 5632, vocabulary 32000, 4 key/value heads of 64 = 256):
    201 tensors, 1,100,048,384 values."""
    d, v, ff, kv = 2048, 32000, 5632, 256
    shapes = [(v, d)]
    for _ in range(22):
        shapes += [(d,), (d, d), (kv, d), (kv, d), (d, d), (d,), (ff, d), (ff, d), (d, ff)]
    shapes += [(d,), (v, d)]
    return tuple(shapes)


def numel(shape) -> int:
    out = 1
    for s in shape:
        out *= int(s)
    return out


WORKLOADS = {
    # 2 ranks, one per island, one 4 MiB float32 buffer each
    "c1": Workload("c1", 1, (1, 1), "f32", "normal_1e-2", "sum", ("none", "bf16"), n=1 << 20),
    # 4 ranks as 2 islands of 2, one 25 MiB float32 DDP bucket each, 1% outliers x100
    "c2": Workload("c2", 2, (2, 2), "f32", "normal_1e-3_outliers", "avg", ("e4m3",), block=256,
                   n=BUCKET_CAP_BYTES // 4),
    # payload sweep: 4 KiB .. 256 MiB of float32 per rank (n = 2^10 .. 2^26)
    "c3": Workload("c3", 3, (2, 2), "f32", "uniform_pm1", "sum", ("none", "bf16", "e4m3"),
                   block=256),
    # 8 ranks as 2 islands of 4, GPT-2-small-shaped bf16 gradients in 25 MiB buckets
    "c4": Workload("c4", 4, (4, 4), "bf16", "student_t3_1e-3", "sum", ("bf16",),
                   tensors=gpt2_small_shapes()),
    # 8 ranks as 2 islands of 4, 1.1B Llama-shaped bf16 gradients, 0.1% zero blocks of 128
    "c5": Workload("c5", 5, (4, 4), "bf16", "normal_1e-3_zero_blocks", "sum", ("e5m2",), block=128,
                   tensors=llama_1b_shapes()),
}

SWEEP_LOG2 = tuple(range(10, 27))  # 2^10 .. 2^26 float32 elements per rank


def seed_of(cid: int, rank: int) -> int:
    return 1000 * cid + rank


def bucket_seed(cid: int, bucket: int, rank: int) -> int:
    """Seed of rank `rank`'s buffer of bucket `bucket` in a bucketed workload
    (the benchmark and the tests draw the same buckets)."""
    return 1_000_000 * cid + 1000 * bucket + rank


# ---------------------------------------------------------------- host side

def draw_host(dist: str, n: int, seed: int) -> np.ndarray:
    """float32 values of the named distribution, n of them, from PCG64(seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if dist == "normal_1e-2":
        x = rng.normal(0.0, 1e-2, n)
    elif dist == "normal_1e-3_outliers":
        x = rng.normal(0.0, 1e-3, n)
        k = n // 100  # exactly 1% of the elements, distinct indices
        idx = rng.permutation(n)[:k]
        x[idx] *= 100.0
    elif dist == "uniform_pm1":
        x = rng.uniform(-1.0, 1.0, n)
    elif dist == "student_t3_1e-3":
        x = rng.standard_t(3, n) * 1e-3
    elif dist == "normal_1e-3_zero_blocks":
        x = rng.normal(0.0, 1e-3, n)
        nblk = n // 128
        k = nblk // 1000  # 0.1% of the whole 128-element blocks
        if k:
            for b in rng.choice(nblk, size=k, replace=False):
                x[b * 128:(b + 1) * 128] = 0.0
    elif dist == "integers":
        x = rng.integers(-1000, 1001, n).astype(np.float64)
    else:
        raise ValueError("unknown distribution %r" % dist)
    return x.astype(np.float32)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 inputs to bf16 patterns (input preparation only), via
    torch's CPU conversion."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def host_rank_inputs(w: Workload, n: int = None, dist: str = None, cid: int = None):
    """W rank buffers as numpy arrays: float32, or uint16 bf16 patterns."""
    n = w.n if n is None else n
    dist = w.dist if dist is None else dist
    cid = w.cid if cid is None else cid
    out = []
    for r in range(w.world_size):
        x = draw_host(dist, n, seed_of(cid, r))
        out.append(x if w.dtype == "f32" else to_bf16_bits(x))
    return out


# -------------------------------------------------------------- device side

def draw_device(dist: str, n: int, seed: int, device, dtype):
    """A torch tensor of n values of the named distribution generated on
    `device` by a torch.Generator seeded with `seed`, cast to `dtype`."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    f32 = torch.float32
    if dist == "normal_1e-2":
        x = torch.randn(n, generator=g, device=device, dtype=f32) * 1e-2
    elif dist == "normal_1e-3_outliers":
        x = torch.randn(n, generator=g, device=device, dtype=f32) * 1e-3
        idx = torch.randperm(n, generator=g, device=device)[: n // 100]
        x[idx] *= 100.0
    elif dist == "uniform_pm1":
        x = torch.rand(n, generator=g, device=device, dtype=f32) * 2.0 - 1.0
    elif dist == "student_t3_1e-3":
        z = torch.randn(n, generator=g, device=device, dtype=f32)
        chi2 = torch.zeros(n, device=device, dtype=f32)
        for _ in range(3):
            chi2 += torch.randn(n, generator=g, device=device, dtype=f32) ** 2
        x = z / torch.sqrt(chi2 / 3.0) * 1e-3
    elif dist == "normal_1e-3_zero_blocks":
        x = torch.randn(n, generator=g, device=device, dtype=f32) * 1e-3
        nblk = n // 128
        k = nblk // 1000
        if k:
            blocks = torch.randperm(nblk, generator=g, device=device)[:k]
            x[: nblk * 128].view(nblk, 128)[blocks] = 0.0
    else:
        raise ValueError("unknown distribution %r" % dist)
    return x.to(dtype)


DTYPE_NAMES = ("f32", "bf16", "f16", "f64", "i8", "u8", "i32", "i64")


def as_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    """Input preparation only: float32 draws as another rank dtype
    (bf16 patterns via torch's cast; integers: x * 1000 rounded and clipped
    to the type's range)."""
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return to_bf16_bits(x)
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "f64":
        return x.astype(np.float64)
    npdt = {"i8": np.int8, "u8": np.uint8, "i32": np.int32, "i64": np.int64}[dtype]
    info = np.iinfo(npdt)
    return np.clip(np.round(x.astype(np.float64) * 1000.0), info.min, info.max).astype(npdt)
