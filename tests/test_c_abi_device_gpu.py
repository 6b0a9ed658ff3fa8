"""The C ABI from a plain C99 program on the GPU: tests/c_abi_device.c builds
against include/gb.h and the CUDA runtime's C API alone, all_reduces and
reduce_scatters four rank buffers, and its results match the oracle bit for
bit."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle as orc
from cross_vendor_gradient_gb300 import binding as B
from tests.gpu_util import assert_bits_equal

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N, NRS = 70003, 70004


def values(r, n, salt):
    j = np.arange(n, dtype=np.int64)
    return (((j * 7 + r * 13 + salt) % 101) - 50).astype(np.float32) * np.float32(0.25)


def test_c_program_all_reduce_and_reduce_scatter(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gcc = shutil.which("gcc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if gcc is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime_api.h")):
        pytest.skip("no gcc or CUDA headers")
    exe = str(tmp_path / "c_abi_device")
    libdir = os.path.dirname(B.LIB_PATH)
    cudalib = os.path.join(cuda, "lib64")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-isystem", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c_abi_device.c"),
                    "-L", libdir, "-lgb", "-L", cudalib, "-lcudart", "-Wl,-rpath," + libdir,
                    "-Wl,-rpath," + cudalib, "-o", exe], check=True)
    out = str(tmp_path / "out.bin")
    run = subprocess.run([exe, out], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr
    got = np.fromfile(out, dtype=np.float32)
    assert got.size == 4 * N + NRS
    xs = [values(r, N, 0) for r in range(4)]
    want = orc.all_reduce(xs, (2, 2), "avg", "e4m3", 256)
    for r in range(4):
        assert_bits_equal(got[r * N:(r + 1) * N], want[r], "all_reduce rank %d" % r)
    xs = [values(r, NRS, 5) for r in range(4)]
    want = orc.reduce_scatter(xs, (2, 2), "sum", "bf16", 256)
    m = NRS // 4
    for r in range(4):
        assert_bits_equal(got[4 * N + r * m:4 * N + (r + 1) * m], want[r], "reduce_scatter rank %d" % r)
