"""bench.py's output contract on the GPU: one JSON line with the metric, the
device-timed value, the roofline of the dominant kernel, the end-to-end
figure through host buffers, the oracle baseline, the kernel count and the
clocks, all self-consistent."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_default_line_contract():
    d = run_bench("--steps", "20", "--warmup", "3")
    assert d["metric"] == "all_reduce algorithm GB/s and % of GB300 HBM roofline vs payload size, per codec"
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3 and d["scaling"] == "weak"
    assert d["vs_baseline"] is None and d["dtype"] == "f32" and "synthetic" in d["data"]
    assert d["config"]["workload"].startswith("c2") and "flushed" in d["config"]["l2"]
    # value = bytes of one rank buffer per step / step time
    n = d["config"]["n"]
    assert abs(d["value"] - n * 4 / (d["ms_per_step"] * 1e-3) / 1e9) < 1e-6 * d["value"]
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["kernel"] in ("k_decode_bcast", "k_reduce_encode")
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    assert abs(r["achieved"] - r["alg_bytes_per_launch"] / (r["avg_launch_ms"] * 1e-3) / 1e9) < 1e-6 * r["achieved"]
    assert 0.3 < r["frac"] < 1.3  # a copy-peak denominator: a little above 1.0 is possible, far above is not
    assert r["traffic"] is None or r["traffic"] > 0
    e = d["e2e"]
    assert e["unit"] == "GB/s" and e["h2d_bytes_per_step"] == 4 * n * 4 and e["d2h_bytes_per_step"] == 4 * n * 4
    assert 0 < e["value"] < d["value"]  # the host link bounds it below the device-resident step
    assert "rows" in e["api"] and e["separate_buffers"]["ms_per_step"] > 0  # both host layouts timed
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    assert d["gpu_launches"] == 20 * 8  # 4 chunks x (encode + decode) per graph-replayed step
    c = d["clocks"]
    assert c["sm_mhz"] > 0 and isinstance(c["reasons"], list)
    k = d["kernels_ms"]  # one-hop steps with and without the phase marks' events
    assert k["step_ms_with_marks"] > 0 and k["step_ms_without_marks"] > 0
    # the metric's curve: 17 payload sizes x 3 codecs of the c3 sweep
    sw = d["sweep"]
    cols = sw["columns"]
    assert cols[:5] == ["bytes_per_rank", "codec", "steps", "ms_per_step", "algbw_gbs"]
    rows = [dict(zip(cols, row)) for row in sw["rows"]]
    assert len(rows) == 51
    assert sorted({r["bytes_per_rank"] for r in rows}) == [4096 << k for k in range(17)]
    for size in {r["bytes_per_rank"] for r in rows}:
        assert sorted(r["codec"] for r in rows if r["bytes_per_rank"] == size) == ["bf16", "e4m3", "none"]
    for r in rows:
        assert r["ms_per_step"] > 0 and r["steps"] >= 5
        assert abs(r["algbw_gbs"] - r["bytes_per_rank"] / (r["ms_per_step"] * 1e-3) / 1e9) < 1e-3 * r["algbw_gbs"]
        assert 0 < r["encode_frac"] < 1.3 and 0 < r["decode_frac"] < 1.3
        assert 0 < r["bridge_frac"] < 1.3
        assert (r["floor_ms"] is not None) == (r["bytes_per_rank"] <= 1 << 20)


def test_reference_arm_contract():
    d = run_bench("--impl", "reference", "--steps", "3", "--warmup", "3")
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
