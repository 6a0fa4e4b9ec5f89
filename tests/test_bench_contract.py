"""bench.py's output line on the GPU: the keys and types every run must carry
(the measured value, the roofline of the dominant kernel, the CPU baseline,
the end-to-end figure, the launch count and the clock record), for our arm
and for the reference arm, on the small 4-rank workload."""
import json
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu

ROOT = Path(__file__).resolve().parent.parent


def _line(*args):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    proc = subprocess.run([sys.executable, "bench.py", "--workload", "qgz_tiny", "--steps", "5",
                           "--warmup", "3", *args], cwd=ROOT, capture_output=True, text=True,
                          timeout=600)
    assert proc.returncode == 0, proc.stderr[-3000:]
    lines = [l for l in proc.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, proc.stdout[-2000:]
    return json.loads(lines[0])


def _has(d, keys, types=(int, float)):
    for k in keys:
        assert k in d, k
        assert d[k] is None or isinstance(d[k], types), (k, d[k])


def test_our_line_carries_the_contract():
    d = _line()
    _has(d, ["value", "ms_per_step"])
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert isinstance(d["metric"], str) and isinstance(d["unit"], str)
    assert d["dtype"] == "f32" and d["data"].startswith("synthetic")
    assert "workload" in d["config"] and "l2" in d["config"]
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    _has(r, ["achieved", "peak", "frac", "traffic"])
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] == 1 and c["value"] > 0 and c["sample"]
    assert c["all_cores"]["cores"] >= 1
    assert d["parity"]["verdict"] == "bit-exact"
    e = d["e2e"]
    _has(e, ["value", "h2d_bytes_per_step", "d2h_bytes_per_step"])
    assert e["h2d_bytes_per_step"] == 4 * 1048576 * 2 and e["d2h_bytes_per_step"] == 1048576 * 4
    assert d["gpu_launches"] == 5 * 2
    k = d["clocks"]
    assert k is None or ("sm_mhz" in k and "sm_max_mhz" in k and isinstance(k["reasons"], list))
    for name, kern in d["kernels"].items():
        _has(kern, ["ms", "GB/s", "frac"])
        assert set(kern["ms_percentiles"]) == {"median", "p10", "p90"}


def test_reference_line_carries_the_contract():
    d = _line("--impl", "reference")
    assert d["impl"] == "reference"
    _has(d, ["value", "ms_per_step"])
    assert d["value"] > 0 and d["unit"] == "elements/s" and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
