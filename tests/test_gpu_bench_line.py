"""The benchmark's JSON line on the GPU: one line with the contract's keys,
the dominant kernel's roofline (measured kernel time, ncu traffic for this
source or null), the end-to-end figure from host buffers, the launch count
and the sampled clocks; the Q2_K-weight decode reported against its integer
pipe."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_contract():
    d = _line(["--gpus", "1", "--steps", "5", "--warmup", "3", "--no-cpu-baseline", "--no-others",
               "--prefill-steps", "2"])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks",
                "prefill"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert abs(d["value"] - 1e3 / d["ms_per_step"]) <= 1e-6 * d["value"]     # one token a step
    assert d["config"]["workload"].startswith("v41_decode_T1")
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and rf["peak"] > 0
    assert 0.3 < rf["frac"] < 1.4 and abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["traffic"] is None or rf["traffic"] >= rf["algorithmic_bytes"]
    e = d["e2e"]
    assert e["unit"] == "tokens/s" and e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= 2 * d["steps"]                               # projection + gate a step
    assert d["clocks"]["sm_max_mhz"] > 0
    p = d["prefill"]
    assert p["roofline"]["bound"] == "tensor" and 0.3 < p["roofline"]["frac"] < 1.4


def test_bench_q2k_weight_decode_reports_integer_pipe():
    d = _line(["--only", "wkvq2k", "--steps", "20", "--warmup", "3", "--no-cpu-baseline"])
    rf = d["roofline"]
    assert rf["bound"] == "alu" and rf["peak"] > 0 and rf["kernel_ms"] > 0
    assert rf["frac"] is None or 0.1 < rf["frac"] < 1.05
    assert 0.0 < rf["hbm_frac"] < 1.0
