"""The benchmark's reference arm on CPU: the JSON line it prints (the oracle
timed on the host cores, W untimed and K timed decode steps), and the silent
exit of every rank but 0 under a multi-rank launch."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None, timeout=600):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_line():
    r = _run(["--impl", "reference", "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 2 and d["warmup"] == 3                  # W >= 3 enforced
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and abs(d["ms_per_step"] - 1e3 / d["value"]) < 1e-6 * d["ms_per_step"]
    assert d["config"]["workload"] == "v41_decode_T1"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["sample"].startswith("2 timed whole decode steps")
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    r = _run(["--impl", "reference", "--steps", "2", "--warmup", "3"],
             {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_q2k_alu_roofline_arithmetic():
    """The Q2_K decode's integer-pipe roofline: the counted ALU warp
    instructions over the launch's event time, against 152 SMs x 4
    sub-partitions x one warp instruction every 2 cycles at the sampled clock;
    a changed kernel (no stored count) reports null, not a stale figure."""
    sys.path.insert(0, ROOT)
    import bench
    r = {"stage_ms": {"gemv": 0.04}, "step_algorithmic_bytes": 82_851_340}
    key = ("gemv_q2k", bench._src_hash("gemv.cu", "common.cuh"))
    saved = dict(bench.NCU_ALU)
    try:
        bench.NCU_ALU.clear()
        bench.NCU_ALU[key] = 15_000_000
        o = bench.q2k_alu_roofline(r, {"sm_mhz": 2000.0}, 6794.5, 152)
        assert o["bound"] == "alu"
        assert abs(o["peak"] - 152 * 4 * 0.5 * 2000e6 / 1e12) < 1e-12           # 0.608 T/s
        assert abs(o["achieved"] - 15e6 / 40e-6 / 1e12) < 1e-12                  # 0.375 T/s
        assert abs(o["frac"] - o["achieved"] / o["peak"]) < 1e-12
        assert abs(o["hbm_frac"] - 82_851_340 / 40e-6 / 1e9 / 6794.5) < 1e-12
        bench.NCU_ALU.clear()
        o = bench.q2k_alu_roofline(r, None, 6794.5, 152)
        assert o["achieved"] is None and o["frac"] is None and o["instructions"] is None
        assert abs(o["peak"] - 152 * 4 * 0.5 * 2070e6 / 1e12) < 1e-12           # default clock
    finally:
        bench.NCU_ALU.clear()
        bench.NCU_ALU.update(saved)
