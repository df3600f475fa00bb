"""bench.py's reference arm (the CPU oracle) on the CPU: one JSON line with the
fields of the benchmark contract, and nothing printed by ranks other than 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(extra_env, *args):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", **extra_env)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _bench({}, "--steps", "1", "--warmup", "0")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key, typ in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                     ("dtype", str), ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)):
        assert isinstance(d[key], typ), key
    assert d["value"] > 0 and d["steps"] == 1 and d["n_gpus"] == 1 and d["vs_baseline"] is None
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["data"] == "synthetic"
    assert isinstance(d["config"]["workload"], str) and d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert isinstance(cb["cores"], int) and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    r = _bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--steps", "1", "--warmup", "0")
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_measured_peaks_record_is_read_flat_or_nested():
    sys.path.insert(0, ROOT)
    from bench import parse_peaks
    want = (7100.0, 2050.0, 1740.0)
    flat = {"hbm_gbs": 7100, "bf16_tflops": 2050, "bf16_tflops_sustained": 1740, "sm_clock_mhz": 2070}
    nested = {"gpu": "GB300", "hbm_gbs": {"value": 7100, "pct_of_nominal": 90},
              "bf16_tflops": {"value": 2050}, "bf16_tflops_sustained": {"value": 1740, "clock_mhz": 1900}}
    units = {"hbm_tbs": 7.1, "bf16_pflops": 2.05, "bf16_pflops_sustained": 1.74}
    for rec in (flat, nested, units):
        assert parse_peaks(rec) == want, rec
    assert parse_peaks({"hbm_gbs": 7100, "bf16_tflops": 2050}) == (7100.0, 2050.0, 2050.0)
    assert parse_peaks({"note": "no measurement"}) is None
