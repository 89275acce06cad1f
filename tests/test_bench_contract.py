"""The benchmark's reference arm (the float64 CPU oracle) prints the JSON line the driver
reads; it needs no GPU, so its contract is checked here."""
import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "cpu_baseline", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1
    assert d["warmup"] >= 3  # the bench raises warm-up to at least 3 steps
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == d["value"] and cpu["cores"] >= 1 and cpu["sample"]
    assert "workload" in d["config"]
    # the reference arm times the oracle alone: neither it nor its oracle child maps the CUDA library
    assert d["product_library_mapped"] == {"arm": False, "oracle_child": False}


def test_host_only_package_users_do_not_map_the_library():
    """Importing the package and its seeded input generators maps no CUDA library (the binding
    maps it on the first call into it)."""
    code = ("import adapter_gemm_segment_gb300 as a, adapter_gemm_segment_gb300.workloads as w; "
            "w.decode_q_proj(seed=1, n=4, layer=0); import bench; print(bench.product_library_mapped())")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip().splitlines()[-1] == "False"
