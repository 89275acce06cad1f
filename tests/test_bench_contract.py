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


def test_concat_metrics_by_hand():
    """The tensor-concatenation figures of the benchmark line on a hand-worked batch:
    idx = [-1, 0, 0, 2] over 3 slots of ranks 8, 16, 4 padded to r_max 16, h_in 10, h_out 6."""
    m = bench.concat_metrics([-1, 0, 0, 2], 10, 6, [8, 16, 4], 16, 3)
    assert m["n_segments"] == 3 and m["distinct_adapters"] == 2  # runs -1, 0, 2
    assert m["concat_elements"] == 3 * 16 * (10 + 6) == 768
    assert m["concat_projection"] == [4, 48] and m["concat_projection_elements"] == 192
    # tokens 0, 0, 2 at r_max 16 multiply 8 + 8 + 12 padded rows out of 48
    assert abs(m["zero_pad_flop_share"] - 28 / 48) < 1e-15
    # touched adapters 0 and 2 store 8 + 12 padded rows out of 32
    assert abs(m["zero_pad_stored_share"] - 20 / 32) < 1e-15
    # concatenated LoRA FLOPs 2*4*48*16 = 6144, of which the 3 LoRA tokens' own blocks 2*3*16*16 = 1536
    assert abs(m["concat_lora_flops_wasted_share"] - 0.75) < 1e-15
    empty = bench.concat_metrics([-1, -1], 10, 6, [8], 8, 1)
    assert empty["n_segments"] == 1 and empty["zero_pad_flop_share"] == 0.0
    assert empty["concat_lora_flops_wasted_share"] == 1.0
