"""bench.py's reference arm (the oracle on the host cores) prints the contract's JSON line on the
CPU; the GB300 arm's L2 labelling follows the workload's resident input bytes."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny_bf16", "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    for key in ("metric", "value", "unit", "ms_per_step", "higher_is_better", "scaling", "vs_baseline", "dtype",
                "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_bf16"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_l2_policy_follows_the_resident_bytes():
    import bench
    from workloads import WORKLOADS
    for name in ("mixtral_bf16_prefill", "dsv3_fp8fp4_decode", "dsv3_fp8fp4_prefill_zipf", "int8_a8w8", "int4_a8w4"):
        assert bench.workload_config(WORKLOADS[name])["l2_policy"] == "inputs larger than L2 (no flush)", name
    assert "fit in L2" in bench.workload_config(WORKLOADS["tiny_bf16"])["l2_policy"]
