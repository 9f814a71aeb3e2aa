"""The benchmark's JSON line on the GPU (small fp32 workload): every key of the
contract, with the roofline, end-to-end, launch-count and clock objects."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bench_json_line_keys():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--workload", "tiny_fp32", "--steps", "5", "--warmup", "3",
                        "--no-cpu-baseline"], cwd=root, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches",
                "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "tiny_fp32" and "model" not in d["config"]
    sys.path.insert(0, root)
    import bench
    from moe_expert_routing_route_gb300 import inputs
    assert d["config"] == bench.workload_config(inputs.CONFIGS["tiny_fp32"], 1)  # the reference arm's too
    assert {"expert_load", "shared_expert_sms"} <= set(d["workload_stats"])
    rl = d["roofline"]
    assert rl["bound"] in ("hbm", "tensor") and rl["unit"] in ("GB/s", "TFLOP/s")
    assert rl["achieved"] > 0 and rl["peak"] > 0 and abs(rl["frac"] - rl["achieved"] / rl["peak"]) < 1e-9
    assert "traffic" in rl
    # whole-layer roofline: reproducible from the stage costs in the line
    sc = rl["stage_costs"]
    assert rl["layer_bytes"] == sum(v["bytes"] for v in sc.values())
    assert rl["layer_flops"] == sum(v["flops"] for v in sc.values())
    assert abs(rl["layer_frac"] - rl["layer_ideal_ms"] / d["ms_per_step"]) < 1e-9
    assert 0 < rl["layer_frac_stagewise"] and rl["layer_frac"] <= rl["layer_frac_stagewise"] + 1e-12
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == e["d2h_bytes_per_step"] == 64 * 256 * 4
    assert d["gpu_launches"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
