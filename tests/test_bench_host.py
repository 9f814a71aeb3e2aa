"""Host-side logic of bench.py on CPU: max-over-ranks timing and the barrier with
two gloo ranks (world_size 2), and the clock-sample summary."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import bench
    world, r, _ = bench.dist_setup()
    bench.barrier(world)
    v = bench.max_over_ranks(10.0 + 5 * rank, world)
    q.put((r, world, v))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 2, 15.0), (1, 2, 15.0)]


def test_clock_summary_window():
    import bench
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.samples = [(1.0, ["1500", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active", "Active"]),
                  (2.0, ["1800", "2070", "1000", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]),
                  (9.0, ["600", "2070", "100", "0x0", "Active", "Not Active", "Not Active", "Not Active"])]
    s = cs.summary(0.5, 2.5)
    assert s["sm_mhz"] == 1650 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    # a window shorter than the sampling period falls back to the nearest sample
    s = cs.summary(8.9, 8.95)
    assert s["reasons"] == ["hw_slowdown"]


def test_reference_arm_json_line_on_cpu():
    """`bench.py --impl reference` times the oracle on host cores; its one JSON line
    carries the contract's keys (run here on the small fp32 workload)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32", "--steps", "2",
                        "--warmup", "1", "--ref-tokens", "8"], cwd=root, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["value"] > 0
    assert d["config"]["workload"] == "tiny_fp32"
    # the same config object as the GPU arm's line, so that the two lines compare as one workload
    sys.path.insert(0, root)
    import bench
    from moe_expert_routing_route_gb300 import inputs
    assert d["config"] == bench.workload_config(inputs.CONFIGS["tiny_fp32"], 1)
    assert d["tokens_per_step"] == 8
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
