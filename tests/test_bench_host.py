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
