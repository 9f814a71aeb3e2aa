"""Benchmark of the MoE layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dsv3_prefill] [--no-cpu-baseline]

One step = one full layer forward (gate GEMM, top-k routing, init-routing,
row permutation, grouped SwiGLU up GEMM, grouped down GEMM, shared expert,
finalize) over one batch of T tokens with inputs resident in HBM.  The default
workload is the DeepSeek-V3-shaped prefill layer: T=4096, H=7168, 256 routed
experts, top-8, I=2048, one shared expert, bf16 (synthetic, seeded).  Weights
(22.6 GB) are far larger than L2, so every step streams them from HBM.

Multi-GPU: the layer does not shard here (one process per GPU runs an
independent replica on its own batch), so N GPUs process N batches per step
("scaling": "weak"); value = tokens of all ranks / max step time over ranks.

--impl reference times the CPU oracle (test infrastructure) on the host cores
on a bounded sample of tokens of the same workload, and prints the same line
with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from moe_expert_routing_route_gb300 import inputs, roofline  # noqa: E402

METRIC = "MoE-layer tokens/sec at 1 GB300; grouped-GEMM % tensor peak; routing GB/s vs HBM"
UNIT = "tokens/s"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
KERNEL_SOURCES = {
    "up": "gemm_tc.cu", "down": "gemm_tc.cu", "shared": "gemm_tc.cu", "gate": "gemm_tc.cu",
    "permute_rows": "permute.cu",
    "init_routing": "permute.cu", "route": "route.cu", "finalize": "finalize.cu",
}


# ---- distributed plumbing (replicas only; used for barrier and max-over-ranks) ----

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- clocks during the timed region ----

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.samples = []  # (host time, fields)
        self.proc = None
        uuid = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            pass
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
               "-lms", "10"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [s.strip() for s in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        rows = [f for (t, f) in self.samples if t0 <= t <= t1 + 0.05]
        if not rows and self.samples:  # window shorter than the sampling period: nearest sample
            rows = [min(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[1]]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for f in rows:
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, f[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(sm) if sm else None, sm_max_mhz=max(smax) if smax else None,
                    reasons=sorted(reasons), samples=len(sm))


# ---- roofline inputs ----

def source_hash(name: str) -> str:
    p = os.path.join(ROOT, "moe_expert_routing_route_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_traffic(stage: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source as it is now (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    for line in open(TRAFFIC_FILE):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == stage and parts[1] == workload:
            src = KERNEL_SOURCES[stage]
            if "fp8" in workload and stage in ("up", "down", "shared"):
                src = "gemm_fp8.cu"  # FP8 layers run their expert GEMMs on the e4m3 kernel
            if parts[3] == source_hash(src):
                return float(parts[2])
    return None


def routing_ops_alone(layer, x, cfg, costs, peaks, steps, stream) -> dict:
    """The routing ops each by itself on the GPU, on this batch's own routing (the layer's
    workspace after its last forward): moe_init_routing (histogram, scan, stable scatter and
    the expanded_x row gather) and moe_finalize_routing (weighted combine plus the shared
    expert's rows).  CUDA events around `steps` calls on the launching stream after one
    warm-up call; each call writes or reads more than L2 holds at the full sizes.  Bytes are
    the algorithmic ones of roofline.stage_costs, against the measured HBM bandwidth."""
    from moe_expert_routing_route_gb300 import binding
    ids = layer.field("topk_ids").clone()
    w = layer.field("topk_w").clone()
    row_idx = layer.field("expanded_row_idx").clone()
    y = layer.field("y_routed").clone()
    ys = layer.field("y_shared").clone() if cfg.S else None
    ws = torch.empty(binding.lib().moe_init_routing_workspace_bytes(cfg.T, cfg.E, cfg.k), dtype=torch.uint8,
                     device=x.device)
    calls = dict(init_routing=lambda: binding.moe_init_routing(x, ids, cfg.E, stream=stream, ws=ws),
                 finalize=lambda: binding.moe_finalize_routing(y, w, row_idx, skip=ys, stream=stream))
    nbytes = dict(init_routing=costs["init_routing"][1] + costs["permute_rows"][1], finalize=costs["finalize"][1])
    res = {}
    for name, call in calls.items():
        call()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(steps):
            call()
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) / steps * 1e3
        gbs = nbytes[name] / (us / 1e6) / 1e9
        res[name] = dict(us=round(us, 2), gbs=round(gbs, 1), frac=round(gbs / peaks["hbm_gbs"], 3))
    return res


# ---- the CPU oracle on a bounded sample ----

def sample_tokens(cfg, n: int, offset: int = 0) -> np.ndarray:
    g = inputs.generator("cpu", cfg.seed + offset, "misc")
    return torch.randperm(cfg.T, generator=g)[:n].sort().values.numpy().astype(np.int32)


def oracle_layer_time(cfg, host: dict, toks: np.ndarray) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.layer(host["x"], host["wg"], host["w_gate"], host["w_up"], host["w2"], host.get("s_gate"),
                 host.get("s_up"), host.get("s2"), k=cfg.k, renorm=cfg.renormalize, bias=host.get("bias"),
                 tokens=toks, n_group=cfg.n_group, topk_group=cfg.topk_group, group_rule=cfg.group_rule)
    return time.perf_counter() - t0


def host_layer(d: dict) -> dict:
    return {k: inputs.to_numpy(v) for k, v in d.items() if isinstance(v, torch.Tensor)}


def cpu_baseline(cfg, host: dict, budget_s: float = 15.0) -> dict:
    import oracle
    # probe with one token per thread (the oracle parallelises over tokens), then
    # scale the sample to the budget; rescale once if it still ran short
    n = min(cfg.T, max(4, oracle.num_threads()))
    t = oracle_layer_time(cfg, host, sample_tokens(cfg, n))
    for attempt in range(2):
        if t >= 0.7 * budget_s or n >= cfg.T:
            break
        n = int(max(4, min(cfg.T, n * budget_s / max(t, 1e-3))))
        t = oracle_layer_time(cfg, host, sample_tokens(cfg, n, offset=1 + attempt))
    return dict(value=n / t, unit=UNIT, cores=min(oracle.num_threads(), n), kind="oracle",
                sample=f"{n} of {cfg.T} tokens of {cfg.name}, whole layer per token in fp64 "
                       f"(gate, routing, shared + {cfg.k} routed SwiGLU experts), {t:.1f} s")


# ---- arms ----

def workload_config(cfg, world: int) -> dict:
    """The bench line's `config`: the workload alone, identical in both arms (the reference arm
    times a sample of the same batch, which its cpu_baseline names)."""
    return dict(workload=cfg.name, T=cfg.T, H=cfg.H, E=cfg.E, k=cfg.k, I=cfg.I, S=cfg.S, global_batch=cfg.T * world,
                parallelism=f"replicas{world}",
                l2="inputs larger than L2: 22.6 GB of expert weights streamed every step"
                if cfg.H == 7168 else "small workload")


def run_reference(args, world, rank):
    cfg = inputs.CONFIGS[args.workload]
    if rank != 0:
        return
    import oracle
    oracle.build()
    # the same seeded workload as the GPU arm (drawn on the GPU when there is one)
    d = inputs.make_layer(cfg, "cuda" if torch.cuda.is_available() else "cpu")
    host = host_layer(d)
    del d
    toks = sample_tokens(cfg, args.ref_tokens)
    for _ in range(args.warmup):
        oracle_layer_time(cfg, host, toks)
    times = [oracle_layer_time(cfg, host, toks) for _ in range(args.steps)]
    per_step = sum(times) / len(times)
    value = args.ref_tokens / per_step
    cores = min(oracle.num_threads(), args.ref_tokens)
    line = dict(metric=METRIC, value=value, unit=UNIT, n_gpus=args.gpus, steps=args.steps, warmup=args.warmup,
                ms_per_step=per_step * 1e3, higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="f64", data="synthetic", impl="reference",
                config=workload_config(cfg, world), tokens_per_step=args.ref_tokens,
                cpu_baseline=dict(value=value, unit=UNIT, cores=cores, kind="oracle",
                                  sample=f"{args.ref_tokens} of {cfg.T} tokens of {cfg.name} per step"),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    from moe_expert_routing_route_gb300 import binding

    cfg = inputs.CONFIGS[args.workload]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build_library()

    d = inputs.make_layer(cfg, dev)
    layer = binding.MoELayer(T=cfg.T, k=cfg.k, w_router=d["wg"], w_gate=d["w_gate"], w_up=d["w_up"], w2=d["w2"],
                             s_gate=d["s_gate"] if cfg.S else None, s_up=d["s_up"] if cfg.S else None,
                             s2=d["s2"] if cfg.S else None, expert_bias=d["bias"], renormalize=cfg.renormalize,
                             n_group=cfg.n_group, topk_group=cfg.topk_group, group_rule=cfg.group_rule,
                             weight_format=cfg.weight_format)
    if cfg.weight_format in ("fp8", "fp8_pow2"):  # the bf16 expert weights are no longer needed on the device
        for key in ("w_gate", "w_up", "w2"):
            d[key] = d[key].cpu() if not args.no_cpu_baseline else None
        torch.cuda.empty_cache()
    x = d["x"]
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    nst = binding.MOE_NUM_STAGES
    if args.ep > 1:
        return run_ours_ep(args, world, rank, local, cfg, layer, x, out)
    for _ in range(args.warmup):
        layer.forward(x, out)
    torch.cuda.synchronize()
    if layer.device_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    # inside the timed region, events around the two routed GEMM stages only (the dominant kernel's
    # duration); the full per-stage table comes from a second pass below
    names = binding.stage_names()
    timed_stages = ("up", "down")
    tev = [[torch.cuda.Event(enable_timing=True) if names[j // 2] in timed_stages else None
            for j in range(2 * nst)] for _ in range(args.steps)]
    for step_evs in tev:  # create the CUDA events before the timed region
        for e in step_evs:
            if e is not None:
                e.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    time.sleep(0.1)
    launches0 = binding.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        layer.forward(x, out, events=tev[i])
    end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    launches = binding.launch_count() - launches0
    clk = clocks.summary(wall0, wall1)
    clocks.stop()
    ms = start.elapsed_time(end) / args.steps
    ms_max = max_over_ranks(ms, world)
    if layer.device_status() != 0:
        raise RuntimeError("device status word set during the timed region")
    timed_ms = {n: sum(tev[i][2 * names.index(n)].elapsed_time(tev[i][2 * names.index(n) + 1])
                       for i in range(args.steps)) / args.steps for n in timed_stages}

    # per-stage times from a second pass of K steps with events recorded between all stages (outside
    # the timed region: 16 event records per forward cost the small layers a quarter of their time)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nst)] for _ in range(args.steps)]
    for step_evs in evs:
        for e in step_evs:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        layer.forward(x, out, events=evs[i])
    torch.cuda.synchronize()
    stage_ms = {name: sum(evs[i][2 * s].elapsed_time(evs[i][2 * s + 1]) for i in range(args.steps)) / args.steps
                for s, name in enumerate(binding.stage_names())}
    if layer.device_status() != 0:
        raise RuntimeError("device status word set during the stage pass")

    graph_ms = None
    if args.graph:
        # the same forward captured once into a CUDA graph ([BLOG §CUDA Graph]) and replayed K times:
        # what a serving loop pays per layer once launch costs are gone
        cs = torch.cuda.Stream()
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            layer.forward(x, out)  # warm-up on the capture stream
        stream.wait_stream(cs)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer.forward(x, out)
        for _ in range(args.warmup):
            graph.replay()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        g0.record()
        for _ in range(args.steps):
            graph.replay()
        g1.record()
        torch.cuda.synchronize()
        graph_ms = max_over_ranks(g0.elapsed_time(g1) / args.steps, world)
        if layer.device_status() != 0:
            raise RuntimeError("device status word set during graph replay")

    # roofline of the dominant kernel
    counts = layer.field("tokens_per_expert").cpu().numpy()
    touched = int((counts > 0).sum())
    load = dict(max=int(counts.max()), mean=float(counts.mean()), min=int(counts.min()),
                empty=int((counts == 0).sum()))  # the realised expert histogram of this batch
    fp8 = cfg.weight_format in ("fp8", "fp8_pow2")
    costs = roofline.stage_costs(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.S, cfg.esize, touched,
                                 weight_bytes=1 if fp8 else None)
    peaks = roofline.load_peaks()
    # the dominant kernel among the main stream's stages (the shared experts run on the second stream,
    # beside the routing steps or, with the SMs split, beside the routed up projection)
    top = max((n for n in stage_ms if n != "shared"), key=stage_ms.get)
    fl, by = costs[top]
    top_ms = timed_ms.get(top, stage_ms[top])  # the timed region's own events where it has them
    rl = roofline.roofline_entry(fl, by, top_ms / 1e3, peaks, sustained=True,
                                 tensor_scale=2.0 if fp8 and top in ("up", "down", "shared") else 1.0)
    rl["traffic"] = measured_traffic(top, cfg.name)
    rl["kernel"] = top
    rl["duration_source"] = "timed region" if top in timed_ms else "stage pass"
    rl["algorithmic_bytes"] = by
    rl["algorithmic_flops"] = fl
    rl["peak_source"] = peaks["source"]
    # the whole layer against the slower of its summed FLOPs at the tensor peak and
    # its summed bytes at HBM bandwidth
    rl.update(roofline.layer_roofline(costs, ms_max / 1e3, peaks, sustained=True,
                                      gemm_tensor_scale=2.0 if fp8 else 1.0))
    rl["stage_costs"] = {name: dict(flops=f_, bytes=b_) for name, (f_, b_) in costs.items()}
    stages = {}
    for name, t in stage_ms.items():
        f_, b_ = costs[name]
        stages[name] = dict(us=round(t * 1e3, 2), tflops=round(f_ / (t / 1e3) / 1e12, 2) if t > 0 else None,
                            gbs=round(b_ / (t / 1e3) / 1e9, 1) if t > 0 else None)
        if name in timed_ms:  # the same stage inside the timed region (events around it alone)
            tt = timed_ms[name]
            stages[name].update(timed_us=round(tt * 1e3, 2), timed_gbs=round(b_ / (tt / 1e3) / 1e9, 1) if tt > 0 else None)
    layer_fl = sum(f for f, _ in costs.values())
    gemm_fl = sum(costs[s][0] for s in ("up", "down", "shared"))
    gemm_ms = sum(stage_ms[s] for s in ("up", "down", "shared"))

    # end to end from pinned host memory through the C ABI
    x_host = x.cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    layer.forward_host(x_host, out_host)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        layer.forward_host(x_host, out_host)
    e2e_s = (time.perf_counter() - t0) / args.steps
    e2e_s = max_over_ranks(e2e_s, world)
    nbytes_io = x.numel() * x.element_size()
    routing_ops = routing_ops_alone(layer, x, cfg, costs, peaks, args.steps, stream)

    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline and not fp8:
        import oracle
        oracle.build()
        cpu = cpu_baseline(cfg, host_layer(d), budget_s=args.cpu_budget)

    if rank == 0:
        tokens = cfg.T * world
        line = dict(metric=METRIC, value=tokens / (ms_max / 1e3), unit=UNIT, n_gpus=world, steps=args.steps,
                    warmup=args.warmup, ms_per_step=ms_max, higher_is_better=True, scaling="weak",
                    vs_baseline=None,
                    # FP8 layers multiply e4m3 codes in the expert GEMMs; gate, routing and outputs stay bf16
                    dtype="e4m3+bf16" if fp8 else cfg.dtype, data="synthetic (seeded N(0,1) x, N(0,1/sqrt(fan_in)) "
                    "weights, random-init DeepSeek-V3-shaped MoE layer)",
                    config=workload_config(cfg, world),
                    # what this batch realised: the expert histogram and the SMs given to the shared experts
                    workload_stats=dict(expert_load=load, shared_expert_sms=layer.shared_expert_sms()),
                    roofline=rl, cpu_baseline=cpu,
                    e2e=dict(value=tokens / e2e_s, unit=UNIT, h2d_bytes_per_step=nbytes_io,
                             d2h_bytes_per_step=nbytes_io),
                    gpu_launches=int(launches), clocks=clk, stages=stages, routing_ops_alone=routing_ops,
                    grouped_gemm=dict(tflops=round(gemm_fl / (gemm_ms / 1e3) / 1e12, 1),
                                      frac_of_bf16_peak=round(gemm_fl / (gemm_ms / 1e3) / 1e12 /
                                                              peaks["bf16_tflops_sustained"], 3)),
                    layer_tflops=round(layer_fl / (ms_max / 1e3) / 1e12, 1))
        if graph_ms is not None:
            line["graph"] = dict(ms_per_step=graph_ms, value=tokens / (graph_ms / 1e3), unit=UNIT)
        print(json.dumps(line), flush=True)


def run_ours_ep(args, world, rank, local, cfg, layer, x, out):
    """The layer through expert-parallel Double-Routing with --ep virtual ranks on one GPU."""
    from moe_expert_routing_route_gb300 import binding
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        layer.forward_ep(x, args.ep, out)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    time.sleep(0.1)
    launches0 = binding.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    start.record(stream)
    for _ in range(args.steps):
        layer.forward_ep(x, args.ep, out)
    end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    launches = binding.launch_count() - launches0
    clk = clocks.summary(wall0, wall1)
    clocks.stop()
    if binding.moe_check_device_status(layer.ws_ep) != 0:
        raise RuntimeError("device status word set during the timed region")
    ms_max = max_over_ranks(start.elapsed_time(end) / args.steps, world)
    layer.forward(x, out)  # the single-routing pass fills the routing fields read below
    counts = layer.field("tokens_per_expert").cpu().numpy()
    costs = roofline.stage_costs(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.S, cfg.esize, int((counts > 0).sum()))
    fl, by = sum(c[0] for c in costs.values()), sum(c[1] for c in costs.values())
    peaks = roofline.load_peaks()
    rl = roofline.roofline_entry(fl, by, ms_max / 1e3, peaks, sustained=True)
    rl.update(kernel="whole layer (double routing)", traffic=None, algorithmic_bytes=by, algorithmic_flops=fl)
    rl.update(roofline.layer_roofline(costs, ms_max / 1e3, peaks, sustained=True))
    if rank == 0:
        tokens = cfg.T * world
        print(json.dumps(dict(metric=METRIC, value=tokens / (ms_max / 1e3), unit=UNIT, n_gpus=world,
                              steps=args.steps, warmup=args.warmup, ms_per_step=ms_max, higher_is_better=True,
                              scaling="weak", vs_baseline=None, dtype=cfg.dtype, data="synthetic",
                              config=dict(workload=cfg.name, ep_virtual_ranks=args.ep, T=cfg.T, H=cfg.H, E=cfg.E,
                                          k=cfg.k, I=cfg.I, S=cfg.S, parallelism=f"replicas{world}"),
                              roofline=rl, cpu_baseline=None, gpu_launches=int(launches), clocks=clk)), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3_prefill", choices=sorted(inputs.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=16, help="tokens per step for --impl reference")
    ap.add_argument("--graph", action="store_true",
                    help="also time K replays of one forward captured into a CUDA graph")
    ap.add_argument("--ep", type=int, default=1,
                    help="run the layer through expert-parallel Double-Routing with this many virtual ranks")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
