"""Algorithmic FLOPs and bytes of each layer step, for roofline fractions.

"Lower latency and higher throughput with multi-node DeepSeek deployment"
(Perplexity blog), §Roofline: the horizontal axis is arithmetic intensity, FLOPs
over memory I/O bytes computed from the kernel's semantics; the ceilings are the
peak tensor throughput and the memory bandwidth.  §Roofline / GroupGEMM: g
groups of [m,k]x[k,n] cost 2*g*m*k*n FLOPs and g*(m*k + n*k + m*n) elements of
I/O; §Roofline / GEMM: one [m,k]x[k,n] costs 2*m*k*n FLOPs and m*k + n*k + m*n
elements.

Bytes here are the compulsory traffic of each step: every input read once,
every output written once, weights of the experts that received at least one
row.  The fused SwiGLU up-projection writes h [rows, I] instead of the [rows, 2I]
GEMM output, so its output term is half the plain GroupGEMM one.
"""
from __future__ import annotations

import json
import os


def gemm_cost(m: int, k: int, n: int):
    """(FLOPs, I/O elements) of one [m,k]x[k,n] GEMM."""
    return 2 * m * k * n, m * k + n * k + m * n


def group_gemm_cost(g: int, m: int, k: int, n: int):
    """(FLOPs, I/O elements) of g equal groups of [m,k]x[k,n]."""
    return 2 * g * m * k * n, g * (m * k + n * k + m * n)


def balanced_tokens_per_expert(batch: int, q_len: int, top_k: int, ranks: int, experts: int) -> float:
    """Average rows per expert when `ranks` data-parallel ranks each route
    batch*q_len tokens to top_k of `experts` experts."""
    return batch * q_len * top_k * ranks / experts


def gemm_part_costs(T: int, H: int, E: int, k: int, I: int, S: int, esize: int, touched: int,
                    weight_bytes: int | None = None) -> dict:
    """{part: (flops, bytes)} of the four expert GEMMs: up/down x routed/shared.

    weight_bytes = 1 (FP8): weights and GEMM inputs are e4m3 codes (plus one fp32
    scale per 128x128 weight tile and per 1x128 input block); outputs stay esize."""
    R = T * k
    b = esize
    SI = S * I
    if weight_bytes is None:
        return {
            "up_routed": (2 * R * H * 2 * I, touched * 2 * I * H * b + R * H * b + R * I * b),
            "up_shared": (2 * T * H * 2 * SI, (2 * SI * H + T * H + T * SI) * b if S else 0),
            "down_routed": (2 * R * I * H, touched * H * I * b + R * I * b + R * H * b),
            "down_shared": (2 * T * SI * H, (H * SI + T * SI + T * H) * b if S else 0),
        }
    wb = weight_bytes
    ws = lambda n, kk: n * kk * wb + (n // 128) * ((kk + 127) // 128) * 4  # noqa: E731  codes + tile scales
    xs = lambda rows, kk: rows * kk * wb + rows * ((kk + 127) // 128) * 4  # noqa: E731  codes + block scales
    return {
        "up_routed": (2 * R * H * 2 * I, touched * ws(2 * I, H) + xs(R, H) + R * I * b),
        "up_shared": (2 * T * H * 2 * SI, (ws(2 * SI, H) + xs(T, H) + T * SI * b) if S else 0),
        "down_routed": (2 * R * I * H, touched * ws(H, I) + xs(R, I) + R * H * b),
        "down_shared": (2 * T * SI * H, (ws(H, SI) + xs(T, SI) + T * H * b) if S else 0),
    }


def stage_costs(T: int, H: int, E: int, k: int, I: int, S: int, esize: int, touched: int,
                weight_bytes: int | None = None) -> dict:
    """{stage: (flops, bytes)} for the eight layer stages.  touched = experts with >= 1 row.
    "shared" is both projections of the shared experts; "up"/"down" the routed ones."""
    R = T * k
    b = esize
    g = gemm_part_costs(T, H, E, k, I, S, esize, touched, weight_bytes)
    add = lambda a, c: (a[0] + c[0], a[1] + c[1])  # noqa: E731
    return {
        "gate": (2 * T * H * E, T * H * b + E * H * b + T * E * 4),
        "route": (0, T * E * 4 + R * 8),
        "init_routing": (0, 2 * R * 4 + R * 4 + (E + 1) * 4 + E * 4),
        "permute_rows": (0, T * H * b + R * H * b + R * 4),
        "shared": add(g["up_shared"], g["down_shared"]),
        "up": g["up_routed"],
        "down": g["down_routed"],
        "finalize": (0, R * H * b + (T * H * b if S else 0) + T * H * b + R * 8),
    }


def layer_flops(T: int, H: int, E: int, k: int, I: int, S: int) -> int:
    return sum(f for f, _ in stage_costs(T, H, E, k, I, S, 2, E).values())


def load_peaks(path: str | None = None) -> dict:
    """Measured peaks of this machine's GPUs if present, else the stated fallback."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    path = path or os.path.join(root, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


GEMM_STAGES = ("shared", "up", "down")


def layer_roofline(costs: dict, seconds: float, peaks: dict, sustained: bool = True,
                   gemm_tensor_scale: float = 1.0) -> dict:
    """The whole layer against its roofline: the ideal time is the slower of all
    stages' FLOPs at the tensor peak and all stages' bytes at HBM bandwidth
    (§Roofline: a kernel cannot beat either ceiling, and the layer's stages run
    back to back on one GPU); frac = ideal time / measured time.

    costs: stage_costs() output.  gemm_tensor_scale applies to the expert GEMM
    stages only (FP8 expert weights: 2, the nominal FP8/bf16 ratio); the gate
    GEMM stays on the bf16 peak."""
    tf = (peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]) * 1e12
    flops = sum(f for f, _ in costs.values())
    nbytes = sum(b for _, b in costs.values())
    t_compute = sum(f / (tf * (gemm_tensor_scale if s in GEMM_STAGES else 1.0)) for s, (f, _) in costs.items())
    t_bytes = nbytes / (peaks["hbm_gbs"] * 1e9)
    ideal = max(t_compute, t_bytes)
    # the stricter per-stage form: each stage at its own ceiling, stages not overlapped
    staged = sum(max(f / (tf * (gemm_tensor_scale if s in GEMM_STAGES else 1.0)), b / (peaks["hbm_gbs"] * 1e9))
                 for s, (f, b) in costs.items())
    return dict(layer_frac=ideal / seconds, layer_bound="tensor" if t_compute > t_bytes else "hbm",
                layer_ideal_ms=ideal * 1e3, layer_flops=flops, layer_bytes=nbytes,
                layer_compute_ms=t_compute * 1e3, layer_bytes_ms=t_bytes * 1e3,
                layer_frac_stagewise=staged / seconds)


def roofline_entry(flops: float, nbytes: float, seconds: float, peaks: dict, sustained: bool = True,
                   tensor_scale: float = 1.0) -> dict:
    """The binding roofline of one kernel: whichever of compute time at the
    tensor peak and byte time at HBM bandwidth is larger.  tensor_scale converts
    the measured bf16 peak to another operand type's (FP8: 2, the nominal
    4.5/2.25 PFLOP/s ratio)."""
    tf = (peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]) * tensor_scale
    t_compute = flops / (tf * 1e12) if flops else 0.0
    t_bytes = nbytes / (peaks["hbm_gbs"] * 1e9)
    if t_compute > t_bytes:
        achieved = flops / seconds / 1e12
        return dict(bound="tensor", achieved=achieved, peak=tf, unit="TFLOP/s", frac=achieved / tf)
    achieved = nbytes / seconds / 1e9
    return dict(bound="hbm", achieved=achieved, peak=peaks["hbm_gbs"], unit="GB/s", frac=achieved / peaks["hbm_gbs"])
