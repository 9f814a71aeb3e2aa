"""Roofline accounting (host logic of the benchmark) pinned to the pages' formulas
and printed numbers (CPU only)."""
import json
import os

import pytest

from moe_expert_routing_route_gb300 import roofline

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "roofline_examples.json")))


def test_worked_example_tokens_per_expert():
    g = GOLDEN["groupgemm_worked_example"]
    assert roofline.balanced_tokens_per_expert(g["batch"], g["q_len"], g["top_k"], g["ranks"],
                                               g["experts"]) == g["m"]


def test_group_gemm_reduces_to_gemm():
    assert roofline.group_gemm_cost(1, 7, 5, 3) == roofline.gemm_cost(7, 5, 3)
    f, b = roofline.group_gemm_cost(4, 7, 5, 3)
    assert f == 4 * roofline.gemm_cost(7, 5, 3)[0] and b == 4 * roofline.gemm_cost(7, 5, 3)[1]


def test_routed_up_projection_is_a_group_gemm_with_half_output():
    """Equal expert loads: the fused SwiGLU up GEMM is the GroupGEMM of the page with
    n = 2I, except that it writes h (I columns) instead of the 2I-wide product."""
    T, H, E, k, I = 4096, 7168, 256, 8, 2048
    m = T * k // E
    fl, el = roofline.group_gemm_cost(E, m, H, 2 * I)
    c = roofline.gemm_part_costs(T, H, E, k, I, 1, 2, touched=E)
    assert c["up_routed"][0] == fl
    assert c["up_routed"][1] == 2 * (el - E * m * I)
    fl2, el2 = roofline.group_gemm_cost(E, m, I, H)
    assert c["down_routed"] == (fl2, 2 * el2)


def test_dsv3_prefill_is_weight_bound_on_measured_peaks():
    """At ~128 rows per expert the grouped GEMM sits left of the ridge point (the
    page: GroupGEMM is memory-bound in most configurations)."""
    T, H, E, k, I = 4096, 7168, 256, 8, 2048
    c = roofline.gemm_part_costs(T, H, E, k, I, 1, 2, touched=E)
    f, b = c["up_routed"]
    peaks = dict(hbm_gbs=6787.2, bf16_tflops=1927.2, bf16_tflops_sustained=1721.0)
    assert f / b < peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    e = roofline.roofline_entry(f, b, 3e-3, peaks)
    assert e["bound"] == "hbm" and e["unit"] == "GB/s"
    assert e["achieved"] == pytest.approx(b / 3e-3 / 1e9)


def test_h100_ridge_point():
    h = GOLDEN["h100_roofline"]
    assert h["tflops"] * 1e12 / (h["tbs"] * 1e12) == pytest.approx(590.7, rel=1e-3)


def test_prefill_table_split_is_consistent():
    p = GOLDEN["prefill_table"]
    tokens = p["requests"] * p["tokens_per_request"]
    for r in p["rows"]:
        total = tokens / (r["latency_ms"] / 1e3)
        assert abs(total - r["total_tokens_s"]) < 1.0
        assert int(total / p["cards"]) == r["per_card_tokens_s"]


def test_stage_costs_sum_the_parts():
    T, H, E, k, I, S = 4096, 2048, 64, 6, 1408, 2
    parts = roofline.gemm_part_costs(T, H, E, k, I, S, 2, touched=E)
    st = roofline.stage_costs(T, H, E, k, I, S, 2, touched=E)
    assert st["shared"] == tuple(a + b for a, b in zip(parts["up_shared"], parts["down_shared"]))
    assert st["up"] == parts["up_routed"] and st["down"] == parts["down_routed"]
    assert list(st) == ["gate", "route", "init_routing", "permute_rows", "shared", "up", "down", "finalize"]


def test_layer_roofline_is_the_slower_ceiling_over_all_stages():
    """dsv3 prefill: the summed bytes at HBM bandwidth exceed the summed FLOPs at the
    sustained tensor peak, so the layer is HBM-bound and frac = (bytes / BW) / time."""
    T, H, E, k, I, S = 4096, 7168, 256, 8, 2048, 1
    costs = roofline.stage_costs(T, H, E, k, I, S, 2, touched=E)
    peaks = dict(hbm_gbs=6787.2, bf16_tflops=1927.2, bf16_tflops_sustained=1721.0)
    lr = roofline.layer_roofline(costs, 4.169e-3, peaks)
    nbytes = sum(b for _, b in costs.values())
    flops = sum(f for f, _ in costs.values())
    assert lr["layer_bound"] == "hbm"
    assert lr["layer_bytes"] == nbytes and lr["layer_flops"] == flops
    assert lr["layer_frac"] == pytest.approx(nbytes / 6787.2e9 / 4.169e-3)
    assert 0.85 < lr["layer_frac"] < 0.95  # 25.2 GB in 4.169 ms
    # the compute ceiling alone: 3.26 TFLOP at 1721 TFLOP/s
    assert lr["layer_compute_ms"] == pytest.approx(flops / 1721e12 * 1e3)


def test_layer_roofline_compute_bound_and_fp8_scale():
    """A skewed 16K-token layer is compute-bound; FP8 expert GEMMs halve the GEMM
    stages' compute time but not the gate's."""
    T, H, E, k, I, S = 16384, 7168, 256, 8, 2048, 1
    costs = roofline.stage_costs(T, H, E, k, I, S, 2, touched=E)
    peaks = dict(hbm_gbs=6787.2, bf16_tflops=1927.2, bf16_tflops_sustained=1721.0)
    lr = roofline.layer_roofline(costs, 12e-3, peaks)
    assert lr["layer_bound"] == "tensor"
    lr8 = roofline.layer_roofline(costs, 12e-3, peaks, gemm_tensor_scale=2.0)
    gate_ms = costs["gate"][0] / 1721e12 * 1e3
    assert lr8["layer_compute_ms"] == pytest.approx(gate_ms + (lr["layer_compute_ms"] - gate_ms) / 2)
