"""Seeded synthetic inputs for the MoE layer, shared by the tests, the smoke check and
the benchmark (both the CUDA path and the CPU oracle are fed from here).

This module draws random numbers and lays them out; it holds none of the layer's
arithmetic.  Every tensor block comes from its own ``torch.Generator`` seeded
from (config seed, tensor tag, block index), so a subset (one expert's weights, a
few tokens) can be regenerated on its own.  Draws happen on the device given;
CPU and CUDA generators give different (equally valid) streams, so a test
generates once and hands the same tensors to both sides.

Recipe (the workloads of the DeepSeek-V3/R1 MoE layer: 256 routed experts,
top-8, one shared expert):
  x ~ N(0, 1); router weight wg [E,H] ~ N(0, 1/sqrt(H)) (standard deviation);
  expert gate/up weights [E,I,H] ~ N(0, 1/sqrt(H)); down weights [E,H,I] ~
  N(0, 1/sqrt(I)); shared experts likewise; values drawn in fp32 and rounded
  (RNE) to the storage dtype.  The skewed workload adds a per-expert bias
  log p_rank(e) with p_i proportional to i^-s over a seeded random ranking of
  the experts (Zipf popularity).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    S: int
    dtype: str  # "f32" | "bf16"
    seed: int
    zipf_s: float | None = None
    renormalize: bool = True
    n_group: int = 1          # > 1: group-limited routing
    topk_group: int = 1
    group_rule: str = "max"   # "max" | "top2_sum"
    weight_format: str = "native"  # "native" | "fp8" (e4m3 expert weights, 128x128 tile scales) | "fp8_pow2"

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def replace(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny fp32 layer, a mid-size bf16 layer, and three
# DeepSeek-V3-shaped layers (prefill, decode, Zipf-skewed long prefill).
CONFIGS = {
    "tiny_fp32": LayerConfig("tiny_fp32", T=64, H=256, E=16, k=2, I=128, S=1, dtype="f32", seed=0),
    "mid_bf16": LayerConfig("mid_bf16", T=4096, H=2048, E=64, k=6, I=1408, S=2, dtype="bf16", seed=1),
    "dsv3_prefill": LayerConfig("dsv3_prefill", T=4096, H=7168, E=256, k=8, I=2048, S=1,
                                dtype="bf16", seed=2),
    "dsv3_decode": LayerConfig("dsv3_decode", T=128, H=7168, E=256, k=8, I=2048, S=1,
                               dtype="bf16", seed=3),
    "dsv3_zipf_prefill": LayerConfig("dsv3_zipf_prefill", T=16384, H=7168, E=256, k=8, I=2048,
                                     S=1, dtype="bf16", seed=4, zipf_s=1.2),
    # The prefill layer with DeepSeek-V3's group-limited routing (8 groups of 32
    # experts, 4 groups kept, group score = sum of its two best scores).
    "dsv3_prefill_grouped": LayerConfig("dsv3_prefill_grouped", T=4096, H=7168, E=256, k=8, I=2048, S=1,
                                        dtype="bf16", seed=2, n_group=8, topk_group=4, group_rule="top2_sum"),
    # The prefill and decode layers with FP8 (e4m3) block-quantised expert weights.
    "dsv3_prefill_fp8": LayerConfig("dsv3_prefill_fp8", T=4096, H=7168, E=256, k=8, I=2048, S=1, dtype="bf16",
                                    seed=2, weight_format="fp8"),
    "dsv3_decode_fp8": LayerConfig("dsv3_decode_fp8", T=128, H=7168, E=256, k=8, I=2048, S=1, dtype="bf16",
                                   seed=3, weight_format="fp8"),
    "dsv3_prefill_slice_fp8": LayerConfig("dsv3_prefill_slice_fp8", T=512, H=7168, E=32, k=8, I=2048, S=1,
                                          dtype="bf16", seed=2, weight_format="fp8"),
    # The same three with power-of-two block scales (products on block-scaled tensor-core MMAs).
    "dsv3_prefill_fp8_pow2": LayerConfig("dsv3_prefill_fp8_pow2", T=4096, H=7168, E=256, k=8, I=2048, S=1,
                                         dtype="bf16", seed=2, weight_format="fp8_pow2"),
    "dsv3_decode_fp8_pow2": LayerConfig("dsv3_decode_fp8_pow2", T=128, H=7168, E=256, k=8, I=2048, S=1,
                                        dtype="bf16", seed=3, weight_format="fp8_pow2"),
    "dsv3_prefill_slice_fp8_pow2": LayerConfig("dsv3_prefill_slice_fp8_pow2", T=512, H=7168, E=32, k=8, I=2048,
                                               S=1, dtype="bf16", seed=2, weight_format="fp8_pow2"),
    # Profiling slice: the DeepSeek-V3 prefill layer's per-expert shape (about 128 rows
    # per expert) on 32 experts, small enough for ncu captures (~5 GB on the device).
    "dsv3_prefill_slice": LayerConfig("dsv3_prefill_slice", T=512, H=7168, E=32, k=8, I=2048, S=1,
                                      dtype="bf16", seed=2),
    # Profiling slice of the skewed long prefill: 512 rows per expert on average over
    # 32 experts with the Zipf(1.2) popularity bias (~3 GB of weights on the device),
    # so the routed GEMMs are compute-bound and unevenly loaded as in the full layer.
    "dsv3_zipf_prefill_slice": LayerConfig("dsv3_zipf_prefill_slice", T=2048, H=7168, E=32, k=8, I=2048, S=1,
                                           dtype="bf16", seed=4, zipf_s=1.2),
}
CONFIG_ORDER = ["tiny_fp32", "mid_bf16", "dsv3_prefill", "dsv3_decode", "dsv3_zipf_prefill"]

_TAGS = dict(x=1, wg=2, w_gate=3, w_up=4, w2=5, s_gate=6, s_up=7, s2=8, zipf=9, logits=10,
             ids=11, y=12, scales=13, misc=14)


def generator(device, seed: int, tag: str, idx: int = 0) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed((int(seed) * 1_000_003 + _TAGS[tag] * 10_007 + int(idx)) % (2**62))
    return g


def _normal(shape, std, dtype, device, seed, tag, idx=0):
    g = generator(device, seed, tag, idx)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    return v.to(dtype)


def _per_expert(n, shape, std, dtype, device, seed, tag):
    out = torch.empty((n,) + tuple(shape), dtype=dtype, device=device)
    for e in range(n):
        out[e].copy_(_normal(shape, std, dtype, device, seed, tag, e))
    return out


def make_layer(cfg: LayerConfig, device="cpu", *, with_weights: bool = True) -> dict:
    """Draw x, router weight, expert weights, shared weights and (Zipf) bias."""
    dt = cfg.torch_dtype
    T, H, E, I, S = cfg.T, cfg.H, cfg.E, cfg.I, cfg.S
    d = dict(cfg=cfg)
    d["x"] = _normal((T, H), 1.0, dt, device, cfg.seed, "x")
    d["wg"] = _normal((E, H), 1.0 / math.sqrt(H), dt, device, cfg.seed, "wg")
    if with_weights:
        d["w_gate"] = _per_expert(E, (I, H), 1.0 / math.sqrt(H), dt, device, cfg.seed, "w_gate")
        d["w_up"] = _per_expert(E, (I, H), 1.0 / math.sqrt(H), dt, device, cfg.seed, "w_up")
        d["w2"] = _per_expert(E, (H, I), 1.0 / math.sqrt(I), dt, device, cfg.seed, "w2")
        d["s_gate"] = _per_expert(S, (I, H), 1.0 / math.sqrt(H), dt, device, cfg.seed, "s_gate")
        d["s_up"] = _per_expert(S, (I, H), 1.0 / math.sqrt(H), dt, device, cfg.seed, "s_up")
        d["s2"] = _per_expert(S, (H, I), 1.0 / math.sqrt(I), dt, device, cfg.seed, "s2")
    d["bias"] = zipf_bias(cfg, device) if cfg.zipf_s else None
    return d


def expert_weights(cfg: LayerConfig, e: int, device="cpu", shared: bool = False):
    """One expert's (gate [I,H], up [I,H], down [H,I]) exactly as make_layer draws them."""
    dt = cfg.torch_dtype
    H, I = cfg.H, cfg.I
    p = ("s_gate", "s_up", "s2") if shared else ("w_gate", "w_up", "w2")
    return (_normal((I, H), 1.0 / math.sqrt(H), dt, device, cfg.seed, p[0], e),
            _normal((I, H), 1.0 / math.sqrt(H), dt, device, cfg.seed, p[1], e),
            _normal((H, I), 1.0 / math.sqrt(I), dt, device, cfg.seed, p[2], e))


def zipf_bias(cfg: LayerConfig, device="cpu") -> torch.Tensor:
    """Per-expert popularity bias log p_rank(e), p_i ~ i^-s normalised over the E ranks,
    ranks a seeded random permutation of the experts (fp32)."""
    g = generator("cpu", cfg.seed, "zipf")
    rank = torch.randperm(cfg.E, generator=g)
    i = torch.arange(1, cfg.E + 1, dtype=torch.float64)
    p = i.pow(-float(cfg.zipf_s))
    p = p / p.sum()
    return torch.log(p[rank]).to(torch.float32).to(device)


# ---- inputs for the single-step tests ---------------------------------------

def random_logits(T: int, E: int, seed: int, device="cpu", ties: str | None = None) -> torch.Tensor:
    """fp32 router logits ~ N(0,1).  ties="quantised" rounds to multiples of 1/8 so
    that many equal values occur; ties="all_equal" makes every logit 0.5."""
    g = generator(device, seed, "logits")
    v = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
    if ties == "quantised":
        v = torch.round(v * 8) / 8
    elif ties == "all_equal":
        v = torch.full_like(v, 0.5)
    return v


def random_ids(T: int, k: int, E: int, seed: int, device="cpu", distinct: bool = True,
               weights: torch.Tensor | None = None) -> torch.Tensor:
    """int32 expert ids [T,k]; distinct per token when asked (sampling without
    replacement, optionally with per-expert weights)."""
    g = generator("cpu", seed, "ids")
    if distinct:
        w = torch.ones(E) if weights is None else weights.to(torch.float64).cpu()
        ids = torch.multinomial(w.expand(T, E).contiguous(), k, replacement=False, generator=g)
    else:
        ids = torch.randint(0, E, (T, k), generator=g)
    return ids.to(torch.int32).to(device)


def random_rows(n: int, H: int, dtype, seed: int, device="cpu", tag: str = "y") -> torch.Tensor:
    return _normal((n, H), 1.0, dtype, device, seed, tag)


def random_scales(T: int, k: int, seed: int, device="cpu") -> torch.Tensor:
    g = generator("cpu", seed, "scales")
    w = torch.rand((T, k), generator=g, dtype=torch.float32) + 0.05
    return (w / w.sum(dim=1, keepdim=True)).to(device)


# ---- marshalling helpers -------------------------------------------------------

def to_numpy(t: torch.Tensor) -> np.ndarray:
    """CPU numpy view for host-side consumers: bf16 tensors as uint16 bit patterns."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
