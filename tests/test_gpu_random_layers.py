"""GPU parity of the whole layer on seeded random configurations: combinations of
T, H, E, k, I, S, dtype, group-limited routing and the GEMM tile shape that the
fixed lists do not spell out, each checked against the oracle on every token."""
import numpy as np
import pytest
import torch

from moe_expert_routing_route_gb300 import inputs
from tests.test_gpu_layer import check_layer, make

pytestmark = pytest.mark.gpu


def _config(i: int) -> tuple[inputs.LayerConfig, str]:
    rng = np.random.default_rng(1000 + i)
    dtype = "f32" if i % 5 == 4 else "bf16"
    E = int(rng.choice([1, 3, 8, 24, 40, 64, 130]))
    k = int(rng.integers(1, min(E, 8) + 1))
    n_group, topk_group, rule = 1, 1, "max"
    if E >= 8 and E % 4 == 0 and i % 3 == 0:  # group-limited routing
        n_group = int(rng.choice([g for g in (2, 4, 8) if E % g == 0]))
        topk_group = int(rng.integers(1, n_group + 1))
        while k > topk_group * (E // n_group):
            topk_group += 1
        rule = "top2_sum" if (E // n_group) >= 2 and i % 2 else "max"
    cfg = inputs.LayerConfig(f"rand{i}", T=int(rng.integers(1, 700)), H=int(rng.choice([64, 136, 256, 264, 512])),
                             E=E, k=k, I=int(rng.choice([64, 128, 200, 256, 384])), S=int(rng.integers(0, 3)),
                             dtype=dtype, seed=2000 + i, renormalize=bool(i % 4 != 1), n_group=n_group,
                             topk_group=topk_group, group_rule=rule)
    tile = ["auto", "single", "pair"][i % 3]
    return cfg, tile


CASES = [_config(i) for i in range(16)]


@pytest.mark.parametrize("cfg,tile", CASES, ids=[f"{c.name}-{t}" for c, t in CASES])
def test_random_layer(oracle, monkeypatch, cfg, tile):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    if tile == "auto":
        monkeypatch.delenv("MOE_GEMM_TILE", raising=False)
    else:
        monkeypatch.setenv("MOE_GEMM_TILE", tile)
    d, layer = make(cfg)
    out = layer.forward(d["x"])
    check_layer(oracle, cfg, d, layer, out)
