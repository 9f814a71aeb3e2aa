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


CASES = [_config(i) for i in range(32)]


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


def _host_config(i: int) -> inputs.LayerConfig:
    """Batches of 1025-3600 tokens: the host-buffer forward copies x in 2-4 chunks and runs the
    gate and top-k chunk by chunk as they arrive."""
    rng = np.random.default_rng(5000 + i)
    dtype = "f32" if i % 4 == 3 else "bf16"
    E = int(rng.choice([8, 32, 64]))
    k = int(rng.integers(1, min(E, 8) + 1))
    return inputs.LayerConfig(f"host{i}", T=int(rng.integers(1025, 3600)), H=int(rng.choice([128, 256, 512])),
                              E=E, k=k, I=int(rng.choice([64, 128, 256])), S=int(rng.integers(0, 3)),
                              dtype=dtype, seed=6000 + i)


HOST_CASES = [_host_config(i) for i in range(10)]


@pytest.mark.parametrize("cfg", HOST_CASES, ids=[c.name for c in HOST_CASES])
def test_random_host_path_matches_device(cfg):
    """The host-buffer forward (chunked copies, chunked gate and top-k) gives the device-buffer
    forward's output bit for bit."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    d, layer = make(cfg)
    dev = layer.forward(d["x"])
    x_host = d["x"].cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    layer.forward_host(x_host, out_host)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    assert torch.equal(out_host, dev.cpu())
