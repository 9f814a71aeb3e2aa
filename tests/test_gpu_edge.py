"""Degenerate inputs through the C ABI on the GPU: an empty batch through every
step and through the layer, and zero rows through the grouped FFN."""
import numpy as np
import pytest
import torch

from moe_expert_routing_route_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build_library()
    binding.lib()


def test_steps_on_an_empty_batch():
    E, k, H = 16, 2, 64
    logits = torch.empty((0, E), device=DEV)
    ids, w = binding.moe_route_topk(logits, k)
    assert ids.shape == (0, k) and w.shape == (0, k)
    x = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    ir = binding.moe_init_routing(x, ids, E)
    torch.cuda.synchronize()
    # the counts and offsets of an empty batch are written, all zero
    assert torch.equal(ir["tokens_per_expert"].cpu(), torch.zeros(E, dtype=torch.int32))
    assert torch.equal(ir["expert_offsets"].cpu(), torch.zeros(E + 1, dtype=torch.int32))
    assert binding.moe_check_device_status(ir["ws"]) == 0
    out = binding.moe_finalize_routing(torch.empty((0, H), dtype=torch.bfloat16, device=DEV), w,
                                       ir["expanded_row_idx"])
    assert out.shape == (0, H)


def test_grouped_ffn_zero_rows():
    E, H, I = 4, 64, 128
    a = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    offs = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    w13 = torch.zeros((E, 2 * 128, H), dtype=torch.bfloat16, device=DEV)
    w2 = torch.zeros((E, H, I), dtype=torch.bfloat16, device=DEV)
    y, ws = binding.moe_grouped_ffn(a, offs, E, I, w13, w2)
    assert y.shape == (0, H)
    assert binding.moe_check_device_status(ws) == 0


@pytest.mark.parametrize("S", [0, 1])
def test_layer_on_an_empty_batch(S):
    cfg = inputs.LayerConfig("empty", T=8, H=256, E=16, k=2, I=128, S=S, dtype="bf16", seed=30)
    d = inputs.make_layer(cfg, DEV)
    layer = binding.MoELayer(T=0, k=cfg.k, w_router=d["wg"], w_gate=d["w_gate"], w_up=d["w_up"], w2=d["w2"],
                             s_gate=d["s_gate"] if S else None, s_up=d["s_up"] if S else None,
                             s2=d["s2"] if S else None)
    x = torch.empty((0, cfg.H), dtype=torch.bfloat16, device=DEV)
    out = layer.forward(x)
    assert out.shape == (0, cfg.H)
    xh = torch.empty((0, cfg.H), dtype=torch.bfloat16).pin_memory()
    oh = torch.empty((0, cfg.H), dtype=torch.bfloat16).pin_memory()
    layer.forward_host(xh, oh)
    torch.cuda.synchronize()
