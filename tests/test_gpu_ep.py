"""GPU parity of expert-parallel Double-Routing on one GPU (re-routing, the
argsort-inverse un-sort, and the layer through W virtual ranks), through the C ABI.

The layer through W virtual ranks is checked three ways: its output against the
oracle's layer (routing, aggregate and per-token), its re-routed rows, their
source indices and the per-expert offsets against the oracle's Double-Routing
chain built from init_routing per rank and re_routing per receiving rank
("DeepSeek-R1 prefill inference optimisation on Atlas A3", §MoE deployment,
steps 1-4), and its output against the single-routing layer bit for bit."""
import numpy as np
import pytest
import torch

from moe_expert_routing_route_gb300 import binding, inputs
from tests._cmp import np_
from tests._layer_check import check_output, check_routing, host_arrays, oracle_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build_library()
    binding.lib()


def _counts(W, El, seed, hi=40):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, hi, size=(W, El)).astype(np.int32)
    if W > 2:
        c[1, :] = 0  # a source that sends nothing
    if El > 2:
        c[:, 2] = 0  # an expert that receives nothing
    return c


@pytest.mark.parametrize("W,El,H", [(1, 1, 8), (4, 5, 64), (8, 32, 512), (3, 300, 40), (32, 8, 16)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_re_routing(oracle, W, El, H, dtype):
    c = _counts(W, El, seed=W * El)
    N = int(c.sum())
    x = inputs.random_rows(max(N, 1), H, dtype, seed=N)[:N]
    got = binding.moe_re_routing(x.to(DEV), torch.from_numpy(c).to(DEV))
    assert binding.moe_check_device_status(got["ws"]) == 0
    ref = oracle.re_routing(np_(x), c)
    assert np.array_equal(got["gathered_ids_unsort"].cpu().numpy(), ref["gathered_ids_unsort"])
    assert np.array_equal(got["tokens_per_local_expert"].cpu().numpy(), ref["tokens_per_local_expert"])
    assert np.array_equal(got["local_offsets"].cpu().numpy(), ref["local_offsets"])
    assert np.array_equal(np_(got["x_sorted"]), ref["x_sorted"])
    # step 6: un-sort, and the page's index_select with the argsort of gathered_ids_unsort
    back = binding.moe_unsort_rows(got["x_sorted"], got["gathered_ids_unsort"])
    assert torch.equal(back.cpu(), x)
    gidx = got["gathered_ids_unsort"]
    assert torch.equal(torch.index_select(got["x_sorted"], 0, gidx.float().argsort().int()).cpu(), x)
    assert np.array_equal(np_(back), oracle.unsort_rows(ref["x_sorted"], ref["gathered_ids_unsort"]))


def test_re_routing_flags_count_mismatch():
    c = torch.tensor([[3, 4], [5, 0]], dtype=torch.int32, device=DEV)
    x = torch.zeros((11, 16), dtype=torch.bfloat16, device=DEV)  # counts add up to 12
    W, El = c.shape
    ws = torch.empty(binding.lib().moe_re_routing_workspace_bytes(W, El), dtype=torch.uint8, device=DEV)
    outs = [torch.empty_like(x), torch.empty(11, dtype=torch.int32, device=DEV),
            torch.empty(El, dtype=torch.int32, device=DEV), torch.empty(El + 1, dtype=torch.int32, device=DEV)]
    st = binding.lib().moe_re_routing(binding._ptr(x), binding.MOE_BF16, binding._ptr(c), W, El, 11, 16,
                                      *[binding._ptr(o) for o in outs], binding._ptr(ws), ws.numel(),
                                      binding._stream())
    assert st == binding.MOE_OK
    assert binding.moe_check_device_status(ws) & binding.MOE_DEVERR_BAD_OFFSETS


def oracle_double_routing(oracle, ids: np.ndarray, x: np.ndarray, E: int, W: int) -> dict:
    """Steps 1-4 of Double-Routing by the oracle: init-routing on each source
    rank's tokens, rank q receives from every source (in source order) the rows
    of its experts [q*E/W, (q+1)*E/W), then re-routes them by local expert."""
    T = ids.shape[0]
    Tp, El = T // W, E // W
    irs = [oracle.init_routing(ids[p * Tp:(p + 1) * Tp], x[p * Tp:(p + 1) * Tp], E) for p in range(W)]
    sorted_rows, gidx, eoff, recv_start = [], [], [], [0]
    for q in range(W):
        recv = np.concatenate([ir["expanded_x"][ir["expert_offsets"][q * El]:ir["expert_offsets"][(q + 1) * El]]
                               for ir in irs])
        counts = np.stack([ir["tokens_per_expert"][q * El:(q + 1) * El] for ir in irs]).astype(np.int32)
        rr = oracle.re_routing(recv, counts)
        base = recv_start[-1]
        sorted_rows.append(rr["x_sorted"])
        gidx.append(rr["gathered_ids_unsort"] + base)
        eoff.append(rr["local_offsets"][:-1] + base)
        recv_start.append(base + len(recv))
    eoff.append(np.array([recv_start[-1]], np.int32))
    return dict(x_sorted=np.concatenate(sorted_rows), gathered_ids_unsort=np.concatenate(gidx).astype(np.int32),
                expert_offsets=np.concatenate(eoff).astype(np.int32), recv_start=np.array(recv_start, np.int32))


EP_CASES = [
    (inputs.LayerConfig("ep_small_bf16", T=256, H=512, E=64, k=6, I=256, S=1, dtype="bf16", seed=41), [1, 2, 4, 8]),
    (inputs.LayerConfig("ep_fp32", T=64, H=128, E=16, k=2, I=64, S=1, dtype="f32", seed=42), [2, 4]),
    (inputs.LayerConfig("ep_noshared_bf16", T=96, H=264, E=24, k=5, I=200, S=0, dtype="bf16", seed=43), [2, 3]),
    (inputs.LayerConfig("ep_grouped_bf16", T=320, H=256, E=64, k=6, I=128, S=2, dtype="bf16", seed=44, n_group=8,
                        topk_group=3, group_rule="top2_sum"), [2, 8]),
    (inputs.LayerConfig("ep_zipf_bf16", T=384, H=256, E=48, k=8, I=128, S=1, dtype="bf16", seed=45, zipf_s=1.2),
     [3, 8]),
    (inputs.CONFIGS["dsv3_prefill"], [2, 8]),
]


@pytest.mark.parametrize("cfg,Ws", EP_CASES, ids=[c.name for c, _ in EP_CASES])
def test_layer_double_routing(oracle, cfg, Ws):
    d = inputs.make_layer(cfg, DEV)
    layer = binding.MoELayer(T=cfg.T, k=cfg.k, w_router=d["wg"], w_gate=d["w_gate"], w_up=d["w_up"], w2=d["w2"],
                             s_gate=d["s_gate"] if cfg.S else None, s_up=d["s_up"] if cfg.S else None,
                             s2=d["s2"] if cfg.S else None, expert_bias=d["bias"], renormalize=cfg.renormalize,
                             n_group=cfg.n_group, topk_group=cfg.topk_group, group_rule=cfg.group_rule)
    single = layer.forward(d["x"])
    n = host_arrays(d)
    full = cfg.T > 1024
    toks = None
    if full:  # a seeded sample of tokens at full size
        g = inputs.generator("cpu", cfg.seed, "misc")
        toks = torch.randperm(cfg.T, generator=g)[:32].sort().values.numpy().astype(np.int32)
    ref = oracle_layer(oracle, cfg, n, toks)
    toks = np.arange(cfg.T, dtype=np.int32) if toks is None else toks
    for W in Ws:
        ep = layer.forward_ep(d["x"], W)
        torch.cuda.synchronize()
        assert binding.moe_check_device_status(layer.ws_ep) == 0
        # routing and output against the oracle (the EP workspace holds the same routing fields)
        gl = layer.field("logits", ws=layer.ws_ep).cpu().numpy()
        ids = layer.field("topk_ids", ws=layer.ws_ep).cpu().numpy()
        w = layer.field("topk_w", ws=layer.ws_ep).cpu().numpy()
        check_routing(oracle, cfg, n, gl, ids, w)
        check_output(cfg, ids, ep, ref, toks)
        # steps 1-4 against the oracle's chain on the GPU's ids
        want = oracle_double_routing(oracle, ids, n["x"], cfg.E, W)
        for name in ("recv_start", "expert_offsets", "gathered_ids_unsort"):
            assert np.array_equal(layer.field_ep(name, W).cpu().numpy(), want[name]), f"W={W} {name}"
        assert np.array_equal(np_(layer.field_ep("x_sorted", W)), want["x_sorted"]), f"W={W} x_sorted"
        # and the single-routing layer, bit for bit
        assert torch.equal(ep, single), f"W={W}"
    del layer, d
    torch.cuda.empty_cache()
