"""GPU parity of the whole layer (moe_layer_forward) against the CPU oracle.

The oracle computes the layer from x and the weights on its own (fp64 logits,
its own routing).  Routing decisions are compared exactly for every token whose
top-k order cannot flip under the measured logit error; for the others the
GPU's choice must be a valid top-k within that error.  Outputs are compared on
every token (small layers) or on a seeded sample of tokens (full-size layers,
in the launch configuration the benchmark times)."""
import numpy as np
import pytest
import torch

from moe_expert_routing_route_gb300 import binding, inputs
from tests._cmp import check_permutation_properties, check_topk_valid, f64, np_, rel_l2, routing_ambiguity

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build_library()
    binding.lib()


def make(cfg):
    d = inputs.make_layer(cfg, DEV)
    layer = binding.MoELayer(T=cfg.T, k=cfg.k, w_router=d["wg"], w_gate=d["w_gate"], w_up=d["w_up"], w2=d["w2"],
                             s_gate=d["s_gate"] if cfg.S else None, s_up=d["s_up"] if cfg.S else None,
                             s2=d["s2"] if cfg.S else None, expert_bias=d["bias"], renormalize=cfg.renormalize,
                             n_group=cfg.n_group, topk_group=cfg.topk_group, group_rule=cfg.group_rule)
    return d, layer


def check_layer(oracle, cfg, d, layer, out, tokens=None):
    n = {k: np_(v) for k, v in d.items() if isinstance(v, torch.Tensor)}
    bias = n.get("bias")
    k, E = cfg.k, cfg.E
    # gate logits (all tokens)
    gl = layer.field("logits").cpu().numpy()
    ref_logits = oracle.gate_logits(n["x"], n["wg"])
    assert rel_l2(gl, ref_logits) <= 1e-5
    maxerr = float(np.abs(gl.astype(np.float64) - ref_logits).max())
    # routing: exact where unambiguous, valid elsewhere
    l32 = ref_logits.astype(np.float32)
    s_ref = (l32 + bias if bias is not None else l32).astype(np.float64)
    amb = routing_ambiguity(s_ref, k, maxerr)
    ids = layer.field("topk_ids").cpu().numpy()
    w = layer.field("topk_w").cpu().numpy()
    if cfg.n_group > 1:
        r_ids, r_w = oracle.route_topk_grouped(l32, k, cfg.n_group, cfg.topk_group, cfg.group_rule,
                                               renorm=cfg.renormalize, bias=bias)
        # ambiguous: a near-tie among the best k+1 experts of the kept groups, or
        # between the last kept group and the next one (a top-2 sum carries the
        # error of two scores)
        gs = E // cfg.n_group
        srt = -np.sort(-s_ref.reshape(len(s_ref), cfg.n_group, gs), axis=2)
        gscore = srt[:, :, 0] + (srt[:, :, 1] if cfg.group_rule == "top2_sum" else 0)
        masked = s_ref.copy()
        for t in range(len(s_ref)):
            keep = np.zeros(cfg.n_group, bool)
            keep[np.unique(r_ids[t] // gs)] = True
            order = np.argsort(-gscore[t], kind="stable")[:cfg.topk_group]
            keep[order] = True
            masked[t][~np.repeat(keep, gs)] = -np.inf
        amb = routing_ambiguity(masked, k, maxerr)
        if cfg.topk_group < cfg.n_group:
            gsorted = -np.sort(-gscore, axis=1)
            amb |= gsorted[:, cfg.topk_group - 1] - gsorted[:, cfg.topk_group] <= 4 * maxerr
    else:
        r_ids, r_w = oracle.route_topk(l32, k, renorm=cfg.renormalize, bias=bias)
    assert np.array_equal(ids[~amb], r_ids[~amb])
    if cfg.n_group == 1:
        for t in np.nonzero(amb)[0]:
            check_topk_valid(ids[t], s_ref[t], maxerr)
    np.testing.assert_allclose(w[~amb], r_w[~amb], rtol=1e-4, atol=1e-6)
    # permutation: properties on the GPU's ids; bit-exact against the oracle when routing agrees
    counts = layer.field("tokens_per_expert").cpu().numpy()
    offsets = layer.field("expert_offsets").cpu().numpy()
    row_idx = layer.field("expanded_row_idx").cpu().numpy()
    ex = np_(layer.field("expanded_x"))
    check_permutation_properties(ids, E, counts, offsets, row_idx, n["x"], ex)
    if np.array_equal(ids, r_ids):
        ir = oracle.init_routing(r_ids, None, E, H=cfg.H)
        assert np.array_equal(row_idx, ir["expanded_row_idx"])
        assert np.array_equal(offsets, ir["expert_offsets"])
    # output
    toks = np.arange(cfg.T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    ref = oracle.layer(n["x"], n["wg"], n["w_gate"], n["w_up"], n["w2"], n.get("s_gate") if cfg.S else None,
                       n.get("s_up") if cfg.S else None, n.get("s2") if cfg.S else None, k=k,
                       renorm=cfg.renormalize, bias=bias, tokens=None if tokens is None else toks,
                       n_group=cfg.n_group, topk_group=cfg.topk_group, group_rule=cfg.group_rule)
    same = np.array([set(ids[t]) == set(ref["ids"][i]) for i, t in enumerate(toks)])
    assert (~same).sum() <= max(1, len(toks) // 100)
    got = f64(out)[toks][same]
    err = rel_l2(got, ref["out"][same])
    tol = 1e-5 if cfg.dtype == "f32" else 1e-2
    assert err <= tol, f"{cfg.name}: rel-L2 {err:.3e}"
    assert binding.moe_check_device_status(layer.ws) == 0
    return err


SMALL = [
    inputs.CONFIGS["tiny_fp32"],
    inputs.CONFIGS["tiny_fp32"].replace(name="tiny_fp32_norenorm", renormalize=False, seed=10),
    inputs.LayerConfig("small_bf16", T=256, H=512, E=64, k=6, I=256, S=2, dtype="bf16", seed=11),
    inputs.LayerConfig("ragged_bf16", T=97, H=264, E=24, k=5, I=200, S=1, dtype="bf16", seed=12),
    inputs.LayerConfig("no_shared_bf16", T=130, H=256, E=32, k=4, I=128, S=0, dtype="bf16", seed=13),
    inputs.LayerConfig("one_token_bf16", T=1, H=128, E=8, k=8, I=128, S=1, dtype="bf16", seed=14),
    inputs.LayerConfig("zipf_bf16", T=512, H=256, E=64, k=8, I=128, S=1, dtype="bf16", seed=15, zipf_s=1.2),
    inputs.LayerConfig("dense_E1_bf16", T=200, H=256, E=1, k=1, I=256, S=1, dtype="bf16", seed=16),
    inputs.LayerConfig("grouped_bf16", T=300, H=256, E=64, k=6, I=128, S=1, dtype="bf16", seed=17, n_group=8,
                       topk_group=3, group_rule="top2_sum"),
    inputs.LayerConfig("grouped_fp32", T=64, H=128, E=16, k=2, I=64, S=1, dtype="f32", seed=18, n_group=4,
                       topk_group=2, group_rule="max"),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
def test_layer_small(oracle, cfg):
    d, layer = make(cfg)
    out = layer.forward(d["x"])
    check_layer(oracle, cfg, d, layer, out)


PAIR = [c for c in SMALL if c.dtype == "bf16" and c.name in ("small_bf16", "ragged_bf16", "zipf_bf16",
                                                                 "grouped_bf16", "dense_E1_bf16")]


@pytest.mark.parametrize("cfg", PAIR, ids=[c.name for c in PAIR])
def test_layer_small_pair_tiles(oracle, monkeypatch, cfg):
    """The whole layer with every bf16 expert GEMM on 256-row pair tiles."""
    monkeypatch.setenv("MOE_GEMM_TILE", "pair")
    d, layer = make(cfg)
    out = layer.forward(d["x"])
    check_layer(oracle, cfg, d, layer, out)


# H sweeps the gate GEMM's k-block count (1 .. 17, with K tails) and T its tile
# count, so the K-split plan takes several slice counts, each slice non-empty.
GATE_SPLIT = [(T, H) for T in (40, 700) for H in (24, 136, 264, 328, 584, 1096)]


@pytest.mark.parametrize("T,H", GATE_SPLIT, ids=[f"T{T}_H{H}" for T, H in GATE_SPLIT])
def test_layer_gate_split_k(oracle, T, H):
    cfg = inputs.LayerConfig(f"gate_{T}_{H}", T=T, H=H, E=40, k=3, I=64, S=0, dtype="bf16", seed=T + H)
    d, layer = make(cfg)
    gl = None
    for _ in range(2):  # the logits region holds stale slices from the first call
        layer.forward(d["x"])
        got = layer.field("logits").cpu().numpy().copy()
        if gl is not None:
            assert np.array_equal(got, gl)
        gl = got
    assert rel_l2(gl, oracle.gate_logits(np_(d["x"]), np_(d["wg"]))) <= 1e-5
    assert binding.moe_check_device_status(layer.ws) == 0


FULL = [("mid_bf16", 96), ("dsv3_prefill", 48), ("dsv3_decode", 32), ("dsv3_zipf_prefill", 32),
        ("dsv3_prefill_grouped", 32)]


@pytest.mark.parametrize("name,n_sample", FULL, ids=[f[0] for f in FULL])
def test_layer_full_size_sampled(oracle, name, n_sample):
    cfg = inputs.CONFIGS[name]
    d, layer = make(cfg)
    out = layer.forward(d["x"])
    g = inputs.generator("cpu", cfg.seed, "misc")
    toks = torch.randperm(cfg.T, generator=g)[:n_sample].sort().values.numpy().astype(np.int32)
    if cfg.zipf_s:
        counts = layer.field("tokens_per_expert").cpu().numpy()
        assert counts.max() > 8 * counts.mean()  # the skew is really there
    check_layer(oracle, cfg, d, layer, out, tokens=toks)
    del layer, d
    torch.cuda.empty_cache()


def test_layer_deterministic_and_graph_capturable(oracle):
    cfg = inputs.LayerConfig("graph_bf16", T=384, H=512, E=64, k=6, I=256, S=1, dtype="bf16", seed=21)
    d, layer = make(cfg)
    x = d["x"]
    out1 = layer.forward(x)
    out2 = layer.forward(x)
    assert torch.equal(out1, out2)
    static_out = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x, out=static_out, stream=s)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x, out=static_out)
    static_out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(static_out, out1)
    # new input through the same graph
    x.copy_(inputs.random_rows(cfg.T, cfg.H, torch.bfloat16, seed=99, tag="x").to(DEV))
    graph.replay()
    torch.cuda.synchronize()
    check_layer(oracle, cfg, d, layer, static_out)


HOST = [
    inputs.LayerConfig("host_bf16", T=256, H=256, E=32, k=4, I=128, S=1, dtype="bf16", seed=22),  # one chunk
    # x and out move in 3 uneven row chunks; the shared experts run chunk by chunk
    inputs.LayerConfig("host_bf16_chunks", T=3001, H=512, E=64, k=6, I=256, S=2, dtype="bf16", seed=24),
    inputs.LayerConfig("host_bf16_noshared", T=2100, H=256, E=16, k=2, I=128, S=0, dtype="bf16", seed=25),
    inputs.LayerConfig("host_fp32_chunks", T=1500, H=128, E=16, k=2, I=64, S=1, dtype="f32", seed=26),
    inputs.LayerConfig("host_fp8_chunks", T=2048, H=512, E=32, k=4, I=256, S=1, dtype="bf16", seed=27,
                       weight_format="fp8"),
]


@pytest.mark.parametrize("cfg", HOST, ids=[c.name for c in HOST])
def test_layer_forward_host_matches_device(cfg):
    """The host-buffer entry point (chunked copies overlapping the shared experts and
    the finalize kernel) gives the device-buffer result bit for bit."""
    d = inputs.make_layer(cfg, DEV)
    layer = binding.MoELayer(T=cfg.T, k=cfg.k, w_router=d["wg"], w_gate=d["w_gate"], w_up=d["w_up"], w2=d["w2"],
                             s_gate=d["s_gate"] if cfg.S else None, s_up=d["s_up"] if cfg.S else None,
                             s2=d["s2"] if cfg.S else None, expert_bias=d["bias"], renormalize=cfg.renormalize,
                             weight_format=cfg.weight_format)
    dev_out = layer.forward(d["x"]).cpu()
    x_host = d["x"].cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    for _ in range(2):  # the second call reuses the buffers the first one filled
        out_host.zero_()
        layer.forward_host(x_host, out_host)
        assert layer.device_status() == 0
        assert torch.equal(out_host, dev_out)


def test_layer_stage_events():
    cfg = inputs.LayerConfig("ev_bf16", T=256, H=256, E=32, k=4, I=128, S=1, dtype="bf16", seed=23)
    d, layer = make(cfg)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * binding.MOE_NUM_STAGES)]
    out = layer.forward(d["x"], events=evs)
    torch.cuda.synchronize()
    times = [evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(binding.MOE_NUM_STAGES)]
    assert all(t >= 0 for t in times)
    names = binding.stage_names()
    # the shared experts overlap routing: they start after the gate and end before "up"
    sh, up, gate = names.index("shared"), names.index("up"), names.index("gate")
    assert evs[2 * gate + 1].elapsed_time(evs[2 * sh]) >= 0
    assert evs[2 * sh + 1].elapsed_time(evs[2 * up]) >= 0
    assert torch.equal(out, layer.forward(d["x"]))
