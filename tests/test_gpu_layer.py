"""GPU parity of the whole layer (moe_layer_forward) against the CPU oracle.

The oracle computes the layer from x and the weights on its own (fp64 logits,
its own routing).  Routing decisions are compared exactly for every token whose
top-k order cannot flip under the measured logit error; for the others the
GPU's choice must be a valid (group-limited) top-k within that error.  Outputs
are compared on every token (small layers and the full-K prefill slice) or on a
seeded sample of tokens (full-size layers, in the launch configuration the
benchmark times), in aggregate and token by token."""
import numpy as np
import pytest
import torch

from moe_expert_routing_route_gb300 import binding, inputs
from tests._cmp import np_, rel_l2
from tests._layer_check import check_layer, host_arrays, oracle_layer

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


ROWS = [c for c in SMALL if c.dtype == "bf16" and c.name in ("small_bf16", "ragged_bf16", "one_token_bf16")]


@pytest.mark.parametrize("tile", ["single", "pair"])
@pytest.mark.parametrize("cfg", ROWS, ids=[c.name for c in ROWS])
def test_layer_small_row_major_weights(oracle, monkeypatch, cfg, tile):
    """bf16 layers take tiled weights by default; the row-major layout stays supported."""
    monkeypatch.setenv("MOE_GEMM_TILE", tile)
    d = inputs.make_layer(cfg, DEV)
    layer = binding.MoELayer(T=cfg.T, k=cfg.k, w_router=d["wg"], w_gate=d["w_gate"], w_up=d["w_up"], w2=d["w2"],
                             s_gate=d["s_gate"] if cfg.S else None, s_up=d["s_up"] if cfg.S else None,
                             s2=d["s2"] if cfg.S else None, expert_bias=d["bias"], renormalize=cfg.renormalize,
                             weight_layout="rows")
    out = layer.forward(d["x"])
    check_layer(oracle, cfg, d, layer, out)
    tiled = make(cfg)[1]
    assert torch.equal(tiled.forward(d["x"]), out)  # the same products, whichever layout


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
    # the host-buffer entry point at full size (x and out in 1024-row chunks or more, the shared
    # experts chunk by chunk as x arrives) gives the device-buffer output bit for bit
    x_host = d["x"].cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    layer.forward_host(x_host, out_host)
    assert layer.device_status() == 0
    assert torch.equal(out_host, out.cpu())
    del layer, d
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def prefill_slice(oracle):
    """The DeepSeek-V3 prefill layer's full K dimensions (H=7168, I=2048, ~128 rows
    per expert) on 32 experts, with the oracle's output for every token."""
    cfg = inputs.CONFIGS["dsv3_prefill_slice"]
    d = inputs.make_layer(cfg, DEV)
    n = host_arrays(d)
    ref = oracle_layer(oracle, cfg, n, None)
    yield cfg, d, n, ref
    del d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("tile", ["auto", "single", "pair"])
def test_layer_prefill_slice_every_token(oracle, monkeypatch, prefill_slice, tile):
    """Every token of a full-K layer against the oracle, under each GEMM tile policy."""
    cfg, d, n, ref = prefill_slice
    if tile != "auto":
        monkeypatch.setenv("MOE_GEMM_TILE", tile)
    layer = binding.MoELayer(T=cfg.T, k=cfg.k, w_router=d["wg"], w_gate=d["w_gate"], w_up=d["w_up"], w2=d["w2"],
                             s_gate=d["s_gate"], s_up=d["s_up"], s2=d["s2"], expert_bias=None,
                             renormalize=cfg.renormalize)
    out = layer.forward(d["x"])
    res = check_layer(oracle, cfg, d, layer, out, n=n, ref=ref)
    assert res["compared"] >= cfg.T - max(1, cfg.T // 100)


def test_layer_prefill_slice_shared_experts_beside_up(oracle, monkeypatch, prefill_slice):
    """Full-K experts, 128 rows per expert: the shared experts on 22 SMs beside the routed
    up projection give the bits of running them first on every SM (the default)."""
    cfg, d, n, ref = prefill_slice
    layer = binding.MoELayer(T=cfg.T, k=cfg.k, w_router=d["wg"], w_gate=d["w_gate"], w_up=d["w_up"], w2=d["w2"],
                             s_gate=d["s_gate"], s_up=d["s_up"], s2=d["s2"], expert_bias=None,
                             renormalize=cfg.renormalize)
    assert layer.shared_expert_sms() == 0
    whole = layer.forward(d["x"])
    monkeypatch.setenv("MOE_SHARED_SMS", "22")
    assert layer.shared_expert_sms() == 22
    split = layer.forward(d["x"])
    assert torch.equal(split, whole)
    check_layer(oracle, cfg, d, layer, split, n=n, ref=ref)


def test_layer_mixed_tiles_zipf(oracle, monkeypatch):
    """A Zipf-skewed layer (1024 rows per expert on average) with pair tiles for each expert's
    256-row blocks and single-CTA tiles for tails of at most 128 rows (MOE_GEMM_MIXED=1, hot and
    cold experts alike): the bits of pair tiles throughout, and the oracle's output."""
    cfg = inputs.LayerConfig("zipf_mixed_bf16", T=2048, H=256, E=16, k=8, I=128, S=1, dtype="bf16", seed=17,
                             zipf_s=1.2)
    monkeypatch.delenv("MOE_GEMM_TILE", raising=False)
    monkeypatch.setenv("MOE_GEMM_MIXED", "1")
    d, layer = make(cfg)
    mixed = layer.forward(d["x"]).clone()
    cnt = layer.field("tokens_per_expert").cpu().numpy()
    assert (((cnt % 256) > 0) & ((cnt % 256) <= 128)).any()
    monkeypatch.setenv("MOE_GEMM_MIXED", "0")
    assert torch.equal(layer.forward(d["x"]), mixed)
    check_layer(oracle, cfg, d, layer, mixed)


FUSED = [c for c in SMALL if c.dtype == "bf16" and c.S > 0 and c.T >= 256]


@pytest.mark.parametrize("cfg", FUSED, ids=[c.name for c in FUSED])
def test_layer_shared_experts_one_launch(oracle, monkeypatch, cfg):
    """The shared experts' up and down projections in one pair-tile launch (the down
    projection's tiles waiting on per-256-row counters) give the bits of two launches."""
    d, layer = make(cfg)
    fused = layer.forward(d["x"])
    assert layer.device_status() == 0
    monkeypatch.setenv("MOE_SHARED_FUSED", "0")
    assert torch.equal(layer.forward(d["x"]), fused)
    check_layer(oracle, cfg, d, layer, fused)


def test_layer_prefill_slice_shared_experts_one_launch(oracle, monkeypatch, prefill_slice):
    """Full-K shared experts (H=7168, I=2048, 512 rows: two m-tiles) in one launch: the
    same bits as two launches, in the same repeated forward."""
    cfg, d, n, ref = prefill_slice
    layer = binding.MoELayer(T=cfg.T, k=cfg.k, w_router=d["wg"], w_gate=d["w_gate"], w_up=d["w_up"], w2=d["w2"],
                             s_gate=d["s_gate"], s_up=d["s_up"], s2=d["s2"], expert_bias=None,
                             renormalize=cfg.renormalize)
    fused = [layer.forward(d["x"]) for _ in range(3)]
    assert layer.device_status() == 0
    assert all(torch.equal(f, fused[0]) for f in fused)
    monkeypatch.setenv("MOE_SHARED_FUSED", "0")
    assert torch.equal(layer.forward(d["x"]), fused[0])
    check_layer(oracle, cfg, d, layer, fused[0], n=n, ref=ref)


SPLIT = [c for c in SMALL if c.dtype == "bf16" and c.S > 0 and c.name in ("small_bf16", "ragged_bf16", "zipf_bf16",
                                                                           "one_token_bf16", "grouped_bf16")]


@pytest.mark.parametrize("cfg", SPLIT, ids=[c.name for c in SPLIT])
def test_layer_shared_experts_on_a_share_of_the_sms(oracle, monkeypatch, cfg):
    """Forcing the split (four SMs for the shared experts, the routed down projection
    joining them) gives the bits of the unsplit layer, and the oracle's results."""
    d, layer = make(cfg)
    monkeypatch.setenv("MOE_SHARED_SMS", "0")
    assert layer.shared_expert_sms() == 0
    whole = layer.forward(d["x"])
    monkeypatch.setenv("MOE_SHARED_SMS", "3")  # rounded up to two pairs
    assert layer.shared_expert_sms() == 4
    split = layer.forward(d["x"])
    assert torch.equal(split, whole)
    check_layer(oracle, cfg, d, layer, split)


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


def test_layer_split_shared_experts_graph_capturable(oracle, monkeypatch):
    """The split schedule (fork before the gate, join before the routed down projection)
    captured into a CUDA graph replays the eager bits."""
    monkeypatch.setenv("MOE_SHARED_SMS", "4")
    cfg = inputs.LayerConfig("graph_split_bf16", T=384, H=512, E=64, k=6, I=256, S=1, dtype="bf16", seed=29)
    d, layer = make(cfg)
    assert layer.shared_expert_sms() == 4
    x = d["x"]
    eager = layer.forward(x)
    static_out = torch.empty_like(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x, out=static_out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(x, out=static_out)
    static_out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(static_out, eager)
    check_layer(oracle, cfg, d, layer, eager)
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
    inputs.LayerConfig("host_fp8_pow2_chunks", T=2048, H=512, E=32, k=4, I=256, S=1, dtype="bf16", seed=28,
                       weight_format="fp8_pow2"),
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
    # the shared experts overlap the gate and routing: they start once the gate has
    # started and end before "up"
    sh, up, gate = names.index("shared"), names.index("up"), names.index("gate")
    assert evs[2 * gate].elapsed_time(evs[2 * sh]) >= 0
    assert evs[2 * sh + 1].elapsed_time(evs[2 * up]) >= 0
    assert torch.equal(out, layer.forward(d["x"]))
    # events for some stages only (the benchmark's timed region): the others are skipped
    dn = names.index("down")
    part = [e if i // 2 in (up, dn) else None for i, e in enumerate(evs)]
    assert torch.equal(layer.forward(d["x"], events=part), out)
    torch.cuda.synchronize()
    assert part[2 * up].elapsed_time(part[2 * up + 1]) >= 0
    assert part[2 * up + 1].elapsed_time(part[2 * dn]) >= 0
