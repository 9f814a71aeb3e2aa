"""GPU parity of the FP8 (e4m3, block-scaled) path against the CPU oracle, through
the C ABI: quantisers bit for bit, the FP8 grouped FFN and the FP8-weight layer
within the bf16 tolerance of the oracle's FP8 definition -- with fp32 block
scales (promotion on CUDA cores) and with power-of-two block scales (applied by
the tensor cores' block-scaled MMA)."""
import numpy as np
import pytest
import torch

from moe_expert_routing_route_gb300 import binding, inputs
from tests._cmp import ROW_TOL, log_parity, np_, per_row_rel_l2, rel_l2
from tests._layer_check import check_output, check_routing, host_arrays

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build_library()
    binding.lib()


@pytest.mark.parametrize("pow2", [False, True], ids=["f32scale", "pow2scale"])
@pytest.mark.parametrize("rows,cols,dtype", [(1, 128, torch.bfloat16), (37, 7168, torch.bfloat16),
                                             (100, 300, torch.float32), (5, 2048, torch.bfloat16),
                                             (64, 40, torch.float32)])
def test_quantize_rows_fp8(oracle, rows, cols, dtype, pow2):
    a = inputs.random_rows(rows, cols, dtype, seed=rows + cols) * 3
    a[0, :5] = 0  # zeros and a partly zero block
    if rows > 2 and dtype == torch.float32:
        a[1] *= 1e-30  # scales near the bottom of the exponent range
        a[2] *= 1e20
    codes, scales = binding.moe_quantize_rows_fp8(a.to(DEV), pow2=pow2)
    rc, rs = oracle.quantize_rows_fp8(np_(a), pow2=pow2)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)


def _boundary_rows(oracle, pow2: bool, rows: int, cols: int, seed: int) -> np.ndarray:
    """fp32 rows whose values, divided by their block's scale, land on or within four fp32 ulps of
    the e4m3 rounding midpoints (between adjacent codes, subnormal ones and the one next to zero
    included).  Each 128-value block starts with its amax A, drawn over 48 decades (the smallest
    below the range where the kernels divide each value); the other values are fl32(M * s) moved
    by -4..4 ulps for random midpoints M, where s is A / 448 in fp32 (or the power of two above
    it), and kept at or below A so that A stays the block's amax."""
    rng = np.random.default_rng(seed)
    vals = np.unique(np.abs(oracle.e4m3_table()[np.isfinite(oracle.e4m3_table())]))  # 0 .. 448
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    a = np.empty((rows, cols), np.float32)
    for r in range(rows):
        for b0 in range(0, cols, 128):
            A = np.float32(10.0 ** rng.uniform(-28, 20))
            s = np.float32(2.0 ** np.ceil(np.log2(float(A) / 448.0))) if pow2 else A / np.float32(448)
            n = min(128, cols - b0)
            m = rng.choice(mids, size=n - 1)
            v = (m * s).astype(np.float32)
            bits = v.view(np.int32) + rng.integers(-4, 5, size=n - 1).astype(np.int32)
            v = np.minimum(bits.view(np.float32), A)
            a[r, b0] = A
            a[r, b0 + 1:b0 + n] = np.where(rng.random(n - 1) < 0.5, -v, v)
    return a


@pytest.mark.parametrize("pow2", [False, True], ids=["f32scale", "pow2scale"])
def test_quantize_rows_fp8_rounding_midpoints(oracle, pow2):
    """The kernels take fl32(v / s) with one division per block (a reciprocal and two fma
    correction steps); on values whose quotients sit at the e4m3 rounding midpoints every code
    must still equal the oracle's, which divides each value."""
    a = _boundary_rows(oracle, pow2, rows=96, cols=1000, seed=11 + pow2)
    codes, scales = binding.moe_quantize_rows_fp8(torch.from_numpy(a).to(DEV), pow2=pow2)
    rc, rs = oracle.quantize_rows_fp8(a, pow2=pow2)
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quantize_rows_fp8_all_zero_block(oracle):
    a = torch.zeros((2, 256), dtype=torch.bfloat16)
    a[1, 200] = 1.5
    codes, scales = binding.moe_quantize_rows_fp8(a.to(DEV))
    want = np.array([[1.0, 1.0], [1.0, np.float32(1.5) / np.float32(448)]], np.float32)
    assert np.array_equal(scales.cpu().numpy(), want)
    assert np.array_equal(codes.cpu().numpy(), oracle.quantize_rows_fp8(np_(a))[0])


@pytest.mark.parametrize("pow2", [False, True], ids=["f32scale", "pow2scale"])
@pytest.mark.parametrize("G,n,k", [(2, 256, 512), (1, 200, 300), (3, 384, 7168)])
def test_quantize_weights_fp8(oracle, G, n, k, pow2):
    w = inputs.random_rows(G * n, k, torch.bfloat16, seed=G * n + k).view(G, n, k)
    codes, scales = binding.moe_quantize_weights_fp8(w.to(DEV), pow2=pow2)
    for g in range(G):
        rc, rs = oracle.quantize_tiles_fp8(np_(w[g]), pow2=pow2)
        assert np.array_equal(codes[g].cpu().numpy(), rc)
        assert np.array_equal(scales[g].cpu().numpy(), rs)


def _oracle_fp8_weights(oracle, n: dict, shared: bool = True, pow2: bool = False):
    q = {}
    parts = [("", "w_gate", "w_up", "w2")] + ([("s", "s_gate", "s_up", "s2")] if shared else [])
    for pre, g, u, d in parts:
        q[pre + "gq"], q[pre + "gs"] = oracle.quantize_experts_fp8(n[g], pow2)
        q[pre + "uq"], q[pre + "us"] = oracle.quantize_experts_fp8(n[u], pow2)
        q[pre + "dq"], q[pre + "ds"] = oracle.quantize_experts_fp8(n[d], pow2)
    return q


@pytest.mark.parametrize("pow2", [False, True], ids=["f32scale", "pow2scale"])
@pytest.mark.parametrize("T,k,E,H,I", [(300, 6, 16, 512, 256), (1000, 2, 8, 256, 384), (64, 8, 64, 256, 128),
                                       (3, 1, 4, 256, 128), (120, 4, 8, 512, 208), (200, 4, 8, 2304, 256)])
def test_grouped_ffn_fp8(oracle, T, k, E, H, I, pow2):
    """I=208: a K tail of 80 in the down projection and padded gate/up packing.  H=2304:
    18 K blocks in the up projection, so with power-of-two scales a tile spans two
    scale-factor groups (16 + 2 blocks)."""
    cfg = inputs.LayerConfig("f", T=T, H=H, E=E, k=k, I=I, S=0, dtype="bf16", seed=T + E)
    d = inputs.make_layer(cfg, "cpu")
    n = {key: np_(v) for key, v in d.items() if isinstance(v, torch.Tensor)}
    ids = inputs.random_ids(T, k, E, seed=T)
    ir = oracle.init_routing(ids.numpy(), n["x"], E)
    xq, xs = oracle.quantize_rows_fp8(ir["expanded_x"], pow2=pow2)
    q = _oracle_fp8_weights(oracle, n, shared=False, pow2=pow2)
    # the GPU quantises the packed gate/up weight; its codes are the oracle's, re-packed
    w13 = binding.moe_pack_w13(d["w_gate"].to(DEV), d["w_up"].to(DEV))
    w13q, w13s = binding.moe_quantize_weights_fp8(w13, pow2=pow2)
    w2q, w2s = binding.moe_quantize_weights_fp8(d["w2"].to(DEV), pow2=pow2)
    if I % 128 == 0:
        e0 = w13q[0].cpu().numpy()
        assert np.array_equal(e0[0:128], q["gq"][0][0:128]) and np.array_equal(e0[128:256], q["uq"][0][0:128])
    y, ws = binding.moe_grouped_ffn_fp8(torch.from_numpy(xq).to(DEV), torch.from_numpy(xs).to(DEV),
                                        torch.from_numpy(ir["expert_offsets"]).to(DEV), E, I, w13q, w13s, w2q, w2s,
                                        pow2=pow2)
    assert binding.moe_check_device_status(ws) == 0
    expert_of_row = np.repeat(np.arange(E, dtype=np.int32), ir["tokens_per_expert"])
    ref = oracle.expert_ffn_rows_fp8(xq, xs, expert_of_row, q, pow2=pow2)
    assert rel_l2(y, ref) <= 1e-2
    rows_err = per_row_rel_l2(y, ref)
    log_parity("ffn_fp8" + ("_pow2" if pow2 else ""), rel_l2=rel_l2(y, ref), worst_token_rel_l2=float(rows_err.max()),
               compared=len(rows_err))
    assert rows_err.max() <= ROW_TOL["bf16"]
    # The up GEMM's epilogue quantises h itself; its codes and scales are those the
    # 1x128 quantiser gives for the bf16 h stored beside them.  Workspace of this
    # entry point: 256-byte header, h [rows, I] bf16, codes [rows, I], scales
    # [rows, scale_ld(I)], each region 256-byte aligned.
    rows, ld = T * k, binding.scale_ld(I)
    up = lambda b: -(-b // 256) * 256  # noqa: E731
    h = ws[256:256 + rows * I * 2].view(torch.bfloat16).view(rows, I)
    o = 256 + up(rows * I * 2)
    hq = ws[o:o + rows * I].view(rows, I)
    o += up(rows * I)
    hs = ws[o:o + rows * ld * 4].view(torch.float32).view(rows, ld)
    rq, rs = binding.moe_quantize_rows_fp8(h, ld_scales=ld, pow2=pow2)
    nb = -(-I // 128)
    assert torch.equal(hq, rq) and torch.equal(hs[:, :nb], rs[:, :nb])
    # and both are the oracle's quantisation of that h
    oq, os_ = oracle.quantize_rows_fp8(np_(h), pow2=pow2)
    assert np.array_equal(hq.cpu().numpy(), oq) and np.array_equal(hs[:, :nb].cpu().numpy(), os_)


FP8_LAYERS = [
    inputs.LayerConfig("fp8_small", T=256, H=512, E=64, k=6, I=256, S=2, dtype="bf16", seed=51,
                       weight_format="fp8"),
    inputs.LayerConfig("fp8_grouped", T=200, H=256, E=32, k=4, I=128, S=1, dtype="bf16", seed=52, n_group=4,
                       topk_group=2, group_rule="top2_sum", weight_format="fp8"),
    inputs.LayerConfig("fp8_noshared", T=130, H=256, E=16, k=2, I=384, S=0, dtype="bf16", seed=53,
                       weight_format="fp8"),
    inputs.LayerConfig("fp8_pow2_small", T=256, H=512, E=64, k=6, I=256, S=2, dtype="bf16", seed=54,
                       weight_format="fp8_pow2"),
    inputs.LayerConfig("fp8_pow2_grouped", T=200, H=2304, E=32, k=4, I=128, S=1, dtype="bf16", seed=55, n_group=4,
                       topk_group=2, group_rule="top2_sum", weight_format="fp8_pow2"),
    inputs.LayerConfig("fp8_pow2_noshared_zipf", T=300, H=256, E=16, k=2, I=384, S=0, dtype="bf16", seed=56,
                       zipf_s=1.2, weight_format="fp8_pow2"),
]


def _check_fp8_layer(oracle, cfg, d, layer, out, tokens=None):
    """Routing as in the bf16 layer (the gate stays bf16), then the output against
    the oracle's FP8 layer, in aggregate and token by token."""
    n = host_arrays(d)
    check_routing(oracle, cfg, n, layer.field("logits").cpu().numpy(), layer.field("topk_ids").cpu().numpy(),
                  layer.field("topk_w").cpu().numpy())
    pow2 = cfg.weight_format == "fp8_pow2"
    q = _oracle_fp8_weights(oracle, n, shared=cfg.S > 0, pow2=pow2)
    toks = np.arange(cfg.T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    ref = oracle.layer_fp8(n["x"], n["wg"], q, k=cfg.k, renorm=cfg.renormalize, bias=n.get("bias"),
                           tokens=None if tokens is None else toks, n_group=cfg.n_group, topk_group=cfg.topk_group,
                           group_rule=cfg.group_rule, pow2=pow2)
    res = check_output(cfg, layer.field("topk_ids").cpu().numpy(), out, ref, toks)
    assert binding.moe_check_device_status(layer.ws) == 0
    return res


def _make(cfg, layout=None):
    d = inputs.make_layer(cfg, DEV)
    layer = binding.MoELayer(T=cfg.T, k=cfg.k, w_router=d["wg"], w_gate=d["w_gate"], w_up=d["w_up"], w2=d["w2"],
                             s_gate=d["s_gate"] if cfg.S else None, s_up=d["s_up"] if cfg.S else None,
                             s2=d["s2"] if cfg.S else None, expert_bias=d["bias"], renormalize=cfg.renormalize,
                             n_group=cfg.n_group, topk_group=cfg.topk_group, group_rule=cfg.group_rule,
                             weight_format=cfg.weight_format, weight_layout=layout)
    return d, layer


@pytest.mark.parametrize("layout", ["tiled", "rows"])
@pytest.mark.parametrize("cfg", FP8_LAYERS, ids=[c.name for c in FP8_LAYERS])
def test_layer_fp8_small(oracle, cfg, layout):
    """FP8 layers with the expert codes in the tiled layout (the default) and row-major."""
    d, layer = _make(cfg, layout)
    out = layer.forward(d["x"])
    _check_fp8_layer(oracle, cfg, d, layer, out)
    # deterministic: a second forward gives the same bits
    assert torch.equal(layer.forward(d["x"]), out)


@pytest.mark.parametrize("name,n_sample", [("dsv3_prefill_fp8", 32), ("dsv3_decode_fp8", 16),
                                           ("dsv3_prefill_fp8_pow2", 32), ("dsv3_decode_fp8_pow2", 16)])
def test_layer_fp8_full_size_sampled(oracle, name, n_sample):
    cfg = inputs.CONFIGS[name]
    d, layer = _make(cfg)
    out = layer.forward(d["x"])
    g = inputs.generator("cpu", cfg.seed, "misc")
    toks = torch.randperm(cfg.T, generator=g)[:n_sample].sort().values.numpy().astype(np.int32)
    _check_fp8_layer(oracle, cfg, d, layer, out, tokens=toks)
    del layer, d
    torch.cuda.empty_cache()


def test_grouped_ffn_fp8_rejects_unsupported_shapes():
    a = torch.zeros((8, 512), dtype=torch.uint8, device=DEV)
    sc = torch.ones((8, 4), dtype=torch.float32, device=DEV)
    with pytest.raises(binding.MoEError):  # I % 16 != 0
        binding.moe_grouped_ffn_fp8(a, sc, None, 1, 200, a, sc, a, sc)
