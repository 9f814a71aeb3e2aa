"""GPU parity of each entry point against the CPU oracle, through the C ABI.

Inputs come from the seeded generators; the oracle never sees a value computed
by the CUDA path.  Integer outputs are compared bit for bit, floating-point
ones within the stated tolerance (bf16 rel-L2 <= 1e-2, fp32 rel-L2 <= 1e-5)."""
import numpy as np
import pytest
import torch

from moe_expert_routing_route_gb300 import binding, inputs
from tests._cmp import ROW_TOL, check_permutation_properties, f64, log_parity, np_, per_row_rel_l2, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build_library()
    binding.lib()


# ---- top-k routing -----------------------------------------------------------------

@pytest.mark.parametrize("T,E,k", [(1, 8, 8), (37, 16, 2), (300, 64, 6), (1000, 256, 8), (65, 160, 7),
                                   (10, 1024, 32), (33, 200, 1), (4096, 256, 8)])
@pytest.mark.parametrize("ties", [None, "quantised"])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_topk(oracle, T, E, k, ties, renorm):
    logits = inputs.random_logits(T, E, seed=T + E + k, ties=ties)
    bias = None
    if E == 256:
        bias = inputs.zipf_bias(inputs.CONFIGS["dsv3_zipf_prefill"])
    ids, w = binding.moe_route_topk(logits.to(DEV), k, renorm, None if bias is None else bias.to(DEV))
    r_ids, r_w = oracle.route_topk(logits.numpy(), k, renorm=renorm, bias=None if bias is None else bias.numpy())
    assert np.array_equal(ids.cpu().numpy(), r_ids)
    np.testing.assert_allclose(w.cpu().numpy(), r_w, rtol=1e-5, atol=1e-7)


def test_route_all_equal_scores():
    logits = inputs.random_logits(9, 32, seed=1, ties="all_equal").to(DEV)
    ids, w = binding.moe_route_topk(logits, 4, True)
    assert np.array_equal(ids.cpu().numpy(), np.tile(np.arange(4), (9, 1)))
    assert torch.all(w == 0.25)


@pytest.mark.parametrize("T,E,k,n_group,topk_group", [(1000, 256, 8, 8, 4), (300, 64, 6, 8, 3), (50, 32, 4, 4, 1),
                                                  (77, 1024, 32, 32, 8), (200, 160, 7, 5, 5), (9, 256, 8, 1, 1)])
@pytest.mark.parametrize("rule", ["max", "top2_sum"])
@pytest.mark.parametrize("ties", [None, "quantised"])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_topk_grouped(oracle, T, E, k, n_group, topk_group, rule, ties, renorm):
    logits = inputs.random_logits(T, E, seed=T + E + n_group, ties=ties)
    bias = inputs.zipf_bias(inputs.CONFIGS["dsv3_zipf_prefill"]) if E == 256 else None
    ids, w = binding.moe_route_topk_grouped(logits.to(DEV), k, n_group, topk_group, rule, renorm,
                                            None if bias is None else bias.to(DEV))
    r_ids, r_w = oracle.route_topk_grouped(logits.numpy(), k, n_group, topk_group, rule, renorm=renorm,
                                           bias=None if bias is None else bias.numpy())
    assert np.array_equal(ids.cpu().numpy(), r_ids)
    np.testing.assert_allclose(w.cpu().numpy(), r_w, rtol=1e-5, atol=1e-7)


def test_route_topk_grouped_rejects_bad_grouping():
    logits = torch.zeros((4, 24), device=DEV)
    for args in [(3, 5, 2), (3, 4, 5), (20, 4, 1), (3, 48, 1)]:  # E % n_group, topk_group > n_group, k too big, n_group > 32
        k, n_group, topk_group = args
        with pytest.raises(binding.MoEError):
            binding.moe_route_topk_grouped(logits, k, n_group, topk_group)


# ---- init-routing ------------------------------------------------------------------

@pytest.mark.parametrize("T,k,E,H,distinct", [
    (1, 1, 1, 8, True),        # a single row
    (64, 2, 16, 256, True),
    (300, 6, 64, 520, True),   # ragged: several hist chunks, H not a multiple of 64
    (4096, 8, 256, 64, True),  # 32 chunks
    (777, 3, 5, 40, False),    # repeated ids inside a token
    (200, 4, 300, 16, True),   # many empty experts
    (2500, 8, 1024, 16, True),
])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_init_routing(oracle, T, k, E, H, distinct, dtype):
    ids = inputs.random_ids(T, k, E, seed=T * 7 + E, distinct=distinct)
    x = inputs.random_rows(T, H, dtype, seed=T + 1, tag="x")
    got = binding.moe_init_routing(x.to(DEV), ids.to(DEV), E)
    assert binding.moe_check_device_status(got["ws"]) == 0
    ref = oracle.init_routing(ids.numpy(), np_(x), E)
    assert np.array_equal(got["tokens_per_expert"].cpu().numpy(), ref["tokens_per_expert"])
    assert np.array_equal(got["expert_offsets"].cpu().numpy(), ref["expert_offsets"])
    assert np.array_equal(got["expanded_row_idx"].cpu().numpy(), ref["expanded_row_idx"])
    assert np.array_equal(np_(got["expanded_x"]), ref["expanded_x"])


def test_init_routing_all_to_one_expert(oracle):
    T, k, E, H = 3000, 1, 8, 32
    ids = torch.full((T, k), 5, dtype=torch.int32)
    x = inputs.random_rows(T, H, torch.bfloat16, seed=2)
    got = binding.moe_init_routing(x.to(DEV), ids.to(DEV), E)
    ref = oracle.init_routing(ids.numpy(), np_(x), E)
    assert np.array_equal(got["expanded_row_idx"].cpu().numpy(), ref["expanded_row_idx"])
    assert np.array_equal(got["expert_offsets"].cpu().numpy(), ref["expert_offsets"])
    assert np.array_equal(np_(got["expanded_x"]), ref["expanded_x"])


def test_init_routing_flags_bad_ids():
    T, k, E, H = 50, 2, 8, 16
    ids = inputs.random_ids(T, k, E, seed=3)
    ids[4, 1] = 8
    ids[20, 0] = -3
    x = inputs.random_rows(T, H, torch.bfloat16, seed=2)
    got = binding.moe_init_routing(x.to(DEV), ids.to(DEV), E)
    assert binding.moe_check_device_status(got["ws"]) & binding.MOE_DEVERR_BAD_EXPERT_ID
    idx = got["expanded_row_idx"].cpu().numpy()
    assert idx[4 * k + 1] == -1 and idx[20 * k] == -1
    assert got["tokens_per_expert"].sum().item() == T * k - 2
    # the workspace status is cleared by the next call
    good = binding.moe_init_routing(x.to(DEV), inputs.random_ids(T, k, E, seed=3).to(DEV), E, ws=got["ws"])
    assert binding.moe_check_device_status(good["ws"]) == 0


# ---- finalize-routing --------------------------------------------------------------

@pytest.mark.parametrize("T,k,H,skip", [(1, 1, 8, False), (64, 2, 256, True), (333, 8, 7168, True),
                                        (129, 6, 2048, False), (50, 32, 40, True)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_finalize(oracle, T, k, H, skip, dtype):
    R = T * k
    y = inputs.random_rows(R, H, dtype, seed=R)
    sk = inputs.random_rows(T, H, dtype, seed=T, tag="misc") if skip else None
    w = inputs.random_scales(T, k, seed=T + k)
    idx = torch.randperm(R, generator=inputs.generator("cpu", 5, "misc")).to(torch.int32)
    out = binding.moe_finalize_routing(y.to(DEV), w.to(DEV), idx.to(DEV), None if sk is None else sk.to(DEV))
    ref = oracle.finalize_routing(np_(y), w.numpy().astype(np.float64), idx.numpy(),
                                  None if sk is None else np_(sk))
    code = 0 if dtype == torch.float32 else 1
    ref_stored = oracle.round_to(ref, code)
    got = f64(out)
    tol = 1e-5 if dtype == torch.float32 else 1e-2
    assert rel_l2(got, ref_stored) <= tol
    # fp32 accumulation (error <= (k+1) u sum|terms|) then one rounding to the
    # stored type (at most one unit in its last place)
    yv = f64(y)[idx.numpy()].reshape(T, k, H)
    mag = np.einsum("tk,tkh->th", np.abs(w.numpy().astype(np.float64)), np.abs(yv))
    if sk is not None:
        mag += np.abs(f64(sk))
    ulp = 2.0 ** -7 if dtype == torch.bfloat16 else 2.0 ** -23
    bound = ulp * np.abs(ref_stored) + (k + 1) * 2.0 ** -24 * mag * (1 + ulp) + 1e-30
    assert np.all(np.abs(got - ref_stored) <= bound)


def test_finalize_identity_reproduces_x():
    """k=1, unit weight, identity experts: the un-permuted rows are x, bit for bit."""
    T, E, k, H = 500, 16, 1, 512
    ids = inputs.random_ids(T, k, E, seed=11)
    x = inputs.random_rows(T, H, torch.bfloat16, seed=12).to(DEV)
    ir = binding.moe_init_routing(x, ids.to(DEV), E)
    out = binding.moe_finalize_routing(ir["expanded_x"], torch.ones((T, k), device=DEV), ir["expanded_row_idx"])
    assert torch.equal(out, x)


def test_finalize_flags_bad_index():
    T, k, H = 10, 2, 16
    y = inputs.random_rows(T * k, H, torch.bfloat16, seed=1).to(DEV)
    idx = torch.arange(T * k, dtype=torch.int32)
    idx[3] = T * k + 5
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    binding.moe_finalize_routing(y, torch.full((T, k), 0.5, device=DEV), idx.to(DEV), ws=ws)
    assert binding.moe_check_device_status(ws) & binding.MOE_DEVERR_BAD_ROW_INDEX


# ---- weight packing ------------------------------------------------------------------

@pytest.mark.parametrize("E,I,H", [(3, 256, 64), (2, 200, 16), (1, 1408, 32)])
def test_pack_w13_layout(E, I, H):
    wg = inputs.random_rows(E * I, H, torch.bfloat16, seed=1).view(E, I, H)
    wu = inputs.random_rows(E * I, H, torch.bfloat16, seed=2).view(E, I, H)
    packed = binding.moe_pack_w13(wg.to(DEV), wu.to(DEV)).cpu()
    Ip = -(-I // 128) * 128
    assert packed.shape == (E, 2 * Ip, H)
    for e in range(E):
        for i in [0, 1, 127, 128, I - 1] + list(range(I, Ip, 37)):
            b, r = divmod(i, 128)
            g_row, u_row = packed[e, 256 * b + r], packed[e, 256 * b + 128 + r]
            if i < I:
                assert torch.equal(g_row, wg[e, i]) and torch.equal(u_row, wu[e, i])
            else:
                assert torch.all(g_row == 0) and torch.all(u_row == 0)


@pytest.mark.parametrize("G,n,K,dtype", [(2, 300, 200, torch.bfloat16), (1, 256, 64, torch.bfloat16),
                                         (3, 512, 7168, torch.bfloat16), (2, 40, 160, torch.uint8)])
def test_tile_weights_layout(G, n, K, dtype):
    """tiled[g][t][b][r] = the 128 bytes of row 256*t + r at byte 128*b, zero past the matrix."""
    if dtype == torch.uint8:
        w = torch.randint(0, 256, (G, n, K), dtype=torch.uint8, generator=inputs.generator("cpu", 7, "misc"))
    else:
        w = inputs.random_rows(G * n, K, dtype, seed=G + n + K).view(G, n, K)
    got = binding.moe_tile_weights(w.to(DEV)).cpu().numpy()
    raw = w.view(torch.uint8).numpy().reshape(G, n, -1) if dtype != torch.uint8 else w.numpy()
    rb = raw.shape[2]
    NT, KB = -(-n // 256), -(-rb // 128)
    pad = np.zeros((G, NT * 256, KB * 128), np.uint8)
    pad[:, :n, :rb] = raw
    want = pad.reshape(G, NT, 256, KB, 128).transpose(0, 1, 3, 2, 4).reshape(-1)
    assert got.shape == want.shape and np.array_equal(got, want)


# ---- gate GEMM -------------------------------------------------------------------------

@pytest.mark.parametrize("T,H,E,dtype", [(1, 64, 8, torch.bfloat16), (300, 512, 64, torch.bfloat16),
                                         (4096, 7168, 256, torch.bfloat16), (129, 264, 40, torch.bfloat16),
                                         (200, 128, 300, torch.bfloat16), (64, 256, 16, torch.float32),
                                         (130, 72, 24, torch.float32)])
def test_gate_logits(oracle, T, H, E, dtype):
    cfg = inputs.LayerConfig("g", T=T, H=H, E=E, k=1, I=8, S=0, dtype="f32" if dtype == torch.float32 else "bf16",
                             seed=T + H)
    d = inputs.make_layer(cfg, DEV, with_weights=False)
    logits = binding.moe_gate_logits(d["x"], d["wg"])
    ref = oracle.gate_logits(np_(d["x"]), np_(d["wg"]))
    assert rel_l2(logits, ref) <= 1e-5
    # fp32 accumulation of exact bf16 products: elementwise within K*u*sum|x w|
    bound = H * 2.0 ** -24 * (np.abs(f64(d["x"])) @ np.abs(f64(d["wg"])).T) + 1e-30
    assert np.all(np.abs(f64(logits) - ref) <= bound)


# ---- grouped expert FFN ----------------------------------------------------------------------

def _close(y, ref, dtype_key: str):
    """Aggregate rel-L2 within the layer tolerance and every row within the per-row bound."""
    tol = 1e-5 if dtype_key == "f32" else 1e-2
    err = rel_l2(y, ref)
    assert err <= tol, err
    rows = per_row_rel_l2(y, ref)
    log_parity("ffn_" + dtype_key, rel_l2=err, worst_token_rel_l2=float(rows.max()), compared=len(rows))
    assert rows.max() <= ROW_TOL[dtype_key], f"row {int(rows.argmax())}: rel-L2 {rows.max():.3e}"
    return err


def _ffn_case(oracle, T, k, E, H, I, dtype, seed, ids=None, tiled=False):
    cfg = inputs.LayerConfig("f", T=T, H=H, E=E, k=k, I=I, S=0,
                             dtype="f32" if dtype == torch.float32 else "bf16", seed=seed)
    d = inputs.make_layer(cfg, "cpu")
    if ids is None:
        ids = inputs.random_ids(T, k, E, seed=seed)
    ir = oracle.init_routing(ids.numpy(), np_(d["x"]), E)
    ex = torch.from_numpy(ir["expanded_x"].view(np.int16)).view(torch.bfloat16) if dtype == torch.bfloat16 \
        else torch.from_numpy(ir["expanded_x"])
    offs = torch.from_numpy(ir["expert_offsets"])
    w13 = binding.moe_pack_w13(d["w_gate"].to(DEV), d["w_up"].to(DEV))
    w2 = d["w2"].to(DEV)
    if tiled:
        w13, w2 = binding.moe_tile_weights(w13), binding.moe_tile_weights(w2)
    y, ws = binding.moe_grouped_ffn(ex.to(DEV), offs.to(DEV), E, I, w13, w2, tiled=tiled)
    assert binding.moe_check_device_status(ws) == 0
    expert_of_row = np.repeat(np.arange(E, dtype=np.int32), ir["tokens_per_expert"])
    ref = oracle.expert_ffn_rows(ir["expanded_x"], expert_of_row, np_(d["w_gate"]), np_(d["w_up"]), np_(d["w2"]))
    return y, ref, ir


@pytest.mark.parametrize("T,k,E,H,I", [
    (300, 6, 64, 512, 256),    # ~28 rows per expert: one ragged m-tile each
    (1000, 2, 8, 512, 384),    # ~250 rows per expert: two m-tiles, ragged tail
    (150, 4, 16, 264, 200),    # K tails (H % 64, I % 64), N tail of the down GEMM, I padded to 256
    (64, 8, 256, 128, 128),    # most experts empty
    (3, 1, 4, 64, 128),        # tiny
])
def test_grouped_ffn_bf16(oracle, T, k, E, H, I):
    y, ref, _ = _ffn_case(oracle, T, k, E, H, I, torch.bfloat16, seed=T + E)
    _close(y, ref, "bf16")


def test_grouped_ffn_bf16_skewed(oracle):
    """One expert holds most rows (many m-tiles), others few or none."""
    T, k, E = 1200, 2, 16
    w = torch.tensor([40.0] + [1.0] * 7 + [0.0] * 0 + [0.5] * 8)
    ids = inputs.random_ids(T, k, E, seed=9, weights=w)
    y, ref, ir = _ffn_case(oracle, T, k, E, 256, 256, torch.bfloat16, seed=3, ids=ids)
    assert ir["tokens_per_expert"].max() > 700
    _close(y, ref, "bf16")


def test_grouped_ffn_dense_single_group(oracle):
    """expert_offsets = NULL: one group of all rows (the shared-expert call)."""
    cfg = inputs.LayerConfig("s", T=333, H=256, E=1, k=1, I=384, S=0, dtype="bf16", seed=4)
    d = inputs.make_layer(cfg, DEV)
    w13 = binding.moe_pack_w13(d["w_gate"], d["w_up"])
    y, _ = binding.moe_grouped_ffn(d["x"], None, 1, 384, w13, d["w2"])
    ref = oracle.expert_ffn_rows(np_(d["x"]), np.zeros(333, np.int32), np_(d["w_gate"]), np_(d["w_up"]),
                                 np_(d["w2"]))
    _close(y, ref, "bf16")


# Both tile shapes of the bf16 GEMM on the same cases: 128-row tiles on one SM,
# and 256-row pair tiles on a two-CTA cluster (tcgen05.mma.cta_group::2).
TILE_CASES = [
    (1000, 2, 8, 512, 384),    # ~250 rows per expert: pair tiles cut inside the peer's half
    (2000, 4, 8, 264, 200),    # ~1000 rows: several pair tiles; K tails; down N tail (264 = 256 + 8)
    (300, 6, 64, 512, 256),    # ~28 rows per expert: the peer's rows lie past the expert
    (64, 8, 256, 128, 128),    # most experts empty
    (3, 1, 4, 64, 128),        # tiny
    (2000, 8, 300, 256, 128),  # more than 256 groups: the pair kernel's 6-stage instantiation
]


@pytest.mark.parametrize("layout", ["rows", "tiled"])
@pytest.mark.parametrize("tile", ["single", "pair"])
@pytest.mark.parametrize("T,k,E,H,I", TILE_CASES)
def test_grouped_ffn_bf16_tile_shapes(oracle, monkeypatch, tile, T, k, E, H, I, layout):
    """Both tile shapes, with the weights row-major and in the tiled layout (whose boxes
    are padded with zero rows and columns past the matrix)."""
    monkeypatch.setenv("MOE_GEMM_TILE", tile)
    y, ref, _ = _ffn_case(oracle, T, k, E, H, I, torch.bfloat16, seed=T + E + 1, tiled=layout == "tiled")
    _close(y, ref, "bf16")


# Launches that take pair tiles (rows >= 256 per group on average) cover each group's 256-row
# blocks with pair tiles and a tail of at most 128 rows with a single-CTA launch.
MIXED_CASES = [
    (1600, 4, 16, 512, 256),   # ~400 rows per expert: one 256-row block, tails around 128
    (3000, 2, 16, 264, 200),   # ~375 rows: tails mostly at most 128; K tails, down N tail
    (2100, 4, 8, 256, 128),    # ~1050 rows: four blocks and short tails
]


def _mixed_ids(T, k, E, seed):
    w = torch.tensor([12.0, 6.0, 3.0] + [1.0] * (E - 3))  # some groups many blocks, some below 128 rows
    return inputs.random_ids(T, k, E, seed=seed, weights=w)


@pytest.mark.parametrize("layout", ["rows", "tiled"])
@pytest.mark.parametrize("skewed", [False, True], ids=["uniform", "skewed"])
@pytest.mark.parametrize("T,k,E,H,I", MIXED_CASES)
def test_grouped_ffn_bf16_mixed_tiles(oracle, monkeypatch, T, k, E, H, I, skewed, layout):
    """Pair tiles for the 256-row blocks plus single-CTA tiles for tails of at most 128 rows
    (MOE_GEMM_MIXED=1; the default for 128 groups or more averaging 512 rows) match the oracle and give
    the bits of pair tiles throughout (MOE_GEMM_MIXED=0)."""
    monkeypatch.delenv("MOE_GEMM_TILE", raising=False)
    monkeypatch.setenv("MOE_GEMM_MIXED", "1")
    ids = _mixed_ids(T, k, E, seed=T + 7) if skewed else None
    y, ref, ir = _ffn_case(oracle, T, k, E, H, I, torch.bfloat16, seed=T + E + 4, ids=ids, tiled=layout == "tiled")
    cnt = ir["tokens_per_expert"]
    assert cnt.sum() >= 256 * E  # the launch takes pair tiles
    assert (((cnt % 256) > 0) & ((cnt % 256) <= 128)).any()  # and some tails go to single tiles
    _close(y, ref, "bf16")
    monkeypatch.setenv("MOE_GEMM_MIXED", "0")
    y0, _, _ = _ffn_case(oracle, T, k, E, H, I, torch.bfloat16, seed=T + E + 4, ids=ids, tiled=layout == "tiled")
    assert torch.equal(y, y0)


@pytest.mark.parametrize("tile", ["single", "pair"])
def test_grouped_ffn_bf16_tile_shapes_skewed_and_dense(oracle, monkeypatch, tile):
    monkeypatch.setenv("MOE_GEMM_TILE", tile)
    T, k, E = 1500, 2, 16
    w = torch.tensor([40.0] + [1.0] * 7 + [0.5] * 8)
    ids = inputs.random_ids(T, k, E, seed=21, weights=w)
    y, ref, ir = _ffn_case(oracle, T, k, E, 256, 128, torch.bfloat16, seed=5, ids=ids)
    assert ir["tokens_per_expert"].max() > 1000
    _close(y, ref, "bf16")
    # one group of all rows, no offsets (the shared-expert call)
    cfg = inputs.LayerConfig("s", T=777, H=320, E=1, k=1, I=256, S=0, dtype="bf16", seed=6)
    d = inputs.make_layer(cfg, DEV)
    w13 = binding.moe_pack_w13(d["w_gate"], d["w_up"])
    y, ws = binding.moe_grouped_ffn(d["x"], None, 1, 256, w13, d["w2"])
    assert binding.moe_check_device_status(ws) == 0
    ref = oracle.expert_ffn_rows(np_(d["x"]), np.zeros(777, np.int32), np_(d["w_gate"]), np_(d["w_up"]),
                                 np_(d["w2"]))
    _close(y, ref, "bf16")


@pytest.mark.parametrize("T,k,E,H,I", [(64, 2, 16, 256, 128), (100, 3, 7, 72, 40)])
def test_grouped_ffn_fp32(oracle, T, k, E, H, I):
    y, ref, _ = _ffn_case(oracle, T, k, E, H, I, torch.float32, seed=T)
    _close(y, ref, "f32")


def test_grouped_ffn_flags_bad_offsets():
    E, rows, H, I = 4, 64, 64, 128
    a = torch.zeros((rows, H), dtype=torch.bfloat16, device=DEV)
    offs = torch.tensor([0, 30, 20, 64, 64], dtype=torch.int32, device=DEV)  # decreasing
    w13 = torch.zeros((E, 2 * 128, H), dtype=torch.bfloat16, device=DEV)
    w2 = torch.zeros((E, H, I), dtype=torch.bfloat16, device=DEV)
    _, ws = binding.moe_grouped_ffn(a, offs, E, I, w13, w2)
    assert binding.moe_check_device_status(ws) & binding.MOE_DEVERR_BAD_OFFSETS


# ---- failure detection: a bounded wait that runs out ------------------------------------

def test_bounded_wait_times_out_and_aborts_without_trapping():
    """An mbarrier nothing arrives on: the limited wait gives up, sets the timeout bit
    and raises the abort flag, and the unlimited waiter leaves through the flag."""
    import time
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    outcome = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.perf_counter()
    st = binding.lib().moe_diag_bounded_wait(50_000_000, binding._ptr(ws), binding._ptr(outcome), binding._stream())
    assert st == binding.MOE_OK
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert binding.moe_check_device_status(ws) == binding.MOE_DEVERR_TIMEOUT
    assert int(outcome.item()) == 3
    assert 0.04 < elapsed < 5.0
    # the context is still usable
    ids, w = binding.moe_route_topk(torch.randn(8, 16, device=DEV), 2)
    torch.cuda.synchronize()
    assert ids.shape == (8, 2)
