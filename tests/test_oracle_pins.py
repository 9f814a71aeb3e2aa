"""Pins of the CPU oracle against things other than itself (CPU only).

Each test checks one oracle function against a closed form, an invariant, a
library routine on a special case, or brute force on tiny inputs, chosen so that
a plausible slip (a dropped term, a wrong sign or index, a transposed operand,
gate and up swapped, an unstable sort) fails at least one of them.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from moe_expert_routing_route_gb300 import inputs

F32, BF16 = 0, 1


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    return inputs.to_numpy(torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16))


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


# ---- storage rounding --------------------------------------------------------

def test_round_to_bf16_matches_torch_cast(oracle):
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(4000).astype(np.float32),
                        # exact ties between two bf16 neighbours: 1 + 2^-8 and 1 + 3*2^-8
                        np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 0.0, -0.0], np.float32)])
    got = oracle.round_to(v.astype(np.float64), BF16)
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, want)
    # ties go to even: 1 + 2^-8 -> 1.0, 1 + 3*2^-8 -> 1 + 2^-6 (upper neighbour is even)
    assert got[-5] == 1.0 and got[-4] == 1 + 2**-6


def test_round_to_f32_matches_numpy(oracle):
    v = np.random.default_rng(1).standard_normal(1000)
    assert np.array_equal(oracle.round_to(v, F32), v.astype(np.float32).astype(np.float64))


# ---- gate GEMM ---------------------------------------------------------------

@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_gate_logits_equals_library_matmul(oracle, dt):
    cfg = inputs.LayerConfig("t", T=37, H=96, E=24, k=2, I=8, S=0, dtype=dt, seed=5)
    d = inputs.make_layer(cfg, with_weights=False)
    x, wg = inputs.to_numpy(d["x"]), inputs.to_numpy(d["wg"])
    got = oracle.gate_logits(x, wg)
    want = d["x"].to(torch.float64).numpy() @ d["wg"].to(torch.float64).numpy().T  # [T,H]x[H,E]
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


# ---- top-k routing -------------------------------------------------------------

def _brute_topk(s: np.ndarray, k: int):
    """Full sort of the experts by (-score, id), truncated to k."""
    return [sorted(range(s.size), key=lambda e: (-float(s[e]), e))[:k] for _ in [0]][0]


@pytest.mark.parametrize("ties", [None, "quantised"])
@pytest.mark.parametrize("use_bias", [False, True])
def test_topk_ids_equal_brute_force_sort(oracle, ties, use_bias):
    T, E, k = 60, 16, 4
    logits = inputs.random_logits(T, E, seed=3, ties=ties).numpy()
    bias = (np.round(np.random.default_rng(2).standard_normal(E) * 4) / 4).astype(np.float32) \
        if use_bias else None
    ids, w = oracle.route_topk(logits, k, renorm=True, bias=bias)
    for t in range(T):
        s = logits[t] + (bias if bias is not None else 0)  # fp32 + fp32 -> fp32
        assert s.dtype == np.float32
        assert list(ids[t]) == _brute_topk(s, k)


def test_topk_weights_are_library_softmax(oracle):
    T, E, k = 40, 32, 6
    logits = inputs.random_logits(T, E, seed=4).numpy()
    ids, w = oracle.route_topk(logits, k, renorm=True)
    _, w_raw = oracle.route_topk(logits, k, renorm=False)
    for t in range(T):
        sel = logits[t][ids[t]].astype(np.float64)
        np.testing.assert_allclose(w[t], scipy.special.softmax(sel), rtol=1e-13)
        full = scipy.special.softmax(logits[t].astype(np.float64))
        np.testing.assert_allclose(w_raw[t], full[ids[t]], rtol=1e-13)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)
    # descending slots: weights are non-increasing along j
    assert np.all(np.diff(w, axis=1) <= 0)


def test_topk_all_equal_scores(oracle):
    T, E, k = 5, 12, 3
    logits = inputs.random_logits(T, E, seed=0, ties="all_equal").numpy()
    ids, w = oracle.route_topk(logits, k, renorm=True)
    assert np.array_equal(ids, np.tile(np.arange(k, dtype=np.int32), (T, 1)))
    assert np.all(w == 1.0 / k)
    _, w_raw = oracle.route_topk(logits, k, renorm=False)
    np.testing.assert_allclose(w_raw, 1.0 / E, rtol=1e-15)


def test_topk_k_equals_E_is_full_softmax(oracle):
    T, E = 7, 8
    logits = inputs.random_logits(T, E, seed=9).numpy()
    ids, w = oracle.route_topk(logits, E, renorm=True)
    for t in range(T):
        assert sorted(ids[t]) == list(range(E))
        np.testing.assert_allclose(w[t], scipy.special.softmax(logits[t].astype(np.float64))[ids[t]],
                                   rtol=1e-13)


def test_topk_bias_moves_selection(oracle):
    logits = np.zeros((1, 8), np.float32)
    logits[0, 3] = 1.0
    bias = np.zeros(8, np.float32)
    bias[6] = 5.0
    ids, w = oracle.route_topk(logits, 2, renorm=True, bias=bias)
    assert list(ids[0]) == [6, 3]
    # the bias feeds the weights too: softmax over (5, 1)
    np.testing.assert_allclose(w[0], scipy.special.softmax(np.array([5.0, 1.0])), rtol=1e-14)


# ---- init-routing --------------------------------------------------------------

@pytest.mark.parametrize("T,k,E,distinct", [(50, 4, 16, True), (33, 3, 5, False), (1, 1, 1, True),
                                            (64, 2, 16, True)])
def test_init_routing_invariants(oracle, T, k, E, distinct):
    ids = inputs.random_ids(T, k, E, seed=T + k, distinct=distinct).numpy()
    x = inputs.to_numpy(inputs.random_rows(T, 24, torch.bfloat16, seed=1))
    r = oracle.init_routing(ids, x, E)
    cnt, off, idx, ex = r["tokens_per_expert"], r["expert_offsets"], r["expanded_row_idx"], r["expanded_x"]
    R = T * k
    assert r["bad"] == 0
    assert cnt.sum() == R
    assert np.array_equal(cnt, np.bincount(ids.ravel(), minlength=E))
    assert off[0] == 0 and np.array_equal(np.diff(off), cnt)
    assert np.array_equal(np.sort(idx), np.arange(R))  # a permutation
    # stable sort by expert: numpy's stable argsort gives dst -> src
    order = np.argsort(ids.ravel(), kind="stable")
    assert np.array_equal(idx[order], np.arange(R))
    # the inverse permutation is the argsort of the permutation (Double-Routing step 6)
    inv = np.argsort(idx)
    assert np.array_equal(idx[inv], np.arange(R))
    # rows: expanded_x[dst] is the source token's row, bit for bit
    assert np.array_equal(ex[idx], x[np.arange(R) // k])
    # stability: ascending src inside each expert's segment
    for e in range(E):
        seg = inv[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)
        assert np.all(ids.ravel()[seg] == e)


def test_init_routing_flags_bad_ids(oracle):
    ids = np.array([[0, 5], [2, -1], [1, 1]], np.int32)
    r = oracle.init_routing(ids, None, 3, H=0)
    assert r["bad"] == 2
    assert r["expanded_row_idx"][1] == -1 and r["expanded_row_idx"][3] == -1
    assert r["tokens_per_expert"].tolist() == [1, 2, 1]


# ---- finalize-routing ----------------------------------------------------------

@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_finalize_identity_experts_k1_reproduces_x(oracle, dt):
    """k=1, unit weight, identity experts (y = expanded_x), no shared: out == x exactly."""
    T, E, k, H = 40, 8, 1, 32
    ids = inputs.random_ids(T, k, E, seed=7).numpy()
    x = inputs.to_numpy(inputs.random_rows(T, H, dt, seed=3))
    r = oracle.init_routing(ids, x, E)
    out = oracle.finalize_routing(r["expanded_x"], np.ones((T, k)), r["expanded_row_idx"])
    xd = x.astype(np.float64) if x.dtype == np.float32 else _bits_to_f64(x)
    assert np.array_equal(out, xd)


def test_finalize_identity_experts_renormalised_weights(oracle):
    T, E, k, H = 30, 16, 4, 20
    logits = inputs.random_logits(T, E, seed=11).numpy()
    ids, w = oracle.route_topk(logits, k, renorm=True)
    x = inputs.random_rows(T, H, torch.float32, seed=5).numpy()
    r = oracle.init_routing(ids, x, E)
    out = oracle.finalize_routing(r["expanded_x"], w, r["expanded_row_idx"])
    np.testing.assert_allclose(out, x.astype(np.float64), rtol=1e-13, atol=1e-13)


def test_finalize_skip_and_one_hot_scales(oracle):
    T, k, H = 6, 3, 10
    R = T * k
    y = inputs.random_rows(R, H, torch.float32, seed=2).numpy()
    skip = inputs.random_rows(T, H, torch.float32, seed=3, tag="misc").numpy()
    idx = np.random.default_rng(0).permutation(R).astype(np.int32)
    zero = np.zeros((T, k))
    assert np.array_equal(oracle.finalize_routing(y, zero, idx, skip), skip.astype(np.float64))
    onehot = np.zeros((T, k))
    onehot[:, 2] = 1.0
    out = oracle.finalize_routing(y, onehot, idx)
    assert np.array_equal(out, y[idx.reshape(T, k)[:, 2]].astype(np.float64))


# ---- expert FFN ------------------------------------------------------------------

def test_ffn_closed_form_detects_gate_up_swap(oracle):
    """H=I=1: y = c * silu(a v) * (b v); silu from torch (a library routine)."""
    a, b, c, v = 2.0, 3.0, 0.5, 1.0
    wg = np.array([[[a]]], np.float32)
    wu = np.array([[[b]]], np.float32)
    w2 = np.array([[[c]]], np.float32)
    y = oracle.expert_ffn_rows(np.array([[v]], np.float32), np.array([0], np.int32), wg, wu, w2)
    want = c * F.silu(torch.tensor(a * v, dtype=torch.float64)).item() * (b * v)
    swapped = c * F.silu(torch.tensor(b * v, dtype=torch.float64)).item() * (a * v)
    assert abs(y[0, 0] - want) < 1e-6 and abs(y[0, 0] - swapped) > 0.1


def test_ffn_zero_up_or_zero_gate_gives_zero(oracle):
    cfg = inputs.LayerConfig("t", T=4, H=16, E=2, k=1, I=8, S=0, dtype="f32", seed=1)
    d = inputs.make_layer(cfg)
    x = d["x"].numpy()
    ex = np.array([0, 1, 0, 1], np.int32)
    zero = np.zeros_like(d["w_up"].numpy())
    assert np.all(oracle.expert_ffn_rows(x, ex, d["w_gate"].numpy(), zero, d["w2"].numpy()) == 0)
    assert np.all(oracle.expert_ffn_rows(x, ex, zero, d["w_up"].numpy(), d["w2"].numpy()) == 0)


def _dense_swiglu(x, wg, wu, w2):
    """Textbook SwiGLU MLP (Shazeer 2020) with torch library ops in fp64."""
    x = x.to(torch.float64)
    return (F.silu(x @ wg.to(torch.float64).T) * (x @ wu.to(torch.float64).T)) @ w2.to(torch.float64).T


def test_layer_E1_k1_is_dense_swiglu_mlp(oracle):
    """One routed expert, top-1 (weight 1) + one shared expert = two dense SwiGLU MLPs."""
    cfg = inputs.LayerConfig("t", T=12, H=48, E=1, k=1, I=40, S=1, dtype="f32", seed=8)
    d = inputs.make_layer(cfg)
    r = oracle.layer(*(inputs.to_numpy(d[n]) for n in
                       ("x", "wg", "w_gate", "w_up", "w2", "s_gate", "s_up", "s2")), k=1)
    assert np.all(r["ids"] == 0) and np.all(r["w"] == 1.0)
    want = (_dense_swiglu(d["x"], d["w_gate"][0], d["w_up"][0], d["w2"][0])
            + _dense_swiglu(d["x"], d["s_gate"][0], d["s_up"][0], d["s2"][0])).numpy()
    np.testing.assert_allclose(r["out"], want, rtol=2e-6, atol=2e-6)


def test_ffn_rows_match_dense_mlp_per_expert(oracle):
    cfg = inputs.LayerConfig("t", T=10, H=40, E=3, k=1, I=24, S=0, dtype="f32", seed=12)
    d = inputs.make_layer(cfg)
    ex = np.array([2, 0, 1, 1, 0, 2, 2, 0, 1, 0], np.int32)
    y = oracle.expert_ffn_rows(d["x"].numpy(), ex, d["w_gate"].numpy(), d["w_up"].numpy(), d["w2"].numpy())
    for e in range(3):
        rows = np.nonzero(ex == e)[0]
        want = _dense_swiglu(d["x"][rows], d["w_gate"][e], d["w_up"][e], d["w2"][e]).numpy()
        np.testing.assert_allclose(y[rows], want, rtol=2e-6, atol=2e-6)


# ---- whole layer: brute force vs the permutation pipeline --------------------------

@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_layer_brute_force_equals_permutation_pipeline(oracle, dt):
    """Per-token loop == route -> init-routing -> expert FFN on expanded rows ->
    finalize with the shared output as skip (same rounding points: exact)."""
    cfg = inputs.LayerConfig("t", T=48, H=64, E=8, k=3, I=32, S=1, dtype=dt, seed=21)
    d = inputs.make_layer(cfg)
    n = {k_: inputs.to_numpy(v) for k_, v in d.items() if isinstance(v, torch.Tensor)}
    r = oracle.layer(n["x"], n["wg"], n["w_gate"], n["w_up"], n["w2"], n["s_gate"], n["s_up"], n["s2"],
                     k=cfg.k)
    logits32 = r["logits64"].astype(np.float32)
    ids, w = oracle.route_topk(logits32, cfg.k, renorm=True)
    assert np.array_equal(ids, r["ids"]) and np.array_equal(w, r["w"])
    ir = oracle.init_routing(ids, n["x"], cfg.E)
    expert_of_row = np.repeat(np.arange(cfg.E, dtype=np.int32), ir["tokens_per_expert"])
    y = oracle.expert_ffn_rows(ir["expanded_x"], expert_of_row, n["w_gate"], n["w_up"], n["w2"])
    ysh = oracle.expert_ffn_rows(n["x"], np.zeros(cfg.T, np.int32), n["s_gate"], n["s_up"], n["s2"])
    code = F32 if dt == "f32" else BF16
    store = (lambda a: a.astype(np.float32)) if dt == "f32" else _bf16_bits
    out = oracle.finalize_routing(store(y), w, ir["expanded_row_idx"], skip=store(ysh))
    assert np.array_equal(oracle.round_to(out, code), r["out"])


def test_layer_token_subset_matches_full(oracle):
    cfg = inputs.LayerConfig("t", T=20, H=32, E=6, k=2, I=16, S=2, dtype="bf16", seed=4)
    d = inputs.make_layer(cfg)
    args = [inputs.to_numpy(d[n]) for n in ("x", "wg", "w_gate", "w_up", "w2", "s_gate", "s_up", "s2")]
    full = oracle.layer(*args, k=2)
    toks = np.array([19, 3, 3, 0], np.int32)
    sub = oracle.layer(*args, k=2, tokens=toks)
    for name in ("ids", "w", "out", "logits64"):
        assert np.array_equal(sub[name], full[name][toks])


def test_layer_two_shared_experts_sum(oracle):
    """S=2 shared experts contribute the sum of two dense SwiGLU MLPs (fp32, E=1, k=1)."""
    cfg = inputs.LayerConfig("t", T=6, H=16, E=1, k=1, I=8, S=2, dtype="f32", seed=13)
    d = inputs.make_layer(cfg)
    r = oracle.layer(*(inputs.to_numpy(d[n]) for n in
                       ("x", "wg", "w_gate", "w_up", "w2", "s_gate", "s_up", "s2")), k=1)
    want = _dense_swiglu(d["x"], d["w_gate"][0], d["w_up"][0], d["w2"][0]).numpy()
    for s in range(2):
        want = want + _dense_swiglu(d["x"], d["s_gate"][s], d["s_up"][s], d["s2"][s]).numpy()
    np.testing.assert_allclose(r["out"], want, rtol=2e-6, atol=2e-6)


def test_layer_zipf_bias_feeds_selection(oracle):
    cfg = inputs.CONFIGS["tiny_fp32"].replace(zipf_s=1.2, T=16)
    d = inputs.make_layer(cfg)
    args = [inputs.to_numpy(d[n]) for n in ("x", "wg", "w_gate", "w_up", "w2", "s_gate", "s_up", "s2")]
    r = oracle.layer(*args, k=cfg.k, bias=d["bias"].numpy())
    s = (r["logits64"].astype(np.float32) + d["bias"].numpy())
    for t in range(cfg.T):
        assert list(r["ids"][t]) == _brute_topk(s[t], cfg.k)


# ---- group-limited top-k -----------------------------------------------------------

@pytest.mark.parametrize("rule", ["max", "top2_sum"])
def test_grouped_topk_single_group_is_flat(oracle, rule):
    """The page's special case: one group holding all experts is flat top-k."""
    logits = inputs.random_logits(50, 32, seed=5, ties="quantised").numpy()
    flat_ids, flat_w = oracle.route_topk(logits, 6)
    for n_group, topk_group in [(1, 1), (4, 4), (8, 8)]:
        ids, w = oracle.route_topk_grouped(logits, 6, n_group, topk_group, rule)
        assert np.array_equal(ids, flat_ids) and np.array_equal(w, flat_w)


def _brute_grouped(s, k, n_group, topk_group, rule):
    gs = s.size // n_group
    gscore = []
    for g in range(n_group):
        top = sorted(s[g * gs:(g + 1) * gs].tolist(), reverse=True)
        gscore.append(np.float32(top[0]) if rule == "max" else np.float32(top[0]) + np.float32(top[1]))
    kept = sorted(range(n_group), key=lambda g: (-float(gscore[g]), g))[:topk_group]
    cand = [e for e in range(s.size) if e // gs in kept]
    return sorted(cand, key=lambda e: (-float(s[e]), e))[:k]


@pytest.mark.parametrize("rule", ["max", "top2_sum"])
@pytest.mark.parametrize("E,n_group,topk_group,k", [(16, 4, 2, 3), (32, 8, 3, 8), (12, 3, 1, 4)])
def test_grouped_topk_brute_force(oracle, rule, E, n_group, topk_group, k):
    T = 60
    logits = inputs.random_logits(T, E, seed=E + k, ties="quantised").numpy()
    bias = (np.round(np.random.default_rng(E).standard_normal(E) * 2) / 4).astype(np.float32)
    ids, w = oracle.route_topk_grouped(logits, k, n_group, topk_group, rule, bias=bias)
    for t in range(T):
        s = logits[t] + bias
        assert list(ids[t]) == _brute_grouped(s, k, n_group, topk_group, rule)
        np.testing.assert_allclose(w[t], scipy.special.softmax(s[ids[t]].astype(np.float64)), rtol=1e-13)


def test_grouped_topk_rules_differ():
    """A group with one large score and weak others: "max" keeps it, "top2_sum" may not."""
    import oracle as o
    s = np.array([[5.0, -9.0, 3.0, 2.9]], np.float32)  # groups {0,1}, {2,3}
    ids_max, _ = o.route_topk_grouped(s, 1, 2, 1, "max")
    ids_sum, _ = o.route_topk_grouped(s, 1, 2, 1, "top2_sum")
    assert ids_max[0, 0] == 0 and ids_sum[0, 0] == 2


def test_layer_grouped_routing_uses_grouped_router(oracle):
    cfg = inputs.LayerConfig("t", T=24, H=32, E=16, k=3, I=16, S=1, dtype="f32", seed=31)
    d = inputs.make_layer(cfg)
    args = [inputs.to_numpy(d[n]) for n in ("x", "wg", "w_gate", "w_up", "w2", "s_gate", "s_up", "s2")]
    r = oracle.layer(*args, k=3, n_group=4, topk_group=2, group_rule="top2_sum")
    ids, w = oracle.route_topk_grouped(r["logits64"].astype(np.float32), 3, 4, 2, "top2_sum")
    assert np.array_equal(r["ids"], ids) and np.array_equal(r["w"], w)
    # the selected experts come from at most two groups
    assert all(len({e // 4 for e in row}) <= 2 for row in r["ids"])


# ---- re-routing (Double-Routing, second permutation) -------------------------------

def test_re_routing_is_a_stable_sort_by_local_expert(oracle):
    rng = np.random.default_rng(3)
    W, El, H = 4, 5, 12
    counts = rng.integers(0, 6, size=(W, El)).astype(np.int32)
    counts[2, :] = 0  # a source that sends nothing
    counts[:, 3] = 0  # an expert that receives nothing
    N = int(counts.sum())
    x = inputs.random_rows(N, H, torch.float32, seed=4).numpy()
    r = oracle.re_routing(x, counts)
    keys = np.concatenate([np.repeat(np.arange(El), counts[p]) for p in range(W)])
    order = np.argsort(keys, kind="stable")  # library stable sort
    assert np.array_equal(r["gathered_ids_unsort"], order)
    assert np.array_equal(r["x_sorted"], x[order])
    assert np.array_equal(r["tokens_per_local_expert"], counts.sum(0))
    assert np.array_equal(np.diff(r["local_offsets"]), counts.sum(0))
    # Double-Routing step 6: index_select with the argsort of gathered_ids_unsort restores arrival order
    back = r["x_sorted"][np.argsort(r["gathered_ids_unsort"])]
    assert np.array_equal(back, x)
    assert np.array_equal(oracle.unsort_rows(r["x_sorted"], r["gathered_ids_unsort"]), x)


def test_double_routing_permutations_compose_to_single_routing(oracle):
    """Init-routing per source rank, block exchange to the expert-owning ranks, then
    re-routing, puts the rows in exactly the single-routing (stable, by expert) order."""
    T, k, E, W, H = 48, 3, 8, 4, 10
    El, Tp = E // W, T // W
    ids = inputs.random_ids(T, k, E, seed=5).numpy()
    x = inputs.random_rows(T, H, torch.float32, seed=6).numpy()
    single = oracle.init_routing(ids, x, E)
    per_src = [oracle.init_routing(ids[p * Tp:(p + 1) * Tp], x[p * Tp:(p + 1) * Tp], E) for p in range(W)]
    sorted_all = []
    for q in range(W):
        blocks, counts = [], []
        for p in range(W):
            off = per_src[p]["expert_offsets"]
            blocks.append(per_src[p]["expanded_x"][off[q * El]:off[(q + 1) * El]])
            counts.append(per_src[p]["tokens_per_expert"][q * El:(q + 1) * El])
        r = oracle.re_routing(np.concatenate(blocks), np.array(counts, np.int32))
        sorted_all.append(r["x_sorted"])
    assert np.array_equal(np.concatenate(sorted_all), single["expanded_x"])


# ---- FP8 (e4m3) block quantisation -------------------------------------------------

def test_e4m3_decode_matches_torch_for_every_code(oracle):
    codes = torch.arange(256, dtype=torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_table()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_cast(oracle):
    rng = np.random.default_rng(0)
    table = oracle.e4m3_table()
    finite = np.sort(np.unique(table[~np.isnan(table)]))
    mids = (finite[:-1] + finite[1:]) / 2  # exact ties: round to the even code
    vals = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(2000) * 1e-2,
                           finite, mids, -mids]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448]
    got = np.array([oracle.e4m3_encode(v) for v in vals], np.uint8)
    want = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # +0/-0 both decode to zero; compare values
    assert np.array_equal(table[got], table[want])
    assert oracle.e4m3_encode(1000.0) == 0x7E and oracle.e4m3_encode(-1000.0) == 0xFE  # saturation


def test_quantize_rows_and_tiles(oracle):
    x = inputs.random_rows(5, 300, torch.bfloat16, seed=1)
    codes, scales = oracle.quantize_rows_fp8(inputs.to_numpy(x))
    assert scales.shape == (5, 3)
    xf = x.to(torch.float64).numpy()
    deq = oracle.e4m3_table()[codes] * np.repeat(scales.astype(np.float64), 128, axis=1)[:, :300]
    # each block's largest magnitude maps to +-448 exactly, every element within half an e4m3 step
    for r in range(5):
        for b in range(3):
            blk = xf[r, b * 128:(b + 1) * 128]
            assert np.isclose(np.abs(blk).max() / scales[r, b], 448.0, rtol=1e-6)
    assert np.all(np.abs(deq - xf) <= np.abs(xf) * 2.0 ** -4 + scales.max() * 2.0 ** -9)
    w = inputs.random_rows(200, 260, torch.float32, seed=2).numpy()
    wc, ws = oracle.quantize_tiles_fp8(w)
    assert ws.shape == (2, 3)
    np.testing.assert_allclose(ws[1, 2], np.abs(w[128:, 256:]).max() / 448, rtol=1e-7)
    zc, zs = oracle.quantize_rows_fp8(np.zeros((1, 128), np.float32))
    assert np.all(zc == 0) and zs[0, 0] == 1.0


def _dequant_torch(codes, scales, rows_per_scale):
    """Library dequantisation: torch's float8_e4m3fn values times the block scales."""
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s = np.repeat(np.repeat(scales.astype(np.float64), rows_per_scale, axis=0), 128, axis=1)
    return v * s[:v.shape[0], :v.shape[1]]


def test_gemm_fp8_is_dequantised_matmul(oracle):
    a = inputs.random_rows(7, 300, torch.bfloat16, seed=3)
    b = inputs.random_rows(260, 300, torch.float32, seed=4).numpy()
    qa, sa = oracle.quantize_rows_fp8(inputs.to_numpy(a))
    qb, sb = oracle.quantize_tiles_fp8(b)
    got = oracle.gemm_fp8(qa, sa, qb, sb)
    want = _dequant_torch(qa, sa, 1) @ _dequant_torch(qb, sb, 128).T
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_gemm_fp8_lossless_case_is_exact(oracle):
    """Small integers with a 448 in every block quantise exactly (scale 1)."""
    rng = np.random.default_rng(5)
    A = rng.integers(-8, 9, size=(4, 256)).astype(np.float32)
    B = rng.integers(-8, 9, size=(128, 256)).astype(np.float32)
    A[:, 0] = 448.0
    A[:, 128] = 448.0
    B[0, :] = 448.0
    qa, sa = oracle.quantize_rows_fp8(A)
    qb, sb = oracle.quantize_tiles_fp8(B)
    assert np.all(sa == 1.0) and np.all(sb == 1.0)
    assert np.array_equal(oracle.gemm_fp8(qa, sa, qb, sb), A.astype(np.float64) @ B.T.astype(np.float64))


def test_layer_fp8_dense_case_composes_the_steps(oracle):
    """E=1, k=1 + one shared expert: the FP8 layer is two FP8 SwiGLU MLPs built
    from the quantiser, the FP8 product and torch's SiLU."""
    cfg = inputs.LayerConfig("t", T=6, H=256, E=1, k=1, I=128, S=1, dtype="bf16", seed=9)
    d = inputs.make_layer(cfg)
    n = {k_: inputs.to_numpy(v) for k_, v in d.items() if isinstance(v, torch.Tensor)}
    q = {}
    for pre, g, u, w2 in (("", "w_gate", "w_up", "w2"), ("s", "s_gate", "s_up", "s2")):
        q[pre + "gq"], q[pre + "gs"] = oracle.quantize_experts_fp8(n[g])
        q[pre + "uq"], q[pre + "us"] = oracle.quantize_experts_fp8(n[u])
        q[pre + "dq"], q[pre + "ds"] = oracle.quantize_experts_fp8(n[w2])
    r = oracle.layer_fp8(n["x"], n["wg"], q, k=1)
    xq, xs = oracle.quantize_rows_fp8(n["x"])

    def mlp(pre):
        g = oracle.gemm_fp8(xq, xs, q[pre + "gq"][0], q[pre + "gs"][0])
        u = oracle.gemm_fp8(xq, xs, q[pre + "uq"][0], q[pre + "us"][0])
        h = (F.silu(torch.from_numpy(g)) * torch.from_numpy(u)).to(torch.bfloat16)
        hq, hs = oracle.quantize_rows_fp8(inputs.to_numpy(h))
        y = oracle.gemm_fp8(hq, hs, q[pre + "dq"][0], q[pre + "ds"][0])
        return oracle.round_to(y, BF16)

    want = oracle.round_to(mlp("s") + mlp(""), BF16)
    # torch's SiLU and the oracle's may differ in the last bit of h before rounding to bf16
    assert np.abs(r["out"] - want).max() <= 1e-2 * np.abs(want).max()
    # and the FP8 layer stays close to the bf16 layer (quantisation error only)
    ref = oracle.layer(*(n[k_] for k_ in ("x", "wg", "w_gate", "w_up", "w2", "s_gate", "s_up", "s2")), k=1)
    assert np.linalg.norm(r["out"] - ref["out"]) / np.linalg.norm(ref["out"]) < 0.1


# ---- FP8 with power-of-two block scales -------------------------------------------------

def _is_pow2(s: np.ndarray) -> bool:
    m, _ = np.frexp(s.astype(np.float64))
    return bool(np.all(m == 0.5))


def test_pow2_scales_are_the_smallest_powers_of_two(oracle):
    """Each scale is a power of two s with amax / s <= 448 < amax / (s / 2): the block's
    largest magnitude lands in (224, 448]; an all-zero block gets 1."""
    x = inputs.random_rows(9, 700, torch.float32, seed=21).numpy() * np.logspace(-3, 3, 9)[:, None]
    x[0, :128] = 0.0
    codes, scales = oracle.quantize_rows_fp8(x.astype(np.float32), pow2=True)
    assert _is_pow2(scales) and scales[0, 0] == 1.0 and np.all(codes[0, :128] == 0)
    for r in range(9):
        for b in range(scales.shape[1]):
            amax = np.abs(x[r, b * 128:(b + 1) * 128]).max()
            if amax == 0:
                continue
            s = float(scales[r, b])
            assert amax / s <= 448.0 < amax / (s / 2)
    # boundaries: exactly 448 * 2^e keeps 2^e, one fp32 step above doubles it
    for e in (-20, -1, 0, 3, 40):
        edge = np.float32(448.0 * 2.0 ** e)
        blk = np.zeros((2, 128), np.float32)
        blk[0, 5] = edge
        blk[1, 5] = np.nextafter(edge, np.float32(np.inf))
        _, s = oracle.quantize_rows_fp8(blk, pow2=True)
        assert s[0, 0] == np.float32(2.0 ** e) and s[1, 0] == np.float32(2.0 ** (e + 1))


def test_pow2_quantisation_is_lossless_on_grid_values(oracle):
    """Values c * s with c on the e4m3 grid and a 448 * s in the block come back as the
    same codes and scale (dividing by a power of two is exact)."""
    rng = np.random.default_rng(22)
    table = oracle.e4m3_table()
    finite = np.flatnonzero(~np.isnan(table) & (np.abs(table) <= 448))
    for e in (-9, 0, 5):
        c = rng.choice(finite, size=(3, 256)).astype(np.uint8)
        c[:, 0] = 0x7E  # 448 in every block
        c[:, 128] = 0xFE  # -448
        v = (table[c] * 2.0 ** e).astype(np.float32)
        codes, scales = oracle.quantize_rows_fp8(v, pow2=True)
        assert np.all(scales == np.float32(2.0 ** e))
        assert np.array_equal(table[codes], table[c])  # +0 / -0 compare equal as values
        wc, ws = oracle.quantize_tiles_fp8(np.tile(v, (43, 1))[:128], pow2=True)
        assert np.all(ws == np.float32(2.0 ** e)) and np.array_equal(table[wc], table[np.tile(c, (43, 1))[:128]])


def test_pow2_dequantised_within_half_a_step(oracle):
    x = inputs.random_rows(6, 300, torch.bfloat16, seed=23)
    xf = x.to(torch.float64).numpy()
    codes, scales = oracle.quantize_rows_fp8(inputs.to_numpy(x), pow2=True)
    deq = oracle.e4m3_table()[codes] * np.repeat(scales.astype(np.float64), 128, axis=1)[:, :300]
    # the code is the nearest grid point of v / s: within half an e4m3 step (relative 2^-4, or the
    # subnormal spacing 2^-9 times s)
    assert np.all(np.abs(deq - xf) <= np.abs(xf) * 2.0 ** -4 + np.repeat(scales, 128, axis=1)[:, :300] * 2.0 ** -10)
    # a power-of-two scale wastes at most one bit of range: amax / s > 224
    assert np.all(np.abs(xf).reshape(6, -1)[:, :256].reshape(6, 2, 128).max(axis=2) / scales[:, :2] > 224)


def test_gemm_fp8_pow2_is_dequantised_matmul(oracle):
    a = inputs.random_rows(7, 300, torch.bfloat16, seed=24)
    b = inputs.random_rows(260, 300, torch.float32, seed=25).numpy()
    qa, sa = oracle.quantize_rows_fp8(inputs.to_numpy(a), pow2=True)
    qb, sb = oracle.quantize_tiles_fp8(b, pow2=True)
    assert _is_pow2(sa) and _is_pow2(sb)
    want = _dequant_torch(qa, sa, 1) @ _dequant_torch(qb, sb, 128).T
    np.testing.assert_allclose(oracle.gemm_fp8(qa, sa, qb, sb), want, rtol=1e-12, atol=1e-12)


def test_layer_fp8_pow2_dense_case_composes_the_steps(oracle):
    """E=1, k=1 + one shared expert with power-of-two scales everywhere: the layer is two
    FP8 SwiGLU MLPs built from the power-of-two quantiser, the FP8 product and torch's SiLU."""
    cfg = inputs.LayerConfig("t", T=6, H=256, E=1, k=1, I=128, S=1, dtype="bf16", seed=26)
    d = inputs.make_layer(cfg)
    n = {k_: inputs.to_numpy(v) for k_, v in d.items() if isinstance(v, torch.Tensor)}
    q = {}
    for pre, g, u, w2 in (("", "w_gate", "w_up", "w2"), ("s", "s_gate", "s_up", "s2")):
        q[pre + "gq"], q[pre + "gs"] = oracle.quantize_experts_fp8(n[g], pow2=True)
        q[pre + "uq"], q[pre + "us"] = oracle.quantize_experts_fp8(n[u], pow2=True)
        q[pre + "dq"], q[pre + "ds"] = oracle.quantize_experts_fp8(n[w2], pow2=True)
    r = oracle.layer_fp8(n["x"], n["wg"], q, k=1, pow2=True)
    xq, xs = oracle.quantize_rows_fp8(n["x"], pow2=True)

    def mlp(pre):
        g = oracle.gemm_fp8(xq, xs, q[pre + "gq"][0], q[pre + "gs"][0])
        u = oracle.gemm_fp8(xq, xs, q[pre + "uq"][0], q[pre + "us"][0])
        h = (F.silu(torch.from_numpy(g)) * torch.from_numpy(u)).to(torch.bfloat16)
        hq, hs = oracle.quantize_rows_fp8(inputs.to_numpy(h), pow2=True)
        assert _is_pow2(hs)
        y = oracle.gemm_fp8(hq, hs, q[pre + "dq"][0], q[pre + "ds"][0])
        return oracle.round_to(y, BF16)

    want = oracle.round_to(mlp("s") + mlp(""), BF16)
    assert np.abs(r["out"] - want).max() <= 1e-2 * np.abs(want).max()
    ref = oracle.layer(*(n[k_] for k_ in ("x", "wg", "w_gate", "w_up", "w2", "s_gate", "s_up", "s2")), k=1)
    assert np.linalg.norm(r["out"] - ref["out"]) / np.linalg.norm(ref["out"]) < 0.1
    # a wrong scale format in the layer (fp32 scales for h) is visible
    r32 = oracle.layer_fp8(n["x"], n["wg"], q, k=1, pow2=False)
    assert not np.array_equal(r32["out"], r["out"])
