"""Whole-layer parity checks against the CPU oracle, shared by the layer, FP8 and
expert-parallel GPU tests (comparison only: no arithmetic of the method here).

Routing: the oracle computes its own fp64 gate logits; the GPU's logits must be
within rel-L2 1e-5 of them.  Ids are compared exactly for every token whose
choice cannot flip under the measured logit error; for the other tokens the
GPU's ids must be a valid top-k (flat routing) or a valid group-limited top-k
(grouped routing) of the oracle's scores within that error.
Outputs: aggregate rel-L2 within the layer tolerance (1e-2 bf16, 1e-5 fp32) and,
for every compared token, its own rel-L2 within the per-token bound."""
from __future__ import annotations

import numpy as np
import torch

from moe_expert_routing_route_gb300 import binding
from tests._cmp import (ROW_TOL, check_grouped_topk_valid, check_permutation_properties, check_topk_valid, f64,
                        group_scores, log_parity, np_, per_row_rel_l2, rel_l2, routing_ambiguity)

LAYER_TOL = {"bf16": 1e-2, "f32": 1e-5}


def host_arrays(d: dict) -> dict:
    return {key: np_(v) for key, v in d.items() if isinstance(v, torch.Tensor)}


def check_routing(oracle, cfg, n: dict, gl: np.ndarray, ids: np.ndarray, w: np.ndarray):
    """Gate logits, ids and weights of the GPU against the oracle.  Returns the
    oracle's ids for all tokens."""
    bias = n.get("bias")
    k, E = cfg.k, cfg.E
    ref_logits = oracle.gate_logits(n["x"], n["wg"])
    assert rel_l2(gl, ref_logits) <= 1e-5
    l32 = ref_logits.astype(np.float32)
    s_ref = (l32 + bias if bias is not None else l32).astype(np.float64)
    # the measured logit error plus one rounding of the (biased) fp32 score
    maxerr = float(np.abs(gl.astype(np.float64) - ref_logits).max()) + 2.0 ** -23 * float(np.abs(s_ref).max())
    if cfg.n_group > 1:
        r_ids, r_w = oracle.route_topk_grouped(l32, k, cfg.n_group, cfg.topk_group, cfg.group_rule,
                                               renorm=cfg.renormalize, bias=bias)
        # ambiguous: a near-tie among the best k+1 experts of the groups that
        # could be kept, or between the last kept group and the next one (a
        # top-2 sum carries the error of two scores)
        gs = E // cfg.n_group
        gscore = group_scores(s_ref, cfg.n_group, cfg.group_rule)
        masked = s_ref.copy()
        for t in range(len(s_ref)):
            keep = np.zeros(cfg.n_group, bool)
            keep[np.unique(r_ids[t] // gs)] = True
            keep[np.argsort(-gscore[t], kind="stable")[:cfg.topk_group]] = True
            masked[t][~np.repeat(keep, gs)] = -np.inf
        amb = routing_ambiguity(masked, k, maxerr)
        if cfg.topk_group < cfg.n_group:
            gsorted = -np.sort(-gscore, axis=1)
            amb |= gsorted[:, cfg.topk_group - 1] - gsorted[:, cfg.topk_group] <= 4 * maxerr
        for t in np.nonzero(amb)[0]:
            check_grouped_topk_valid(ids[t], s_ref[t], cfg.n_group, cfg.topk_group, cfg.group_rule, maxerr)
    else:
        r_ids, r_w = oracle.route_topk(l32, k, renorm=cfg.renormalize, bias=bias)
        amb = routing_ambiguity(s_ref, k, maxerr)
        for t in np.nonzero(amb)[0]:
            check_topk_valid(ids[t], s_ref[t], maxerr)
    assert np.array_equal(ids[~amb], r_ids[~amb])
    np.testing.assert_allclose(w[~amb], r_w[~amb], rtol=1e-4, atol=1e-6)
    return r_ids


def check_output(cfg, ids: np.ndarray, out, ref: dict, toks: np.ndarray) -> dict:
    """out [T,H] of the GPU on tokens toks against the oracle's ref (ids, out for
    those tokens).  Tokens whose id sets differ (near-ties, at most 1%) are left
    out of the comparison.  Returns the aggregate and worst per-token rel-L2."""
    same = np.array([set(ids[t]) == set(ref["ids"][i]) for i, t in enumerate(toks)])
    assert (~same).sum() <= max(1, len(toks) // 100)
    got = f64(out)[toks][same]
    want = ref["out"][same]
    err = rel_l2(got, want)
    rows = per_row_rel_l2(got, want)
    assert err <= LAYER_TOL[cfg.dtype], f"{cfg.name}: rel-L2 {err:.3e}"
    worst = int(np.argmax(rows)) if rows.size else -1
    assert rows.size == 0 or rows.max() <= ROW_TOL[cfg.dtype], \
        f"{cfg.name}: token {toks[same][worst]} rel-L2 {rows.max():.3e}"
    res = dict(rel_l2=err, worst_token_rel_l2=float(rows.max()) if rows.size else 0.0, compared=int(same.sum()))
    log_parity(cfg.name, **res)
    return res


def oracle_layer(oracle, cfg, n: dict, toks: np.ndarray | None):
    return oracle.layer(n["x"], n["wg"], n["w_gate"], n["w_up"], n["w2"], n.get("s_gate") if cfg.S else None,
                        n.get("s_up") if cfg.S else None, n.get("s2") if cfg.S else None, k=cfg.k,
                        renorm=cfg.renormalize, bias=n.get("bias"), tokens=toks, n_group=cfg.n_group,
                        topk_group=cfg.topk_group, group_rule=cfg.group_rule)


def check_layer(oracle, cfg, d, layer, out, tokens=None, n=None, ref=None):
    """Routing, permutation and output of one moe_layer_forward call."""
    n = host_arrays(d) if n is None else n
    gl = layer.field("logits").cpu().numpy()
    ids = layer.field("topk_ids").cpu().numpy()
    w = layer.field("topk_w").cpu().numpy()
    r_ids = check_routing(oracle, cfg, n, gl, ids, w)
    # permutation: properties on the GPU's ids; bit-exact against the oracle when routing agrees
    counts = layer.field("tokens_per_expert").cpu().numpy()
    offsets = layer.field("expert_offsets").cpu().numpy()
    row_idx = layer.field("expanded_row_idx").cpu().numpy()
    ex = np_(layer.field("expanded_x"))
    check_permutation_properties(ids, cfg.E, counts, offsets, row_idx, n["x"], ex)
    if np.array_equal(ids, r_ids):
        ir = oracle.init_routing(r_ids, None, cfg.E, H=cfg.H)
        assert np.array_equal(row_idx, ir["expanded_row_idx"])
        assert np.array_equal(offsets, ir["expert_offsets"])
    toks = np.arange(cfg.T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    if ref is None:
        ref = oracle_layer(oracle, cfg, n, None if tokens is None else toks)
    res = check_output(cfg, ids, out, ref, toks)
    assert binding.moe_check_device_status(layer.ws) == 0
    return res
