"""Comparison helpers shared by the tests (no arithmetic of the method here)."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from moe_expert_routing_route_gb300 import inputs


def f64(a) -> np.ndarray:
    """Values of a torch tensor or a numpy array (bf16 bit patterns included) as fp64."""
    if isinstance(a, torch.Tensor):
        return a.detach().cpu().to(torch.float64).numpy()
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return a.astype(np.float64)


def rel_l2(got, want) -> float:
    got, want = f64(got), f64(want)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def np_(t):
    return inputs.to_numpy(t)


def routing_ambiguity(scores: np.ndarray, k: int, err: float) -> np.ndarray:
    """True for tokens whose top-k (with slot order) could flip under a score
    perturbation of at most `err` per element: some adjacent gap among the k+1
    best scores is <= 2*err."""
    T, E = scores.shape
    srt = -np.sort(-scores, axis=1)[:, :min(k + 1, E)]
    with np.errstate(invalid="ignore"):
        gaps = srt[:, :-1] - srt[:, 1:]  # -inf entries (masked experts) never count as ties
    return np.any(np.nan_to_num(gaps, nan=np.inf) <= 2 * err, axis=1)


def check_topk_valid(ids: np.ndarray, scores: np.ndarray, err: float):
    """ids [k] must be distinct and a top-k of `scores` (descending) up to 2*err."""
    k = ids.size
    assert len(set(ids.tolist())) == k, "duplicate expert ids"
    s = scores[ids]
    assert np.all(s[:-1] >= s[1:] - 2 * err), "slots not in descending order"
    rest = np.setdiff1d(np.arange(scores.size), ids)
    if rest.size:
        assert s.min() >= scores[rest].max() - 2 * err, "a better expert was left out"


def check_permutation_properties(ids: np.ndarray, E: int, counts, offsets, row_idx, x=None, ex=None):
    """Init-routing outputs that hold for any ids: counts = histogram, offsets =
    exclusive scan, row_idx a stable expert-major permutation, rows copied."""
    R = ids.size
    counts, offsets, row_idx = np.asarray(counts), np.asarray(offsets), np.asarray(row_idx)
    assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts) and offsets[-1] == R
    assert np.array_equal(np.sort(row_idx), np.arange(R))
    inv = np.argsort(row_idx)
    flat = ids.ravel()
    for e in np.nonzero(counts)[0]:
        seg = inv[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
    if x is not None:
        k = ids.shape[1]
        assert np.array_equal(ex[row_idx], x[np.arange(R) // k])


def per_row_rel_l2(got, want) -> np.ndarray:
    """rel-L2 of each row (token) separately: ||got_r - want_r|| / ||want_r||."""
    got, want = f64(got), f64(want)
    got, want = got.reshape(len(got), -1), want.reshape(len(want), -1)
    den = np.linalg.norm(want, axis=1)
    return np.linalg.norm(got - want, axis=1) / np.where(den > 0, den, 1.0)


# Per-token (per-row) tolerance next to the aggregate one: the layer tolerance
# (rel-L2 <= 1e-2 bf16, 1e-5 fp32) held by every token, not only on average.  One
# wrong row among thousands barely moves an aggregate rel-L2, but fails this.
ROW_TOL = {"bf16": 1e-2, "f32": 1e-5}


def group_scores(scores: np.ndarray, n_group: int, rule: str) -> np.ndarray:
    """Group score of each expert group: its best score ("max") or the sum of its
    two best ("top2_sum").  scores [E] or [T,E]."""
    s = np.atleast_2d(scores)
    g = -np.sort(-s.reshape(len(s), n_group, -1), axis=2)
    out = g[:, :, 0] + (g[:, :, 1] if rule == "top2_sum" else 0.0)
    return out if scores.ndim == 2 else out[0]


def check_grouped_topk_valid(ids: np.ndarray, scores: np.ndarray, n_group: int, topk_group: int, rule: str,
                             err: float):
    """Group-limited routing, valid within a score error of `err` per expert: there
    is a set K of topk_group groups that is a top-topk_group set of the group
    scores (within the error of a group score: 2*err for "max", 4*err for a sum
    of two), such that ids lie in K and are a valid top-k of the scores of K's
    experts (within 2*err).  K exists iff the greedy choice exists: the groups of
    ids, plus the best-scoring other groups whose experts all score no more than
    the weakest chosen one (+ 2*err)."""
    E = scores.size
    gs = E // n_group
    k = ids.size
    assert len(set(ids.tolist())) == k, "duplicate expert ids"
    s = scores[ids]
    assert np.all(s[:-1] >= s[1:] - 2 * err), "slots not in descending order"
    gsc = group_scores(scores, n_group, rule)
    gtol = (4 if rule == "top2_sum" else 2) * err
    chosen = sorted(set((ids // gs).tolist()))
    assert len(chosen) <= topk_group, "ids span more groups than are kept"
    gmax = scores.reshape(n_group, gs).max(axis=1)
    cand = [g for g in np.argsort(-gsc, kind="stable") if g not in chosen and gmax[g] <= s.min() + 2 * err]
    K = chosen + [int(g) for g in cand[:topk_group - len(chosen)]]
    assert len(K) == topk_group, "no valid set of kept groups holds these ids"
    rest = [g for g in range(n_group) if g not in K]
    if rest:
        assert gsc[K].min() >= gsc[rest].max() - gtol, "a better group was left out"
    in_k = np.concatenate([np.arange(g * gs, (g + 1) * gs) for g in K])
    others = np.setdiff1d(in_k, ids)
    if others.size:
        assert s.min() >= scores[others].max() - 2 * err, "a better expert of a kept group was left out"


def log_parity(name: str, **values):
    """Append the measured errors of one comparison to the file MOE_PARITY_LOG names
    (nothing when it is unset): the record behind the tolerances."""
    path = os.environ.get("MOE_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(config=name, **values)) + "\n")
