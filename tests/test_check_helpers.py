"""The parity checkers themselves (CPU only): the validity checks used for tokens
whose routing can flip under the measured logit error accept the oracle's own
choices and reject planted mistakes."""
import numpy as np
import pytest

from moe_expert_routing_route_gb300 import inputs
from tests._cmp import check_grouped_topk_valid, check_topk_valid, group_scores, per_row_rel_l2


def _grouped(oracle, T, E, k, n_group, topk_group, rule, seed):
    logits = inputs.random_logits(T, E, seed=seed).numpy()
    ids, _ = oracle.route_topk_grouped(logits, k, n_group, topk_group, rule)
    return logits.astype(np.float64), ids


@pytest.mark.parametrize("rule", ["max", "top2_sum"])
@pytest.mark.parametrize("E,k,n_group,topk_group", [(64, 6, 8, 3), (256, 8, 8, 4), (32, 4, 4, 1), (40, 5, 5, 5)])
def test_grouped_validity_accepts_the_oracle(oracle, rule, E, k, n_group, topk_group):
    s, ids = _grouped(oracle, 200, E, k, n_group, topk_group, rule, seed=E + k)
    for t in range(len(s)):
        check_grouped_topk_valid(ids[t], s[t], n_group, topk_group, rule, err=0.0)
        check_grouped_topk_valid(ids[t], s[t], n_group, topk_group, rule, err=1e-6)


@pytest.mark.parametrize("rule", ["max", "top2_sum"])
def test_grouped_validity_rejects_planted_mistakes(oracle, rule):
    E, k, n_group, topk_group = 64, 6, 8, 3
    s, ids = _grouped(oracle, 100, E, k, n_group, topk_group, rule, seed=7)
    gs = E // n_group
    caught = dict(group=0, order=0, weaker=0, dup=0)
    for t in range(len(s)):
        gsc = group_scores(s[t], n_group, rule)
        kept = set((ids[t] // gs).tolist())
        # (1) the last id moved to the best expert of the weakest group (never a kept group
        # when its score is clearly below the kept ones)
        worst = int(np.argmin(gsc))
        if worst not in kept and gsc[worst] < np.sort(gsc)[-topk_group] - 0.1:
            bad = ids[t].copy()
            bad[-1] = worst * gs + int(np.argmax(s[t][worst * gs:(worst + 1) * gs]))
            if s[t][bad[-1]] < s[t][bad[-2]]:
                with pytest.raises(AssertionError):
                    check_grouped_topk_valid(bad, s[t], n_group, topk_group, rule, err=1e-6)
                caught["group"] += 1
        # (2) two slots swapped out of descending order
        if s[t][ids[t][0]] - s[t][ids[t][1]] > 1e-3:
            bad = ids[t].copy()
            bad[[0, 1]] = bad[[1, 0]]
            with pytest.raises(AssertionError):
                check_grouped_topk_valid(bad, s[t], n_group, topk_group, rule, err=1e-6)
            caught["order"] += 1
        # (3) the last id replaced by the weakest expert of the first kept group
        g0 = ids[t][0] // gs
        members = np.arange(g0 * gs, (g0 + 1) * gs)
        weakest = int(members[np.argmin(s[t][members])])
        if weakest not in ids[t] and s[t][weakest] < s[t][ids[t][-1]] - 1e-3:
            bad = ids[t].copy()
            bad[-1] = weakest
            with pytest.raises(AssertionError):
                check_grouped_topk_valid(bad, s[t], n_group, topk_group, rule, err=1e-6)
            caught["weaker"] += 1
        # (4) a duplicate id
        bad = ids[t].copy()
        bad[-1] = bad[0]
        with pytest.raises(AssertionError):
            check_grouped_topk_valid(bad, s[t], n_group, topk_group, rule, err=1e-6)
        caught["dup"] += 1
    assert min(caught.values()) >= 10, caught


def test_grouped_validity_accepts_either_side_of_a_group_tie():
    """Two groups whose scores tie within the error: keeping either is valid."""
    n_group, topk_group, gs = 4, 3, 4
    s = np.array([5.0, 1, 0, 0,  4.0, 0.5, 0, 0,  3.0, 0.2, 0, 0,  3.0 + 1e-7, 0.1, 0, 0])
    for last in (8, 12):
        ids = np.array([0, 4, last])
        check_grouped_topk_valid(ids, s, n_group, topk_group, "max", err=1e-7)
    with pytest.raises(AssertionError):  # a clear gap: only group 3 is valid
        s2 = s.copy()
        s2[12] = 3.5
        check_grouped_topk_valid(np.array([0, 4, 8]), s2, n_group, topk_group, "max", err=1e-7)


def test_flat_validity_rejects_a_left_out_better_expert():
    s = np.array([0.9, 0.1, 0.8, 0.7, 0.2])
    check_topk_valid(np.array([0, 2, 3]), s, err=0.0)
    with pytest.raises(AssertionError):
        check_topk_valid(np.array([0, 2, 4]), s, err=0.0)
    check_topk_valid(np.array([0, 2, 4]), s, err=0.3)  # within the error


def test_per_row_rel_l2_isolates_one_bad_row():
    rng = np.random.default_rng(0)
    want = rng.standard_normal((2400, 64))
    got = want.copy()
    got[17] *= 1.3
    errs = per_row_rel_l2(got, want)
    assert errs[17] == pytest.approx(0.3) and np.all(np.delete(errs, 17) == 0)
    # the aggregate barely moves: the reason for the per-row bound
    agg = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert agg < 1e-2
