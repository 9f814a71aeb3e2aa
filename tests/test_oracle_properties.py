"""Randomised properties of the oracle (CPU only).  The fixed-example pins in
test_oracle_pins.py check each function against an independent computation;
these draw many small shapes -- dense ties, E not a multiple of 32, k up to E,
empty experts -- and check the defining properties on every draw."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

SETTINGS = settings(max_examples=30, deadline=None, derandomize=True)


@st.composite
def routing_case(draw):
    E = draw(st.integers(1, 70))
    k = draw(st.integers(1, min(E, 9)))
    T = draw(st.integers(1, 40))
    levels = draw(st.sampled_from([3, 8, 1000]))  # few levels: many exact ties
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    logits = (rng.integers(0, levels, size=(T, E)) / 4.0 - 1.0).astype(np.float32)
    return logits, k


@SETTINGS
@given(routing_case(), st.booleans())
def test_topk_is_the_stable_sort_prefix(oracle, case, renorm):
    logits, k = case
    ids, w = oracle.route_topk(logits, k, renorm=renorm)
    T, E = logits.shape
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        assert list(ids[t]) == order
    if renorm:
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)  # slots in descending score order carry non-increasing weights


@SETTINGS
@given(routing_case())
def test_group_limited_routing_with_one_group_is_flat(oracle, case):
    logits, k = case
    ids, w = oracle.route_topk(logits, k)
    gids, gw = oracle.route_topk_grouped(logits, k, 1, 1, "max")
    assert np.array_equal(ids, gids)
    np.testing.assert_array_equal(w, gw)


@st.composite
def ids_case(draw):
    E = draw(st.integers(1, 50))
    k = draw(st.integers(1, min(E, 8)))
    T = draw(st.integers(0, 60))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    # each token draws k distinct experts, from a skewed subset so that some experts stay empty
    pool = rng.permutation(E)[:max(k, E // 2 + 1)]
    ids = np.stack([rng.choice(pool, size=k, replace=False) for _ in range(T)]).astype(np.int32) \
        if T else np.zeros((0, k), np.int32)
    return ids, E


@SETTINGS
@given(ids_case())
def test_init_routing_defining_properties(oracle, case):
    ids, E = case
    T, k = ids.shape
    H = 4
    x = np.arange(T * H, dtype=np.float32).reshape(T, H)
    ir = oracle.init_routing(ids, x, E)
    flat = ids.ravel()
    counts = ir["tokens_per_expert"]
    offsets = ir["expert_offsets"]
    row_idx = ir["expanded_row_idx"]
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts) and offsets[-1] == T * k
    assert np.array_equal(np.sort(row_idx), np.arange(T * k))  # a permutation
    # the sorted order is numpy's stable argsort by expert id
    assert np.array_equal(np.argsort(flat, kind="stable"), np.argsort(row_idx))
    if T:
        assert np.array_equal(ir["expanded_x"][row_idx], x[np.arange(T * k) // k])


@SETTINGS
@given(ids_case(), st.integers(0, 2 ** 31 - 1))
def test_finalize_is_the_weighted_gather(oracle, case, seed):
    ids, E = case
    T, k = ids.shape
    if T == 0:
        return
    H = 8
    rng = np.random.default_rng(seed)
    ir = oracle.init_routing(ids, None, E, H=H)
    row_idx = ir["expanded_row_idx"]
    y = rng.standard_normal((T * k, H)).astype(np.float32)  # stored values (fp32)
    w = rng.random((T, k))
    skip = rng.standard_normal((T, H)).astype(np.float32)
    out = oracle.finalize_routing(y, w, row_idx, skip=skip)  # fp64 sums
    want = skip.astype(np.float64) + np.einsum("tj,tjh->th", w, y[row_idx].astype(np.float64).reshape(T, k, H))
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


@SETTINGS
@given(st.lists(st.floats(-500.0, 500.0, allow_nan=False, width=32), min_size=1, max_size=64))
def test_e4m3_encode_is_nearest_and_monotone(oracle, values):
    table = oracle.e4m3_table()  # value of every code
    finite = np.isfinite(table)
    for v in values:
        c = oracle.e4m3_encode(v)
        d = table[c]
        assert np.isfinite(d) and abs(d) <= 448.0
        # no finite code is strictly nearer to v (saturated at +-448)
        vc = min(max(v, -448.0), 448.0)
        assert np.all(np.abs(table[finite] - vc) >= abs(d - vc) - 1e-12)
    enc = [table[oracle.e4m3_encode(v)] for v in sorted(values)]
    assert all(a <= b for a, b in zip(enc, enc[1:]))


@st.composite
def re_routing_case(draw):
    W = draw(st.integers(1, 6))
    El = draw(st.integers(1, 9))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, draw(st.sampled_from([1, 3, 6])), size=(W, El)).astype(np.int32)
    return counts


@SETTINGS
@given(re_routing_case())
def test_re_routing_is_the_stable_sort_by_local_expert(oracle, counts):
    """Rows arrive source after source, each source's rows in local-expert order; the
    second routing sorts them by local expert, stably (arrival order inside an expert),
    and the un-sort puts every row back where it arrived."""
    W, El = counts.shape
    N, H = int(counts.sum()), 3
    x = np.arange(N * H, dtype=np.float32).reshape(N, H)  # every row distinct
    r = oracle.re_routing(x, counts)
    keys = np.concatenate([np.repeat(np.arange(El), counts[p]) for p in range(W)]) if N else np.zeros(0, int)
    order = np.argsort(keys, kind="stable")
    assert np.array_equal(r["gathered_ids_unsort"], order)
    assert np.array_equal(r["x_sorted"], x[order])
    assert np.array_equal(r["tokens_per_local_expert"], counts.sum(0))
    assert r["local_offsets"][0] == 0 and np.array_equal(np.diff(r["local_offsets"]), counts.sum(0))
    assert np.array_equal(oracle.unsort_rows(r["x_sorted"], r["gathered_ids_unsort"]), x)


@st.composite
def fp8_rows_case(draw):
    rows = draw(st.integers(1, 4))
    cols = draw(st.integers(1, 400))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    mag = 10.0 ** rng.uniform(-6, 6, size=(rows, 1))  # a magnitude per row, 12 decades apart at most
    a = (rng.standard_normal((rows, cols)) * mag).astype(np.float32)
    nb = (cols + 127) // 128
    for r in range(rows):  # some all-zero blocks
        for b in range(nb):
            if rng.random() < 0.15:
                a[r, b * 128:(b + 1) * 128] = 0.0
    return a


@SETTINGS
@given(fp8_rows_case(), st.booleans())
def test_fp8_row_blocks_scales_and_codes(oracle, a, pow2):
    """1x128 blocks: fp32 scales put the block's largest magnitude at 448, power-of-two
    scales are the smallest 2^e that keep it at or below 448; an all-zero block gets
    scale 1 and zero codes; every element decodes within half an e4m3 step."""
    rows, cols = a.shape
    codes, scales = oracle.quantize_rows_fp8(a, pow2=pow2)
    nb = (cols + 127) // 128
    assert codes.shape == (rows, cols) and scales.shape == (rows, nb)
    table = oracle.e4m3_table()
    for r in range(rows):
        for b in range(nb):
            blk = a[r, b * 128:(b + 1) * 128].astype(np.float64)
            s = float(scales[r, b])
            amax = np.abs(blk).max()
            deq = table[codes[r, b * 128:(b + 1) * 128]]
            if amax == 0:
                assert s == 1.0 and np.all(deq == 0)
                continue
            if pow2:
                assert s == 2.0 ** np.round(np.log2(s))
                assert amax / s <= 448.0 < amax / (s / 2)
            else:
                assert np.isclose(amax / s, 448.0, rtol=1e-6)
            sub = 2.0 ** -10 if pow2 else 2.0 ** -9
            assert np.all(np.abs(deq * s - blk) <= np.abs(blk) * 2.0 ** -4 + s * sub)
