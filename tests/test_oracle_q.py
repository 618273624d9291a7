"""Pins of the oracle's q construction and integer draw.

"PP1 q transport and scheduling design", section "Distribution contract and
precision": integer counts summing exactly to M = 2^24, floor plus largest
remainders with ties to the lowest token id, FP64 allocation, sparse top-k
support chosen first, a 24-bit draw returning the first cumulative count
strictly greater than the draw.

Pins used here (none re-types the oracle's formulas):
* closed forms for uniform rows (lowest-id ties at full vocabulary size);
* the exact-integer Hamilton apportionment of M with quotas M*E_v/S, which
  the FP64 allocation must reproduce whenever no two fractional parts are
  within FP64 rounding of each other;
* the integer weights against numpy's float64 exp;
* the top-k support against numpy's stable sort;
* temperature as an exact rescaling;
* every one of the 2^24 draws, whose histogram must equal the counts.
"""
import json
import os

import numpy as np
import pytest

M = 1 << 24


def hamilton(E, support):
    """Exact largest-remainder apportionment of M over quotas M*E_v/S
    (integer arithmetic; ties to the lowest id)."""
    ids = [v for v in range(len(E)) if support[v]]
    S = sum(int(E[v]) for v in ids)
    floors, rems = {}, {}
    for v in ids:
        num = M * int(E[v])
        floors[v], rems[v] = divmod(num, S)
    R = M - sum(floors.values())
    order = sorted(ids, key=lambda v: (-rems[v], v))
    counts = np.zeros(len(E), np.int64)
    for v in ids:
        counts[v] = floors[v]
    for v in order[:R]:
        counts[v] += 1
    # smallest gap between distinct remainders, relative to S (FP64 can only
    # disagree with the exact order when this is below ~2^-45)
    r_sorted = sorted(set(rems.values()))
    gap = min((b - a for a, b in zip(r_sorted, r_sorted[1:])), default=S) / S
    return counts, R, gap


# ------------------------------------------------------------- closed forms
def test_uniform_full_vocab_lowest_id_rule(oracle):
    V = 129280
    c, _, _, st = oracle.q_build(np.zeros((1, V), np.float32))
    assert st[0] == 0
    base, extra = divmod(M, V)
    assert (base, extra) == (129, 100096)
    expect = np.full(V, base, np.uint32)
    expect[:extra] += 1
    assert np.array_equal(c[0], expect)


@pytest.mark.parametrize("V,expect", [(3, [5592406, 5592405, 5592405]), (8, [1 << 21] * 8),
                                      (1, [M]), (2, [1 << 23, 1 << 23])])
def test_uniform_small(oracle, V, expect):
    c, _, _, st = oracle.q_build(np.full((1, V), 3.25, np.float32))
    assert st[0] == 0 and c[0].tolist() == expect


@pytest.mark.parametrize("n", [1, 2, 4, 64, 512, 4096, 65536])
def test_uniform_power_of_two_support(oracle, n):
    V = 129280
    rng = np.random.default_rng(n)
    x = np.full(V, -np.inf, np.float32)
    sup = rng.choice(V, size=n, replace=False)
    x[sup] = -7.5
    c, _, _, st = oracle.q_build(x[None])
    assert st[0] == 0
    assert np.all(c[0, sup] == M // n)
    assert c[0].sum() == M


def test_single_finite_logit_gets_all_mass(oracle):
    x = np.full(1000, -np.inf, np.float32)
    x[417] = 12.0
    c, _, _, st = oracle.q_build(x[None])
    assert st[0] == 0 and c[0, 417] == M and c[0].sum() == M


def test_top1_goes_to_lowest_id_of_tied_maxima(oracle):
    x = np.linspace(-5, 5, 4099).astype(np.float32)
    x[[100, 2000, 4098]] = 9.0
    c, ids, nnz, st = oracle.q_build(x[None], top_k=1)
    assert st[0] == 0 and nnz[0] == 1 and ids[0, 0] == 100 and c[0, 0] == M


# -------------------------------------------- exact apportionment (Hamilton)
def _rows(rng, V):
    yield rng.normal(0, 2, V).astype(np.float32)
    yield rng.normal(0, 6, V).astype(np.float32)
    r = (-1.1 * np.log1p(rng.permutation(V)) + rng.normal(0, 0.3, V)).astype(np.float32)
    yield r
    m = r.copy()
    m[rng.random(V) < 0.3] = -np.inf
    yield m
    yield np.round(rng.normal(0, 2, V) * 2) .astype(np.float32) / 2  # many exact ties


@pytest.mark.parametrize("V", [2, 3, 5, 8, 13, 16, 257, 4099])
def test_allocation_matches_exact_hamilton(oracle, V):
    rng = np.random.default_rng(V)
    checked = 0
    for x in _rows(rng, V):
        st, E, sup, S = oracle.q_weights_row(x)
        if st != 0:
            continue
        c, _, _, st2 = oracle.q_build(x[None])
        assert st2[0] == 0
        exact, R, gap = hamilton(E, sup)
        assert gap > 2.0 ** -40  # FP64 allocation cannot reorder these remainders
        assert np.array_equal(c[0].astype(np.int64), exact)
        assert 0 <= R < M
        checked += 1
    assert checked >= 4


@pytest.mark.slow
def test_allocation_matches_exact_hamilton_full_vocab(oracle):
    rng = np.random.default_rng(99)
    V = 129280
    for x in list(_rows(rng, V))[:3]:
        st, E, sup, S = oracle.q_weights_row(x)
        assert st == 0
        c, _, _, _ = oracle.q_build(x[None])
        exact, R, gap = hamilton(E, sup)
        if gap > 2.0 ** -40:
            assert np.array_equal(c[0].astype(np.int64), exact)
        else:  # near-equal remainders: counts still within one of the quota
            assert np.abs(c[0].astype(np.int64) - exact).max() <= 1
        assert c[0].sum() == M


# ------------------------------------------------------ integer weights E_v
def test_weights_follow_softmax_numerator(oracle):
    rng = np.random.default_rng(5)
    V = 4099
    x = rng.normal(0, 3, V).astype(np.float32)
    x[rng.random(V) < 0.1] = -np.inf
    st, E, sup, S = oracle.q_weights_row(x, T=0.7)
    assert st == 0
    y = x.astype(np.float64) * float(np.float32(1.0) / np.float32(0.7))
    ref = np.where(np.isfinite(y), np.exp(y - y[np.isfinite(y)].max()), 0.0) * 2.0 ** 40
    # exp_ds is within 1 ulp of exp; the fp32 temperature multiply and the
    # shift by the max add a few more ulp of the exponent
    err = np.abs(E.astype(np.float64) - ref)
    assert np.all(err <= 1.0 + 2e-6 * ref)
    assert E.max() == 1 << 40
    assert S == int(E.sum())
    assert np.array_equal(sup, np.isfinite(x))


def test_temperature_is_an_exact_rescaling(oracle):
    rng = np.random.default_rng(11)
    x = rng.normal(0, 2, 20000).astype(np.float32)
    c1, _, _, _ = oracle.q_build((2 * x)[None], temperature=1.0)
    c2, _, _, _ = oracle.q_build(x[None], temperature=0.5)
    assert np.array_equal(c1, c2)
    c3, _, _, _ = oracle.q_build(x[None])
    c4, _, _, _ = oracle.q_build((x / 4)[None], temperature=0.25)
    assert np.array_equal(c3, c4)


# --------------------------------------------------------------- sparse q
@pytest.mark.parametrize("k", [1, 2, 16, 256, 5000])
def test_topk_support_and_layout(oracle, k):
    rng = np.random.default_rng(k)
    V = 4099
    x = np.round(rng.normal(0, 2, V) * 8).astype(np.float32) / 8  # many ties
    x[rng.random(V) < 0.05] = -np.inf
    c, ids, nnz, st = oracle.q_build(x[None], top_k=k)
    assert st[0] == 0
    finite = np.flatnonzero(np.isfinite(x))
    order = finite[np.lexsort((finite, -x[finite]))]  # by value desc, then id asc
    support = np.sort(order[:k])
    n = nnz[0]
    got = ids[0, :n]
    assert np.all(np.diff(got) > 0)
    assert set(got.tolist()) <= set(support.tolist())
    assert np.all(c[0, :n] > 0) and c[0, :n].sum() == M
    assert np.all(ids[0, n:] == -1) and np.all(c[0, n:] == 0)
    # the same counts as a dense build restricted to that support
    xs = np.full(V, -np.inf, np.float32)
    xs[support] = x[support]
    cd, _, _, _ = oracle.q_build(xs[None])
    assert np.array_equal(cd[0, got], c[0, :n])
    assert cd[0].sum() == M and np.count_nonzero(cd[0]) == n


def test_topk_larger_than_support_equals_dense(oracle):
    x = np.full(300, -np.inf, np.float32)
    x[::7] = np.arange(43, dtype=np.float32) / 10
    cd, _, _, _ = oracle.q_build(x[None])
    cs, ids, nnz, _ = oracle.q_build(x[None], top_k=256)
    n = nnz[0]
    assert np.array_equal(cd[0, ids[0, :n]], cs[0, :n])
    assert np.count_nonzero(cd[0]) == n


# ------------------------------------------------------------ refusals
@pytest.mark.parametrize("bad,T,code", [
    ("nan", 1.0, 1), ("pinf", 1.0, 1), ("allninf", 1.0, 2), ("ok", 0.0, 4), ("ok", -1.0, 4),
    ("ok", float("inf"), 4), ("ok", float("nan"), 4), ("ok", 1e-39, 4), ("big", 0.5, 1)])
def test_refusals(oracle, bad, T, code):
    x = np.linspace(-3, 3, 64).astype(np.float32)
    if bad == "nan":
        x[5] = np.nan
    elif bad == "pinf":
        x[9] = np.inf
    elif bad == "allninf":
        x[:] = -np.inf
    elif bad == "big":
        x[3] = 3e38
    c, _, _, st = oracle.q_build(x[None], temperature=T)
    assert st[0] == code and c.sum() == 0
    c, ids, nnz, st = oracle.q_build(x[None], temperature=T, top_k=8)
    assert st[0] == code and c.sum() == 0 and nnz[0] == 0 and np.all(ids == -1)


def test_q_wire_sizes_match_the_page(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "q_sizes_depth5.json")))
    V, depth = g["vocab"], g["depth"]
    # dense counts are one 32-bit word per token (the page's FP32 q carries
    # the same number of words); sparse entries are (int32 id, 32-bit count)
    assert depth * V * 4 == g["dense_fp32_bytes_per_request"]
    assert 4 * depth * V * 4 == g["dense_fp32_bytes_per_four_requests"]
    for k, b in g["sparse_bytes_per_request"].items():
        assert depth * int(k) * 8 == b
    assert g["dense_tp2_shard_tokens"] * 2 == V
    assert depth * g["dense_tp2_shard_tokens"] * 4 == g["dense_tp2_shard_bytes_per_rank"]


# ------------------------------------------------------------- the draw
@pytest.mark.parametrize("which", ["dense8", "sparse", "onehot", "uniform3"])
def test_every_draw_enumerated(oracle, which):
    rng = np.random.default_rng(3)
    ids = None
    if which == "dense8":
        cuts = np.sort(rng.choice(np.arange(1, M), size=7, replace=False))
        counts = np.diff(np.concatenate([[0], cuts, [M]])).astype(np.uint32)
        counts[2] = 0
        counts[3] += np.uint32(np.diff(np.concatenate([[0], cuts, [M]]))[2])
    elif which == "sparse":
        ids = np.array([3, 17, 18, 40000, 129279], np.int32)
        counts = np.array([1, M - 10, 4, 3, 2], np.uint32)
    elif which == "onehot":
        counts = np.zeros(16, np.uint32)
        counts[9] = M
    else:
        counts = np.array([5592406, 5592405, 5592405], np.uint32)
    assert counts.sum() == M
    D = np.arange(M, dtype=np.uint32)
    tok = oracle.categorical_pick_many(counts, D, ids)
    keys = np.arange(counts.size) if ids is None else ids
    assert np.all(tok >= 0)
    for i, key in enumerate(keys):
        assert int((tok == key).sum()) == int(counts[i])
    # the draw is the first cumulative count strictly greater than D
    cum = np.cumsum(counts.astype(np.int64))
    edge = cum[:-1]
    edge = edge[edge < M]
    after = oracle.categorical_pick_many(counts, edge.astype(np.uint32), ids)
    nxt = np.searchsorted(cum, edge, side="right")
    assert np.array_equal(after, np.asarray(keys)[nxt])


def test_draft_sample_refuses_wrong_mass(oracle):
    counts = np.full((1, 8), 1 << 21, np.uint32)
    tok, st = oracle.draft_sample(counts, None, None, 0, 1, 1, seed=5)
    assert st[0] == 0 and 0 <= tok[0] < 8
    counts[0, 3] += 1
    tok, st = oracle.draft_sample(counts, None, None, 0, 1, 1, seed=5)
    assert st[0] == 5 and tok[0] == -1


@pytest.mark.slow
def test_c4_tie_rows_straddle_the_threshold(oracle):
    """C4's tied-argmax rows (1 % of the draft rows): with the stored tuner
    offsets the oracle splits every tied group at the grant threshold, some
    members getting the remaining ticket and the others not, the members
    granted being the lowest ids ("PP1 q transport and scheduling design",
    Distribution contract and precision: ties by lowest global token id)."""
    from draft_sampling_verification_gb300 import workloads as W
    wl = W.config4()
    assert wl.notes.get("tie_rows_straddling") == len(wl.notes["tie_rows"]) >= 12
    assert wl.notes.get("lowest_id_decisive_rows", 0) >= len(wl.notes["tie_rows"])
    for b, j, ids, tuners in wl.notes["tie_rows"]:
        x = wl.draft[b, j]
        assert np.all(x[ids] == x.max()) and np.isfinite(x[tuners]).all()
        counts, _, _, st = oracle.q_build(x[None, :], None, 0)
        c = counts[0, ids]
        assert st[0] == 0 and c.max() == c.min() + 1, (b, j, c)
        # the lowest ids of the group hold the extra ticket
        granted = c == c.max()
        assert np.all(granted[:int(granted.sum())]), (b, j, c)
