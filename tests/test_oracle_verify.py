"""Pins of the oracle's target p, greedy verifier and ratio verifier.

"PP1 q transport and scheduling design": ratio tests and full-vocabulary
residual sampling with the target p and the dyadic q must preserve p ("q can
approximate the draft arbitrarily poorly and still preserve p under correct
verification"), and the CPU suite carries a toy selection-bias regression
(uniform q = p; admitting the first draw only when it is token 0 gives output
mass 3/4 instead of 1/2).  "DeepSeek-V4.1 DSpark", State and sampling
contracts: greedy verification matches the target argmax.

Pins: p against scipy's softmax; every acceptance draw enumerated; the exact
measure of every residual pick found by bisection over the 32-bit draw; the
committed-token distribution on V = 8, depth 2 computed exactly from those
measures and compared with p; a Monte Carlo run of the request-level
verifier; the selection-bias negative control.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import softmax

M = 1 << 24


# ------------------------------------------------------------- target p
def test_target_p_matches_scipy_softmax(oracle):
    rng = np.random.default_rng(1)
    z = rng.normal(0, 3, (4, 4099)).astype(np.float32)
    z[1, rng.random(4099) < 0.2] = -np.inf
    z[2, :] = -np.inf
    z[2, 17] = 4.0
    p, am, st = oracle.target_probs(z)
    assert np.all(st == 0)
    for r in range(4):
        zr = z[r].astype(np.float64)
        ref = softmax(np.where(np.isfinite(zr), zr, -np.inf))
        assert np.abs(p[r] - ref).max() <= 1e-15
        assert am[r] == int(np.argmax(zr))  # numpy returns the first maximum
    assert p[1][~np.isfinite(z[1])].max() == 0.0
    assert p[2, 17] == 1.0


def test_target_argmax_ties_to_lowest_id(oracle):
    z = np.zeros((1, 64), np.float32)
    z[0, [7, 3, 50]] = 2.0
    _, am, _ = oracle.target_probs(z)
    assert am[0] == 3


@pytest.mark.parametrize("bad,code", [("nan", 1), ("pinf", 1), ("allninf", 2)])
def test_target_refusals(oracle, bad, code):
    z = np.zeros((1, 16), np.float32)
    if bad == "nan":
        z[0, 4] = np.nan
    elif bad == "pinf":
        z[0, 4] = np.inf
    else:
        z[:] = -np.inf
    _, am, st = oracle.target_probs(z)
    assert st[0] == code and am[0] == -1


# ------------------------------------------------------------ ratio test
@pytest.mark.parametrize("P,c", [(1, 1), (3, 7), (M // 3, M // 2), (5000, 1 << 20), (M, M),
                                 (M - 1, M), (123457, 99991), (0, 5)])
def test_every_acceptance_draw_enumerated(oracle, P, c):
    # p = P / 2^24 is exact; the accepted draws are U < P*2^24/c
    U = np.arange(M, dtype=np.uint32)
    acc = oracle.ratio_accept_many(U, c, P / float(M))
    expect = min(M, -(-(P * M) // c))
    assert int(acc.sum()) == expect
    assert np.all(acc[:expect]) and not np.any(acc[expect:])


# ------------------------------------------------- residual pick measures
def pick_measure(oracle, p, c):
    """Exact fraction of the 2^32 residual draws that pick each token."""
    V = p.size
    def pick(w):
        return oracle.residual_pick(p, c, w)[0]
    # pick(w) is non-decreasing in w: bisect the first w reaching each token
    first = np.zeros(V + 1, np.int64)
    first[V] = 1 << 32
    for v in range(1, V):
        lo, hi = 0, 1 << 32  # pick(lo-1) < v <= pick(hi) (hi virtual)
        while lo < hi:
            mid = (lo + hi) // 2
            if pick(mid) >= v:
                hi = mid
            else:
                lo = mid + 1
        first[v] = lo
    first[0] = 0
    return np.diff(first) / float(1 << 32)


def test_residual_pick_measures(oracle):
    rng = np.random.default_rng(2)
    V = 8
    p = softmax(rng.normal(0, 1.5, V))
    counts = np.array([0, M // 2, M // 4, 0, M // 8, M // 16, M // 16, 0], np.uint32)
    q = counts / float(M)
    r = np.maximum(p - q, 0)
    meas = pick_measure(oracle, p, counts)
    assert np.abs(meas - r / r.sum()).max() <= 2.0 ** -31
    # bonus draw: the weights are p itself
    meas = pick_measure(oracle, p, None)
    assert np.abs(meas - p).max() <= 2.0 ** -31
    # zero residual mass: draws from p, flagged degenerate
    onehot = np.zeros(V)
    onehot[3] = 1.0
    c = np.zeros(V, np.uint32)
    c[3] = M
    tok, fl = oracle.residual_pick(onehot, c, 12345)
    assert tok == 3 and fl & oracle.FLAG_DEGENERATE


def band_runs(oracle, p, c, first, bit):
    """Lengths (in draws) of the runs of draws flagged `bit` at the start and at
    the end of each token's run of draws [first[v], first[v+1])."""
    def fl(w):
        return oracle.residual_pick(p, c, w)[1] & bit
    out = []
    for v in range(p.size):
        a, e = int(first[v]), int(first[v + 1])
        if e <= a:
            out.append((0, 0))
            continue
        mid = (a + e) // 2
        lo, hi = a, mid  # first unflagged draw of the leading run
        while lo < hi:
            m = (lo + hi) // 2
            if fl(m):
                lo = m + 1
            else:
                hi = m
        lead = lo - a
        lo, hi = mid, e  # first draw of the trailing run
        while lo < hi:
            m = (lo + hi) // 2
            if fl(m):
                hi = m
            else:
                lo = m + 1
        out.append((lead, e - lo))
    return np.array(out, np.int64)


def test_boundary_band_measures(oracle):
    """The two readings of "a draw within 1e-6 of a cumulative boundary".
    Absolute: every edge carries a band of 1e-6 (probability units) on each
    side, whatever the token's mass.  Relative: the band of a token's edges is
    1e-6 of that token's own mass, so a uniform draw falls in it with
    probability 2e-6 on any row; it lies inside the absolute band."""
    # dyadic masses: every edge sits exactly on a draw, Z = 1
    p = np.array([2.0 ** -1, 2.0 ** -3, 2.0 ** -3, 2.0 ** -6, 2.0 ** -4, 2.0 ** -6, 2.0 ** -5,
                  2.0 ** -3])
    assert p.sum() == 1.0
    first = np.concatenate([[0], np.cumsum(p) * 2.0 ** 32]).astype(np.int64)
    rel = band_runs(oracle, p, None, first, oracle.FLAG_NEAR_BOUNDARY_REL)
    ab = band_runs(oracle, p, None, first, oracle.FLAG_NEAR_BOUNDARY)
    width = 1e-6 * 2.0 ** 32  # draws per 1e-6 of probability
    # absolute band: the same run at every edge
    assert np.all(np.abs(ab - width) <= 1.5)
    # relative band: runs proportional to the token's own mass, both ends
    assert np.all(np.abs(rel - p[:, None] * width) <= 1.5)
    assert abs(rel.sum() / 2.0 ** 32 - 2e-6) <= p.size * 2 * 2.0 ** -32
    assert np.all(rel <= ab)
    # residual weights max(p - q, 0): a token's band follows its residual mass
    c = np.zeros(8, np.uint32)
    c[0] = 1 << 23          # q(0) = 1/2 = p(0): no residual, no band
    c[2] = 1 << 20          # q(2) = 1/16: residual 1/16
    c[4] = (1 << 20) + (1 << 19)  # q(4) = 3/32 > p(4): no residual
    r = np.maximum(p - c / float(M), 0.0)
    Z = r.sum()
    first_r = np.concatenate([[0], np.cumsum(r / Z) * 2.0 ** 32]).astype(np.int64)
    rel_r = band_runs(oracle, p, c, first_r, oracle.FLAG_NEAR_BOUNDARY_REL)
    assert np.all(rel_r[r == 0] == 0)
    t_width = 1e-6 / Z * 2.0 ** 32  # t = w * 2^-32 * Z
    assert np.all(np.abs(rel_r - r[:, None] * t_width) <= 1.5)


# ----------------------------------- exact committed distribution, V = 8
def accept_prob(oracle, c, p):
    U = np.arange(M, dtype=np.uint32)
    return oracle.ratio_accept_many(U, int(c), float(p)).mean()


def row_committed_dist(oracle, p, counts):
    """Distribution of the token committed at one row: the draft d ~ q,
    accepted with the enumerated probability, else the residual pick."""
    q = counts / float(M)
    res = pick_measure(oracle, p, counts)
    out = np.zeros(p.size)
    acc_total = 0.0
    for d in range(p.size):
        if counts[d] == 0:
            continue
        a = accept_prob(oracle, counts[d], p[d])
        out[d] += q[d] * a
        out += q[d] * (1 - a) * res
        acc_total += q[d] * a
    return out, acc_total


@pytest.mark.slow
def test_ratio_verifier_preserves_p_exactly(oracle):
    rng = np.random.default_rng(8)
    V, depth = 8, 2
    zt = rng.normal(0, 1.5, (depth + 1, V)).astype(np.float32)
    zt[1, 6] = -np.inf  # a token the target forbids
    p, _, st = oracle.target_probs(zt)
    assert np.all(st == 0)
    xd = rng.normal(0, 1.5, (depth, V)).astype(np.float32)
    xd[0, 2] = -np.inf  # a token the draft never proposes
    counts, _, _, qst = oracle.q_build(xd)
    assert np.all(qst == 0)
    d0, acc0 = row_committed_dist(oracle, p[0], counts[0])
    d1, acc1 = row_committed_dist(oracle, p[1], counts[1])
    bonus = pick_measure(oracle, p[2], None)
    # position 0 ~ p_0; position 1, given the first draft accepted, ~ p_1;
    # the bonus, given both accepted, ~ p_2
    assert np.abs(d0 - p[0]).max() <= 1e-6
    assert np.abs(d1 - p[1]).max() <= 1e-6
    assert np.abs(bonus - p[2]).max() <= 1e-6
    assert 0.05 < acc0 < 1.0 and 0.05 < acc1 < 1.0


def test_ratio_verifier_request_level_monte_carlo(oracle):
    rng = np.random.default_rng(9)
    V, depth, B = 8, 2, 30000
    zt = rng.normal(0, 1.0, (depth + 1, V)).astype(np.float32)
    p, _, _ = oracle.target_probs(zt)
    xd = rng.normal(0, 1.0, (depth, V)).astype(np.float32)
    counts, _, _, _ = oracle.q_build(xd)
    qrep = np.tile(counts, (B, 1))
    drafts, st = oracle.draft_sample(qrep, None, None, 0, B, depth, seed=77)
    assert np.all(st == 0)
    z = np.broadcast_to(zt, (B, depth + 1, V))
    acc, com, flags, vst = oracle.verify_ratio(z, drafts.reshape(B, depth), qrep, None, None, 0,
                                               seed=78)
    assert np.all(vst == 0)
    assert np.all(com[np.arange(B), acc] >= 0)

    def chi2(samples, probs):
        n = samples.size
        h = np.bincount(samples, minlength=V)
        keep = probs * n > 5
        return (((h - probs * n) ** 2) / np.maximum(probs * n, 1e-12))[keep].sum(), keep.sum() - 1

    for pos, cond in [(0, acc >= 0), (1, acc >= 1), (2, acc >= 2)]:
        x2, dof = chi2(com[cond, pos], p[pos])
        assert x2 < dof + 6 * np.sqrt(2 * dof), (pos, x2, dof)
    # the accepted drafts are the drafts, and nothing after the commit
    for b in range(200):
        L = acc[b]
        assert np.array_equal(com[b, :L], drafts.reshape(B, depth)[b, :L])
        assert np.all(com[b, L + 1:] == -1)


def test_selection_bias_negative_control(oracle, golden_dir):
    """The distribution check must flag the page's selection-biased policy."""
    g = json.load(open(os.path.join(golden_dir, "selection_bias_toy.json")))
    p = np.array([0.5, 0.5])
    counts = np.array([M // 2, M // 2], np.uint32)
    q = counts / float(M)
    # correct fixed-depth verification (depth 1): the committed first token
    correct, _ = row_committed_dist(oracle, p, counts)
    # planted mistake: admit the draft only when it is token 0, else fall
    # back to target-only sampling from p
    biased = np.zeros(2)
    biased[0] += q[0] * 1.0
    biased += q[1] * p
    assert abs(correct[0] - g["correct_output_mass_token0"]) <= 1e-6
    assert abs(biased[0] - g["biased_output_mass_token0"]) <= 1e-12
    assert np.abs(correct - p).max() <= 1e-6      # the check accepts the verifier
    assert np.abs(biased - p).max() > 0.2         # and rejects the biased policy


def test_ratio_special_cases(oracle):
    V = 16
    # q one-hot on x with p(x) = 1: always accepted
    z = np.full((2, V), -np.inf, np.float32)
    z[0, 5] = 0.0
    z[1, :] = 0.0
    c = np.zeros((1, V), np.uint32)
    c[0, 5] = M
    for seed in range(50):
        acc, com, fl, st = oracle.verify_ratio(z[None], np.array([[5]]), c, None, None, 0, seed)
        assert st[0] == 0 and acc[0] == 1 and com[0, 0] == 5
    # p(x) = 0: always rejected, and the correction is drawn from p itself
    z2 = np.zeros((2, V), np.float32)
    z2[0, 5] = -np.inf
    p, _, _ = oracle.target_probs(z2)
    meas = pick_measure(oracle, p[0], c[0])
    assert np.abs(meas - p[0]).max() <= 2.0 ** -31
    for seed in range(50):
        acc, com, fl, st = oracle.verify_ratio(z2[None], np.array([[5]]), c, None, None, 0, seed)
        assert st[0] == 0 and acc[0] == 0 and com[0, 0] != 5 and com[0, 1] == -1


def test_ratio_refusals(oracle):
    V, depth = 16, 2
    z = np.zeros((1, depth + 1, V), np.float32)
    c = np.full((depth, V), M // V, np.uint32)
    d = np.array([[1, 2]], np.int32)
    # draft out of range
    _, com, _, st = oracle.verify_ratio(z, np.array([[1, 16]]), c, None, None, 0, 0)
    assert st[0] == oracle.BAD_DRAFT and np.all(com == -1)
    # zero q at the proposed token
    c0 = c.copy()
    c0[0, 1] = 0
    c0[0, 2] += M // V
    _, com, _, st = oracle.verify_ratio(z, d, c0, None, None, 0, 0)
    assert st[0] == oracle.BAD_DRAFT and np.all(com == -1)
    # non-finite target row
    zb = z.copy()
    zb[0, 0, 3] = np.nan
    acc, com, _, st = oracle.verify_ratio(zb, d, c, None, None, 0, 0)
    assert st[0] == oracle.NONFINITE and acc[0] == 0 and np.all(com == -1)
    # sparse q with unsorted ids
    ids = np.array([[2, 1] + [-1] * 2, [1, 2] + [-1] * 2], np.int32)
    sc = np.array([[M // 2, M // 2, 0, 0], [M // 2, M // 2, 0, 0]], np.uint32)
    nnz = np.array([2, 2], np.int32)
    _, com, _, st = oracle.verify_ratio(z, d, sc, ids, nnz, 4, 0)
    assert st[0] == oracle.BAD_Q


# ---------------------------------------------------------------- greedy
def test_greedy_all_accept_and_first_mismatch(oracle):
    rng = np.random.default_rng(4)
    V, depth = 4099, 5
    z = rng.normal(0, 2, (3, depth + 1, V)).astype(np.float32)
    am = z.argmax(axis=2).astype(np.int32)
    drafts = am[:, :depth].copy()
    drafts[1, 3] = (drafts[1, 3] + 1) % V
    drafts[2, 0] = (drafts[2, 0] + 7) % V
    acc, com, st = oracle.verify_greedy(z, drafts)
    assert np.all(st == 0)
    assert acc.tolist() == [5, 3, 0]
    assert com[0].tolist() == am[0].tolist()
    assert com[1].tolist() == am[1, :4].tolist() + [-1, -1]
    assert com[2].tolist() == [am[2, 0]] + [-1] * 5


def test_greedy_stops_reading_after_mismatch(oracle):
    V, depth = 32, 3
    z = np.zeros((1, depth + 1, V), np.float32)
    z[0, :, 4] = 1.0
    z[0, 2, :] = np.nan  # never reached: mismatch at row 1
    acc, com, st = oracle.verify_greedy(z, np.array([[4, 5, 4]], np.int32))
    assert st[0] == 0 and acc[0] == 1 and com[0].tolist() == [4, 4, -1, -1]
    acc, com, st = oracle.verify_greedy(z, np.array([[4, 4, 4]], np.int32))
    assert st[0] == oracle.NONFINITE and acc[0] == 0 and np.all(com == -1)
