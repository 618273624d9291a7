"""The oracle's stochastic (match) verifier ("DeepSeek-V4.1 DSpark", State and
sampling contracts: each row draws from the target's p with its own noise, a
matching proposal is accepted, the first mismatch stops verification and
commits the draw).  Pins: the committed tokens follow p position by position
(chi-square at the request level, as for the ratio verifier); the acceptance
rate equals sum_x q(x) p(x), the probability that an independent draw from p
equals a draft drawn from q; the extremes (p on the draft: every proposal
accepted; p away from it: none); a row after the mismatch is never read."""
import numpy as np
import pytest

from oracle import oracle as O

M = 1 << 24


def setup(rng, V=8, depth=2, B=20000, seed=31):
    zt = rng.normal(0, 1.0, (depth + 1, V)).astype(np.float32)
    p, _, _ = O.target_probs(zt)
    xd = rng.normal(0, 1.0, (depth, V)).astype(np.float32)
    counts, _, _, _ = O.q_build(xd)
    qrep = np.tile(counts, (B, 1))
    drafts, st = O.draft_sample(qrep, None, None, 0, B, depth, seed=seed)
    assert np.all(st == 0)
    z = np.broadcast_to(zt, (B, depth + 1, V))
    return zt, p, counts, drafts.reshape(B, depth), z


def chi2(samples, probs):
    n = samples.size
    h = np.bincount(samples, minlength=probs.size)
    keep = probs * n > 5
    x2 = (((h - probs * n) ** 2) / np.maximum(probs * n, 1e-12))[keep].sum()
    return x2, keep.sum() - 1


def test_match_verifier_preserves_p(oracle):
    rng = np.random.default_rng(41)
    zt, p, counts, drafts, z = setup(rng)
    acc, com, fl, st = O.verify_match(z, drafts, seed=42)
    assert np.all(st == 0)
    for pos, cond in [(0, acc >= 0), (1, acc >= 1), (2, acc >= 2)]:
        x2, dof = chi2(com[cond, pos], p[pos])
        assert x2 < dof + 6 * np.sqrt(2 * dof), (pos, x2, dof)
    B = acc.size
    for b in range(300):
        L = acc[b]
        assert np.array_equal(com[b, :L], drafts[b, :L])
        assert np.all(com[b, L + 1:] == -1)
        # a rejection commits a token other than the draft it rejected
        if L < drafts.shape[1]:
            assert com[b, L] != drafts[b, L]


def test_match_acceptance_rate(oracle):
    rng = np.random.default_rng(43)
    zt, p, counts, drafts, z = setup(rng, B=40000)
    acc, com, fl, st = O.verify_match(z, drafts, seed=44)
    q0 = counts[0] / float(M)
    rate = float((q0 * p[0]).sum())
    n = acc.size
    got = float((acc >= 1).mean())
    assert abs(got - rate) < 5 * np.sqrt(rate * (1 - rate) / n), (got, rate)


def test_match_extremes(oracle):
    V, depth, B = 16, 3, 64
    rng = np.random.default_rng(45)
    drafts = rng.integers(0, V, (B, depth)).astype(np.int32)
    z = np.full((B, depth + 1, V), -30.0, np.float32)
    for b in range(B):
        for j in range(depth):
            z[b, j, drafts[b, j]] = 30.0         # p all but one-hot on the draft
        z[b, depth, 5] = 30.0
    acc, com, fl, st = O.verify_match(z, drafts, seed=46)
    assert np.all(st == 0) and np.all(acc == depth)
    assert np.all(com[:, depth] == 5)
    z2 = np.full((B, depth + 1, V), 0.0, np.float32)
    for b in range(B):
        z2[b, 0, drafts[b, 0]] = -np.inf         # the first draft is impossible
    acc, com, fl, st = O.verify_match(z2, drafts, seed=47)
    assert np.all(st == 0) and np.all(acc == 0)
    assert np.all(com[np.arange(B), 0] != drafts[:, 0])


def test_match_stops_reading(oracle):
    V, depth = 16, 3
    drafts = np.array([[1, 2, 3]], np.int32)
    z = np.full((1, depth + 1, V), 0.0, np.float32)
    z[0, 0, 1] = -np.inf                          # row 0 cannot match: L = 0
    z[0, 2, 4] = np.nan                           # a later row is never read
    acc, com, fl, st = O.verify_match(z, drafts, seed=48)
    assert st[0] == 0 and acc[0] == 0
    z[0, 0, 7] = np.nan                           # the row read is refused
    acc, com, fl, st = O.verify_match(z, drafts, seed=48)
    assert st[0] == O.NONFINITE and acc[0] == 0 and np.all(com[0] == -1)
    bad = np.array([[1, V, 3]], np.int32)
    acc, com, fl, st = O.verify_match(np.zeros((1, depth + 1, V), np.float32), bad, seed=48)
    assert st[0] == O.BAD_DRAFT
