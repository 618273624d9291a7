"""GPU Monte Carlo of the committed-token distribution: the library's draft
draw, ratio verification and stochastic (match) verification over 10^7
requests that share one set of small-vocabulary rows, each request with its
own Philox counters.

"PP1 q transport and scheduling design": ratio tests and the full-vocabulary
residual must preserve the target p whatever q is, and the v2 message design
asks for independent CPU/GPU distribution and RNG tests.  "DeepSeek-V4.1
DSpark", State and sampling contracts: the stochastic verifier keeps the
target distribution.  So, for every position j, the token committed at j by
the requests that reach j follows p_j (the oracle's FP64 softmax of target
row j): a chi-square test per position.  The acceptance rate at position j
is the exact sum over v of min(p_j(v), q_j(v)) for the ratio test and of
p_j(v) q_j(v) for the match test: a binomial z test per position.  q comes
from the oracle's q build; the drafts are the library's own draws from it.
"""
import numpy as np
import pytest
import torch
from scipy.stats import chi2

import draft_sampling_verification_gb300 as ds
from oracle import oracle as O

pytestmark = pytest.mark.gpu

N_REQ = 10_000_000
DEPTH = 5
P_MIN = 1e-6   # smallest chi-square p-value accepted (the seeds are fixed)
Z_MAX = 5.0    # largest |z| of an acceptance rate


def rows(V, seed):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1.0, (DEPTH + 1, V)).astype(np.float32)
    xd = (zt[:DEPTH] + rng.normal(0, 0.7, (DEPTH, V))).astype(np.float32)
    counts, _, _, st = O.q_build(xd, None, 0)
    assert np.all(st == 0)
    p, _, pst = O.target_probs(zt)
    assert np.all(pst == 0)
    return zt, counts, p


def check(mode, p, q, acc, com):
    """Chi-square of the committed tokens at every position reached often
    enough, and the z test of each acceptance rate."""
    V = p.shape[1]
    reached = np.ones(acc.size, bool)
    for j in range(DEPTH + 1):
        n = int(reached.sum())
        if n < 50 * V:
            break
        tok = com[reached, j]
        assert tok.min() >= 0 and tok.max() < V
        obs = np.bincount(tok, minlength=V).astype(np.float64)
        exp = n * p[j]
        keep = exp > 0
        assert obs[~keep].sum() == 0, (mode, j, "a token of zero probability")
        stat = ((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum()
        pval = chi2.sf(stat, int(keep.sum()) - 1)
        assert pval > P_MIN, (mode, j, n, stat, pval)
        if j < DEPTH:
            a = np.minimum(p[j], q[j]).sum() if mode == "ratio" else (p[j] * q[j]).sum()
            k = int((acc[reached] > j).sum())
            z = (k - n * a) / np.sqrt(n * a * (1 - a))
            assert abs(z) < Z_MAX, (mode, j, n, k, a, z)
        reached &= acc > j


@pytest.mark.parametrize("V,seed", [(8, 71), (16, 72)])
def test_committed_tokens_follow_p(V, seed):
    zt, counts, p = rows(V, seed)
    q = counts.astype(np.float64) / float(1 << 24)
    dev = torch.device("cuda")
    t = torch.from_numpy(zt).to(dev).unsqueeze(0).expand(N_REQ, DEPTH + 1, V).reshape(
        N_REQ * (DEPTH + 1), V)
    c = torch.from_numpy(counts.view(np.int32)).to(dev).unsqueeze(0).expand(
        N_REQ, DEPTH, V).reshape(N_REQ * DEPTH, V)
    qd = {"counts": c, "ids": None, "nnz": None, "top_k": 0}
    run_seed = 1000 + V
    tok, sst = ds.draft_sample(qd, N_REQ, DEPTH, V, run_seed)
    torch.cuda.synchronize()
    assert int((sst != 0).sum()) == 0
    # the drafts themselves follow q at every position
    for j in range(DEPTH):
        obs = torch.bincount(tok[:, j].long(), minlength=V).cpu().numpy().astype(np.float64)
        exp = N_REQ * q[j]
        keep = exp > 0
        assert obs[~keep].sum() == 0
        stat = ((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum()
        assert chi2.sf(stat, int(keep.sum()) - 1) > P_MIN, ("draft", j, stat)
    for mode in ("ratio", "match"):
        if mode == "ratio":
            acc, com, fl, st = ds.verify_ratio(t, tok, qd, run_seed)
        else:
            acc, com, fl, st = ds.verify_match(t, tok, run_seed)
        torch.cuda.synchronize()
        assert int((st != 0).sum()) == 0
        check(mode, p, q, acc.cpu().numpy(), com.cpu().numpy())
    del t, c
    torch.cuda.empty_cache()


def test_negative_control_is_detected():
    """The same statistics reject a committed distribution that is not p:
    the drafts' own q (what a verifier that accepts every draft would
    commit) fails the chi-square at position 0."""
    V = 8
    zt, counts, p = rows(V, 71)
    q = counts.astype(np.float64) / float(1 << 24)
    dev = torch.device("cuda")
    c = torch.from_numpy(counts.view(np.int32)).to(dev).unsqueeze(0).expand(
        N_REQ // 10, DEPTH, V).reshape(N_REQ // 10 * DEPTH, V)
    qd = {"counts": c, "ids": None, "nnz": None, "top_k": 0}
    tok, _ = ds.draft_sample(qd, N_REQ // 10, DEPTH, V, 5)
    obs = torch.bincount(tok[:, 0].long(), minlength=V).cpu().numpy().astype(np.float64)
    exp = (N_REQ // 10) * p[0]
    stat = ((obs - exp) ** 2 / exp).sum()
    assert chi2.sf(stat, V - 1) < P_MIN
    assert np.abs(q[0] - p[0]).max() > 0.01
