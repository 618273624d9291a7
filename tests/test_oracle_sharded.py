"""The oracle's vocabulary-sharded emulator ("PP1 q transport and scheduling
design", Sparse support and vocabulary-sharded TP2 follow-up) equals the
unsharded functions: the same counts for dense and top-k rows (all-reduce
max and sums, a globally coordinated remaining-ticket grant, the merge of
the shards' local top-k), the same draft draw (the shard chosen by its count
total), and the same ratio-verification outputs (p from (max, shifted sum)
partials, the residual shard chosen by its residual mass) -- for 1, 2, 3, 4
and 7 shards, on rows with ties, masks, a single finite logit and ragged
shard sizes."""
import numpy as np
import pytest

from oracle import oracle as O

M = 1 << 24


def rows(V, rng, n=2):
    out = []
    for _ in range(n):
        out.append(rng.normal(0, 2, V))
        z = -1.1 * np.log1p(rng.permutation(V)) + rng.normal(0, 0.3, V)
        out.append(z)
        zm = z.copy()
        zm[rng.random(V) < 0.3] = -np.inf
        out.append(zm)
        out.append(np.round(rng.normal(0, 2, V) * 4) / 4)   # exact ties
    out.append(np.zeros(V))
    one = np.full(V, -np.inf)
    one[rng.integers(V)] = 1.0
    out.append(one)
    return np.array(out, np.float32)


def dense_of(counts, ids, nnz, V):
    out = np.zeros((counts.shape[0], V), np.uint32)
    for r in range(counts.shape[0]):
        n = int(nnz[r])
        out[r, ids[r, :n]] = counts[r, :n]
    return out


@pytest.mark.parametrize("V", [7, 64, 1001])
@pytest.mark.parametrize("top_k", [0, 5, 40])
def test_sharded_q_equals_unsharded(oracle, V, top_k):
    if top_k > V:
        pytest.skip("top_k > V")
    rng = np.random.default_rng(V + top_k)
    x = rows(V, rng)
    temps = rng.choice([1.0, 0.7, 1.3], x.shape[0]).astype(np.float32)
    c, ids, nnz, st = O.q_build(x, temps, top_k)
    ref = c if top_k == 0 else dense_of(c, ids, nnz, V)
    for n_sh in (1, 2, 3, 4, 7):
        cs, sts = O.q_build_sharded(x, n_sh, temps, top_k)
        assert np.array_equal(sts, st), n_sh
        assert np.array_equal(cs, ref), n_sh


def test_sharded_draw_equals_unsharded(oracle):
    rng = np.random.default_rng(3)
    V = 1001
    x = rows(V, rng, n=1)
    c, _, _, st = O.q_build(x)
    D = np.concatenate([[0, M - 1], rng.integers(0, M, 300)]).astype(np.uint32)
    for r in range(c.shape[0]):
        if st[r] != 0:
            continue
        for n_sh in (2, 3, 7):
            got = np.array([O.draw_sharded(c[r], n_sh, d) for d in D])
            want = np.array([int(np.searchsorted(np.cumsum(c[r].astype(np.uint64)), d,
                                                 side="right")) for d in D])
            assert np.array_equal(got, want), (r, n_sh)


def test_sharded_ratio_verification_equals_unsharded(oracle):
    rng = np.random.default_rng(4)
    B, depth, V = 40, 5, 333
    xd = rng.normal(0, 1.5, (B, depth, V)).astype(np.float32)
    counts, _, _, st = O.q_build(xd.reshape(-1, V))
    assert np.all(st == 0)
    drafts, sst = O.draft_sample(counts, None, None, 0, B, depth, seed=7)
    zt = np.concatenate([xd, rng.normal(0, 1.5, (B, 1, V)).astype(np.float32)], axis=1)
    zt = (zt + rng.normal(0, 0.7, zt.shape)).astype(np.float32)
    ref = O.verify_ratio(zt, drafts.reshape(B, depth), counts, None, None, 0, seed=8)
    for n_sh in (2, 3, 4):
        got = O.verify_ratio_sharded(zt, drafts.reshape(B, depth), counts, n_sh, seed=8)
        flagged = ((got[2] & 3) != 0) | ((ref[2] & 3) != 0)
        same = (got[0] == ref[0]) & (got[1] == ref[1]).all(axis=1) & (got[3] == ref[3])
        assert np.all(same | flagged), n_sh
        assert same.sum() >= B - 1
