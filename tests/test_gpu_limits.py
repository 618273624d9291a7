"""GPU parity at the ABI's limits: V = DSPARK_MAX_V (131,072), depth =
DSPARK_MAX_DEPTH (8), top_k = DSPARK_MAX_TOPK (1,024); the q build with its
draw, both verification modes, and the whole step in both schedules,
against the oracle (counts, tokens and greedy outputs bit for bit, ratio
outputs outside the oracle's tolerance band)."""
import numpy as np
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from oracle import oracle as O
from parity import compare_verify, np_

pytestmark = pytest.mark.gpu

V, DEPTH, K = 131072, 8, 1024


def inputs(B, seed):
    rng = np.random.default_rng(seed)
    perm = np.argsort(rng.random((B * DEPTH, V)), axis=1)
    xd = (-1.1 * np.log1p(perm) + rng.normal(0, 0.3, (B * DEPTH, V))).astype(np.float32)
    xd[:, rng.random(V) < 0.05] = -np.inf
    xt = np.empty((B, DEPTH + 1, V), np.float32)
    xt[:, :DEPTH] = xd.reshape(B, DEPTH, V) + rng.normal(0, 0.7, (B, DEPTH, V))
    xt[:, DEPTH] = rng.normal(0, 2, (B, V))
    bf = torch.from_numpy(xt).to(torch.bfloat16)
    return xd, bf, bf.float().numpy()


@pytest.mark.parametrize("top_k", [0, K])
def test_max_vocab_and_depth(oracle, top_k):
    B, seed = 3, 77
    xd, bf, zt = inputs(B, 5 + top_k)
    d = torch.from_numpy(xd).cuda()
    t = bf.cuda().reshape(B * (DEPTH + 1), V)
    req = torch.tensor([7, 1, 30000], dtype=torch.int32).cuda()
    q, tok = ds.q_build_sample(d, B, DEPTH, seed, None, top_k, req)
    torch.cuda.synchronize()
    counts, ids, nnz, st = O.q_build(xd, None, top_k)
    assert np.array_equal(np_(q["status"]), st)
    assert np.array_equal(np_(q["counts"]).view(np.uint32), counts)
    if top_k:
        assert np.array_equal(np_(q["ids"]), ids) and np.array_equal(np_(q["nnz"]), nnz)
    req_np = np.array([7, 1, 30000], np.uint32)
    drafts, sst = O.draft_sample(counts, ids, nnz, top_k, B, DEPTH, seed, req_np, V=V)
    assert np.array_equal(np_(tok).reshape(-1), drafts)
    drafts = drafts.reshape(B, DEPTH)
    g = ds.verify_greedy(t, tok)
    r = ds.verify_ratio(t, tok, q, seed, req)
    torch.cuda.synchronize()
    acc, com, gst = O.verify_greedy(zt, drafts)
    assert np.array_equal(np_(g[0]), acc) and np.array_equal(np_(g[1]), com)
    assert np.array_equal(np_(g[2]), gst)
    ref = O.verify_ratio(zt, drafts, counts, ids, nnz, top_k, seed, req_np)
    c = compare_verify(r, ref, "ratio")
    assert c.mismatch == 0 and c.requests == B, c


@pytest.mark.parametrize("schedule", [ds.SCHEDULE_ONE_LAUNCH, ds.SCHEDULE_SEPARATE])
def test_max_sizes_whole_step(oracle, schedule):
    B, seed = 3, 91
    xd, bf, zt = inputs(B, 11)
    d = torch.from_numpy(xd).cuda()
    t = bf.cuda().reshape(B * (DEPTH + 1), V)
    q, tok, outs = ds.spec_step(d, t, B, DEPTH, seed, None, None, ("greedy", "ratio"),
                                schedule=schedule)
    torch.cuda.synchronize()
    counts, _, _, st = O.q_build(xd, None, 0)
    assert np.array_equal(np_(q["counts"]).view(np.uint32), counts)
    drafts, _ = O.draft_sample(counts, None, None, 0, B, DEPTH, seed, None, V=V)
    assert np.array_equal(np_(tok).reshape(-1), drafts)
    acc, com, gst = O.verify_greedy(zt, drafts.reshape(B, DEPTH))
    ga, gc, gs = outs["greedy"]
    assert np.array_equal(np_(ga), acc) and np.array_equal(np_(gc), com)
    ref = O.verify_ratio(zt, drafts.reshape(B, DEPTH), counts, None, None, 0, seed, None)
    c = compare_verify(outs["ratio"], ref, "ratio")
    assert c.mismatch == 0, c
