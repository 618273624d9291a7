"""GPU parity of the Markov-conditioned draft chain (dspark_q_chain_sample)
against the oracle, bit for bit: counts, draft tokens, statuses and margins,
for fp32 and bf16 base logits, with and without a bias table, with
temperatures, for a bias that forces the next token, ragged vocabularies and
refused rows."""
import numpy as np
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from oracle import oracle as O
from parity import np_

pytestmark = pytest.mark.gpu


def run(x, bias, anchors, seed, temps=None, bf16=False):
    B, depth, V = x.shape
    xh = torch.from_numpy(x.reshape(B * depth, V))
    if bf16:  # rounded on the host; the oracle reads the widened bf16 rows
        xh = xh.to(torch.bfloat16)
        x = xh.float().numpy().reshape(B, depth, V)
    xd = xh.cuda()
    bt = None if bias is None else torch.from_numpy(bias).cuda()
    tt = None if temps is None else torch.from_numpy(temps).cuda()
    at = torch.from_numpy(np.asarray(anchors, np.int32)).cuda()
    q, tok, mg = ds.q_chain_sample(xd, B, depth, seed, at, bt, tt)
    torch.cuda.synchronize()
    ref = O.q_chain(x, temps, bias, np.asarray(anchors), seed)
    return (np_(q["counts"]).view(np.uint32), np_(tok), np_(q["status"]), np_(mg)), ref


def check(g, ref):
    gc, gt, gs, gm = g
    rc, rt, rs, rm = ref
    assert np.array_equal(gs, rs), (gs, rs)
    assert np.array_equal(gt, rt), (gt, rt)
    bad = np.flatnonzero((gc != rc).any(axis=1))
    assert bad.size == 0, bad[:8]
    assert np.array_equal(gm.view(np.uint32), rm.view(np.uint32)), (gm, rm)


@pytest.mark.parametrize("V,bf16,with_bias", [(300, False, True), (4099, False, True),
                                              (129280, False, True), (129280, True, True),
                                              (4099, False, False)])
def test_chain_matches_oracle(oracle, V, bf16, with_bias):
    rng = np.random.default_rng(V + int(bf16))
    B, depth = 3, 5
    x = rng.normal(0, 2, (B, depth, V)).astype(np.float32)
    x[1, 2] = np.round(x[1, 2] * 2) / 2                # ties in one row
    bias = rng.normal(0, 1.5, (7, V)).astype(np.float32) if with_bias else None
    temps = rng.choice([1.0, 0.7, 1.3], B * depth).astype(np.float32)
    g, ref = run(x, bias, rng.integers(0, V, B), 21, temps, bf16)
    check(g, ref)


def test_chain_follows_forced_map(oracle):
    V, depth, B = 64, 5, 4
    f = (np.arange(V) * 7 + 3) % V
    bias = np.zeros((V, V), np.float32)
    bias[np.arange(V), f] = 40.0
    x = np.zeros((B, depth, V), np.float32)
    anchors = np.arange(B) * 5 + 1
    g, ref = run(x, bias, anchors, 13)
    check(g, ref)
    prev = anchors
    for j in range(depth):
        assert np.array_equal(g[1][:, j], f[prev])
        prev = g[1][:, j]


def test_chain_refusals(oracle):
    rng = np.random.default_rng(5)
    B, depth, V = 3, 4, 1000
    x = rng.normal(0, 1, (B, depth, V)).astype(np.float32)
    x[0, 1, 7] = np.nan
    x[2, 3, :] = -np.inf
    g, ref = run(x, rng.normal(0, 1, (3, V)).astype(np.float32), [0, V, 5], 5)
    check(g, ref)
    st = g[2].reshape(B, depth)
    assert st[0, 0] == 0 and np.all(st[0, 1:] == ds.ST_NONFINITE)
    assert np.all(st[1] == ds.ST_BAD_DRAFT)
    assert st[2, 3] == ds.ST_ZERO_MASS
