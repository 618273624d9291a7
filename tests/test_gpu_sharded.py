"""GPU parity of the vocabulary-sharded q build and draft draw
(dspark_q_build_sample_sharded) with the unsharded one and the oracle:
counts (dense, or sparse ids / counts / nnz on a top-k support merged from
the ranks' local top-k), tokens and statuses bit for bit for 1, 2, 3 and 8
emulated ranks,
fp32 and bf16 rows, temperatures, refused rows, rows of massive exact ties
(the remaining tickets go to the lowest ids across the shard boundaries),
and the rows of a workload."""
import numpy as np
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from draft_sampling_verification_gb300 import workloads as W
from oracle import oracle as O
from parity import compare_verify, dev_inputs, np_, oracle_q, oracle_sample

pytestmark = pytest.mark.gpu


def rows(V, rng, n=2):
    out = []
    for _ in range(n):
        out.append(rng.normal(0, 2, V))
        z = -1.1 * np.log1p(rng.permutation(V)) + rng.normal(0, 0.3, V)
        out.append(z)
        zm = z.copy()
        zm[rng.random(V) < 0.3] = -np.inf
        out.append(zm)
    one = np.full(V, -np.inf)
    one[rng.integers(V)] = 1.0
    out.append(one)
    # exact ties: a flat row, and two levels in blocks that straddle shards
    out.append(np.zeros(V))
    out.append(np.where((np.arange(V) // 7) % 2 == 0, 0.0, 0.5))
    return np.array(out, np.float32)


def unsharded(x_dev, B, depth, seed, temps):
    q, tok = ds.q_build_sample(x_dev, B, depth, seed, temps, 0)
    return q, tok


@pytest.mark.parametrize("V", [5, 257, 4099, 129280])
@pytest.mark.parametrize("n_shards", [1, 2, 3, 8])
def test_sharded_equals_unsharded(oracle, V, n_shards):
    rng = np.random.default_rng(V * 10 + n_shards)
    x = rows(V, rng, n=1 if V > 10000 else 2)
    x = x[: (x.shape[0] // 1)]
    depth = 1
    B = x.shape[0]
    temps = rng.choice([1.0, 0.7, 1.3], B).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    tt = torch.from_numpy(temps).cuda()
    q1, t1 = unsharded(xd, B, depth, 17, tt)
    q2, t2 = ds.q_build_sample_sharded(xd, B, depth, n_shards, 17, tt)
    torch.cuda.synchronize()
    assert torch.equal(q2["status"], q1["status"])
    assert torch.equal(q2["counts"], q1["counts"])
    assert torch.equal(t2, t1)
    if V <= 4099:
        ref = O.q_build(x, temps, 0)
        assert np.array_equal(np_(q2["counts"]).view(np.uint32), ref[0])


def test_sharded_bf16_and_refusals(oracle):
    rng = np.random.default_rng(7)
    V = 4099
    x = rows(V, rng, n=1)
    x[0, 5] = np.nan
    x[1, :] = -np.inf
    x[2, 9] = 3e38
    temps = np.array([1.0, 1.0, 0.5, 0.0] + [1.0] * (x.shape[0] - 4), np.float32)
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    tt = torch.from_numpy(temps).cuda()
    B = x.shape[0]
    q1, t1 = unsharded(xd, B, 1, 3, tt)
    q2, t2 = ds.q_build_sample_sharded(xd, B, 1, 2, 3, tt)
    torch.cuda.synchronize()
    assert torch.equal(q2["status"], q1["status"])
    assert torch.equal(q2["counts"], q1["counts"]) and torch.equal(t2, t1)
    st = np_(q2["status"])
    assert st[0] == ds.ST_NONFINITE and st[1] == ds.ST_ZERO_MASS and st[3] == ds.ST_BAD_TEMPERATURE


def test_sharded_workload_rows(oracle):
    wl = W.config4(B=8)
    d, t, temps, req = dev_inputs(wl)
    q1, t1 = ds.q_build_sample(d, wl.B, wl.depth, wl.seed, temps, 0, req)
    q2, t2 = ds.q_build_sample_sharded(d, wl.B, wl.depth, 2, wl.seed, temps, request_ids=req)
    torch.cuda.synchronize()
    assert torch.equal(q2["status"], q1["status"])
    assert torch.equal(q2["counts"], q1["counts"])
    assert torch.equal(t2, t1)


def dense_of(counts, ids, nnz, V):
    out = np.zeros((counts.shape[0], V), np.uint32)
    for r in range(counts.shape[0]):
        n = int(nnz[r])
        out[r, ids[r, :n]] = counts[r, :n]
    return out


@pytest.mark.parametrize("V,k", [(5, 3), (257, 7), (4099, 256), (4099, 1024), (129280, 64),
                                 (129280, 1024)])
@pytest.mark.parametrize("n_shards", [1, 2, 3, 8])
def test_sharded_topk_equals_unsharded(oracle, V, k, n_shards):
    rng = np.random.default_rng(V * 31 + k + n_shards)
    x = rows(V, rng, n=1 if V > 10000 else 2)
    # ties at the cut: every id of a block shares one value
    tied = np.full(V, -3.0)
    tied[(np.arange(V) % 5) == 0] = 1.0
    x = np.vstack([x, tied[None, :].astype(np.float32)])
    B = x.shape[0]
    temps = rng.choice([1.0, 0.7, 1.3], B).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    tt = torch.from_numpy(temps).cuda()
    q1, t1 = ds.q_build_sample(xd, B, 1, 23, tt, k)
    q2, t2 = ds.q_build_sample_sharded(xd, B, 1, n_shards, 23, tt, top_k=k)
    torch.cuda.synchronize()
    assert torch.equal(q2["status"], q1["status"])
    assert torch.equal(q2["nnz"], q1["nnz"])
    assert torch.equal(q2["ids"], q1["ids"])
    assert torch.equal(q2["counts"], q1["counts"])
    assert torch.equal(t2, t1)
    if V <= 4099:
        ref, st = O.q_build_sharded(x, n_shards, temps, k)
        assert np.array_equal(np_(q2["status"]), st)
        got = dense_of(np_(q2["counts"]).view(np.uint32), np_(q2["ids"]), np_(q2["nnz"]), V)
        assert np.array_equal(got, ref)


def test_sharded_topk_refusals_and_workload(oracle):
    rng = np.random.default_rng(11)
    V = 4099
    x = rows(V, rng, n=1)
    x[0, 5] = np.nan
    x[1, :] = -np.inf
    x[2, 9] = 3e38
    temps = np.array([1.0, 1.0, 0.5, 0.0] + [1.0] * (x.shape[0] - 4), np.float32)
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    tt = torch.from_numpy(temps).cuda()
    B = x.shape[0]
    q1, t1 = ds.q_build_sample(xd, B, 1, 3, tt, 32)
    q2, t2 = ds.q_build_sample_sharded(xd, B, 1, 2, 3, tt, top_k=32)
    torch.cuda.synchronize()
    for key in ("status", "nnz", "ids", "counts"):
        assert torch.equal(q2[key], q1[key]), key
    assert torch.equal(t2, t1)
    st = np_(q2["status"])
    assert st[0] == ds.ST_NONFINITE and st[1] == ds.ST_ZERO_MASS and st[3] == ds.ST_BAD_TEMPERATURE
    wl = W.config3(B=8)
    d, t, temps, req = dev_inputs(wl)
    q1, t1 = ds.q_build_sample(d, wl.B, wl.depth, wl.seed, temps, wl.top_k, req)
    q2, t2 = ds.q_build_sample_sharded(d, wl.B, wl.depth, 2, wl.seed, temps, wl.top_k, req)
    torch.cuda.synchronize()
    for key in ("status", "nnz", "ids", "counts"):
        assert torch.equal(q2[key], q1[key]), key
    assert torch.equal(t2, t1)


@pytest.mark.parametrize("target", ["bf16", "f32"])
def test_cluster_verify_is_the_sharded_verifier(oracle, target):
    """The ratio verifier's cluster CTAs are the ranks of a vocabulary-sharded
    verifier: each combines its slice into (max, shifted sum) partials for p,
    and the residual draw picks the CTA by its residual mass, then the token
    inside.  With V = 129,280 the CTAs' slices (4 for bf16 rows, 8 for fp32)
    are the oracle's contiguous shards, and the outputs equal the sharded
    oracle's on every request outside the oracle's band.  q and
    drafts come from the oracle."""
    wl = W.config4(B=8)
    n_sh = 4 if target == "bf16" else 8
    _, t, _, req = dev_inputs(wl)
    if target == "f32":
        t = t.float()
    qref = oracle_q(wl)
    drafts = oracle_sample(wl, qref)[0].reshape(wl.B, wl.depth)
    counts = qref[0]
    q = {"counts": torch.from_numpy(counts.view(np.int32)).cuda(), "ids": None, "nnz": None,
         "top_k": 0}
    dd = torch.from_numpy(np.ascontiguousarray(drafts, np.int32)).cuda()
    g = ds.verify_ratio(t, dd, q, wl.seed, req)
    torch.cuda.synchronize()
    ref = O.verify_ratio_sharded(wl.target_f32(), drafts, counts, n_sh, wl.seed, wl.request_ids)
    c = compare_verify(g, ref, "ratio")
    assert c.mismatch == 0 and c.requests == wl.B, c
