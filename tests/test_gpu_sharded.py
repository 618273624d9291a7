"""GPU parity of the vocabulary-sharded q build and draft draw
(dspark_q_build_sample_sharded) with the unsharded one and the oracle:
counts, tokens and statuses bit for bit for 1, 2, 3 and 8 emulated ranks,
fp32 and bf16 rows, temperatures, refused rows, rows of massive exact ties
(the remaining tickets go to the lowest ids across the shard boundaries),
and the rows of a workload."""
import numpy as np
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from draft_sampling_verification_gb300 import workloads as W
from oracle import oracle as O
from parity import dev_inputs, np_

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
    q2, t2 = ds.q_build_sample_sharded(d, wl.B, wl.depth, 2, wl.seed, temps, req)
    torch.cuda.synchronize()
    assert torch.equal(q2["status"], q1["status"])
    assert torch.equal(q2["counts"], q1["counts"])
    assert torch.equal(t2, t1)
