"""GPU parity of q construction and the draft draw against the oracle:
bit-exact counts, sparse ids, nnz, statuses and tokens, on random rows of
many lengths (ragged slices, a single element, full vocabulary), strided and
unaligned rows, bf16 logits, the degenerate and refused rows, and the draft
rows of every workload."""
import numpy as np
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from draft_sampling_verification_gb300 import workloads as W
from parity import compare_q, np_

pytestmark = pytest.mark.gpu

M = 1 << 24


def rows_for(V, rng, n_each=2):
    out = []
    for _ in range(n_each):
        out.append(rng.normal(0, 2, V))
        out.append(rng.normal(0, 9, V))
        z = -1.1 * np.log1p(rng.permutation(V)) + rng.normal(0, 0.3, V)
        out.append(z)
        zm = z.copy()
        zm[rng.random(V) < 0.3] = -np.inf
        if np.isfinite(zm).sum() == 0:
            zm[0] = 0.0
        out.append(zm)
        out.append(np.round(rng.normal(0, 2, V) * 4) / 4)   # heavy exact ties
    out.append(np.zeros(V))                                   # uniform row
    one = np.full(V, -np.inf)
    one[rng.integers(V)] = 3.0
    out.append(one)                                           # one finite logit
    return np.array(out, np.float32)


def run_q(x, temps, top_k, ld_pad=0, dtype=torch.float32, offset=0):
    n, V = x.shape
    buf = torch.zeros(n * (V + ld_pad) + offset + 8, dtype=torch.float32, device="cuda")
    view = buf[offset:offset + n * (V + ld_pad)].view(n, V + ld_pad)[:, :V]
    view.copy_(torch.from_numpy(x))
    if dtype == torch.bfloat16:
        bb = torch.zeros(n * (V + ld_pad) + offset + 8, dtype=torch.bfloat16, device="cuda")
        view = bb[offset:offset + n * (V + ld_pad)].view(n, V + ld_pad)[:, :V]
        view.copy_(torch.from_numpy(x).to(torch.bfloat16))
    t = None if temps is None else torch.from_numpy(np.asarray(temps, np.float32)).cuda()
    q = ds.q_build(view, t, top_k)
    torch.cuda.synchronize()
    return q, view


def host_rows(x, dtype):
    """The rows the kernels read, made on the host: bf16 rounding by the CPU,
    widened exactly back to fp32."""
    if dtype == torch.bfloat16:
        return torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    return x


@pytest.mark.parametrize("V", [1, 2, 3, 8, 13, 257, 4099, 65537, 129280])
@pytest.mark.parametrize("top_k", [0, 1, 16, 256])
def test_q_build_random_rows(oracle, V, top_k):
    if top_k > V:
        pytest.skip("top_k > V")
    rng = np.random.default_rng(V * 7 + top_k)
    x = rows_for(V, rng, n_each=1 if V > 10000 else 2)
    temps = rng.choice([1.0, 0.7, 1.3, 0.25], size=x.shape[0]).astype(np.float32)
    q, _ = run_q(x, temps, top_k)
    compare_q(q, oracle.q_build(x, temps, top_k))


@pytest.mark.parametrize("ld_pad,offset", [(3, 1), (1, 2), (5, 3)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_q_build_strided_unaligned(oracle, ld_pad, offset, dtype):
    rng = np.random.default_rng(ld_pad + 10 * offset)
    V = 4099
    x = rows_for(V, rng, n_each=1)
    q, view = run_q(x, None, 0, ld_pad=ld_pad, dtype=dtype, offset=offset)
    xr = host_rows(x, dtype)
    compare_q(q, oracle.q_build(xr, None, 0))
    qs, _ = run_q(x, None, 64, ld_pad=ld_pad, dtype=dtype, offset=offset)
    compare_q(qs, oracle.q_build(xr, None, 64))


@pytest.mark.parametrize("top_k", [1, 256, 1024])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_q_topk_stream_orders(oracle, top_k, dtype):
    """Top-k rows whose order defeats the streaming filter (ascending: every
    element is a candidate, so the buffer is cut back many times) or makes it
    trivial (descending), with exact ties straddling every cut, at the full
    vocabulary and the largest k."""
    rng = np.random.default_rng(top_k)
    V = 129280
    asc = np.sort(rng.normal(0, 3, V)).astype(np.float32)
    tied = np.round(asc * 2) / 2                     # long runs of equal values
    x = np.stack([asc, asc[::-1], tied, tied[::-1],
                  np.repeat(np.arange(V // 640, dtype=np.float32), 640)[:V]])
    q, view = run_q(x, [1.0, 1.0, 0.7, 1.3, 1.0], top_k, dtype=dtype)
    xr = host_rows(x, dtype)
    compare_q(q, oracle.q_build(xr, [1.0, 1.0, 0.7, 1.3, 1.0], top_k))


@pytest.mark.parametrize("V", [4099, 129280])
@pytest.mark.parametrize("top_k", [2, 7, 256, 1000, 1024])
def test_q_topk_allocation_edges(oracle, V, top_k):
    """Supports that steer the allocation's selects and its id ordering:
    equal logits (every remainder equal, the grants go to the lowest ids;
    with k a power of two every remainder is zero and nothing is granted),
    two tied groups, support ids packed at the start of the row with one at
    its end (one id bucket holds nearly all of them), ties at the support's
    cut, and a single finite value."""
    if top_k > V:
        pytest.skip("top_k > V")
    rng = np.random.default_rng(V + top_k)
    rows = []
    r = np.full(V, -np.inf, np.float32)
    pos = rng.choice(V, size=min(V, top_k + 3), replace=False)
    r[pos] = 1.0                                        # k + 3 equal logits
    rows.append(r)
    r = np.full(V, -np.inf, np.float32)
    pos = rng.choice(V, size=min(V, top_k + 5), replace=False)
    r[pos[: len(pos) // 2]] = 2.0                       # two tied groups
    r[pos[len(pos) // 2:]] = 1.0
    rows.append(r)
    r = rng.normal(-40, 1, V).astype(np.float32)
    r[: top_k - 1] = rng.normal(3, 1, top_k - 1)        # ids 0 .. k-2 and V-1
    r[V - 1] = 2.5
    rows.append(r)
    r = np.round(rng.normal(0, 1, V) * 2).astype(np.float32) / 2   # ties at the cut
    rows.append(r)
    r = np.full(V, -np.inf, np.float32)
    r[rng.integers(V)] = 0.5                            # one finite value
    rows.append(r)
    x = np.stack(rows)
    temps = np.array([1.0, 0.7, 1.0, 1.3, 1.0], np.float32)
    q, _ = run_q(x, temps, top_k)
    compare_q(q, oracle.q_build(x, temps, top_k))


def test_q_topk_batch_invariance():
    rng = np.random.default_rng(19)
    V = 129280
    x = rows_for(V, rng, n_each=1)
    full, _ = run_q(x, None, 256)
    for r in (0, 2, x.shape[0] - 1):
        alone, _ = run_q(x[r:r + 1], None, 256)
        for key in ("counts", "ids", "nnz", "status"):
            assert torch.equal(alone[key][0], full[key][r]), key


def test_q_build_uniform_full_vocab_closed_form():
    V = 129280
    q, _ = run_q(np.zeros((3, V), np.float32), [1.0, 0.5, 2.0], 0)
    c = np_(q["counts"])
    expect = np.full(V, 129, np.int64)
    expect[:100096] += 1
    for r in range(3):
        assert np.array_equal(c[r], expect)
    assert np.all(np_(q["status"]) == 0)


def test_q_build_refusals(oracle):
    V = 5000
    rng = np.random.default_rng(3)
    x = rng.normal(0, 2, (6, V)).astype(np.float32)
    x[0, 17] = np.nan
    x[1, 4999] = np.inf
    x[2, :] = -np.inf
    x[3, 5] = 3e38
    temps = np.array([1.0, 1.0, 1.0, 0.5, 0.0, np.inf], np.float32)
    for top_k in (0, 32):
        q, _ = run_q(x, temps, top_k)
        ref = oracle.q_build(x, temps, top_k)
        compare_q(q, ref)
        assert np_(q["status"]).tolist() == [1, 1, 2, 1, 4, 4]
        assert np_(q["counts"]).sum() == 0


def test_q_build_batch_invariance():
    rng = np.random.default_rng(9)
    V = 129280
    x = rows_for(V, rng, n_each=1)
    full, _ = run_q(x, None, 0)
    for r in (0, 3, x.shape[0] - 1):
        alone, _ = run_q(x[r:r + 1], None, 0)
        assert torch.equal(alone["counts"][0], full["counts"][r])


WORKLOADS = [
    ("c1", {}), ("c2", {}), ("c3", {"B": 8}), ("c4", {"B": 24}),
    ("c5", {"B": 4, "variant": "accept"}), ("c5", {"B": 4, "variant": "reject"}),
    ("c5", {"B": 4, "variant": "mixed", "top_k": 0}),
]


def _wl(name, kw):
    if name == "c5":
        return W.config5(**kw)
    return {"c1": W.config1, "c2": W.config2, "c3": W.config3, "c4": W.config4}[name](**kw)


@pytest.mark.parametrize("name,kw", WORKLOADS)
def test_workload_q_and_draft_sample(oracle, name, kw):
    wl = _wl(name, kw)
    x = wl.draft.reshape(wl.B * wl.depth, wl.V)
    q, _ = run_q(x, wl.temperature, wl.top_k)
    ref = oracle.q_build(x, wl.temperature, wl.top_k)
    compare_q(q, ref)
    req = torch.from_numpy(wl.request_ids.view(np.int32)).cuda()
    tok, st = ds.draft_sample(q, wl.B, wl.depth, wl.V, wl.seed, req)
    rtok, rst = oracle.draft_sample(ref[0], ref[1], ref[2], wl.top_k, wl.B, wl.depth, wl.seed,
                                    wl.request_ids, V=wl.V)
    assert np.array_equal(np_(st).ravel(), rst)
    assert np.array_equal(np_(tok).ravel(), rtok)
    # the fused entry: same counts and the same draws in one launch
    d = torch.from_numpy(np.ascontiguousarray(wl.draft)).cuda()
    temps = torch.from_numpy(wl.temperature).cuda()
    qf, ftok = ds.q_build_sample(d, wl.B, wl.depth, wl.seed, temps, wl.top_k, req)
    torch.cuda.synchronize()
    compare_q(qf, ref)
    assert np.array_equal(np_(ftok).ravel(), rtok)


@pytest.mark.parametrize("V", [1, 3, 257, 4099])
@pytest.mark.parametrize("top_k", [0, 2, 64])
def test_fused_sample_small_and_refused(oracle, V, top_k):
    if top_k > V:
        pytest.skip("top_k > V")
    rng = np.random.default_rng(V + top_k)
    B, depth = 3, 4
    x = rows_for(V, rng, n_each=1)[: B * depth]
    while x.shape[0] < B * depth:
        x = np.concatenate([x, rng.normal(0, 1, (1, V)).astype(np.float32)])
    x[5, 0] = np.nan          # a refused row inside the batch
    temps = np.ones(B * depth, np.float32)
    temps[7] = 0.0            # another one
    req = np.array([5, 0, 77], np.uint32)
    xt = torch.from_numpy(x).cuda()
    qf, ftok = ds.q_build_sample(xt, B, depth, 1234, torch.from_numpy(temps).cuda(), top_k,
                                 torch.from_numpy(req.view(np.int32)).cuda())
    torch.cuda.synchronize()
    ref = oracle.q_build(x, temps, top_k)
    compare_q(qf, ref)
    rtok, rst = oracle.draft_sample(ref[0], ref[1], ref[2], top_k, B, depth, 1234, req, V=V)
    rtok = np.where(ref[3] == 0, rtok, -1)
    assert np.array_equal(np_(ftok).ravel(), rtok)


def test_draft_sample_refuses_bad_rows(oracle):
    V, depth = 300, 2
    counts = np.zeros((4, V), np.uint32)
    counts[:, 7] = M
    counts[1, 7] -= 1                      # wrong mass
    counts[2, 7] = M // 2
    counts[2, 299] = M // 2
    counts[3, :] = M // V
    counts[3, :M - (M // V) * V] += 1
    ct = torch.from_numpy(counts.view(np.int32)).cuda()
    q = {"counts": ct, "ids": None, "nnz": None, "top_k": 0}
    tok, st = ds.draft_sample(q, 2, depth, V, 123)
    rtok, rst = oracle.draft_sample(counts, None, None, 0, 2, depth, 123)
    assert np.array_equal(np_(st).ravel(), rst) and rst.tolist()[:2] == [0, 5]
    assert np.array_equal(np_(tok).ravel(), rtok)
    # sparse: unsorted ids, zero count, nnz out of range, out-of-range id
    ids = np.array([[3, 9, -1, -1], [9, 3, -1, -1], [3, 9, -1, -1], [3, 9, 12, -1],
                    [3, 400, -1, -1], [5, -1, -1, -1]], np.int32)
    sc = np.array([[M - 5, 5, 0, 0], [M - 5, 5, 0, 0], [M, 0, 0, 0], [1, 2, M - 3, 0],
                   [M - 1, 1, 0, 0], [M, 0, 0, 0]], np.uint32)
    nnz = np.array([2, 2, 2, 3, 2, 0], np.int32)
    q = {"counts": torch.from_numpy(sc.view(np.int32)).cuda(),
         "ids": torch.from_numpy(ids).cuda(), "nnz": torch.from_numpy(nnz).cuda(), "top_k": 4}
    tok, st = ds.draft_sample(q, 3, 2, V, 77)
    rtok, rst = oracle.draft_sample(sc, ids, nnz, 4, 3, 2, 77, V=V)
    assert rst.tolist() == [0, 5, 5, 0, 5, 5]
    assert np.array_equal(np_(st).ravel(), rst)
    assert np.array_equal(np_(tok).ravel(), rtok)
