"""GPU parity of the received-q path (dspark_q_pack, dspark_q_validate)
against the oracle, bit for bit: wire values, Fletcher-64 checksums,
statuses and recovered counts, on dense rows of many lengths (aligned and
unaligned starts), sparse rows, the rows the q build makes for the
workloads, and one damaged row per refusal."""
import numpy as np
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from draft_sampling_verification_gb300 import workloads as W
from oracle import oracle as O
from parity import compare_q, dev_inputs, np_, oracle_q

pytestmark = pytest.mark.gpu


def oracle_rows(V, top_k, n, seed):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 2, (n, V)).astype(np.float32)
    x[0] = np.round(x[0] * 2) / 2          # ties
    counts, ids, nnz, st = O.q_build(x, None, top_k)
    return counts, ids, nnz


def gpu_pack(counts, ids, nnz, top_k, V):
    c = torch.from_numpy(counts.view(np.int32)).cuda()
    i = None if ids is None else torch.from_numpy(ids).cuda()
    z = None if nnz is None else torch.from_numpy(nnz).cuda()
    q = {"counts": c, "ids": i, "nnz": z, "top_k": top_k}
    qf, cs = ds.q_pack(q, V)
    torch.cuda.synchronize()
    return qf, cs, i, z


@pytest.mark.parametrize("V,top_k", [(1, 0), (5, 0), (257, 0), (4099, 0), (129280, 0),
                                     (257, 1), (4099, 16), (129280, 256)])
def test_pack_and_validate_match_oracle(oracle, V, top_k):
    n = 4 if V > 10000 else 9
    counts, ids, nnz = oracle_rows(V, top_k, n, V + top_k)
    qf, cs, i, z = gpu_pack(counts, ids, nnz, top_k, V)
    q_ref, cs_ref = O.q_pack(counts, ids, nnz, top_k)
    assert np.array_equal(np_(qf).view(np.uint32), q_ref.view(np.uint32))
    assert np.array_equal(np_(cs).view(np.uint64), cs_ref)
    toks = np.array([ids[r][0] if top_k else int(np.argmax(counts[r])) for r in range(n)],
                    np.int32)
    st, rec = ds.q_validate(qf, V, i, z, top_k, torch.from_numpy(toks).cuda(), cs)
    torch.cuda.synchronize()
    st_ref, rec_ref = O.q_validate(q_ref, ids, nnz, top_k, V, toks, cs_ref)
    assert np.array_equal(np_(st), st_ref) and np.all(st_ref == 0)
    assert np.array_equal(np_(rec).view(np.uint32), rec_ref)
    assert np.array_equal(rec_ref, counts)


def test_unaligned_dense_rows(oracle):
    # V = 4099: every row after the first starts off a 16-byte boundary
    V, n = 4099, 7
    counts, _, _ = oracle_rows(V, 0, n, 3)
    qf, cs, _, _ = gpu_pack(counts, None, None, 0, V)
    q_ref, cs_ref = O.q_pack(counts)
    assert np.array_equal(np_(cs).view(np.uint64), cs_ref)
    # a received buffer at an odd offset
    buf = torch.zeros(n * V + 3, dtype=torch.float32, device="cuda")
    view = buf[3:].view(n, V)
    view.copy_(qf)
    st, rec = ds.q_validate(view, V, expect=cs)
    torch.cuda.synchronize()
    assert np.all(np_(st) == 0) and np.array_equal(np_(rec).view(np.uint32), counts)


def damaged_dense(q, V):
    hot = int(np.argmax(q[0]))
    out = []
    for kind in ("nan", "inf", "neg", "nondyadic", "above1", "mass"):
        qq = q.copy()
        v = qq[0, hot]
        qq[0, hot] = {"nan": np.nan, "inf": np.inf, "neg": -v, "above1": np.float32(1.5),
                      "nondyadic": np.nextafter(v, np.float32(2)),
                      "mass": v + np.float32(2.0 ** -24)}[kind]
        out.append(qq)
    return out


def test_dense_refusals_match_oracle(oracle):
    V = 4099
    counts, _, _ = oracle_rows(V, 0, 1, 11)
    q_ref, cs_ref = O.q_pack(counts)
    rows = damaged_dense(q_ref, V)
    q_all = np.concatenate(rows + [q_ref, q_ref, q_ref, q_ref])
    n = q_all.shape[0]
    expect = np.concatenate([np.repeat(cs_ref, len(rows)), cs_ref, cs_ref ^ np.uint64(1),
                             cs_ref, cs_ref])
    cold = np.flatnonzero(counts[0] == 0)
    toks = np.full(n, int(np.argmax(counts[0])), np.int32)
    toks[-2] = V
    toks[-1] = int(cold[0]) if cold.size else -1
    seen = set()
    for use_expect in (False, True):
        ex = expect if use_expect else None
        st, rec = ds.q_validate(torch.from_numpy(q_all).cuda(), V,
                                tokens=torch.from_numpy(toks).cuda(),
                                expect=None if ex is None else torch.from_numpy(ex.view(np.int64)).cuda())
        torch.cuda.synchronize()
        st_ref, rec_ref = O.q_validate(q_all, None, None, 0, V, toks, ex)
        assert np.array_equal(np_(st), st_ref), (use_expect, np_(st), st_ref)
        assert np.array_equal(np_(rec).view(np.uint32), rec_ref)
        seen |= set(st_ref.tolist())
    assert seen >= {O.OK, O.BAD_Q, O.BAD_CHECKSUM, O.BAD_DRAFT}


def test_sparse_refusals_match_oracle(oracle):
    V, k = 4099, 16
    counts, ids, nnz = oracle_rows(V, k, 1, 12)
    q_ref, cs_ref = O.q_pack(counts, ids, nnz, k)
    n = int(nnz[0])
    qs, iss, ns = [], [], []
    for kind in ("ok", "dup", "unsorted", "range", "pad", "zero", "nnz0", "nnzbig", "tokout"):
        qq, ii, nn = q_ref.copy(), ids.copy(), nnz.copy()
        if kind == "dup":
            ii[0, 1] = ii[0, 0]
        elif kind == "unsorted":
            ii[0, [0, 1]] = ii[0, [1, 0]]
        elif kind == "range":
            ii[0, n - 1] = V
        elif kind == "pad":
            ii[0, n - 1] = -1
        elif kind == "zero":
            qq[0, 0] = 0.0
        elif kind == "nnz0":
            nn[0] = 0
        elif kind == "nnzbig":
            nn[0] = k + 1
        qs.append(qq)
        iss.append(ii)
        ns.append(nn)
    q_all, i_all, n_all = np.concatenate(qs), np.concatenate(iss), np.concatenate(ns)
    toks = np.full(len(qs), int(ids[0][1]), np.int32)
    toks[-1] = int(np.setdiff1d(np.arange(V), ids[0][:n])[0])
    for ex in (None, np.repeat(cs_ref, len(qs))):
        st, rec = ds.q_validate(torch.from_numpy(q_all).cuda(), V, torch.from_numpy(i_all).cuda(),
                                torch.from_numpy(n_all).cuda(), k, torch.from_numpy(toks).cuda(),
                                None if ex is None else torch.from_numpy(ex.view(np.int64)).cuda())
        torch.cuda.synchronize()
        st_ref, rec_ref = O.q_validate(q_all, i_all, n_all, k, V, toks, ex)
        assert np.array_equal(np_(st), st_ref), (np_(st), st_ref)
        assert np.array_equal(np_(rec).view(np.uint32), rec_ref)


@pytest.mark.parametrize("name", ["c4", "c3"])
def test_workload_rows_round_trip(oracle, name):
    wl = W.by_name(name, B=8)
    d, t, temps, req = dev_inputs(wl)
    q, tok = ds.q_build_sample(d, wl.B, wl.depth, wl.seed, temps, wl.top_k, req)
    qf, cs = ds.q_pack(q, wl.V)
    st, rec = ds.q_validate(qf, wl.V, q["ids"], q["nnz"], wl.top_k, tok.reshape(-1), cs)
    torch.cuda.synchronize()
    assert np.all(np_(st) == 0)
    assert torch.equal(rec, q["counts"])
    # the checksums of the oracle's own q, which the GPU's q must equal
    qref = oracle_q(wl)
    compare_q(q, qref)
    counts, ids, nnz, _ = qref
    _, cs_ref = O.q_pack(counts, ids, nnz, wl.top_k)
    assert np.array_equal(np_(cs).view(np.uint64), cs_ref)
