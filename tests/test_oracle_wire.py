"""The oracle's received-q functions against what fixes them: Fletcher-64's
published test vectors, the exactness of q = c / M in FP32 that the pages
state ("PP1 q transport and scheduling design", Distribution contract and
precision), pack-then-validate round trips on oracle-built q rows, and one
case for each refusal the pages list (Versioned v2 message design)."""
import json
import os

import numpy as np
import pytest

from oracle import oracle as O

M = 1 << 24


def words_of(b: bytes) -> np.ndarray:
    b = b + b"\0" * (-len(b) % 4)
    return np.frombuffer(b, "<u4")


def test_fletcher64_published_vectors(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "fletcher64.json")))
    for v in g["vectors"]:
        assert O.fletcher64(words_of(v["ascii"].encode())) == int(v["fletcher64"], 16), v


def test_fletcher64_sensitivity():
    # a changed word, two swapped words and a dropped zero word all change it
    w = np.arange(1, 65, dtype=np.uint32) * np.uint32(2654435761)
    base = O.fletcher64(w)
    w2 = w.copy()
    w2[10] ^= 1
    w3 = w.copy()
    w3[[3, 4]] = w3[[4, 3]]
    assert O.fletcher64(w2) != base and O.fletcher64(w3) != base
    assert O.fletcher64(np.append(w, np.uint32(0))) != base


def test_counts_are_exact_in_fp32():
    # every c in [0, M] survives c / M -> FP32 -> * M (edges and a sample)
    rng = np.random.default_rng(5)
    c = np.concatenate([np.arange(0, 4096), M - np.arange(0, 4096),
                        rng.integers(0, M + 1, 200000)]).astype(np.uint64)
    q = (c.astype(np.float64) / M).astype(np.float32)
    assert np.array_equal(q.astype(np.float64) * M, c.astype(np.float64))


def built_rows(V, top_k, n=6, seed=1):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 2, (n, V)).astype(np.float32)
    counts, ids, nnz, st = O.q_build(x, None, top_k)
    assert np.all(st == 0)
    return counts, ids, nnz


@pytest.mark.parametrize("V,top_k", [(5, 0), (257, 0), (4099, 0), (257, 16), (4099, 64)])
def test_pack_validate_round_trip(oracle, V, top_k):
    counts, ids, nnz = built_rows(V, top_k)
    q, cs = O.q_pack(counts, ids, nnz, top_k)
    assert np.all(q[:, :counts.shape[1]].astype(np.float64) * M == counts)
    toks = np.array([ids[r][0] if top_k else int(np.argmax(counts[r])) for r in range(len(q))])
    st, rec = O.q_validate(q, ids, nnz, top_k, V, toks, cs)
    assert np.all(st == O.OK)
    assert np.array_equal(rec, counts)
    # the checksum is that of the payload words taken by hand
    r = 0
    if top_k:
        payload = np.concatenate([ids[r][:nnz[r]].view(np.uint32), q[r][:nnz[r]].view(np.uint32)])
    else:
        payload = q[r].view(np.uint32)
    assert int(cs[r]) == O.fletcher64(payload)


def refuse(q, ids, nnz, top_k, V, tokens=None, expect=None):
    st, rec = O.q_validate(q, ids, nnz, top_k, V, tokens, expect)
    assert np.all(rec[st != 0] == 0)
    return st


def test_dense_refusals(oracle):
    V = 257
    counts, _, _ = built_rows(V, 0, n=1)
    q, cs = O.q_pack(counts)
    hot = int(np.argmax(counts[0]))
    cold = int(np.flatnonzero(counts[0] == 0)[0]) if np.any(counts[0] == 0) else None
    cases = []
    for mod in ("nan", "inf", "neg", "nondyadic", "above1", "mass"):
        qq = q.copy()
        if mod == "nan":
            qq[0, hot] = np.nan
        elif mod == "inf":
            qq[0, hot] = np.inf
        elif mod == "neg":
            qq[0, hot] = -qq[0, hot]
        elif mod == "nondyadic":
            qq[0, hot] = np.nextafter(qq[0, hot], np.float32(2))
        elif mod == "above1":
            qq[0, hot] = np.float32(1.5)
        elif mod == "mass":
            # one ticket more: every value still dyadic, the mass M + 1
            qq[0, hot] = qq[0, hot] + np.float32(2.0 ** -24)
        cases.append((mod, qq))
    for mod, qq in cases:
        assert refuse(qq, None, None, 0, V)[0] == O.BAD_Q, mod
    # a changed payload with the sender's checksum: the checksum speaks first
    qq = q.copy()
    qq[0, hot] = np.nan
    assert refuse(qq, None, None, 0, V, expect=cs)[0] == O.BAD_CHECKSUM
    # a valid row whose checksum was damaged in transit
    assert refuse(q, None, None, 0, V, expect=cs ^ np.uint64(1))[0] == O.BAD_CHECKSUM
    # the proposed token: outside [0, V), or with q = 0
    assert refuse(q, None, None, 0, V, tokens=np.array([V]))[0] == O.BAD_DRAFT
    assert refuse(q, None, None, 0, V, tokens=np.array([-1]))[0] == O.BAD_DRAFT
    if cold is not None:
        assert refuse(q, None, None, 0, V, tokens=np.array([cold]))[0] == O.BAD_DRAFT
    assert refuse(q, None, None, 0, V, tokens=np.array([hot]), expect=cs)[0] == O.OK


def test_sparse_refusals(oracle):
    V, k = 4099, 16
    counts, ids, nnz = built_rows(V, k, n=1)
    q, cs = O.q_pack(counts, ids, nnz, k)
    n = int(nnz[0])
    assert n >= 3
    base = (q, ids.copy(), nnz.copy())

    def case(fn):
        qq, ii, nn = base[0].copy(), base[1].copy(), base[2].copy()
        fn(qq, ii, nn)
        return refuse(qq, ii, nn, k, V)[0]

    def dup(qq, ii, nn):
        ii[0, 1] = ii[0, 0]

    def unsorted(qq, ii, nn):
        ii[0, [0, 1]] = ii[0, [1, 0]]

    def out_of_range(qq, ii, nn):
        ii[0, n - 1] = V

    def padded(qq, ii, nn):
        ii[0, n - 1] = -1

    def listed_zero(qq, ii, nn):
        qq[0, 0] = 0.0

    def nnz_zero(qq, ii, nn):
        nn[0] = 0

    def nnz_big(qq, ii, nn):
        nn[0] = k + 1

    for fn in (dup, unsorted, out_of_range, padded, listed_zero, nnz_zero, nnz_big):
        assert case(fn) == O.BAD_Q, fn.__name__
    # a token outside the support is refused, one inside it is not
    outside = int(np.setdiff1d(np.arange(V), ids[0][:n])[0])
    assert refuse(q, ids, nnz, k, V, tokens=np.array([outside]))[0] == O.BAD_DRAFT
    assert refuse(q, ids, nnz, k, V, tokens=np.array([ids[0][1]]), expect=cs)[0] == O.OK
