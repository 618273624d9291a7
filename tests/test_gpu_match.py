"""GPU parity of stochastic (match) verification (dspark_verify_match)
against the oracle: integer outputs bit for bit on every request except
those whose draw the ORACLE finds within 1e-6 (probability units) of a
cumulative boundary (the benchmark definition's band; the GPU's own flags
excuse nothing), on the workloads' rows (fp32 and bf16 targets), the
all-accept and all-reject extremes, ragged vocabularies and refused rows.
Band cases under both readings (absolute, and relative to the picked
token's own mass) are counted and printed in pytest's summary; the relative
reading's must stay under 1e-4 of the verify rows."""
import numpy as np
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from draft_sampling_verification_gb300 import workloads as W
from oracle import oracle as O
from parity import (BAND_BOUND, VerifyCounts, compare_verify, dev_inputs, np_, oracle_q,
                    oracle_sample)

pytestmark = pytest.mark.gpu

STATS = VerifyCounts()  # match comparisons of the workload tests


def run(wl, drafts_np=None):
    d, t, temps, req = dev_inputs(wl)
    if drafts_np is None:  # the oracle's drafts, given to both sides
        drafts_np = oracle_sample(wl, oracle_q(wl))[0].reshape(wl.B, wl.depth)
    drafts = np.ascontiguousarray(drafts_np, dtype=np.int32)
    tok = torch.from_numpy(drafts).cuda()
    g = ds.verify_match(t, tok, wl.seed, req)
    torch.cuda.synchronize()
    ref = O.verify_match(wl.target_f32(), drafts, wl.seed, wl.request_ids)
    return g, ref


@pytest.mark.parametrize("name,kw", [("c1", {}), ("c2", {}), ("c4", {"B": 48}),
                                     ("c3", {"B": 16}),
                                     ("c5:8:accept:sparse", {}),
                                     ("c5:8:reject:sparse", {})])
def test_match_workloads(oracle, name, kw):
    global STATS
    wl = W.by_name(name, **kw)
    g, ref = run(wl)
    c = compare_verify(g, ref, "match")
    STATS += c
    assert c.mismatch == 0, (name, c)
    acc = np_(g[0])
    assert np.all(np_(g[3]) == 0)
    if "accept" in name:
        assert acc.mean() > 2.0


@pytest.mark.parametrize("V", [1, 5, 257, 4099])
def test_match_ragged_and_refused(oracle, V):
    rng = np.random.default_rng(V + 7)
    B, depth = 6, 5
    wl = W.config1(B=B, V=V)
    wl.target = rng.normal(0, 2, (B, depth + 1, V)).astype(np.float32)
    drafts = rng.integers(0, V, (B, depth)).astype(np.int32)
    wl.target[1, 0, V // 2] = np.nan       # refused at row 0
    wl.target[2, depth, 0] = np.inf        # refused only if every proposal matched
    drafts[3, 2] = V                       # an out-of-range draft: BAD_DRAFT
    g, ref = run(wl, drafts)
    c = compare_verify(g, ref, "match")
    assert c.mismatch == 0, (V, c)
    st = np_(g[3])
    assert st[1] == ds.ST_NONFINITE and st[3] == ds.ST_BAD_DRAFT


def test_zz_match_band_budget():
    """Over the workload tests above: the relative band's cases stay under
    1e-4 of the verify rows (the absolute reading's rate is printed)."""
    if STATS.rows == 0:
        pytest.skip("no match verification ran")
    print("match verification:", STATS)
    assert STATS.mismatch == 0
    assert STATS.band_rel <= BAND_BOUND * STATS.rows
