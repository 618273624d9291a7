"""The bounds-checked build of the library (libdspark_checked.so, compiled
with DSPARK_CHECKED): the small-vocabulary parity set run through it, with
every checked index site passing (no failure counted by
dspark_checked_status).  It stands in for the memory checker, which this
pool does not run: each checked site tests its index against its bound and
records a failure instead of making the access.

Small vocabularies (V in {1, 2, 3, 8, 257, 4099}) make every slice ragged
(empty CTAs, partial edge groups, single elements), where an index slip is
most likely; the outputs must still equal the oracle's as in the other
parity tests (greedy bit-exact, ratio and match outside the oracle's band)."""
import ctypes
import os

import numpy as np
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from draft_sampling_verification_gb300 import _lib, build
from draft_sampling_verification_gb300 import workloads as W
from oracle import oracle as O
from parity import compare_q, compare_verify, dev_inputs, np_, oracle_q, oracle_sample

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked_lib():
    path = build.LIB_CHECKED
    if not os.path.exists(path):
        build.build(checked=True)
    saved = _lib._lib
    _lib._lib = None
    lib = _lib.load(path)
    yield lib
    _lib._lib = saved


def status(lib):
    out = (ctypes.c_uint32 * 3)()
    assert lib.dspark_checked_status(out) == 0
    return list(out)


def small_workload(V, dtype, top_k, seed):
    rng = np.random.default_rng(seed)
    B, depth = 6, 3
    xd = rng.normal(0, 1.5, (B, depth, V)).astype(np.float32)
    xt = np.concatenate([xd, rng.normal(0, 1.5, (B, 1, V)).astype(np.float32)], axis=1)
    xt = xt + rng.normal(0, 0.5, xt.shape).astype(np.float32)
    if V >= 8:
        xd[0, 1] = np.round(xd[0, 1] * 2) / 2          # exact ties
        xd[1, 0, : V // 3] = -np.inf                   # a masked third
        xt[1, 0, : V // 3] = -np.inf
    tgt = W.f32_to_bf16_bits(xt) if dtype == "bf16" else xt
    temps = rng.choice([1.0, 0.7], B * depth).astype(np.float32)
    return W.Workload("checked", B, depth, V, xd, tgt, dtype, temps, top_k, 5,
                      ("greedy", "ratio"), np.arange(B, dtype=np.uint32) * 5 + 2)


@pytest.mark.parametrize("V", [1, 2, 3, 8, 257, 4099])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_vocab_parity_under_checks(oracle, checked_lib, V, dtype):
    assert status(checked_lib)[2] == 1, "not the checked build"
    for top_k in (0, min(V, 4)):
        wl = small_workload(V, dtype, top_k, V * 7 + top_k)
        d, t, temps, req = dev_inputs(wl)
        q = ds.q_build(d, temps, top_k)
        tok, sst = ds.draft_sample(q, wl.B, wl.depth, V, wl.seed, req)
        torch.cuda.synchronize()
        qref = oracle_q(wl)
        compare_q(q, qref)
        rtok, _ = oracle_sample(wl, qref)
        assert np.array_equal(np_(tok).ravel(), rtok)
        drafts = rtok.reshape(wl.B, wl.depth)
        z = wl.target_f32()
        g = ds.verify_greedy(t, tok)
        r = ds.verify_ratio(t, tok, q, wl.seed, req)
        m = ds.verify_match(t, tok, wl.seed, req)
        torch.cuda.synchronize()
        acc, com, gst = O.verify_greedy(z, drafts)
        assert np.array_equal(np_(g[0]), acc) and np.array_equal(np_(g[1]), com)
        ref = O.verify_ratio(z, drafts, qref[0], qref[1], qref[2], top_k, wl.seed,
                             wl.request_ids)
        assert compare_verify(r, ref, "ratio").mismatch == 0
        refm = O.verify_match(z, drafts, wl.seed, wl.request_ids)
        assert compare_verify(m, refm, "match").mismatch == 0
        if top_k == 0:
            # the whole step in both schedules, and the Markov chain
            for sched in (ds.SCHEDULE_ONE_LAUNCH, ds.SCHEDULE_SEPARATE):
                q2, tok2, outs = ds.spec_step(d, t, wl.B, wl.depth, wl.seed, temps, req,
                                              schedule=sched)
                torch.cuda.synchronize()
                assert torch.equal(q2["counts"], q["counts"]) and torch.equal(tok2, tok)
                assert torch.equal(outs["greedy"][0], g[0]) and torch.equal(outs["ratio"][1],
                                                                            r[1])
            anchors = torch.arange(wl.B, dtype=torch.int32, device="cuda") % V
            bias = torch.from_numpy(np.random.default_rng(V).normal(
                0, 1, (3, V)).astype(np.float32)).cuda()
            cq, ctok, cmg = ds.q_chain_sample(d, wl.B, wl.depth, wl.seed, anchors, bias, temps,
                                              req)
            torch.cuda.synchronize()
            cref = O.q_chain(wl.draft, wl.temperature, bias.cpu().numpy(),
                             np.arange(wl.B) % V, wl.seed, wl.request_ids)
            assert np.array_equal(np_(cq["counts"]).view(np.uint32), cref[0])
            assert np.array_equal(np_(ctok), cref[1])
    fails, site, checked = status(checked_lib)
    assert checked == 1 and fails == 0, "checked site %d failed %d times" % (site, fails)


def test_zz_a_failing_site_is_counted(checked_lib):
    """The counters themselves: one deliberately failing site (it guards no
    access) is reported once, with its source file's number (2, the debug
    entry points), and the counters are cleared by the read."""
    status(checked_lib)
    assert checked_lib.dspark_debug_check_selftest(None) == 0
    torch.cuda.synchronize()
    fails, site, checked = status(checked_lib)
    assert checked == 1 and fails == 1 and site // 10000 == 2, (fails, site)
    assert status(checked_lib)[:2] == [0, 0]
