"""GPU parity of the whole speculative step (dspark_spec_step), in both of
its schedules: every output is bit-identical to the separate calls (dspark_q_build_sample, then
dspark_verify_greedy / dspark_verify_ratio on the same stream), and matches
the oracle as those calls do (counts, tokens and greedy outputs bit-exact;
ratio outputs bit-exact outside the oracle's tolerance band), on the dense workloads at
full size, both target dtypes, one or both modes, ragged vocabularies and
refused rows."""
import numpy as np
import pytest
import torch

import draft_sampling_verification_gb300 as ds
from draft_sampling_verification_gb300 import workloads as W
from parity import (compare_q, compare_verify, dev_inputs, np_, oracle_q, oracle_sample,
                    oracle_verify)

pytestmark = pytest.mark.gpu


def separate(d, t, wl, temps, req, modes):
    q, tok = ds.q_build_sample(d, wl.B, wl.depth, wl.seed, temps, 0, req)
    outs = {}
    if "greedy" in modes:
        outs["greedy"] = ds.verify_greedy(t, tok)
    if "ratio" in modes:
        outs["ratio"] = ds.verify_ratio(t, tok, q, wl.seed, req)
    torch.cuda.synchronize()
    return q, tok, outs


def fused(d, t, wl, temps, req, modes, schedule=ds.SCHEDULE_ONE_LAUNCH):
    q, tok, outs = ds.spec_step(d, t, wl.B, wl.depth, wl.seed, temps, req, modes,
                                schedule=schedule)
    torch.cuda.synchronize()
    return q, tok, outs


def assert_same(a, b):
    qa, ta, oa = a
    qb, tb, ob = b
    assert torch.equal(qa["counts"], qb["counts"])
    assert torch.equal(qa["status"], qb["status"])
    assert torch.equal(ta, tb)
    assert sorted(oa) == sorted(ob)
    for m in oa:
        for x, y in zip(oa[m], ob[m]):
            assert torch.equal(x, y), m


def check_oracle(wl, res, modes):
    q, tok, outs = res
    qref = oracle_q(wl)
    compare_q(q, qref)
    # the oracle verifies the oracle's own drafts, which the GPU's must equal
    rtok, _ = oracle_sample(wl, qref)
    assert np.array_equal(np_(tok).ravel(), rtok)
    drafts = rtok.reshape(wl.B, wl.depth)
    for m in modes:
        g = outs[m]
        if m == "greedy":
            g = (g[0], g[1], torch.zeros_like(g[0]), g[2])
        c = compare_verify(g, oracle_verify(wl, m, drafts, qref), m)
        assert c.mismatch == 0, (wl.name, m, c)


@pytest.mark.parametrize("name", ["c1", "c2", "c4"])
def test_spec_step_workloads(oracle, name):
    kw = {"B": 32} if name == "c4" else {}
    wl = W.by_name(name, **kw)
    d, t, temps, req = dev_inputs(wl)
    modes = ("greedy", "ratio")
    a = fused(d, t, wl, temps, req, modes)
    sep = separate(d, t, wl, temps, req, modes)
    assert_same(a, sep)
    # the two-kernel schedule (one verify pass for both modes) and the
    # automatic choice give the same outputs
    for sched in (ds.SCHEDULE_SEPARATE, ds.SCHEDULE_AUTO):
        assert_same(fused(d, t, wl, temps, req, modes, sched), sep)
    check_oracle(wl, a, modes)


@pytest.mark.parametrize("modes", [("greedy",), ("ratio",)])
@pytest.mark.parametrize("tdtype", ["f32", "bf16"])
def test_spec_step_one_mode(oracle, modes, tdtype):
    wl = W.config3(B=8, top_k=0)
    if tdtype == "bf16":
        wl.target = W.f32_to_bf16_bits(wl.target)
        wl.target_dtype = "bf16"
    d, t, temps, req = dev_inputs(wl)
    a = fused(d, t, wl, temps, req, modes)
    assert_same(a, separate(d, t, wl, temps, req, modes))
    check_oracle(wl, a, modes)


@pytest.mark.parametrize("V", [1, 5, 257, 4099])
def test_spec_step_ragged_and_refused(oracle, V):
    rng = np.random.default_rng(V)
    B, depth = 6, 5
    wl = W.config1(B=B, V=V)
    wl.draft = rng.normal(0, 2, (B, depth, V)).astype(np.float32)
    wl.target = (wl.draft[:, [0, 1, 2, 3, 4, 4]] + rng.normal(0, 0.5, (B, depth + 1, V))).astype(
        np.float32)
    wl.draft[1, 2, 0] = np.nan          # a refused q row: its request is BAD_DRAFT
    wl.temperature[4 * depth + 1] = 0.0  # a refused temperature
    wl.target[3, 0, V // 2] = np.inf     # a refused target row (if it is read)
    d, t, temps, req = dev_inputs(wl)
    modes = ("greedy", "ratio")
    a = fused(d, t, wl, temps, req, modes)
    sep = separate(d, t, wl, temps, req, modes)
    assert_same(a, sep)
    assert_same(fused(d, t, wl, temps, req, modes, ds.SCHEDULE_SEPARATE), sep)
    check_oracle(wl, a, modes)
    st_r = np_(a[2]["ratio"][3])
    assert st_r[1] == 6 and st_r[4] == 6  # BAD_DRAFT


def verify_both(t, wl, q, tok, req, modes):
    B, depth = wl.B, wl.depth
    dev = t.device
    mk = lambda *s: torch.empty(s, dtype=torch.int32, device=dev)
    g = (mk(B), mk(B, depth + 1), mk(B)) if "greedy" in modes else None
    r = (mk(B), mk(B, depth + 1), mk(B), mk(B)) if "ratio" in modes else None
    ds.dspark_verify(t, B, depth, tok, g, r, q["counts"], q["ids"], q["nnz"], q["top_k"],
                     wl.seed, req)
    torch.cuda.synchronize()
    outs = {}
    if g:
        outs["greedy"] = g
    if r:
        outs["ratio"] = r
    return outs


@pytest.mark.parametrize("case", ["c3_topk", "c4_dense", "c4_greedy_only", "c3_ratio_only"])
def test_verify_one_pass_equals_separate_calls(case):
    """dspark_verify (both modes in one pass over the target rows) gives
    each mode's outputs exactly as dspark_verify_greedy / _ratio do, with a
    sparse (top-k) or a dense q."""
    wl = W.config3(B=8) if case.startswith("c3") else W.config4(B=16)
    modes = {"c3_topk": ("greedy", "ratio"), "c4_dense": ("greedy", "ratio"),
             "c4_greedy_only": ("greedy",), "c3_ratio_only": ("ratio",)}[case]
    d, t, temps, req = dev_inputs(wl)
    q, tok = ds.q_build_sample(d, wl.B, wl.depth, wl.seed, temps, wl.top_k, req)
    ref = {}
    if "greedy" in modes:
        ref["greedy"] = ds.verify_greedy(t, tok)
    if "ratio" in modes:
        ref["ratio"] = ds.verify_ratio(t, tok, q, wl.seed, req)
    got = verify_both(t, wl, q, tok, req, modes)
    assert sorted(got) == sorted(ref)
    for m in ref:
        for x, y in zip(got[m], ref[m]):
            assert torch.equal(x, y), (case, m)


@pytest.mark.parametrize("name,schedule", [("c2", ds.SCHEDULE_AUTO), ("c4", ds.SCHEDULE_SEPARATE),
                                           ("c4", ds.SCHEDULE_ONE_LAUNCH)])
def test_spec_step_host_equals_device_step(oracle, name, schedule):
    """dspark_spec_step_host (host buffers, its own staging and copies) gives
    the device step's outputs bit for bit, on two streams at once."""
    wl = W.config2() if name == "c2" else W.config4(B=8)
    d, t, temps, req = dev_inputs(wl)
    ref_q, ref_tok, ref = fused(d, t, wl, temps, req, wl.modes, schedule)
    B, depth, V = wl.B, wl.depth, wl.V
    h_d = d.cpu().pin_memory()
    h_t = t.cpu().pin_memory()
    h_temp = temps.cpu().pin_memory()
    h_req = req.cpu().pin_memory()
    sb = ds.dspark_spec_step_host_staging_bytes(B, depth, V, ds._dtype_code(h_d),
                                                ds._dtype_code(h_t))
    outs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    stagings = []
    for s in streams:
        pin = lambda shape: torch.full(shape, -9, dtype=torch.int32).pin_memory()
        o = {"tok": pin((B, depth)), "rst": pin((B * depth,))}
        if "greedy" in wl.modes:
            o["greedy"] = (pin((B,)), pin((B, depth + 1)), pin((B,)))
        if "ratio" in wl.modes:
            o["ratio"] = (pin((B,)), pin((B, depth + 1)), pin((B,)), pin((B,)))
        stg = torch.empty((sb,), dtype=torch.uint8, device="cuda")
        stagings.append(stg)
        ds.dspark_spec_step_host(h_d, h_t, B, depth, h_temp, wl.seed, h_req, o["tok"], o["rst"],
                                 stg, greedy_out=o.get("greedy"), ratio_out=o.get("ratio"),
                                 stream=s, schedule=schedule)
        outs.append(o)
    torch.cuda.synchronize()
    for o, stg in zip(outs, stagings):
        assert torch.equal(o["tok"], ref_tok.cpu())
        assert torch.equal(o["rst"], ref_q["status"].cpu())
        # the q counts stay at the start of the staging buffer
        counts = stg[: B * depth * V * 4].view(torch.int32).view(B * depth, V)
        assert torch.equal(counts, ref_q["counts"])
        for m in wl.modes:
            assert all(torch.equal(x, y.cpu()) for x, y in zip(o[m], ref[m])), m
