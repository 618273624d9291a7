"""Runs one workload through the CUDA library and through the CPU oracle.

Both sides get the same seeded inputs (``workloads``).  The CUDA side goes
through the Python binding of the C ABI; the oracle side through its ctypes
front end.  Nothing here computes any step of the method.
"""
from __future__ import annotations

import numpy as np
import torch

import draft_sampling_verification_gb300 as ds
from oracle import oracle as O


def dev_inputs(wl):
    """Device tensors of a workload (target bf16 kept as bf16)."""
    d = torch.from_numpy(np.ascontiguousarray(wl.draft)).cuda()
    if wl.target_dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(wl.target)).cuda()
    else:
        t = torch.from_numpy(np.ascontiguousarray(wl.target).view(np.int16)).cuda().view(
            torch.bfloat16)
    temps = torch.from_numpy(wl.temperature).cuda()
    req = torch.from_numpy(wl.request_ids.view(np.int32)).cuda()
    return d, t, temps, req


def np_(t):
    return None if t is None else t.cpu().numpy()


def gpu_q(wl, d=None, temps=None):
    if d is None:
        d, _, temps, _ = dev_inputs(wl)
    q = ds.q_build(d, temps, wl.top_k)
    torch.cuda.synchronize()
    return q


def oracle_q(wl):
    x = wl.draft.reshape(wl.B * wl.depth, wl.V)
    return O.q_build(x, wl.temperature, wl.top_k)


def compare_q(q, ref):
    """Bit-exact comparison of counts / ids / nnz / status."""
    counts, ids, nnz, status = ref
    assert np.array_equal(np_(q["status"]), status), "status differs"
    gc = np_(q["counts"]).view(np.uint32)
    bad = np.flatnonzero((gc != counts).any(axis=1))
    assert bad.size == 0, "counts differ in rows %s" % bad[:10]
    if q["top_k"] > 0:
        assert np.array_equal(np_(q["nnz"]), nnz)
        assert np.array_equal(np_(q["ids"]), ids)


def oracle_sample(wl, qref):
    counts, ids, nnz, _ = qref
    return O.draft_sample(counts, ids, nnz, wl.top_k, wl.B, wl.depth, wl.seed,
                          wl.request_ids, V=wl.V)


def oracle_verify(wl, mode, drafts, qref):
    z = wl.target_f32()
    counts, ids, nnz, _ = qref
    if mode == "greedy":
        acc, com, st = O.verify_greedy(z, drafts)
        return acc, com, np.zeros(wl.B, np.uint32), st
    return O.verify_ratio(z, drafts, counts, ids, nnz, wl.top_k, wl.seed, wl.request_ids)


def compare_verify(gpu, ref, mode):
    """Returns (unflagged mismatches, flagged mismatches, flagged requests,
    requests).  Integer outputs must match bit for bit, except on ratio
    requests that either side flags (a decision with |u*q - p| <= 1e-6*q, or
    a final draw within 1e-6 of a cumulative boundary)."""
    ga, gc, gf, gs = [np_(x) for x in gpu]
    ra, rc, rf, rs = ref
    if mode == "greedy":
        assert np.array_equal(gs, rs)
        assert np.array_equal(ga, ra)
        assert np.array_equal(gc, rc)
        return 0, 0, 0, ga.size
    gf = gf.view(np.uint32)
    flagged = ((gf & 3) != 0) | ((rf & 3) != 0)
    same = (ga == ra) & (gc == rc).all(axis=1) & (gs == rs)
    return (int((~same & ~flagged).sum()), int((~same & flagged).sum()), int(flagged.sum()),
            ga.size)
