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


# Ratio and match verification flags.  The GPU sets AMBIG_ACCEPT and
# NEAR_BOUNDARY (absolute band) from its own fp32 p; the oracle sets the same
# two from FP64 p, and NEAR_BOUNDARY_REL, the band relative to the picked
# token's own mass.  Only the oracle's flags excuse a request, and only those
# of the benchmark definition's band (AMBIG_ACCEPT or NEAR_BOUNDARY).
F_AMBIG, F_NEAR, F_NEAR_REL = 1, 2, 8
BAND_BOUND = 1e-4  # band cases per verify row


class VerifyCounts:
    """Counts of one comparison of the GPU's verification outputs with the
    oracle's, or a sum of them.

    requests, rows        requests compared, their verify rows (depth + 1 each)
    ambig                 oracle: a ratio decision with |u*q - p| <= 1e-6*q
    near_abs / near_rel   oracle: the final draw within 1e-6 (probability
                          units) / within 1e-6 of the picked token's own mass
                          of a cumulative boundary
    band_abs / band_rel   oracle band cases under the absolute / relative
                          reading of the draw's band (ambig counts in both)
    gpu_only              the GPU flags a request that the oracle does not
                          (not an excuse: such a request must match)
    mismatch              requests whose outputs differ outside the oracle's
                          band (absolute reading, the definition's): must be 0
    band_mismatch         requests whose outputs differ inside it (allowed)
    rel_mismatch          requests whose outputs differ outside the relative
                          band (what that reading's parity would count)
    """
    FIELDS = ("requests", "rows", "ambig", "near_abs", "near_rel", "band_abs", "band_rel",
              "gpu_only", "mismatch", "band_mismatch", "rel_mismatch")

    def __init__(self, **kw):
        for f in self.FIELDS:
            setattr(self, f, int(kw.get(f, 0)))

    def __iadd__(self, o):
        for f in self.FIELDS:
            setattr(self, f, getattr(self, f) + getattr(o, f))
        return self

    def as_dict(self):
        return {f: getattr(self, f) for f in self.FIELDS}

    def __repr__(self):
        return "VerifyCounts(%s)" % ", ".join("%s=%d" % kv for kv in self.as_dict().items())


# every comparison of the session, by mode, for the summary pytest prints
SESSION = {}


def record(mode, c):
    SESSION.setdefault(mode, VerifyCounts())
    SESSION[mode] += c


def compare_verify(gpu, ref, mode):
    """Compares one batch of GPU verification outputs (accept_len, committed,
    flags, status) with the oracle's and returns VerifyCounts.  Greedy
    outputs must be bit-exact (asserted here).  Ratio / match outputs must be
    bit-exact on every request the oracle does not put in the band (counted
    in `mismatch`, asserted by the caller); the GPU's own flags excuse
    nothing."""
    ga, gc, gf, gs = [np_(x) for x in gpu]
    ra, rc, rf, rs = ref
    n = ga.size
    rows = n * gc.shape[1]  # depth + 1 verify rows per request
    if mode == "greedy":
        assert np.array_equal(gs, rs)
        assert np.array_equal(ga, ra)
        assert np.array_equal(gc, rc)
        c = VerifyCounts(requests=n, rows=rows)
        record(mode, c)
        return c
    gf = gf.view(np.uint32)
    rf = np.asarray(rf).view(np.uint32)
    ambig = (rf & F_AMBIG) != 0
    near_abs = (rf & F_NEAR) != 0
    near_rel = (rf & F_NEAR_REL) != 0
    band_abs = ambig | near_abs
    band_rel = ambig | near_rel
    gpu_only = ((gf & (F_AMBIG | F_NEAR)) != 0) & ~band_abs
    same = (ga == ra) & (gc == rc).all(axis=1) & (gs == rs)
    c = VerifyCounts(requests=n, rows=rows, ambig=ambig.sum(), near_abs=near_abs.sum(),
                     near_rel=near_rel.sum(), band_abs=band_abs.sum(), band_rel=band_rel.sum(),
                     gpu_only=gpu_only.sum(), mismatch=(~same & ~band_abs).sum(),
                     band_mismatch=(~same & band_abs).sum(),
                     rel_mismatch=(~same & ~band_rel).sum())
    record(mode, c)
    return c
