"""Seeded synthetic inputs for the draft-sampling / verification path.

This module only draws logits; it holds none of the method's arithmetic and is
the one piece shared by the test suite (feeding both the CUDA library and the
CPU oracle) and the benchmark.  Every array comes from
``numpy.random.default_rng(1000 + config index)`` (PCG64) unless a seed is
given.  Shapes follow the anchor-as-first block of the remote DSpark drafter
contract (section 2): ``depth`` draft rows per request and ``depth + 1``
target rows (row j scores the token drafted at position j; row ``depth``
gives the bonus).  Vocabulary 129,280 and the noise token 128,799 are the
drafter's (same section).

Recipes (sizes at full scale):

* C1  B=1: draft ~ N(0, 2^2) fp32; target rows 0..4 = draft + N(0, 0.5^2),
  row 5 = an independent N(0, 2^2) row + N(0, 0.5^2); T = 1; dense q;
  greedy and ratio; Philox seed 0.
* C2  B=4: draft ~ N(0, 3^2) fp32 with the noise token masked to -inf;
  target = bf16(0.8 * unmasked draft + N(0, 1)) (not masked); T = 0.7;
  dense q; ratio; seed 1.
* C3  B=64: Zipf rows, logit(v) = -1.1 ln(rank(v)) + N(0, 0.3^2) with rank a
  seeded affine permutation of the ids (rank = (a v + b) mod V + 1, a coprime
  with V); target = draft + N(0, 0.7^2) fp32; sparse top-256 q; ratio; seed 2.
* C4  B=256: Zipf draft fp32, target = bf16(draft + N(0, 0.7^2)); per
  (request, position) exactly 10 % of ids (a seeded affine selection) masked
  to -inf in both the draft row and its target row (target row 5 has its own
  mask); 1 % of draft rows carry a top logit shared by g in {3, 5, 7} ids
  spread over the vocabulary (0.5 above the row's own maximum), so the draft
  argmax sits on g tied remainders.  In each such row two more unmasked
  ids, the tuners, get the logits (group logit - delta) and (group logit -
  delta_fine), the offsets chosen per row with the oracle
  (tests/golden/make_c4_ties.py, stored in tests/golden/c4_tie_rows.json) so
  that the group straddles the grant threshold: some of its members get the
  remaining ticket and the rest do not, and the lowest-id rule decides
  which; dense q; greedy and ratio; seed 3.
* C5  sweep B in {1, 8, 32, 128, 512, 1024} with the C3 generators, sparse
  top-256 or dense q, three target variants: ``mixed`` (as C3), ``accept``
  (draft argmax raised by 30 nats so q is one-hot, target = draft), and
  ``reject`` (+20 nats on 16 ids outside the draft's top 256 in every target
  row); seed 4.
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass, field
from math import gcd

import numpy as np

V_FULL = 129280
NOISE_TOKEN = 128799
DEPTH = 5
TOP_K = 256
SWEEP_B = (1, 8, 32, 128, 512, 1024)


@dataclass
class Workload:
    name: str
    B: int
    depth: int
    V: int
    draft: np.ndarray          # [B, depth, V] float32
    target: np.ndarray         # [B, depth+1, V] float32, or uint16 bf16 bit patterns
    target_dtype: str          # "f32" or "bf16"
    temperature: np.ndarray    # [B*depth] float32
    top_k: int                 # 0 = dense q
    seed: int                  # Philox seed of the draws
    modes: tuple               # verification modes run on this workload
    request_ids: np.ndarray    # [B] uint32
    notes: dict = field(default_factory=dict)

    def target_f32(self) -> np.ndarray:
        """Target logits as fp32 (bf16 widened exactly)."""
        if self.target_dtype == "f32":
            return self.target
        return (self.target.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.reshape(-1).view(np.uint32)
    out = np.empty(u.size, np.uint16)
    step = 1 << 24
    for s in range(0, u.size, step):
        c = u[s:s + step]
        r = (c >> 16) & 1
        r += c
        r += 0x7FFF  # no wrap for any non-NaN pattern (at most 0xFF807FFF)
        r >>= 16
        out[s:s + step] = r
    nan = np.isnan(x.reshape(-1))
    if nan.any():
        out[nan] = 0x7FC0
    return out.reshape(x.shape)


def _normal(rng, shape, sigma):
    out = rng.standard_normal(shape, dtype=np.float32)
    out *= np.float32(sigma)
    return out


def _affine_params(rng, n_rows, V):
    """Per row (a, b) of a seeded affine permutation v -> (a v + b) mod V."""
    a = np.empty(n_rows, np.int64)
    for i in range(n_rows):
        while True:
            cand = int(rng.integers(1, V)) if V > 1 else 1
            if gcd(cand, V) == 1:
                a[i] = cand
                break
    b = rng.integers(0, max(V, 1), size=n_rows, dtype=np.int64)
    return a, b


def _affine_ranks(a, b, V):
    v = np.arange(V, dtype=np.int64)
    return (a[:, None] * v[None, :] + b[:, None]) % V


def zipf_rows(rng, n_rows, V, slope=1.1, noise=0.3, chunk=64):
    """logit(v) = -slope * ln(rank(v) + 1) + N(0, noise^2), seeded permutation."""
    table = (-slope * np.log1p(np.arange(V, dtype=np.float64))).astype(np.float32)
    a, b = _affine_params(rng, n_rows, V)
    out = np.empty((n_rows, V), np.float32)
    for s in range(0, n_rows, chunk):
        e = min(n_rows, s + chunk)
        np.take(table, _affine_ranks(a[s:e], b[s:e], V), out=out[s:e])
        out[s:e] += _normal(rng, (e - s, V), noise)
    return out


def affine_masks(rng, n_rows, V, n_mask, chunk=64):
    """Per row exactly n_mask masked ids: those whose affine rank is < n_mask."""
    a, b = _affine_params(rng, n_rows, V)
    out = np.empty((n_rows, V), bool)
    for s in range(0, n_rows, chunk):
        e = min(n_rows, s + chunk)
        np.less(_affine_ranks(a[s:e], b[s:e], V), n_mask, out=out[s:e])
    return out


def _temps(B, depth, T):
    return np.full(B * depth, T, np.float32)


def _req(B):
    return np.arange(B, dtype=np.uint32)


def config1(B=1, V=V_FULL, depth=DEPTH, rng=None):
    rng = rng or np.random.default_rng(1001)
    xd = _normal(rng, (B, depth, V), 2.0)
    xt = np.empty((B, depth + 1, V), np.float32)
    xt[:, :depth] = xd + _normal(rng, (B, depth, V), 0.5)
    xt[:, depth] = _normal(rng, (B, V), 2.0) + _normal(rng, (B, V), 0.5)
    return Workload("C1 B=%d gaussian fp32 dense T=1" % B, B, depth, V, xd, xt, "f32",
                    _temps(B, depth, 1.0), 0, 0, ("greedy", "ratio"), _req(B))


def config2(B=4, V=V_FULL, depth=DEPTH, rng=None):
    rng = rng or np.random.default_rng(1002)
    raw = _normal(rng, (B, depth, V), 3.0)
    xd = raw.copy()
    if V > NOISE_TOKEN:
        xd[:, :, NOISE_TOKEN] = -np.inf
    t = np.empty((B, depth + 1, V), np.float32)
    t[:, :depth] = np.float32(0.8) * raw + _normal(rng, (B, depth, V), 1.0)
    t[:, depth] = np.float32(0.8) * _normal(rng, (B, V), 3.0) + _normal(rng, (B, V), 1.0)
    return Workload("C2 B=%d gaussian fp32 draft / bf16 target dense T=0.7" % B, B, depth, V,
                    xd, f32_to_bf16_bits(t), "bf16", _temps(B, depth, 0.7), 0, 1, ("ratio",),
                    _req(B))


def config3(B=64, V=V_FULL, depth=DEPTH, rng=None, top_k=TOP_K, variant="mixed", seed=2,
            name="C3"):
    rng = rng or np.random.default_rng(1003)
    xd = zipf_rows(rng, B * depth, V).reshape(B, depth, V)
    xt = np.empty((B, depth + 1, V), np.float32)
    if variant == "accept":
        am = xd.argmax(axis=2)
        bi, ji = np.meshgrid(np.arange(B), np.arange(depth), indexing="ij")
        xd[bi, ji, am] += np.float32(30.0)
        xt[:, :depth] = xd
    else:
        xt[:, :depth] = xd + _normal(rng, (B, depth, V), 0.7)
    xt[:, depth] = zipf_rows(rng, B, V) + _normal(rng, (B, V), 0.7)
    if variant == "reject":
        k = min(top_k if top_k > 0 else TOP_K, V)
        for b in range(B):
            for j in range(depth + 1):
                row = xd[b, min(j, depth - 1)]
                top = np.argpartition(-row, k - 1)[:k] if k < V else np.arange(V)
                pool = np.setdiff1d(np.arange(V), top)
                if pool.size == 0:
                    continue
                pick = rng.choice(pool, size=min(16, pool.size), replace=False)
                xt[b, j, pick] += np.float32(20.0)
    modes = ("ratio",) if name == "C3" else ("greedy", "ratio")
    return Workload("%s B=%d zipf fp32 %s %s" % (name, B, "top-%d" % top_k if top_k else "dense",
                                                  variant),
                    B, depth, V, xd, xt, "f32", _temps(B, depth, 1.0), top_k, seed, modes,
                    _req(B), {"variant": variant})


_C4_TIES = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "tests",
                        "golden", "c4_tie_rows.json")


def c4_tie_tuning():
    """The stored tuner offsets of the C4 tie rows (B = 256), or None."""
    try:
        with open(_C4_TIES) as f:
            return json.load(f)
    except OSError:
        return None


def config4(B=256, V=V_FULL, depth=DEPTH, rng=None, tie_fraction=0.01, mask_fraction=0.10,
            tuning="stored"):
    """tuning: "stored" applies the stored tuner offsets when they were made
    for this workload (B = 256 at full size, default generator), None leaves
    every tuner at its own Zipf logit (the raw rows the offsets are chosen on)."""
    table = c4_tie_tuning() if (tuning == "stored" and rng is None) else None
    if table is not None and (table.get("B"), table.get("V"), table.get("depth")) != (B, V, depth):
        table = None
    rng = rng or np.random.default_rng(1004)
    xd = zipf_rows(rng, B * depth, V).reshape(B, depth, V)
    n_mask = int(round(mask_fraction * V))
    masks = affine_masks(rng, B * (depth + 1), V, n_mask).reshape(B, depth + 1, V)
    tie_rows = []
    n_tie = max(1, int(round(tie_fraction * B * depth))) if V >= 16 else 0
    offsets = {(e["b"], e["j"]): (np.float32(float.fromhex(e["delta"])),
                                  np.float32(float.fromhex(e["delta_fine"])))
               for e in (table or {}).get("rows", [])}
    for r in rng.choice(B * depth, size=min(n_tie, B * depth), replace=False):
        b, j = divmod(int(r), depth)
        g = int(rng.choice([3, 5, 7]))
        free = np.flatnonzero(~masks[b, j])
        pick = rng.choice(free, size=g + 2, replace=False)
        ids = np.sort(pick[:g])
        tuners = [int(pick[g]), int(pick[g + 1])]
        top = np.float32(xd[b, j].max() + np.float32(0.5))
        xd[b, j, ids] = top
        if (b, j) in offsets:
            for t, dlt in zip(tuners, offsets[(b, j)]):
                xd[b, j, t] = np.float32(top - dlt)
        tie_rows.append((b, j, ids.tolist(), tuners))
    xt = np.empty((B, depth + 1, V), np.float32)
    xt[:, :depth] = xd + _normal(rng, (B, depth, V), 0.7)
    xt[:, depth] = zipf_rows(rng, B, V) + _normal(rng, (B, V), 0.7)
    for b in range(B):
        xd[b][masks[b, :depth]] = -np.inf
        xt[b][masks[b]] = -np.inf
    notes = {"tie_rows": tie_rows}
    if table is not None:
        notes.update({k: table[k] for k in ("tie_rows_straddling", "lowest_id_decisive_rows")
                      if k in table})
    return Workload("C4 B=%d zipf fp32 draft / bf16 target dense, 10%% mask, 1%% ties" % B, B,
                    depth, V, xd, f32_to_bf16_bits(xt), "bf16", _temps(B, depth, 1.0), 0, 3,
                    ("greedy", "ratio"), _req(B), notes)


def config5(B, variant="mixed", top_k=TOP_K, V=V_FULL, depth=DEPTH, rng=None):
    rng = rng or np.random.default_rng(1005)
    return config3(B=B, V=V, depth=depth, rng=rng, top_k=top_k, variant=variant, seed=4,
                   name="C5")


def by_name(name: str, **kw) -> Workload:
    """'c1'..'c4', or 'c5:<B>:<variant>:<sparse|dense>'; keyword B overrides the batch."""
    name = name.lower()
    if name.startswith("c5"):
        parts = name.split(":")
        B = int(parts[1]) if len(parts) > 1 else 1024
        B = kw.pop("B", B)
        variant = parts[2] if len(parts) > 2 else "mixed"
        q = parts[3] if len(parts) > 3 else "sparse"
        return config5(B, variant=variant, top_k=TOP_K if q == "sparse" else 0, **kw)
    return {"c1": config1, "c2": config2, "c3": config3, "c4": config4}[name](**kw)
