"""Writes c4_tie_rows.json: for every tied-argmax row of the C4 workload
(B = 256, depth 5, V = 129,280), the offset delta of its tuner token's logit
and of a second, finer tuner below the tied group's, chosen so that the ORACLE's allocation of the row
splits the group at the grant threshold (some members get the remaining
ticket, the others do not: the lowest-id rule decides), and the number of
C4 draft rows whose grant the lowest-id rule decides at all.

"PP1 q transport and scheduling design", Distribution contract and
precision: the remaining tickets go to the largest remainders, ties by
lowest global token id.  The benchmark definition's C4 asks for 1 % of rows
whose draft argmax sits on tied remainders; the survey of the scope asks the
generator to keep re-drawing until the oracle confirms that the tied group
straddles the threshold.  Re-drawing at random succeeds about once in
N / g tries (N ~ 116,000 supported tokens), so the search steers instead:
one more token's weight moves the row's weight sum S, which moves the
group's remainder frac(2^64 / S) while leaving the other remainders almost
where they are.  The steering estimate below is only a guide; a row is
accepted only when the oracle's own counts show the split.

Test infrastructure: runs the oracle and numpy only.  Usage (repository
root): python tests/golden/make_c4_ties.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from draft_sampling_verification_gb300 import workloads as W  # noqa: E402
from oracle import oracle as O  # noqa: E402

M = 1 << 24
OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c4_tie_rows.json")


def remainders(E):
    """Steering guide: the FP64 split of the row's weights (floor, fraction)
    and the remaining tickets, as the method states them."""
    k = np.float64(M) / np.float64(int(E.sum()))
    a = E.astype(np.float64) * k
    f = np.floor(a)
    return a, a - f, M - int(f.sum())


def split_by_oracle(x, ids):
    counts, _, _, st = O.q_build(x[None, :], None, 0)
    c = counts[0, ids]
    return st[0] == 0 and c.min() != c.max(), counts[0]


def tune_row(x, ids, tuners, max_iter=120):
    """(delta, delta_fine) (float32) such that the oracle splits the group,
    or None.  The coarse tuner (about e^-2 of a member's weight) moves the
    group's remainder in steps of a few 1e-3; the fine one (about e^-17)
    in steps far below the window, whose width is about g / N."""
    g = len(ids)
    top = x[ids[0]]
    tc, tf = tuners
    deltas = [np.float32(2.0), np.float32(17.0)]
    fine_max = 2.0 ** 17
    for _ in range(max_iter):
        x[tc] = np.float32(top - deltas[0])
        x[tf] = np.float32(top - deltas[1])
        st, E, sup, S = O.q_weights_row(x)
        if st != 0:
            return None
        a, r, R = remainders(E)
        rt = r[ids[0]]
        above = int(np.count_nonzero(r[sup] > rt))
        at = int(np.count_nonzero(r[sup] == rt))
        if above < R < above + at:
            ok, _ = split_by_oracle(x, ids)
            if ok:
                return deltas
        # move the group's remainder to the middle of the window where
        # R - g < #(remainders above it) < R
        others = np.ones(x.size, bool)
        others[ids] = False
        rho = np.sort(r[sup & others])[::-1]
        # the widest gap (rho[i], rho[i - 1]) with R - g < i < R
        cand = [i for i in range(max(1, R - g + 1), R) if i < rho.size]
        if not cand:
            return None
        i = max(cand, key=lambda c: rho[c - 1] - rho[c])
        target = 0.5 * (rho[i] + rho[i - 1])
        d = target - rt
        d -= np.round(d)  # the nearest way round, in (-0.5, 0.5]
        dS = -d * float(E.sum()) / a[ids[0]]
        if abs(dS) < 1.0:
            # narrower than one unit of the fine tuner's weight: move the
            # coarse tuner by one step instead, which redraws the landscape
            deltas[0] = np.nextafter(deltas[0], np.float32(np.inf))
            continue
        Ef = float(E[tf]) + dS
        if 16.0 < Ef < fine_max:
            deltas[1] = np.float32(-np.log(Ef / 2.0 ** 40))
        else:
            Ec = float(E[tc]) + dS - (fine_max / 2 - float(E[tf]))
            if not (0.0 < Ec < 2.0 ** 40):
                return None
            deltas[0] = np.float32(-np.log(Ec / 2.0 ** 40))
            deltas[1] = np.float32(-np.log(fine_max / 2 / 2.0 ** 40))
    return None


def lowest_id_decides(counts, E, sup):
    """True if some tokens of equal weight (hence equal remainder) got
    different counts: the grant cut a group of equal remainders."""
    idx = np.flatnonzero(sup)
    order = np.lexsort((counts[idx], E[idx]))
    e, c = E[idx][order], counts[idx][order]
    same_e = e[1:] == e[:-1]
    return bool(np.any(same_e & (c[1:] != c[:-1])))


def main():
    wl = W.config4(tuning=None)
    rows = []
    for b, j, ids, tuners in wl.notes["tie_rows"]:
        x = wl.draft[b, j].copy()
        deltas = tune_row(x, np.array(ids), tuners)
        if deltas is None:
            raise SystemExit("no split found for row (%d, %d)" % (b, j))
        rows.append({"b": b, "j": j, "ids": ids, "tuners": tuners,
                     "delta": float(deltas[0]).hex(), "delta_fine": float(deltas[1]).hex()})
        print("row (%d, %d): g = %d, deltas %s %s" % (b, j, len(ids), deltas[0], deltas[1]),
              flush=True)
    table = {"B": wl.B, "V": wl.V, "depth": wl.depth, "rows": rows,
             "tie_rows_straddling": len(rows)}
    with open(OUT, "w") as f:
        json.dump(table, f, indent=1)
    # the tuned workload: every tie row split by the oracle; count the rows
    # the lowest-id rule decides
    wl = W.config4()
    n_dec = 0
    for b in range(wl.B):
        for j in range(wl.depth):
            st, E, sup, S = O.q_weights_row(wl.draft[b, j])
            counts, _, _, st2 = O.q_build(wl.draft[b, j][None, :], None, 0)
            n_dec += int(st == 0 and st2[0] == 0 and lowest_id_decides(counts[0], E, sup))
    for e in rows:
        ok, _ = split_by_oracle(wl.draft[e["b"], e["j"]], np.array(e["ids"]))
        assert ok, e
    table["lowest_id_decisive_rows"] = n_dec
    with open(OUT, "w") as f:
        json.dump(table, f, indent=1)
    print("tie rows split: %d; rows decided by the lowest-id rule: %d of %d"
          % (len(rows), n_dec, wl.B * wl.depth))


if __name__ == "__main__":
    main()
