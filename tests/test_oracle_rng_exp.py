"""Pins of the oracle's Philox4x32-10 and of its deterministic exp (exp_ds).

exp_ds is pinned against numpy's float64 exp (a library routine) and its
mathematical properties; Philox on the CPU by its avalanche behaviour and
output uniformity, and bit for bit by cuRAND's Philox4_32_10 in the GPU test
``test_gpu_rng.py``.
"""
import numpy as np
import pytest


def _floats_between(lo_bits, hi_bits, step):
    return np.arange(lo_bits, hi_bits, step, dtype=np.uint64).astype(np.uint32).view(np.float32)


def test_exp_ds_error_below_one_ulp(oracle):
    # a dense sample of every negative float in [-87, 0] (every 53rd bit pattern)
    d = _floats_between(0x80000000, 0xC2AE0001, 53)
    d = d[(d >= -87.0) & (d <= 0.0)]
    e = oracle.exp_ds(d).astype(np.float64)
    ref = np.exp(d.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    err = np.abs(e - ref) / ulp
    assert err.max() <= 1.0, (err.max(), d[err.argmax()])


def test_exp_ds_special_values(oracle):
    d = np.array([0.0, -0.0, -np.inf, -87.0, -87.00001, -1000.0, -1e-30], np.float32)
    e = oracle.exp_ds(d)
    assert e[0] == 1.0 and e[1] == 1.0
    assert e[2] == 0.0 and e[4] == 0.0 and e[5] == 0.0
    assert e[3] > 0.0 and np.isfinite(e[3]) and e[3] >= np.float32(2.0 ** -126)
    assert e[6] == 1.0


def test_exp_ds_never_above_one_and_monotone(oracle):
    # windows of consecutive floats around every switch of n = rint(d/ln2)
    # and near 0, checked for monotonicity float by float
    windows = [np.float32(-0.0)]
    for n in range(0, 126):
        windows.append(np.float32(-(n + 0.5) * np.log(2.0)))
    for c in windows:
        b = int(np.array([c], np.float32).view(np.uint32)[0])
        lo = max(b - 4000, 0x80000000)
        d = np.arange(lo, b + 4000, dtype=np.uint64).astype(np.uint32).view(np.float32)
        d = d[(d >= -87.0) & (d <= 0.0)]
        d = np.sort(d)
        e = oracle.exp_ds(d)
        assert np.all(np.diff(e.astype(np.float64)) >= 0.0)
        assert e.max() <= 1.0


def test_exp_ds_weight_vanishes_below_minus_28(oracle):
    # exhaustive over every float in [-87, -28): floor(exp_ds(d) * 2^40) == 0,
    # i.e. such tokens get integer weight 0 whatever the row
    lo = int(np.array([-28.0], np.float32).view(np.uint32)[0]) + 1
    hi = int(np.array([-87.0], np.float32).view(np.uint32)[0]) + 1
    d = np.arange(lo, hi, dtype=np.uint64).astype(np.uint32).view(np.float32)
    e = oracle.exp_ds(d).astype(np.float64)
    assert np.all(np.floor(e * 2.0 ** 40) == 0.0)
    # and just above -28 the weight is still positive
    assert np.floor(float(oracle.exp_ds(np.array([-27.0], np.float32))[0]) * 2.0 ** 40) > 0


def test_philox_avalanche(oracle):
    rng = np.random.default_rng(7)
    flips = []
    for _ in range(24):
        ctr = rng.integers(0, 2 ** 32, size=4, dtype=np.uint64).astype(np.uint32)
        key = rng.integers(0, 2 ** 32, size=2, dtype=np.uint64).astype(np.uint32)
        base = oracle.philox4x32_10(ctr, key)
        for bit in range(192):
            c2, k2 = ctr.copy(), key.copy()
            if bit < 128:
                c2[bit // 32] ^= np.uint32(1 << (bit % 32))
            else:
                k2[(bit - 128) // 32] ^= np.uint32(1 << (bit % 32))
            out = oracle.philox4x32_10(c2, k2)
            flips.append(int(np.unpackbits((base ^ out).view(np.uint8)).sum()))
    flips = np.array(flips)
    # 10 rounds mix completely: mean 64 of 128 bits, no input bit leaves
    # the output nearly unchanged
    assert abs(flips.mean() - 64.0) < 0.5
    assert flips.min() >= 30


def test_philox_counter_words_all_matter_and_outputs_uniform(oracle):
    # word 0 of consecutive counters (request ids) is uniform: chi-square on
    # the top 8 bits over 2^16 draws
    draws = np.array([oracle.draw_u32(12345, r, 3, 1) for r in range(1 << 16)], np.uint64)
    hist = np.bincount((draws >> 24).astype(np.int64), minlength=256)
    expected = (1 << 16) / 256.0
    chi2 = ((hist - expected) ** 2 / expected).sum()
    assert chi2 < 340.0  # 255 dof, p ~ 3e-4
    # every counter word and both key halves change the draw
    base = oracle.draw_u32(0, 0, 0, 0)
    assert oracle.draw_u32(0, 1, 0, 0) != base
    assert oracle.draw_u32(0, 0, 1, 0) != base
    assert oracle.draw_u32(0, 0, 0, 1) != base
    assert oracle.draw_u32(1, 0, 0, 0) != base
    assert oracle.draw_u32(1 << 32, 0, 0, 0) != base
    out = oracle.philox4x32_10([0, 0, 0, 1], [0, 0])
    assert int(out[0]) != base
