"""The certified float split of the dense q kernels (the float path of
q_dense.cuh and tp.cu), modelled on CPU with IEEE float32 / float64
arithmetic: whenever the split certifies itself, its floor and its fraction
bin floor(2048 r) equal those of the FP64 allocation a = RN64(E k),
k = RN64(2^24 / RN64(S)), computed directly; and it leaves only a small
fraction of elements to the exact integer path.  Every step of the model is
one correctly rounded float32 operation, as in the kernels."""
import numpy as np

F32, F64 = np.float32, np.float64
MARGIN = F32(0.5) - F32(2.0 ** -12) - F32(2.0 ** -15)


def weights(rng, n):
    """Integer-valued float32 weights E = floor(e 2^40), e in (2^-28, 1]."""
    d = rng.uniform(-19.0, 0.0, n)
    e = np.exp(d).astype(F32)
    return np.floor(e.astype(F64) * 2.0 ** 40).astype(F32)


def model(E, khi, klo):
    p1 = (E * khi).astype(F32)
    e1 = (E.astype(F64) * F64(khi) - p1.astype(F64)).astype(F32)  # exact: the fma residual
    p2 = (E * klo).astype(F32)
    f0 = np.floor(p1)
    fr = ((p1 - f0).astype(F32) + (e1 + p2).astype(F32)).astype(F32)
    fb = (fr * F32(2048.0)).astype(F32)
    G = np.floor(fb)
    cert = (np.abs(((fb - G).astype(F32) - F32(0.5)).astype(F32)) < MARGIN) & (f0 < F32(524285.0))
    f = f0.astype(np.int64) + np.floor_divide(G.astype(np.int64), 2048)
    b = np.mod(G.astype(np.int64), 2048)
    return cert, f, b


def exact(E, S):
    k = F64(2.0 ** 24) / F64(S)          # RN64(2^24 / RN64(S)); S < 2^53 here
    a = E.astype(F64) * k                 # RN64(E k)
    f = np.floor(a)
    r = a - f                             # exact
    return f.astype(np.int64), np.floor(r * 2048.0).astype(np.int64), r > 0


def test_certified_split_equals_fp64_allocation():
    rng = np.random.default_rng(2024)
    total = certified = 0
    for _ in range(20):
        S = int(rng.integers(1 << 40, 1 << 52))
        k = F64(2.0 ** 24) / F64(S)
        khi = F32(k)
        klo = F32(k - F64(khi))
        E = weights(rng, 50000)
        E = E[E <= S]
        cert, f, b = model(E, khi, klo)
        fx, bx, pos = exact(E, S)
        ok = cert & (E > 0)
        assert np.array_equal(f[ok], fx[ok])
        assert np.array_equal(b[ok], bx[ok])
        assert np.all(pos[ok])            # a certified element has r > 0
        total += int((E > 0).sum())
        certified += int(ok.sum())
    assert total > 500000
    assert total - certified < 2e-3 * total  # the exact path takes a small remainder


def test_certification_rejects_near_integer_fractions():
    # weights whose fraction 2048 r sits within 2^-13 of an integer are not certified
    S = 1 << 44
    k = F64(2.0 ** 24) / F64(S)           # a power of two: a = E 2^-20 exactly
    khi, klo = F32(k), F32(0.0)
    E = (np.arange(1, 4097, dtype=np.int64) << 9).astype(F32)   # fractions on the 2^-11 grid
    cert, f, b = model(E, khi, klo)
    assert not cert.any()
