"""GPU pins of the building blocks: the library's Philox and exp_ds weights
against the oracle (bit for bit, over large and exhaustive input sets), and
the oracle's Philox against cuRAND's Philox4_32_10 (a library routine, which
pins the round constants the CPU tests cannot)."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

from draft_sampling_verification_gb300 import _lib

pytestmark = pytest.mark.gpu


def _call(name, *args):
    rc = getattr(_lib.load(), name)(*args)
    assert rc == 0, (name, rc)


def lib_philox(ctr, seed):
    c = torch.from_numpy(ctr.view(np.int32)).cuda().contiguous()
    out = torch.empty_like(c)
    _call("dspark_debug_philox", ctypes.c_void_p(c.data_ptr()), seed, ctr.shape[0],
          ctypes.c_void_p(out.data_ptr()), None)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32)


def lib_weights(d):
    dt = torch.from_numpy(d).cuda()
    e = torch.empty_like(dt)
    E = torch.empty(d.size, dtype=torch.int64, device="cuda")
    _call("dspark_debug_exp_weights", ctypes.c_void_p(dt.data_ptr()), d.size,
          ctypes.c_void_p(e.data_ptr()), ctypes.c_void_p(E.data_ptr()), None)
    torch.cuda.synchronize()
    return e.cpu().numpy(), E.cpu().numpy().view(np.uint64)


def test_library_philox_matches_oracle(oracle):
    rng = np.random.default_rng(0)
    n = 20000
    ctr = rng.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    ctr[:100, 3] = 0
    for seed in (0, 1, 0xDEADBEEFCAFEF00D):
        out = lib_philox(ctr, seed)
        key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
        for i in range(0, n, 97):
            assert np.array_equal(out[i], oracle.philox4x32_10(ctr[i], key)), (seed, i)


CURAND_SRC = r"""
#include <curand_kernel.h>
#include <cstdint>
__global__ void k(const unsigned long long* seed, const unsigned long long* subseq,
                  const unsigned long long* offset, uint4* out, int n) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  curandStatePhilox4_32_10_t st;
  curand_init(seed[i], subseq[i], offset[i], &st);
  out[i] = curand4(&st);
}
extern "C" int run(const unsigned long long* seed, const unsigned long long* subseq,
                   const unsigned long long* offset, uint4* out, int n) {
  k<<<(n + 127) / 128, 128>>>(seed, subseq, offset, out, n);
  return (int)cudaDeviceSynchronize();
}
"""


@pytest.fixture(scope="module")
def curand_lib():
    d = tempfile.mkdtemp()
    src = os.path.join(d, "pin.cu")
    so = os.path.join(d, "pin.so")
    open(src, "w").write(CURAND_SRC)
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                    "-Xcompiler", "-fPIC", "-o", so, src], check=True)
    return ctypes.CDLL(so)


def test_oracle_philox_matches_curand(oracle, curand_lib):
    # curand_init(seed, subsequence, offset) starts Philox4_32_10 at counter
    # (offset/4 as the low 64 bits, subsequence as the high 64 bits) with key
    # (seed low, seed high); curand4 then returns the block at that counter.
    rng = np.random.default_rng(1)
    n = 4096
    a = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64)
    b = rng.integers(0, 2 ** 20, size=n, dtype=np.uint64)
    c = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64)
    dd = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64)
    seed = rng.integers(0, 2 ** 63, size=n, dtype=np.uint64)
    seed[:8] = 0
    a[:8] = 0
    offset = (a + (b << np.uint64(32))) * np.uint64(4)
    subseq = c + (dd << np.uint64(32))
    t = [torch.from_numpy(x.view(np.int64)).cuda() for x in (seed, subseq, offset)]
    out = torch.empty((n, 4), dtype=torch.int32, device="cuda")
    rc = curand_lib.run(*[ctypes.c_void_p(x.data_ptr()) for x in t],
                        ctypes.c_void_p(out.data_ptr()), n)
    assert rc == 0
    got = out.cpu().numpy().view(np.uint32)
    for i in range(n):
        ctr = np.array([a[i], b[i], c[i], dd[i]], np.uint64).astype(np.uint32)
        key = np.array([int(seed[i]) & 0xFFFFFFFF, int(seed[i]) >> 32], np.uint32)
        assert np.array_equal(got[i], oracle.philox4x32_10(ctr, key)), i


def _float_range(lo, hi, step):
    bl = int(np.array([lo], np.float32).view(np.uint32)[0])
    bh = int(np.array([hi], np.float32).view(np.uint32)[0])
    a, b = min(bl, bh), max(bl, bh)
    return np.arange(a, b + 1, step, dtype=np.uint64).astype(np.uint32).view(np.float32)


@pytest.mark.parametrize("lo,hi,step", [(-0.0, -1.0, 31), (-1.0, -28.0, 29), (-28.0, -87.5, 7)])
def test_library_exp_weights_bit_exact(oracle, lo, hi, step):
    d = _float_range(lo, hi, step)
    d = np.concatenate([d, np.array([0.0, -0.0, -np.inf, -87.0, -28.0, -27.999998, -30.0,
                                     -29.999998, -100.0, -1e30, -3.4e38], np.float32)])
    e, E = lib_weights(d)
    ref = oracle.exp_ds(d)
    assert np.array_equal(e.view(np.uint32), ref.view(np.uint32))
    refE = np.floor(ref.astype(np.float64) * 2.0 ** 40).astype(np.uint64)
    assert np.array_equal(E, refE)


def test_library_exp_weights_every_float(oracle):
    """Every fp32 d in [-28, 0] (1.1e9 values, where the integer weight
    floor(exp_ds(d) * 2^40) is not zero) and +0, chunk by chunk: the
    library's exp_ds and weight bit for bit equal to the oracle's.  The
    clamp region below -28 (weight 0, then exp_ds 0 below -87) is sampled in
    the test above."""
    from concurrent.futures import ThreadPoolExecutor
    lo = int(np.array([-0.0], np.float32).view(np.uint32)[0])      # 0x80000000
    hi = int(np.array([-28.0], np.float32).view(np.uint32)[0])     # 0xC1E00000
    chunk = 1 << 26
    dev = torch.device("cuda")
    e = torch.empty(chunk, dtype=torch.float32, device=dev)
    E = torch.empty(chunk, dtype=torch.int64, device=dev)

    def oracle_part(d):  # the oracle's C loop runs with the GIL released
        return oracle.exp_ds(d)

    with ThreadPoolExecutor(max_workers=16) as pool:
        starts = list(range(lo, hi + 1, chunk)) + [None]
        for a in starts:
            if a is None:  # +0 and the first negative patterns once more
                bits = np.array([0, lo, lo + 1, hi], np.uint32)
            else:
                bits = np.arange(a, min(hi + 1, a + chunk), dtype=np.uint64).astype(np.uint32)
            d = bits.view(np.float32)
            n = d.size
            dt = torch.from_numpy(d).to(dev)
            _call("dspark_debug_exp_weights", ctypes.c_void_p(dt.data_ptr()), n,
                  ctypes.c_void_p(e.data_ptr()), ctypes.c_void_p(E.data_ptr()), None)
            parts = np.array_split(d, 16)
            ref = np.concatenate(list(pool.map(oracle_part, parts)))
            torch.cuda.synchronize()
            ge = e[:n].cpu().numpy()
            gE = E[:n].cpu().numpy().view(np.uint64)
            bad = np.flatnonzero(ge.view(np.uint32) != ref.view(np.uint32))
            assert bad.size == 0, ("exp_ds", d[bad[:5]])
            refE = np.floor(ref.astype(np.float64) * 2.0 ** 40).astype(np.uint64)
            bad = np.flatnonzero(gE != refE)
            assert bad.size == 0, ("weight", d[bad[:5]])


def test_library_alloc_scale_matches_fp64():
    """k = RN64(2^24 / RN64(S)), khi = RN32(k), klo = RN32(k - khi) from the
    kernels' integer arithmetic equal numpy's FP64 / FP32 roundings."""
    rng = np.random.default_rng(5)
    S = [rng.integers(1 << 40, 1 << 57, size=20000, dtype=np.uint64)]
    edges = []
    for e in range(40, 58):
        for d in (-3, -2, -1, 0, 1, 2, 3):
            edges.append((1 << e) + d)
        edges.append((1 << e) + (1 << max(0, e - 53)))      # a tie at the 53-bit rounding
        edges.append((1 << e) + 3 * (1 << max(0, e - 54)))
    S.append(np.array(edges, np.uint64))
    S.append(np.array([1, 2, 3, 129280 << 40, (1 << 57) - 1], np.uint64))
    S = np.concatenate(S)
    St = torch.from_numpy(S.view(np.int64)).cuda()
    mk = torch.empty_like(St)
    ek = torch.empty(S.size, dtype=torch.int32, device="cuda")
    khi = torch.empty(S.size, dtype=torch.float32, device="cuda")
    klo = torch.empty(S.size, dtype=torch.float32, device="cuda")
    _call("dspark_debug_alloc_scale", ctypes.c_void_p(St.data_ptr()), S.size,
          ctypes.c_void_p(mk.data_ptr()), ctypes.c_void_p(ek.data_ptr()),
          ctypes.c_void_p(khi.data_ptr()), ctypes.c_void_p(klo.data_ptr()), None)
    torch.cuda.synchronize()
    kd = np.float64(2.0 ** 24) / S.astype(np.float64)
    bits = kd.view(np.uint64)
    ref_mk = (bits & np.uint64((1 << 52) - 1)) | np.uint64(1 << 52)
    ref_ek = ((bits >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64) - 1075
    ref_khi = kd.astype(np.float32)
    ref_klo = (kd - ref_khi.astype(np.float64)).astype(np.float32)
    assert np.array_equal(mk.cpu().numpy().view(np.uint64), ref_mk)
    assert np.array_equal(ek.cpu().numpy().astype(np.int64), ref_ek)
    assert np.array_equal(khi.cpu().numpy().view(np.uint32), ref_khi.view(np.uint32))
    assert np.array_equal(klo.cpu().numpy().view(np.uint32), ref_klo.view(np.uint32))
