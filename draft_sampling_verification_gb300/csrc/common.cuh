// common.cuh -- device helpers shared by the library's kernels: Philox4x32-10,
// the deterministic fp32 exponential exp_ds, the exact FP64 allocation split,
// logit loads and block / cluster reductions.
//
// Everything on the q path must round exactly as written (IEEE RN, no FTZ,
// no contraction): those expressions use the explicit __f*_rn intrinsics.
#pragma once

#include <cooperative_groups.h>
#include <cstdint>
#include <cuda_runtime.h>

#include "dspark.h"

namespace cg = cooperative_groups;

namespace dspark {

constexpr uint32_t kM = DSPARK_M;

// ------------------------------------------------- bounds-checked build
// In the checked build of the library (compiled with DSPARK_CHECKED), every
// DSPARK_CHECK(cond) site tests an index against its bound before the access
// it guards; a failing site skips the access (a load yields a neutral value)
// and is recorded in this translation unit's counters: the number of
// failures and the first failing site (source line + 10000 * DSPARK_TU, the
// file's number).  dspark_checked_status reads and clears them.  No trap, no
// assert.  In the normal build the macro is the constant true: the condition
// is not even evaluated.
#ifndef DSPARK_TU
#define DSPARK_TU 0
#endif
#ifdef DSPARK_CHECKED
static __device__ uint32_t g_check_fail;
static __device__ uint32_t g_check_site;
__device__ __forceinline__ bool check_ok(bool ok, uint32_t site) {
  if (!ok) {
    atomicAdd(&g_check_fail, 1u);
    atomicCAS(&g_check_site, 0u, site);
  }
  return ok;
}
#define DSPARK_CHECK(cond) (::dspark::check_ok((cond), (uint32_t)(__LINE__ + 10000 * DSPARK_TU)))
// this translation unit's counters added into out[0] (failures) and out[1]
// (first site, if none yet), then cleared (host; synchronises the device)
static inline cudaError_t check_collect(uint32_t* out) {
  uint32_t v[2] = {0u, 0u};
  cudaError_t e = cudaMemcpyFromSymbol(&v[0], g_check_fail, 4);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v[1], g_check_site, 4);
  const uint32_t zero = 0u;
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_check_fail, &zero, 4);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_check_site, &zero, 4);
  out[0] += v[0];
  if (out[1] == 0u) out[1] = v[1];
  return e;
}
#define DSPARK_CHECK_COLLECTOR(name) \
  cudaError_t dspark_check_collect_##name(uint32_t* out) { return ::dspark::check_collect(out); }
#else
#define DSPARK_CHECK(cond) true
#define DSPARK_CHECK_COLLECTOR(name)
#endif

// ---------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies of
// counter words 0 and 2 (multipliers 0xD2511F53, 0xCD9E8D57); the key is
// advanced by the Weyl increments 0x9E3779B9, 0xBB67AE85 between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    if (i > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Word 0 of Philox(key = seed, counter = (request, row, purpose, 0)).
__device__ __forceinline__ uint32_t draw_u32(uint64_t seed, uint32_t request, uint32_t row,
                                             uint32_t purpose) {
  return philox4x32_10(make_uint4(request, row, purpose, 0u), (uint32_t)seed,
                       (uint32_t)(seed >> 32))
      .x;
}

// ----------------------------------------------------------------- exp_ds
// Deterministic fp32 e^d for d <= 0 (0 below -87): Cody-Waite reduction
// n = rint(d * log2(e)), r = d - n*ln2 with ln2 split into a 16-bit-fraction
// high part (n*hi exact for |n| <= 127) and the float nearest the rest, then
// the degree-7 Taylor polynomial of e^r in Horner form (one fma per step) and
// an exact scaling by 2^n.  Constants: float nearest 1/ln2; ln2 truncated
// to 16 fraction bits; float nearest (ln2 - that); floats nearest 1/k!.
constexpr float kL2E = 0x1.715476p+0f;
constexpr float kLn2Hi = 0x1.62e4p-1f;
constexpr float kLn2Lo = 0x1.7f7d1cp-20f;
constexpr float kInvFact2 = 0x1p-1f;
constexpr float kInvFact3 = 0x1.555556p-3f;
constexpr float kInvFact4 = 0x1.555556p-5f;
constexpr float kInvFact5 = 0x1.111112p-7f;
constexpr float kInvFact6 = 0x1.6c16c2p-10f;
constexpr float kInvFact7 = 0x1.a01a02p-13f;

// rint(t) for |t| < 2^22 by adding and removing 1.5 * 2^23 (each addition
// rounds to nearest, ties to even, exactly once); *ni gets rint(t) as int.
__device__ __forceinline__ float rint_magic(float t, int* ni) {
  const float tm = __fadd_rn(t, 12582912.0f);
  *ni = __float_as_int(tm) - 0x4B400000;
  return __fsub_rn(tm, 12582912.0f);
}

// exp_ds(d) * 2^k for d in [-87, 0]: the scaling by 2^(n + k) is an exact
// add to the exponent field of p (p is in [0.7, 1.42)), valid while the
// result stays a normal float, i.e. n + k >= -126.
__device__ __forceinline__ float exp_ds_pow2(float d, int k) {
  int ni;
  const float n = rint_magic(__fmul_rn(d, kL2E), &ni);
  float r = __fmaf_rn(-n, kLn2Hi, d);
  r = __fmaf_rn(-n, kLn2Lo, r);
  float p = kInvFact7;
  p = __fmaf_rn(p, r, kInvFact6);
  p = __fmaf_rn(p, r, kInvFact5);
  p = __fmaf_rn(p, r, kInvFact4);
  p = __fmaf_rn(p, r, kInvFact3);
  p = __fmaf_rn(p, r, kInvFact2);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  return __int_as_float(__float_as_int(p) + ((ni + k) << 23));
}

__device__ __forceinline__ float exp_ds(float d) {
  if (!(d >= -87.0f)) return 0.0f;
  return exp_ds_pow2(d, 0);
}

// floor(exp_ds(d) * 2^40) as an exact float for any d <= 0 (or -inf): the
// distance is clamped at -30, where, as everywhere below -28, the weight is 0.
__device__ __forceinline__ float weight40(float d) {
  return floorf(exp_ds_pow2(fmaxf(d, -30.0f), 40));
}

// ------------------------------------------------- packed fp32x2 arithmetic
// Two fp32 lanes per instruction (sm_100 and later).  Written as inline PTX
// with an explicit rounding modifier so that no multiply and add are ever
// contracted into one fma: each lane is exactly the single-rounded scalar
// operation named (mul / add / fma, .rn or .rm).
__device__ __forceinline__ uint64_t f2_pack(float2 v) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(d);
}
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(d);
}
__device__ __forceinline__ float2 add2_rm(float2 a, float2 b) {  // rounded down
  uint64_t d;
  asm("add.rm.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_pack(a)), "l"(f2_pack(b)));
  return f2_unpack(d);
}
__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(f2_pack(a)), "l"(f2_pack(b)), "l"(f2_pack(c)));
  return f2_unpack(d);
}
__device__ __forceinline__ float2 fma2_rm(float2 a, float2 b, float2 c) {  // rounded down
  uint64_t d;
  asm("fma.rm.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(f2_pack(a)), "l"(f2_pack(b)), "l"(f2_pack(c)));
  return f2_unpack(d);
}
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

// weight40 of two distances at once, the reduction and the polynomial on the
// packed fp32x2 pipe: every lane goes through exactly the single-rounded
// operations of weight40, so each result is bit-identical to weight40 of
// that lane.  Differences from the scalar sequence, all exact: the rint
// offset carries the +40 of the scaling (1.5 * 2^23 + 40 rounds t as
// 1.5 * 2^23 does, the parity of the offset being even), so the bits of tm
// shifted left by 23 are (n + 40) << 23 modulo 2^32 (the offset's own bits
// vanish there); fma(n, -c, x) equals fma(-n, c, x).  The rounding of
// t = RN(d * log2(e)) to an integer decides ties (t = k + 1/2 exactly), so
// that step stays on the scalar pipe: a packed product feeding a packed add
// measured different there (the rounding of the product was not seen), while
// the scalar pair matches the oracle on every float.
__device__ __forceinline__ float2 weight40x2(float2 d) {
  constexpr float kMag40 = 12582952.0f;  // 1.5 * 2^23 + 40
  d.x = fmaxf(d.x, -30.0f);
  d.y = fmaxf(d.y, -30.0f);
  const float2 tm = make_float2(__fadd_rn(__fmul_rn(d.x, kL2E), kMag40),
                                __fadd_rn(__fmul_rn(d.y, kL2E), kMag40));
  const float2 n = add2_rn(tm, f2(-kMag40));
  float2 r = fma2_rn(n, f2(-kLn2Hi), d);
  r = fma2_rn(n, f2(-kLn2Lo), r);
  float2 q = fma2_rn(f2(kInvFact7), r, f2(kInvFact6));
  q = fma2_rn(q, r, f2(kInvFact5));
  q = fma2_rn(q, r, f2(kInvFact4));
  q = fma2_rn(q, r, f2(kInvFact3));
  q = fma2_rn(q, r, f2(kInvFact2));
  q = fma2_rn(q, r, f2(1.0f));
  q = fma2_rn(q, r, f2(1.0f));
  const float ex = __int_as_float(__float_as_int(q.x) + (__float_as_int(tm.x) << 23));
  const float ey = __int_as_float(__float_as_int(q.y) + (__float_as_int(tm.y) << 23));
  return make_float2(floorf(ex), floorf(ey));
}

// Integer weight E = floor(exp_ds(d) * 2^40) of a token at distance d <= 0
// from the row maximum.  Below d = -28 the weight is 0 for every float d
// (exp_ds(d) < 2^-40 there), so the polynomial is skipped.
__device__ __forceinline__ float weight_float(float d) {
  return (d >= -28.0f) ? exp_ds(d) : 0.0f;
}

// E = floor(e * 2^40) for e in {0} U [2^-126, 1], returned as (Ei, se) with
// E = Ei << se and Ei < 2^24.
__device__ __forceinline__ void weight_split(float e, uint32_t* Ei, int* se) {
  const uint32_t b = __float_as_uint(e);
  const int ef = (int)(b >> 23);  // e >= 0
  const uint32_t p24 = (b & 0x7FFFFFu) | 0x800000u;
  const int sh = ef - 110;  // e = p24 * 2^(ef-150); E = p24 * 2^(ef-110) floored
  if (e == 0.0f || sh <= -24) {
    *Ei = 0u;
    *se = 0;
  } else if (sh >= 0) {
    *Ei = p24;
    *se = sh;
  } else {
    *Ei = p24 >> (-sh);
    *se = 0;
  }
}

// E as (Ei, se) from its exact float value Ef (an integer < 2^41 with at most
// 24 significant bits): E = Ei << se.
__device__ __forceinline__ void weight_split_ef(float Ef, uint32_t* Ei, int* se) {
  const uint32_t b = __float_as_uint(Ef);
  const int ex = (int)(b >> 23);
  const uint32_t m24 = (b & 0x7FFFFFu) | 0x800000u;
  if (Ef == 0.0f) {
    *Ei = 0u;
    *se = 0;
  } else if (ex >= 150) {
    *Ei = m24;
    *se = ex - 150;
  } else {
    *Ei = m24 >> (150 - ex);  // exact: Ef is an integer
    *se = 0;
  }
}

__device__ __forceinline__ uint64_t weight_u64(float e) {
  uint32_t Ei;
  int se;
  weight_split(e, &Ei, &se);
  return (uint64_t)Ei << se;
}

// ------------------------------------------------- FP64 allocation split
// k = RN64(2^24 / RN64(S)) is passed as mk * 2^ek (mk in [2^52, 2^53)).
// a = RN64(E * k) is computed exactly with integer arithmetic (the product
// of a <= 24-bit E and the 53-bit mk rounded to 53 bits, ties to even),
// which is bit-identical to the FP64 multiply.  a = A * 2^-t with t >= 28;
// floor(a) = A >> t; the fraction is r = (A mod 2^t) * 2^-t.
struct AllocSplit {
  uint32_t f;      // floor(a)  (<= 2^24)
  uint64_t rnum;   // A mod 2^t
  int t;           // fraction bits
};

__device__ __forceinline__ AllocSplit alloc_split(uint32_t Ei, int se, uint64_t mk, int ek) {
  AllocSplit out;
  if (Ei == 0u) {
    out.f = 0u;
    out.rnum = 0ull;
    out.t = 64;
    return out;
  }
  const unsigned __int128 P = (unsigned __int128)Ei * (unsigned __int128)mk;  // < 2^77
  const uint64_t Phi = (uint64_t)(P >> 64);
  const int nb = Phi ? (128 - __clzll((long long)Phi)) : (64 - __clzll((long long)(uint64_t)P));
  int s = nb - 53;  // >= 0 since P >= 2^52
  uint64_t A;
  if (s == 0) {
    A = (uint64_t)P;
  } else {
    A = (uint64_t)(P >> s);
    const uint64_t rem = (uint64_t)P & ((1ull << s) - 1ull);  // s <= 24
    const uint64_t half = 1ull << (s - 1);
    if (rem > half || (rem == half && (A & 1ull))) ++A;
    if (A == (1ull << 53)) {
      A >>= 1;
      ++s;
    }
  }
  const int t = -(s + se + ek);
  out.t = t;
  if (t >= 64) {
    out.f = 0u;
    out.rnum = A;
  } else {
    out.f = (uint32_t)(A >> t);
    out.rnum = A & ((1ull << t) - 1ull);
  }
  return out;
}

// Bucket of the fraction: floor(r * 4096).
__device__ __forceinline__ uint32_t frac_bucket(const AllocSplit& a) {
  const int sh = a.t - 12;
  return (sh >= 64) ? 0u : (uint32_t)(a.rnum >> sh);
}

// Exact fraction r = rnum * 2^-t as its FP64 bit pattern (monotone in r,
// equal for equal r), built with integer operations: rnum < 2^53, so the
// double is exact and normal for the t that occur (t <= ~90).
__device__ __forceinline__ uint64_t frac_key(const AllocSplit& a) {
  if (a.rnum == 0ull) return 0ull;
  const int nb = 64 - __clzll((long long)a.rnum);        // bits of rnum, 1..53
  const uint64_t mant = a.rnum << (53 - nb);              // [2^52, 2^53)
  const uint64_t bexp = (uint64_t)(1023 + (nb - 1) - a.t);
  return (bexp << 52) | (mant & ((1ull << 52) - 1ull));
}

// The allocation scale k = RN64(2^24 / RN64(S)) for S >= 1, exactly as the
// FP64 operations would round it, with integer arithmetic only (FP64 is slow
// on this GPU): k = mk * 2^ek with mk in [2^52, 2^53); also khi = RN32(k) and
// klo = RN32(k - khi).
// floor(2^116 / m) and the remainder *rem, for m in (2^52, 2^53), without a
// 128-bit division (a long software loop on the GPU): Newton's iteration
// y <- y + y (2^116 - y m) / 2^116 from a seed of the fp32 reciprocal of m's
// top 32 bits (relative error below 2^-22), twice (error below 2^-44, then a
// few units), then exact corrections on the 128-bit remainder.
__device__ __forceinline__ uint64_t div_2p116(uint64_t m, uint64_t* rem) {
  const unsigned __int128 num = (unsigned __int128)1 << 116;
  const uint32_t mh = (uint32_t)(m >> 21);  // [2^31, 2^32)
  const float f = __fmul_rn(__frcp_rn(__uint2float_rn(mh)), 0x1p95f);  // ~ 2^95 / mh <= 2^64
  uint64_t y = (f >= 0x1p64f) ? ~0ull : __float2ull_rz(f);
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const unsigned __int128 p = (unsigned __int128)y * m;
    // e = 2^116 - y m, |e| < 2^95; y += y e / 2^116 with e taken to 2^52
    if (p <= num) {
      const uint64_t eh = (uint64_t)((num - p) >> 52);
      y += (uint64_t)(((unsigned __int128)y * eh) >> 64);
    } else {
      const uint64_t eh = (uint64_t)((p - num) >> 52);
      y -= (uint64_t)(((unsigned __int128)y * eh) >> 64);
    }
  }
  // exact: y m <= 2^116 < (y + 1) m (a few steps at most; bounded)
  unsigned __int128 p = (unsigned __int128)y * m;
  for (int i = 0; i < 64 && p > num; ++i) {
    --y;
    p -= m;
  }
  unsigned __int128 r = num - p;
  for (int i = 0; i < 64 && r >= m; ++i) {
    ++y;
    r -= m;
  }
  *rem = (uint64_t)r;
  return y;
}

struct AllocScale {
  uint64_t mk;
  int ek;
  float khi, klo;
};

__device__ __forceinline__ float pow2f(int e) {  // 2^e for a normal float exponent
  return __int_as_float((e + 127) << 23);
}

__device__ __forceinline__ AllocScale alloc_scale(uint64_t S) {
  // RN64(S) = m * 2^E, m in [2^52, 2^53)
  const int nb = 64 - __clzll((long long)S);
  uint64_t m;
  int E;
  if (nb <= 53) {
    m = S << (53 - nb);
    E = nb - 53;
  } else {
    const int sh = nb - 53;
    m = S >> sh;
    const uint64_t rem = S & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (m & 1ull))) ++m;
    E = sh;
    if (m == (1ull << 53)) {
      m >>= 1;
      ++E;
    }
  }
  // k = RN64(2^(24 - E) / m)
  uint64_t t;
  int ke;
  if (m == (1ull << 52)) {
    t = 1ull << 52;
    ke = 24 - E - 104;
  } else {
    // q = floor(2^116 / m) in (2^63, 2^64); drop 11 bits with round-to-nearest-even
    uint64_t r;
    const uint64_t q = div_2p116(m, &r);
    t = q >> 11;
    const uint32_t d = (uint32_t)(q & 2047u);
    if (d > 1024u || (d == 1024u && (r != 0ull || (t & 1ull)))) ++t;
    ke = 11 - 116 + 24 - E;
    if (t == (1ull << 53)) {
      t >>= 1;
      ++ke;
    }
  }
  AllocScale o;
  o.mk = t;
  o.ek = ke;
  // khi = RN32(k): the top 24 bits of t, rounded to nearest even
  uint64_t hm = t >> 29;
  const uint64_t dr = t & ((1ull << 29) - 1ull);
  if (dr > (1ull << 28) || (dr == (1ull << 28) && (hm & 1ull))) ++hm;
  o.khi = __fmul_rn((float)(uint32_t)hm, pow2f(ke + 29));  // hm <= 2^24: exact
  // klo = RN32(k - khi) = RN32((t - hm 2^29) 2^ke), the difference exact in 64 bits
  const long long diff = (long long)t - (long long)(hm << 29);
  o.klo = __fmul_rn(__ll2float_rn(diff), pow2f(ke));
  return o;
}

// ------------------------------------------------------------ logit loads
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(((uint32_t)h) << 16);
}

__device__ __forceinline__ float load_logit(const void* row, int dtype, int64_t v) {
  if (dtype == DSPARK_F32) return __ldg(reinterpret_cast<const float*>(row) + v);
  return bf16_to_f32(__ldg(reinterpret_cast<const unsigned short*>(row) + v));
}

// Monotone unsigned key of a float (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float y) {
  const uint32_t u = __float_as_uint(y);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ------------------------------------------------------ block reductions
template <typename T, typename Op>
__device__ __forceinline__ T warp_reduce(T v, Op op) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Reduces over the block; every thread gets the result.  `scratch` holds at
// least 32 elements; the call contains two __syncthreads().
template <typename T, typename Op>
__device__ __forceinline__ T block_reduce(T v, Op op, T* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = warp_reduce(v, op);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  T r = scratch[0];
  for (int i = 1; i < nw; ++i) r = op(r, scratch[i]);
  return r;
}

struct OpAddU64 {
  __device__ uint64_t operator()(uint64_t a, uint64_t b) const { return a + b; }
};
struct OpAddU32 {
  __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return a + b; }
};
struct OpOrU32 {
  __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return a | b; }
};
struct OpMaxF {
  __device__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct OpMinU64 {
  __device__ uint64_t operator()(uint64_t a, uint64_t b) const { return a < b ? a : b; }
};
struct OpMaxU64 {
  __device__ uint64_t operator()(uint64_t a, uint64_t b) const { return a > b ? a : b; }
};

// 32-bit sums and ors over a full warp by the hardware warp reduction
__device__ __forceinline__ uint32_t warp_reduce(uint32_t v, OpAddU32) {
  return __reduce_add_sync(0xffffffffu, v);
}
__device__ __forceinline__ uint32_t warp_reduce(uint32_t v, OpOrU32) {
  return __reduce_or_sync(0xffffffffu, v);
}
// 64-bit sums over a full warp by three 32-bit warp reductions of 24-, 24-
// and 16-bit pieces (each sum stays below 2^29): exact for any total below
// 2^64, and measured far faster than shuffling 64-bit values five times.
__device__ __forceinline__ uint64_t warp_reduce(uint64_t v, OpAddU64) {
  const uint32_t a = __reduce_add_sync(0xffffffffu, (uint32_t)v & 0xFFFFFFu);
  const uint32_t b = __reduce_add_sync(0xffffffffu, (uint32_t)(v >> 24) & 0xFFFFFFu);
  const uint32_t c = __reduce_add_sync(0xffffffffu, (uint32_t)(v >> 48));
  return (uint64_t)a + ((uint64_t)b << 24) + ((uint64_t)c << 48);
}

// Inclusive scan over the block for one uint32 per thread; returns the
// inclusive prefix, *total gets the block total.  scratch >= 32 words.
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* scratch,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  uint32_t before = 0, all = 0;
  for (int i = 0; i < nw; ++i) {
    const uint32_t s = scratch[i];
    if (i < warp) before += s;
    all += s;
  }
  *total = all;
  return v + before;
}

// Inclusive scan over the block for one uint64 per thread; *total gets the
// block total.  scratch >= 32 elements.
__device__ __forceinline__ uint64_t block_inclusive_scan_u64(uint64_t v, uint64_t* scratch,
                                                             uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  uint64_t before = 0, all = 0;
  for (int i = 0; i < nw; ++i) {
    const uint64_t s = scratch[i];
    if (i < warp) before += s;
    all += s;
  }
  *total = all;
  return v + before;
}

// -------------------------------------------------- TMA bulk copy, mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_bulk(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (src 16-byte aligned, bytes a
// multiple of 16); nothing waits for it.
__device__ __forceinline__ void l2_prefetch_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One try_wait with a suspend-time hint: the thread may sleep in hardware
// (up to the hint) until the phase completes instead of spinning.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase), "r"(1000000u)
      : "memory");
  return ok != 0u;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `phase` of `bar` for at most kWaitLimitNs; false on timeout.
// Between polls the thread sleeps with an exponential backoff (64 ns .. 1 us),
// so a waiting warp takes almost no issue slots from the rest of the SM.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t phase) {
  if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = global_ns();
  uint32_t nap = 64;
  while (global_ns() - t0 < kWaitLimitNs) {
    __nanosleep(nap);
    if (mbar_try_wait(bar, phase)) return true;
    nap = nap < 1024u ? 2u * nap : 1024u;
  }
  return false;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Waits (at most kWaitLimitNs) until *flag >= target, another CTA's release
// seen through an acquire load; false on timeout.
static __device__ __noinline__ bool wait_count(const uint32_t* flag, uint32_t target) {
  if (ld_acquire(flag) >= target) return true;
  const uint64_t t0 = global_ns();
  uint32_t nap = 64;
  while (global_ns() - t0 < kWaitLimitNs) {
    __nanosleep(nap);
    if (ld_acquire(flag) >= target) return true;
    nap = nap < 1024u ? 2u * nap : 1024u;
  }
  return false;
}

// Float holding an integer in [0, 2^23) to int, by the 2^23 offset trick.
__device__ __forceinline__ int small_float_to_int(float v) {
  return __float_as_int(__fadd_rn(v, 8388608.0f)) - 0x4B000000;
}

}  // namespace dspark
