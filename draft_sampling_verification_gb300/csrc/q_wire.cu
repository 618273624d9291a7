// q_wire.cu -- the wire form of a q row and its validation on receipt
// ("PP1 q transport and scheduling design", Distribution contract and
// precision: q travels as little-endian FP32 values q = c / M, each exact;
// the receiver recovers c by multiplying by M, requires an integer and checks
// the mass in uint64.  Versioned v2 message design: the reply carries the q
// values, the sparse ids and a checksum; the receiver refuses non-finite,
// negative or non-dyadic values, a wrong mass, duplicate, unsorted,
// out-of-range or padded ids, and a zero q at the proposed token).
//
// Payload words: a dense row is its V FP32 bit patterns in id order; a
// sparse row is its nnz int32 ids, then their nnz FP32 bit patterns.  The
// byte checksum is Fletcher-64 of those words: A = sum w_i and
// B = sum (n - i) w_i, both modulo 2^32 - 1, checksum = B << 32 | A.  Both
// sums split over threads, so one CTA streams a row once with every thread
// independent until a single block reduction.
//
// One CTA of 256 threads per row.  Dense rows whose start is 16-byte aligned
// move 4 elements per 128-bit access; other rows one element per access.
#define DSPARK_TU 5  // this file's number in the checked build's site codes
#include "common.cuh"

namespace dspark {
namespace {

constexpr int kWThr = 256;
constexpr uint64_t kFlMod = 0xFFFFFFFFull;  // 2^32 - 1

// x modulo 2^32 - 1, for any 64-bit x
__device__ __forceinline__ uint64_t fold_mod(uint64_t x) {
  x = (x & kFlMod) + (x >> 32);  // < 2^33
  x = (x & kFlMod) + (x >> 32);  // <= 2^32
  return x >= kFlMod ? x - kFlMod : x;
}

// Per-thread Fletcher partials: word i of an n-word payload adds w to A and
// (n - i) * w to B.  (n - i) <= 2^18 and w < 2^32, so B grows by < 2^50 per
// word; it is folded every 256 words.
struct Fl {
  uint64_t a = 0, b = 0;
  int since = 0;
  __device__ __forceinline__ void add(uint32_t w, int64_t i, int64_t n) {
    a += w;
    b += (uint64_t)(n - i) * w;
    if (++since == 256) {
      a = fold_mod(a);
      b = fold_mod(b);
      since = 0;
    }
  }
};

struct WShared {
  uint64_t r64[32];
  uint64_t r64b[32];
  uint32_t r32[32];
};

// Block-wide A and B (each < 2^32 - 1 after the fold), in every thread.
__device__ __forceinline__ uint64_t fletcher_block(Fl fl, WShared& sh) {
  uint64_t a = fold_mod(fl.a), b = fold_mod(fl.b);  // < 2^32 each
  a = block_reduce(a, OpAddU64(), sh.r64);           // < 2^40
  b = block_reduce(b, OpAddU64(), sh.r64b);
  return (fold_mod(b) << 32) | fold_mod(a);
}

struct PackParams {
  const uint32_t* counts;
  const int32_t* ids;
  const int32_t* nnz;
  int top_k;
  int V;
  float* q;
  uint64_t* checksum;
};

__global__ void __launch_bounds__(kWThr) q_pack_kernel(PackParams p) {
  __shared__ WShared sh;
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const bool sparse = p.top_k > 0;
  const int width = sparse ? p.top_k : p.V;
  const uint32_t* c = p.counts + (int64_t)row * width;
  float* q = p.q + (int64_t)row * width;
  Fl fl;
  if (!sparse) {
    const int64_t n = p.V;
    const bool vec =
        ((reinterpret_cast<uintptr_t>(c) | reinterpret_cast<uintptr_t>(q)) & 15u) == 0;
    if (vec) {
      const int ng = p.V >> 2;
      const uint4* c4 = reinterpret_cast<const uint4*>(c);
      float4* q4 = reinterpret_cast<float4*>(q);
#pragma unroll 4
      for (int g = tid; g < ng; g += kWThr) {
        const uint4 cc = __ldcs(c4 + g);
        const float4 qq = make_float4(__uint2float_rn(cc.x) * 0x1p-24f,
                                      __uint2float_rn(cc.y) * 0x1p-24f,
                                      __uint2float_rn(cc.z) * 0x1p-24f,
                                      __uint2float_rn(cc.w) * 0x1p-24f);
        __stcs(q4 + g, qq);
        const int64_t i = 4 * (int64_t)g;
        fl.add(__float_as_uint(qq.x), i, n);
        fl.add(__float_as_uint(qq.y), i + 1, n);
        fl.add(__float_as_uint(qq.z), i + 2, n);
        fl.add(__float_as_uint(qq.w), i + 3, n);
      }
      for (int v = 4 * ng + tid; v < p.V; v += kWThr) {
        const float qv = __uint2float_rn(c[v]) * 0x1p-24f;
        q[v] = qv;
        fl.add(__float_as_uint(qv), v, n);
      }
    } else {
#pragma unroll 4
      for (int v = tid; v < p.V; v += kWThr) {
        const float qv = __uint2float_rn(__ldcs(c + v)) * 0x1p-24f;
        __stcs(q + v, qv);
        fl.add(__float_as_uint(qv), v, n);
      }
    }
  } else {
    const int32_t* id = p.ids + (int64_t)row * width;
    const int nz = max(0, min(p.nnz[row], width));
    const int64_t n = 2 * (int64_t)nz;
    for (int i = tid; i < width; i += kWThr) {
      const float qv = (i < nz) ? __uint2float_rn(c[i]) * 0x1p-24f : 0.0f;
      q[i] = qv;
      if (i < nz) {
        fl.add((uint32_t)id[i], i, n);
        fl.add(__float_as_uint(qv), nz + i, n);
      }
    }
  }
  const uint64_t cs = fletcher_block(fl, sh);
  if (tid == 0) p.checksum[row] = cs;
}

struct ValParams {
  const float* q;
  const int32_t* ids;
  const int32_t* nnz;
  int top_k;
  int V;
  const int32_t* tokens;   // [rows] or null
  const uint64_t* expect;  // [rows] or null
  uint32_t* counts;        // [rows][width] or null
  int32_t* status;
};

// Count of one received value: q * 2^24 when q is finite, not negative,
// dyadic and at most 1; else flags the row.
__device__ __forceinline__ uint32_t recover(float v, uint32_t& bad) {
  const float cm = v * 0x1p24f;  // exact: a power-of-two scale of a value <= 1
  const bool ok = (v >= 0.0f) && (v <= 1.0f) && (cm == truncf(cm));  // NaN fails v >= 0
  bad |= ok ? 0u : 1u;
  return ok ? (uint32_t)cm : 0u;
}

__global__ void __launch_bounds__(kWThr) q_validate_kernel(ValParams p) {
  __shared__ WShared sh;
  __shared__ int found;
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const bool sparse = p.top_k > 0;
  const int width = sparse ? p.top_k : p.V;
  const float* q = p.q + (int64_t)row * width;
  uint32_t* cout = p.counts ? p.counts + (int64_t)row * width : nullptr;
  const int token = p.tokens ? p.tokens[row] : -1;
  if (tid == 0) found = 0;
  __syncthreads();
  Fl fl;
  uint64_t mass = 0;
  uint32_t bad = 0;
  bool size_bad = false;  // a sparse entry count outside [1, top_k]
  int nz = 0;
  if (!sparse) {
    const int64_t n = p.V;
    const bool vec = ((reinterpret_cast<uintptr_t>(q) |
                       (cout ? reinterpret_cast<uintptr_t>(cout) : 0)) & 15u) == 0;
    int done = 0;
    if (vec) {
      const int ng = p.V >> 2;
      const float4* q4 = reinterpret_cast<const float4*>(q);
#pragma unroll 4
      for (int g = tid; g < ng; g += kWThr) {
        const float4 qq = __ldcs(q4 + g);
        const uint4 cc = make_uint4(recover(qq.x, bad), recover(qq.y, bad),
                                    recover(qq.z, bad), recover(qq.w, bad));
        if (cout) __stcs(reinterpret_cast<uint4*>(cout) + g, cc);
        mass += (uint64_t)cc.x + cc.y + cc.z + cc.w;
        const int i = 4 * g;
        if (token >= i && token < i + 4) {
          const uint32_t ct = token == i       ? cc.x
                              : token == i + 1 ? cc.y
                              : token == i + 2 ? cc.z
                                               : cc.w;
          if (ct > 0u) found = 1;
        }
        fl.add(__float_as_uint(qq.x), i, n);
        fl.add(__float_as_uint(qq.y), i + 1, n);
        fl.add(__float_as_uint(qq.z), i + 2, n);
        fl.add(__float_as_uint(qq.w), i + 3, n);
      }
      done = 4 * ng;
    }
    for (int v = done + tid; v < p.V; v += kWThr) {
      const float qv = q[v];
      const uint32_t cv = recover(qv, bad);
      if (cout) cout[v] = cv;
      mass += cv;
      if (v == token && cv > 0u) found = 1;
      fl.add(__float_as_uint(qv), v, n);
    }
  } else {
    const int32_t* id = p.ids + (int64_t)row * width;
    nz = p.nnz[row];
    if (nz < 1 || nz > width) {
      size_bad = true;
      nz = 0;
    }
    const int64_t n = 2 * (int64_t)nz;
    for (int i = tid; i < width; i += kWThr) {
      uint32_t cv = 0;
      if (i < nz) {
        const float qv = q[i];
        const int32_t v = id[i];
        cv = recover(qv, bad);
        // canonical support: ascending ids in [0, V), no zero entry
        if (v < 0 || v >= p.V || cv == 0u || (i > 0 && id[i - 1] >= v)) bad |= 1u;
        if (v == token && cv > 0u) found = 1;
        mass += cv;
        fl.add((uint32_t)v, i, n);
        fl.add(__float_as_uint(qv), nz + i, n);
      }
      if (cout) cout[i] = cv;
    }
  }
  const uint64_t cs = fletcher_block(fl, sh);
  mass = block_reduce(mass, OpAddU64(), sh.r64);
  bad = block_reduce(bad, OpOrU32(), sh.r32);
  // the payload's size, then its checksum, then its values, then the token
  int st = DSPARK_ST_OK;
  if (size_bad) st = DSPARK_ST_BAD_Q;
  else if (p.expect && cs != p.expect[row]) st = DSPARK_ST_BAD_CHECKSUM;
  else if (bad || mass != (uint64_t)DSPARK_M) st = DSPARK_ST_BAD_Q;
  else if (p.tokens && (token < 0 || token >= p.V || !found)) st = DSPARK_ST_BAD_DRAFT;
  if (st != DSPARK_ST_OK && cout)
    for (int i = tid; i < width; i += kWThr) cout[i] = 0u;
  if (tid == 0) p.status[row] = st;
}

}  // namespace

cudaError_t launch_q_pack(const uint32_t* counts, const int32_t* ids, const int32_t* nnz,
                          int top_k, int n_rows, int V, float* q, uint64_t* checksum,
                          cudaStream_t stream) {
  PackParams p{counts, ids, nnz, top_k, V, q, checksum};
  q_pack_kernel<<<n_rows, kWThr, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_q_validate(const float* q, const int32_t* ids, const int32_t* nnz, int top_k,
                              int n_rows, int V, const int32_t* tokens, const uint64_t* expect,
                              uint32_t* counts, int32_t* status, cudaStream_t stream) {
  ValParams p{q, ids, nnz, top_k, V, tokens, expect, counts, status};
  q_validate_kernel<<<n_rows, kWThr, 0, stream>>>(p);
  return cudaGetLastError();
}

DSPARK_CHECK_COLLECTOR(q_wire)

}  // namespace dspark
