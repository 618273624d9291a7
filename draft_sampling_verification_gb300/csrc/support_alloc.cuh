// support_alloc.cuh -- the 2^24-ticket allocation on a small support and the
// sparse outputs ("PP1 q transport and scheduling design", Distribution
// contract and precision: for a sparse q the weights are normalised on the
// support and the tickets are allocated there; Sparse support: the support
// ids travel in ascending order).  Shared by the top-k q kernel and the
// vocabulary-sharded top-k merge.
//
// On at most DSPARK_MAX_TOPK entries the allocation runs in FP64 as the
// method states it: E = floor(exp_ds(y - m) * 2^40), S = sum E,
// a = RN64(E * RN64(2^24 / RN64(S))), f = floor a, r = a - f, and the
// R = M - sum f largest r (lowest id first) get one more ticket.  The nonzero
// counts are written in ascending id order; the draft draw takes the first id
// whose inclusive cumulative count exceeds the 24-bit draw.
#pragma once
#include "common.cuh"

namespace dspark {
namespace {

constexpr int kSupThr = 256;                 // threads of the calling block
constexpr int kSupCap = DSPARK_MAX_TOPK;     // largest support
constexpr int kSupScratch = 16 * kSupCap + 4 * kSupCap;  // bytes of scratch

struct SupShared {
  double kd;  // RN64(2^24 / RN64(S))
  uint64_t red64[32];
  uint32_t red32[32];
  int found;
};

struct OpMaxU32Sup {
  __device__ uint32_t operator()(uint32_t a, uint32_t b) const { return a > b ? a : b; }
};

__device__ __forceinline__ float sup_key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Allocation on the support keys[i] (float_key of a finite y; -0 taken as +0)
// with ids[i], i < ns <= kSupCap, then the outputs of one row: counts and ids
// [k] (nonzero counts in ascending id order, then id -1 / count 0), *nnz_out,
// *status_out, and the token (if token_out) of the 24-bit draw D.  `st` is
// the row's status so far (anything but OK writes an empty row).  scratch:
// kSupScratch bytes of shared memory, 16-byte aligned.  Every thread of the
// block calls it.
__device__ void support_alloc_emit(int st, int ns, int k, const uint32_t* keys,
                                   const int32_t* ids, unsigned char* scratch, SupShared& sh,
                                   uint32_t* cnt_out, int32_t* ids_out, int32_t* nnz_out,
                                   int32_t* status_out, int32_t* token_out, uint32_t D) {
  const int tid = threadIdx.x;
  // one 16-byte record per entry {r low, r high, id, count}: r in [0, 1) as
  // its bit pattern (the same order as the values, compared in integer
  // arithmetic: FP64 compares are slow here)
  uint4* ent = reinterpret_cast<uint4*>(scratch);
  float* e_arr = reinterpret_cast<float*>(scratch + 16 * kSupCap);
  if (tid == 0) sh.found = -1;
  if (st == DSPARK_ST_OK) {
    uint32_t mk = 0u;
    for (int i = tid; i < ns; i += kSupThr) mk = max(mk, keys[i]);
    mk = block_reduce(mk, OpMaxU32Sup(), sh.red32);
    const float m = sup_key_float(mk);
    uint64_t S = 0;
    for (int i = tid; i < ns; i += kSupThr) {
      const float e = weight40(__fsub_rn(sup_key_float(keys[i]), m));
      e_arr[i] = e;
      S += (uint64_t)__float2ull_rz(e);
    }
    S = block_reduce(S, OpAddU64(), sh.red64);
    // one FP64 division for the block (FP64 is slow here)
    if (tid == 0) sh.kd = __ddiv_rn(16777216.0, __ull2double_rn(S));
    __syncthreads();
    const double kd = sh.kd;
    uint64_t F = 0;
    uint32_t npos = 0;
    for (int i = tid; i < ns; i += kSupThr) {
      const double a = __dmul_rn((double)e_arr[i], kd);
      const double f = floor(a);
      const uint64_t rb = (uint64_t)__double_as_longlong(__dsub_rn(a, f));
      ent[i] = make_uint4((uint32_t)rb, (uint32_t)(rb >> 32), (uint32_t)ids[i], (uint32_t)f);
      F += (uint64_t)f;
      npos += (rb != 0u) ? 1u : 0u;
    }
    F = block_reduce(F, OpAddU64(), sh.red64);
    npos = block_reduce(npos, OpAddU32(), sh.red32);
    if (F > (uint64_t)DSPARK_M) {
      st = DSPARK_ST_ALLOC_INCONSISTENT;
    } else {
      const uint64_t R = (uint64_t)DSPARK_M - F;
      if (R >= (uint64_t)DSPARK_M || R > (uint64_t)npos) {
        st = DSPARK_ST_ALLOC_INCONSISTENT;
      } else {
        // the R largest remainders (lowest id first among equal ones):
        // rank = the entries that come before this one
        uint32_t grant[kSupCap / kSupThr];
#pragma unroll
        for (int q = 0; q < kSupCap / kSupThr; ++q) {
          const int i = tid + q * kSupThr;
          grant[q] = 0u;
          if (i < ns) {
            const uint4 ei = ent[i];
            const uint64_t ri = ((uint64_t)ei.y << 32) | ei.x;
            uint32_t rank = 0;
#pragma unroll 8
            for (int j = 0; j < ns; ++j) {
              const uint4 ej = ent[j];
              const uint64_t rj = ((uint64_t)ej.y << 32) | ej.x;
              rank += (uint32_t)(rj > ri) | ((uint32_t)(rj == ri) & (uint32_t)(ej.z < ei.z));
            }
            grant[q] = ((uint64_t)rank < R) ? 1u : 0u;
          }
        }
        __syncthreads();  // every rank is taken before the counts change
        uint64_t csum = 0;
#pragma unroll
        for (int q = 0; q < kSupCap / kSupThr; ++q) {
          const int i = tid + q * kSupThr;
          if (i < ns) {
            const uint32_t c = ent[i].w + grant[q];
            ent[i].w = c;
            csum += c;
          }
        }
        csum = block_reduce(csum, OpAddU64(), sh.red64);
        if (csum != (uint64_t)DSPARK_M) st = DSPARK_ST_ALLOC_INCONSISTENT;
      }
    }
  }

  // ---- outputs: nonzero counts in ascending id order, the draw
  uint32_t nnz = 0;
  if (st == DSPARK_ST_OK) {
    const uint2* ic = reinterpret_cast<const uint2*>(ent);  // {id, count} at odd halves
    for (int i = tid; i < ns; i += kSupThr) {
      const uint2 mine = ic[2 * i + 1];
      const uint32_t c = mine.y, idi = mine.x;
      if (c == 0u) continue;
      nnz += 1u;
      uint32_t pos = 0, before = 0;
#pragma unroll 8
      for (int j = 0; j < ns; ++j) {
        const uint2 o = ic[2 * j + 1];
        const uint32_t pre = (uint32_t)(o.y > 0u) & (uint32_t)(o.x < idi);
        pos += pre;
        before += pre ? o.y : 0u;
      }
      if (DSPARK_CHECK(pos < (uint32_t)k)) {
        ids_out[pos] = (int32_t)idi;
        cnt_out[pos] = c;
      }
      if (before <= D && D - before < c) sh.found = (int32_t)idi;
    }
    nnz = block_reduce(nnz, OpAddU32(), sh.red32);
  }
  for (int i = (int)nnz + tid; i < k; i += kSupThr) {
    ids_out[i] = -1;
    cnt_out[i] = 0u;
  }
  __syncthreads();
  if (tid == 0) {
    *nnz_out = (int32_t)nnz;
    *status_out = st;
    if (token_out) *token_out = (st == DSPARK_ST_OK) ? sh.found : -1;
  }
}

}  // namespace
}  // namespace dspark
