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
constexpr int kSupBuckets = 256;             // id buckets of the output ordering
// bytes of scratch: the entries' records and weights, the select's histogram
// and gathered values, four arrays over the id buckets, the entries in
// bucket order
constexpr int kSupScratch = 16 * kSupCap + 4 * kSupCap + 4 * 256 + 8 * 32 +
                            4 * 4 * kSupBuckets + 4 * kSupCap;

struct SupShared {
  double kd;  // RN64(2^24 / RN64(S))
  uint64_t red64[32];
  uint32_t red32[32];
  int found;
  uint64_t sel_v;  // the select's result and counts
  uint32_t sel_digit, sel_above, sel_equal, n_list;
};

// Block-wide radix select over 64-bit values: the r-th largest
// (1 <= r <= the number of taken entries) of val(i) over i < n with take(i);
// *above gets the number of taken values above it, *equal the number equal.
// The digit passes (8 bits) start at the byte holding the highest bit where
// the taken values' min and max differ; once the selected bin holds at most
// 32 values they are gathered and one warp finishes.  hist: 256 words and
// list: 32 values of shared memory.  Every thread calls it; it starts with a
// __syncthreads() and its result is uniform.
template <typename Val, typename Take>
__device__ uint64_t sup_select_desc(int n, uint32_t r, Val val, Take take, uint32_t* hist,
                                    uint64_t* list, SupShared& sh, uint32_t* above,
                                    uint32_t* equal) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kW = kSupThr / 32;
  __syncthreads();
  uint64_t vmin = ~0ull, vmax = 0ull;
  uint32_t cnt = 0u;
  for (int i = (int)threadIdx.x; i < n; i += kSupThr)
    if (take(i)) {
      const uint64_t v = val(i);
      vmin = min(vmin, v);
      vmax = max(vmax, v);
      ++cnt;
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    vmin = min(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
    vmax = max(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
  }
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  if (lane == 0) {
    sh.red64[warp] = vmin;
    sh.red64[kW + warp] = vmax;
    sh.red32[warp] = cnt;
  }
  __syncthreads();
  vmin = ~0ull;
  vmax = 0ull;
  cnt = 0u;
  for (int w = 0; w < kW; ++w) {
    vmin = min(vmin, sh.red64[w]);
    vmax = max(vmax, sh.red64[kW + w]);
    cnt += sh.red32[w];
  }
  if (vmin >= vmax) {  // every taken value is the same
    *above = 0u;
    *equal = cnt;
    return vmin;
  }
  int shift = (63 - __clzll((long long)(vmin ^ vmax))) & ~7;
  uint64_t mask = (shift == 56) ? 0ull : ~((1ull << (shift + 8)) - 1ull);
  uint64_t prefix = vmin & mask;
  uint32_t above_acc = 0, eq = cnt;
  for (; shift >= 0; shift -= 8) {
    __syncthreads();
    hist[threadIdx.x] = 0u;  // kSupThr == 256 bins
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kSupThr) {
      const int i = i0 + (int)threadIdx.x;
      uint32_t bin = 0xFFFFFFFFu;
      if (i < n && take(i)) {
        const uint64_t v = val(i);
        if ((v & mask) == prefix) bin = (uint32_t)(v >> shift) & 255u;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (bin != 0xFFFFFFFFu && lane == __ffs(peers) - 1)
        atomicAdd(&hist[bin], (uint32_t)__popc(peers));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l scans bins 255 - 8l down to 248 - 8l
      uint32_t c[8], sacc = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        sacc += c[j];
      }
      uint32_t incl = sacc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const uint32_t excl = incl - sacc;
      if (excl < r && r <= incl) {
        uint32_t acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc < r && r <= acc + c[j]) {
            sh.sel_digit = (uint32_t)(255 - 8 * lane - j);
            sh.sel_above = acc;
            sh.sel_equal = c[j];
          }
          acc += c[j];
        }
      }
    }
    __syncthreads();
    const uint32_t d = sh.sel_digit, ab = sh.sel_above;
    eq = sh.sel_equal;
    r -= ab;
    above_acc += ab;
    prefix |= (uint64_t)d << shift;
    mask |= 255ull << shift;
    if (shift > 0 && eq <= 32u) {
      // the selected bin's values, gathered; warp 0 takes the r-th largest
      if (threadIdx.x == 0) sh.n_list = 0u;
      __syncthreads();
      for (int i = (int)threadIdx.x; i < n; i += kSupThr)
        if (take(i)) {
          const uint64_t v = val(i);
          if ((v & mask) == prefix) {
            const uint32_t j = atomicAdd(&sh.n_list, 1u);
            if (DSPARK_CHECK(j < 32u)) list[j] = v;
          }
        }
      __syncthreads();
      if (warp == 0) {
        const uint64_t v = (lane < (int)eq) ? list[lane] : 0ull;
        uint32_t gt = 0, ge = 0;
        for (int m = 0; m < (int)eq; ++m) {
          const uint64_t u = __shfl_sync(0xffffffffu, v, m);
          gt += (u > v) ? 1u : 0u;
          ge += (u >= v) ? 1u : 0u;
        }
        const bool hit = lane < (int)eq && gt < r && r <= ge;
        const unsigned msk = __ballot_sync(0xffffffffu, hit);
        if (msk != 0u && lane == __ffs(msk) - 1) {
          sh.sel_v = v;
          sh.sel_above = gt;
          sh.sel_equal = ge - gt;
        }
      }
      __syncthreads();
      *above = above_acc + sh.sel_above;
      *equal = sh.sel_equal;
      return sh.sel_v;
    }
  }
  *above = above_acc;
  *equal = eq;
  return prefix;
}

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
  uint32_t* hist = reinterpret_cast<uint32_t*>(scratch + 20 * kSupCap);
  uint64_t* list = reinterpret_cast<uint64_t*>(hist + 256);
  uint32_t* bcount = reinterpret_cast<uint32_t*>(list + 32);  // [kSupBuckets] each
  uint32_t* bstart = bcount + kSupBuckets;
  uint32_t* bcur = bstart + kSupBuckets;
  uint32_t* bmass = bcur + kSupBuckets;
  uint32_t* border = bmass + kSupBuckets;  // [kSupCap]
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
        // the R largest remainders, lowest id first among equal ones: T is
        // the R-th largest remainder (a radix select over the remainders'
        // bit patterns, which order like the values); every remainder above
        // T is granted, and of those equal to T the R - above lowest ids
        auto rkey = [&](int i) -> uint64_t {
          const uint4 e = ent[i];
          return ((uint64_t)e.y << 32) | e.x;
        };
        uint64_t T = ~0ull;
        int32_t id_cut = 0x7FFFFFFF;
        if (R > 0) {
          uint32_t ab, eqc;
          T = sup_select_desc(
              ns, (uint32_t)R, rkey, [&](int i) { return rkey(i) != 0ull; }, hist, list, sh,
              &ab, &eqc);
          const uint32_t need = (uint32_t)R - ab;
          if (need < eqc) {
            uint32_t ab2, eq2;
            const uint64_t nid = sup_select_desc(
                ns, need, [&](int i) -> uint64_t { return (uint64_t)(~ent[i].z); },
                [&](int i) { return rkey(i) == T; }, hist, list, sh, &ab2, &eq2);
            id_cut = (int32_t)~(uint32_t)nid;
          }
        }
        __syncthreads();  // every record is read before the counts change
        uint64_t csum = 0;
        for (int i = tid; i < ns; i += kSupThr) {
          const uint64_t ri = rkey(i);
          const bool g = R > 0 && ri != 0ull &&
                         (ri > T || (ri == T && (int32_t)ent[i].z <= id_cut));
          const uint32_t c = ent[i].w + (g ? 1u : 0u);
          ent[i].w = c;
          csum += c;
        }
        csum = block_reduce(csum, OpAddU64(), sh.red64);
        if (csum != (uint64_t)DSPARK_M) st = DSPARK_ST_ALLOC_INCONSISTENT;
      }
    }
  }

  // ---- outputs: nonzero counts in ascending id order, the draw.  The
  // nonzero entries go to kSupBuckets buckets of the id range [lo, hi]
  // (bucket (id - lo) * kSupBuckets / (hi - lo + 1): ascending ids, ascending
  // buckets); a bucket's place and the count mass before it come from scans
  // over the buckets, an entry's place inside its bucket from the bucket's
  // few other entries.
  uint32_t nnz = 0;
  if (st == DSPARK_ST_OK) {
    int32_t ilo = 0x7FFFFFFF, ihi = -1;
    for (int i = tid; i < ns; i += kSupThr)
      if (ent[i].w != 0u) {
        ilo = min(ilo, (int32_t)ent[i].z);
        ihi = max(ihi, (int32_t)ent[i].z);
      }
    ilo = __reduce_min_sync(0xffffffffu, ilo);
    ihi = __reduce_max_sync(0xffffffffu, ihi);
    const int lane = tid & 31, warp = tid >> 5;
    __syncthreads();
    if (lane == 0) {
      sh.red32[warp] = (uint32_t)ilo;
      sh.red32[16 + warp] = (uint32_t)ihi;
    }
    for (int bk = tid; bk < kSupBuckets; bk += kSupThr) {
      bcount[bk] = 0u;
      bmass[bk] = 0u;
    }
    __syncthreads();
    ilo = 0x7FFFFFFF;
    ihi = -1;
    for (int w = 0; w < kSupThr / 32; ++w) {
      ilo = min(ilo, (int32_t)sh.red32[w]);
      ihi = max(ihi, (int32_t)sh.red32[16 + w]);
    }
    const uint64_t span = (ihi >= ilo) ? (uint64_t)(ihi - ilo) + 1u : 1u;
    auto bucket = [&](int32_t id) -> int {
      return (int)(((uint64_t)(id - ilo) * (uint64_t)kSupBuckets) / span);
    };
    for (int i = tid; i < ns; i += kSupThr) {
      const uint32_t c = ent[i].w;
      if (c == 0u) continue;
      const int bk = bucket((int32_t)ent[i].z);
      if (!DSPARK_CHECK(bk >= 0 && bk < kSupBuckets)) continue;
      atomicAdd(&bcount[bk], 1u);
      atomicAdd(&bmass[bk], c);
    }
    __syncthreads();
    if (warp == 0) {
      // exclusive scans of the bucket sizes and masses (lane l: buckets 8l .. 8l+7)
      constexpr int kPer = kSupBuckets / 32;
      uint32_t cs[kPer], ms[kPer], ct = 0, mt = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        cs[j] = bcount[kPer * lane + j];
        ms[j] = bmass[kPer * lane + j];
        ct += cs[j];
        mt += ms[j];
      }
      uint32_t ci = ct, mi = mt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t tc = __shfl_up_sync(0xffffffffu, ci, o);
        const uint32_t tm = __shfl_up_sync(0xffffffffu, mi, o);
        if (lane >= o) {
          ci += tc;
          mi += tm;
        }
      }
      uint32_t c0 = ci - ct, m0 = mi - mt;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        bstart[kPer * lane + j] = c0;
        bcur[kPer * lane + j] = c0;
        bmass[kPer * lane + j] = m0;  // now the mass before the bucket
        c0 += cs[j];
        m0 += ms[j];
      }
    }
    __syncthreads();
    for (int i = tid; i < ns; i += kSupThr) {
      if (ent[i].w == 0u) continue;
      const int bk = bucket((int32_t)ent[i].z);
      if (!DSPARK_CHECK(bk >= 0 && bk < kSupBuckets)) continue;
      const uint32_t j = atomicAdd(&bcur[bk], 1u);
      if (DSPARK_CHECK(j < (uint32_t)kSupCap)) border[j] = (uint32_t)i;
    }
    __syncthreads();
    for (int i = tid; i < ns; i += kSupThr) {
      const uint32_t c = ent[i].w;
      if (c == 0u) continue;
      const int32_t idi = (int32_t)ent[i].z;
      const int bk = bucket(idi);
      if (!DSPARK_CHECK(bk >= 0 && bk < kSupBuckets)) continue;
      nnz += 1u;
      uint32_t pos = bstart[bk], before = bmass[bk];
      const uint32_t e1 = bcur[bk];  // the bucket's end
      for (uint32_t j = bstart[bk]; j < e1; ++j) {
        if (!DSPARK_CHECK(j < (uint32_t)kSupCap && border[j] < (uint32_t)ns)) break;
        const uint4 o = ent[border[j]];
        if ((int32_t)o.z < idi) {
          pos += 1u;
          before += o.w;
        }
      }
      if (DSPARK_CHECK(pos < (uint32_t)k)) {
        ids_out[pos] = idi;
        cnt_out[pos] = c;
      }
      if (before <= D && D - before < c) sh.found = idi;
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
