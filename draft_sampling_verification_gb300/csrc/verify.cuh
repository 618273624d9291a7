// verify.cuh -- device code of verification (see verify.cu), shared by the
// verify kernels and the fused speculative-step kernel.
#pragma once
#include "common.cuh"

namespace dspark {
namespace vfy {
namespace {  // device code private to each translation unit that includes it

constexpr int kVCluster = 8;
constexpr int kVThreads = 256;
constexpr uint64_t kNearTol = 70368745ull;   // ceil(1e-6 * 2^46)

enum VerifyMode { kGreedy = 0, kRatio = 1 };

struct VParams {
  const void* z;
  int dtype;
  int64_t ld;
  int B;
  int depth;
  int V;
  const int32_t* drafts;
  const uint32_t* counts;
  const int32_t* ids;
  const int32_t* nnz;
  int top_k;
  uint64_t seed;
  const uint32_t* request_ids;
  // greedy outputs (null when the mode is not run)
  int32_t* g_accept_len;
  int32_t* g_committed;
  int32_t* g_status;
  // ratio outputs (null when the mode is not run)
  int32_t* r_accept_len;
  int32_t* r_committed;
  uint32_t* r_flags;
  int32_t* r_status;
  int chunk;
};

constexpr int kVTma = 4;
constexpr int kVMaxBlocks = 160;  // blocks of 32 groups per slice (fp32: <= 129)

struct __align__(16) VX {
  float m;        // max of the slice (NaN-propagating)
  float s;        // sum of exp(z - m) over the slice (ratio mode)
  float amv;      // argmax value (greedy mode)
  int ami;        // argmax id, lowest among the maxima
  uint64_t z;     // fixed-point draw mass of the slice
  uint64_t cs;    // q mass of the slice (dense residual rows)
  uint32_t fl;    // bit0: a bulk copy timed out
  uint32_t pad[3];
};

constexpr int kVMaxNC = 8;  // the largest verify cluster

struct VSh2 {
  VX x[2];
  // every CTA's partials, pushed here by each CTA before the cluster barrier
  // ([buffer][writer's rank]), so that after it the merge reads local memory
  VX px[2][kVMaxNC];
  union {
    uint64_t bsum[kVMaxBlocks];  // final draw: the mass of each block of 32 groups
    // then, in the drawing CTA's token search once its block is found: a
    // sparse q row's counts over that block's ids
    uint32_t qblk[32 * 8];
  };
  float wm[8], ws[8];
  int wai[8];
  uint64_t wz[8], wc[8];
  float M, S, AMV;
  int AMI;
  uint32_t FL;
  uint64_t Z, before, CS;
  int q_ok;
  uint32_t q_c;
  int timeout;
  int found;
  uint32_t near;
  int m_pick;       // match mode: the row's drawn token, pushed by the CTA that drew it
  int m_st;
  uint32_t m_flags;
  int dec;          // ratio decision of the row: 1 accept, 0 reject, -1 refuse (status in dst)
  int dst;
  uint32_t dflags;
};

// A load of q (counts, sparse ids): through the read-only data path when q
// was written before the launch, a plain (coherent) load when the same launch
// wrote it (the one-launch step, whose q rows are finished by other clusters
// and published with release / acquire on the per-request row counter).
template <bool kCoh, typename T>
__device__ __forceinline__ T ldq(const T* p) {
  if (kCoh) return *p;
  return __ldg(p);
}

// The final draw's fixed-point weight floor(r * 2^46), r in [0, 1], as
// hi * 2^23 + lo with hi = floor(r 2^23) and lo = floor((r 2^23 - hi) 2^23),
// read from the bits of round-down sums with 2^23 (each exact: the sums lie
// in [2^23, 2^24], where floats are the integers): no float-to-integer
// conversion, and the sums of a block fit 32-bit integers.
struct Fix46 {
  uint32_t hi, lo;
};
__device__ __forceinline__ Fix46 fix46(float r) {
  const float a = __fmul_rn(r, 8388608.0f);                     // r * 2^23, exact
  const float t1 = __fadd_rd(a, 8388608.0f);                    // 2^23 + floor(a)
  const float f = __fsub_rn(a, __fsub_rn(t1, 8388608.0f));      // a - floor(a), exact
  const float t2 = __fmaf_rd(f, 8388608.0f, 8388608.0f);        // 2^23 + floor(f 2^23)
  return {__float_as_uint(t1) - 0x4B000000u, __float_as_uint(t2) - 0x4B000000u};
}
__device__ __forceinline__ uint64_t fix46_u64(Fix46 w) {
  return ((uint64_t)w.hi << 23) + w.lo;
}
// fix46 of two weights on the packed fp32x2 pipe, lane for lane the scalar
// steps (-floor(a) is formed as 2^23 - t1, exactly), added to (hi, lo) as the
// raw bits of t1 and t2: each element adds 0x4B000000 to both, which the
// caller removes once per group (sums modulo 2^32, the true sums far below).
__device__ __forceinline__ void fix46x2_add(float2 r, uint32_t& hi, uint32_t& lo) {
  const float2 a = mul2_rn(r, f2(8388608.0f));
  const float2 t1 = add2_rm(a, f2(8388608.0f));
  const float2 f = add2_rn(a, fma2_rn(t1, f2(-1.0f), f2(8388608.0f)));
  const float2 t2 = fma2_rm(f, f2(8388608.0f), f2(8388608.0f));
  hi += __float_as_uint(t1.x) + __float_as_uint(t1.y);
  lo += __float_as_uint(t2.x) + __float_as_uint(t2.y);
}

constexpr float kLog2e = 1.4426950408889634f;

// 2^x by the hardware approximation (ex2.approx: a few units in the last place
// of relative error; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float e;
  asm("ex2.approx.f32 %0, %1;" : "=f"(e) : "f"(x));
  return e;
}

struct OpMaxNaNv {
  __device__ float operator()(float a, float b) const {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
  }
};

// max of two bf16 pairs, lane by lane; NaN when either lane is NaN
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

struct OpAddF {
  __device__ float operator()(float a, float b) const { return __fadd_rn(a, b); }
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void am_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// Verification of request b on one 8-CTA cluster (every CTA calls it with the
// same b): greedy (kG) and/or ratio (kR) mode over target rows of dtype kDt,
// both modes sharing each row's statistics; rows are read in order until
// every mode has decided.  `mbar` holds kVTma initialised mbarriers whose
// current phase parity is `phase` (updated here).  The draft tokens come from
// drafts_sm (shared memory of every CTA) when given, else from p.drafts; the
// count of draft j in its dense q row from cnt_sm when given, else from
// p.counts.
// kMatch: the stochastic (match) mode instead of the ratio mode, with the same
// outputs (r_*): every row draws from its own p (purpose MATCH) and a draw
// equal to the proposal accepts it.
// kCohQ: q was written by this same launch (see ldq).
template <bool kG, bool kR, int kDt, int NC = kVCluster, bool kMatch = false,
          bool kCohQ = false>
__device__ __forceinline__ void verify_request(const VParams& p, int b, VSh2& sh,
                                               unsigned char* vbuf, uint64_t* mbar,
                                               uint32_t& phase, const int32_t* drafts_sm,
                                               const uint32_t* cnt_sm) {
  constexpr int EPG = (kDt == DSPARK_F32) ? 4 : 8;  // elements per 16-byte group
  constexpr int ESZ = (kDt == DSPARK_F32) ? 4 : 2;
  cg::cluster_group cluster = cg::this_cluster();
  const float* vf = reinterpret_cast<const float*>(vbuf);
  const uint16_t* vh = reinterpret_cast<const uint16_t*>(vbuf);
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int depth = p.depth, V = p.V;
  const int lo = rank * p.chunk;
  const int n = max(0, min(V, lo + p.chunk) - lo);
  const int32_t* drafts_g = drafts_sm ? nullptr : p.drafts + (int64_t)b * depth;
  auto draft = [&](int j) -> int { return drafts_sm ? drafts_sm[j] : drafts_g[j]; };
  const uint32_t req = p.request_ids ? p.request_ids[b] : (uint32_t)b;

  int st0 = DSPARK_ST_OK;
  for (int j = 0; j < depth; ++j) {
    const int x = draft(j);
    if (x < 0 || x >= V) st0 = DSPARK_ST_BAD_DRAFT;
  }
  if (tid == 0) {
    sh.timeout = 0;
    // read only after a push (every draw has exactly one drawing CTA); a
    // missing push would stop the request uniformly
    sh.m_pick = -1;
    sh.m_st = DSPARK_ST_INTERNAL;
    sh.m_flags = 0u;
  }
  __syncthreads();
  int st_g = st0, st_r = st0;  // per-mode statuses
  static_assert(!(kR && kMatch), "the ratio and the match mode share the r_* outputs");
  constexpr bool kD = kR || kMatch;  // a mode that draws from p (needs the row sums)
  bool need_g = kG && st0 == DSPARK_ST_OK, need_r = kD && st0 == DSPARK_ST_OK;
  int L_g = depth, pick_g = -1;
  int xi = 0;
  int L = depth, pick = -1;  // ratio mode
  uint32_t flags = 0;
  int writer = -1;
  bool drawn = false;

  // the slice buffer holds chunk elements plus one 16-byte group of slack
  const int slice_groups = (p.chunk * ESZ + 32) / 16;
  (void)slice_groups;  // read by the checked build's bounds only
  auto val = [&](int s) -> float {
    if (!DSPARK_CHECK(s >= 0 && s < slice_groups * EPG)) return -INFINITY;
    if (kDt == DSPARK_F32) return vf[s];
    return __uint_as_float(((uint32_t)vh[s]) << 16);
  };
  // the EPG values of group g
  auto group = [&](int g, float* z) {
    if (!DSPARK_CHECK(g >= 0 && g < slice_groups)) {
#pragma unroll
      for (int i = 0; i < EPG; ++i) z[i] = -INFINITY;
      return;
    }
    if (kDt == DSPARK_F32) {
      const float4 q = reinterpret_cast<const float4*>(vbuf)[g];
      z[0] = q.x;
      z[1] = q.y;
      z[2] = q.z;
      z[3] = q.w;
    } else {
      const uint4 q = reinterpret_cast<const uint4*>(vbuf)[g];
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        z[2 * i] = __uint_as_float(w[i] << 16);
        z[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  };

  for (int j = 0; j <= depth && (need_g || need_r); ++j) {
    const char* zrow = reinterpret_cast<const char*>(p.z) +
                       ((int64_t)b * (depth + 1) + j) * p.ld * ESZ;
    const int off = (int)((reinterpret_cast<uintptr_t>(zrow + (int64_t)lo * ESZ) / ESZ) % EPG);
    const int ng = (off + n + EPG - 1) / EPG;
    const int g_first = (off == 0) ? 0 : 1;
    const int g_last = (off + n) / EPG - 1;
    const int n_int = max(0, g_last - g_first + 1);
    const char* gbase = zrow + (int64_t)(lo - off) * ESZ;  // 16-byte aligned
    __syncthreads();  // every read of the previous row's slice is done
    if (tid == 0 && n_int > 0) {
      fence_proxy_async_smem();
      for (int c = 0; c < kVTma; ++c) {
        const int g0 = g_first + (n_int * c) / kVTma, g1 = g_first + (n_int * (c + 1)) / kVTma;
        const uint32_t bytes = (uint32_t)(g1 - g0) * 16u;
        mbar_arrive_expect_tx(&mbar[c], bytes);
        if (bytes) tma_load_bulk(vbuf + 16 * g0, gbase + 16 * g0, bytes, &mbar[c]);
      }
      if (j < depth) {
        // the next row's part towards L2 while this row is decided: it is
        // read next unless this row decides every mode
        const char* nrow = zrow + p.ld * ESZ;
        const uintptr_t a0 = (reinterpret_cast<uintptr_t>(nrow + (int64_t)lo * ESZ) + 15u) &
                             ~(uintptr_t)15u;
        const uintptr_t a1 = reinterpret_cast<uintptr_t>(nrow + (int64_t)(lo + n) * ESZ) &
                             ~(uintptr_t)15u;
        if (a1 > a0) prefetch_l2(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
      }
    }
    if (tid < 2 * EPG) {
      const int g = (tid < EPG) ? 0 : ng - 1;
      if (g >= 0 && !(n_int > 0 && g >= g_first && g <= g_last)) {
        const int s = g * EPG + (tid % EPG);
        const bool in = (s >= off && s < off + n);
        if (kDt == DSPARK_F32)
          reinterpret_cast<float*>(vbuf)[s] =
              in ? __ldg(reinterpret_cast<const float*>(gbase) + s) : -INFINITY;
        else
          reinterpret_cast<uint16_t*>(vbuf)[s] =
              in ? __ldg(reinterpret_cast<const unsigned short*>(gbase) + s) : (uint16_t)0xFF80u;
      }
    }
    // ratio mode: the inputs of the decision, fetched while the copies fly
    float zx = 0.0f;
    uint32_t cx = 0u, U = 0u;
    const uint32_t* qrow = nullptr;  // dense counts row j
    const int32_t* sids = nullptr;   // sparse row j
    const uint32_t* scnt = nullptr;
    int snnz = 0;
    if (kR && need_r && j < depth) {
      const int x = draft(j);
      const int64_t qr = (int64_t)b * depth + j;
      if (p.top_k == 0) {
        qrow = p.counts + qr * V;
        if (tid == 0 && DSPARK_CHECK(x >= 0 && x < V))
          cx = cnt_sm ? cnt_sm[j] : ldq<kCohQ>(qrow + x);
      } else {
        // canonical sparse row: 1 <= nnz <= top_k, ids strictly ascending in
        // [0, V), counts > 0, total M
        const int32_t* ids = p.ids + qr * p.top_k;
        const uint32_t* cn = p.counts + qr * p.top_k;
        const int nz = p.nnz[qr];
        if (tid == 0) {
          sh.q_ok = 1;
          sh.q_c = 0u;
        }
        __syncthreads();
        uint64_t tot = 0;
        if (nz < 1 || nz > p.top_k) {
          if (tid == 0) sh.q_ok = 0;
        } else {
          for (int i = tid; i < nz; i += kVThreads) {
            if (!DSPARK_CHECK(i < p.top_k)) break;
            const int id = ids[i];
            const uint32_t cc = cn[i];
            if (id < 0 || id >= V || cc == 0u || (i > 0 && ids[i - 1] >= id)) sh.q_ok = 0;
            if (id == x) sh.q_c = cc;
            tot += cc;
          }
        }
        tot = block_reduce(tot, OpAddU64(), sh.wz);
        if (tid == 0 && nz >= 1 && nz <= p.top_k && tot != (uint64_t)kM) sh.q_ok = 0;
        __syncthreads();
        if (tid == 0) cx = sh.q_c;
        sids = ids;
        scnt = cn;
        snnz = nz;
      }
      if (tid == 0) {
        zx = DSPARK_CHECK(x >= 0 && x < V) ? load_logit(zrow, kDt, x) : -INFINITY;
        U = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_ACCEPT) >> 8;
      }
    }
    if (n_int > 0) {
      if (tid == 0)
        for (int c = 0; c < kVTma; ++c)
          if (!mbar_wait_bounded(&mbar[c], phase)) sh.timeout = 1;
      phase ^= 1u;
    }
    __syncthreads();

    // ---- row statistics of this slice.  Pass 1: the max, group by group
    // (bf16 pairs by one packed max), and for the greedy argmax the group
    // where each thread first met its own maximum.  Pass 2: the sum of exp
    // relative to the CTA's max; the CTA's argmax is the lowest id holding
    // that max, found in those groups.
    const bool trk = kG && need_g;
    float mx = -INFINITY, tmx = -INFINITY;
    int tg = -1;
    for (int g = tid; g < ng; g += kVThreads) {
      float gm = -INFINITY;
      if (DSPARK_CHECK(g < slice_groups)) {
        if (kDt == DSPARK_F32) {
          const float4 q = reinterpret_cast<const float4*>(vbuf)[g];
          gm = OpMaxNaNv()(OpMaxNaNv()(q.x, q.y), OpMaxNaNv()(q.z, q.w));
        } else {
          const uint4 q = reinterpret_cast<const uint4*>(vbuf)[g];
          const uint32_t m2 = bf16x2_max_nan(bf16x2_max_nan(q.x, q.y), bf16x2_max_nan(q.z, q.w));
          gm = OpMaxNaNv()(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
        }
      }
      mx = OpMaxNaNv()(mx, gm);
      if (trk && gm > tmx) {
        tmx = gm;
        tg = g;
      }
    }
    mx = warp_reduce(mx, OpMaxNaNv());
    if (lane == 0) sh.wm[warp] = mx;
    __syncthreads();
    float cm = sh.wm[0];  // the CTA's max
    for (int w = 1; w < kVThreads / 32; ++w) cm = OpMaxNaNv()(cm, sh.wm[w]);
    const bool cm_fin = cm > -INFINITY && cm < INFINITY;
    int ami = 0x7FFFFFFF;
    if (trk && cm_fin && tg >= 0 && tmx == cm) {
      float z[EPG];
      group(tg, z);
#pragma unroll
      for (int i = EPG - 1; i >= 0; --i)
        if (z[i] == cm) ami = lo - off + tg * EPG + i;
    }
    float sm = 0.0f;
    if (kD && need_r && cm_fin) {
      // each term by the hardware base-2 exponential (relative error a few
      // 2^-23) of RN(RN(z - cm) log2 e), pairs of arguments on the packed
      // pipe, the terms added in element order
      for (int g = tid; g < ng; g += kVThreads) {
        float z[EPG];
        group(g, z);
#pragma unroll
        for (int i = 0; i < EPG; i += 2) {
          const float2 t = mul2_rn(add2_rn(make_float2(z[i], z[i + 1]), f2(-cm)), f2(kLog2e));
          sm += ex2_approx(t.x);
          sm += ex2_approx(t.y);
        }
      }
    }
    if (kD && need_r) sm = warp_reduce(sm, OpAddF());
    if (trk) ami = __reduce_min_sync(0xffffffffu, ami);
    if (lane == 0) {
      sh.ws[warp] = sm;
      sh.wai[warp] = ami;
    }
    __syncthreads();
    if (tid == 0) {
      float s = 0.0f;
      int ai = 0x7FFFFFFF;
      for (int w = 0; w < kVThreads / 32; ++w) {
        if (kD && need_r) s += sh.ws[w];
        if (trk) ai = min(ai, sh.wai[w]);
      }
      VX& e = sh.x[xi];
      e.m = cm;
      e.s = s;
      e.amv = (ai != 0x7FFFFFFF) ? cm : -INFINITY;
      e.ami = ai;
      e.fl = sh.timeout ? 1u : 0u;
    }
    if (warp == 0) {
      // this CTA's partials into every peer's slot for it (lane r writes rank r)
      __syncwarp();
      if (lane < NC) *cluster.map_shared_rank(&sh.px[xi][rank], lane) = sh.x[xi];
    }
    cluster.sync();
    if (warp == 0) {
      // every CTA's partials, from local memory, merged by one lane in rank
      // order (identical in every CTA): warp shuffles queue behind the other
      // CTAs' shared-memory traffic here, and the whole cluster waits on
      // this.  The flags, the max and the argmax (lowest id among the maxima)
      // are exact; each slice's sum is rescaled to the row max and the
      // rescaled sums are added in rank order.
      bool bad = false;
      float m = -INFINITY, s = 0.0f, av = -INFINITY;
      int ai = 0x7FFFFFFF;
      uint32_t fl = 0;
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < NC; ++r) {
          const VX& e = sh.px[xi][r];
          bad = bad || !(e.m < INFINITY);  // NaN or +inf
          if (e.m < INFINITY) m = fmaxf(m, e.m);
          fl |= e.fl;
          if (kG && need_g) am_merge(av, ai, e.amv, e.ami);
        }
        if (kD && need_r && m > -INFINITY) {
#pragma unroll
          for (int r = 0; r < NC; ++r) {
            const VX& e = sh.px[xi][r];
            if (e.m > -INFINITY && e.m < INFINITY) s += e.s * expf(e.m - m);
          }
        }
      }
      if (lane == 0) {
        sh.M = bad ? NAN : m;
        sh.S = s;
        sh.AMV = av;
        sh.AMI = ai;
        sh.FL = fl;
        if (kR && need_r && j < depth && !bad && m > -INFINITY && !(fl & 1u)) {
          // the ratio test: accept iff U * c < p(x) * 2^48
          int dec = 0, dst = DSPARK_ST_OK;
          uint32_t dfl = 0;
          if (p.top_k > 0 && !sh.q_ok) {
            dec = -1;
            dst = DSPARK_ST_BAD_Q;
          } else if (cx == 0u) {
            dec = -1;
            dst = DSPARK_ST_BAD_DRAFT;
          } else {
            const float px = (zx == -INFINITY) ? 0.0f : __fdiv_rn(expf(zx - m), s);
            const double uc = (double)((uint64_t)U * (uint64_t)cx);
            const double p48 = (double)px * 281474976710656.0;
            if (fabs(uc * 0x1p-48 - (double)px) <= 1e-6 * ((double)cx * 0x1p-24))
              dfl = DSPARK_FLAG_AMBIG_ACCEPT;
            dec = (uc < p48) ? 1 : 0;
          }
          sh.dec = dec;
          sh.dst = dst;
          sh.dflags = dfl;
        }
      }
    }
    xi ^= 1;
    __syncthreads();
    const float M = sh.M, S = sh.S;
    // a refused row refuses the modes still reading it
    int row_st = DSPARK_ST_OK;
    if (sh.FL & 1u) row_st = DSPARK_ST_TIMEOUT;
    else if (!(M < INFINITY)) row_st = DSPARK_ST_NONFINITE;
    else if (M == -INFINITY) row_st = DSPARK_ST_ZERO_MASS;
    if (row_st != DSPARK_ST_OK) {
      if (need_g) st_g = row_st;
      if (need_r) st_r = row_st;
      break;
    }
    if (kG && need_g && (j == depth || sh.AMI != draft(j))) {
      L_g = j;
      pick_g = sh.AMI;
      need_g = false;
    }
    if (!(kD && need_r)) continue;

    // ---- ratio test of draft j (decided above by thread 0), or the match
    //      mode's draw from p_j
    bool use_q = false;
    uint32_t purpose = DSPARK_PURPOSE_BONUS;
    if (kMatch) {
      L = j;
      purpose = DSPARK_PURPOSE_MATCH;
    } else if (j < depth) {
      if (sh.dec < 0) {
        st_r = sh.dst;
        need_r = false;
        continue;
      }
      flags |= sh.dflags;
      if (sh.dec == 1) continue;  // accepted
      L = j;
      use_q = true;
      purpose = DSPARK_PURPOSE_RESIDUAL;
      if (qrow && tid == 0) {
        // the counts of this slice are read next: start them towards L2
        const uintptr_t a0 = (reinterpret_cast<uintptr_t>(qrow + lo) + 15) & ~(uintptr_t)15;
        const uintptr_t a1 = reinterpret_cast<uintptr_t>(qrow + lo + n) & ~(uintptr_t)15;
        if (a1 > a0) prefetch_l2(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
      }
    } else {
      L = depth;
    }

    // ---- final draw over row j: residual max(p - q, 0) or p itself
    const uint32_t wdraw = draw_u32(p.seed, req, (uint32_t)j, purpose);
    // p(v) = 2^((z - M) log2(e) - log2(S)) by the hardware base-2 exponential
    // (relative error a few 2^-23; -inf gives 0), one rounding of the argument
    const float nlgS = -log2f(S);
    auto pv = [&](float z) -> float {
      return ex2_approx(__fmaf_rn(__fsub_rn(z, M), kLog2e, nlgS));
    };
    auto wfix = [&](float r) -> uint64_t { return fix46_u64(fix46(r)); };
    const int nblk = (ng + 31) / 32;
    const bool qvec = qrow != nullptr &&
                      (reinterpret_cast<uintptr_t>(qrow + lo - off) & 15u) == 0u;
    // the EPG counts of group g of the dense q row (128-bit loads for a full,
    // aligned group; 0 outside the slice)
    auto load_q = [&](int g, uint32_t* qv) {
#pragma unroll
      for (int i = 0; i < EPG; ++i) qv[i] = 0u;
      if (qvec && g >= g_first && g <= g_last) {
        const uint4* qp = reinterpret_cast<const uint4*>(qrow + lo - off) + g * (EPG / 4);
#pragma unroll
        for (int k = 0; k < EPG / 4; ++k) {
          const uint4 t4 = ldq<kCohQ>(qp + k);
          qv[4 * k] = t4.x;
          qv[4 * k + 1] = t4.y;
          qv[4 * k + 2] = t4.z;
          qv[4 * k + 3] = t4.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < EPG; ++i) {
          const int s = g * EPG + i;
          if (s >= off && s < off + n) qv[i] = ldq<kCohQ>(qrow + (lo - off + s));
        }
      }
    };
    for (int attempt = 0; attempt < 2; ++attempt) {
      const bool dense_q = use_q && qrow != nullptr;
      const bool sparse_qm = use_q && sids != nullptr;
      uint64_t zs = 0, cs = 0;
      // the counts of a thread's next group are loaded one step ahead, so that
      // their latency overlaps the current group's arithmetic
      uint32_t qn[EPG];
#pragma unroll
      for (int i = 0; i < EPG; ++i) qn[i] = 0u;
      if (dense_q && tid < ng) load_q(tid, qn);
      for (int gb = 0; gb < ng; gb += kVThreads) {
        const int g = gb + tid;
        uint32_t ghi = 0, glo = 0;  // the group's weights: sum hi * 2^23 + sum lo
        uint32_t qv[EPG];
#pragma unroll
        for (int i = 0; i < EPG; ++i) qv[i] = qn[i];
        if (dense_q && g + kVThreads < ng) load_q(g + kVThreads, qn);
        if (g < ng) {
          float z[EPG];
          group(g, z);
          // pairs on the packed fp32x2 pipe: p as pv, max(p - c 2^-24, 0)
          // (c 2^-24 is exact, so one fma), the fixed-point weight as fix46
          uint32_t gc = 0;
#pragma unroll
          for (int i = 0; i < EPG; i += 2) {
            const float2 t = fma2_rn(add2_rn(make_float2(z[i], z[i + 1]), f2(-M)), f2(kLog2e),
                                     f2(nlgS));
            float2 r = make_float2(ex2_approx(t.x), ex2_approx(t.y));
            if (dense_q) {
              gc += qv[i] + qv[i + 1];
              r = fma2_rn(make_float2((float)qv[i], (float)qv[i + 1]), f2(-0x1p-24f), r);
              r.x = fmaxf(r.x, 0.0f);
              r.y = fmaxf(r.y, 0.0f);
            }
            fix46x2_add(r, ghi, glo);
          }
          ghi -= (uint32_t)EPG * 0x4B000000u;
          glo -= (uint32_t)EPG * 0x4B000000u;
          cs += gc;
        }
        // one block = the 32 groups of one warp in one iteration: each half
        // is at most 32 * EPG * 2^23 <= 2^31, summed by the 32-bit warp
        // reduction
        const uint32_t bhi = __reduce_add_sync(0xffffffffu, ghi);
        const uint32_t blo = __reduce_add_sync(0xffffffffu, glo);
        const uint64_t bs = ((uint64_t)bhi << 23) + blo;
        if (lane == 0 && gb / 32 + warp < nblk) sh.bsum[gb / 32 + warp] = bs;
        zs += ((uint64_t)ghi << 23) + glo;
      }
      __syncthreads();
      if (sparse_qm) {
        // support ids in this slice: their weight is max(p - q, 0), not p
        for (int i = tid; i < snnz; i += kVThreads) {
          const int v = ldq<kCohQ>(sids + i);
          if (v < lo || v >= lo + n) continue;
          const int s = v - lo + off;
          const float pr = pv(val(s));
          const float r = fmaxf(__fsub_rn(pr, (float)ldq<kCohQ>(scnt + i) * 0x1p-24f), 0.0f);
          const uint64_t d = wfix(pr) - wfix(r);
          if (!DSPARK_CHECK((s / EPG) / 32 < kVMaxBlocks)) continue;
          atomicAdd(reinterpret_cast<unsigned long long*>(&sh.bsum[(s / EPG) / 32]),
                    (unsigned long long)(0ull - d));
          zs -= d;
        }
      }
      zs = warp_reduce(zs, OpAddU64());
      cs = warp_reduce(cs, OpAddU64());
      if (lane == 0) {
        sh.wz[warp] = zs;
        sh.wc[warp] = cs;
      }
      __syncthreads();
      if (tid == 0) {
        uint64_t a = 0, c2 = 0;
        for (int w = 0; w < kVThreads / 32; ++w) {
          a += sh.wz[w];
          c2 += sh.wc[w];
        }
        sh.x[xi].z = a;
        sh.x[xi].cs = c2;
      }
      if (warp == 0) {
        // this CTA's masses into every peer's slot for it
        __syncwarp();
        if (lane < NC) {
          VX* dst = cluster.map_shared_rank(&sh.px[xi][rank], lane);
          dst->z = sh.x[xi].z;
          dst->cs = sh.x[xi].cs;
        }
      }
      cluster.sync();
      if (warp == 0) {
        // every CTA's masses, from local memory, summed exactly by one lane
        if (lane == 0) {
          uint64_t before = 0, Z = 0, CS = 0;
#pragma unroll
          for (int r = 0; r < NC; ++r) {
            const uint64_t zr = sh.px[xi][r].z;
            if (r < rank) before += zr;
            Z += zr;
            CS += sh.px[xi][r].cs;
          }
          sh.Z = Z;
          sh.before = before;
          sh.CS = CS;
        }
      }
      xi ^= 1;
      __syncthreads();
      const uint64_t Z = sh.Z, before = sh.before;
      const uint64_t mine = sh.x[xi ^ 1].z;
      if (dense_q && sh.CS != (uint64_t)kM) {
        st_r = DSPARK_ST_BAD_Q;
        break;
      }
      if (Z == 0ull && use_q) {  // no residual mass: draw from p instead
        flags |= DSPARK_FLAG_DEGENERATE;
        use_q = false;
        continue;
      }
      const uint64_t T = __umul64hi((uint64_t)wdraw << 32, Z);  // floor(w * Z / 2^32) < Z
      drawn = true;
      writer = -1;
      if (T >= before && T - before < mine) {
        // the block holding T, then the token inside it (warp 0)
        if (warp == 0) {
          const uint64_t t = T - before;
          uint64_t base = 0;
          int blk = -1;
          for (int k0 = 0; k0 < nblk && blk < 0; k0 += 32) {
            const int k = k0 + lane;
            const uint64_t v = (k < nblk && DSPARK_CHECK(k < kVMaxBlocks)) ? sh.bsum[k] : 0ull;
            uint64_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint64_t u = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += u;
            }
            const bool hit = (k < nblk) && v > 0ull && t - base < incl && t - base >= incl - v;
            const unsigned msk = __ballot_sync(0xffffffffu, hit);
            if (msk) {
              const int l = __ffs(msk) - 1;
              blk = k0 + l;
              base += __shfl_sync(0xffffffffu, incl - v, l);
            } else {
              base += __shfl_sync(0xffffffffu, incl, 31);
            }
          }
          int found = -1;
          uint32_t near = 0u;
          if (blk >= 0) {
            const int g = blk * 32 + lane;
            uint64_t wv[EPG];
            uint64_t gsum = 0;
            // the block's counts: a dense row's by 128-bit loads, issued
            // before any arithmetic; a sparse row's support ids that fall in
            // the block's id range, found by the whole warp and scattered
            // into shared memory
            uint32_t qv[EPG];
#pragma unroll
            for (int i = 0; i < EPG; ++i) qv[i] = 0u;
            if (use_q && qrow && g < ng) load_q(g, qv);
            if (use_q && sids) {
              const int v0 = lo - off + blk * 32 * EPG;  // id of the block's first position
#pragma unroll
              for (int i = 0; i < EPG; ++i) sh.qblk[i * 32 + lane] = 0u;
              __syncwarp();
              for (int k = lane; k < snnz; k += 32) {
                const int id = ldq<kCohQ>(sids + k);
                const int rel = id - v0;
                if (rel >= 0 && rel < 32 * EPG) sh.qblk[rel] = ldq<kCohQ>(scnt + k);
              }
              __syncwarp();
#pragma unroll
              for (int i = 0; i < EPG; ++i) {
                const int s = g * EPG + i;
                qv[i] = (s >= off && s < off + n) ? sh.qblk[lane * EPG + i] : 0u;
              }
            }
            if (g < ng) {
              float z[EPG];
              group(g, z);
#pragma unroll
              for (int i = 0; i < EPG; ++i) {
                const int s = g * EPG + i;
                const bool in = (s >= off && s < off + n);
                float r = pv(z[i]);
                if (use_q && in) r = fmaxf(__fsub_rn(r, (float)qv[i] * 0x1p-24f), 0.0f);
                wv[i] = wfix(r);
                gsum += wv[i];
              }
            } else {
#pragma unroll
              for (int i = 0; i < EPG; ++i) wv[i] = 0ull;
            }
            uint64_t incl = gsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint64_t u = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += u;
            }
            const uint64_t tb = t - base;  // position inside the block
            const bool hit = gsum > 0ull && tb < incl && tb >= incl - gsum;
            const unsigned msk = __ballot_sync(0xffffffffu, hit);
            if (msk && lane == __ffs(msk) - 1) {
              uint64_t cum = incl - gsum;
              for (int i = 0; i < EPG; ++i) {
                const uint64_t prev = cum;
                cum += wv[i];
                if (tb < cum) {
                  found = lo - off + g * EPG + i;
                  near = (tb - prev <= kNearTol || cum - tb <= kNearTol) ? 1u : 0u;
                  break;
                }
              }
              sh.found = found;
              sh.near = near;
            }
            if (!msk && lane == 0) {
              sh.found = -1;
              sh.near = 0u;
            }
          } else if (lane == 0) {
            sh.found = -1;
            sh.near = 0u;
          }
        }
        __syncthreads();
        pick = sh.found;
        if (sh.near) flags |= DSPARK_FLAG_NEAR_BOUNDARY;
        if (pick < 0) st_r = DSPARK_ST_INTERNAL;
        writer = rank;
      }
      break;
    }
    if (kMatch) {
      // only the CTA that drew the token knows it: it pushes the token, the
      // status and the boundary flag to every CTA, so that all of them take
      // the same decision (and the same barriers) below
      if (writer == rank && tid == 0)
        for (int r = 0; r < NC; ++r) {
          VSh2* peer = cluster.map_shared_rank(&sh, r);
          peer->m_pick = pick;
          peer->m_st = st_r;
          peer->m_flags = flags;
        }
      cluster.sync();
      pick = sh.m_pick;
      st_r = sh.m_st;
      flags |= sh.m_flags;
      // a draw equal to the proposal accepts it, and the next row draws
      if (st_r == DSPARK_ST_OK && j < depth && pick == draft(j)) continue;
    }
    need_r = false;
  }

  // outputs: greedy and ratio refusals by rank 0; after a ratio draw, by the
  // CTA that found the token
  if (kG && rank == 0 && tid == 0 && DSPARK_CHECK(b < p.B && L_g <= depth)) {
    int32_t* com = p.g_committed + (int64_t)b * (depth + 1);
    if (st_g != DSPARK_ST_OK) {
      p.g_accept_len[b] = 0;
      for (int i = 0; i <= depth; ++i) com[i] = -1;
    } else {
      p.g_accept_len[b] = L_g;
      for (int i = 0; i < L_g; ++i) com[i] = draft(i);
      com[L_g] = pick_g;
      for (int i = L_g + 1; i <= depth; ++i) com[i] = -1;
    }
    p.g_status[b] = st_g;
  }
  const bool i_write = drawn ? (writer == rank) : (rank == 0);
  if (kD && i_write && tid == 0 && DSPARK_CHECK(b < p.B && L <= depth)) {
    int32_t* com = p.r_committed + (int64_t)b * (depth + 1);
    if (st_r != DSPARK_ST_OK) {
      p.r_accept_len[b] = 0;
      for (int i = 0; i <= depth; ++i) com[i] = -1;
      if (p.r_flags) p.r_flags[b] = 0u;
    } else {
      p.r_accept_len[b] = L;
      for (int i = 0; i < L; ++i) com[i] = draft(i);
      com[L] = pick;
      for (int i = L + 1; i <= depth; ++i) com[i] = -1;
      if (p.r_flags) p.r_flags[b] = flags;
    }
    p.r_status[b] = st_r;
  }
  cluster.sync();  // no CTA leaves while a peer may still read its shared memory
}

}  // namespace
}  // namespace vfy
}  // namespace dspark
