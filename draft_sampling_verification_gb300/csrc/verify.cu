// verify.cu -- greedy and standard ratio verification, one 8-CTA cluster per
// request, plus the target distribution p of a batch of rows.
//
// "PP1 q transport and scheduling design": ratio tests and full-vocabulary
// residual sampling with the target p (T = 1) and the dyadic q; separate
// acceptance and correction/bonus RNG domains.  "DeepSeek-V4.1 DSpark",
// State and sampling contracts: greedy verification matches the target
// argmax and stops at the first mismatch.
//
// A request's target rows are visited in order; each CTA streams one eighth
// of the row (128-bit loads) keeping an online max / sum of exp and the first
// argmax, the cluster combines the eight partials in rank order (identical
// in every CTA), and the request stops at the deciding row, so rows after
// the first rejection are never read.  The correction / bonus draw re-reads
// row L (an L2 hit) and scans exact 46-bit fixed-point residual weights.
#include "common.cuh"

namespace dspark {

constexpr int kVCluster = 8;
constexpr int kVThreads = 256;
constexpr float kTwo46f = 70368744177664.0f;
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
  int32_t* accept_len;
  int32_t* committed;
  uint32_t* flags;
  int32_t* status;
  int chunk;
};

struct RowStat {
  float m;      // max logit
  float s;      // sum exp(z - m)
  float amv;    // argmax value
  int ami;      // argmax id (lowest among maxima)
  uint32_t bad; // bit0 NaN/+inf
};

struct VPub {
  RowStat st;
  uint64_t z;       // residual mass of this CTA's slice (fixed point)
  uint64_t csum;    // q mass of this CTA's slice (dense rows)
  int pick;
  uint32_t pick_near;
};

struct VShared {
  VPub pub;
  float redf[32];
  uint32_t red32[32];
  uint64_t red64[32];
  int redi[32];
  int q_ok;         // sparse row check result
  uint32_t q_c;     // count at the draft token
};

__device__ __forceinline__ RowStat stat_identity() {
  RowStat r;
  r.m = -INFINITY;
  r.s = 0.0f;
  r.amv = -INFINITY;
  r.ami = 0x7FFFFFFF;
  r.bad = 0u;
  return r;
}

// Merge b into a; a holds lower ids than b when `a_first` (argmax ties).
__device__ __forceinline__ RowStat stat_merge(RowStat a, RowStat b) {
  RowStat r;
  r.m = fmaxf(a.m, b.m);
  if (r.m == -INFINITY) {
    r.s = 0.0f;
  } else {
    const float sa = (a.m == -INFINITY) ? 0.0f : a.s * expf(a.m - r.m);
    const float sb = (b.m == -INFINITY) ? 0.0f : b.s * expf(b.m - r.m);
    r.s = sa + sb;
  }
  if (b.amv > a.amv || (b.amv == a.amv && b.ami < a.ami)) {
    r.amv = b.amv;
    r.ami = b.ami;
  } else {
    r.amv = a.amv;
    r.ami = a.ami;
  }
  r.bad = a.bad | b.bad;
  return r;
}

__device__ __forceinline__ void stat_push(RowStat& st, float zv, int v) {
  if (isnan(zv) || zv == INFINITY) {
    st.bad |= 1u;
    return;
  }
  if (zv > st.amv) {
    st.amv = zv;
    st.ami = v;
  }
  if (zv == -INFINITY) return;
  if (zv > st.m) {
    st.s = (st.m == -INFINITY) ? 1.0f : st.s * expf(st.m - zv) + 1.0f;
    st.m = zv;
  } else {
    st.s += expf(zv - st.m);
  }
}

// Calls fn(v, z) for every element v in [lo, lo+n) of a logit row, each
// thread visiting its elements in increasing v; 128-bit loads where aligned.
template <typename Fn>
__device__ __forceinline__ void row_foreach(const void* row, int dtype, int lo, int n, Fn fn) {
  if (n <= 0) return;
  if (dtype == DSPARK_F32) {
    const float* r = reinterpret_cast<const float*>(row);
    const int off = (int)((reinterpret_cast<uintptr_t>(r + lo) >> 2) & 3);
    const int ng = (off + n + 3) >> 2;
    const float* base = r + lo - off;
    for (int g = threadIdx.x; g < ng; g += blockDim.x) {
      const int s0 = 4 * g;
      if (s0 >= off && s0 + 3 < off + n) {
        const float4 q = __ldg(reinterpret_cast<const float4*>(base + s0));
        const int v0 = lo - off + s0;
        fn(v0, q.x);
        fn(v0 + 1, q.y);
        fn(v0 + 2, q.z);
        fn(v0 + 3, q.w);
      } else {
        for (int i = 0; i < 4; ++i) {
          const int s = s0 + i;
          if (s >= off && s < off + n) fn(lo - off + s, __ldg(base + s));
        }
      }
    }
  } else {
    const unsigned short* r = reinterpret_cast<const unsigned short*>(row);
    const int off = (int)((reinterpret_cast<uintptr_t>(r + lo) >> 1) & 7);
    const int ng = (off + n + 7) >> 3;
    const unsigned short* base = r + lo - off;
    for (int g = threadIdx.x; g < ng; g += blockDim.x) {
      const int s0 = 8 * g;
      if (s0 >= off && s0 + 7 < off + n) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(base + s0));
        const int v0 = lo - off + s0;
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        for (int i = 0; i < 4; ++i) {
          fn(v0 + 2 * i, __uint_as_float(w[i] << 16));
          fn(v0 + 2 * i + 1, __uint_as_float(w[i] & 0xFFFF0000u));
        }
      } else {
        for (int i = 0; i < 8; ++i) {
          const int s = s0 + i;
          if (s >= off && s < off + n) fn(lo - off + s, bf16_to_f32(__ldg(base + s)));
        }
      }
    }
  }
}

__device__ RowStat block_stat(RowStat st, VShared& sh) {
  // warp level
  for (int o = 16; o > 0; o >>= 1) {
    RowStat b;
    b.m = __shfl_xor_sync(0xffffffffu, st.m, o);
    b.s = __shfl_xor_sync(0xffffffffu, st.s, o);
    b.amv = __shfl_xor_sync(0xffffffffu, st.amv, o);
    b.ami = __shfl_xor_sync(0xffffffffu, st.ami, o);
    b.bad = __shfl_xor_sync(0xffffffffu, st.bad, o);
    st = stat_merge(st, b);
  }
  __shared__ RowStat wst[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) wst[warp] = st;
  __syncthreads();
  RowStat r = wst[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = stat_merge(r, wst[i]);
  return r;
}

// Stats of [lo, lo+n) of one row, reduced over the block.
__device__ RowStat slice_stat(const void* row, int dtype, int lo, int n, VShared& sh) {
  RowStat st = stat_identity();
  row_foreach(row, dtype, lo, n, [&](int v, float zv) { stat_push(st, zv, v); });
  return block_stat(st, sh);
}

// ------------------------------------------------------- verification
// One 8-CTA cluster per request.  Each target row's slice arrives in shared
// memory by bulk copies (interior 16-byte groups) and plain loads (the two
// partial edge groups); the statistics are two cheap passes over it (max and
// first argmax; sum of exp relative to the thread's own max), merged per
// block and then across the cluster in rank order.  The exchange slots are
// double-buffered, so each exchange costs one cluster barrier.  The final
// draw computes exact 46-bit fixed-point weights of row L once, keeps the
// mass of every block of 32 groups, and the CTA holding the draw finds its
// block from those sums and its token with one warp.
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

struct VSh2 {
  VX x[2];
  uint64_t mbar[kVTma];
  uint64_t bsum[kVMaxBlocks];
  float wm[8], ws[8], wam[8];
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
  int dec;          // ratio decision of the row: 1 accept, 0 reject, -1 refuse (status in dst)
  int dst;
  uint32_t dflags;
};

struct OpMaxNaNv {
  __device__ float operator()(float a, float b) const {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
  }
};

struct OpAddF {
  __device__ float operator()(float a, float b) const { return __fadd_rn(a, b); }
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// (m, s) pairs: s is a sum of exp(z - m); merged to the larger m.
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) {
    m = M;
    s = 0.0f;
    return;
  }
  const float a = (m == -INFINITY) ? 0.0f : s * expf(m - M);
  const float c = (m2 == -INFINITY) ? 0.0f : s2 * expf(m2 - M);
  m = M;
  s = a + c;
}

__device__ __forceinline__ void am_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

template <int kMode, int kDt>
__global__ void __cluster_dims__(kVCluster, 1, 1) __launch_bounds__(kVThreads, 3)
    verify_kernel(VParams p) {
  constexpr int EPG = (kDt == DSPARK_F32) ? 4 : 8;  // elements per 16-byte group
  constexpr int ESZ = (kDt == DSPARK_F32) ? 4 : 2;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ VSh2 sh;
  extern __shared__ __align__(128) unsigned char vbuf[];
  const float* vf = reinterpret_cast<const float*>(vbuf);
  const uint16_t* vh = reinterpret_cast<const uint16_t*>(vbuf);
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / kVCluster;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int depth = p.depth, V = p.V;
  const int lo = rank * p.chunk;
  const int n = max(0, min(V, lo + p.chunk) - lo);
  const int32_t* drafts = p.drafts + (int64_t)b * depth;
  const uint32_t req = p.request_ids ? p.request_ids[b] : (uint32_t)b;

  int status = DSPARK_ST_OK;
  for (int j = 0; j < depth; ++j) {
    const int x = drafts[j];
    if (x < 0 || x >= V) status = DSPARK_ST_BAD_DRAFT;
  }
  if (tid == 0) {
    for (int c = 0; c < kVTma; ++c) mbar_init(&sh.mbar[c], 1);
    mbar_init_fence();
    sh.timeout = 0;
  }
  __syncthreads();
  uint32_t phase = 0;
  int xi = 0;
  int L = depth, pick = -1;
  uint32_t flags = 0;
  int writer = -1;
  bool drawn = false;

  auto val = [&](int s) -> float {
    if (kDt == DSPARK_F32) return vf[s];
    return __uint_as_float(((uint32_t)vh[s]) << 16);
  };
  // the EPG values of group g
  auto group = [&](int g, float* z) {
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

  for (int j = 0; j <= depth && status == DSPARK_ST_OK; ++j) {
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
        mbar_arrive_expect_tx(&sh.mbar[c], bytes);
        if (bytes) tma_load_bulk(vbuf + 16 * g0, gbase + 16 * g0, bytes, &sh.mbar[c]);
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
    if (kMode == kRatio && j < depth) {
      const int x = drafts[j];
      const int64_t qr = (int64_t)b * depth + j;
      if (p.top_k == 0) {
        qrow = p.counts + qr * V;
        if (tid == 0) cx = __ldg(qrow + x);
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
        zx = load_logit(zrow, kDt, x);
        U = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_ACCEPT) >> 8;
      }
    }
    if (n_int > 0) {
      if (tid == 0)
        for (int c = 0; c < kVTma; ++c)
          if (!mbar_wait_bounded(&sh.mbar[c], phase)) sh.timeout = 1;
      phase ^= 1u;
    }
    __syncthreads();

    // ---- row statistics of this slice
    float mx = -INFINITY, sm = 0.0f, amv = -INFINITY;
    int ami = 0x7FFFFFFF;
    for (int g = tid; g < ng; g += kVThreads) {
      float z[EPG];
      group(g, z);
#pragma unroll
      for (int i = 0; i < EPG; ++i) {
        mx = OpMaxNaNv()(mx, z[i]);
        if (kMode == kGreedy && z[i] > amv) {
          amv = z[i];
          ami = lo - off + g * EPG + i;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mx = OpMaxNaNv()(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (kMode == kGreedy) {
        const float a2 = __shfl_xor_sync(0xffffffffu, amv, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, ami, o);
        am_merge(amv, ami, a2, i2);
      }
    }
    if (lane == 0) {
      sh.wm[warp] = mx;
      sh.wam[warp] = amv;
      sh.wai[warp] = ami;
    }
    __syncthreads();
    float cm = sh.wm[0];  // the CTA's max
    for (int w = 1; w < kVThreads / 32; ++w) cm = OpMaxNaNv()(cm, sh.wm[w]);
    if (kMode == kRatio) {
      // the sum of exp relative to the CTA's max: a plain sum
      if (cm > -INFINITY && cm < INFINITY)
        for (int g = tid; g < ng; g += kVThreads) {
          float z[EPG];
          group(g, z);
#pragma unroll
          for (int i = 0; i < EPG; ++i) sm += expf(__fsub_rn(z[i], cm));
        }
      sm = warp_reduce(sm, OpAddF());
      if (lane == 0) sh.ws[warp] = sm;
      __syncthreads();
    }
    if (tid == 0) {
      float m = cm, s = 0.0f, av = sh.wam[0];
      int ai = sh.wai[0];
      for (int w = 0; w < kVThreads / 32; ++w) {
        if (kMode == kRatio) s += sh.ws[w];
        else if (w > 0) am_merge(av, ai, sh.wam[w], sh.wai[w]);
      }
      VX& e = sh.x[xi];
      e.m = m;
      e.s = s;
      e.amv = av;
      e.ami = ai;
      e.fl = sh.timeout ? 1u : 0u;
    }
    cluster.sync();
    if (tid == 0) {
      // peers' partials in rank order (identical in every CTA)
      float m = -INFINITY, s = 0.0f, av = -INFINITY;
      int ai = 0x7FFFFFFF;
      uint32_t fl = 0;
      bool bad = false;
      for (int r = 0; r < kVCluster; ++r) {
        const VX* e = cluster.map_shared_rank(&sh.x[xi], r);
        const float m2 = e->m;
        fl |= e->fl;
        if (!(m2 < INFINITY)) bad = true;  // NaN or +inf in that slice
        if (kMode == kRatio) ms_merge(m, s, bad ? -INFINITY : m2, bad ? 0.0f : e->s);
        else {
          m = fmaxf(m, m2);
          am_merge(av, ai, e->amv, e->ami);
        }
      }
      sh.M = bad ? NAN : m;
      sh.S = s;
      sh.AMV = av;
      sh.AMI = ai;
      sh.FL = fl;
      if (kMode == kRatio && j < depth && !bad && m > -INFINITY && !(fl & 1u)) {
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
    xi ^= 1;
    __syncthreads();
    const float M = sh.M, S = sh.S;
    if (sh.FL & 1u) {
      status = DSPARK_ST_TIMEOUT;
      break;
    }
    if (!(M < INFINITY)) {
      status = DSPARK_ST_NONFINITE;
      break;
    }
    if (M == -INFINITY) {
      status = DSPARK_ST_ZERO_MASS;
      break;
    }
    if (kMode == kGreedy) {
      if (j == depth || sh.AMI != drafts[j]) {
        L = j;
        pick = sh.AMI;
        break;
      }
      continue;
    }

    // ---- ratio test of draft j (decided above by thread 0)
    bool use_q = false;
    uint32_t purpose = DSPARK_PURPOSE_BONUS;
    if (j < depth) {
      if (sh.dec < 0) {
        status = sh.dst;
        break;
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
    const float invS = __frcp_rn(S);
    auto pv = [&](float z) -> float {
      return (z == -INFINITY) ? 0.0f : __fmul_rn(expf(z - M), invS);
    };
    auto wfix = [&](float r) -> uint64_t { return __float2ull_rz(__fmul_rn(r, kTwo46f)); };
    // q of the sparse row at id v (binary search; -1 ids never match)
    auto sparse_q = [&](int v) -> uint32_t {
      int a = 0, e = snnz - 1;
      while (a <= e) {
        const int mid = (a + e) >> 1;
        const int id = __ldg(sids + mid);
        if (id == v) return __ldg(scnt + mid);
        if (id < v) a = mid + 1;
        else e = mid - 1;
      }
      return 0u;
    };
    const int nblk = (ng + 31) / 32;
    const bool qvec = qrow != nullptr &&
                      (reinterpret_cast<uintptr_t>(qrow + lo - off) & 15u) == 0u;
    for (int attempt = 0; attempt < 2; ++attempt) {
      const bool dense_q = use_q && qrow != nullptr;
      const bool sparse_qm = use_q && sids != nullptr;
      uint64_t zs = 0, cs = 0;
      for (int gb = 0; gb < ng; gb += kVThreads) {
        const int g = gb + tid;
        uint64_t gsum = 0;
        if (g < ng) {
          // the counts first (128-bit loads for a full, aligned group), then
          // the weights
          uint32_t qv[EPG];
#pragma unroll
          for (int i = 0; i < EPG; ++i) qv[i] = 0u;
          if (dense_q) {
            if (qvec && g >= g_first && g <= g_last) {
              const uint4* qp = reinterpret_cast<const uint4*>(qrow + lo - off) + g * (EPG / 4);
#pragma unroll
              for (int k = 0; k < EPG / 4; ++k) {
                const uint4 t4 = __ldg(qp + k);
                qv[4 * k] = t4.x;
                qv[4 * k + 1] = t4.y;
                qv[4 * k + 2] = t4.z;
                qv[4 * k + 3] = t4.w;
              }
            } else {
#pragma unroll
              for (int i = 0; i < EPG; ++i) {
                const int s = g * EPG + i;
                if (s >= off && s < off + n) qv[i] = __ldg(qrow + (lo - off + s));
              }
            }
          }
          float z[EPG];
          group(g, z);
#pragma unroll
          for (int i = 0; i < EPG; ++i) {
            float r = pv(z[i]);
            if (dense_q) {
              cs += qv[i];
              r = fmaxf(__fsub_rn(r, (float)qv[i] * 0x1p-24f), 0.0f);
            }
            gsum += wfix(r);
          }
        }
        // one block = the 32 groups of one warp in one iteration
        const uint64_t bs = warp_reduce(gsum, OpAddU64());
        if (lane == 0 && gb / 32 + warp < nblk) sh.bsum[gb / 32 + warp] = bs;
        zs += gsum;
      }
      __syncthreads();
      if (sparse_qm) {
        // support ids in this slice: their weight is max(p - q, 0), not p
        for (int i = tid; i < snnz; i += kVThreads) {
          const int v = __ldg(sids + i);
          if (v < lo || v >= lo + n) continue;
          const int s = v - lo + off;
          const float pr = pv(val(s));
          const float r = fmaxf(__fsub_rn(pr, (float)__ldg(scnt + i) * 0x1p-24f), 0.0f);
          const uint64_t d = wfix(pr) - wfix(r);
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
      cluster.sync();
      if (tid == 0) {
        uint64_t before = 0, Z = 0, CS = 0;
        for (int r = 0; r < kVCluster; ++r) {
          const VX* e = cluster.map_shared_rank(&sh.x[xi], r);
          const uint64_t zr = e->z;
          if (r < rank) before += zr;
          Z += zr;
          CS += e->cs;
        }
        sh.Z = Z;
        sh.before = before;
        sh.CS = CS;
      }
      xi ^= 1;
      __syncthreads();
      const uint64_t Z = sh.Z, before = sh.before;
      const uint64_t mine = sh.x[xi ^ 1].z;
      if (dense_q && sh.CS != (uint64_t)kM) {
        status = DSPARK_ST_BAD_Q;
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
            const uint64_t v = (k < nblk) ? sh.bsum[k] : 0ull;
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
            if (g < ng) {
              float z[EPG];
              group(g, z);
#pragma unroll
              for (int i = 0; i < EPG; ++i) {
                const int s = g * EPG + i;
                const bool in = (s >= off && s < off + n);
                float r = pv(z[i]);
                if (use_q && in) {
                  const uint32_t q = qrow ? __ldg(qrow + (lo - off + s)) : sparse_q(lo - off + s);
                  r = fmaxf(__fsub_rn(r, (float)q * 0x1p-24f), 0.0f);
                }
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
        if (pick < 0) status = DSPARK_ST_INTERNAL;
        writer = rank;
      }
      break;
    }
    break;
  }

  // outputs: greedy and refusals by rank 0; after a draw, by the CTA that
  // found the token
  const bool i_write = drawn ? (writer == rank) : (rank == 0);
  if (i_write && tid == 0) {
    int32_t* com = p.committed + (int64_t)b * (depth + 1);
    if (status != DSPARK_ST_OK) {
      p.accept_len[b] = 0;
      for (int i = 0; i <= depth; ++i) com[i] = -1;
      if (p.flags) p.flags[b] = 0u;
    } else {
      p.accept_len[b] = L;
      for (int i = 0; i < L; ++i) com[i] = drafts[i];
      com[L] = pick;
      for (int i = L + 1; i <= depth; ++i) com[i] = -1;
      if (p.flags) p.flags[b] = flags;
    }
    p.status[b] = status;
  }
  cluster.sync();  // no CTA leaves while a peer may still read its shared memory
}

// ------------------------------------------------------------ target p
struct PParams {
  const void* z;
  int dtype;
  int64_t ld;
  int n_rows;
  int V;
  float* p_out;
  int32_t* argmax;
  int32_t* status;
  int chunk;
};

__global__ void __cluster_dims__(kVCluster, 1, 1) __launch_bounds__(kVThreads, 2)
    target_probs_kernel(PParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ VShared sh;
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.x / kVCluster;
  const int lo = rank * p.chunk;
  const int n = max(0, min(p.V, lo + p.chunk) - lo);
  const void* zr = reinterpret_cast<const char*>(p.z) + (int64_t)row * p.ld * (p.dtype == DSPARK_F32 ? 4 : 2);
  const RowStat mine = slice_stat(zr, p.dtype, lo, n, sh);
  if (threadIdx.x == 0) sh.pub.st = mine;
  cluster.sync();
  RowStat st = cluster.map_shared_rank(&sh.pub, 0)->st;
  for (int r = 1; r < kVCluster; ++r) st = stat_merge(st, cluster.map_shared_rank(&sh.pub, r)->st);
  cluster.sync();
  int status = DSPARK_ST_OK;
  if (st.bad) status = DSPARK_ST_NONFINITE;
  else if (st.m == -INFINITY) status = DSPARK_ST_ZERO_MASS;
  if (p.p_out) {
    float* out = p.p_out + (int64_t)row * p.V;
    if (status == DSPARK_ST_OK) {
      row_foreach(zr, p.dtype, lo, n, [&](int v, float zv) {
        out[v] = (zv == -INFINITY) ? 0.0f : __fdiv_rn(expf(zv - st.m), st.s);
      });
    } else {
      for (int v = lo + threadIdx.x; v < lo + n; v += blockDim.x) out[v] = 0.0f;
    }
  }
  if (rank == 0 && threadIdx.x == 0) {
    if (p.argmax) p.argmax[row] = (status == DSPARK_ST_OK) ? st.ami : -1;
    p.status[row] = status;
  }
}

static int verify_chunk(int V) {
  int c = (V + kVCluster - 1) / kVCluster;
  return (c + 7) & ~7;
}

cudaError_t launch_verify(int mode, const void* z, int dtype, int64_t ld, int B, int depth, int V,
                          const int32_t* drafts, const uint32_t* counts, const int32_t* ids,
                          const int32_t* nnz, int top_k, uint64_t seed,
                          const uint32_t* request_ids, int32_t* accept_len, int32_t* committed,
                          uint32_t* flags, int32_t* status, cudaStream_t stream) {
  VParams p;
  p.z = z;
  p.dtype = dtype;
  p.ld = ld;
  p.B = B;
  p.depth = depth;
  p.V = V;
  p.drafts = drafts;
  p.counts = counts;
  p.ids = ids;
  p.nnz = nnz;
  p.top_k = top_k;
  p.seed = seed;
  p.request_ids = request_ids;
  p.accept_len = accept_len;
  p.committed = committed;
  p.flags = flags;
  p.status = status;
  p.chunk = verify_chunk(V);
  // the slice buffer: chunk elements plus one 16-byte group of slack
  const int esz = (dtype == DSPARK_F32) ? 4 : 2;
  const int smem = p.chunk * esz + 32;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    kern<<<B * kVCluster, kVThreads, smem, stream>>>(p);
    return cudaGetLastError();
  };
  if (mode == kGreedy)
    return dtype == DSPARK_F32 ? go(verify_kernel<kGreedy, DSPARK_F32>)
                               : go(verify_kernel<kGreedy, DSPARK_BF16>);
  return dtype == DSPARK_F32 ? go(verify_kernel<kRatio, DSPARK_F32>)
                             : go(verify_kernel<kRatio, DSPARK_BF16>);
}

cudaError_t launch_target_probs(const void* z, int dtype, int64_t ld, int n_rows, int V,
                                float* p_out, int32_t* argmax, int32_t* status,
                                cudaStream_t stream) {
  PParams p;
  p.z = z;
  p.dtype = dtype;
  p.ld = ld;
  p.n_rows = n_rows;
  p.V = V;
  p.p_out = p_out;
  p.argmax = argmax;
  p.status = status;
  p.chunk = verify_chunk(V);
  target_probs_kernel<<<n_rows * kVCluster, kVThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dspark
