// q_dense.cu -- dyadic24-standard-v1 q construction for dense rows (no top-k
// support), optionally fused with the draft draw ("PP1 q transport and
// scheduling design", Distribution contract and precision: proposal
// construction, integer draw).
//
// One 8-CTA thread-block cluster per draft row, 256 threads per CTA, three
// CTAs per SM.  Each CTA keeps one eighth of the row in shared memory for the
// whole build (TMA bulk copies), so the row is read from HBM once and the
// counts are written once.  Row-wide values go through distributed shared
// memory: every CTA publishes its partial, and after a cluster barrier one
// warp of every CTA combines all eight in rank order, so all CTAs hold
// identical values.
//
// Passes over the resident slice (per element, branch-free in the common
// case; the rare cases are voted per warp and handled out of line):
//   A  m = max x with NaN propagation (NaN or +inf anywhere refuses the row);
//      with a temperature, m = RN(max x * RN(1/T)) -- RN is monotone.
//   B  E = floor(exp_ds(y - m) * 2^40) as an exact float, in place; S = sum E.
//   C  a = RN64(E * RN64(2^24 / RN64(S))): with k = khi + klo + d (khi =
//      RN32(k), klo = RN32(k - khi), |d| <= 2^-48 k) and p1 + e1 = E * khi
//      exactly (fma), p2 = RN32(E * klo): a = p1 + e1 + p2 + eta with
//      |eta| <= 2^-46.9 a.  With f0 = floor(p1), fr = RN(RN(p1 - f0) +
//      RN(e1 + p2)):  |2048 (a - f0) - 2048 fr| <= 2^-13 + 2^-34.4 p1.  When
//      2048 fr is at least 2^-12 + 2^-34 p1 away from every integer (a few
//      ulps of margin for the test itself), G = floor(2048 fr) gives
//      floor(a) = f0 + floor(G / 2048), r > 0 and floor(2048 r) = G mod 2048
//      exactly.  The other elements (about 1 in 2000) take the exact integer
//      split afterwards.  Each element becomes one word
//          f << 13 | grant << 12 | (r > 0) << 11 | floor(2048 r)
//      (floors >= 2^19 - 1, at most 32 per row, are kept aside), and a
//      2048-bin histogram of floor(2048 r) is built.
//   E  the bin holding the grant threshold is found on the cluster-wide
//      histogram; counts = f + [bin above it] are written with 128-bit
//      stores; the members of the threshold bin are listed.
// The members (about V / 2048 per row) are then ranked on their exact
// fractions, lowest id first on ties, and the first R - (grants above) get
// their ticket.  The optional draft draw scans the counts still held in
// shared memory in the CTA whose range holds the draw.
#include "common.cuh"

namespace dspark {
namespace {

constexpr int kCl = 8;                   // CTAs per cluster: one row
constexpr int kThr = 256;                // threads per CTA
constexpr int kWarps = kThr / 32;
constexpr int kBins = 2048;              // fraction buckets, floor(2048 r)
constexpr int kFine = kBins / 64;        // fine bins per coarse bin
constexpr int kCandCap = 64;             // threshold-bin members listed per CTA
constexpr int kUncCap = 128;             // elements left to the exact split per CTA
constexpr int kEscCap = 40;              // floors >= kFMax, at most 32 per row
constexpr int kTma = 4;                  // bulk copies (and mbarriers) per slice
constexpr uint32_t kFMax = (1u << 19) - 1u;
constexpr uint32_t kEsc = kFMax << 13;   // word of an element whose floor is kept aside
constexpr uint32_t kPos = 1u << 11;      // r > 0
constexpr uint32_t kGrant = 1u << 12;    // member granted its ticket
constexpr uint32_t kLowMask = 0x1FFFu;   // grant | pos | bucket
constexpr uint32_t kNoThr = 0x1FFFu;     // threshold when no ticket is granted

struct __align__(16) Cand {
  uint64_t key;  // exact fraction (FP64 bit pattern)
  int32_t v;     // token id
  int32_t s;     // slice position
};

struct __align__(16) Esc {
  int32_t s;
  uint32_t f;
  uint32_t low;  // grant | pos | bucket, as in a word
  uint32_t pad;
};

// Scalars a CTA publishes to its peers (read remotely field by field).
struct __align__(16) Pub {
  float mx;         // max of the raw logits (NaN-propagating)
  uint32_t flags1;  // after pass A: bit2 timeout
  uint32_t F;       // sum of floors
  uint32_t csum;    // sum of the counts written before member grants
  uint64_t S;       // sum of E
  uint64_t kmin, kmax;
  uint32_t ncand;   // members of the threshold bin
  uint32_t n_eq;    // id-order rank exchange
  uint32_t n_grant; // granted members (many-member path)
  uint32_t flags2;  // after pass B: bit0 a finite logit overflowed to -inf
  uint32_t flags3;  // after pass C: bit1 internal (escape list full)
  uint32_t pad;
  uint32_t coarse[64];
};

struct DShared {
  union {
    uint32_t hist[kBins];
    Cand all[kBins * 4 / (int)sizeof(Cand)];  // every member of the row (512)
  };
  Cand cand[kCandCap];
  int32_t unc[kUncCap];
  Esc esc[kEscCap];
  Pub pub;
  uint64_t mbar[kTma];
  uint64_t wred64[kWarps];
  uint32_t wred32[kWarps];
  uint32_t wred32b[kWarps];
  float wredf[kWarps];
  uint32_t peers_csum[kCl];
  uint32_t peers_ncand[kCl];
  uint32_t grants[kCl];
  uint32_t gco[64];
  uint32_t gfi[64];
  uint64_t mk;
  uint64_t gmin, gmax;
  int ek;
  float khi, klo;
  float m, invT;
  int bad_T, timeout, status;
  uint32_t n_cand, n_unc, n_esc;
  uint32_t R, Rin, thr, total, fits;
  int sel_bin;
  uint32_t sel_above, sel_count, scan_base;
};
constexpr int kAllCap = kBins * 4 / (int)sizeof(Cand);

struct Params {
  const void* x;
  int dtype;
  int64_t ld;
  int n_rows;
  int V;
  const float* temperature;
  uint32_t* counts;
  int32_t* status;
  int chunk;  // elements per CTA, multiple of 4
  int32_t* tokens;  // optional fused draw (nullptr: none)
  uint64_t seed;
  const uint32_t* request_ids;
  int depth;
};

__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

struct OpMaxNaN {
  __device__ float operator()(float a, float b) const { return fmax_nan(a, b); }
};

// Warp w's value -> one value for the block, in warp 0 (lane 0 holds it).
// The caller issues the __syncthreads between the writes and the reads.
template <typename T, typename Op>
__device__ __forceinline__ T warp0_combine(const T* part, T ident, Op op) {
  const int lane = threadIdx.x & 31;
  return warp_reduce(lane < kWarps ? part[lane] : ident, op);
}

// Exact split of a = RN64(E * k) for one element: word (or escape entry),
// floor, histogram.  Used for the elements the float test leaves open.
__device__ __forceinline__ uint32_t exact_word(float Ef, uint64_t mk, int ek, DShared& sh, int s,
                                               uint32_t* F, uint32_t* internal) {
  uint32_t Ei;
  int se;
  weight_split_ef(Ef, &Ei, &se);
  const AllocSplit a = alloc_split(Ei, se, mk, ek);
  const bool pos = a.rnum != 0ull;
  const int sh11 = a.t - 11;
  const uint32_t b = (!pos || sh11 >= 64) ? 0u : (uint32_t)(a.rnum >> sh11);
  *F += a.f;
  if (pos) atomicAdd(&sh.hist[b], 1u);
  const uint32_t low = (pos ? kPos : 0u) | b;
  if (a.f < kFMax) return (a.f << 13) | low;
  const uint32_t q = atomicAdd(&sh.n_esc, 1u);
  if (q < (uint32_t)kEscCap) {
    sh.esc[q].s = s;
    sh.esc[q].f = a.f;
    sh.esc[q].low = low;
  } else {
    *internal = 1u;
  }
  return kEsc;
}

__device__ __forceinline__ int esc_find(const DShared& sh, int s) {
  const uint32_t ne = min(sh.n_esc, (uint32_t)kEscCap);
  for (uint32_t j = 0; j < ne; ++j)
    if (sh.esc[j].s == s) return (int)j;
  return -1;
}

// Count of slice position s once the grants are settled.
__device__ __forceinline__ uint32_t count_of(const DShared& sh, const uint32_t* slu, int s,
                                             uint32_t thr) {
  const uint32_t w = slu[s];
  if (w != kEsc) return (w >> 13) + (((w & kLowMask) > thr) ? 1u : 0u);
  const int j = esc_find(sh, s);
  return j < 0 ? 0u : sh.esc[j].f + ((sh.esc[j].low > thr) ? 1u : 0u);
}

// Warp 0: the bin b in g[0..63] where the count accumulated from bin 63 down
// reaches `need` (bin 0 if it never does); *above = the count above b.
__device__ __forceinline__ void warp_select64(const uint32_t* g, uint32_t need, int* bin,
                                              uint32_t* above) {
  const int lane = threadIdx.x & 31;
  const uint32_t g0 = g[2 * lane], g1 = g[2 * lane + 1];
  const uint32_t pair = g0 + g1;
  uint32_t suf = pair;  // sum over lanes >= lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += t;
  }
  const uint32_t ab1 = suf - pair;
  const uint32_t ab0 = ab1 + g1;
  const bool hit1 = ab1 < need && need <= ab1 + g1;
  const bool hit0 = ab0 < need && need <= ab0 + g0;
  const unsigned m1 = __ballot_sync(0xffffffffu, hit1);
  const unsigned m0 = __ballot_sync(0xffffffffu, hit0);
  const uint32_t total = __shfl_sync(0xffffffffu, suf, 0);
  if (m1) {
    const int l = __ffs(m1) - 1;
    *bin = 2 * l + 1;
    *above = __shfl_sync(0xffffffffu, ab1, l);
  } else if (m0) {
    const int l = __ffs(m0) - 1;
    *bin = 2 * l;
    *above = __shfl_sync(0xffffffffu, ab0, l);
  } else {
    *bin = 0;
    *above = total - __shfl_sync(0xffffffffu, g0, 0);
  }
}

// After a cluster barrier that published hist and pub.coarse (nbins bins,
// 64 coarse bins of nbins / 64): the bin where the cluster-wide count from
// the top bin down reaches `need` (1 <= need <= total).  Warp 0 works, the
// block waits; sel_bin / sel_above / sel_count are identical in every CTA.
__device__ void select_cluster(cg::cluster_group& cluster, DShared& sh, int nbins,
                               uint32_t need) {
  const int per = nbins / 64;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 64) {
    uint32_t g = 0;
#pragma unroll
    for (int r = 0; r < kCl; ++r) g += *cluster.map_shared_rank(&sh.pub.coarse[threadIdx.x], r);
    sh.gco[threadIdx.x] = g;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    int sb;
    uint32_t above;
    warp_select64(sh.gco, need, &sb, &above);
    for (int i = lane; i < 64; i += 32) {
      uint32_t g = 0;
      if (i < per)
#pragma unroll
        for (int r = 0; r < kCl; ++r) g += cluster.map_shared_rank(&sh.hist[0], r)[sb * per + i];
      sh.gfi[i] = g;
    }
    __syncwarp();
    int b;
    uint32_t ab2;
    warp_select64(sh.gfi, need - above, &b, &ab2);
    if (lane == 0) {
      sh.sel_bin = sb * per + b;
      sh.sel_above = above + ab2;
      sh.sel_count = sh.gfi[b];
    }
  }
  __syncthreads();
}

// Rank, in id order over the whole cluster, of every slice position s with
// pred(s); calls fn(s, rank).  One cluster barrier.
template <typename Pred, typename Fn>
__device__ void ordered_ranks(cg::cluster_group& cluster, DShared& sh, int ngroups, Pred pred,
                              Fn fn) {
  uint32_t cnt = 0;
  for (int g = threadIdx.x; g < ngroups; g += kThr)
    for (int i = 0; i < 4; ++i) cnt += pred(4 * g + i) ? 1u : 0u;
  cnt = block_reduce(cnt, OpAddU32(), sh.wred32);
  if (threadIdx.x == 0) sh.pub.n_eq = cnt;
  cluster.sync();
  if (threadIdx.x == 0) {
    uint32_t base = 0;
    const int me = (int)cluster.block_rank();
    for (int r = 0; r < me; ++r) base += *cluster.map_shared_rank(&sh.pub.n_eq, r);
    sh.scan_base = base;
  }
  __syncthreads();
  uint32_t base = sh.scan_base;
  for (int t0 = 0; t0 < ngroups; t0 += kThr) {
    const int g = t0 + threadIdx.x;
    uint32_t mine = 0;
    bool hit[4] = {false, false, false, false};
    if (g < ngroups)
      for (int i = 0; i < 4; ++i) {
        hit[i] = pred(4 * g + i);
        mine += hit[i] ? 1u : 0u;
      }
    uint32_t total;
    const uint32_t incl = block_inclusive_scan(mine, sh.wred32, &total);
    uint32_t rank = base + incl - mine;
    for (int i = 0; i < 4; ++i)
      if (hit[i]) fn(4 * g + i, rank++);
    base += total;
    __syncthreads();
  }
}

__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kThr, 3)
    q_dense_kernel(Params p) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ DShared sh;
  extern __shared__ __align__(128) float sl[];
  uint32_t* slu = reinterpret_cast<uint32_t*>(sl);

  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.x / kCl;
  const int V = p.V;
  const int lo = rank * p.chunk;
  const int hi = min(V, lo + p.chunk);
  const int n = max(0, hi - lo);
  const int esz = (p.dtype == DSPARK_F32) ? 4 : 2;
  const char* xrow = reinterpret_cast<const char*>(p.x) + (int64_t)row * p.ld * esz;
  // offset of element lo inside its 4-element group of the source row
  const int off = (int)((reinterpret_cast<uintptr_t>(xrow + (int64_t)lo * esz) / esz) & 3);
  const int ngroups = (off + n + 3) >> 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* crow = p.counts + (int64_t)row * V;

  // ---- temperature, barriers, slice
  const bool use_tma_dtype = (p.dtype == DSPARK_F32);
  const int g_first = (off == 0) ? 0 : 1;
  const int g_last = (off + n) / 4 - 1;  // last group fully inside the slice
  const int n_int = max(0, g_last - g_first + 1);
  if (tid == 0) {
    const float T = p.temperature ? p.temperature[row] : 1.0f;
    const float iT = __frcp_rn(T);
    sh.invT = iT;
    sh.bad_T = (!(isfinite(T) && T > 0.0f) || !(isfinite(iT) && iT >= 0x1p-126f)) ? 1 : 0;
    sh.n_cand = 0;
    sh.n_unc = 0;
    sh.n_esc = 0;
    sh.timeout = 0;
    if (use_tma_dtype && n_int > 0) {
      for (int c = 0; c < kTma; ++c) mbar_init(&sh.mbar[c], 1);
      mbar_init_fence();
    }
  }
  __syncthreads();
  const float invT = sh.invT;
  const bool bad_T = sh.bad_T != 0;
  const bool scale = (invT != 1.0f);
  const bool use_tma = use_tma_dtype && n_int > 0;
  const float* xbase = reinterpret_cast<const float*>(xrow) + lo - off;  // group 0 start
  int chunk_lo[kTma + 1];
#pragma unroll
  for (int c = 0; c <= kTma; ++c) chunk_lo[c] = g_first + (n_int * c) / kTma;
  if (use_tma && tid == 0) {
    // issued even for a bad temperature, so that no copy is left pending
    for (int c = 0; c < kTma; ++c) {
      const int g0 = chunk_lo[c], g1 = chunk_lo[c + 1];
      const uint32_t bytes = (uint32_t)(g1 - g0) * 16u;
      mbar_arrive_expect_tx(&sh.mbar[c], bytes);
      if (bytes) tma_load_bulk(sl + 4 * g0, xbase + 4 * g0, bytes, &sh.mbar[c]);
    }
  }
  if (use_tma_dtype) {
    // partial edge groups by plain loads, -inf padding
    if (tid < 8) {
      const int g = (tid < 4) ? 0 : ngroups - 1;
      if (g >= 0 && !(n_int > 0 && g >= g_first && g <= g_last)) {
        const int s = 4 * g + (tid & 3);
        sl[s] = (s >= off && s < off + n) ? __ldg(xbase + s) : -INFINITY;
      }
    }
  } else {
    for (int g = tid; g < ngroups; g += kThr)
      for (int i = 0; i < 4; ++i) {
        const int s = 4 * g + i;
        sl[s] = (s >= off && s < off + n) ? load_logit(xrow, p.dtype, (int64_t)(lo - off + s))
                                          : -INFINITY;
      }
  }
  __syncthreads();

  // ---- pass A: NaN-propagating max of the raw logits
  float mx = -INFINITY;
  for (int c = 0; c < kTma; ++c) {
    int g0 = use_tma ? chunk_lo[c] : (c == 0 ? 0 : ngroups);
    int g1 = use_tma ? chunk_lo[c + 1] : ngroups;
    if (c == 0) g0 = 0;                 // the head edge group
    if (c == kTma - 1) g1 = ngroups;    // the tail edge group
    if (use_tma) {
      if (tid == 0 && !mbar_wait_bounded(&sh.mbar[c], 0)) sh.timeout = 1;
      __syncthreads();
    }
    for (int g = g0 + tid; g < g1; g += kThr) {
      const float4 v = reinterpret_cast<const float4*>(sl)[g];
      mx = fmax_nan(mx, fmax_nan(fmax_nan(v.x, v.y), fmax_nan(v.z, v.w)));
    }
  }
  mx = warp_reduce(mx, OpMaxNaN());
  if (lane == 0) sh.wredf[warp] = mx;
  __syncthreads();
  if (warp == 0) {
    const float m2 = warp0_combine(sh.wredf, -INFINITY, OpMaxNaN());
    if (lane == 0) {
      sh.pub.mx = m2;
      sh.pub.flags1 = sh.timeout ? 4u : 0u;
    }
  }
  cluster.sync();  // S1
  if (warp == 0) {
    float mm = -INFINITY;
    uint32_t fl = 0;
    if (lane < kCl) {
      mm = *cluster.map_shared_rank(&sh.pub.mx, lane);
      fl = *cluster.map_shared_rank(&sh.pub.flags1, lane);
    }
    mm = warp_reduce(mm, OpMaxNaN());
    fl = warp_reduce(fl, OpOrU32());
    if (lane == 0) {
      int st = DSPARK_ST_OK;
      float m = mm;
      if (scale) m = __fmul_rn(mm, invT);
      if (bad_T) st = DSPARK_ST_BAD_TEMPERATURE;
      else if (fl & 4u) st = DSPARK_ST_TIMEOUT;
      else if (!(mm < INFINITY)) st = DSPARK_ST_NONFINITE;   // NaN or +inf
      else if (mm == -INFINITY) st = DSPARK_ST_ZERO_MASS;     // every logit -inf
      else if (!(m > -INFINITY && m < INFINITY)) st = DSPARK_ST_NONFINITE;  // overflow
      sh.status = st;
      sh.m = m;
    }
  }
  __syncthreads();
  if (sh.status != DSPARK_ST_OK) {
    const int st = sh.status;
    for (int v = lo + tid; v < hi; v += kThr) crow[v] = 0u;
    if (rank == 0 && tid == 0) {
      p.status[row] = st;
      if (p.tokens) p.tokens[row] = -1;
    }
    cluster.sync();  // peers may still read this CTA's pub
    return;
  }
  const float m = sh.m;

  // ---- pass B: E = floor(exp_ds(y - m) * 2^40) in place, S = sum E
  uint64_t S = 0;
  uint32_t ovf = 0;
  if (scale) {
    for (int g = tid; g < ngroups; g += kThr) {
      const float4 x4 = reinterpret_cast<const float4*>(sl)[g];
      const float xx[4] = {x4.x, x4.y, x4.z, x4.w};
      float ee[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float y = __fmul_rn(xx[i], invT);
        // a finite logit whose scaled value overflows to -inf refuses the row
        ovf |= (y == -INFINITY && xx[i] != -INFINITY) ? 1u : 0u;
        ee[i] = weight40(__fsub_rn(y, m));
        S += __float2ull_rz(ee[i]);
      }
      reinterpret_cast<float4*>(sl)[g] = make_float4(ee[0], ee[1], ee[2], ee[3]);
    }
  } else {
#pragma unroll 2
    for (int g = tid; g < ngroups; g += kThr) {
      const float4 x4 = reinterpret_cast<const float4*>(sl)[g];
      const float e0 = weight40(__fsub_rn(x4.x, m));
      const float e1 = weight40(__fsub_rn(x4.y, m));
      const float e2 = weight40(__fsub_rn(x4.z, m));
      const float e3 = weight40(__fsub_rn(x4.w, m));
      S += __float2ull_rz(e0) + __float2ull_rz(e1) + __float2ull_rz(e2) + __float2ull_rz(e3);
      reinterpret_cast<float4*>(sl)[g] = make_float4(e0, e1, e2, e3);
    }
  }
  for (int i = tid; i < kBins; i += kThr) sh.hist[i] = 0u;
  S = warp_reduce(S, OpAddU64());
  ovf = warp_reduce(ovf, OpOrU32());
  if (lane == 0) {
    sh.wred64[warp] = S;
    sh.wred32[warp] = ovf;
  }
  __syncthreads();
  if (warp == 0) {
    const uint64_t s2 = warp0_combine(sh.wred64, (uint64_t)0, OpAddU64());
    const uint32_t o2 = warp0_combine(sh.wred32, 0u, OpOrU32());
    if (lane == 0) {
      sh.pub.S = s2;
      sh.pub.flags2 = o2;
    }
  }
  cluster.sync();  // S2
  if (warp == 0) {
    uint64_t sv = 0;
    uint32_t fl = 0;
    if (lane < kCl) {
      sv = *cluster.map_shared_rank(&sh.pub.S, lane);
      fl = *cluster.map_shared_rank(&sh.pub.flags2, lane);
    }
    sv = warp_reduce(sv, OpAddU64());
    fl = warp_reduce(fl, OpOrU32());
    if (lane == 0) {
      const double kd = __ddiv_rn(16777216.0, __ull2double_rn(sv));
      const uint64_t kbits = (uint64_t)__double_as_longlong(kd);
      sh.mk = (kbits & ((1ull << 52) - 1ull)) | (1ull << 52);
      sh.ek = (int)((kbits >> 52) & 0x7FF) - 1075;
      const float khi = __double2float_rn(kd);
      sh.khi = khi;
      sh.klo = __double2float_rn(__dsub_rn(kd, (double)khi));
      sh.status = (fl & 1u) ? DSPARK_ST_NONFINITE : DSPARK_ST_OK;
    }
  }
  __syncthreads();
  if (sh.status != DSPARK_ST_OK) {
    const int st = sh.status;
    for (int v = lo + tid; v < hi; v += kThr) crow[v] = 0u;
    if (rank == 0 && tid == 0) {
      p.status[row] = st;
      if (p.tokens) p.tokens[row] = -1;
    }
    cluster.sync();
    return;
  }
  const uint64_t mk = sh.mk;
  const int ek = sh.ek;
  const float khi = sh.khi, klo = sh.klo;

  // ---- pass C: words and fraction histogram
  uint32_t F = 0, internal = 0;
  // the trip count is the same for every thread (warp votes inside)
  for (int gb = 0; gb < ngroups; gb += kThr) {
    const int g = gb + tid;
    const bool valid = g < ngroups;
    const float4 e4 = valid ? reinterpret_cast<const float4*>(sl)[g] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float ee[4] = {e4.x, e4.y, e4.z, e4.w};
    uint32_t w[4];
    bool open[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float Ef = ee[i];
      const float p1 = __fmul_rn(Ef, khi);
      const float e1 = __fmaf_rn(Ef, khi, -p1);
      const float p2 = __fmul_rn(Ef, klo);
      const float f0 = floorf(p1);
      const float fr = __fadd_rn(__fsub_rn(p1, f0), __fadd_rn(e1, p2));
      const float fb = __fmul_rn(fr, 2048.0f);
      const float G = floorf(fb);
      const float h = __fmaf_rn(p1, -0x1p-34f, 0.5f - 0x1p-12f);
      const bool cert = fabsf(__fsub_rn(__fsub_rn(fb, G), 0.5f)) < h &&
                        f0 < (float)(kFMax - 2u);
      // f0 and G as integers (both below 2^22 in magnitude here)
      const int f0i = __float_as_int(__fadd_rn(f0, 12582912.0f)) - 0x4B400000;
      const int Gi = __float_as_int(__fadd_rn(G, 12582912.0f)) - 0x4B400000;
      const uint32_t f = (uint32_t)(f0i + (Gi >> 11));
      const uint32_t b = (uint32_t)Gi & (kBins - 1u);
      const bool zero = (Ef == 0.0f);
      open[i] = !(cert || zero);
      w[i] = zero ? 0u : ((f << 13) | kPos | b);
      if (cert && !zero) {
        F += f;
        atomicAdd(&sh.hist[b], 1u);
      }
    }
    const bool any_open = open[0] || open[1] || open[2] || open[3];
    if (__any_sync(0xffffffffu, any_open)) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (open[i]) {
          const uint32_t j = atomicAdd(&sh.n_unc, 1u);
          if (j < (uint32_t)kUncCap) {
            sh.unc[j] = 4 * g + i;
            w[i] = __float_as_uint(ee[i]);  // E kept for the exact split
          } else {
            w[i] = exact_word(ee[i], mk, ek, sh, 4 * g + i, &F, &internal);
          }
        }
    }
    if (valid) reinterpret_cast<uint4*>(slu)[g] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __syncthreads();
  {
    const uint32_t nu = min(sh.n_unc, (uint32_t)kUncCap);
    for (uint32_t j = tid; j < nu; j += kThr) {
      const int s = sh.unc[j];
      slu[s] = exact_word(__uint_as_float(slu[s]), mk, ek, sh, s, &F, &internal);
    }
  }
  F = warp_reduce(F, OpAddU32());
  internal = warp_reduce(internal, OpOrU32());
  if (lane == 0) {
    sh.wred32[warp] = F;
    sh.wred32b[warp] = internal;
  }
  __syncthreads();
  // coarse histogram: warp w sums coarse bins 8w .. 8w+7
#pragma unroll
  for (int c = 0; c < 64 / kWarps; ++c) {
    const int cb = warp * (64 / kWarps) + c;
    const uint32_t s = warp_reduce(sh.hist[cb * kFine + lane], OpAddU32());
    if (lane == 0) sh.pub.coarse[cb] = s;
  }
  if (warp == 0) {
    const uint32_t f2 = warp0_combine(sh.wred32, 0u, OpAddU32());
    const uint32_t i2 = warp0_combine(sh.wred32b, 0u, OpOrU32());
    if (lane == 0) {
      sh.pub.F = f2;
      sh.pub.flags3 = i2 ? 2u : 0u;
    }
  }
  cluster.sync();  // S3
  // combine F, flags and the coarse histogram; find the threshold bin
  if (tid < 64) {
    uint32_t gsum = 0;
#pragma unroll
    for (int r = 0; r < kCl; ++r) gsum += *cluster.map_shared_rank(&sh.pub.coarse[tid], r);
    sh.gco[tid] = gsum;
  }
  if (warp == 2) {
    uint32_t fa = 0, fl = 0;
    if (lane < kCl) {
      fa = *cluster.map_shared_rank(&sh.pub.F, lane);
      fl = *cluster.map_shared_rank(&sh.pub.flags3, lane);
    }
    fa = warp_reduce(fa, OpAddU32());
    fl = warp_reduce(fl, OpOrU32());
    if (lane == 0) {
      sh.wred32[0] = fa;
      sh.wred32b[0] = fl;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t npos = warp_reduce(sh.gco[lane] + sh.gco[lane + 32], OpAddU32());
    const uint32_t Fa = sh.wred32[0], fl = sh.wred32b[0];
    int st = DSPARK_ST_OK;
    if (fl & 2u) st = DSPARK_ST_INTERNAL;
    else if (Fa == 0u || Fa > kM || kM - Fa > npos) st = DSPARK_ST_ALLOC_INCONSISTENT;
    const uint32_t R = (st == DSPARK_ST_OK) ? kM - Fa : 0u;
    int bstar = -1;
    uint32_t Rin = 0;
    if (R > 0) {
      int sb;
      uint32_t above;
      warp_select64(sh.gco, R, &sb, &above);
      for (int i = lane; i < 64; i += 32) {
        uint32_t g = 0;
        if (i < kFine)
#pragma unroll
          for (int r = 0; r < kCl; ++r) g += cluster.map_shared_rank(&sh.hist[0], r)[sb * kFine + i];
        sh.gfi[i] = g;
      }
      __syncwarp();
      int b;
      uint32_t ab2;
      warp_select64(sh.gfi, R - above, &b, &ab2);
      bstar = sb * kFine + b;
      Rin = R - above - ab2;
    }
    if (lane == 0) {
      sh.status = st;
      sh.R = R;
      sh.Rin = Rin;
      sh.thr = (bstar >= 0) ? (kPos | (uint32_t)bstar) : kNoThr;
    }
  }
  __syncthreads();
  int status = sh.status;
  const uint32_t R = sh.R, Rin = sh.Rin, thr = sh.thr;

  // ---- pass E: counts = f + [bin above the threshold bin]; members listed
  uint32_t csum = 0;
  const int offc = (int)((reinterpret_cast<uintptr_t>(crow + lo) / 4) & 3);
  if (status == DSPARK_ST_OK) {
    // the trip count is the same for every thread (warp votes inside)
    for (int gb = 0; gb < ngroups; gb += kThr) {
      const int g = gb + tid;
      const bool valid = g < ngroups;
      const uint4 w4 = valid ? reinterpret_cast<const uint4*>(slu)[g] : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
      uint32_t c[4];
      bool odd = false;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t low = ww[i] & kLowMask;
        c[i] = (ww[i] >> 13) + ((low > thr) ? 1u : 0u);
        odd = odd || low == thr || ww[i] == kEsc;
      }
      if (__any_sync(0xffffffffu, odd)) {
        if (odd)
          for (int i = 0; i < 4; ++i) {
            const int s = 4 * g + i;
            uint32_t low = ww[i] & kLowMask;
            if (ww[i] == kEsc) {
              const int j = esc_find(sh, s);
              low = j < 0 ? 0u : sh.esc[j].low;
              c[i] = j < 0 ? 0u : sh.esc[j].f + ((low > thr) ? 1u : 0u);
            }
            if (low == thr && s >= off && s < off + n) {
              const uint32_t q = atomicAdd(&sh.n_cand, 1u);
              if (q < (uint32_t)kCandCap) {
                sh.cand[q].v = lo - off + s;
                sh.cand[q].s = s;
              }
            }
          }
      }
      const int s0 = 4 * g;
      if (!valid) continue;
      if (s0 >= off && s0 + 3 < off + n) {
        csum += c[0] + c[1] + c[2] + c[3];
        if (offc == off)
          *reinterpret_cast<uint4*>(crow + lo - off + s0) = make_uint4(c[0], c[1], c[2], c[3]);
        else
          for (int i = 0; i < 4; ++i) crow[lo - off + s0 + i] = c[i];
      } else {
        for (int i = 0; i < 4; ++i) {
          const int s = s0 + i;
          if (s < off || s >= off + n) continue;
          csum += c[i];
          crow[lo - off + s] = c[i];
        }
      }
    }
  }
  __syncthreads();
  // exact fractions of the listed members
  auto exact_key = [&](int s) -> uint64_t {
    const float x = load_logit(xrow, p.dtype, (int64_t)(lo - off + s));
    const float y = scale ? __fmul_rn(x, invT) : x;
    uint32_t Ei;
    int se;
    weight_split_ef(weight40(__fsub_rn(y, m)), &Ei, &se);
    return frac_key(alloc_split(Ei, se, mk, ek));
  };
  const uint32_t my_cand = sh.n_cand;
  for (uint32_t j = tid; j < min(my_cand, (uint32_t)kCandCap); j += kThr)
    sh.cand[j].key = exact_key(sh.cand[j].s);
  csum = warp_reduce(csum, OpAddU32());
  if (lane == 0) sh.wred32[warp] = csum;
  __syncthreads();
  if (warp == 0) {
    const uint32_t c2 = warp0_combine(sh.wred32, 0u, OpAddU32());
    if (lane == 0) {
      sh.pub.csum = c2;
      sh.pub.ncand = my_cand;
    }
  }
  cluster.sync();  // S4
  if (warp == 0) {
    uint32_t nc = 0, over = 0;
    if (lane < kCl) {
      const uint32_t cs = *cluster.map_shared_rank(&sh.pub.csum, lane);
      nc = *cluster.map_shared_rank(&sh.pub.ncand, lane);
      sh.peers_csum[lane] = cs;
      sh.peers_ncand[lane] = nc;
      sh.grants[lane] = 0u;
      over = nc > (uint32_t)kCandCap ? 1u : 0u;
    }
    over = warp_reduce(over, OpOrU32());
    const uint32_t tot = warp_reduce(nc, OpAddU32());
    if (lane == 0) {
      sh.total = tot;
      sh.fits = (!over && tot <= (uint32_t)kAllCap) ? 1u : 0u;
    }
  }
  __syncthreads();
  const uint32_t total = sh.total;
  const bool fits = sh.fits != 0u;

  // grant one member: its word (or escape entry) gets the grant bit and its
  // count f + 1 is written
  auto grant_member = [&](int s) {
    const uint32_t w = slu[s];
    uint32_t f;
    if (w == kEsc) {
      const int j = esc_find(sh, s);
      if (j < 0) return;
      sh.esc[j].low |= kGrant;
      f = sh.esc[j].f;
    } else {
      slu[s] = w | kGrant;
      f = w >> 13;
    }
    crow[lo - off + s] = f + 1u;
  };

  if (R > 0 && fits && Rin > 0) {
    // every CTA ranks every member: granted iff fewer than Rin members come
    // before it in (fraction desc, id asc)
    Cand* all = sh.all;
    for (int t = tid; t < (int)total; t += kThr) {
      int r = 0;
      uint32_t base = 0;
      while (r < kCl - 1 && (uint32_t)t >= base + sh.peers_ncand[r]) {
        base += sh.peers_ncand[r];
        ++r;
      }
      const Cand* src = cluster.map_shared_rank(&sh.cand[0], r) + (t - base);
      Cand e;
      e.key = src->key;
      e.v = src->v;
      e.s = src->s;
      all[t] = e;
    }
    __syncthreads();
    // tpm threads per member, each scanning a stride of the list
    int tpm = 32;
    while (tpm > 1 && (int)total * tpm > kThr) tpm >>= 1;
    for (int i0 = 0; i0 < (int)total; i0 += kThr / tpm) {
      const int i = i0 + tid / tpm;
      const int part = tid % tpm;
      uint32_t before = 0;
      uint64_t ki = 0;
      int vi = 0;
      if (i < (int)total) {
        ki = all[i].key;
        vi = all[i].v;
        for (int j = part; j < (int)total; j += tpm) {
          const uint64_t kj = all[j].key;
          before += (kj > ki || (kj == ki && all[j].v < vi)) ? 1u : 0u;
        }
      }
      for (int o = tpm >> 1; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
      if (i < (int)total && part == 0 && before < Rin) {
        const int owner = vi / p.chunk;
        atomicAdd(&sh.grants[owner], 1u);
        if (owner == rank) grant_member(all[i].s);
      }
    }
    __syncthreads();
  } else if (R > 0 && !fits && Rin > 0) {
    // many members: the exact fraction threshold by 8-bit radix levels over
    // the keys (unless they all hold one fraction), then the remaining tickets
    // go to the lowest ids holding the threshold fraction
    auto is_member = [&](int s) -> bool {
      if (s < off || s >= off + n) return false;
      const uint32_t w = slu[s];
      if (w != kEsc) return (w & kLowMask) == thr;
      const int j = esc_find(sh, s);
      return j >= 0 && sh.esc[j].low == thr;
    };
    uint64_t kmin = ~0ull, kmax = 0ull;
    for (int g = tid; g < ngroups; g += kThr)
      for (int i = 0; i < 4; ++i)
        if (is_member(4 * g + i)) {
          const uint64_t key = exact_key(4 * g + i);
          kmin = min(kmin, key);
          kmax = max(kmax, key);
        }
    kmin = block_reduce(kmin, OpMinU64(), sh.wred64);
    kmax = block_reduce(kmax, OpMaxU64(), sh.wred64);
    if (tid == 0) {
      sh.pub.kmin = kmin;
      sh.pub.kmax = kmax;
    }
    cluster.sync();
    if (tid == 0) {
      uint64_t a = ~0ull, b = 0ull;
      for (int r = 0; r < kCl; ++r) {
        a = min(a, *cluster.map_shared_rank(&sh.pub.kmin, r));
        b = max(b, *cluster.map_shared_rank(&sh.pub.kmax, r));
      }
      sh.gmin = a;
      sh.gmax = b;
    }
    __syncthreads();
    const uint64_t gmin = sh.gmin, gmax = sh.gmax;
    const bool one_key = (gmin == gmax);
    uint64_t thrk = gmin, prefix = 0ull;
    uint32_t need = Rin;
    if (!one_key) {
      for (int lvl = 0; lvl < 8; ++lvl) {
        const int sft = 56 - 8 * lvl;
        cluster.sync();  // peers are done reading this CTA's histogram
        for (int i = tid; i < 256; i += kThr) sh.hist[i] = 0u;
        __syncthreads();
        for (int g = tid; g < ngroups; g += kThr)
          for (int i = 0; i < 4; ++i) {
            const int s = 4 * g + i;
            if (!is_member(s)) continue;
            const uint64_t key = exact_key(s);
            if (lvl > 0 && (key >> (sft + 8)) != prefix) continue;
            atomicAdd(&sh.hist[(key >> sft) & 255u], 1u);
          }
        __syncthreads();
        if (tid < 64)
          sh.pub.coarse[tid] = sh.hist[4 * tid] + sh.hist[4 * tid + 1] + sh.hist[4 * tid + 2] +
                               sh.hist[4 * tid + 3];
        cluster.sync();
        select_cluster(cluster, sh, 256, need);
        prefix = (prefix << 8) | (uint64_t)sh.sel_bin;
        need -= sh.sel_above;
      }
      thrk = prefix;
    }
    uint32_t mine = 0;
    if (!one_key)
      for (int g = tid; g < ngroups; g += kThr)
        for (int i = 0; i < 4; ++i) {
          const int s = 4 * g + i;
          if (is_member(s) && exact_key(s) > thrk) {
            grant_member(s);
            ++mine;
          }
        }
    __syncthreads();
    // members granted above are no longer members (their low bits changed)
    ordered_ranks(
        cluster, sh, ngroups,
        [&](int s) -> bool { return is_member(s) && (one_key || exact_key(s) == thrk); },
        [&](int s, uint32_t rk) {
          if (rk < need) {
            grant_member(s);
            ++mine;
          }
        });
    mine = block_reduce(mine, OpAddU32(), sh.wred32);
    if (tid == 0) sh.pub.n_grant = mine;
    cluster.sync();
    if (tid < kCl) sh.grants[tid] = *cluster.map_shared_rank(&sh.pub.n_grant, tid);
    __syncthreads();
  }

  // ---- totals: every CTA's count sum; the row must hold exactly M
  uint32_t cbefore = 0, my_total = 0, all_total = 0;
  for (int r = 0; r < kCl; ++r) {
    const uint32_t cr = sh.peers_csum[r] + sh.grants[r];
    if (r < rank) cbefore += cr;
    if (r == rank) my_total = cr;
    all_total += cr;
  }
  if (status == DSPARK_ST_OK && all_total != kM) status = DSPARK_ST_ALLOC_INCONSISTENT;
  __syncthreads();  // member counts are written before any zeroing below
  if (status != DSPARK_ST_OK)
    for (int v = lo + tid; v < hi; v += kThr) crow[v] = 0u;
  if (rank == 0 && tid == 0) {
    p.status[row] = status;
    if (p.tokens && status != DSPARK_ST_OK) p.tokens[row] = -1;
  }
  // every remote read of this CTA's shared memory is done: arrive now, wait
  // before leaving
  cluster.barrier_arrive();

  // ---- fused draft draw: the CTA whose range holds D scans its counts
  if (p.tokens && status == DSPARK_ST_OK) {
    const int b = row / p.depth, j = row % p.depth;
    const uint32_t req = p.request_ids ? p.request_ids[b] : (uint32_t)b;
    const uint32_t D = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_PROPOSAL) >> 8;
    if (D >= cbefore && D - cbefore < my_total) {
      // one contiguous segment of slice positions per warp
      const int ns = 4 * ngroups;
      const int seg = (ns + kWarps - 1) / kWarps;
      const int a0 = warp * seg, a1 = min(ns, a0 + seg);
      uint32_t ssum = 0;
      for (int s = a0 + lane; s < a1; s += 32) ssum += count_of(sh, slu, s, thr);
      ssum = warp_reduce(ssum, OpAddU32());
      if (lane == 0) sh.wred32[warp] = ssum;
      __syncthreads();
      uint32_t sb = cbefore;
      for (int w2 = 0; w2 < warp; ++w2) sb += sh.wred32[w2];
      if (D >= sb && D - sb < sh.wred32[warp]) {
        uint32_t base = sb;
        for (int s0 = a0; s0 < a1; s0 += 32) {
          const int s = s0 + lane;
          const uint32_t cv = (s < a1) ? count_of(sh, slu, s, thr) : 0u;
          uint32_t incl = cv;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
          }
          const uint32_t tile = __shfl_sync(0xffffffffu, incl, 31);
          if (D - base < tile) {
            const bool hit = cv > 0u && D - base < incl && D - base >= incl - cv;
            const unsigned msk = __ballot_sync(0xffffffffu, hit);
            if (lane == 0 && msk) p.tokens[row] = lo - off + s0 + __ffs(msk) - 1;
            break;
          }
          base += tile;
        }
      }
    }
  }
  cluster.barrier_wait();  // no CTA leaves while a peer may still read its shared memory
}

}  // namespace

int q_dense_smem_bytes(int chunk) { return (chunk + 4) * 4; }

cudaError_t launch_q_dense(const void* x, int dtype, int64_t ld, int n_rows, int V,
                           const float* temperature, uint32_t* counts, int32_t* status,
                           int32_t* tokens, uint64_t seed, const uint32_t* request_ids, int depth,
                           cudaStream_t stream) {
  Params p;
  p.x = x;
  p.dtype = dtype;
  p.ld = ld;
  p.n_rows = n_rows;
  p.V = V;
  p.temperature = temperature;
  p.counts = counts;
  p.status = status;
  int chunk = (V + kCl - 1) / kCl;
  chunk = (chunk + 3) & ~3;
  p.chunk = chunk;
  p.tokens = tokens;
  p.seed = seed;
  p.request_ids = request_ids;
  p.depth = depth > 0 ? depth : 1;
  const int smem = q_dense_smem_bytes(chunk);
  cudaError_t err =
      cudaFuncSetAttribute(q_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(q_dense_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  q_dense_kernel<<<n_rows * kCl, kThr, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dspark
