// q_dense.cuh -- device code of the dense q build (see q_dense.cu), shared by
// the q kernel and the fused speculative-step kernel.
#pragma once
#include "common.cuh"

namespace dspark {
namespace qdense {
namespace {  // device code private to each translation unit that includes it

constexpr int kCl = 8;                   // CTAs per cluster: one row
constexpr int kThr = 256;                // threads per CTA
constexpr int kWarps = kThr / 32;
constexpr int kBins = 2048;              // fraction buckets, floor(2048 r)
constexpr int kFine = kBins / 64;        // fine bins per coarse bin
constexpr int kCandCap = 56;             // threshold-bin members listed per CTA
constexpr int kBlkCap = 130;             // count sums of 32-group blocks (<= 129 per slice)
constexpr int kWin = 3072;               // slice positions compacted per window (many members)
constexpr int kTab = 64;                 // distinct member fractions kept per CTA
constexpr int kEscCap = 40;              // floors >= kFMax, at most 32 per row
constexpr int kTma = 4;                  // bulk copies (and mbarriers) per slice
constexpr uint32_t kFMax = (1u << 19) - 1u;
constexpr uint32_t kEsc = kFMax << 13;   // word of an element whose floor is kept aside
constexpr uint32_t kPos = 1u << 11;      // r > 0
constexpr uint32_t kGrant = 1u << 12;    // member granted its ticket
constexpr uint32_t kLowMask = 0x1FFFu;   // grant | pos | bucket
constexpr uint32_t kNoThr = 0x1FFFu;     // threshold when no ticket is granted
// certification half-width: 2048 fr must lie within this of a half-integer
constexpr float kHalfMargin = 0.5f - 0x1p-12f - 0x1p-15f;

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

// Values a CTA publishes for its peers to read (field by field).
struct __align__(16) Pub {
  uint64_t kmin, kmax;
  uint32_t n_eq;    // id-order rank exchange
  uint32_t n_grant; // granted members (many-member path)
  uint32_t flags4;  // many-member path: bit0 a table of fractions overflowed
  uint32_t pad;
  uint32_t coarse[64];
};

// Scalars every CTA writes into every peer's copy before a cluster barrier
// (slot = the writer's rank), so that after it each CTA reads local memory.
struct __align__(16) Push {
  uint64_t S[kCl];      // sum of E
  float mx[kCl];        // max of the raw logits (NaN-propagating)
  uint32_t fl1[kCl];    // after pass A: bit2 timeout
  uint32_t fl2[kCl];    // after pass B: bit0 a finite logit overflowed to -inf
  uint32_t F[kCl];      // sum of floors
  uint32_t fl3[kCl];    // after pass C: bit1 internal (escape list full)
  uint32_t csum[kCl];   // sum of the counts written before member grants
  uint32_t ncand[kCl];  // members of the threshold bin
  float t1[kCl], t2[kCl];  // Markov chain rows: each CTA's two largest finite z
};

// Many-member path: member positions compacted per window, then the table of
// distinct exact fractions (read by peers), then every peer's table merged.
// steps of 32 slice positions in one warp's segment of the slice, at most
constexpr int kAtSteps = ((DSPARK_MAX_V / kCl + 8) / kWarps + 31) / 32 + 1;

struct ManyShared {
  union {
    uint16_t list[kWin];
    struct {
      uint64_t key[kCl * kTab];
      uint32_t cnt[kCl * kTab];
    } merged;
    uint32_t atm[kWarps * kAtSteps];  // members at the threshold fraction, per step
  };
  uint64_t tkey[kTab];
  uint32_t tcnt[kTab];
  uint8_t state[kTab];  // 0 below the threshold fraction, 1 above, 2 at it
};

struct DShared {
  union {
    uint32_t hist[kBins + 16];  // + dummy bins taking the elements that do not count
    Cand all[kBins * 4 / (int)sizeof(Cand)];  // every member of the row (512)
    ManyShared many;
  };
  Cand cand[kCandCap];
  uint32_t bsum[kBlkCap];  // count sum of each block of 32 groups
  Esc esc[kEscCap];
  Pub pub;
  Push push;
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
  uint32_t n_cand, n_esc;
  uint32_t R, Rin, thr, total, fits;
  uint64_t thrk;
  uint32_t need, fovf;
  uint32_t wcnt[kWarps];
  int sel_bin;
  uint32_t sel_above, sel_count, scan_base;
  uint32_t draw;  // the row's 24-bit draft draw (fused draw only)
  uint32_t n_merged;  // many-member path: non-empty merged table slots
  float top1, top2;   // Markov chain rows: the row's two largest finite z
  int chain_tok;      // Markov chain rows: the drawn token, stored by the drawing CTA
  float wt1[kWarps], wt2[kWarps];
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

// top two of {a1, a2} and {b1, b2} (a1 >= a2, b1 >= b2)
__device__ __forceinline__ void top2_merge(float& a1, float& a2, float b1, float b2) {
  if (b1 > a1) {
    a2 = fmaxf(a1, b2);
    a1 = b1;
  } else {
    a2 = fmaxf(a2, b1);
  }
}

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
__device__ __noinline__ uint32_t exact_word(float Ef, uint64_t mk, int ek, DShared& sh, int s,
                                               uint32_t* F, uint32_t* internal) {
  uint32_t Ei;
  int se;
  weight_split_ef(Ef, &Ei, &se);
  const AllocSplit a = alloc_split(Ei, se, mk, ek);
  const bool pos = a.rnum != 0ull;
  const int sh11 = a.t - 11;
  const uint32_t b = (!pos || sh11 >= 64) ? 0u : (uint32_t)(a.rnum >> sh11);
  *F += a.f;
  if (pos && DSPARK_CHECK(b < (uint32_t)kBins)) atomicAdd(&sh.hist[b], 1u);
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

// The float split of one weight (see the file comment): the word, its floor,
// its bucket, and whether the float result is certified.
struct FloatSplit {
  uint32_t word, f, b;
  bool cert, zero;
};
__device__ __forceinline__ FloatSplit float_split(float Ef, float khi, float klo) {
  FloatSplit o;
  const float p1 = __fmul_rn(Ef, khi);
  const float e1 = __fmaf_rn(Ef, khi, -p1);
  const float p2 = __fmul_rn(Ef, klo);
  const float f0 = floorf(p1);
  const float fr = __fadd_rn(__fsub_rn(p1, f0), __fadd_rn(e1, p2));
  const float fb = __fmul_rn(fr, 2048.0f);
  const float G = floorf(fb);
  o.cert = fabsf(__fsub_rn(__fsub_rn(fb, G), 0.5f)) < kHalfMargin && f0 < (float)(kFMax - 2u);
  // f0 and G as integers (|G| < 2^13 here): f = f0 + floor(G / 2048)
  const int f0i = __float_as_int(__fadd_rn(f0, 12582912.0f)) - 0x4B400000;
  const int Gi = __float_as_int(__fadd_rn(G, 12582912.0f)) - 0x4B400000;
  o.f = (uint32_t)(f0i + (Gi >> 11));
  o.b = (uint32_t)Gi & (kBins - 1u);
  o.zero = (Ef == 0.0f);
  o.word = o.zero ? 0u : ((o.f << 13) | kPos | o.b);
  return o;
}

// float_split of two weights at once on the packed fp32x2 pipe, lane for
// lane bit-identical to float_split: floor(p1) is the rounded-down sum
// p1 + 1.5 * 2^23 (exact for 0 <= p1 < 2^22, and p1 >= 2^22 is never
// certified: the test below is p1 < kFMax - 2, i.e. floor(p1) < kFMax - 2);
// 2048 fr is taken as fma(u, 2048, 2048 RN(e1 + p2)) with u = p1 - floor(p1)
// exact, which equals RN(RN(u + RN(e1 + p2)) * 2048) because scaling by
// 2^11 commutes with rounding (no value here is subnormal); the same
// rounded-down sum gives floor(2048 fr).  klo2k = 2048 * klo (exact).  The
// floor f and the bucket come from the bits of the two sums: bits(t0) =
// 0x4B400000 + floor(p1), bits(tG) = 0x4B400000 + G with G in [-1, 2049],
// and 0x4B400000 is a multiple of 2048.
struct FloatSplit2 {
  uint32_t word[2], f[2], b[2];
  bool cert[2], zero[2];
};
__device__ __forceinline__ FloatSplit2 float_split2(float2 E, float khi, float klo2k) {
  constexpr float kMag = 12582912.0f;  // 1.5 * 2^23
  const float2 K = f2(khi);
  const float2 p1 = mul2_rn(E, K);
  const float2 e1 = fma2_rn(E, K, make_float2(-p1.x, -p1.y));
  const float2 p2s = mul2_rn(E, f2(klo2k));
  const float2 t0 = add2_rm(p1, f2(kMag));
  const float2 f0 = add2_rn(t0, f2(-kMag));
  const float2 u = add2_rn(p1, make_float2(-f0.x, -f0.y));
  const float2 vs = fma2_rn(e1, f2(2048.0f), p2s);
  const float2 fb = fma2_rn(u, f2(2048.0f), vs);
  const float2 tG = add2_rm(fb, f2(kMag));
  const float2 G = add2_rn(tG, f2(-kMag));
  const float2 xh = add2_rn(add2_rn(fb, make_float2(-G.x, -G.y)), f2(-0.5f));
  FloatSplit2 o;
  const float ee[2] = {E.x, E.y}, pp[2] = {p1.x, p1.y}, hh[2] = {xh.x, xh.y};
  const uint32_t bt0[2] = {__float_as_uint(t0.x), __float_as_uint(t0.y)};
  const uint32_t btg[2] = {__float_as_uint(tG.x), __float_as_uint(tG.y)};
#pragma unroll
  for (int l = 0; l < 2; ++l) {
    o.cert[l] = fabsf(hh[l]) < kHalfMargin && pp[l] < (float)(kFMax - 2u);
    o.f[l] = bt0[l] + (btg[l] >> 11) - (0x4B400000u + (0x4B400000u >> 11));
    o.b[l] = btg[l] & (kBins - 1u);
    o.zero[l] = (ee[l] == 0.0f);
    o.word[l] = o.zero[l] ? 0u : ((o.f[l] << 13) | kPos | o.b[l]);
  }
  return o;
}

// Exact sum of the integer weights E (integer floats <= 2^40) without a
// float-to-integer conversion: E = hi * 2^20 + lo with hi = floor(E / 2^20)
// read from the bits of the round-down sum E * 2^-20 + 2^23, and lo = E -
// hi * 2^20 (exact) from the bits of lo + 2^23; the bits are summed as 32-bit
// integers (modulo 2^32, the 2^23 offsets removed at the end: a thread's hi
// and lo sums stay far below 2^32).
struct WeightSum {
  uint32_t hi, lo, n;  // sums of the offset bits, and the number of weights
};
__device__ __forceinline__ void sum_weights2(float2 E, WeightSum& w) {
  const float2 t = fma2_rm(E, f2(0x1p-20f), f2(8388608.0f));
  const float2 l = add2_rn(fma2_rn(add2_rn(t, f2(-8388608.0f)), f2(-1048576.0f), E),
                           f2(8388608.0f));
  w.hi += __float_as_uint(t.x) + __float_as_uint(t.y);
  w.lo += __float_as_uint(l.x) + __float_as_uint(l.y);
  w.n += 2u;
}
__device__ __forceinline__ uint64_t weight_sum_total(const WeightSum& w) {
  return ((uint64_t)(w.hi - w.n * 0x4B000000u) << 20) + (uint64_t)(w.lo - w.n * 0x4B000000u);
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
        for (int r = 0; r < kCl; ++r)
          if (DSPARK_CHECK(sb * per + i < nbins))
            g += cluster.map_shared_rank(&sh.hist[0], r)[sb * per + i];
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

// One draft row on one 8-CTA cluster (every CTA of the cluster calls it with
// the same row).  `mbar` holds kTma initialised mbarriers whose current phase
// parity is `phase` (updated here).  When `ready` is given (a fused launch),
// ready[row / depth] is incremented once the row's counts, status and token
// are visible device-wide.  When next_row >= 0, this CTA's part of that row
// is prefetched into L2 while this row is built (the same cluster takes it
// next, so its bulk copies then read L2).  A Markov chain row (chain true)
// builds z = RN(x + bias) with the bias row zbias (fp32, element v at
// zbias[v]; z = x when zbias is null), formed in shared memory as the slice
// lands, and sh.top1 / sh.top2 get the row's two largest finite z; its
// drawn token reaches every CTA's sh.chain_tok.  Returns the row's status,
// the same in every CTA of the cluster.
__device__ __forceinline__ int q_dense_row(const Params& p, int row, DShared& sh, float* sl,
                                           uint64_t* mbar, uint32_t& phase, uint32_t* ready,
                                           int next_row = -1, bool chain = false,
                                           const float* zbias = nullptr) {
  cg::cluster_group cluster = cg::this_cluster();
  uint32_t* slu = reinterpret_cast<uint32_t*>(sl);

  const int rank = (int)cluster.block_rank();
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
  const int slice_cap = p.chunk + 4;  // floats of the slice buffer
  // this CTA's count position s of the row (checked build: inside [lo, hi))
  auto in_row = [&](int s) -> bool { return DSPARK_CHECK(lo - off + s >= lo && lo - off + s < hi); };

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
    sh.n_esc = 0;
    sh.timeout = 0;
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
    // the buffer's earlier generic-proxy writes (a previous item of a fused
    // launch) are ordered before the bulk copies into it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    // issued even for a bad temperature, so that no copy is left pending
    for (int c = 0; c < kTma; ++c) {
      const int g0 = chunk_lo[c], g1 = chunk_lo[c + 1];
      const uint32_t bytes = (uint32_t)(g1 - g0) * 16u;
      mbar_arrive_expect_tx(&mbar[c], bytes);
      if (bytes) tma_load_bulk(sl + 4 * g0, xbase + 4 * g0, bytes, &mbar[c]);
    }
  }
  if (zbias && tid == 64) {
    // a chain row's bias part, into L2 for the loads of chunks 1 .. kTma-1
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(zbias + lo) + 15u) & ~(uintptr_t)15u;
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(zbias + hi) & ~(uintptr_t)15u;
    if (a1 > a0) l2_prefetch_bulk(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
  }
  if (tid == 32 && p.tokens) {
    // the draft draw, while the slice lands
    const int b = row / p.depth, j = row % p.depth;
    const uint32_t req = p.request_ids ? p.request_ids[b] : (uint32_t)b;
    sh.draw = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_PROPOSAL) >> 8;
  }
  if (use_tma_dtype) {
    // partial edge groups by plain loads, -inf padding
    if (tid < 8) {
      const int g = (tid < 4) ? 0 : ngroups - 1;
      if (g >= 0 && !(n_int > 0 && g >= g_first && g <= g_last)) {
        const int s = 4 * g + (tid & 3);
        if (DSPARK_CHECK(s < slice_cap))
          sl[s] = (s >= off && s < off + n) ? __ldg(xbase + s) : -INFINITY;
      }
    }
  } else {
    for (int g = tid; g < ngroups; g += kThr)
      for (int i = 0; i < 4; ++i) {
        const int s = 4 * g + i;
        if (DSPARK_CHECK(s < slice_cap))
          sl[s] = (s >= off && s < off + n) ? load_logit(xrow, p.dtype, (int64_t)(lo - off + s))
                                            : -INFINITY;
      }
  }
  __syncthreads();

  // ---- pass A: NaN-propagating max of the raw logits (of z for a chain row)
  float mx = -INFINITY;
  float zt1 = -INFINITY, zt2 = -INFINITY;  // chain rows: the thread's two largest finite z
  // chain rows: the bias values of a group (0 outside the slice), by one
  // 128-bit load when the bias row is aligned like the slice's groups
  const bool bvec = zbias && ((reinterpret_cast<uintptr_t>(zbias + (lo - off)) & 15u) == 0u);
  auto bias4 = [&](int g) -> float4 {
    if (bvec && g >= g_first && g <= g_last)
      return __ldg(reinterpret_cast<const float4*>(zbias + (lo - off)) + g);
    float b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int s = 4 * g + i;
      b[i] = (s >= off && s < off + n) ? __ldg(zbias + (lo - off + s)) : 0.0f;
    }
    return make_float4(b[0], b[1], b[2], b[3]);
  };
  constexpr int kBPre = 4;  // groups of a chunk per thread whose bias is loaded together
  for (int c = 0; c < kTma; ++c) {
    int g0 = use_tma ? chunk_lo[c] : (c == 0 ? 0 : ngroups);
    int g1 = use_tma ? chunk_lo[c + 1] : ngroups;
    if (c == 0) g0 = 0;                 // the head edge group
    if (c == kTma - 1) g1 = ngroups;    // the tail edge group
    if (use_tma) {
      if (tid == 0 && !mbar_wait_bounded(&mbar[c], phase)) sh.timeout = 1;
      __syncthreads();
    }
    // chain rows: the chunk's bias values, loaded together once the chunk
    // has landed (from L2: the row's bias part was prefetched at its start).
    // Loading them before the wait, or a chunk ahead, measured slower.
    float4 bpre[kBPre];
    if (zbias) {
#pragma unroll
      for (int k = 0; k < kBPre; ++k) {
        const int g = g0 + tid + k * kThr;
        bpre[k] = (g < g1) ? bias4(g) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
    if (!chain) {
      for (int g = g0 + tid; g < g1; g += kThr) {
        const float4 v = reinterpret_cast<const float4*>(sl)[g];
        mx = fmax_nan(mx, fmax_nan(fmax_nan(v.x, v.y), fmax_nan(v.z, v.w)));
      }
    } else {
      // z = RN(x + bias) in place (the -inf padding of the edge groups stays)
      int k = 0;
      for (int g = g0 + tid; g < g1; g += kThr, ++k) {
        const float4 v = reinterpret_cast<const float4*>(sl)[g];
        float z[4] = {v.x, v.y, v.z, v.w};
        if (zbias) {
          float4 b4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
          for (int kk = 0; kk < kBPre; ++kk)
            if (kk == k) b4 = bpre[kk];
          if (k >= kBPre) b4 = bias4(g);
          const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int s = 4 * g + i;
            if (s >= off && s < off + n) z[i] = __fadd_rn(z[i], bb[i]);
          }
          reinterpret_cast<float4*>(sl)[g] = make_float4(z[0], z[1], z[2], z[3]);
        }
        // the two largest z (with multiplicity); a row holding +inf or NaN
        // is refused, and -inf changes neither
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          mx = fmax_nan(mx, z[i]);
          zt2 = fmaxf(zt2, fminf(zt1, z[i]));
          zt1 = fmaxf(zt1, z[i]);
        }
      }
    }
  }
  if (use_tma) phase ^= 1u;
  mx = warp_reduce(mx, OpMaxNaN());
  if (lane == 0) sh.wredf[warp] = mx;
  if (chain) {
    // the CTA's two largest finite z (warp 0 of the block, then pushed)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float o1 = __shfl_xor_sync(0xffffffffu, zt1, o);
      const float o2 = __shfl_xor_sync(0xffffffffu, zt2, o);
      top2_merge(zt1, zt2, o1, o2);
    }
    if (lane == 0) {
      sh.wt1[warp] = zt1;
      sh.wt2[warp] = zt2;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const float m2 = warp0_combine(sh.wredf, -INFINITY, OpMaxNaN());
    float c1 = -INFINITY, c2 = -INFINITY;
    if (chain) {
      for (int w = 0; w < kWarps; ++w) top2_merge(c1, c2, sh.wt1[w], sh.wt2[w]);
    }
    if (lane < kCl) {
      *cluster.map_shared_rank(&sh.push.mx[rank], lane) = m2;
      *cluster.map_shared_rank(&sh.push.fl1[rank], lane) = sh.timeout ? 4u : 0u;
      if (chain) {
        *cluster.map_shared_rank(&sh.push.t1[rank], lane) = c1;
        *cluster.map_shared_rank(&sh.push.t2[rank], lane) = c2;
      }
    }
  }
  cluster.sync();  // S1
  // every thread of this CTA has read the previous row's token by now, and
  // no peer stores this row's before S4
  if (chain && tid == 64) sh.chain_tok = -1;
  if (chain && warp == 1 && lane == 0) {
    float c1 = -INFINITY, c2 = -INFINITY;
    for (int r = 0; r < kCl; ++r) top2_merge(c1, c2, sh.push.t1[r], sh.push.t2[r]);
    sh.top1 = c1;
    sh.top2 = c2;
  }
  // the cluster's values by one lane straight from shared memory: warp
  // shuffles and reductions queue behind the other CTAs' shared-memory
  // traffic here, and these few lines hold the whole CTA
  if (warp == 0 && lane == 0) {
    float mm = -INFINITY;
    uint32_t fl = 0;
    for (int r = 0; r < kCl; ++r) {
      mm = fmax_nan(mm, sh.push.mx[r]);
      fl |= sh.push.fl1[r];
    }
    {
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
    if (rank == 0 && tid == 0 && DSPARK_CHECK(row < p.n_rows)) {
      p.status[row] = st;
      if (p.tokens) p.tokens[row] = -1;
    }
    cluster.sync();  // peers may still read this CTA's pub
    if (ready && rank == 0 && tid == 0 && DSPARK_CHECK(row / p.depth < (p.n_rows + p.depth - 1) / p.depth)) {
      __threadfence();
      atomicAdd(&ready[row / p.depth], 1u);
    }
    return st;
  }
  const float m = sh.m;
  if (next_row >= 0 && use_tma_dtype && tid == 0) {
    // this CTA's aligned part of the next row, into L2
    const char* nrow = reinterpret_cast<const char*>(p.x) + (int64_t)next_row * p.ld * 4;
    const uintptr_t a0 = (reinterpret_cast<uintptr_t>(nrow + (int64_t)lo * 4) + 15u) & ~(uintptr_t)15u;
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(nrow + (int64_t)hi * 4) & ~(uintptr_t)15u;
    if (a1 > a0) l2_prefetch_bulk(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
  }

  // ---- pass B: E = floor(exp_ds(y - m) * 2^40) in place, S = sum E
  //      (pairs of elements on the packed fp32x2 pipe)
  WeightSum sw = {0u, 0u, 0u};
  uint32_t ovf = 0;
  const float2 mneg = f2(-m);
  if (scale) {
    const float2 iT2 = f2(invT);
    for (int g = tid; g < ngroups; g += kThr) {
      const float4 x4 = reinterpret_cast<const float4*>(sl)[g];
      const float2 ya = mul2_rn(make_float2(x4.x, x4.y), iT2);
      const float2 yb = mul2_rn(make_float2(x4.z, x4.w), iT2);
      // a finite logit whose scaled value overflows to -inf refuses the row
      ovf |= ((ya.x == -INFINITY && x4.x != -INFINITY) || (ya.y == -INFINITY && x4.y != -INFINITY) ||
              (yb.x == -INFINITY && x4.z != -INFINITY) || (yb.y == -INFINITY && x4.w != -INFINITY))
                 ? 1u : 0u;
      const float2 ea = weight40x2(add2_rn(ya, mneg));
      const float2 eb = weight40x2(add2_rn(yb, mneg));
      sum_weights2(ea, sw);
      sum_weights2(eb, sw);
      reinterpret_cast<float4*>(sl)[g] = make_float4(ea.x, ea.y, eb.x, eb.y);
    }
  } else {
#pragma unroll 2
    for (int g = tid; g < ngroups; g += kThr) {
      const float4 x4 = reinterpret_cast<const float4*>(sl)[g];
      const float2 ea = weight40x2(add2_rn(make_float2(x4.x, x4.y), mneg));
      const float2 eb = weight40x2(add2_rn(make_float2(x4.z, x4.w), mneg));
      sum_weights2(ea, sw);
      sum_weights2(eb, sw);
      reinterpret_cast<float4*>(sl)[g] = make_float4(ea.x, ea.y, eb.x, eb.y);
    }
  }
  uint64_t S = weight_sum_total(sw);
  for (int i = tid; i < kBins + 16; i += kThr) sh.hist[i] = 0u;
  S = warp_reduce(S, OpAddU64());
  ovf = warp_reduce(ovf, OpOrU32());
  if (lane == 0) {
    sh.wred64[warp] = S;
    sh.wred32[warp] = ovf;
  }
  __syncthreads();
  if (warp == 0) {
    uint64_t s2 = 0;
    uint32_t o2 = 0;
    for (int w = 0; w < kWarps; ++w) {  // every lane, the same sums
      s2 += sh.wred64[w];
      o2 |= sh.wred32[w];
    }
    if (lane < kCl) {
      *cluster.map_shared_rank(&sh.push.S[rank], lane) = s2;
      *cluster.map_shared_rank(&sh.push.fl2[rank], lane) = o2;
    }
  }
  cluster.sync();  // S2
  if (warp == 0 && lane == 0) {
    uint64_t sv = 0;
    uint32_t fl = 0;
    for (int r = 0; r < kCl; ++r) {
      sv += sh.push.S[r];
      fl |= sh.push.fl2[r];
    }
    {
      const AllocScale ks = alloc_scale(sv);  // sv >= 2^40: the max has weight 2^40
      sh.mk = ks.mk;
      sh.ek = ks.ek;
      sh.khi = ks.khi;
      sh.klo = ks.klo;
      sh.status = (fl & 1u) ? DSPARK_ST_NONFINITE : DSPARK_ST_OK;
    }
  }
  __syncthreads();
  if (sh.status != DSPARK_ST_OK) {
    const int st = sh.status;
    for (int v = lo + tid; v < hi; v += kThr) crow[v] = 0u;
    if (rank == 0 && tid == 0 && DSPARK_CHECK(row < p.n_rows)) {
      p.status[row] = st;
      if (p.tokens) p.tokens[row] = -1;
    }
    cluster.sync();
    if (ready && rank == 0 && tid == 0 && DSPARK_CHECK(row / p.depth < (p.n_rows + p.depth - 1) / p.depth)) {
      __threadfence();
      atomicAdd(&ready[row / p.depth], 1u);
    }
    return st;
  }
  const uint64_t mk = sh.mk;
  const int ek = sh.ek;
  const float khi = sh.khi, klo = sh.klo;

  // ---- pass C: words and fraction histogram (pairs on the fp32x2 pipe)
  const float klo2k = __fmul_rn(klo, 2048.0f);
  uint32_t F = 0, internal = 0;
  uint32_t gmask = 0;  // bit it: group tid + 256 it holds an element the float split left open
  {
    int it = 0;
    for (int g = tid; g < ngroups; g += kThr, ++it) {
      const float4 e4 = reinterpret_cast<const float4*>(sl)[g];
      const FloatSplit2 fa = float_split2(make_float2(e4.x, e4.y), khi, klo2k);
      const FloatSplit2 fc = float_split2(make_float2(e4.z, e4.w), khi, klo2k);
      bool any_open = false;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const FloatSplit2& fs = (i < 2) ? fa : fc;
        const int l = i & 1;
        const bool counted = fs.cert[l] && !fs.zero[l];
        any_open = any_open || !(fs.cert[l] || fs.zero[l]);
        // branch-free: the elements that do not count go to a dummy bin
        F += counted ? fs.f[l] : 0u;
        const uint32_t bin = counted ? fs.b[l] : kBins + (tid & 15);
        if (DSPARK_CHECK(bin < (uint32_t)(kBins + 16))) atomicAdd(&sh.hist[bin], 1u);
      }
      gmask |= any_open ? (1u << it) : 0u;
      // a group with an open element keeps its four weights for the refinement
      reinterpret_cast<uint4*>(slu)[g] =
          any_open ? make_uint4(__float_as_uint(e4.x), __float_as_uint(e4.y),
                                __float_as_uint(e4.z), __float_as_uint(e4.w))
                   : make_uint4(fa.word[0], fa.word[1], fc.word[0], fc.word[1]);
    }
  }
  // the flagged groups: the certified elements get their word (counted above),
  // the open ones (about 1 in 2000) the exact split
  for (uint32_t m2 = gmask; m2 != 0u; m2 &= m2 - 1u) {
    const int g = tid + kThr * (__ffs(m2) - 1);
    const uint4 e4 = reinterpret_cast<const uint4*>(slu)[g];
    const float ee[4] = {__uint_as_float(e4.x), __uint_as_float(e4.y), __uint_as_float(e4.z),
                         __uint_as_float(e4.w)};
    const FloatSplit2 fa = float_split2(make_float2(ee[0], ee[1]), khi, klo2k);
    const FloatSplit2 fc = float_split2(make_float2(ee[2], ee[3]), khi, klo2k);
    for (int i = 0; i < 4; ++i) {
      const FloatSplit2& fs = (i < 2) ? fa : fc;
      const int l = i & 1;
      const int s = 4 * g + i;
      if (DSPARK_CHECK(s < slice_cap))
        slu[s] = (fs.cert[l] || fs.zero[l]) ? fs.word[l]
                                            : exact_word(ee[i], mk, ek, sh, s, &F, &internal);
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
    if (lane < kCl) {
      *cluster.map_shared_rank(&sh.push.F[rank], lane) = f2;
      *cluster.map_shared_rank(&sh.push.fl3[rank], lane) = i2 ? 2u : 0u;
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
      fa = sh.push.F[lane];
      fl = sh.push.fl3[lane];
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
          for (int r = 0; r < kCl; ++r)
            if (DSPARK_CHECK(sb * kFine + i < kBins))
              g += cluster.map_shared_rank(&sh.hist[0], r)[sb * kFine + i];
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

  // ---- pass E: counts = f + [bin above the threshold bin], 128-bit stores;
  // groups holding a member of the threshold bin are flagged and listed after
  // the loop; escapes are corrected from their list
  const uint32_t carry_k = kLowMask - thr;
  const uint32_t esc_c = (kEsc + carry_k) >> 13;  // what the loop writes for an escape
  if (status == DSPARK_ST_OK) {
    const bool vec = ((reinterpret_cast<uintptr_t>(crow + lo) / 4) & 3) == (uintptr_t)off;
    uint32_t* cbase = crow + lo - off;  // slice position s is cbase[s]
    uint32_t mmask = 0;                 // bit it: group tid + 256 it holds a member
    int it = 0;
    // the trip count is the same for every thread (one warp reduction per step)
    for (int gb = 0; gb < ngroups; gb += kThr, ++it) {
      const int g = gb + tid;
      const bool valid = g < ngroups;
      const uint4 w4 = valid ? reinterpret_cast<const uint4*>(slu)[g] : make_uint4(0u, 0u, 0u, 0u);
      // f + [low > thr]: low + (kLowMask - thr) carries into bit 13 exactly
      // when low > thr
      const uint32_t c0 = (w4.x + carry_k) >> 13, c1 = (w4.y + carry_k) >> 13;
      const uint32_t c2 = (w4.z + carry_k) >> 13, c3 = (w4.w + carry_k) >> 13;
      const uint32_t xm = min(min((w4.x ^ thr) & kLowMask, (w4.y ^ thr) & kLowMask),
                              min((w4.z ^ thr) & kLowMask, (w4.w ^ thr) & kLowMask));
      mmask |= (valid && xm == 0u) ? (1u << it) : 0u;
      const bool full = valid && g >= g_first && g <= g_last;  // all four inside the slice
      uint32_t gsum = 0;
      if (full && in_row(4 * g) && in_row(4 * g + 3)) {
        gsum = c0 + c1 + c2 + c3;
        if (vec) {
          reinterpret_cast<uint4*>(cbase)[g] = make_uint4(c0, c1, c2, c3);
        } else {
          cbase[4 * g] = c0;
          cbase[4 * g + 1] = c1;
          cbase[4 * g + 2] = c2;
          cbase[4 * g + 3] = c3;
        }
      }
      // one block = the 32 groups of one warp in one step
      const uint32_t bs = __reduce_add_sync(0xffffffffu, gsum);
      if (lane == 0 && gb / 32 + warp < kBlkCap) sh.bsum[gb / 32 + warp] = bs;
    }
    __syncthreads();
    // partial edge groups (first and last): element by element
    if (tid < 8) {
      const int g = (tid < 4) ? 0 : ngroups - 1;
      const bool dup = (tid >= 4 && g == 0);
      const bool edge = g >= 0 && !(g >= g_first && g <= g_last);
      const int s = 4 * g + (tid & 3);
      if (!dup && edge && s >= off && s < off + n) {
        // an escape is stored by the correction below, which expects esc_c here
        const uint32_t w = slu[s];
        const uint32_t c = (w + carry_k) >> 13;
        if (w != kEsc && in_row(s)) cbase[s] = c;
        if (DSPARK_CHECK(g / 32 < kBlkCap)) atomicAdd(&sh.bsum[g / 32], c);
      }
    }
    // escapes: the right count, and the block sum corrected
    for (uint32_t j = tid; j < min(sh.n_esc, (uint32_t)kEscCap); j += kThr) {
      const int s = sh.esc[j].s;
      if (s < off || s >= off + n) continue;
      const uint32_t low = sh.esc[j].low;
      const uint32_t c = sh.esc[j].f + ((low > thr) ? 1u : 0u);
      if (in_row(s)) cbase[s] = c;
      if (DSPARK_CHECK(((s >> 2) >> 5) < kBlkCap)) atomicAdd(&sh.bsum[(s >> 2) >> 5], c - esc_c);
      if (low == thr) {
        const uint32_t q = atomicAdd(&sh.n_cand, 1u);
        if (q < (uint32_t)kCandCap) {
          sh.cand[q].v = lo - off + s;
          sh.cand[q].s = s;
        }
      }
    }
    // members of the threshold bin, from the flagged groups
    for (uint32_t m2 = mmask; m2 != 0u; m2 &= m2 - 1u) {
      const int g = tid + kThr * (__ffs(m2) - 1);
      for (int i = 0; i < 4; ++i) {
        const int s = 4 * g + i;
        if (s < off || s >= off + n || (slu[s] & kLowMask) != thr || slu[s] == kEsc) continue;
        const uint32_t q = atomicAdd(&sh.n_cand, 1u);
        if (q < (uint32_t)kCandCap) {
          sh.cand[q].v = lo - off + s;
          sh.cand[q].s = s;
        }
      }
    }
  }
  __syncthreads();
  // the CTA's count sum (before member grants), from the block sums
  if (warp == 0 && status == DSPARK_ST_OK) {
    const int nblk = (ngroups + 31) / 32;
    uint32_t t = 0;
    for (int k = lane; k < nblk; k += 32)
      if (DSPARK_CHECK(k < kBlkCap)) t += sh.bsum[k];
    t = __reduce_add_sync(0xffffffffu, t);
    if (lane == 0) sh.wred32[0] = t;
  }
  // exact fractions of the listed members
  auto key_of_x = [&](float x) -> uint64_t {
    const float y = scale ? __fmul_rn(x, invT) : x;
    uint32_t Ei;
    int se;
    weight_split_ef(weight40(__fsub_rn(y, m)), &Ei, &se);
    return frac_key(alloc_split(Ei, se, mk, ek));
  };
  // the logit of slice position s again (the slice holds other values by
  // now); a chain row's is z = RN(x + bias)
  auto x_at = [&](int s) -> float {
    if (!in_row(s)) return 0.0f;
    const float x = load_logit(xrow, p.dtype, (int64_t)(lo - off + s));
    return zbias ? __fadd_rn(x, __ldg(zbias + (lo - off + s))) : x;
  };
  auto exact_key = [&](int s) -> uint64_t { return key_of_x(x_at(s)); };
  const uint32_t my_cand = sh.n_cand;
  for (uint32_t j = tid; j < min(my_cand, (uint32_t)kCandCap); j += kThr)
    sh.cand[j].key = exact_key(sh.cand[j].s);
  __syncthreads();
  if (warp == 0 && lane < kCl) {
    *cluster.map_shared_rank(&sh.push.csum[rank], lane) =
        (status == DSPARK_ST_OK) ? sh.wred32[0] : 0u;
    *cluster.map_shared_rank(&sh.push.ncand[rank], lane) = my_cand;
  }
  cluster.sync();  // S4
  if (warp == 0) {
    uint32_t nc = 0, over = 0;
    if (lane < kCl) {
      const uint32_t cs = sh.push.csum[lane];
      nc = sh.push.ncand[lane];
      sh.peers_csum[lane] = cs;
      sh.peers_ncand[lane] = nc;
      sh.grants[lane] = 0u;  // lane < kCl
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
    if (in_row(s)) crow[lo - off + s] = f + 1u;
    if (DSPARK_CHECK(((s >> 2) >> 5) < kBlkCap)) atomicAdd(&sh.bsum[(s >> 2) >> 5], 1u);
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
      if (!DSPARK_CHECK((t - base) < (uint32_t)kCandCap && t < kAllCap)) continue;
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
        if (DSPARK_CHECK(owner >= 0 && owner < kCl)) atomicAdd(&sh.grants[owner], 1u);
        if (owner == rank) grant_member(all[i].s);
      }
    }
    __syncthreads();
  } else if (R > 0 && !fits && Rin > 0) {
    // many members (exact ties): every member's exact fraction is computed
    // once, on compacted windows so that whole warps work, and counted in a
    // small table of distinct fractions per CTA; the row's tables give the
    // threshold fraction, and the remaining tickets go to the lowest ids
    // holding it.  More distinct fractions than a table holds: 8-bit radix
    // levels over the exact fractions.
    ManyShared& ms = sh.many;
    constexpr uint32_t kMark = kGrant;  // marked member: grant bit set, pos bit clear
    auto low_of = [&](int s) -> uint32_t {
      const uint32_t w = slu[s];
      if (w != kEsc) return w & kLowMask;
      const int j = esc_find(sh, s);
      return j < 0 ? 0u : sh.esc[j].low;
    };
    auto set_low = [&](int s, uint32_t low) {
      const uint32_t w = slu[s];
      if (w != kEsc) {
        slu[s] = (w & ~kLowMask) | low;
        return;
      }
      const int j = esc_find(sh, s);
      if (j >= 0) sh.esc[j].low = low;
    };
    auto is_member = [&](int s) -> bool { return s >= off && s < off + n && low_of(s) == thr; };
    auto cls_state = [&](uint32_t low) -> int {  // -1: not a marked member
      return ((low & (kMark | kPos)) == kMark) ? (int)ms.state[low & (kTab - 1)] : -1;
    };
    const int npos = 4 * ngroups;
    if (tid < kTab) {
      ms.tkey[tid] = ~0ull;
      ms.tcnt[tid] = 0u;
    }
    uint32_t tovf = 0;
    uint64_t kmn = ~0ull, kmx = 0ull;
    for (int wb = 0; wb < npos; wb += kWin) {
      constexpr int kPer = kWin / kThr;  // positions per thread in a window
      const int p0 = wb + tid * kPer;
      uint32_t bits = 0, cnt = 0;
      for (int i = 0; i < kPer; ++i)
        if (p0 + i < npos && is_member(p0 + i)) {
          bits |= 1u << i;
          ++cnt;
        }
      uint32_t tot;
      const uint32_t incl = block_inclusive_scan(cnt, sh.wred32, &tot);
      uint32_t o = incl - cnt;
      for (int i = 0; i < kPer; ++i)
        if ((bits >> i) & 1u) {
          if (DSPARK_CHECK(o < (uint32_t)kWin)) ms.list[o] = (uint16_t)(p0 + i);
          ++o;
        }
      __syncthreads();
      // four rounds of members at a time: their logits are reloaded together
      for (uint32_t j4 = 0; j4 < tot; j4 += 4 * kThr) {
        float xs[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t j = j4 + u * kThr + tid;
          xs[u] = j < tot ? x_at((int)ms.list[j]) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
        const uint32_t j0 = j4 + u * kThr;
        if (j0 >= tot) break;  // the same for every thread
        const uint32_t j = j0 + tid;
        const bool valid = j < tot;
        const int sp = valid ? (int)ms.list[j] : 0;
        const uint64_t key = valid ? key_of_x(xs[u]) : ~0ull;
        if (valid) {
          kmn = min(kmn, key);
          kmx = max(kmx, key);
        }
        const unsigned grp = __match_any_sync(0xffffffffu, key);
        const int leader = __ffs(grp) - 1;
        uint32_t cls = kTab;
        if (valid && lane == leader) {
          int h = (int)((key ^ (key >> 23) ^ (key >> 41)) & (uint64_t)(kTab - 1));
          for (int t = 0; t < kTab; ++t) {
            const unsigned long long old = atomicCAS(
                reinterpret_cast<unsigned long long*>(&ms.tkey[h]), ~0ull, (unsigned long long)key);
            if (old == ~0ull || old == key) {
              atomicAdd(&ms.tcnt[h], (uint32_t)__popc(grp));
              cls = (uint32_t)h;
              break;
            }
            h = (h + 1) & (kTab - 1);
          }
        }
        cls = __shfl_sync(0xffffffffu, cls, leader);
        if (valid) {
          if (cls < (uint32_t)kTab) set_low(sp, kMark | cls);
          else tovf = 1u;
        }
        }
      }
      __syncthreads();
    }
    tovf = block_reduce(tovf, OpOrU32(), sh.wred32);
    kmn = block_reduce(kmn, OpMinU64(), sh.wred64);
    kmx = block_reduce(kmx, OpMaxU64(), sh.wred64);
    if (tid == 0) {
      sh.pub.flags4 = tovf;
      sh.pub.kmin = kmn;
      sh.pub.kmax = kmx;
    }
    cluster.sync();  // tables published
    if (warp == 0) {
      // every peer's flags and key range, fetched at once (lane r reads rank r)
      uint32_t fo = 0;
      uint64_t a = ~0ull, bb = 0ull;
      if (lane < kCl) {
        fo = *cluster.map_shared_rank(&sh.pub.flags4, lane);
        a = *cluster.map_shared_rank(&sh.pub.kmin, lane);
        bb = *cluster.map_shared_rank(&sh.pub.kmax, lane);
      }
      fo = warp_reduce(fo, OpOrU32());
      a = warp_reduce(a, OpMinU64());
      bb = warp_reduce(bb, OpMaxU64());
      if (lane == 0) {
        sh.fovf = fo;
        sh.gmin = a;
        sh.gmax = bb;
      }
    }
    __syncthreads();
    uint32_t mine = 0;
    if (sh.fovf == 0u) {
      // every table of the row, merged here
      if (tid == 0) {
        sh.thrk = 0ull;
        sh.need = 0u;
        sh.n_merged = 0u;
      }
      __syncthreads();
      // the non-empty slots of every table of the row, gathered here (a
      // fraction held by several CTAs keeps one slot per CTA)
      for (int t = tid; t < kCl * kTab; t += kThr) {
        const int r = t / kTab, slot = t % kTab;
        const uint32_t c = *cluster.map_shared_rank(&ms.tcnt[slot], r);
        if (c == 0u) continue;
        const uint32_t q = atomicAdd(&sh.n_merged, 1u);
        if (!DSPARK_CHECK(q < (uint32_t)(kCl * kTab))) continue;
        ms.merged.key[q] = *cluster.map_shared_rank(&ms.tkey[slot], r);
        ms.merged.cnt[q] = c;
      }
      __syncthreads();
      const int nmg = (int)sh.n_merged;
      // the threshold fraction holds the Rin-th ticket: above < Rin <= above + at
      for (int t = tid; t < nmg; t += kThr) {
        const uint64_t kt = ms.merged.key[t];
        uint32_t above = 0, at = 0;
        for (int u = 0; u < nmg; ++u) {
          const uint32_t cu = ms.merged.cnt[u];
          const uint64_t ku = ms.merged.key[u];
          above += (ku > kt) ? cu : 0u;
          at += (ku == kt) ? cu : 0u;
        }
        if (above < Rin && Rin <= above + at) {
          sh.thrk = kt;
          sh.need = Rin - above;
        }
      }
      __syncthreads();
      const uint64_t thrk = sh.thrk;
      if (tid < kTab) {
        const uint64_t kt = ms.tkey[tid];
        ms.state[tid] = (ms.tcnt[tid] == 0u) ? 0 : (kt > thrk ? 1 : (kt == thrk ? 2 : 0));
      }
      __syncthreads();
      // members above the threshold fraction get their ticket, those below
      // none; those at it are counted per warp segment (id order)
      const int seg = (npos + kWarps - 1) / kWarps;
      const int a0 = warp * seg, a1 = min(npos, a0 + seg);
      uint32_t* atm = ms.atm + warp * kAtSteps;  // the merged tables are no longer read
      uint32_t wat = 0;
      for (int s0 = a0; s0 < a1; s0 += 32) {
        const int sp = s0 + lane;
        const int stt = (sp < a1) ? cls_state(low_of(sp)) : -1;
        if (stt == 1) {
          set_low(sp, thr);
          grant_member(sp);
          ++mine;
        } else if (stt == 0) {
          set_low(sp, thr);
        }
        const unsigned at = __ballot_sync(0xffffffffu, stt == 2);
        if (lane == 0 && DSPARK_CHECK(warp * kAtSteps + ((s0 - a0) >> 5) < kWarps * kAtSteps))
          atm[(s0 - a0) >> 5] = at;
        wat += (uint32_t)__popc(at);
      }
      if (lane == 0) sh.wcnt[warp] = wat;
      __syncthreads();
      if (tid == 0) {
        uint32_t t = 0;
        for (int w = 0; w < kWarps; ++w) t += sh.wcnt[w];
        sh.pub.n_eq = t;
      }
      cluster.sync();
      if (warp == 0) {
        // members at the threshold in the lower ranks, fetched at once
        const uint32_t e = lane < rank ? *cluster.map_shared_rank(&sh.pub.n_eq, lane) : 0u;
        const uint32_t base = warp_reduce(e, OpAddU32());
        if (lane == 0) sh.scan_base = base;
      }
      __syncthreads();
      uint32_t base = sh.scan_base;
      for (int w = 0; w < warp; ++w) base += sh.wcnt[w];
      const uint32_t need = sh.need;
      for (int s0 = a0; s0 < a1; s0 += 32) {
        const unsigned msk = atm[(s0 - a0) >> 5];
        if (msk == 0u) continue;  // the same for the whole warp
        const int sp = s0 + lane;
        const bool at = (msk >> lane) & 1u;
        if (at) {
          const uint32_t rk = base + (uint32_t)__popc(msk & ((1u << lane) - 1u));
          set_low(sp, thr);
          if (rk < need) {
            grant_member(sp);
            ++mine;
          }
        }
        base += (uint32_t)__popc(msk);
      }
      __syncthreads();
    } else {
      // the members marked in the tables become plain members again
      for (int sp = tid; sp < npos; sp += kThr)
        if (cls_state(low_of(sp)) >= 0) set_low(sp, thr);
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
    }
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
  if (rank == 0 && tid == 0 && DSPARK_CHECK(row < p.n_rows)) {
    p.status[row] = status;
    if (p.tokens && status != DSPARK_ST_OK) p.tokens[row] = -1;
  }
  bool signal = ready && status != DSPARK_ST_OK && rank == 0 && tid == 0;
  // every remote read of this CTA's shared memory is done: arrive now, wait
  // before leaving.  A chain row arrives after the draw instead, whose token
  // the drawing CTA stores into every CTA's sh.chain_tok first.
  if (!chain) cluster.barrier_arrive();

  // ---- fused draft draw: the CTA whose range holds D finds the block of 32
  // groups holding it from the block sums, then the token inside it (warp 0)
  if (p.tokens && status == DSPARK_ST_OK) {
    const uint32_t D = sh.draw;
    if (warp == 0 && D >= cbefore && D - cbefore < my_total) {
      const uint32_t t = D - cbefore;
      const int nblk = (ngroups + 31) / 32;
      uint32_t base = 0;
      int blk = -1;
      for (int k0 = 0; k0 < nblk && blk < 0; k0 += 32) {
        const int k = k0 + lane;
        const uint32_t v = (k < nblk) ? sh.bsum[k] : 0u;
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
        const bool hit = v > 0u && t - base < incl && t - base >= incl - v;
        const unsigned msk = __ballot_sync(0xffffffffu, hit);
        if (msk) {
          const int l = __ffs(msk) - 1;
          blk = k0 + l;
          base += __shfl_sync(0xffffffffu, incl - v, l);
        } else {
          base += __shfl_sync(0xffffffffu, incl, 31);
        }
      }
      int token = -1;
      if (blk >= 0) {
        const int g = blk * 32 + lane;
        uint32_t cv[4] = {0u, 0u, 0u, 0u};
        uint32_t gs = 0;
        if (g < ngroups)
          for (int i = 0; i < 4; ++i) {
            cv[i] = DSPARK_CHECK(4 * g + i < slice_cap) ? count_of(sh, slu, 4 * g + i, thr) : 0u;
            gs += cv[i];
          }
        uint32_t incl = gs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
        const uint32_t tb = t - base;
        const bool hit = gs > 0u && tb < incl && tb >= incl - gs;
        if (hit) {
          uint32_t cum = incl - gs;
          for (int i = 0; i < 4; ++i) {
            cum += cv[i];
            if (tb < cum) {
              token = lo - off + 4 * g + i;
              break;
            }
          }
        }
        const unsigned msk = __ballot_sync(0xffffffffu, hit);
        if (msk) token = __shfl_sync(0xffffffffu, token, __ffs(msk) - 1);
      }
      if (lane == 0) {
        if (DSPARK_CHECK(row < p.n_rows)) p.tokens[row] = token;
        signal = ready != nullptr;
      }
      if (chain && lane < kCl) *cluster.map_shared_rank(&sh.chain_tok, lane) = token;
    }
  }
  if (chain) cluster.barrier_arrive();
  cluster.barrier_wait();  // no CTA leaves while a peer may still read its shared memory
  if (signal && DSPARK_CHECK(row / p.depth < (p.n_rows + p.depth - 1) / p.depth)) {
    // every CTA's counts were written before its arrive, the token before
    // this point: make them visible device-wide, then count the row done
    __threadfence();
    atomicAdd(&ready[row / p.depth], 1u);
  }
  return status;
}

}  // namespace
}  // namespace qdense
}  // namespace dspark
