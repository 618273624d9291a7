// tp.cu -- the vocabulary-sharded q build and draft draw, emulated on one GPU
// ("PP1 q transport and scheduling design", Sparse support and
// vocabulary-sharded TP2 follow-up: each rank computes its logit max and
// shifted sum and an all-reduce gives the global normalisation; the remaining
// tickets are coordinated globally; the leader's one integer draw picks the
// shard by its count mass, then the token inside it).
//
// The vocabulary is split into n_sh contiguous shards of ceil(V / n_sh) ids.
// Each kernel below runs one CTA per (row, shard) -- the work of one rank --
// and every exchange between ranks goes through a per-row record in the
// caller's workspace between launches: a rank only reads the other ranks'
// partials, never their rows.
//   1  local max of y and the validity flags
//   2  all-reduce max (each rank combines the partials); E and its uint64 sum
//   3  all-reduce the sum; exact floors f, the fraction histogram (2048 bins
//      of floor(2048 r)), the floor sum and the count of r > 0
//   4  all-reduce F, the histograms and the counts; the bin holding the
//      grant threshold; counts f + [bin above it]; each rank's table of the
//      distinct exact fractions in that bin, with their counts
//   5  the leader merges the tables: the threshold fraction T and each
//      rank's quota of members at T (ranks in id order, so the lowest ids
//      come first); a refused row is zeroed here
//   6  each rank grants its members above T, and its quota of members at T
//      to its lowest ids (an id-ordered block scan); its count total.  The
//      threshold-bin members are marked in the counts by step 4, so only
//      they are split again here
//   7  the leader's draw: the shard by the count totals, the token inside
// Floors and fractions are exact integer splits of E * RN64(2^24 / RN64(S)),
// so the counts equal those of the unsharded build bit for bit.
//
// Top-k rows (same follow-up: a global top-k merge of the ranks' local
// top-k): each rank selects its local top k by (y desc, id asc) with a radix
// select over its shard and sends those candidates; the leader merges the at
// most n_sh * k candidates into the global top k by the same order (the
// global top k is a subset of the union of the local ones) and allocates the
// tickets on that support.  The leader's draw over the support in id order is
// the draw that picks the shard by its count total, then the token inside.
#define DSPARK_TU 8  // this file's number in the checked build's site codes
#include "support_alloc.cuh"

namespace dspark {
namespace {

constexpr int kTpThr = 256;
constexpr int kTpMaxShards = 8;
constexpr int kTpBins = 2048;
constexpr int kTpTab = 1024;  // distinct threshold-bin fractions per shard
constexpr uint64_t kTpEmpty = ~0ull;  // an empty table slot (no fraction key is all ones)
constexpr uint32_t kTpMark = 0x80000000u;  // a count marked as a threshold-bin member (f < 2^31)

// One draft row's exchange record.
struct TpRow {
  float mx[kTpMaxShards];
  uint32_t fl[kTpMaxShards];  // bit0 NaN / +inf / overflow, bit1 a finite y
  uint64_t S[kTpMaxShards];
  uint64_t F[kTpMaxShards];
  uint32_t npos[kTpMaxShards];
  uint64_t C[kTpMaxShards];
  uint32_t over[kTpMaxShards];   // the shard's table overflowed
  uint32_t nc[kTpMaxShards];     // top-k rows: the shard's candidates
  uint32_t quota[kTpMaxShards];  // members at T granted in the shard
  uint64_t T;                    // the threshold fraction's key
  int32_t st;                    // the row's status after the grant step
  uint32_t hist[kTpMaxShards][kTpBins];
  uint64_t tab_key[kTpMaxShards][kTpTab];  // top-k rows: candidates (key << 32 | id)
  uint32_t tab_cnt[kTpMaxShards][kTpTab];
};

struct TpParams {
  const void* x;
  int dtype;
  int64_t ld;
  int V;
  int n_sh;
  int depth;
  const float* temperature;
  uint64_t seed;
  const uint32_t* request_ids;
  uint32_t* counts;
  int32_t* tokens;
  int32_t* status;
  TpRow* ws;
  int top_k;     // 0: dense rows
  int32_t* ids;  // top-k rows: [rows][top_k]
  int32_t* nnz;  // top-k rows: [rows]
};

struct TpShared {
  uint64_t r64[32];
  uint32_t r32[32];
  float rf[32];
  uint32_t hist[kTpBins];
  int found;
  int gs_bstar;     // grant_state: the threshold bin and the tickets inside it
  uint32_t gs_rin;
};

struct OpMaxNaNTp {
  __device__ float operator()(float a, float b) const {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
  }
};

struct Shard {
  int row, s, lo, hi;
};

__device__ __forceinline__ Shard shard_of(const TpParams& p) {
  Shard sh;
  sh.row = blockIdx.x / p.n_sh;
  sh.s = blockIdx.x % p.n_sh;
  const int vs = (p.V + p.n_sh - 1) / p.n_sh;
  sh.lo = min(p.V, sh.s * vs);
  sh.hi = min(p.V, sh.lo + vs);
  return sh;
}

__device__ __forceinline__ float inv_temp(const TpParams& p, int row, bool* bad) {
  const float T = p.temperature ? p.temperature[row] : 1.0f;
  const float iT = __frcp_rn(T);
  *bad = !(isfinite(T) && T > 0.0f) || !(isfinite(iT) && iT >= 0x1p-126f);
  return iT;
}

__device__ __forceinline__ float y_of(const TpParams& p, int row, int v, float invT) {
  const char* xrow = reinterpret_cast<const char*>(p.x) +
                     (int64_t)row * p.ld * (p.dtype == DSPARK_F32 ? 4 : 2);
  const float x = load_logit(xrow, p.dtype, v);
  return invT == 1.0f ? x : __fmul_rn(x, invT);
}

// The row's status from every rank's flags, and the global max (all-reduce).
__device__ __forceinline__ int row_state(const TpParams& p, const TpRow& w, bool badT, float* m) {
  float mm = -INFINITY;
  uint32_t fl = 0;
  for (int s = 0; s < p.n_sh; ++s) {
    mm = fmaxf(mm, w.mx[s]);
    fl |= w.fl[s];
  }
  *m = mm;
  if (badT) return DSPARK_ST_BAD_TEMPERATURE;
  if (fl & 1u) return DSPARK_ST_NONFINITE;
  if (!(fl & 2u)) return DSPARK_ST_ZERO_MASS;
  return DSPARK_ST_OK;
}

// floor(2048 r) of an exact split (r = rnum / 2^t)
__device__ __forceinline__ uint32_t bin_of(const AllocSplit& a) {
  if (a.rnum == 0ull) return 0u;
  return (uint32_t)(a.t >= 11 ? (a.rnum >> (a.t - 11)) : (a.rnum << (11 - a.t)));
}

__device__ __forceinline__ AllocSplit split_of(float y, float m, uint64_t mk, int ek) {
  uint32_t Ei;
  int se;
  weight_split_ef(weight40(__fsub_rn(y, m)), &Ei, &se);
  return alloc_split(Ei, se, mk, ek);
}

// The dense kernel's certified float split of a = RN64(E k): with k = khi +
// klo + d (|d| <= 2^-48 k), p1 + e1 = E khi exactly (fma) and p2 = RN32(E klo),
// fr = RN(RN(p1 - f0) + RN(e1 + p2)) is within 2^-13 + 2^-34.4 p1 of
// 2048 (a - f0) / 2048.  When 2048 fr is at least 2^-12 + 2^-15 from every
// integer and p1 < 2^19, floor(a) = f0 + floor(G / 2048) and the bin
// floor(2048 r) = G mod 2048 (G = floor(2048 fr)) are exact and r > 0;
// otherwise cert is false and the exact integer split decides (about 1
// element in 2,000).  E = 0 is certified with f = 0 and no fraction.
struct TpFast {
  uint32_t f, bin;
  bool cert, zero;
};
__device__ __forceinline__ TpFast tp_fast_split(float Ef, float khi, float klo) {
  TpFast o;
  const float p1 = __fmul_rn(Ef, khi);
  const float e1 = __fmaf_rn(Ef, khi, -p1);
  const float p2 = __fmul_rn(Ef, klo);
  const float f0 = floorf(p1);
  const float fr = __fadd_rn(__fsub_rn(p1, f0), __fadd_rn(e1, p2));
  const float fb = __fmul_rn(fr, 2048.0f);
  const float G = floorf(fb);
  o.zero = (Ef == 0.0f);
  o.cert = o.zero || (fabsf(__fsub_rn(__fsub_rn(fb, G), 0.5f)) < 0.5f - 0x1p-12f - 0x1p-15f &&
                      f0 < 524285.0f);  // 2^19 - 3
  const int f0i = __float_as_int(__fadd_rn(f0, 12582912.0f)) - 0x4B400000;
  const int Gi = __float_as_int(__fadd_rn(G, 12582912.0f)) - 0x4B400000;
  o.f = o.zero ? 0u : (uint32_t)(f0i + (Gi >> 11));
  o.bin = (uint32_t)Gi & (kTpBins - 1u);
  return o;
}

__global__ void __launch_bounds__(kTpThr) tp_max_kernel(TpParams p) {
  __shared__ TpShared sh;
  const Shard d = shard_of(p);
  bool badT;
  const float invT = inv_temp(p, d.row, &badT);
  float mx = -INFINITY;
  uint32_t fl = 0;
  if (!badT)
    for (int v = d.lo + threadIdx.x; v < d.hi; v += kTpThr) {
      const char* xrow = reinterpret_cast<const char*>(p.x) +
                         (int64_t)d.row * p.ld * (p.dtype == DSPARK_F32 ? 4 : 2);
      const float x = load_logit(xrow, p.dtype, v);
      if (!(x < INFINITY)) fl |= 1u;  // NaN or +inf
      const float y = invT == 1.0f ? x : __fmul_rn(x, invT);
      if (fabsf(y) == INFINITY && fabsf(x) < INFINITY) fl |= 1u;  // overflow
      if (y > -INFINITY && y < INFINITY) {
        fl |= 2u;
        mx = fmaxf(mx, y);
      }
    }
  mx = block_reduce(mx, OpMaxNaNTp(), sh.rf);
  fl = block_reduce(fl, OpOrU32(), sh.r32);
  if (threadIdx.x == 0) {
    p.ws[d.row].mx[d.s] = mx;
    p.ws[d.row].fl[d.s] = fl;
  }
}

__global__ void __launch_bounds__(kTpThr) tp_weights_kernel(TpParams p) {
  __shared__ TpShared sh;
  const Shard d = shard_of(p);
  const TpRow& w = p.ws[d.row];
  bool badT;
  const float invT = inv_temp(p, d.row, &badT);
  float m;
  const int st = row_state(p, w, badT, &m);
  uint64_t S = 0;
  if (st == DSPARK_ST_OK)
    for (int v = d.lo + threadIdx.x; v < d.hi; v += kTpThr)
      S += __float2ull_rz(weight40(__fsub_rn(y_of(p, d.row, v, invT), m)));
  S = block_reduce(S, OpAddU64(), sh.r64);
  if (threadIdx.x == 0) p.ws[d.row].S[d.s] = S;
}

__global__ void __launch_bounds__(kTpThr) tp_floors_kernel(TpParams p) {
  __shared__ TpShared sh;
  const Shard d = shard_of(p);
  TpRow& w = p.ws[d.row];
  bool badT;
  const float invT = inv_temp(p, d.row, &badT);
  float m;
  const int st = row_state(p, w, badT, &m);
  for (int i = threadIdx.x; i < kTpBins; i += kTpThr) sh.hist[i] = 0u;
  __syncthreads();
  uint64_t F = 0;
  uint32_t npos = 0;
  if (st == DSPARK_ST_OK) {
    uint64_t S = 0;
    for (int s = 0; s < p.n_sh; ++s) S += w.S[s];
    const AllocScale k = alloc_scale(S);
    for (int v = d.lo + threadIdx.x; v < d.hi; v += kTpThr) {
      const float Ef = weight40(__fsub_rn(y_of(p, d.row, v, invT), m));
      const TpFast q = tp_fast_split(Ef, k.khi, k.klo);
      uint32_t f = q.f, bin = q.bin;
      bool pos = !q.zero;
      if (!q.cert) {
        uint32_t Ei;
        int se;
        weight_split_ef(Ef, &Ei, &se);
        const AllocSplit a = alloc_split(Ei, se, k.mk, k.ek);
        f = a.f;
        pos = a.rnum != 0ull;
        bin = bin_of(a);
      }
      p.counts[(int64_t)d.row * p.V + v] = f;
      F += f;
      if (pos) {
        ++npos;
        atomicAdd(&sh.hist[bin], 1u);
      }
    }
  }
  F = block_reduce(F, OpAddU64(), sh.r64);
  npos = block_reduce(npos, OpAddU32(), sh.r32);
  for (int i = threadIdx.x; i < kTpBins; i += kTpThr) w.hist[d.s][i] = sh.hist[i];
  for (int i = threadIdx.x; i < kTpTab; i += kTpThr) {
    w.tab_key[d.s][i] = kTpEmpty;
    w.tab_cnt[d.s][i] = 0u;
  }
  if (threadIdx.x == 0) {
    w.F[d.s] = F;
    w.npos[d.s] = npos;
    w.over[d.s] = 0u;
  }
}

// The threshold bin and the tickets granted inside it, from every rank's
// partials (each rank computes the same values).  Every thread of the block
// calls it: the ranks' histograms are added into sh.hist, and a scan over the
// bins from the top (eight per thread) finds the bin holding the R-th ticket.
__device__ int grant_state(const TpParams& p, const TpRow& w, int st, TpShared& sh,
                           uint32_t* R, int* bstar, uint32_t* Rin) {
  *R = 0;
  *bstar = -1;
  *Rin = 0;
  if (st != DSPARK_ST_OK) return st;
  uint64_t F = 0, npos = 0;
  for (int s = 0; s < p.n_sh; ++s) {
    F += w.F[s];
    npos += w.npos[s];
  }
  if (F == 0 || F > (uint64_t)kM || (uint64_t)kM - F > npos) return DSPARK_ST_ALLOC_INCONSISTENT;
  *R = (uint32_t)((uint64_t)kM - F);
  if (*R == 0) return st;
  static_assert(kTpBins == 8 * kTpThr, "eight bins per thread");
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  __syncthreads();  // earlier readers of sh.hist are done
  for (int b = t; b < kTpBins; b += kTpThr) {
    uint32_t c = 0;
    for (int s = 0; s < p.n_sh; ++s) c += w.hist[s][b];
    sh.hist[b] = c;
  }
  if (t == 0) {
    sh.gs_bstar = -1;
    sh.gs_rin = 0u;
  }
  __syncthreads();
  // thread t holds bins kTpBins - 8t - 1 down to kTpBins - 8t - 8
  const int bt = kTpBins - 8 * t - 1;
  uint32_t c[8], tot = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = sh.hist[bt - j];
    tot += c[j];
  }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) sh.r32[warp] = incl;
  __syncthreads();
  for (int w2 = 0; w2 < warp; ++w2) incl += sh.r32[w2];
  const uint32_t excl = incl - tot, r = *R;
  if (excl < r && r <= incl) {
    uint32_t acc = excl;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (acc < r && r <= acc + c[j]) {
        sh.gs_bstar = bt - j;
        sh.gs_rin = r - acc;
      }
      acc += c[j];
    }
  }
  __syncthreads();
  *bstar = sh.gs_bstar;
  *Rin = sh.gs_rin;
  return st;
}

// One element of the grant pass: an element above the threshold bin gets
// f + 1; a member of the bin is marked in its count and returns true with
// its exact fraction's key.
__device__ __forceinline__ bool grant_one(const TpParams& p, const Shard& d, int v, float invT,
                                          float m, const AllocScale& k, int bstar,
                                          uint64_t* key) {
  const float Ef = weight40(__fsub_rn(y_of(p, d.row, v, invT), m));
  const TpFast q = tp_fast_split(Ef, k.khi, k.klo);
  if (q.zero) return false;
  int b = (int)q.bin;
  uint32_t f = q.f;
  AllocSplit a;
  if (!q.cert || b == bstar) {  // the exact split: open elements, and the key of a member
    uint32_t Ei;
    int se;
    weight_split_ef(Ef, &Ei, &se);
    a = alloc_split(Ei, se, k.mk, k.ek);
    if (a.rnum == 0ull) return false;
    b = (int)bin_of(a);
    f = a.f;
  }
  uint32_t* c = p.counts + (int64_t)d.row * p.V + v;
  if (b > bstar) *c = f + 1u;
  if (b != bstar) return false;
  *c = f | kTpMark;  // its exact split was taken above
  *key = frac_key(a);
  return true;
}

__global__ void __launch_bounds__(kTpThr) tp_grant_kernel(TpParams p) {
  __shared__ TpShared sh;
  const Shard d = shard_of(p);
  TpRow& w = p.ws[d.row];
  bool badT;
  const float invT = inv_temp(p, d.row, &badT);
  float m;
  int st = row_state(p, w, badT, &m);
  uint32_t R, Rin;
  int bstar;
  st = grant_state(p, w, st, sh, &R, &bstar, &Rin);
  if (st != DSPARK_ST_OK || R == 0) return;
  uint64_t S = 0;
  for (int s = 0; s < p.n_sh; ++s) S += w.S[s];
  const AllocScale k = alloc_scale(S);
  for (int v0 = d.lo; v0 < d.hi; v0 += kTpThr) {  // whole warps: the table insert below
    const int v = v0 + (int)threadIdx.x;
    uint64_t key = kTpEmpty;
    const bool member = v < d.hi && grant_one(p, d, v, invT, m, k, bstar, &key);
    // count the members' fractions in the shard's table (open addressing),
    // one atomic per distinct fraction in the warp (members are rare: most
    // warps skip the match)
    if (!__any_sync(0xffffffffu, member)) continue;
    const unsigned grp = __match_any_sync(0xffffffffu, member ? key : kTpEmpty);
    if (member && (int)(threadIdx.x & 31u) == __ffs(grp) - 1) {
      uint32_t h = (uint32_t)((key * 0x9E3779B97F4A7C15ull) >> 54) & (kTpTab - 1);
      bool done = false;
      for (int probe = 0; probe < kTpTab && !done; ++probe) {
        unsigned long long* slot =
            reinterpret_cast<unsigned long long*>(&w.tab_key[d.s][(h + probe) & (kTpTab - 1)]);
        const unsigned long long prev = atomicCAS(slot, (unsigned long long)kTpEmpty, key);
        if (prev == kTpEmpty || prev == key) {
          atomicAdd(&w.tab_cnt[d.s][(h + probe) & (kTpTab - 1)], (uint32_t)__popc(grp));
          done = true;
        }
      }
      if (!done) w.over[d.s] = 1u;
    }
  }
}

// The leader of each row: merges the ranks' tables into the threshold
// fraction T and each rank's quota of members at T, writes the status (and
// zeroes a refused row).
__global__ void __launch_bounds__(kTpThr) tp_threshold_kernel(TpParams p) {
  __shared__ TpShared sh;
  const int row = blockIdx.x;
  TpRow& w = p.ws[row];
  bool badT;
  inv_temp(p, row, &badT);
  float m;
  int st = row_state(p, w, badT, &m);
  uint32_t R, Rin;
  int bstar;
  st = grant_state(p, w, st, sh, &R, &bstar, &Rin);
  bool over = false;
  for (int s = 0; s < p.n_sh; ++s) over |= w.over[s] != 0u;
  if (st == DSPARK_ST_OK && R > 0 && over) st = DSPARK_ST_INTERNAL;
  __shared__ uint64_t keys[kTpTab];
  __shared__ uint32_t cnts[kTpTab];
  __shared__ uint32_t nk;
  __shared__ uint64_t Tsh;
  if (threadIdx.x == 0) {
    nk = 0u;
    Tsh = kTpEmpty;
    sh.found = -1;
  }
  __syncthreads();
  if (st == DSPARK_ST_OK && R > 0) {
    // the ranks' non-empty slots, gathered (a fraction held by several
    // ranks keeps one slot per rank; the counts still add up)
    const int n = p.n_sh * kTpTab;
    for (int i = threadIdx.x; i < n; i += kTpThr) {
      const uint64_t ki = w.tab_key[i / kTpTab][i % kTpTab];
      if (ki == kTpEmpty) continue;
      const uint32_t j = atomicAdd(&nk, 1u);
      if (j < (uint32_t)kTpTab) {
        keys[j] = ki;
        cnts[j] = w.tab_cnt[i / kTpTab][i % kTpTab];
      }
    }
    __syncthreads();
    if (nk > (uint32_t)kTpTab) {
      st = DSPARK_ST_INTERNAL;  // more distinct fractions than the gather holds
    } else {
      // T: the fraction with (members above it) < Rin <= (members at or above it)
      for (uint32_t i = threadIdx.x; i < nk; i += kTpThr) {
        const uint64_t ki = keys[i];
        uint64_t above = 0, at = 0;
        for (uint32_t j = 0; j < nk; ++j) {
          if (keys[j] > ki) above += cnts[j];
          else if (keys[j] == ki) at += cnts[j];
        }
        if (above < Rin && Rin <= above + at) {
          Tsh = ki;  // every slot holding T writes the same values
          sh.found = (int)(Rin - above);
        }
      }
      __syncthreads();
      if (sh.found < 0) st = DSPARK_ST_INTERNAL;  // the tables miss members of the bin
    }
  }
  // each rank's members at T (every thread scans part of every table), then
  // each rank's quota of them, ranks in id order
  const bool want = st == DSPARK_ST_OK && R > 0;
  uint32_t at_s[kTpMaxShards];
  for (int s = 0; s < p.n_sh; ++s) {
    uint32_t c = 0;
    if (want)
      for (int j = threadIdx.x; j < kTpTab; j += kTpThr)
        if (w.tab_key[s][j] == Tsh) c += w.tab_cnt[s][j];
    at_s[s] = block_reduce(c, OpAddU32(), sh.r32);
  }
  if (threadIdx.x == 0) {
    uint32_t need = want ? (uint32_t)sh.found : 0u;
    for (int s = 0; s < p.n_sh; ++s) {
      const uint32_t q = min(need, at_s[s]);
      w.quota[s] = q;
      need -= q;
    }
    w.T = st == DSPARK_ST_OK ? Tsh : kTpEmpty;
  }
  if (st != DSPARK_ST_OK)
    for (int v = threadIdx.x; v < p.V; v += kTpThr) p.counts[(int64_t)row * p.V + v] = 0u;
  if (threadIdx.x == 0) {
    w.st = st;
    p.status[row] = st;
    if (p.tokens && st != DSPARK_ST_OK) p.tokens[row] = -1;
  }
}

// Each rank grants its marked members above T, and its quota of members at
// T to its lowest ids, and sums its counts.  The members at T are listed as
// they are met and ranked by id afterwards; more of them than the list holds
// (long exact ties) are granted by an id-ordered block scan instead.
constexpr int kTpAtCap = 1024;
__global__ void __launch_bounds__(kTpThr) tp_ties_kernel(TpParams p) {
  __shared__ TpShared sh;
  __shared__ int32_t at_ids[kTpAtCap];
  __shared__ uint32_t n_at;
  const Shard d = shard_of(p);
  TpRow& w = p.ws[d.row];
  uint64_t C = 0;
  if (threadIdx.x == 0) n_at = 0u;
  __syncthreads();
  if (w.st == DSPARK_ST_OK) {
    bool badT;
    const float invT = inv_temp(p, d.row, &badT);
    float m;
    row_state(p, w, badT, &m);
    uint64_t S = 0;
    for (int s = 0; s < p.n_sh; ++s) S += w.S[s];
    const AllocScale k = alloc_scale(S);
    const uint64_t T = w.T;
    const uint32_t quota = w.quota[d.s];
    uint32_t* crow = p.counts + (int64_t)d.row * p.V;
    for (int v = d.lo + (int)threadIdx.x; v < d.hi; v += kTpThr) {
      uint32_t c = crow[v];
      if ((c & kTpMark) != 0u) {
        c &= ~kTpMark;
        const uint64_t key = frac_key(split_of(y_of(p, d.row, v, invT), m, k.mk, k.ek));
        if (key > T) {
          c += 1u;
        } else if (key == T && quota > 0u) {
          const uint32_t j = atomicAdd(&n_at, 1u);
          if (j < (uint32_t)kTpAtCap) at_ids[j] = v;
        }
        crow[v] = c;
      }
      C += c;
    }
    __syncthreads();
    const uint32_t na = n_at;
    if (na <= (uint32_t)kTpAtCap) {
      // the quota's lowest ids among the listed members
      for (uint32_t i = threadIdx.x; i < na; i += kTpThr) {
        const int32_t vi = at_ids[i];
        uint32_t rank = 0;
        for (uint32_t j = 0; j < na; ++j) rank += (at_ids[j] < vi) ? 1u : 0u;
        if (rank < quota) {
          crow[vi] += 1u;
          C += 1u;
        }
      }
    } else {
      // every member at T again, in id order (their counts are unmarked now)
      uint32_t base = 0;
      for (int v0 = d.lo; v0 < d.hi; v0 += kTpThr) {
        const int v = v0 + (int)threadIdx.x;
        uint32_t at = 0;
        if (v < d.hi) {
          const AllocSplit a = split_of(y_of(p, d.row, v, invT), m, k.mk, k.ek);
          at = (a.rnum != 0ull && frac_key(a) == T) ? 1u : 0u;
        }
        if (__syncthreads_or(at)) {  // uniform over the block
          uint32_t tot;
          const uint32_t incl = block_inclusive_scan(at, sh.r32, &tot);
          if (at && base + incl - 1u < quota) {
            crow[v] += 1u;
            C += 1u;
          }
          base += tot;
          __syncthreads();
        }
      }
    }
  }
  C = block_reduce(C, OpAddU64(), sh.r64);
  if (threadIdx.x == 0) w.C[d.s] = C;
}

// The leader's draw picks the shard by the count totals; that rank finds the
// token (the first id whose cumulative count exceeds the draw).
__global__ void __launch_bounds__(kTpThr) tp_draw_kernel(TpParams p) {
  __shared__ TpShared sh;
  const Shard d = shard_of(p);
  if (p.status[d.row] != DSPARK_ST_OK) return;
  const TpRow& w = p.ws[d.row];
  uint64_t before = 0;
  for (int s = 0; s < d.s; ++s) before += w.C[s];
  const int b = d.row / p.depth, j = d.row % p.depth;
  const uint32_t req = p.request_ids ? p.request_ids[b] : (uint32_t)b;
  const uint64_t D = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_PROPOSAL) >> 8;
  if (!(D >= before && D - before < w.C[d.s])) return;
  const uint32_t t = (uint32_t)(D - before);  // < the shard's total <= 2^24
  // each thread sums a contiguous run of the shard; one block scan finds the
  // run holding t, and its thread walks it
  const uint32_t* crow = p.counts + (int64_t)d.row * p.V;
  const int L = (d.hi - d.lo + kTpThr - 1) / kTpThr;
  const int a0 = min(d.hi, d.lo + (int)threadIdx.x * L), a1 = min(d.hi, a0 + L);
  uint32_t mine = 0;
  for (int v = a0; v < a1; ++v) mine += crow[v];
  uint32_t tot;
  const uint32_t incl = block_inclusive_scan(mine, sh.r32, &tot);
  const uint32_t excl = incl - mine;
  if (mine > 0u && excl <= t && t < incl) {
    uint32_t cum = excl;
    for (int v = a0; v < a1; ++v) {
      cum += crow[v];
      if (t < cum) {
        p.tokens[d.row] = v;
        break;
      }
    }
  }
}

// ------------------------------------------------------------ top-k rows
static_assert(DSPARK_MAX_TOPK <= kTpTab, "a shard's candidates fit in its table");
constexpr int kTkCand = kTpMaxShards * DSPARK_MAX_TOPK;  // the leader's merge buffer

struct TkShared {
  uint32_t hist[256];
  uint32_t r32[32];
  float rf[32];
  uint32_t sel_digit, sel_above, sel_equal;
  uint32_t n;
};

// Block-wide radix select (8-bit digits, most significant first): the r-th
// largest value of val(i) over i < n with take(i) (1 <= r <= the count);
// *above: the entries with a larger value, *equal: those equal to it.  The
// lanes of a warp that fall in one bin add to it with one atomic.  Called by
// every thread of the block; the result is uniform.
template <int kBits, typename T, typename Val, typename Take>
__device__ T radix_select_desc(int n, uint32_t r, Val val, Take take, TkShared& sh,
                               uint32_t* above, uint32_t* equal) {
  const int lane = threadIdx.x & 31;
  T prefix = 0, mask = 0;
  uint32_t above_acc = 0, eq = 0;
  for (int shift = kBits - 8; shift >= 0; shift -= 8) {
    __syncthreads();
    sh.hist[threadIdx.x] = 0u;  // kTpThr == 256 bins
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kTpThr) {
      const int i = i0 + (int)threadIdx.x;
      uint32_t bin = 0xFFFFFFFFu;
      if (i < n && take(i)) {
        const T v = val(i);
        if ((v & mask) == prefix) bin = (uint32_t)(v >> shift) & 255u;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (bin != 0xFFFFFFFFu && lane == __ffs(peers) - 1)
        atomicAdd(&sh.hist[bin], (uint32_t)__popc(peers));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l holds bins 255 - 8l down to 248 - 8l
      uint32_t c[8], t = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sh.hist[255 - 8 * lane - j];
        t += c[j];
      }
      uint32_t incl = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      const uint32_t excl = incl - t;
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
    const uint32_t ab = sh.sel_above;
    eq = sh.sel_equal;
    r -= ab;
    above_acc += ab;
    prefix |= (T)sh.sel_digit << shift;
    mask |= (T)255u << shift;
  }
  *above = above_acc;
  *equal = eq;
  return prefix;
}

// Order key of y for the support: larger y, larger key; -0 taken as +0.
__device__ __forceinline__ uint32_t tk_key(float y) { return float_key(__fadd_rn(y, 0.0f)); }

// Each rank: validity flags and max of its shard (as the dense rows), then its
// local top k by (y desc, id asc) -- every finite element when it holds at
// most k -- sent as (key << 32 | id) records.
__global__ void __launch_bounds__(kTpThr) tp_topk_local_kernel(TpParams p) {
  __shared__ TkShared sh;
  const Shard d = shard_of(p);
  TpRow& w = p.ws[d.row];
  bool badT;
  const float invT = inv_temp(p, d.row, &badT);
  float mx = -INFINITY;
  uint32_t fl = 0, nfin = 0;
  if (!badT)
    for (int v = d.lo + threadIdx.x; v < d.hi; v += kTpThr) {
      const char* xrow = reinterpret_cast<const char*>(p.x) +
                         (int64_t)d.row * p.ld * (p.dtype == DSPARK_F32 ? 4 : 2);
      const float x = load_logit(xrow, p.dtype, v);
      if (!(x < INFINITY)) fl |= 1u;  // NaN or +inf
      const float y = invT == 1.0f ? x : __fmul_rn(x, invT);
      if (fabsf(y) == INFINITY && fabsf(x) < INFINITY) fl |= 1u;  // overflow
      if (y > -INFINITY && y < INFINITY) {
        fl |= 2u;
        ++nfin;
        mx = fmaxf(mx, y);
      }
    }
  mx = block_reduce(mx, OpMaxNaNTp(), sh.rf);
  fl = block_reduce(fl, OpOrU32(), sh.r32);
  nfin = block_reduce(nfin, OpAddU32(), sh.r32);
  if (threadIdx.x == 0) {
    w.mx[d.s] = mx;
    w.fl[d.s] = fl;
    sh.n = 0u;
  }
  __syncthreads();
  const int k = p.top_k;
  uint32_t nc = 0;
  if (!badT && !(fl & 1u) && nfin > 0u) {
    auto key_at = [&](int i, uint32_t* key) -> bool {  // i: position in the shard
      const float y = y_of(p, d.row, d.lo + i, invT);
      *key = tk_key(y);
      return y > -INFINITY;
    };
    const int n = d.hi - d.lo;
    uint32_t T = 0u, need = 0xFFFFFFFFu;  // take key > T, and `need` lowest ids at T
    if (nfin > (uint32_t)k) {
      uint32_t above, equal;
      T = radix_select_desc<32, uint32_t>(
          n, (uint32_t)k,
          [&](int i) {
            uint32_t key;
            key_at(i, &key);
            return key;
          },
          [&](int i) {
            uint32_t key;
            return key_at(i, &key);
          },
          sh, &above, &equal);
      need = (uint32_t)k - above;
    }
    // the candidates, in id order (ties at T: the lowest ids)
    uint32_t base = 0;
    for (int i0 = 0; i0 < n; i0 += kTpThr) {
      const int i = i0 + (int)threadIdx.x;
      uint32_t key = 0u;
      const bool fin = i < n && key_at(i, &key);
      const bool at = fin && nfin > (uint32_t)k && key == T;
      const bool hi = fin && (nfin <= (uint32_t)k || key > T);
      uint32_t tot;
      const uint32_t incl = block_inclusive_scan(at ? 1u : 0u, sh.r32, &tot);
      if (hi || (at && base + incl <= need)) {
        const uint32_t j = atomicAdd(&sh.n, 1u);
        w.tab_key[d.s][j] = ((uint64_t)key << 32) | (uint32_t)(d.lo + i);
      }
      base += tot;
      __syncthreads();
    }
    nc = sh.n;
  }
  if (threadIdx.x == 0) w.nc[d.s] = nc;
}

// The leader of each row: the global top k of the ranks' candidates, the
// allocation on it, the outputs and the draw.
__global__ void __launch_bounds__(kTpThr) tp_topk_merge_kernel(TpParams p) {
  __shared__ TkShared sh;
  __shared__ SupShared ssh;
  extern __shared__ __align__(16) unsigned char dyn[];
  uint64_t* cand = reinterpret_cast<uint64_t*>(dyn);                   // [kTkCand]
  uint32_t* skeys = reinterpret_cast<uint32_t*>(cand + kTkCand);       // [top_k]
  int32_t* sids = reinterpret_cast<int32_t*>(skeys + DSPARK_MAX_TOPK); // [top_k]
  unsigned char* scratch = reinterpret_cast<unsigned char*>(sids + DSPARK_MAX_TOPK);
  const int row = blockIdx.x;
  const TpRow& w = p.ws[row];
  const int k = p.top_k;
  bool badT;
  inv_temp(p, row, &badT);
  float m;
  const int st = row_state(p, w, badT, &m);
  int n = 0;
  if (st == DSPARK_ST_OK) {
    for (int s = 0; s < p.n_sh; ++s) {
      const int ns = (int)w.nc[s];
      for (int i = threadIdx.x; i < ns; i += kTpThr) cand[n + i] = w.tab_key[s][i];
      n += ns;
    }
  }
  if (threadIdx.x == 0) sh.n = 0u;
  __syncthreads();
  int ns = min(n, k);
  if (st == DSPARK_ST_OK) {
    // the k largest (key, -id): a record's order value is key << 32 | ~id
    auto ord = [&](int i) { return cand[i] ^ 0xFFFFFFFFull; };
    uint64_t C = 0ull;
    if (n > k) {
      uint32_t above, equal;
      C = radix_select_desc<64, uint64_t>(n, (uint32_t)k, ord, [](int) { return true; }, sh,
                                          &above, &equal);
    }
    for (int i = threadIdx.x; i < n; i += kTpThr)
      if (ord(i) >= C) {
        const uint32_t j = atomicAdd(&sh.n, 1u);  // exactly min(n, k) qualify
        skeys[j] = (uint32_t)(cand[i] >> 32);
        sids[j] = (int32_t)(uint32_t)cand[i];
      }
    __syncthreads();
  }
  uint32_t D = 0;
  if (p.tokens) {
    const int b = row / p.depth, j = row % p.depth;
    const uint32_t req = p.request_ids ? p.request_ids[b] : (uint32_t)b;
    D = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_PROPOSAL) >> 8;
  }
  support_alloc_emit(st, ns, k, skeys, sids, scratch, ssh, p.counts + (int64_t)row * k,
                     p.ids + (int64_t)row * k, p.nnz + row, p.status + row,
                     p.tokens ? p.tokens + row : nullptr, D);
}

constexpr int kTkMergeSmem =
    kTkCand * 8 + DSPARK_MAX_TOPK * 8 + kSupScratch;  // candidates, support, scratch

}  // namespace

int64_t q_sharded_workspace_bytes(int n_rows) { return (int64_t)n_rows * sizeof(TpRow); }

cudaError_t launch_q_sharded(const void* x, int dtype, int64_t ld, int B, int depth, int V,
                             int n_sh, const float* temperature, int top_k, uint64_t seed,
                             const uint32_t* request_ids, uint32_t* counts, int32_t* ids,
                             int32_t* nnz, int32_t* tokens, int32_t* status, void* workspace,
                             cudaStream_t stream) {
  TpParams p{x,           dtype,  ld,     V,      n_sh,
             depth,       temperature, seed, request_ids, counts,
             tokens,      status, static_cast<TpRow*>(workspace), top_k, ids, nnz};
  const int rows = B * depth;
  const int units = rows * n_sh;
  if (top_k > 0) {
    cudaError_t e = cudaFuncSetAttribute(tp_topk_merge_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTkMergeSmem);
    if (e != cudaSuccess) return e;
    tp_topk_local_kernel<<<units, kTpThr, 0, stream>>>(p);
    tp_topk_merge_kernel<<<rows, kTpThr, kTkMergeSmem, stream>>>(p);
    return cudaGetLastError();
  }
  tp_max_kernel<<<units, kTpThr, 0, stream>>>(p);
  tp_weights_kernel<<<units, kTpThr, 0, stream>>>(p);
  tp_floors_kernel<<<units, kTpThr, 0, stream>>>(p);
  tp_grant_kernel<<<units, kTpThr, 0, stream>>>(p);
  tp_threshold_kernel<<<rows, kTpThr, 0, stream>>>(p);
  tp_ties_kernel<<<units, kTpThr, 0, stream>>>(p);
  if (tokens) tp_draw_kernel<<<units, kTpThr, 0, stream>>>(p);
  return cudaGetLastError();
}

DSPARK_CHECK_COLLECTOR(tp)

}  // namespace dspark
