// q_build.cu -- dyadic24-standard-v1 q construction (and, optionally, the
// draft draw from it), one 8-CTA thread-block cluster per draft row
// ("PP1 q transport and scheduling design", Distribution contract and
// precision: proposal construction, sparse top-k, integer draw).
//
// Each CTA holds one eighth of the row in shared memory for the whole build;
// the slice arrives by TMA bulk copies, so the row is read from HBM once.
// Cluster-wide values (row max, weight sum, floor sum, remainder histograms)
// are exchanged through distributed shared memory: each CTA publishes its
// partial, and after a cluster barrier every CTA combines all of them in rank
// order, so all hold identical values.
//
// Dense rows, passes over the resident slice:
//   A  validate, y = x * RN(1/T) in place, row max
//   B  E = floor(exp_ds(y - m) * 2^40) (as an exact float) in place, S = sum E
//   C  a = RN64(E * RN64(2^24 / RN64(S))) split into floor f and fraction r.
//      With k = khi + klo + d (khi = RN32(k), klo = RN32(k - khi),
//      |d| <= 2^-48 k), p1 + e1 = E * khi exactly (fma), p2 = RN32(E * klo):
//      a = p1 + e1 + p2 + eta with |eta| <= 2^-46.9 a (including the FP64
//      rounding of a).  With f0 = floor(p1), fr = RN(RN(p1 - f0) + RN(e1 + p2)),
//      fi = floor(fr), frc = fr - fi:  |(a - f0 - fi) - frc| <= 2^-24 (1 +
//      |e1 + p2|) + 2^-45.9 a <= 2^-24 + 2^-45 p1.  So when 4096 frc is
//      farther than 2^-12 + 2^-33 p1 from every integer, floor(a) = f0 + fi,
//      r > 0 and floor(4096 r) = floor(4096 frc).  The few other elements
//      take the exact integer path afterwards.  Packed (f, r > 0, bin) in
//      place; 4096-bin histogram; F = sum f.
//   D  the members of the bin holding the grant threshold: exact fractions,
//      ranked by (fraction desc, id asc)
//   E  counts = f + grant, written with 128-bit stores; total checked == M;
//      optionally the draft draw over the counts kept in shared memory.
// Top-k rows: a 4096-bin histogram of the distance to the row max (1/64-nat
// bins, monotone in y) finds the bins holding the k largest; those candidates
// are gathered in the cluster's first CTA, sorted by (y desc, id asc), and
// the first k are allocated with FP64.
#include "common.cuh"

namespace dspark {

constexpr int kQCluster = 8;
constexpr int kQThreads = 512;
constexpr int kHistBins = 4096;
constexpr int kCandCap = 256;       // members of the threshold bin, per CTA
constexpr int kEscCap = 48;         // floors >= 2^19 (at most 32 per row)
constexpr int kUncCap = 1024;       // elements left to the exact split, per CTA
constexpr int kSupCap = 1024;       // support candidates per CTA (aliases the histogram)
constexpr int kGatherCap = 2048;    // support candidates per row (leader)
constexpr int kAllCap = 1024;       // members of the threshold bin, per row
constexpr int kChunkMax = DSPARK_MAX_V / kQCluster;  // 16384 elements per CTA
constexpr int kTmaChunks = 4;
constexpr uint32_t kEscape = 0xFFFFE000u;            // f field all ones
constexpr uint32_t kFMaxPacked = (1u << 19) - 1u;    // f below this is packed inline

struct QParams {
  const void* x;
  int dtype;
  int64_t ld;
  int n_rows;
  int V;
  const float* temperature;
  int top_k;
  uint32_t* counts;
  int32_t* ids;
  int32_t* nnz;
  int32_t* status;
  int chunk;  // elements per CTA, multiple of 4
  // optional fused draft draw (tokens == nullptr: none)
  int32_t* tokens;
  uint64_t seed;
  const uint32_t* request_ids;
  int depth;
};

// Scalars each CTA publishes to its cluster peers.
struct PubS {
  float max;
  uint32_t flags;  // bit0 nonfinite, bit1 internal, bit2 timeout
  uint32_t nfinite;
  uint32_t npos;
  uint64_t S;
  uint64_t F;
  uint64_t csum;
  uint64_t kmin, kmax;
  uint32_t ncand;
  uint32_t n_eq;    // ordered_ranks: matching elements of this CTA
  uint32_t nsup;
  uint32_t n_grant; // members of this CTA granted a ticket (separate from
                    // n_eq: a peer may still read n_eq when this is written)
};

struct QPub {
  PubS s;
  uint32_t coarse[64];
};

struct Cand {
  uint64_t key;
  int32_t v;
  int32_t s;
};

struct Esc {
  int32_t s;
  uint32_t f;
  uint32_t bucket;
  uint32_t pos;
};

struct Sup {
  uint32_t key;
  int32_t v;
  float y;
  uint32_t pad;
};

struct QShared {
  union {  // one of: the histogram, the support candidates, all members
    uint32_t hist[kHistBins];
    Sup sup[kSupCap];
    Cand allc[kAllCap];
  };
  uint32_t grant_bits[kChunkMax / 32 + 2];
  Cand cand[kCandCap];
  Esc esc[kEscCap];
  int32_t unc[kUncCap];
  QPub pub;
  PubS peers[kQCluster];  // local copy of every CTA's published scalars
  int timeout;
  uint64_t mbar[kTmaChunks];
  uint32_t gcoarse[64];
  uint32_t gfine[64];
  uint64_t red64[32];
  uint32_t red32[32];
  float redf[32];
  uint32_t n_cand, n_esc, n_sup, n_unc;
  int sel_bin;
  uint32_t sel_above, sel_count;
  uint32_t scan_base;
  int found;
  uint32_t grants[kQCluster];
  uint64_t peers_csum[kQCluster];
  uint32_t segsum[32];
  uint64_t mk;
  int ek;
  float khi, klo;
};

// Leader-only arrays of the sparse allocation (aliased onto the slice).
struct SparseEntry {
  double r;
  uint64_t E;
  int32_t v;
  uint32_t f;
  float y;
  uint32_t c;
};

__device__ __forceinline__ void set_bit(uint32_t* bits, int s) {
  atomicOr(&bits[s >> 5], 1u << (s & 31));
}
__device__ __forceinline__ bool get_bit(const uint32_t* bits, int s) {
  return (bits[s >> 5] >> (s & 31)) & 1u;
}

__device__ __forceinline__ uint32_t pack(uint32_t f, uint32_t pos, uint32_t bucket) {
  return (f << 13) | (pos << 12) | bucket;
}

// After a cluster barrier: eight threads copy every CTA's published scalars
// into this CTA's shared memory; the block then reads them locally.
__device__ __forceinline__ void gather_pubs(cg::cluster_group& cluster, QShared& sh) {
  if (threadIdx.x < kQCluster)
    sh.peers[threadIdx.x] = cluster.map_shared_rank(&sh.pub, threadIdx.x)->s;
  __syncthreads();
}

__device__ void publish_coarse(QShared& sh, int nbins) {
  const int per = nbins / 64;
  for (int c = threadIdx.x; c < 64; c += blockDim.x) {
    uint32_t s = 0;
    for (int i = 0; i < per; ++i) s += sh.hist[c * per + i];
    sh.pub.coarse[c] = s;
  }
}

// Warp 0: the bin b in g[0..63] where the count accumulated from bin 63 down
// reaches `need` (bin 0 if it never does); *above = the count in the bins
// above b.  At most one bin satisfies above(b) < need <= above(b) + g[b].
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
  const uint32_t ab1 = suf - pair;  // count above bin 2*lane+1
  const uint32_t ab0 = ab1 + g1;    // count above bin 2*lane
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

// After a cluster barrier that published hist / coarse: the bin b where the
// cluster-wide count, accumulated from the top bin down, reaches `need`
// (1 <= need <= total).  All CTAs agree.  The histograms must not change
// until every CTA has passed its next cluster barrier.
__device__ void select_from_cluster(cg::cluster_group& cluster, QShared& sh, int nbins,
                                    uint32_t need) {
  const int per = nbins / 64;
  if (threadIdx.x < 64) {
    uint32_t v[kQCluster];
#pragma unroll
    for (int r = 0; r < kQCluster; ++r)
      v[r] = cluster.map_shared_rank(&sh.pub, r)->coarse[threadIdx.x];
    uint32_t g = 0;
#pragma unroll
    for (int r = 0; r < kQCluster; ++r) g += v[r];
    sh.gcoarse[threadIdx.x] = g;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    int sb;
    uint32_t above;
    warp_select64(sh.gcoarse, need, &sb, &above);
    if (threadIdx.x == 0) {
      sh.sel_bin = sb;
      sh.sel_above = above;
    }
  }
  __syncthreads();
  const int sb = sh.sel_bin;
  if (threadIdx.x < 64) {
    uint32_t g = 0;
    if (threadIdx.x < per) {
      uint32_t v[kQCluster];
#pragma unroll
      for (int r = 0; r < kQCluster; ++r)
        v[r] = cluster.map_shared_rank(&sh.hist[0], r)[sb * per + threadIdx.x];
#pragma unroll
      for (int r = 0; r < kQCluster; ++r) g += v[r];
    }
    sh.gfine[threadIdx.x] = g;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    int b;
    uint32_t above;
    warp_select64(sh.gfine, need - sh.sel_above, &b, &above);
    if (threadIdx.x == 0) {
      sh.sel_count = sh.gfine[b];
      sh.sel_above = sh.sel_above + above;
      sh.sel_bin = sb * per + b;
    }
  }
  __syncthreads();
}

// Rank, in id order over the whole cluster, of every element for which
// pred(s) holds; calls fn(s, rank).  One cluster barrier.
template <typename Pred, typename Fn>
__device__ void ordered_ranks(cg::cluster_group& cluster, QShared& sh, int ngroups, Pred pred,
                              Fn fn) {
  uint32_t cnt = 0;
  for (int g = threadIdx.x; g < ngroups; g += blockDim.x)
    for (int i = 0; i < 4; ++i) cnt += pred(4 * g + i) ? 1u : 0u;
  cnt = block_reduce(cnt, OpAddU32(), sh.red32);
  if (threadIdx.x == 0) sh.pub.s.n_eq = cnt;
  cluster.sync();
  gather_pubs(cluster, sh);
  if (threadIdx.x == 0) {
    uint32_t base = 0;
    const int me = (int)cluster.block_rank();
    for (int r = 0; r < me; ++r) base += sh.peers[r].n_eq;
    sh.scan_base = base;
  }
  __syncthreads();
  uint32_t base = sh.scan_base;
  for (int t0 = 0; t0 < ngroups; t0 += blockDim.x) {
    const int g = t0 + threadIdx.x;
    uint32_t mine = 0;
    bool hit[4] = {false, false, false, false};
    if (g < ngroups)
      for (int i = 0; i < 4; ++i) {
        hit[i] = pred(4 * g + i);
        mine += hit[i] ? 1u : 0u;
      }
    uint32_t total;
    const uint32_t incl = block_inclusive_scan(mine, sh.red32, &total);
    uint32_t rank = base + incl - mine;
    for (int i = 0; i < 4; ++i)
      if (hit[i]) fn(4 * g + i, rank++);
    base += total;
    __syncthreads();
  }
}

// In-place bitonic sort of n (a power of two) entries in shared memory by
// `less` (ascending).  Every thread of the block must call it.
template <typename T, typename Less>
__device__ void bitonic_sort(T* a, int n, Less less) {
  for (int kx = 2; kx <= n; kx <<= 1)
    for (int j = kx >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int l = i ^ j;
        if (l > i) {
          const bool up = ((i & kx) == 0);
          if (up ? less(a[l], a[i]) : less(a[i], a[l])) {
            const T t = a[i];
            a[i] = a[l];
            a[l] = t;
          }
        }
      }
      __syncthreads();
    }
}

// Exact split (floor, r > 0, bin) of a = RN64(E * k) by integer arithmetic.
__device__ __forceinline__ void exact_pack(float Ef, uint64_t mk, int ek, uint32_t* f_out,
                                           uint32_t* pos_out, uint32_t* bucket_out) {
  uint32_t Ei;
  int se;
  weight_split_ef(Ef, &Ei, &se);
  const AllocSplit a = alloc_split(Ei, se, mk, ek);
  *f_out = a.f;
  *pos_out = (a.rnum != 0ull) ? 1u : 0u;
  *bucket_out = *pos_out ? frac_bucket(a) : 0u;
}

__global__ void __cluster_dims__(kQCluster, 1, 1) __launch_bounds__(kQThreads, 2)
    q_build_kernel(QParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ QShared sh;
  extern __shared__ __align__(128) float sl[];
  uint32_t* slu = reinterpret_cast<uint32_t*>(sl);

  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.x / kQCluster;
  const int V = p.V;
  const int lo = rank * p.chunk;
  const int hi = min(V, lo + p.chunk);
  const int n = max(0, hi - lo);
  const int esz = (p.dtype == DSPARK_F32) ? 4 : 2;
  const char* xrow = reinterpret_cast<const char*>(p.x) + (int64_t)row * p.ld * esz;
  // offset of element lo inside its 4-element group of the source row
  const int off = (int)((reinterpret_cast<uintptr_t>(xrow + (int64_t)lo * esz) / esz) & 3);
  const int ngroups = (off + n + 3) >> 2;
  const bool sparse = p.top_k > 0;
  const int tid = threadIdx.x;

  // ---- temperature (identical decision in every CTA)
  const float T = p.temperature ? p.temperature[row] : 1.0f;
  const float invT = __frcp_rn(T);
  const bool bad_T = !(isfinite(T) && T > 0.0f) || !(isfinite(invT) && invT >= 0x1p-126f);
  const bool scale = (invT != 1.0f);

  // ---- the slice: full 16-byte groups by TMA, partial edge groups by plain loads
  const bool use_tma = (p.dtype == DSPARK_F32) && !bad_T;
  const int g_first = (off == 0) ? 0 : 1;
  const int g_last = (off + n) / 4 - 1;  // last group fully inside the slice
  const int n_int = max(0, g_last - g_first + 1);
  if (tid == 0) {
    sh.n_cand = 0;
    sh.n_esc = 0;
    sh.n_sup = 0;
    sh.n_unc = 0;
    sh.timeout = 0;
    if (use_tma && n_int > 0) {
      for (int c = 0; c < kTmaChunks; ++c) mbar_init(&sh.mbar[c], 1);
      mbar_init_fence();
    }
  }
  for (int i = tid; i < kChunkMax / 32 + 2; i += blockDim.x) sh.grant_bits[i] = 0u;
  __syncthreads();
  const float* xbase = reinterpret_cast<const float*>(xrow) + lo - off;  // group 0 start
  int chunk_lo[kTmaChunks + 1];
  for (int c = 0; c <= kTmaChunks; ++c)
    chunk_lo[c] = g_first + (int)(((int64_t)n_int * c) / kTmaChunks);
  if (use_tma && n_int > 0 && tid == 0) {
    for (int c = 0; c < kTmaChunks; ++c) {
      const int g0 = chunk_lo[c], g1 = chunk_lo[c + 1];
      const uint32_t bytes = (uint32_t)(g1 - g0) * 16u;
      mbar_arrive_expect_tx(&sh.mbar[c], bytes);
      if (bytes) tma_load_bulk(sl + 4 * g0, xbase + 4 * g0, bytes, &sh.mbar[c]);
    }
  }
  if (!bad_T) {
    if (use_tma) {
      // edge groups (partial) by plain loads, -inf padding
      for (int i = tid; i < 8; i += blockDim.x) {
        const int g = (i < 4) ? 0 : ngroups - 1;
        if (g < 0 || (g >= g_first && g <= g_last)) continue;
        const int s = 4 * g + (i & 3);
        sl[s] = (s >= off && s < off + n) ? __ldg(xbase + s) : -INFINITY;
      }
    } else {
      for (int g = tid; g < ngroups; g += blockDim.x)
        for (int i = 0; i < 4; ++i) {
          const int s = 4 * g + i;
          sl[s] = (s >= off && s < off + n) ? load_logit(xrow, p.dtype, (int64_t)(lo - off + s))
                                            : -INFINITY;
        }
    }
  }
  __syncthreads();

  // ---- pass A: validate, y, max
  uint32_t flags = 0, nfin = 0;
  float mx = -INFINITY;
  if (!bad_T) {
    for (int c = 0; c < kTmaChunks; ++c) {
      int g0 = chunk_lo[c], g1 = chunk_lo[c + 1];
      if (c == 0) g0 = 0;                       // the head edge group
      if (c == kTmaChunks - 1) g1 = ngroups;    // the tail edge group
      if (use_tma && n_int > 0) {
        if (tid == 0 && !mbar_wait_bounded(&sh.mbar[c], 0)) sh.timeout = 1;
        __syncthreads();
      }
      for (int g = g0 + tid; g < g1; g += blockDim.x) {
        float4 v = reinterpret_cast<const float4*>(sl)[g];
        float xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x = xv[i];
          if (!(x < INFINITY)) flags |= 1u;  // NaN or +inf
          float y = x;
          if (scale) {
            y = __fmul_rn(x, invT);
            if ((x > -INFINITY) && !(y > -INFINITY && y < INFINITY)) flags |= 1u;
          }
          xv[i] = y;
          mx = fmaxf(mx, y);
          nfin += (y > -INFINITY) ? 1u : 0u;
        }
        if (scale) reinterpret_cast<float4*>(sl)[g] = make_float4(xv[0], xv[1], xv[2], xv[3]);
      }
    }
  }
  flags = block_reduce(flags, OpOrU32(), sh.red32);
  nfin = block_reduce(nfin, OpAddU32(), sh.red32);
  mx = block_reduce(mx, OpMaxF(), sh.redf);
  if (tid == 0) {
    sh.pub.s.flags = flags | (sh.timeout ? 4u : 0u);
    sh.pub.s.nfinite = nfin;
    sh.pub.s.max = mx;
  }
  cluster.sync();  // S1
  gather_pubs(cluster, sh);
  uint32_t nfin_all = 0, flags_all = 0;
  float m = -INFINITY;
  for (int r = 0; r < kQCluster; ++r) {
    nfin_all += sh.peers[r].nfinite;
    flags_all |= sh.peers[r].flags;
    m = fmaxf(m, sh.peers[r].max);
  }
  int status = DSPARK_ST_OK;
  if (bad_T) status = DSPARK_ST_BAD_TEMPERATURE;
  else if (flags_all & 4u) status = DSPARK_ST_TIMEOUT;
  else if (flags_all & 1u) status = DSPARK_ST_NONFINITE;
  else if (m == -INFINITY) status = DSPARK_ST_ZERO_MASS;

  // ------------------------------------------------------------ top-k rows
  if (sparse) {
    if (status != DSPARK_ST_OK) {
      cluster.sync();  // peers may still read this CTA's pub
      if (rank == 0) {
        for (int i = tid; i < p.top_k; i += blockDim.x) {
          p.ids[(int64_t)row * p.top_k + i] = -1;
          p.counts[(int64_t)row * p.top_k + i] = 0u;
        }
        if (tid == 0) {
          p.nnz[row] = 0;
          p.status[row] = status;
          if (p.tokens) p.tokens[row] = -1;
        }
      }
      return;
    }
    const uint32_t kk = min((uint32_t)p.top_k, nfin_all);
    const bool all_finite = (kk == nfin_all);
    // histogram of the distance to the max on a 1/64-nat grid, bins reversed
    // so that the largest y sit in the top bin (monotone in y, so a bin cut
    // keeps every element at least as large as any element it drops)
    auto dbin = [&](float y) -> uint32_t {
      const float d = __fmul_rn(__fsub_rn(m, y), 64.0f);
      return (d < 4095.0f) ? 4095u - (uint32_t)d : 0u;
    };
    uint32_t b1 = 0, cand_total = nfin_all, my_cand = 0;
    if (!all_finite) {
      for (int i = tid; i < kHistBins; i += blockDim.x) sh.hist[i] = 0u;
      __syncthreads();
      for (int g = tid; g < ngroups; g += blockDim.x) {
        const float4 v = reinterpret_cast<const float4*>(sl)[g];
        const float yy[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (yy[i] > -INFINITY) atomicAdd(&sh.hist[dbin(yy[i])], 1u);
      }
      __syncthreads();
      publish_coarse(sh, kHistBins);
      cluster.sync();
      select_from_cluster(cluster, sh, kHistBins, kk);
      b1 = (uint32_t)sh.sel_bin;
      cand_total = sh.sel_above + sh.sel_count;
      for (int i = tid; i < kHistBins; i += blockDim.x)
        if ((uint32_t)i >= b1) my_cand += sh.hist[i];
      my_cand = block_reduce(my_cand, OpAddU32(), sh.red32);
    } else {
      my_cand = nfin;
    }
    if (tid == 0) sh.pub.s.ncand = my_cand;
    cluster.sync();  // S2: histograms no longer read remotely
    gather_pubs(cluster, sh);
    bool gather = cand_total <= (uint32_t)kGatherCap;
    for (int r = 0; r < kQCluster; ++r) gather = gather && sh.peers[r].ncand <= (uint32_t)kSupCap;
    auto push = [&](int s, uint32_t key) {
      const uint32_t i = atomicAdd(&sh.n_sup, 1u);
      if (i < kSupCap) {
        sh.sup[i].key = key;
        sh.sup[i].v = lo + s - off;
        sh.sup[i].y = sl[s];
      }
    };
    if (gather) {
      // candidates: every finite element of a bin at or above b1
      for (int g = tid; g < ngroups; g += blockDim.x)
        for (int i = 0; i < 4; ++i) {
          const int s = 4 * g + i;
          const float y = sl[s];
          if (!(y > -INFINITY)) continue;
          if (all_finite || dbin(y) >= b1) push(s, float_key(y));
        }
    } else {
      // too many candidates: exact radix select of the k-th largest float key
      // (12, 12 and 8 bits), then the lowest ids among the elements holding
      // that key
      uint32_t prefix = 0, need = kk, n_eq_all = 0;
      const int shifts[3] = {20, 8, 0};
      const int widths[3] = {12, 12, 8};
      for (int lvl = 0; lvl < 3; ++lvl) {
        const int nb = 1 << widths[lvl];
        for (int i = tid; i < nb; i += blockDim.x) sh.hist[i] = 0u;
        __syncthreads();
        const int hs = shifts[lvl] + widths[lvl];
        for (int g = tid; g < ngroups; g += blockDim.x)
          for (int i = 0; i < 4; ++i) {
            const float y = sl[4 * g + i];
            if (!(y > -INFINITY)) continue;
            const uint32_t key = float_key(y);
            if (hs < 32 && (key >> hs) != prefix) continue;
            atomicAdd(&sh.hist[(key >> shifts[lvl]) & (nb - 1)], 1u);
          }
        __syncthreads();
        publish_coarse(sh, nb);
        cluster.sync();
        select_from_cluster(cluster, sh, nb, need);
        need -= sh.sel_above;
        n_eq_all = sh.sel_count;
        prefix = (prefix << widths[lvl]) | (uint32_t)sh.sel_bin;
        cluster.sync();
      }
      const uint32_t thr = prefix, need_eq = need;
      for (int g = tid; g < ngroups; g += blockDim.x)
        for (int i = 0; i < 4; ++i) {
          const int s = 4 * g + i;
          const float y = sl[s];
          if (!(y > -INFINITY)) continue;
          const uint32_t key = float_key(y);
          if (key > thr || (key == thr && need_eq >= n_eq_all)) push(s, key);
        }
      if (need_eq < n_eq_all) {
        __syncthreads();
        ordered_ranks(
            cluster, sh, ngroups,
            [&](int s) -> bool {
              if (s < off || s >= off + n) return false;
              const float y = sl[s];
              return (y > -INFINITY) && float_key(y) == thr;
            },
            [&](int s, uint32_t rk) {
              if (rk < need_eq) push(s, thr);
            });
      }
    }
    __syncthreads();
    if (tid == 0) sh.pub.s.nsup = sh.n_sup;
    cluster.sync();  // S3: candidate lists complete everywhere

    if (rank == 0) {
      gather_pubs(cluster, sh);
      __shared__ uint32_t base_of[kQCluster + 1];
      __shared__ int bad_gather;
      if (tid == 0) {
        uint32_t acc = 0;
        bad_gather = 0;
        for (int r = 0; r < kQCluster; ++r) {
          base_of[r] = acc;
          const uint32_t ns = sh.peers[r].nsup;
          if (ns > (uint32_t)kSupCap) bad_gather = 1;
          acc += ns;
        }
        base_of[kQCluster] = acc;
        if (acc > (uint32_t)kGatherCap || acc < kk || (!gather && acc != kk)) bad_gather = 1;
      }
      __syncthreads();
      const int ncand = bad_gather ? 0 : (int)base_of[kQCluster];
      // gather the candidates into the leader's slice memory and sort them by
      // (key desc, id asc): the first kk form the support
      Sup* cl = reinterpret_cast<Sup*>(sl);
      for (int r = 0; r < kQCluster && !bad_gather; ++r) {
        const Sup* rs = cluster.map_shared_rank(&sh.sup[0], r);
        const int cnt = (int)(base_of[r + 1] - base_of[r]);
        for (int i = tid; i < cnt; i += blockDim.x) cl[base_of[r] + i] = rs[i];
      }
      int np2 = 1;
      while (np2 < ncand) np2 <<= 1;
      for (int i = ncand + tid; i < np2; i += blockDim.x) {
        Sup e;
        e.key = 0u;
        e.v = 0x7FFFFFFF;
        e.y = -INFINITY;
        e.pad = 0u;
        cl[i] = e;
      }
      __syncthreads();
      if (ncand > 1)
        bitonic_sort(cl, np2, [](const Sup& a, const Sup& b) {
          return a.key > b.key || (a.key == b.key && a.v < b.v);
        });
      const int nsup = bad_gather ? 0 : (int)kk;
      SparseEntry* ent = reinterpret_cast<SparseEntry*>(
          reinterpret_cast<char*>(sl) + (size_t)kGatherCap * sizeof(Sup));
      for (int i = tid; i < nsup; i += blockDim.x) {
        SparseEntry e;
        e.v = cl[i].v;
        e.y = cl[i].y;
        ent[i] = e;
      }
      __syncthreads();
      // weights, sum, FP64 allocation (order-independent)
      uint64_t S = 0;
      for (int i = tid; i < nsup; i += blockDim.x) {
        const float e = weight_float(__fsub_rn(ent[i].y, m));
        ent[i].E = weight_u64(e);
        S += ent[i].E;
      }
      S = block_reduce(S, OpAddU64(), sh.red64);
      __shared__ double kd_sh;
      if (tid == 0) kd_sh = __ddiv_rn(16777216.0, __ull2double_rn(S));
      __syncthreads();
      const double kd = kd_sh;
      uint64_t F = 0;
      uint32_t npos = 0;
      for (int i = tid; i < nsup; i += blockDim.x) {
        const double a = __dmul_rn(__ull2double_rn(ent[i].E), kd);
        const double f = floor(a);
        ent[i].f = (uint32_t)f;
        ent[i].r = __dsub_rn(a, f);
        F += (uint64_t)ent[i].f;
        npos += (ent[i].r > 0.0) ? 1u : 0u;
      }
      F = block_reduce(F, OpAddU64(), sh.red64);
      npos = block_reduce(npos, OpAddU32(), sh.red32);
      int st = bad_gather ? DSPARK_ST_INTERNAL : DSPARK_ST_OK;
      if (st == DSPARK_ST_OK &&
          (F == 0 || F > (uint64_t)kM || (uint64_t)kM - F > (uint64_t)npos))
        st = DSPARK_ST_ALLOC_INCONSISTENT;
      const uint32_t R = (st == DSPARK_ST_OK) ? (uint32_t)((uint64_t)kM - F) : 0u;
      int np2s = 1;
      while (np2s < nsup) np2s <<= 1;
      for (int i = nsup + tid; i < np2s; i += blockDim.x) {
        SparseEntry e;
        e.v = 0x7FFFFFFF;
        e.r = -1.0;
        e.E = 0;
        e.f = 0;
        e.y = -INFINITY;
        e.c = 0;
        ent[i] = e;
      }
      __syncthreads();
      bitonic_sort(ent, np2s, [](const SparseEntry& a, const SparseEntry& b) {
        return a.r > b.r || (a.r == b.r && a.v < b.v);
      });
      for (int i = tid; i < nsup; i += blockDim.x)
        ent[i].c = ent[i].f + ((uint32_t)i < R ? 1u : 0u);
      __syncthreads();
      bitonic_sort(ent, np2s, [](const SparseEntry& a, const SparseEntry& b) { return a.v < b.v; });
      uint64_t csum = 0;
      for (int i = tid; i < nsup; i += blockDim.x) csum += ent[i].c;
      csum = block_reduce(csum, OpAddU64(), sh.red64);
      if (st == DSPARK_ST_OK && csum != (uint64_t)kM) st = DSPARK_ST_ALLOC_INCONSISTENT;
      int32_t* ids = p.ids + (int64_t)row * p.top_k;
      uint32_t* cnt = p.counts + (int64_t)row * p.top_k;
      uint32_t written = 0;
      // optional draft draw: the first support id, in id order, whose
      // inclusive cumulative count exceeds D
      uint32_t D = 0;
      if (p.tokens) {
        const int b = row / p.depth, j = row % p.depth;
        const uint32_t req = p.request_ids ? p.request_ids[b] : (uint32_t)b;
        D = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_PROPOSAL) >> 8;
      }
      if (tid == 0) sh.found = -1;
      __syncthreads();
      if (st == DSPARK_ST_OK) {
        uint32_t base = 0, cbase = 0;
        for (int t0 = 0; t0 < nsup; t0 += blockDim.x) {
          const int i = t0 + tid;
          const uint32_t c = (i < nsup) ? ent[i].c : 0u;
          const uint32_t nz = c > 0u ? 1u : 0u;
          uint32_t tot;
          const uint32_t incl = block_inclusive_scan(nz, sh.red32, &tot);
          if (nz) {
            ids[base + incl - 1] = ent[i].v;
            cnt[base + incl - 1] = c;
          }
          base += tot;
          uint32_t ctot;
          const uint32_t cincl = block_inclusive_scan(c, sh.red32, &ctot);
          if (c > 0u && cbase + cincl > D && cbase + cincl - c <= D) sh.found = ent[i].v;
          cbase += ctot;
          __syncthreads();
        }
        written = base;
      }
      for (int i = (int)written + tid; i < p.top_k; i += blockDim.x) {
        ids[i] = -1;
        cnt[i] = 0u;
      }
      __syncthreads();
      if (tid == 0) {
        p.nnz[row] = (int32_t)written;
        p.status[row] = st;
        if (p.tokens) p.tokens[row] = (st == DSPARK_ST_OK) ? sh.found : -1;
      }
    }
    cluster.sync();  // leader done reading the peers' candidate lists
    return;
  }

  // ------------------------------------------------------------ dense rows
  uint32_t* crow = p.counts + (int64_t)row * V;
  if (status != DSPARK_ST_OK) {
    for (int v = lo + tid; v < hi; v += blockDim.x) crow[v] = 0u;
    if (rank == 0 && tid == 0) {
      p.status[row] = status;
      if (p.tokens) p.tokens[row] = -1;
    }
    cluster.sync();  // peers may still read this CTA's pub
    return;
  }

  // ---- pass B: E (exact float) in place, S
  uint64_t S = 0;
  for (int g = tid; g < ngroups; g += blockDim.x) {
    const float4 y4 = reinterpret_cast<const float4*>(sl)[g];
    float yy[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float e = weight_float(__fsub_rn(yy[i], m));
      const float Ef = floorf(__fmul_rn(e, 0x1p40f));  // exact, < 2^41
      yy[i] = Ef;
      S += __float2ull_rz(Ef);                           // exact
    }
    reinterpret_cast<float4*>(sl)[g] = make_float4(yy[0], yy[1], yy[2], yy[3]);
  }
  S = block_reduce(S, OpAddU64(), sh.red64);
  if (tid == 0) sh.pub.s.S = S;
  for (int i = tid; i < kHistBins; i += blockDim.x) sh.hist[i] = 0u;
  cluster.sync();  // S3
  gather_pubs(cluster, sh);
  if (tid == 0) {
    uint64_t S_all = 0;
    for (int r = 0; r < kQCluster; ++r) S_all += sh.peers[r].S;
    const double kd = __ddiv_rn(16777216.0, __ull2double_rn(S_all));
    const uint64_t kbits = (uint64_t)__double_as_longlong(kd);
    sh.mk = (kbits & ((1ull << 52) - 1ull)) | (1ull << 52);
    sh.ek = (int)((kbits >> 52) & 0x7FF) - 1075;
    sh.khi = __double2float_rn(kd);
    sh.klo = __double2float_rn(__dsub_rn(kd, (double)sh.khi));
  }
  __syncthreads();
  const uint64_t mk = sh.mk;
  const int ek = sh.ek;
  const float khi = sh.khi, klo = sh.klo;

  // ---- pass C: floor / fraction split, histogram, packed in place
  uint32_t F = 0, npos = 0, internal = 0;
  for (int g = tid; g < ngroups; g += blockDim.x) {
    const float4 e4 = reinterpret_cast<const float4*>(sl)[g];
    const float ee[4] = {e4.x, e4.y, e4.z, e4.w};
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float Ef = ee[i];
      const float p1 = __fmul_rn(Ef, khi);
      const float e1 = __fmaf_rn(Ef, khi, -p1);
      const float p2 = __fmul_rn(Ef, klo);
      const float f0 = floorf(p1);
      const float w = __fadd_rn(e1, p2);
      const float fr = __fadd_rn(__fsub_rn(p1, f0), w);
      const float fi = floorf(fr);
      const float frc = __fsub_rn(fr, fi);
      const float fb = __fmul_rn(frc, 4096.0f);
      const float bk = floorf(fb);
      const float dist = fminf(__fsub_rn(fb, bk), __fsub_rn(__fadd_rn(bk, 1.0f), fb));
      const float eps = __fmaf_rn(p1, 0x1p-33f, 0x1p-12f);
      const float ff = __fadd_rn(f0, fi);
      if (Ef == 0.0f) {
        pk[i] = 0u;
      } else if (dist > eps && ff < (float)kFMaxPacked) {
        const uint32_t fu = (uint32_t)small_float_to_int(ff);
        const uint32_t bu = (uint32_t)small_float_to_int(bk);
        F += fu;
        ++npos;
        atomicAdd(&sh.hist[bu], 1u);
        pk[i] = pack(fu, 1u, bu);
      } else {
        // exact path after the loop (E stays in place)
        const uint32_t j = atomicAdd(&sh.n_unc, 1u);
        if (j < kUncCap) {
          sh.unc[j] = 4 * g + i;
          pk[i] = __float_as_uint(Ef);
        } else {
          uint32_t fu, pos, bu;
          exact_pack(Ef, mk, ek, &fu, &pos, &bu);
          F += fu;
          npos += pos;
          if (pos) atomicAdd(&sh.hist[bu], 1u);
          if (fu < kFMaxPacked) {
            pk[i] = pack(fu, pos, bu);
          } else {
            const uint32_t q = atomicAdd(&sh.n_esc, 1u);
            if (q < kEscCap) {
              sh.esc[q].s = 4 * g + i;
              sh.esc[q].f = fu;
              sh.esc[q].bucket = bu;
              sh.esc[q].pos = pos;
            } else {
              internal = 1u;
            }
            pk[i] = kEscape;
          }
        }
      }
    }
    reinterpret_cast<uint4*>(slu)[g] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  __syncthreads();
  // elements whose fraction lies within the error bound of a bin edge
  const uint32_t n_unc = min(sh.n_unc, (uint32_t)kUncCap);
  for (uint32_t j = tid; j < n_unc; j += blockDim.x) {
    const int s = sh.unc[j];
    uint32_t fu, pos, bu;
    exact_pack(__uint_as_float(slu[s]), mk, ek, &fu, &pos, &bu);
    F += fu;
    npos += pos;
    if (pos) atomicAdd(&sh.hist[bu], 1u);
    if (fu < kFMaxPacked) {
      slu[s] = pack(fu, pos, bu);
    } else {
      const uint32_t q = atomicAdd(&sh.n_esc, 1u);
      if (q < kEscCap) {
        sh.esc[q].s = s;
        sh.esc[q].f = fu;
        sh.esc[q].bucket = bu;
        sh.esc[q].pos = pos;
      } else {
        internal = 1u;
      }
      slu[s] = kEscape;
    }
  }
  const uint64_t F64 = block_reduce((uint64_t)F, OpAddU64(), sh.red64);
  npos = block_reduce(npos, OpAddU32(), sh.red32);
  internal = block_reduce(internal, OpOrU32(), sh.red32);
  if (tid == 0) {
    sh.pub.s.F = F64;
    sh.pub.s.npos = npos;
    sh.pub.s.flags = internal ? 2u : 0u;
  }
  publish_coarse(sh, kHistBins);
  cluster.sync();  // S4
  gather_pubs(cluster, sh);
  uint64_t F_all = 0;
  uint32_t npos_all = 0, flags2 = 0;
  for (int r = 0; r < kQCluster; ++r) {
    F_all += sh.peers[r].F;
    npos_all += sh.peers[r].npos;
    flags2 |= sh.peers[r].flags;
  }
  if (flags2 & 2u) status = DSPARK_ST_INTERNAL;
  else if (F_all == 0 || F_all > (uint64_t)kM || (uint64_t)kM - F_all > (uint64_t)npos_all)
    status = DSPARK_ST_ALLOC_INCONSISTENT;
  const uint32_t R = (status == DSPARK_ST_OK) ? (uint32_t)((uint64_t)kM - F_all) : 0u;

  const uint32_t n_esc = min(sh.n_esc, (uint32_t)kEscCap);
  auto unpack = [&](uint32_t w, int s, uint32_t* f, uint32_t* pos, uint32_t* bucket) {
    if (w == kEscape) {
      *f = 0u;
      *pos = 0u;
      *bucket = 0u;
      for (uint32_t j = 0; j < n_esc; ++j)
        if (sh.esc[j].s == s) {
          *f = sh.esc[j].f;
          *pos = sh.esc[j].pos;
          *bucket = sh.esc[j].bucket;
        }
      return;
    }
    *f = w >> 13;
    *pos = (w >> 12) & 1u;
    *bucket = w & 0xFFFu;
  };
  auto exact_key = [&](int s) -> uint64_t {
    const int v = lo + s - off;
    float y = load_logit(xrow, p.dtype, v);
    if (scale) y = __fmul_rn(y, invT);
    const float e = weight_float(__fsub_rn(y, m));
    uint32_t Ei;
    int se;
    weight_split(e, &Ei, &se);
    return frac_key(alloc_split(Ei, se, mk, ek));
  };

  int bstar = kHistBins;  // no grants when R == 0
  uint32_t Rin = 0;       // grants inside bin bstar
  if (R > 0) {
    select_from_cluster(cluster, sh, kHistBins, R);
    bstar = sh.sel_bin;
    Rin = R - sh.sel_above;
  }

  // ---- pass E: counts = f + [bin > bstar]; the members of bin bstar get f
  // for now, their exact fraction, and a place in the member list
  uint32_t csum = 0;
  uint64_t kmin = ~0ull, kmax = 0ull;
  const int offc = (int)((reinterpret_cast<uintptr_t>(crow + lo) / 4) & 3);
  if (status == DSPARK_ST_OK) {
    for (int g = tid; g < ngroups; g += blockDim.x) {
      const uint4 w4 = reinterpret_cast<const uint4*>(slu)[g];
      const uint32_t ww[4] = {w4.x, w4.y, w4.z, w4.w};
      uint32_t c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int s = 4 * g + i;
        uint32_t f, pos, b;
        unpack(ww[i], s, &f, &pos, &b);
        c[i] = f + ((pos && (int)b > bstar) ? 1u : 0u);
        if (pos && (int)b == bstar && s >= off && s < off + n) {
          const uint64_t key = exact_key(s);
          kmin = min(kmin, key);
          kmax = max(kmax, key);
          const uint32_t j = atomicAdd(&sh.n_cand, 1u);
          if (j < kCandCap) {
            sh.cand[j].key = key;
            sh.cand[j].v = lo + s - off;
            sh.cand[j].s = s;
          }
        }
      }
      const int s0 = 4 * g;
      const bool full = (s0 >= off) && (s0 + 3 < off + n);
      if (full) {
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
  const uint64_t csum64 = block_reduce((uint64_t)csum, OpAddU64(), sh.red64);
  kmin = block_reduce(kmin, OpMinU64(), sh.red64);
  kmax = block_reduce(kmax, OpMaxU64(), sh.red64);
  if (tid == 0) {
    sh.pub.s.csum = csum64;
    sh.pub.s.ncand = sh.n_cand;
    sh.pub.s.kmin = kmin;
    sh.pub.s.kmax = kmax;
  }
  cluster.sync();  // S5
  gather_pubs(cluster, sh);
  if (tid < kQCluster) sh.peers_csum[tid] = sh.peers[tid].csum;
  uint32_t total_members = 0;
  bool fits = true;
  uint64_t gmin = ~0ull, gmax = 0ull;
  for (int r = 0; r < kQCluster; ++r) {
    total_members += sh.peers[r].ncand;
    fits = fits && (sh.peers[r].ncand <= (uint32_t)kCandCap);
    gmin = min(gmin, sh.peers[r].kmin);
    gmax = max(gmax, sh.peers[r].kmax);
  }
  fits = fits && total_members <= (uint32_t)kAllCap;
  // grants[r]: members of CTA r granted a ticket
  if (tid < kQCluster) sh.grants[tid] = 0u;
  __syncthreads();
  if (R > 0 && fits) {
    // every CTA sorts all members by (fraction desc, id asc); the first Rin
    // are granted
    Cand* all = sh.allc;
    // one remote load per thread: entry t comes from the CTA whose range of
    // the concatenated lists holds t
    for (int t = tid; t < (int)total_members; t += blockDim.x) {
      int r = 0;
      uint32_t base = 0;
      while (r < kQCluster - 1 && (uint32_t)t >= base + sh.peers[r].ncand) {
        base += sh.peers[r].ncand;
        ++r;
      }
      all[t] = cluster.map_shared_rank(&sh.cand[0], r)[t - base];
    }
    int np2 = 1;
    while (np2 < (int)total_members) np2 <<= 1;
    for (int i = (int)total_members + tid; i < np2; i += blockDim.x) {
      Cand e;
      e.key = 0ull;
      e.v = 0x7FFFFFFF;
      e.s = -1;
      all[i] = e;
    }
    __syncthreads();
    auto cand_less = [](const Cand& a, const Cand& b) {
      return a.key > b.key || (a.key == b.key && a.v < b.v);
    };
    if (np2 <= 32) {
      // one warp, one entry per lane, shuffles only
      if (tid < 32 && np2 > 1) {
        Cand c = all[tid < np2 ? tid : 0];
        for (int kx = 2; kx <= np2; kx <<= 1)
          for (int jx = kx >> 1; jx > 0; jx >>= 1) {
            Cand o;
            o.key = __shfl_xor_sync(0xffffffffu, c.key, jx);
            o.v = __shfl_xor_sync(0xffffffffu, c.v, jx);
            o.s = __shfl_xor_sync(0xffffffffu, c.s, jx);
            const bool lower = (tid & jx) == 0;
            const bool up = (tid & kx) == 0;
            // the lower lane keeps the "smaller" (by cand_less) when ascending
            const bool o_first = cand_less(o, c);
            if (tid < np2 && (lower == up ? o_first : !o_first)) c = o;
          }
        if (tid < np2) all[tid] = c;
      }
      __syncthreads();
    } else {
      bitonic_sort(all, np2, cand_less);
    }
    for (int i = tid; i < (int)min(Rin, total_members); i += blockDim.x) {
      const int owner = all[i].v / p.chunk;
      atomicAdd(&sh.grants[owner], 1u);
      if (owner == rank) set_bit(sh.grant_bits, all[i].s);
    }
    __syncthreads();
  } else if (R > 0) {
    // many members: the exact fraction threshold by 8-bit radix levels unless
    // they all hold the same fraction, then the remaining tickets go to the
    // lowest ids holding the threshold fraction
    auto is_member = [&](int s) -> bool {
      if (s < off || s >= off + n) return false;
      uint32_t f, pos, b;
      unpack(slu[s], s, &f, &pos, &b);
      return pos && (int)b == bstar;
    };
    uint64_t thr = gmin, prefix = 0ull;
    uint32_t need = Rin;
    if (gmin != gmax) {
      for (int lvl = 0; lvl < 8; ++lvl) {
        const int sft = 56 - 8 * lvl;
        __syncthreads();
        for (int i = tid; i < 256; i += blockDim.x) sh.hist[i] = 0u;
        __syncthreads();
        for (int g = tid; g < ngroups; g += blockDim.x)
          for (int i = 0; i < 4; ++i) {
            const int s = 4 * g + i;
            if (!is_member(s)) continue;
            const uint64_t key = exact_key(s);
            if (lvl > 0 && (key >> (sft + 8)) != prefix) continue;
            atomicAdd(&sh.hist[(key >> sft) & 255u], 1u);
          }
        __syncthreads();
        publish_coarse(sh, 256);
        cluster.sync();
        select_from_cluster(cluster, sh, 256, need);
        prefix = (prefix << 8) | (uint64_t)sh.sel_bin;
        need -= sh.sel_above;
        cluster.sync();
      }
      thr = prefix;
    }
    uint32_t mine = 0;
    // with a single fraction among the members no key is recomputed: every
    // member holds the threshold fraction
    const bool one_key = (gmin == gmax);
    if (!one_key)
      for (int g = tid; g < ngroups; g += blockDim.x)
        for (int i = 0; i < 4; ++i) {
          const int s = 4 * g + i;
          if (is_member(s) && exact_key(s) > thr) {
            set_bit(sh.grant_bits, s);
            ++mine;
          }
        }
    __syncthreads();
    ordered_ranks(
        cluster, sh, ngroups,
        [&](int s) -> bool { return is_member(s) && (one_key || exact_key(s) == thr); },
        [&](int s, uint32_t rk) {
          if (rk < need) {
            set_bit(sh.grant_bits, s);
            ++mine;
          }
        });
    mine = block_reduce(mine, OpAddU32(), sh.red32);
    if (tid == 0) sh.pub.s.n_grant = mine;
    cluster.sync();
    gather_pubs(cluster, sh);
    if (tid < kQCluster) sh.grants[tid] = sh.peers[tid].n_grant;
    __syncthreads();
  }
  // patch this CTA's granted members (their counts were written as f)
  if (R > 0) {
    const int nc = fits ? (int)sh.n_cand : 0;
    for (int j = tid; j < nc; j += blockDim.x) {
      const int s = sh.cand[j].s;
      if (get_bit(sh.grant_bits, s)) {
        uint32_t f, pos, b;
        unpack(slu[s], s, &f, &pos, &b);
        crow[lo - off + s] = f + 1u;
      }
    }
    if (!fits)
      for (int g = tid; g < ngroups; g += blockDim.x)
        for (int i = 0; i < 4; ++i) {
          const int s = 4 * g + i;
          if (s < off || s >= off + n || !get_bit(sh.grant_bits, s)) continue;
          uint32_t f, pos, b;
          unpack(slu[s], s, &f, &pos, &b);
          crow[lo - off + s] = f + 1u;
        }
  }
  uint64_t csum_all = 0, cbefore = 0, my_total = 0;
  for (int r = 0; r < kQCluster; ++r) {
    const uint64_t cr = sh.peers_csum[r] + sh.grants[r];
    if (r < rank) cbefore += cr;
    if (r == rank) my_total = cr;
    csum_all += cr;
  }
  if (status == DSPARK_ST_OK && csum_all != (uint64_t)kM) status = DSPARK_ST_ALLOC_INCONSISTENT;
  __syncthreads();  // the member patches are written before any re-read below
  if (status != DSPARK_ST_OK)
    for (int v = lo + tid; v < hi; v += blockDim.x) crow[v] = 0u;
  if (rank == 0 && tid == 0) {
    p.status[row] = status;
    if (p.tokens && status != DSPARK_ST_OK) p.tokens[row] = -1;
  }
  // every remote read of this row is done: arrive now, wait before leaving
  cluster.barrier_arrive();
  // ---- fused draft draw: the CTA whose slice holds D scans its counts,
  // rebuilt from the packed words still in shared memory
  if (p.tokens && status == DSPARK_ST_OK) {
    const int b = row / p.depth, j = row % p.depth;
    const uint32_t req = p.request_ids ? p.request_ids[b] : (uint32_t)b;
    const uint64_t D = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_PROPOSAL) >> 8;
    if (D >= cbefore && D < cbefore + my_total) {
      auto count_at = [&](int s) -> uint32_t {
        if (s < off || s >= off + n) return 0u;
        uint32_t f, pos, bb;
        unpack(slu[s], s, &f, &pos, &bb);
        const bool gr =
            pos && ((int)bb > bstar || ((int)bb == bstar && get_bit(sh.grant_bits, s)));
        return f + (gr ? 1u : 0u);
      };
      // one contiguous segment of slice positions per warp
      const int lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
      const int ns = 4 * ngroups;
      const int seg = (ns + nw - 1) / nw;
      const int a0 = warp * seg, a1 = min(ns, a0 + seg);
      uint32_t ssum = 0;
      for (int s = a0 + lane; s < a1; s += 32) ssum += count_at(s);
      ssum = warp_reduce(ssum, OpAddU32());
      if (lane == 0) sh.segsum[warp] = ssum;
      __syncthreads();
      uint64_t sb = cbefore;
      for (int w = 0; w < warp; ++w) sb += sh.segsum[w];
      if (D >= sb && D < sb + sh.segsum[warp]) {
        uint64_t base = sb;
        for (int s0 = a0; s0 < a1; s0 += 32) {
          const int s = s0 + lane;
          const uint32_t cv = (s < a1) ? count_at(s) : 0u;
          uint32_t incl = cv;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
          }
          const uint32_t tile = __shfl_sync(0xffffffffu, incl, 31);
          if (D < base + tile) {
            const bool hit = cv > 0u && base + incl > D && base + incl - cv <= D;
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

int q_build_smem_bytes(int chunk, int top_k) {
  int slice = (chunk + 4) * 4;
  if (top_k > 0) {
    const int need = kGatherCap * (int)sizeof(Sup) + 1024 * (int)sizeof(SparseEntry);
    if (slice < need) slice = need;
  }
  return slice;
}

cudaError_t launch_q_build(const void* x, int dtype, int64_t ld, int n_rows, int V,
                           const float* temperature, int top_k, uint32_t* counts, int32_t* ids,
                           int32_t* nnz, int32_t* status, int32_t* tokens, uint64_t seed,
                           const uint32_t* request_ids, int depth, cudaStream_t stream) {
  QParams p;
  p.x = x;
  p.dtype = dtype;
  p.ld = ld;
  p.n_rows = n_rows;
  p.V = V;
  p.temperature = temperature;
  p.top_k = top_k;
  p.counts = counts;
  p.ids = ids;
  p.nnz = nnz;
  p.status = status;
  int chunk = (V + kQCluster - 1) / kQCluster;
  chunk = (chunk + 3) & ~3;
  p.chunk = chunk;
  p.tokens = tokens;
  p.seed = seed;
  p.request_ids = request_ids;
  p.depth = depth > 0 ? depth : 1;
  const int smem = q_build_smem_bytes(chunk, top_k);
  cudaError_t err =
      cudaFuncSetAttribute(q_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  q_build_kernel<<<n_rows * kQCluster, kQThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dspark

