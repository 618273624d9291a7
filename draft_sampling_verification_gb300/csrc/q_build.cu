// q_build.cu -- dyadic24-standard-v1 q construction, one 8-CTA thread-block
// cluster per draft row ("PP1 q transport and scheduling design",
// Distribution contract and precision: proposal construction, sparse top-k).
//
// Each CTA holds one eighth of the row in shared memory for the whole build;
// the row is read from HBM once.  Cluster-wide values (row max, weight sum,
// floor sum, remainder histograms) are exchanged through distributed shared
// memory.  Passes over the resident slice:
//   A  load, validate, y = x * RN(1/T), row max
//   (top-k) three radix-select levels on the float key of y for the support
//   B  e = exp_ds(y - m) in place, S = sum floor(e * 2^40)
//   C  exact FP64-equivalent split of a = E * k into floor f and fraction r,
//      4096-bin histogram of floor(r * 4096), packed (f, r > 0, bin) in place
//   D  the bin holding the grant threshold: exact fractions of its members,
//      ranked by (fraction desc, id asc)
//   E  counts = f + grant, written to HBM; the total is checked to be M.
// Sparse rows gather their (<= top_k) support in the cluster's first CTA,
// which allocates with FP64 arithmetic directly.
#include "common.cuh"

namespace dspark {

constexpr int kQCluster = 8;
constexpr int kQThreads = 256;
constexpr int kHistBins = 4096;
constexpr int kCandCap = 256;
constexpr int kEscCap = 48;
constexpr int kChunkMax = DSPARK_MAX_V / kQCluster;  // 16384 elements per CTA
constexpr uint32_t kEscape = 0xFFFFE000u;            // f field all ones
constexpr uint32_t kFMaxPacked = (1u << 19) - 1u;    // f < this is packed inline

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
};

struct QPub {
  float max;
  uint32_t flags;  // bit0 nonfinite, bit1 internal
  uint32_t nfinite;
  uint32_t npos;
  uint64_t S;
  uint64_t F;
  uint64_t csum;
  uint64_t kmin, kmax;
  uint32_t ncand;
  uint32_t n_eq;   // tie-group members in this CTA
  uint32_t nsup;
  uint32_t coarse[64];
};

struct Cand {
  uint64_t key;
  int32_t v;  // token id
  int32_t s;  // slice index
};

struct Esc {
  int32_t s;
  uint32_t f;
  uint32_t bucket;
  uint32_t pos;
};

struct Sup {
  int32_t v;
  float y;
};

struct QShared {
  uint32_t hist[kHistBins];
  uint32_t grant_bits[kChunkMax / 32 + 2];
  Cand cand[kCandCap];
  Esc esc[kEscCap];
  Sup sup[DSPARK_MAX_TOPK];
  QPub pub;
  uint32_t gcoarse[64];
  uint32_t gfine[64];
  uint64_t red64[32];
  uint32_t red32[32];
  float redf[32];
  uint32_t n_cand, n_esc, n_sup;
  int sel_bin;
  uint32_t sel_above, sel_count;
  uint32_t scan_base;
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

__device__ __forceinline__ void set_bit(uint32_t* bits, int s) { atomicOr(&bits[s >> 5], 1u << (s & 31)); }
__device__ __forceinline__ bool get_bit(const uint32_t* bits, int s) { return (bits[s >> 5] >> (s & 31)) & 1u; }

__device__ __forceinline__ uint32_t pack(uint32_t f, uint32_t pos, uint32_t bucket) {
  return (f << 13) | (pos << 12) | bucket;
}

// Coarse sums (64 superbins) of the local histogram into pub.coarse.
__device__ void publish_coarse(QShared& sh, int nbins) {
  const int per = nbins / 64;
  for (int c = threadIdx.x; c < 64; c += blockDim.x) {
    uint32_t s = 0;
    for (int i = 0; i < per; ++i) s += sh.hist[c * per + i];
    sh.pub.coarse[c] = s;
  }
}

// After a cluster sync that published hist/coarse: finds the bin b where the
// cluster-wide count, accumulated from the top bin down, reaches `need`
// (need >= 1 and <= total).  Result in sh.sel_*; all CTAs agree.  The caller
// must cluster-sync before the histograms are modified again.
__device__ void select_from_cluster(cg::cluster_group& cluster, QShared& sh, int nbins,
                                    uint32_t need) {
  const int per = nbins / 64;
  if (threadIdx.x < 64) {
    uint32_t g = 0;
    for (int r = 0; r < kQCluster; ++r) g += cluster.map_shared_rank(&sh.pub, r)->coarse[threadIdx.x];
    sh.gcoarse[threadIdx.x] = g;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t acc = 0;
    int sb = 63;
    for (; sb > 0; --sb) {
      if (acc + sh.gcoarse[sb] >= need) break;
      acc += sh.gcoarse[sb];
    }
    sh.sel_bin = sb;
    sh.sel_above = acc;
  }
  __syncthreads();
  const int sb = sh.sel_bin;
  if (threadIdx.x < per) {
    uint32_t g = 0;
    for (int r = 0; r < kQCluster; ++r) g += cluster.map_shared_rank(&sh.hist[0], r)[sb * per + threadIdx.x];
    sh.gfine[threadIdx.x] = g;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t acc = sh.sel_above;
    int b = per - 1;
    for (; b > 0; --b) {
      if (acc + sh.gfine[b] >= need) break;
      acc += sh.gfine[b];
    }
    sh.sel_bin = sb * per + b;
    sh.sel_above = acc;
    sh.sel_count = sh.gfine[b];
  }
  __syncthreads();
}

// Exclusive count, in id order over the whole cluster, of the elements for
// which pred(s) holds; calls fn(s, rank) for each of them.  One cluster sync.
template <typename Pred, typename Fn>
__device__ void ordered_ranks(cg::cluster_group& cluster, QShared& sh, int ngroups, Pred pred,
                              Fn fn) {
  // local count
  uint32_t cnt = 0;
  for (int g = threadIdx.x; g < ngroups; g += blockDim.x)
    for (int i = 0; i < 4; ++i) cnt += pred(4 * g + i) ? 1u : 0u;
  cnt = block_reduce(cnt, OpAddU32(), sh.red32);
  if (threadIdx.x == 0) sh.pub.n_eq = cnt;
  cluster.sync();
  if (threadIdx.x == 0) {
    uint32_t base = 0;
    const int me = (int)cluster.block_rank();
    for (int r = 0; r < me; ++r) base += cluster.map_shared_rank(&sh.pub, r)->n_eq;
    sh.scan_base = base;
  }
  __syncthreads();
  uint32_t base = sh.scan_base;
  // tiles of blockDim.x groups, scanned in id order
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

__global__ void __cluster_dims__(kQCluster, 1, 1) __launch_bounds__(kQThreads, 2)
    q_build_kernel(QParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ QShared sh;
  extern __shared__ __align__(16) float sl[];
  uint32_t* slu = reinterpret_cast<uint32_t*>(sl);

  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.x / kQCluster;
  const int V = p.V;
  const int lo = rank * p.chunk;
  const int hi = min(V, lo + p.chunk);
  const int n = max(0, hi - lo);
  const char* xrow = reinterpret_cast<const char*>(p.x) +
                     (int64_t)row * p.ld * (p.dtype == DSPARK_F32 ? 4 : 2);
  const int esz = (p.dtype == DSPARK_F32) ? 4 : 2;
  // offset of element lo inside its 4-element group of the source row
  const int off = (int)((reinterpret_cast<uintptr_t>(xrow + (int64_t)lo * esz) / esz) & 3);
  const int ngroups = (off + n + 3) >> 2;
  const bool sparse = p.top_k > 0;
  const int tid = threadIdx.x;

  if (tid == 0) {
    sh.n_cand = 0;
    sh.n_esc = 0;
    sh.n_sup = 0;
  }
  for (int i = tid; i < kChunkMax / 32 + 2; i += blockDim.x) sh.grant_bits[i] = 0u;

  // ---- temperature (identical decision in every CTA)
  const float T = p.temperature ? p.temperature[row] : 1.0f;
  const float invT = __frcp_rn(T);
  const bool bad_T = !(isfinite(T) && T > 0.0f) || !(isfinite(invT) && invT >= 0x1p-126f);
  int status = DSPARK_ST_OK;
  if (bad_T) status = DSPARK_ST_BAD_TEMPERATURE;

  // ---- pass A: load, validate, y, max
  uint32_t flags = 0, nfin = 0;
  float mx = -INFINITY;
  if (!bad_T) {
    const bool vec = (p.dtype == DSPARK_F32);
    for (int g = tid; g < ngroups; g += blockDim.x) {
      float xv[4];
      const int s0 = 4 * g;
      const bool full = (s0 >= off) && (s0 + 3 < off + n);
      if (vec && full) {
        const float4 q = __ldg(reinterpret_cast<const float4*>(
            reinterpret_cast<const float*>(xrow) + lo - off + s0));
        xv[0] = q.x; xv[1] = q.y; xv[2] = q.z; xv[3] = q.w;
      } else {
        for (int i = 0; i < 4; ++i) {
          const int s = s0 + i;
          xv[i] = (s >= off && s < off + n) ? load_logit(xrow, p.dtype, (int64_t)(lo - off + s))
                                            : -INFINITY;
        }
      }
      float yv[4];
      for (int i = 0; i < 4; ++i) {
        const float x = xv[i];
        if (isnan(x) || x == INFINITY) flags |= 1u;
        const float y = __fmul_rn(x, invT);
        if (isfinite(x) && !isfinite(y)) flags |= 1u;
        yv[i] = y;
        if (y > -INFINITY) {
          ++nfin;
          mx = fmaxf(mx, y);
        }
      }
      reinterpret_cast<float4*>(sl)[g] = make_float4(yv[0], yv[1], yv[2], yv[3]);
    }
  }
  flags = block_reduce(flags, OpOrU32(), sh.red32);
  nfin = block_reduce(nfin, OpAddU32(), sh.red32);
  mx = block_reduce(mx, OpMaxF(), sh.redf);
  if (tid == 0) {
    sh.pub.flags = flags;
    sh.pub.nfinite = nfin;
    sh.pub.max = mx;
  }
  cluster.sync();  // S1
  uint32_t nfin_all = 0, flags_all = 0;
  float m = -INFINITY;
  for (int r = 0; r < kQCluster; ++r) {
    const QPub* q = cluster.map_shared_rank(&sh.pub, r);
    nfin_all += q->nfinite;
    flags_all |= q->flags;
    m = fmaxf(m, q->max);
  }
  if (status == DSPARK_ST_OK) {
    if (flags_all & 1u) status = DSPARK_ST_NONFINITE;
    else if (nfin_all == 0) status = DSPARK_ST_ZERO_MASS;
  }
  cluster.sync();  // S2: pubs may be rewritten below

  // ---- sparse: top-k support by radix select on the float key of y
  if (status == DSPARK_ST_OK && sparse) {
    const uint32_t kk = min((uint32_t)p.top_k, nfin_all);
    uint32_t thr = 0;          // threshold key (elements with key > thr are in)
    uint32_t need_eq = 0;      // how many with key == thr are in (lowest ids)
    uint32_t n_eq_all = 0;
    bool all_finite = (kk == nfin_all);
    if (!all_finite) {
      uint32_t prefix = 0, need = kk;
      const int shifts[3] = {20, 8, 0};
      const int widths[3] = {12, 12, 8};
      for (int lvl = 0; lvl < 3; ++lvl) {
        const int nb = 1 << widths[lvl];
        for (int i = tid; i < nb; i += blockDim.x) sh.hist[i] = 0u;
        __syncthreads();
        const int hs = shifts[lvl] + widths[lvl];  // bits above this level
        for (int g = tid; g < ngroups; g += blockDim.x) {
          const float4 y4 = reinterpret_cast<const float4*>(sl)[g];
          const float yy[4] = {y4.x, y4.y, y4.z, y4.w};
          for (int i = 0; i < 4; ++i) {
            if (!(yy[i] > -INFINITY)) continue;
            const uint32_t key = float_key(yy[i]);
            if (hs < 32 && (key >> hs) != prefix) continue;
            atomicAdd(&sh.hist[(key >> shifts[lvl]) & (nb - 1)], 1u);
          }
        }
        __syncthreads();
        publish_coarse(sh, nb);
        cluster.sync();
        select_from_cluster(cluster, sh, nb, need);
        const uint32_t b = (uint32_t)sh.sel_bin;
        need -= sh.sel_above;
        n_eq_all = sh.sel_count;
        prefix = (prefix << widths[lvl]) | b;
        cluster.sync();
      }
      thr = prefix;
      need_eq = need;
    }
    // membership: key > thr, or key == thr among the need_eq lowest ids
    auto in_sup_strict = [&](int s) -> bool {
      if (s < off || s >= off + n) return false;
      const float y = sl[s];
      if (!(y > -INFINITY)) return false;
      return all_finite || float_key(y) > thr;
    };
    auto push = [&](int s) {
      const uint32_t i = atomicAdd(&sh.n_sup, 1u);
      if (i < DSPARK_MAX_TOPK) {
        sh.sup[i].v = lo + s - off;
        sh.sup[i].y = sl[s];
      }
    };
    for (int g = tid; g < ngroups; g += blockDim.x)
      for (int i = 0; i < 4; ++i)
        if (in_sup_strict(4 * g + i)) push(4 * g + i);
    if (!all_finite) {
      auto is_eq = [&](int s) -> bool {
        if (s < off || s >= off + n) return false;
        const float y = sl[s];
        return (y > -INFINITY) && float_key(y) == thr;
      };
      if (need_eq >= n_eq_all) {
        for (int g = tid; g < ngroups; g += blockDim.x)
          for (int i = 0; i < 4; ++i)
            if (is_eq(4 * g + i)) push(4 * g + i);
      } else {
        __syncthreads();
        ordered_ranks(cluster, sh, ngroups, is_eq, [&](int s, uint32_t rk) {
          if (rk < need_eq) push(s);
        });
      }
    }
    __syncthreads();
    if (tid == 0) sh.pub.nsup = sh.n_sup;
    cluster.sync();  // support lists complete everywhere

    if (rank == 0) {
      // gather the support into the leader's slice memory
      SparseEntry* ent = reinterpret_cast<SparseEntry*>(sl);
      __shared__ uint32_t base_of[kQCluster + 1];
      __shared__ int bad_gather;
      if (tid == 0) {
        uint32_t acc = 0;
        bad_gather = 0;
        for (int r = 0; r < kQCluster; ++r) {
          base_of[r] = acc;
          const uint32_t ns = cluster.map_shared_rank(&sh.pub, r)->nsup;
          if (ns > DSPARK_MAX_TOPK) bad_gather = 1;
          acc += ns;
        }
        base_of[kQCluster] = acc;
        if (acc != kk) bad_gather = 1;
      }
      __syncthreads();
      const int nsup = bad_gather ? 0 : (int)base_of[kQCluster];
      if (!bad_gather) {
        for (int r = 0; r < kQCluster; ++r) {
          const Sup* rs = cluster.map_shared_rank(&sh.sup[0], r);
          const int cnt = (int)(base_of[r + 1] - base_of[r]);
          for (int i = tid; i < cnt; i += blockDim.x) {
            SparseEntry e;
            e.v = rs[i].v;
            e.y = rs[i].y;
            ent[base_of[r] + i] = e;
          }
        }
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
      const double kd = __ddiv_rn(16777216.0, __ull2double_rn(S));
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
      // order by (fraction desc, id asc), grant the first R, restore id order
      int np2 = 1;
      while (np2 < nsup) np2 <<= 1;
      for (int i = nsup + tid; i < np2; i += blockDim.x) {
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
      bitonic_sort(ent, np2, [](const SparseEntry& a, const SparseEntry& b) {
        return a.r > b.r || (a.r == b.r && a.v < b.v);
      });
      for (int i = tid; i < nsup; i += blockDim.x) ent[i].c = ent[i].f + ((uint32_t)i < R ? 1u : 0u);
      __syncthreads();
      bitonic_sort(ent, np2, [](const SparseEntry& a, const SparseEntry& b) { return a.v < b.v; });
      // total check and compaction of nonzero counts in id order
      uint64_t csum = 0;
      for (int i = tid; i < nsup; i += blockDim.x) csum += ent[i].c;
      csum = block_reduce(csum, OpAddU64(), sh.red64);
      if (st == DSPARK_ST_OK && csum != (uint64_t)kM) st = DSPARK_ST_ALLOC_INCONSISTENT;
      int32_t* ids = p.ids + (int64_t)row * p.top_k;
      uint32_t* cnt = p.counts + (int64_t)row * p.top_k;
      uint32_t written = 0;
      if (st == DSPARK_ST_OK) {
        uint32_t base = 0;
        for (int t0 = 0; t0 < nsup; t0 += blockDim.x) {
          const int i = t0 + tid;
          const uint32_t nz = (i < nsup && ent[i].c > 0) ? 1u : 0u;
          uint32_t tot;
          const uint32_t incl = block_inclusive_scan(nz, sh.red32, &tot);
          if (nz) {
            ids[base + incl - 1] = ent[i].v;
            cnt[base + incl - 1] = ent[i].c;
          }
          base += tot;
          __syncthreads();
        }
        written = base;
      }
      for (int i = (int)written + tid; i < p.top_k; i += blockDim.x) {
        ids[i] = -1;
        cnt[i] = 0u;
      }
      if (tid == 0) {
        p.nnz[row] = (int32_t)written;
        p.status[row] = st;
      }
    }
    cluster.sync();  // leader done reading remote support lists
    return;
  }

  if (status != DSPARK_ST_OK) {
    if (sparse) {
      if (rank == 0) {
        for (int i = tid; i < p.top_k; i += blockDim.x) {
          p.ids[(int64_t)row * p.top_k + i] = -1;
          p.counts[(int64_t)row * p.top_k + i] = 0u;
        }
        if (tid == 0) {
          p.nnz[row] = 0;
          p.status[row] = status;
        }
      }
    } else {
      uint32_t* crow = p.counts + (int64_t)row * V;
      for (int v = lo + tid; v < hi; v += blockDim.x) crow[v] = 0u;
      if (rank == 0 && tid == 0) p.status[row] = status;
    }
    return;  // no remote access after S2
  }

  // ---- pass B: e in place, S
  uint64_t S = 0;
  for (int g = tid; g < ngroups; g += blockDim.x) {
    const float4 y4 = reinterpret_cast<const float4*>(sl)[g];
    float e[4];
    e[0] = weight_float(__fsub_rn(y4.x, m));
    e[1] = weight_float(__fsub_rn(y4.y, m));
    e[2] = weight_float(__fsub_rn(y4.z, m));
    e[3] = weight_float(__fsub_rn(y4.w, m));
    for (int i = 0; i < 4; ++i) S += weight_u64(e[i]);
    reinterpret_cast<float4*>(sl)[g] = make_float4(e[0], e[1], e[2], e[3]);
  }
  S = block_reduce(S, OpAddU64(), sh.red64);
  if (tid == 0) sh.pub.S = S;
  for (int i = tid; i < kHistBins; i += blockDim.x) sh.hist[i] = 0u;
  cluster.sync();  // S3
  uint64_t S_all = 0;
  for (int r = 0; r < kQCluster; ++r) S_all += cluster.map_shared_rank(&sh.pub, r)->S;
  const double kd = __ddiv_rn(16777216.0, __ull2double_rn(S_all));
  const uint64_t kbits = (uint64_t)__double_as_longlong(kd);
  const uint64_t mk = (kbits & ((1ull << 52) - 1ull)) | (1ull << 52);
  const int ek = (int)((kbits >> 52) & 0x7FF) - 1075;

  // ---- pass C: floor / fraction split, histogram, packed in place
  uint64_t F = 0;
  uint32_t npos = 0, internal = 0;
  for (int g = tid; g < ngroups; g += blockDim.x) {
    const float4 e4 = reinterpret_cast<const float4*>(sl)[g];
    const float ee[4] = {e4.x, e4.y, e4.z, e4.w};
    uint32_t pk[4];
    for (int i = 0; i < 4; ++i) {
      uint32_t Ei;
      int se;
      weight_split(ee[i], &Ei, &se);
      const AllocSplit a = alloc_split(Ei, se, mk, ek);
      const uint32_t pos = (a.rnum != 0ull) ? 1u : 0u;
      const uint32_t bucket = pos ? frac_bucket(a) : 0u;
      F += a.f;
      if (pos) {
        ++npos;
        atomicAdd(&sh.hist[bucket], 1u);
      }
      if (a.f < kFMaxPacked) {
        pk[i] = pack(a.f, pos, bucket);
      } else {
        const uint32_t j = atomicAdd(&sh.n_esc, 1u);
        if (j < kEscCap) {
          sh.esc[j].s = 4 * g + i;
          sh.esc[j].f = a.f;
          sh.esc[j].bucket = bucket;
          sh.esc[j].pos = pos;
        } else {
          internal = 1u;
        }
        pk[i] = kEscape;
      }
    }
    reinterpret_cast<uint4*>(slu)[g] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  F = block_reduce(F, OpAddU64(), sh.red64);
  npos = block_reduce(npos, OpAddU32(), sh.red32);
  internal = block_reduce(internal, OpOrU32(), sh.red32);
  if (tid == 0) {
    sh.pub.F = F;
    sh.pub.npos = npos;
    sh.pub.flags = internal ? 2u : 0u;
  }
  publish_coarse(sh, kHistBins);
  cluster.sync();  // S4
  uint64_t F_all = 0;
  uint32_t npos_all = 0, flags2 = 0;
  for (int r = 0; r < kQCluster; ++r) {
    const QPub* q = cluster.map_shared_rank(&sh.pub, r);
    F_all += q->F;
    npos_all += q->npos;
    flags2 |= q->flags;
  }
  if (flags2 & 2u) status = DSPARK_ST_INTERNAL;
  else if (F_all == 0 || F_all > (uint64_t)kM || (uint64_t)kM - F_all > (uint64_t)npos_all)
    status = DSPARK_ST_ALLOC_INCONSISTENT;
  const uint32_t R = (status == DSPARK_ST_OK) ? (uint32_t)((uint64_t)kM - F_all) : 0u;

  auto unpack = [&](int s, uint32_t* f, uint32_t* pos, uint32_t* bucket) {
    const uint32_t w = slu[s];
    if (w == kEscape) {
      const uint32_t ne = min(sh.n_esc, (uint32_t)kEscCap);
      for (uint32_t j = 0; j < ne; ++j)
        if (sh.esc[j].s == s) {
          *f = sh.esc[j].f;
          *pos = sh.esc[j].pos;
          *bucket = sh.esc[j].bucket;
          return;
        }
      *f = 0u;
      *pos = 0u;
      *bucket = 0u;
      return;
    }
    *f = w >> 13;
    *pos = (w >> 12) & 1u;
    *bucket = w & 0xFFFu;
  };

  int bstar = kHistBins;  // no grants when R == 0
  uint32_t Rin = 0;       // grants inside bin bstar
  if (R > 0) {
    select_from_cluster(cluster, sh, kHistBins, R);
    bstar = sh.sel_bin;
    Rin = R - sh.sel_above;
  }
  cluster.sync();  // S5: histograms no longer read remotely

  if (R > 0) {
    // ---- pass D: exact fractions of the members of bin bstar
    auto exact_key = [&](int s) -> uint64_t {
      const int v = lo + s - off;
      const float y = __fmul_rn(load_logit(xrow, p.dtype, v), invT);
      const float e = weight_float(__fsub_rn(y, m));
      uint32_t Ei;
      int se;
      weight_split(e, &Ei, &se);
      return frac_key(alloc_split(Ei, se, mk, ek));
    };
    auto is_member = [&](int s) -> bool {
      if (s < off || s >= off + n) return false;
      uint32_t f, pos, b;
      unpack(s, &f, &pos, &b);
      return pos && (int)b == bstar;
    };
    uint64_t kmin = ~0ull, kmax = 0ull;
    for (int g = tid; g < ngroups; g += blockDim.x)
      for (int i = 0; i < 4; ++i) {
        const int s = 4 * g + i;
        if (!is_member(s)) continue;
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
    kmin = block_reduce(kmin, OpMinU64(), sh.red64);
    kmax = block_reduce(kmax, OpMaxU64(), sh.red64);
    if (tid == 0) {
      sh.pub.ncand = sh.n_cand;
      sh.pub.kmin = kmin;
      sh.pub.kmax = kmax;
    }
    cluster.sync();  // S6
    bool fits = true;
    uint64_t gmin = ~0ull, gmax = 0ull;
    for (int r = 0; r < kQCluster; ++r) {
      const QPub* q = cluster.map_shared_rank(&sh.pub, r);
      fits = fits && (q->ncand <= (uint32_t)kCandCap);
      gmin = min(gmin, q->kmin);
      gmax = max(gmax, q->kmax);
    }
    if (fits) {
      // rank every local candidate against all candidates of the cluster
      const int nc = (int)sh.n_cand;
      for (int j = tid; j < nc; j += blockDim.x) {
        const uint64_t key = sh.cand[j].key;
        const int v = sh.cand[j].v;
        uint32_t rk = 0;
        for (int r = 0; r < kQCluster; ++r) {
          const QPub* q = cluster.map_shared_rank(&sh.pub, r);
          const Cand* rc = cluster.map_shared_rank(&sh.cand[0], r);
          const int rn = (int)q->ncand;
          for (int l = 0; l < rn; ++l) {
            const uint64_t k2 = rc[l].key;
            rk += (k2 > key || (k2 == key && rc[l].v < v)) ? 1u : 0u;
          }
        }
        if (rk < Rin) set_bit(sh.grant_bits, sh.cand[j].s);
      }
    } else {
      // many members: narrow the exact key by 8-bit radix levels unless
      // every member holds the same fraction, then grant the remaining
      // tickets to the lowest ids holding the threshold fraction
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
      // members with key > thr are granted; key == thr by id order
      for (int g = tid; g < ngroups; g += blockDim.x)
        for (int i = 0; i < 4; ++i) {
          const int s = 4 * g + i;
          if (is_member(s) && exact_key(s) > thr) set_bit(sh.grant_bits, s);
        }
      __syncthreads();
      ordered_ranks(
          cluster, sh, ngroups,
          [&](int s) -> bool { return is_member(s) && exact_key(s) == thr; },
          [&](int s, uint32_t rk) {
            if (rk < need) set_bit(sh.grant_bits, s);
          });
    }
  }
  __syncthreads();

  // ---- pass E: counts = f + grant
  uint32_t* crow = p.counts + (int64_t)row * V;
  uint64_t csum = 0;
  const int offc = (int)((reinterpret_cast<uintptr_t>(crow + lo) / 4) & 3);
  auto count_at = [&](int s) -> uint32_t {
    uint32_t f, pos, b;
    unpack(s, &f, &pos, &b);
    uint32_t g = 0;
    if (pos) g = ((int)b > bstar || ((int)b == bstar && get_bit(sh.grant_bits, s))) ? 1u : 0u;
    return f + g;
  };
  if (status == DSPARK_ST_OK) {
    for (int g = tid; g < ngroups; g += blockDim.x) {
      const int s0 = 4 * g;
      const bool full = (s0 >= off) && (s0 + 3 < off + n);
      if (full && offc == off) {
        uint4 c4;
        c4.x = count_at(s0);
        c4.y = count_at(s0 + 1);
        c4.z = count_at(s0 + 2);
        c4.w = count_at(s0 + 3);
        csum += (uint64_t)c4.x + c4.y + c4.z + c4.w;
        *reinterpret_cast<uint4*>(crow + lo - off + s0) = c4;
      } else {
        for (int i = 0; i < 4; ++i) {
          const int s = s0 + i;
          if (s < off || s >= off + n) continue;
          const uint32_t c = count_at(s);
          csum += c;
          crow[lo - off + s] = c;
        }
      }
    }
  }
  csum = block_reduce(csum, OpAddU64(), sh.red64);
  if (tid == 0) sh.pub.csum = csum;
  cluster.sync();  // S7
  uint64_t csum_all = 0;
  for (int r = 0; r < kQCluster; ++r) csum_all += cluster.map_shared_rank(&sh.pub, r)->csum;
  if (status == DSPARK_ST_OK && csum_all != (uint64_t)kM) status = DSPARK_ST_ALLOC_INCONSISTENT;
  if (status != DSPARK_ST_OK)
    for (int v = lo + tid; v < hi; v += blockDim.x) crow[v] = 0u;
  if (rank == 0 && tid == 0) p.status[row] = status;
  cluster.sync();  // S8: no CTA leaves while a peer still reads its pub
}

int q_build_smem_bytes(int chunk, int top_k) {
  int slice = (chunk + 4) * 4;
  if (top_k > 0) {
    const int need = (int)sizeof(SparseEntry) * 1024;
    if (slice < need) slice = need;
  }
  return slice;
}

cudaError_t launch_q_build(const void* x, int dtype, int64_t ld, int n_rows, int V,
                           const float* temperature, int top_k, uint32_t* counts, int32_t* ids,
                           int32_t* nnz, int32_t* status, cudaStream_t stream) {
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
  const int smem = q_build_smem_bytes(chunk, top_k);
  cudaError_t err = cudaFuncSetAttribute(q_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  q_build_kernel<<<n_rows * kQCluster, kQThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dspark
