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

__device__ __forceinline__ const void* row_ptr(const VParams& p, int64_t r) {
  return reinterpret_cast<const char*>(p.z) + r * p.ld * (p.dtype == DSPARK_F32 ? 4 : 2);
}

// Fixed-point weight of token v for the final draw: residual max(p - q, 0)
// (qrow != NULL: dense counts; qsm: sparse lookup) or p itself.
struct DrawWeights {
  float m, s;
  const uint32_t* qrow;      // dense counts row or NULL
  const int32_t* sids;       // sparse ids row or NULL
  const uint32_t* scnt;      // sparse counts row
  int snnz;
  bool use_q;
};

__device__ __forceinline__ uint32_t q_count(const DrawWeights& w, int v) {
  if (w.qrow) return __ldg(w.qrow + v);
  if (w.sids) {
    int a = 0, b = w.snnz - 1;
    while (a <= b) {
      const int mid = (a + b) >> 1;
      const int id = __ldg(w.sids + mid);
      if (id == v) return __ldg(w.scnt + mid);
      if (id < v) a = mid + 1;
      else b = mid - 1;
    }
  }
  return 0u;
}

__device__ __forceinline__ uint64_t draw_weight(const DrawWeights& w, int v, float zv) {
  const float pv = (zv == -INFINITY) ? 0.0f : __fdiv_rn(expf(zv - w.m), w.s);
  float r = pv;
  if (w.use_q) {
    const float qv = (float)q_count(w, v) * 0x1p-24f;
    r = fmaxf(pv - qv, 0.0f);
  }
  return (uint64_t)__float2ull_rz(__fmul_rn(r, kTwo46f));
}

template <int kMode>
__global__ void __cluster_dims__(kVCluster, 1, 1) __launch_bounds__(kVThreads, 2)
    verify_kernel(VParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ VShared sh;
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / kVCluster;
  const int tid = threadIdx.x;
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
  int L = depth, pick = -1;
  uint32_t flags = 0;
  int writer = -1;     // rank of the CTA that found the drawn token
  bool drawn = false;  // the request reached its final draw (same in every CTA)

  for (int j = 0; j <= depth && status == DSPARK_ST_OK; ++j) {
    const void* row = row_ptr(p, (int64_t)b * (depth + 1) + j);
    const RowStat mine = slice_stat(row, p.dtype, lo, n, sh);
    if (tid == 0) sh.pub.st = mine;
    cluster.sync();
    RowStat st = cluster.map_shared_rank(&sh.pub, 0)->st;
    for (int r = 1; r < kVCluster; ++r) st = stat_merge(st, cluster.map_shared_rank(&sh.pub, r)->st);
    cluster.sync();  // pubs free again
    if (st.bad) {
      status = DSPARK_ST_NONFINITE;
      break;
    }
    if (st.m == -INFINITY) {
      status = DSPARK_ST_ZERO_MASS;
      break;
    }
    if (kMode == kGreedy) {
      if (j == depth || st.ami != drafts[j]) {
        L = j;
        pick = st.ami;
        break;
      }
      continue;
    }
    // ---- ratio verification
    DrawWeights w;
    w.m = st.m;
    w.s = st.s;
    w.qrow = nullptr;
    w.sids = nullptr;
    w.scnt = nullptr;
    w.snnz = 0;
    w.use_q = false;
    uint32_t purpose = DSPARK_PURPOSE_BONUS;
    if (j < depth) {
      const int x = drafts[j];
      const int64_t qr = (int64_t)b * depth + j;
      uint32_t c;
      if (p.top_k == 0) {
        w.qrow = p.counts + qr * V;
        c = __ldg(w.qrow + x);
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
        if (nz < 1 || nz > p.top_k) {
          if (tid == 0) sh.q_ok = 0;
        } else {
          uint64_t tot = 0;
          for (int i = tid; i < nz; i += blockDim.x) {
            const int id = ids[i];
            const uint32_t cc = cn[i];
            if (id < 0 || id >= V || cc == 0u || (i > 0 && ids[i - 1] >= id)) sh.q_ok = 0;
            if (id == x) sh.q_c = cc;
            tot += cc;
          }
          tot = block_reduce(tot, OpAddU64(), sh.red64);
          if (tid == 0 && tot != (uint64_t)kM) sh.q_ok = 0;
        }
        __syncthreads();
        if (!sh.q_ok) {
          status = DSPARK_ST_BAD_Q;
          break;
        }
        c = sh.q_c;
        w.sids = ids;
        w.scnt = cn;
        w.snnz = nz;
      }
      if (c == 0u) {
        status = DSPARK_ST_BAD_DRAFT;
        break;
      }
      const float zx = load_logit(row, p.dtype, x);
      const float px = (zx == -INFINITY) ? 0.0f : __fdiv_rn(expf(zx - st.m), st.s);
      const uint32_t U = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_ACCEPT) >> 8;
      const double uc = (double)((uint64_t)U * (uint64_t)c);
      const double p48 = (double)px * 281474976710656.0;
      if (fabs(uc * 0x1p-48 - (double)px) <= 1e-6 * ((double)c * 0x1p-24))
        flags |= DSPARK_FLAG_AMBIG_ACCEPT;
      if (uc < p48) continue;  // accepted
      L = j;
      w.use_q = true;
      purpose = DSPARK_PURPOSE_RESIDUAL;
      if (p.top_k == 0) {
        // the dense residual row must carry mass M
        uint64_t cs = 0;
        for (int v = lo + tid; v < lo + n; v += blockDim.x) cs += __ldg(w.qrow + v);
        cs = block_reduce(cs, OpAddU64(), sh.red64);
        if (tid == 0) sh.pub.csum = cs;
        cluster.sync();
        uint64_t all = 0;
        for (int r = 0; r < kVCluster; ++r) all += cluster.map_shared_rank(&sh.pub, r)->csum;
        cluster.sync();
        if (all != (uint64_t)kM) {
          status = DSPARK_ST_BAD_Q;
          break;
        }
      }
    } else {
      L = depth;
    }
    // ---- final draw over row j: residual (ratio rejection) or p (bonus)
    const uint32_t wdraw = draw_u32(p.seed, req, (uint32_t)j, purpose);
    for (int attempt = 0; attempt < 2; ++attempt) {
      uint64_t zs = 0;
      row_foreach(row, p.dtype, lo, n, [&](int v, float zv) { zs += draw_weight(w, v, zv); });
      zs = block_reduce(zs, OpAddU64(), sh.red64);
      if (tid == 0) sh.pub.z = zs;
      cluster.sync();
      uint64_t before = 0, Z = 0;
      for (int r = 0; r < kVCluster; ++r) {
        const uint64_t zr = cluster.map_shared_rank(&sh.pub, r)->z;
        if (r < rank) before += zr;
        Z += zr;
      }
      cluster.sync();
      if (Z == 0ull && w.use_q) {  // no residual mass: draw from p instead
        flags |= DSPARK_FLAG_DEGENERATE;
        w.use_q = false;
        continue;
      }
      const uint64_t T = __umul64hi((uint64_t)wdraw << 32, Z);  // floor(w * Z / 2^32) < Z
      // exactly one CTA's slice holds T; it walks its slice in id order and
      // writes the request's outputs
      drawn = true;
      writer = -1;
      const bool mine_has = (T >= before) && (T < before + zs);
      if (mine_has) {
        // ordered scan over groups of this slice
        __shared__ int found;
        __shared__ uint32_t found_near;
        if (tid == 0) {
          found = -1;
          found_near = 0u;
        }
        __syncthreads();
        const int gsz = (p.dtype == DSPARK_F32) ? 4 : 8;
        const int offs = (p.dtype == DSPARK_F32)
                             ? (int)((reinterpret_cast<uintptr_t>(reinterpret_cast<const float*>(row) + lo) >> 2) & 3)
                             : (int)((reinterpret_cast<uintptr_t>(reinterpret_cast<const unsigned short*>(row) + lo) >> 1) & 7);
        const int ng = (offs + n + gsz - 1) / gsz;
        uint64_t base = before;
        for (int t0 = 0; t0 < ng; t0 += blockDim.x) {
          const int g = t0 + tid;
          uint64_t wv[8];
          uint64_t mysum = 0;
          for (int i = 0; i < gsz; ++i) {
            const int s = g * gsz + i;
            wv[i] = 0;
            if (g < ng && s >= offs && s < offs + n) {
              const int v = lo - offs + s;
              wv[i] = draw_weight(w, v, load_logit(row, p.dtype, v));
            }
            mysum += wv[i];
          }
          uint64_t tot;
          const uint64_t incl = block_inclusive_scan_u64(mysum, sh.red64, &tot);
          uint64_t cum = base + incl - mysum;
          if (T >= cum && T < cum + mysum) {
            for (int i = 0; i < gsz; ++i) {
              const uint64_t prev = cum;
              cum += wv[i];
              if (T < cum) {
                found = lo - offs + g * gsz + i;
                found_near = (T - prev <= kNearTol || cum - T <= kNearTol) ? 1u : 0u;
                break;
              }
            }
          }
          base += tot;
          __syncthreads();
          if (found >= 0) break;
        }
        pick = found;
        if (found_near) flags |= DSPARK_FLAG_NEAR_BOUNDARY;
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
  cluster.sync();
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
  if (mode == kGreedy)
    verify_kernel<kGreedy><<<B * kVCluster, kVThreads, 0, stream>>>(p);
  else
    verify_kernel<kRatio><<<B * kVCluster, kVThreads, 0, stream>>>(p);
  return cudaGetLastError();
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
