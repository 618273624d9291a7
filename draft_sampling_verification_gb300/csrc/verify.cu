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
#define DSPARK_TU 9  // this file's number in the checked build's site codes
#include <mutex>

#include "verify.cuh"

namespace dspark {
using namespace vfy;

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
//
// Cluster size: bf16 rows take 5-CTA clusters (a 51 KB slice per CTA, four
// CTAs per SM within 64 registers), so more requests walk their row chains
// at once, each on shorter slices, than with 4 or 8 CTAs at three per SM.
// fp32 rows take 8 (a 64 KB slice, three CTAs per SM), or 7 (a 72 KB slice,
// still three per SM) when the batch does not fit the GPU at once with 8:
// one more request in eight is resident, at a slice an eighth longer.
template <bool kG, bool kR, int kDt, bool kMatch, int NC>
__global__ void __cluster_dims__(NC, 1, 1)
    __launch_bounds__(kVThreads, (kDt == DSPARK_BF16) ? 4 : 3)
    verify_kernel(VParams p) {
  __shared__ VSh2 sh;
  __shared__ uint64_t mbar[kVTma];
  extern __shared__ __align__(128) unsigned char vbuf[];
  if (threadIdx.x == 0) {
    for (int c = 0; c < kVTma; ++c) mbar_init(&mbar[c], 1);
    mbar_init_fence();
  }
  __syncthreads();
  uint32_t phase = 0;
  verify_request<kG, kR, kDt, NC, kMatch>(p, blockIdx.x / NC, sh, vbuf, mbar, phase, nullptr,
                                          nullptr);
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

static int verify_chunk(int V, int nc) {
  int c = (V + nc - 1) / nc;
  return (c + 7) & ~7;
}

// Clusters of a verify kernel resident at once for a dynamic shared size,
// per device and cluster size (queried once).
template <typename K>
int verify_wave(K kern, int nc, int smem) {
  static std::mutex mu;
  static int cached[64][9][2];  // [device][cluster size] {smem, clusters}
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || nc < 1 || nc > 8) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev][nc][0] == smem && cached[dev][nc][1] > 0) return cached[dev][nc][1];
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nc * 64);
  cfg.blockDim = dim3(kVThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = nc;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cached[dev][nc][0] = smem;
  cached[dev][nc][1] = n;
  return n;
}

// Launches verify_kernel<kG, kR, kDt, kMatch, NC> for the p.B requests:
// bf16 rows on 5-CTA clusters; fp32 rows on 8, or on 7 when the batch does
// not fit at once on 8-CTA clusters and more 7-CTA clusters do.
template <bool kG, bool kR, int kDt, bool kMatch>
cudaError_t launch_verify_kernel(VParams p, cudaStream_t stream) {
  constexpr int esz = (kDt == DSPARK_F32) ? 4 : 2;
  auto go = [&](auto kern, int nc) -> cudaError_t {
    p.chunk = verify_chunk(p.V, nc);
    // the slice buffer: chunk elements plus one 16-byte group of slack
    const int smem = p.chunk * esz + 32;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    kern<<<p.B * nc, kVThreads, smem, stream>>>(p);
    return cudaGetLastError();
  };
  if constexpr (kDt == DSPARK_BF16) {
    return go(verify_kernel<kG, kR, kDt, kMatch, 5>, 5);
  } else {
    const int w8 = verify_wave(verify_kernel<kG, kR, kDt, kMatch, 8>, 8,
                               verify_chunk(p.V, 8) * esz + 32);
    if (w8 > 0 && p.B > w8) {
      const int w7 = verify_wave(verify_kernel<kG, kR, kDt, kMatch, 7>, 7,
                                 verify_chunk(p.V, 7) * esz + 32);
      if (w7 > w8) return go(verify_kernel<kG, kR, kDt, kMatch, 7>, 7);
    }
    return go(verify_kernel<kG, kR, kDt, kMatch, 8>, 8);
  }
}

cudaError_t launch_verify_modes(const void* z, int dtype, int64_t ld, int B, int depth, int V,
                                const int32_t* drafts, const uint32_t* counts, const int32_t* ids,
                                const int32_t* nnz, int top_k, uint64_t seed,
                                const uint32_t* request_ids, int32_t* g_acc, int32_t* g_com,
                                int32_t* g_st, int32_t* r_acc, int32_t* r_com, uint32_t* r_flags,
                                int32_t* r_st, cudaStream_t stream) {
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
  p.g_accept_len = g_acc;
  p.g_committed = g_com;
  p.g_status = g_st;
  p.r_accept_len = r_acc;
  p.r_committed = r_com;
  p.r_flags = r_flags;
  p.r_status = r_st;
  const bool g = g_acc != nullptr, r = r_acc != nullptr;
  if (dtype == DSPARK_F32) {
    if (g && r) return launch_verify_kernel<true, true, DSPARK_F32, false>(p, stream);
    if (g) return launch_verify_kernel<true, false, DSPARK_F32, false>(p, stream);
    return launch_verify_kernel<false, true, DSPARK_F32, false>(p, stream);
  }
  if (g && r) return launch_verify_kernel<true, true, DSPARK_BF16, false>(p, stream);
  if (g) return launch_verify_kernel<true, false, DSPARK_BF16, false>(p, stream);
  return launch_verify_kernel<false, true, DSPARK_BF16, false>(p, stream);
}

// The match mode: its outputs take the ratio mode's slots.
cudaError_t launch_verify_match(const void* z, int dtype, int64_t ld, int B, int depth, int V,
                                const int32_t* drafts, uint64_t seed,
                                const uint32_t* request_ids, int32_t* accept_len,
                                int32_t* committed, uint32_t* flags, int32_t* status,
                                cudaStream_t stream) {
  VParams p;
  p.z = z;
  p.dtype = dtype;
  p.ld = ld;
  p.B = B;
  p.depth = depth;
  p.V = V;
  p.drafts = drafts;
  p.counts = nullptr;
  p.ids = nullptr;
  p.nnz = nullptr;
  p.top_k = 0;
  p.seed = seed;
  p.request_ids = request_ids;
  p.g_accept_len = nullptr;
  p.g_committed = nullptr;
  p.g_status = nullptr;
  p.r_accept_len = accept_len;
  p.r_committed = committed;
  p.r_flags = flags;
  p.r_status = status;
  return dtype == DSPARK_F32 ? launch_verify_kernel<false, false, DSPARK_F32, true>(p, stream)
                             : launch_verify_kernel<false, false, DSPARK_BF16, true>(p, stream);
}

cudaError_t launch_verify(int mode, const void* z, int dtype, int64_t ld, int B, int depth, int V,
                          const int32_t* drafts, const uint32_t* counts, const int32_t* ids,
                          const int32_t* nnz, int top_k, uint64_t seed,
                          const uint32_t* request_ids, int32_t* accept_len, int32_t* committed,
                          uint32_t* flags, int32_t* status, cudaStream_t stream) {
  if (mode == kGreedy)
    return launch_verify_modes(z, dtype, ld, B, depth, V, drafts, counts, ids, nnz, top_k, seed,
                               request_ids, accept_len, committed, status, nullptr, nullptr,
                               nullptr, nullptr, stream);
  return launch_verify_modes(z, dtype, ld, B, depth, V, drafts, counts, ids, nnz, top_k, seed,
                             request_ids, nullptr, nullptr, nullptr, accept_len, committed, flags,
                             status, stream);
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
  p.chunk = verify_chunk(V, kVCluster);
  target_probs_kernel<<<n_rows * kVCluster, kVThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

// The verifier's optional statistics from its per-request flags: one CTA
// counts, for each DSPARK_FLAG_* bit k (ambiguous decision, draw near a
// boundary, degenerate residual), the requests carrying it into stats[k].
__global__ void __launch_bounds__(256) verify_stats_kernel(const uint32_t* flags, int B,
                                                           uint32_t* stats) {
  __shared__ uint32_t part[3][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t c[3] = {0u, 0u, 0u};
  for (int b = threadIdx.x; b < B; b += 256) {
    const uint32_t f = flags[b];
#pragma unroll
    for (int k = 0; k < 3; ++k) c[k] += (f >> k) & 1u;
  }
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    c[k] = __reduce_add_sync(0xffffffffu, c[k]);
    if (lane == 0) part[k][warp] = c[k];
  }
  __syncthreads();
  if (threadIdx.x < 3) {
    uint32_t t = 0;
    for (int w = 0; w < 8; ++w) t += part[threadIdx.x][w];
    stats[threadIdx.x] = t;
  }
}

cudaError_t launch_verify_stats(const uint32_t* flags, int B, uint32_t* stats,
                                cudaStream_t stream) {
  verify_stats_kernel<<<1, 256, 0, stream>>>(flags, B, stats);
  return cudaGetLastError();
}

DSPARK_CHECK_COLLECTOR(verify)

}  // namespace dspark
