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
//
// One cluster per row, launched in row order: with G clusters resident at
// once, row r + G starts about when row r ends, so each cluster prefetches
// its part of row r + G into L2 while it builds row r, and that row's bulk
// copies then read L2.  (A persistent grid of G clusters taking rows
// r, r + G, ... measured 15% slower: fixed placements keep the slow CTAs
// slow, where fresh clusters rebalance.)
#define DSPARK_TU 3  // this file's number in the checked build's site codes
#include <mutex>

#include "q_dense.cuh"

namespace dspark {
using namespace qdense;

__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kThr, 3)
    q_dense_kernel(Params p, int ahead) {
  __shared__ DShared sh;
  __shared__ uint64_t mbar[kTma];
  extern __shared__ __align__(128) float sl[];
  if (threadIdx.x == 0) {
    for (int c = 0; c < kTma; ++c) mbar_init(&mbar[c], 1);
    mbar_init_fence();
  }
  __syncthreads();
  uint32_t phase = 0;
  const int row = blockIdx.x / kCl;
  q_dense_row(p, row, sh, sl, mbar, phase, nullptr,
              (ahead > 0 && row + ahead < p.n_rows) ? row + ahead : -1);
}

namespace {
// Clusters of q_dense_kernel resident at once for a dynamic shared size, per
// device (queried once).
int q_dense_wave(int smem) {
  static std::mutex mu;
  static int cached[64][2];  // {smem, clusters}
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev][0] == smem && cached[dev][1] > 0) return cached[dev][1];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCl * 64);
  cfg.blockDim = dim3(kThr);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = kCl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (void*)q_dense_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cached[dev][0] = smem;
  cached[dev][1] = n;
  return n;
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
  q_dense_kernel<<<n_rows * kCl, kThr, smem, stream>>>(p, q_dense_wave(smem));
  return cudaGetLastError();
}

DSPARK_CHECK_COLLECTOR(q_dense)

}  // namespace dspark
