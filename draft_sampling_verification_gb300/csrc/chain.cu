// chain.cu -- the Markov-conditioned draft chain ("Remote DSpark drafter --
// wire and state contract", section 2: the sequential Markov step adds the
// bias row of the previous sampled token to the base logits, the anchor at
// step 0; section 6.3: the optional margin is top1 - top2 of (base + Markov)
// logits at each step).
//
// One 8-CTA cluster per request walks its draft rows in order.  For row j
// every CTA writes z = RN(x + bias[prev mod n_bias]) over its eighth of the
// row into the caller's workspace and keeps the top two finite z; the
// workspace writes are made visible to the bulk copies (an async-proxy fence,
// then a cluster barrier), and the dense q build with its draft draw (the
// q_dense row code) runs on z.  The drawn token goes to every CTA through
// distributed shared memory and conditions row j + 1.  A refused row refuses
// the rest of its chain with the same status.
#include <cfloat>

#include "q_dense.cuh"

namespace dspark {
namespace {

using qdense::kCl;
using qdense::kThr;

struct ChainParams {
  const void* x;  // base logits, row r at x + r * ld elements
  int dtype;
  int64_t ld;
  const float* bias;  // [n_bias][bias_ld] or null
  int64_t bias_ld;
  int n_bias;
  const int32_t* anchors;  // [B]
  float* ws;               // [B * depth][V]: z rows
  float* margins;          // [B * depth] or null
  int depth;
  int V;
};

struct ChainShared {
  float t1[kCl], t2[kCl];  // pushed to rank 0: each CTA's top two finite z
  int tok, st;             // pushed by rank 0: the row's token and status
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

__device__ __noinline__ void chain_q_row(const qdense::Params& qp, int row, qdense::DShared& sh,
                                         float* sl, uint64_t* mbar, uint32_t& phase) {
  qdense::q_dense_row(qp, row, sh, sl, mbar, phase, nullptr);
}

__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kThr, 3)
    q_chain_kernel(qdense::Params qp, ChainParams cp) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ qdense::DShared sh;
  __shared__ uint64_t mbar[qdense::kTma];
  __shared__ ChainShared cs;
  __shared__ float wt1[kThr / 32], wt2[kThr / 32];
  extern __shared__ __align__(128) float sl[];
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int c = 0; c < qdense::kTma; ++c) mbar_init(&mbar[c], 1);
    mbar_init_fence();
  }
  __syncthreads();
  uint32_t phase = 0;
  const int b = blockIdx.x / kCl;
  const int V = cp.V, depth = cp.depth;
  const int chunk = (V + kCl - 1) / kCl;
  const int lo = min(V, rank * chunk), hi = min(V, lo + chunk);
  const int esz = (cp.dtype == DSPARK_F32) ? 4 : 2;
  const int anchor = cp.anchors[b];
  int prev = anchor;
  int refused = (anchor < 0 || anchor >= V) ? DSPARK_ST_BAD_DRAFT : DSPARK_ST_OK;

  for (int j = 0; j < depth; ++j) {
    const int row = b * depth + j;
    if (refused != DSPARK_ST_OK) {
      for (int v = lo + tid; v < hi; v += kThr) qp.counts[(int64_t)row * V + v] = 0u;
      if (rank == 0 && tid == 0) {
        qp.status[row] = refused;
        qp.tokens[row] = -1;
        if (cp.margins) cp.margins[row] = 0.0f;
      }
      continue;
    }
    // ---- z over this CTA's range, and its top two finite values
    const char* xrow = reinterpret_cast<const char*>(cp.x) + (int64_t)row * cp.ld * esz;
    const float* brow = cp.bias ? cp.bias + (int64_t)(prev % cp.n_bias) * cp.bias_ld : nullptr;
    float* zrow = cp.ws + (int64_t)row * V;
    float t1 = -INFINITY, t2 = -INFINITY;
    for (int v = lo + tid; v < hi; v += kThr) {
      const float x = load_logit(xrow, cp.dtype, v);
      const float z = brow ? __fadd_rn(x, __ldg(brow + v)) : x;
      zrow[v] = z;
      if (z > -INFINITY && z < INFINITY) top2_merge(t1, t2, z, -INFINITY);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float o1 = __shfl_xor_sync(0xffffffffu, t1, o);
      const float o2 = __shfl_xor_sync(0xffffffffu, t2, o);
      top2_merge(t1, t2, o1, o2);
    }
    if (lane == 0) {
      wt1[warp] = t1;
      wt2[warp] = t2;
    }
    // the workspace rows are read next by bulk copies (the async proxy)
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      float c1 = wt1[0], c2 = wt2[0];
      for (int w = 1; w < kThr / 32; ++w) top2_merge(c1, c2, wt1[w], wt2[w]);
      ChainShared* r0 = cluster.map_shared_rank(&cs, 0);
      r0->t1[rank] = c1;
      r0->t2[rank] = c2;
    }
    cluster.sync();
    float m1 = -INFINITY, m2 = -INFINITY;
    if (rank == 0 && tid == 0)
      for (int r = 0; r < kCl; ++r) top2_merge(m1, m2, cs.t1[r], cs.t2[r]);

    // ---- the dense q of z and its draft draw
    chain_q_row(qp, row, sh, sl, mbar, phase);

    // ---- the drawn token (and status) to every CTA
    __threadfence();
    cluster.sync();
    if (rank == 0 && tid == 0) {
      const int tok = *reinterpret_cast<volatile const int32_t*>(qp.tokens + row);
      const int st = *reinterpret_cast<volatile const int32_t*>(qp.status + row);
      if (cp.margins) {
        float mg = 0.0f;
        if (st == DSPARK_ST_OK) {
          mg = (m2 == -INFINITY) ? FLT_MAX : __fsub_rn(m1, m2);
          if (!(mg <= FLT_MAX)) mg = FLT_MAX;
        }
        cp.margins[row] = mg;
      }
      for (int r = 0; r < kCl; ++r) {
        ChainShared* peer = cluster.map_shared_rank(&cs, r);
        peer->tok = tok;
        peer->st = st;
      }
    }
    cluster.sync();
    if (cs.st != DSPARK_ST_OK || cs.tok < 0) refused = (cs.st != DSPARK_ST_OK) ? cs.st
                                                                               : DSPARK_ST_INTERNAL;
    else prev = cs.tok;
  }
}

}  // namespace

cudaError_t launch_q_chain(const void* x, int dtype, int64_t ld, int B, int depth, int V,
                           const float* temperature, const float* bias, int64_t bias_ld,
                           int n_bias, const int32_t* anchors, uint64_t seed,
                           const uint32_t* request_ids, float* workspace, uint32_t* counts,
                           int32_t* tokens, int32_t* status, float* margins,
                           cudaStream_t stream) {
  qdense::Params qp;
  qp.x = workspace;
  qp.dtype = DSPARK_F32;
  qp.ld = V;
  qp.n_rows = B * depth;
  qp.V = V;
  qp.temperature = temperature;
  qp.counts = counts;
  qp.status = status;
  int qchunk = (V + kCl - 1) / kCl;
  qchunk = (qchunk + 3) & ~3;
  qp.chunk = qchunk;
  qp.tokens = tokens;
  qp.seed = seed;
  qp.request_ids = request_ids;
  qp.depth = depth;
  ChainParams cp{x, dtype, ld, bias, bias_ld, n_bias, anchors, workspace, margins, depth, V};
  const int smem = (qchunk + 4) * 4;
  cudaError_t e =
      cudaFuncSetAttribute(q_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(q_chain_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  q_chain_kernel<<<B * kCl, kThr, smem, stream>>>(qp, cp);
  return cudaGetLastError();
}

}  // namespace dspark
