// chain.cu -- the Markov-conditioned draft chain ("Remote DSpark drafter --
// wire and state contract", section 2: the sequential Markov step adds the
// bias row of the previous sampled token to the base logits, the anchor at
// step 0; section 6.3: the optional margin is top1 - top2 of (base + Markov)
// logits at each step).
//
// One 8-CTA cluster per request walks its draft rows in order.  For row j
// the dense q build with its draft draw (the q_dense row code) runs on
// z = RN(x + bias[prev mod n_bias]), formed in shared memory as each CTA's
// eighth of the base row lands (the bias row is read alongside), and the
// same pass keeps the row's two largest z for the margin.  The CTA that
// draws the token stores it into every CTA's shared memory before the row's
// last cluster barrier, and it conditions row j + 1; the next row's base part
// is prefetched into L2 meanwhile, its bias part when the row starts.  A
// refused row refuses the rest of its chain with the same status.
#define DSPARK_TU 1  // this file's number in the checked build's site codes
#include <cfloat>

#include "q_dense.cuh"

namespace dspark {
namespace {

using qdense::kCl;
using qdense::kThr;

struct ChainParams {
  const float* bias;  // [n_bias][bias_ld] or null
  int64_t bias_ld;
  int n_bias;
  const int32_t* anchors;  // [B]
  float* margins;          // [B * depth] or null
  int depth;
  int V;
};

__device__ __noinline__ int chain_q_row(const qdense::Params& qp, int row, qdense::DShared& sh,
                                        float* sl, uint64_t* mbar, uint32_t& phase,
                                        int next_row, const float* zbias) {
  return qdense::q_dense_row(qp, row, sh, sl, mbar, phase, nullptr, next_row, true, zbias);
}

__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kThr, 3)
    q_chain_kernel(qdense::Params qp, ChainParams cp) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ qdense::DShared sh;
  __shared__ uint64_t mbar[qdense::kTma];
  extern __shared__ __align__(128) float sl[];
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int c = 0; c < qdense::kTma; ++c) mbar_init(&mbar[c], 1);
    mbar_init_fence();
  }
  __syncthreads();
  uint32_t phase = 0;
  const int b = blockIdx.x / kCl;
  const int V = cp.V, depth = cp.depth;
  const int lo = min(V, rank * qp.chunk), hi = min(V, lo + qp.chunk);
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
    const float* brow = cp.bias ? cp.bias + (int64_t)(prev % cp.n_bias) * cp.bias_ld : nullptr;
    const int st = chain_q_row(qp, row, sh, sl, mbar, phase, (j + 1 < depth) ? row + 1 : -1, brow);
    // the drawn token is in this CTA's shared memory (stored before the
    // row's last cluster barrier), the status the same in every CTA
    const int tok = sh.chain_tok;
    if (cp.margins && rank == 0 && tid == 0) {
      float mg = 0.0f;
      if (st == DSPARK_ST_OK) {
        const float m1 = sh.top1, m2 = sh.top2;
        mg = (m2 == -INFINITY) ? FLT_MAX : __fsub_rn(m1, m2);
        if (!(mg <= FLT_MAX)) mg = FLT_MAX;
      }
      cp.margins[row] = mg;
    }
    if (st != DSPARK_ST_OK) refused = st;
    else if (tok < 0) refused = DSPARK_ST_INTERNAL;
    else prev = tok;
  }
}

}  // namespace

cudaError_t launch_q_chain(const void* x, int dtype, int64_t ld, int B, int depth, int V,
                           const float* temperature, const float* bias, int64_t bias_ld,
                           int n_bias, const int32_t* anchors, uint64_t seed,
                           const uint32_t* request_ids, uint32_t* counts, int32_t* tokens,
                           int32_t* status, float* margins, cudaStream_t stream) {
  qdense::Params qp;
  qp.x = x;
  qp.dtype = dtype;
  qp.ld = ld;
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
  ChainParams cp{bias, bias_ld, n_bias, anchors, margins, depth, V};
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

DSPARK_CHECK_COLLECTOR(chain)

}  // namespace dspark
