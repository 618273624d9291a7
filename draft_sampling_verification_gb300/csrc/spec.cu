// spec.cu -- the whole speculative step in one call ("PP1 q transport and
// scheduling design", Distribution contract and precision; "DeepSeek-V4.1
// DSpark", State and sampling contracts): the dense dyadic q of every draft
// row with its draft draw (the q_dense row code) and the greedy and/or ratio
// verification of every request (the verify code).  Outputs are those of
// dspark_q_build_sample followed by dspark_verify_greedy /
// dspark_verify_ratio, whichever schedule runs.
//
// Two schedules:
//   separate    the q_dense kernel, then one verify kernel doing every
//               requested mode in one pass over the target rows.
//   one launch  persistent 8-CTA clusters, as many as fit at once, take work
//               items from a counter in the caller's workspace: one q row, or
//               one request's verification.  The items are interleaved so
//               that a request's verification comes about two waves of rows
//               after its own rows: it then overlaps other clusters' q
//               builds, and its rows are normally done when it starts (each
//               finished row increments the request's counter in the
//               workspace; the verifying cluster waits on it with a bounded
//               wait).  It pays off only while all items fit in one wave.
#define DSPARK_TU 7  // this file's number in the checked build's site codes
#include <mutex>

#include "q_dense.cuh"
#include "verify.cuh"

namespace dspark {
namespace {

static_assert(qdense::kCl == vfy::kVCluster && qdense::kThr == vfy::kVThreads &&
                  qdense::kTma == vfy::kVTma,
              "the q and verify phases share one cluster shape and one set of mbarriers");

struct SpecShared {
  union {
    qdense::DShared q;
    vfy::VSh2 v;
  };
};

struct WorkParams {
  uint32_t* next;   // item counter (zero at launch)
  uint32_t* ready;  // [B] finished q rows per request (zero at launch)
  int B, depth, lag, n_items;
};

// Item k of the interleaved order: the q rows of requests [0, l) (l =
// min(lag, B)); then for each request r in [l, B) its q rows followed by the
// verification of request r - lag; then the verifications of the last l
// requests.
__device__ __forceinline__ void decode_item(int k, const WorkParams& w, bool* verify, int* idx) {
  const int l = min(w.lag, w.B);
  const int n1 = l * w.depth;
  if (k < n1) {
    *verify = false;
    *idx = k;
    return;
  }
  k -= n1;
  const int n2 = (w.B - l) * (w.depth + 1);
  if (k < n2) {
    const int r = l + k / (w.depth + 1), o = k % (w.depth + 1);
    *verify = (o == w.depth);
    *idx = *verify ? r - w.lag : r * w.depth + o;
    return;
  }
  *verify = true;
  *idx = (w.B - l) + (k - n2);
}

// The two phases as calls, so that each is register-allocated on its own.
__device__ __noinline__ void q_row(const qdense::Params& qp, int row, qdense::DShared& sh,
                                   float* sl, uint64_t* mbar, uint32_t& phase, uint32_t* ready) {
  qdense::q_dense_row(qp, row, sh, sl, mbar, phase, ready);
}

template <bool kG, bool kR, int kDt>
__device__ __noinline__ void verify_call(const vfy::VParams& vp, int b, vfy::VSh2& sh,
                                         unsigned char* dyn, uint64_t* mbar, uint32_t& phase) {
  // q rows come from other clusters of this launch: coherent loads of q
  vfy::verify_request<kG, kR, kDt, vfy::kVCluster, false, true>(vp, b, sh, dyn, mbar, phase,
                                                                 nullptr, nullptr);
}

template <bool kG, bool kR, int kDt>
__global__ void __cluster_dims__(qdense::kCl, 1, 1) __launch_bounds__(qdense::kThr, 3)
    spec_step_kernel(qdense::Params qp, vfy::VParams vp, WorkParams wp) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ SpecShared sh;
  __shared__ uint64_t mbar[qdense::kTma];
  __shared__ int item_slot;
  __shared__ int wait_ok;
  extern __shared__ __align__(128) unsigned char dyn[];
  const int rank = (int)cluster.block_rank();
  if (threadIdx.x == 0) {
    for (int c = 0; c < qdense::kTma; ++c) mbar_init(&mbar[c], 1);
    mbar_init_fence();
  }
  __syncthreads();
  uint32_t phase = 0;
  for (;;) {
    if (rank == 0 && threadIdx.x == 0) {
      const int k = (int)atomicAdd(wp.next, 1u);
      for (int r = 0; r < qdense::kCl; ++r) *cluster.map_shared_rank(&item_slot, r) = k;
    }
    cluster.sync();
    const int k = item_slot;
    if (k >= wp.n_items) break;
    bool is_v;
    int idx;
    decode_item(k, wp, &is_v, &idx);
    if (!DSPARK_CHECK(is_v ? (idx >= 0 && idx < wp.B) : (idx >= 0 && idx < wp.B * wp.depth)))
      continue;
    if (!is_v) {
      q_row(qp, idx, sh.q, reinterpret_cast<float*>(dyn), mbar, phase, wp.ready);
      continue;
    }
    // the request's q rows must be finished (normally long since)
    if (rank == 0 && threadIdx.x == 0) {
      const int ok = wait_count(&wp.ready[idx], (uint32_t)wp.depth) ? 1 : 0;
      __threadfence();
      for (int r = 0; r < qdense::kCl; ++r) *cluster.map_shared_rank(&wait_ok, r) = ok;
    }
    cluster.sync();
    if (wait_ok) {
      verify_call<kG, kR, kDt>(vp, idx, sh.v, dyn, mbar, phase);
    } else if (rank == 0 && threadIdx.x == 0) {
      // rows not finished within the wait limit: the request is refused
      const int depth = wp.depth;
      if (kG) {
        vp.g_accept_len[idx] = 0;
        for (int i = 0; i <= depth; ++i) vp.g_committed[(int64_t)idx * (depth + 1) + i] = -1;
        vp.g_status[idx] = DSPARK_ST_TIMEOUT;
      }
      if (kR) {
        vp.r_accept_len[idx] = 0;
        for (int i = 0; i <= depth; ++i) vp.r_committed[(int64_t)idx * (depth + 1) + i] = -1;
        if (vp.r_flags) vp.r_flags[idx] = 0u;
        vp.r_status[idx] = DSPARK_ST_TIMEOUT;
      }
    }
  }
}

}  // namespace

cudaError_t launch_q_dense(const void* x, int dtype, int64_t ld, int n_rows, int V,
                           const float* temperature, uint32_t* counts, int32_t* status,
                           int32_t* tokens, uint64_t seed, const uint32_t* request_ids, int depth,
                           cudaStream_t stream);
cudaError_t launch_verify_modes(const void* z, int dtype, int64_t ld, int B, int depth, int V,
                                const int32_t* drafts, const uint32_t* counts, const int32_t* ids,
                                const int32_t* nnz, int top_k, uint64_t seed,
                                const uint32_t* request_ids, int32_t* g_acc, int32_t* g_com,
                                int32_t* g_st, int32_t* r_acc, int32_t* r_com, uint32_t* r_flags,
                                int32_t* r_st, cudaStream_t stream);

// The schedule DSPARK_SCHEDULE_AUTO takes.  Upper bound on resident 8-CTA
// clusters: three CTAs per SM on 152 SMs.  Beyond it the items cannot all run
// in one wave and the separate launches are faster (a verification item holds
// a q-sized cluster slot while it is latency-bound); with one request there is
// nothing to overlap.
int spec_step_schedule(int B, int depth) {
  constexpr int kMaxWave = (152 * 3) / qdense::kCl;
  return (B < 2 || B * (depth + 1) > kMaxWave) ? DSPARK_SCHEDULE_SEPARATE
                                               : DSPARK_SCHEDULE_ONE_LAUNCH;
}

cudaError_t launch_spec_step(const void* xd, int d_dtype, int64_t ld_d, const void* xt,
                             int t_dtype, int64_t ld_t, int B, int depth, int V,
                             const float* temperature, uint64_t seed,
                             const uint32_t* request_ids, uint32_t* counts, int32_t* tokens,
                             int32_t* row_status, int32_t* g_acc, int32_t* g_com, int32_t* g_st,
                             int32_t* r_acc, int32_t* r_com, uint32_t* r_flags, int32_t* r_st,
                             uint32_t* workspace, int schedule, cudaStream_t stream) {
  const int n_items = B * depth + B;
  if (schedule == DSPARK_SCHEDULE_AUTO) schedule = spec_step_schedule(B, depth);
  if (schedule == DSPARK_SCHEDULE_SEPARATE) {
    cudaError_t e = launch_q_dense(xd, d_dtype, ld_d, B * depth, V, temperature, counts,
                                   row_status, tokens, seed, request_ids, depth, stream);
    if (e != cudaSuccess) return e;
    return launch_verify_modes(xt, t_dtype, ld_t, B, depth, V, tokens, counts, nullptr, nullptr,
                               0, seed, request_ids, g_acc, g_com, g_st, r_acc, r_com, r_flags,
                               r_st, stream);
  }

  qdense::Params qp;
  qp.x = xd;
  qp.dtype = d_dtype;
  qp.ld = ld_d;
  qp.n_rows = B * depth;
  qp.V = V;
  qp.temperature = temperature;
  qp.counts = counts;
  qp.status = row_status;
  int qchunk = (V + qdense::kCl - 1) / qdense::kCl;
  qchunk = (qchunk + 3) & ~3;
  qp.chunk = qchunk;
  qp.tokens = tokens;
  qp.seed = seed;
  qp.request_ids = request_ids;
  qp.depth = depth;

  vfy::VParams vp;
  vp.z = xt;
  vp.dtype = t_dtype;
  vp.ld = ld_t;
  vp.B = B;
  vp.depth = depth;
  vp.V = V;
  vp.drafts = tokens;
  vp.counts = counts;
  vp.ids = nullptr;
  vp.nnz = nullptr;
  vp.top_k = 0;
  vp.seed = seed;
  vp.request_ids = request_ids;
  vp.g_accept_len = g_acc;
  vp.g_committed = g_com;
  vp.g_status = g_st;
  vp.r_accept_len = r_acc;
  vp.r_committed = r_com;
  vp.r_flags = r_flags;
  vp.r_status = r_st;
  int vchunk = (V + vfy::kVCluster - 1) / vfy::kVCluster;
  vchunk = (vchunk + 7) & ~7;
  vp.chunk = vchunk;

  WorkParams wp;
  wp.next = workspace;
  wp.ready = workspace + 1;
  wp.B = B;
  wp.depth = depth;
  wp.n_items = n_items;

  using SpecKernel = void (*)(qdense::Params, vfy::VParams, WorkParams);
  const bool g = g_acc != nullptr, r = r_acc != nullptr;
  SpecKernel kern;
  if (t_dtype == DSPARK_F32)
    kern = (g && r) ? spec_step_kernel<true, true, DSPARK_F32>
           : g      ? spec_step_kernel<true, false, DSPARK_F32>
                    : spec_step_kernel<false, true, DSPARK_F32>;
  else
    kern = (g && r) ? spec_step_kernel<true, true, DSPARK_BF16>
           : g      ? spec_step_kernel<true, false, DSPARK_BF16>
                    : spec_step_kernel<false, true, DSPARK_BF16>;

  const int esz_t = (t_dtype == DSPARK_F32) ? 4 : 2;
  const int smem = max((qchunk + 4) * 4, vchunk * esz_t + 32);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  // as many clusters as are resident at once (at most one per item)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(qdense::kCl * 1024);
  cfg.blockDim = dim3(qdense::kThr);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  int ncl = 0;
  if (cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg) != cudaSuccess || ncl < 1) {
    cudaGetLastError();
    ncl = 1;
  }
  ncl = min(ncl, n_items);
  // a request's verification comes about two waves of rows after its rows
  wp.lag = (2 * ncl + depth - 1) / depth;
  e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t) * (size_t)(B + 1), stream);
  if (e != cudaSuccess) return e;
  kern<<<ncl * qdense::kCl, qdense::kThr, smem, stream>>>(qp, vp, wp);
  return cudaGetLastError();
}

// ---- the no-allocation variant's scratch
//
// A file-scope device array stands in for the caller's workspace: one copy
// per device (each device's module has its own), its address looked up once
// per device with cudaGetSymbolAddress and cached.  Every call on a device
// uses the same array, so calls that may overlap (other streams, other host
// threads) race on it.  The one-launch schedule zeroes the words it uses on
// the stream before its kernel, as with a caller's workspace.
constexpr int kMaxDevices = 64;
static __device__ __align__(256) uint32_t g_spec_workspace[DSPARK_SPEC_STATIC_MAX_B + 1];

// The calling thread's current device's copy of the array; nullptr if the
// device or the lookup fails.
uint32_t* static_spec_workspace() {
  static std::mutex mu;
  static uint32_t* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_spec_workspace) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = static_cast<uint32_t*>(p);
  }
  return addr[dev];
}

DSPARK_CHECK_COLLECTOR(spec)

}  // namespace dspark
