// sample.cu -- one draft token per row from its dyadic q ("PP1 q transport
// and scheduling design", Distribution contract and precision: a uniform
// 24-bit integer D and exact integer cumulative counts; the token is the first
// whose inclusive cumulative count exceeds D).
//
// One CTA per row.  Dense rows: 16 warps each sum a contiguous segment of the
// row (coalesced 32-bit loads), a block prefix over the segment totals finds
// the segment holding D, and that warp scans its segment in id order.
// Sparse rows (<= 1024 entries) are checked for canonical form and scanned
// by one warp.
#define DSPARK_TU 6  // this file's number in the checked build's site codes
#include "common.cuh"

namespace dspark {

constexpr int kSThreads = 512;
constexpr int kSWarps = kSThreads / 32;

struct SParams {
  const uint32_t* counts;
  const int32_t* ids;
  const int32_t* nnz;
  int top_k;
  int B;
  int depth;
  int V;
  uint64_t seed;
  const uint32_t* request_ids;
  int32_t* tokens;
  int32_t* status;
};

__global__ void __launch_bounds__(kSThreads) draft_sample_kernel(SParams p) {
  __shared__ uint64_t seg_sum[kSWarps];
  __shared__ int bad;
  __shared__ int result;
  const int r = blockIdx.x;
  const int b = r / p.depth, j = r % p.depth;
  const uint32_t req = p.request_ids ? p.request_ids[b] : (uint32_t)b;
  const uint32_t D = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_PROPOSAL) >> 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    bad = 0;
    result = -1;
  }
  __syncthreads();

  if (p.top_k == 0) {
    const uint32_t* row = p.counts + (int64_t)r * p.V;
    const int seg = (p.V + kSWarps - 1) / kSWarps;
    const int s_lo = warp * seg, s_hi = min(p.V, s_lo + seg);
    uint64_t sum = 0;
    for (int v = s_lo + lane; v < s_hi; v += 32) sum += __ldg(row + v);
    sum = warp_reduce(sum, OpAddU64());
    if (lane == 0) seg_sum[warp] = sum;
    __syncthreads();
    uint64_t before = 0, total = 0;
    for (int w = 0; w < kSWarps; ++w) {
      if (w < warp) before += seg_sum[w];
      total += seg_sum[w];
    }
    if (total != (uint64_t)kM) {
      if (threadIdx.x == 0) bad = 1;
    } else if ((uint64_t)D >= before && (uint64_t)D < before + seg_sum[warp]) {
      // this warp's segment holds D: scan it 32 ids at a time
      uint64_t base = before;
      for (int v0 = s_lo; v0 < s_hi; v0 += 32) {
        const int v = v0 + lane;
        const uint32_t c = (v < s_hi) ? __ldg(row + v) : 0u;
        uint32_t incl = c;
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const uint32_t tile = __shfl_sync(0xffffffffu, incl, 31);
        if ((uint64_t)D < base + tile) {
          const bool hit = (base + incl > (uint64_t)D) && (base + incl - c <= (uint64_t)D);
          const unsigned m = __ballot_sync(0xffffffffu, hit && c > 0u);
          if (lane == 0 && m) result = v0 + __ffs(m) - 1;
          break;
        }
        base += tile;
      }
    }
  } else {
    const int32_t* ids = p.ids + (int64_t)r * p.top_k;
    const uint32_t* cn = p.counts + (int64_t)r * p.top_k;
    const int nz = p.nnz[r];
    if (warp == 0) {
      int ok = (nz >= 1 && nz <= p.top_k) ? 1 : 0;
      uint64_t total = 0;
      if (ok)
        for (int i = lane; i < nz; i += 32) {
          const int id = ids[i];
          const uint32_t c = cn[i];
          if (id < 0 || id >= p.V || c == 0u || (i > 0 && ids[i - 1] >= id)) ok = 0;
          total += c;
        }
      total = warp_reduce(total, OpAddU64());
      ok = __all_sync(0xffffffffu, ok) && total == (uint64_t)kM;
      if (!ok) {
        if (lane == 0) bad = 1;
      } else {
        uint64_t base = 0;
        for (int i0 = 0; i0 < nz; i0 += 32) {
          const int i = i0 + lane;
          const uint32_t c = (i < nz) ? cn[i] : 0u;
          uint32_t incl = c;
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
          }
          const uint32_t tile = __shfl_sync(0xffffffffu, incl, 31);
          if ((uint64_t)D < base + tile) {
            const bool hit = (base + incl > (uint64_t)D) && (base + incl - c <= (uint64_t)D);
            const unsigned m = __ballot_sync(0xffffffffu, hit && c > 0u);
            if (lane == 0 && m && DSPARK_CHECK(i0 + __ffs(m) - 1 < nz))
              result = ids[i0 + __ffs(m) - 1];
            break;
          }
          base += tile;
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int st = bad ? DSPARK_ST_BAD_Q : (result >= 0 ? DSPARK_ST_OK : DSPARK_ST_INTERNAL);
    p.status[r] = st;
    p.tokens[r] = (st == DSPARK_ST_OK) ? result : -1;
  }
}

cudaError_t launch_draft_sample(const uint32_t* counts, const int32_t* ids, const int32_t* nnz,
                                int top_k, int B, int depth, int V, uint64_t seed,
                                const uint32_t* request_ids, int32_t* tokens, int32_t* status,
                                cudaStream_t stream) {
  SParams p;
  p.counts = counts;
  p.ids = ids;
  p.nnz = nnz;
  p.top_k = top_k;
  p.B = B;
  p.depth = depth;
  p.V = V;
  p.seed = seed;
  p.request_ids = request_ids;
  p.tokens = tokens;
  p.status = status;
  draft_sample_kernel<<<B * depth, kSThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

DSPARK_CHECK_COLLECTOR(sample)

}  // namespace dspark
