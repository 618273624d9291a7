// q_topk.cu -- dyadic24-standard-v1 q on a global top-k support, optionally
// with the draft draw ("PP1 q transport and scheduling design", Distribution
// contract and precision: for a sparse q the global support is chosen first,
// the weights are normalised on it, and the 2^24 tickets are allocated there;
// "Sparse support and vocabulary-sharded TP2 follow-up": an exact global
// top-k with deterministic ties).
//
// One CTA per draft row.  The support is the k largest y = RN(x * RN(1/T))
// with the lowest id first among equal y: an order on distinct (y, id) pairs.
//
// Main pass: a sample of 2048 elements spread over the row (plain loads)
// gives a filter value t, the j-th largest finite y of the sample, with j set
// so that about half the candidate buffer is expected to clear it.  The row
// is then streamed from HBM once: each warp owns one contiguous range and
// its own ring of TMA bulk copies (no block barrier while streaming), and an
// element whose y >= t joins the candidate buffer in shared memory.  The
// per-element work is a load, a NaN-propagating max, a multiply and a
// compare.  If at least k elements cleared t and the buffer did not
// overflow, the candidates hold the top k (every element outside is below
// the k-th largest), and a block-wide radix select on y, then on id among
// the elements tied at the cut, picks it exactly.
//
// Exact pass, only when the sample misled (the buffer overflowed, or fewer
// than k elements cleared t): the row is streamed again in ascending id
// order through a block-wide ring, and the buffer holds a superset of the
// top k of the prefix read so far.  An element enters it only if y > thr,
// thr the k-th largest y of the buffer after its last compaction; the filter
// is exact because the buffer then holds k elements with y >= thr, each with
// a lower id than any element still to come.  When the buffer fills, the
// same radix select cuts it back to the top k of the prefix.  Rows in
// ascending order of y make every element a candidate there: correct, slow.
//
// The allocation then runs on the at most k survivors (support_alloc.cuh):
// FP64 as the method states it, the nonzero counts in ascending id order,
// and the draft draw on them.
#define DSPARK_TU 4  // this file's number in the checked build's site codes
#include "support_alloc.cuh"

namespace dspark {
namespace {

constexpr int kKThr = 256;
constexpr int kKStages = 4;                        // ring slots
constexpr int kKStageElems = 2048;                 // elements per stage (8 KB f32, 4 KB bf16)
constexpr int kKStageBytes = kKStageElems * 4;     // ring slot size
constexpr int kKCap = 4096;                        // candidate buffer entries
constexpr int kKCompact = kKCap - kKStageElems;    // most entries before a stage
constexpr int kKSupCap = DSPARK_MAX_TOPK;          // largest k
constexpr int kKSample = 2048;                     // sampled elements (64 segments of 32)
constexpr int kKWarps = kKThr / 32;
// Per-warp rings of two 2 KB slots: measured faster than four 1 KB slots
// (fewer waits per element) and than one block-wide ring of 8 KB slots (whose
// refill waits for the slowest warp).
constexpr int kKWStage = 512;                      // elements per warp stage
constexpr int kKWSub = kKWStage / 256;             // 8 elements per lane each
constexpr int kKWStageBytes = kKWStage * 4;        // warp ring slot size
constexpr int kKWSlots = 2;                        // warp ring depth
static_assert(kKWStage % 256 == 0, "whole 256-element steps");
// the warps' rings share the ring with the exact streaming pass (not at once)
static_assert(kKWarps * kKWSlots * kKWStageBytes <= kKStages * kKStageBytes,
              "the warps' rings fit in the ring");
static_assert(kKSample == 8 * kKThr && kKSample <= kKCap, "8 sample keys per thread");
static_assert(kSupScratch <= kKStages * kKStageBytes && kKThr == kSupThr,
              "the allocation's scratch fits in the ring");

struct KParams {
  const void* x;
  int dtype;
  int64_t ld;
  int V;
  const float* temperature;
  int top_k;
  uint32_t* counts;  // [rows][top_k]
  int32_t* ids;      // [rows][top_k]
  int32_t* nnz;      // [rows]
  int32_t* status;   // [rows]
  int32_t* tokens;   // [rows] or null (no draw)
  uint64_t seed;
  const uint32_t* request_ids;
  int depth;
};

struct KShared {
  SupShared sup;                         // the allocation on the support
  uint64_t mbar[kKStages];               // the exact streaming pass
  uint64_t wbar[kKWarps * kKWSlots];     // the warps' rings
  uint64_t red64[32];
  uint32_t red32[32];
  float redf[32];
  uint32_t hist[256];
  uint32_t count;      // entries in the candidate buffer
  uint32_t n_fin;      // finite elements of the sample
  uint32_t n_tmp;
  uint32_t sel_digit, sel_above, sel_equal;
  float thr;           // an element is a candidate iff y > thr
  float invT;
  int bad_T;
  int timeout;
};

__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

struct OpMaxNaN {
  __device__ float operator()(float a, float b) const { return fmax_nan(a, b); }
};

// Inverse of float_key.
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Block-wide radix select: the r-th largest (1 <= r <= the number of taken
// entries) of val(i) over the entries i < n with take(i).  *above gets the
// number of taken entries with a larger value, *equal the number equal to
// it.  Called by every thread (n uniform); it starts with a __syncthreads()
// and its result is uniform.
// The bytes above the highest bit where the taken values' min and max differ
// are common to all of them, so the 8-bit digit passes start at the byte
// holding that bit.  In a pass, the lanes of a warp that fall in one bin add
// to it with a single atomic (candidate values share their high bits, so
// plain per-lane atomics would serialise on a few bins).  Once the selected
// bin holds at most 32 values, they are gathered and one warp finishes.
template <typename Val, typename Take>
__device__ uint32_t select_desc(int n, uint32_t r, Val val, Take take, KShared& sh,
                                uint32_t* above, uint32_t* equal) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  uint32_t vmin = 0xFFFFFFFFu, vmax = 0u, cnt = 0u;
  for (int i = (int)threadIdx.x; i < n; i += kKThr)
    if (take(i)) {
      const uint32_t v = val(i);
      vmin = min(vmin, v);
      vmax = max(vmax, v);
      ++cnt;
    }
  vmin = __reduce_min_sync(0xffffffffu, vmin);
  vmax = __reduce_max_sync(0xffffffffu, vmax);
  cnt = __reduce_add_sync(0xffffffffu, cnt);
  if (lane == 0) {
    sh.red32[warp] = vmin;
    sh.red32[kKWarps + warp] = vmax;
    sh.red32[2 * kKWarps + warp] = cnt;
  }
  __syncthreads();
  vmin = 0xFFFFFFFFu;
  vmax = 0u;
  cnt = 0u;
  for (int w = 0; w < kKWarps; ++w) {
    vmin = min(vmin, sh.red32[w]);
    vmax = max(vmax, sh.red32[kKWarps + w]);
    cnt += sh.red32[2 * kKWarps + w];
  }
  if (vmin >= vmax) {  // every taken value is the same
    *above = 0u;
    *equal = cnt;
    return vmin;
  }
  int shift = (31 - __clz(vmin ^ vmax)) & ~7;
  uint32_t mask = (shift == 24) ? 0u : ~((1u << (shift + 8)) - 1u);
  uint32_t prefix = vmin & mask, above_acc = 0, eq = cnt;
  for (; shift >= 0; shift -= 8) {
    __syncthreads();
    sh.hist[threadIdx.x] = 0u;  // kKThr == 256 bins
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kKThr) {
      const int i = i0 + (int)threadIdx.x;
      uint32_t bin = 0xFFFFFFFFu;
      if (i < n && take(i)) {
        const uint32_t v = val(i);
        if ((v & mask) == prefix) bin = (v >> shift) & 255u;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (bin != 0xFFFFFFFFu && lane == __ffs(peers) - 1)
        atomicAdd(&sh.hist[bin], (uint32_t)__popc(peers));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l scans bins 255 - 8l down to 248 - 8l
      uint32_t c[8], sacc = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sh.hist[255 - 8 * lane - j];
        sacc += c[j];
      }
      uint32_t incl = sacc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const uint32_t excl = incl - sacc;
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
    const uint32_t d = sh.sel_digit, ab = sh.sel_above;
    eq = sh.sel_equal;
    r -= ab;
    above_acc += ab;
    prefix |= d << shift;
    mask |= 255u << shift;
    if (shift > 0 && eq <= 32u) {
      // the selected bin's values, gathered; warp 0 takes the r-th largest
      if (threadIdx.x == 0) sh.n_tmp = 0u;
      __syncthreads();
      for (int i = (int)threadIdx.x; i < n; i += kKThr)
        if (take(i)) {
          const uint32_t v = val(i);
          if ((v & mask) == prefix) {
            const uint32_t j = atomicAdd(&sh.n_tmp, 1u);
            if (DSPARK_CHECK(j < 32u)) sh.hist[j] = v;
          }
        }
      __syncthreads();
      if (warp == 0) {
        const uint32_t v = (lane < (int)eq) ? sh.hist[lane] : 0u;
        uint32_t gt = 0, ge = 0;
        for (int m = 0; m < (int)eq; ++m) {
          const uint32_t u = __shfl_sync(0xffffffffu, v, m);
          gt += (u > v) ? 1u : 0u;
          ge += (u >= v) ? 1u : 0u;
        }
        const bool hit = lane < (int)eq && gt < r && r <= ge;
        const unsigned msk = __ballot_sync(0xffffffffu, hit);
        if (msk != 0u && lane == __ffs(msk) - 1) {
          sh.sel_digit = v;
          sh.sel_above = gt;
          sh.sel_equal = ge - gt;
        }
      }
      __syncthreads();
      *above = above_acc + sh.sel_above;
      *equal = sh.sel_equal;
      return sh.sel_digit;
    }
  }
  *above = above_acc;
  *equal = eq;
  return prefix;
}

// Cuts the buffer (n > k entries) back to the k that come first by (y desc,
// id asc), and sets the stream filter to their smallest y.
__device__ void keep_top_k(int n, int k, uint32_t* keys, int32_t* ids, uint32_t* tkeys,
                           int32_t* tids, KShared& sh) {
  uint32_t above, equal;
  const uint32_t T = select_desc(
      n, (uint32_t)k, [&](int i) { return keys[i]; }, [](int) { return true; }, sh, &above,
      &equal);
  // the (k - above) lowest ids among the entries whose key is T (all of them
  // when that is every such entry)
  int32_t id_max = 0x7FFFFFFF;
  if (equal != (uint32_t)k - above) {
    uint32_t above2, equal2;
    const uint32_t nid = select_desc(
        n, (uint32_t)k - above, [&](int i) { return ~(uint32_t)ids[i]; },
        [&](int i) { return keys[i] == T; }, sh, &above2, &equal2);
    id_max = (int32_t)~nid;
  }
  if (threadIdx.x == 0) sh.n_tmp = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kKThr) {
    const uint32_t kk = keys[i];
    const int32_t id = ids[i];
    if (kk > T || (kk == T && id <= id_max)) {
      const uint32_t j = atomicAdd(&sh.n_tmp, 1u);  // exactly k entries qualify
      if (j < (uint32_t)k) {
        tkeys[j] = kk;
        tids[j] = id;
      }
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < k; i += kKThr) {
    keys[i] = tkeys[i];
    ids[i] = tids[i];
  }
  if (threadIdx.x == 0) {
    sh.count = (uint32_t)k;
    sh.thr = key_float(T);
  }
  __syncthreads();
}

// Appends this thread's candidates (bit i of m: element i, value y[i], id
// idb + i, plus `jump` for i >= 4).  Candidates are rare after the first
// compaction, so each thread that has some takes its slots with one atomic.
__device__ __forceinline__ void append(uint32_t m, const float (&y)[8], int idb, int jump,
                                       uint32_t* keys, int32_t* ids, KShared& sh) {
  uint32_t j = atomicAdd(&sh.count, (uint32_t)__popc(m));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if ((m >> i) & 1u) {
      if (j < (uint32_t)kKCap) {
        // -0 and +0 are equal y: one key for both
        keys[j] = float_key(__fadd_rn(y[i], 0.0f));
        ids[j] = idb + i + (i >= 4 ? jump : 0);
      }
      ++j;
    }
  }
}

// Per-element step on up to 8 logits: the NaN-propagating max of x, the
// scaled value, the overflow check and the candidate mask.
__device__ __forceinline__ uint32_t scan8(const float (&x)[8], float (&y)[8], float invT,
                                         bool may_ovf, float thr, float& mx, uint32_t& ovf) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    mx = fmax_nan(mx, x[i]);
    y[i] = __fmul_rn(x[i], invT);
    // a finite logit whose scaled value overflows (to either infinity)
    if (may_ovf) ovf |= (fabsf(y[i]) == INFINITY && fabsf(x[i]) < INFINITY) ? 1u : 0u;
    m |= (y[i] > thr) ? (1u << i) : 0u;
  }
  return m;
}

// Up to 8 logits of a stage slot for thread t of `nt` (4-element f32 groups t
// and t + nt, or the 8-element bf16 group t); -inf past the `ne` elements
// the slot holds.  Element i has id idb + i (+ jump for i >= 4).
__device__ __forceinline__ void load8(const unsigned char* slot, int ne, int t, int nt, bool f32,
                                      int e0, float (&x)[8], int& idb, int& jump) {
  if (f32) {
    const float4* r4 = reinterpret_cast<const float4*>(slot);
    const int groups = ne >> 2;
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    const float4 a = (t < groups) ? r4[t] : ninf;
    const float4 b = (t + nt < groups) ? r4[t + nt] : ninf;
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    idb = e0 + 4 * t;
    jump = 4 * nt - 4;
  } else {
    const uint4* r4 = reinterpret_cast<const uint4*>(slot);
    const int groups = ne >> 3;
    const uint4 w = (t < groups) ? r4[t]
                                 : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(ww[i] << 16);
      x[2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
    }
    idb = e0 + 8 * t;
    jump = 0;
  }
}

// The exact streaming build of the candidate buffer: the whole row again,
// in ascending id order, with the filter raised at every compaction.  Used
// when the sampled threshold of the main path does not fit the row (the
// buffer overflowed, or fewer than k elements cleared it).  Recomputes mx and
// ovf; sets sh.timeout if a copy does not land.
__device__ __noinline__ void stream_adaptive(const KParams& p, const char* xrow, int h0, int nb,
                                             float invT, bool may_ovf, unsigned char* ring,
                                             uint32_t* keys, int32_t* ids, uint32_t* tkeys,
                                             int32_t* tids, KShared& sh, float& mx,
                                             uint32_t& ovf) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V, k = p.top_k;
  const bool f32 = (p.dtype == DSPARK_F32);
  const int esz = f32 ? 4 : 2;
  const int n_stages = (nb + kKStageElems - 1) / kKStageElems;
  // Compact once the buffer holds 512 entries (or k) beyond the k it keeps:
  // early cuts are cheap (the select runs over few entries) and raise the
  // filter soon; never above kKCompact, so that a stage always fits.
  const int trigger = min(kKCompact, max(2 * k, k + 512));
  __syncthreads();
  if (tid == 0) {
    sh.count = 0u;
    sh.thr = -INFINITY;
  }
  mx = -INFINITY;
  ovf = 0;
  auto issue = [&](int s) {
    const int e0 = h0 + s * kKStageElems;
    const int ne = min(kKStageElems, h0 + nb - e0);
    const uint32_t bytes = (uint32_t)ne * (uint32_t)esz;  // a multiple of 16
    uint64_t* bar = &sh.mbar[s % kKStages];
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar, bytes);
    tma_load_bulk(ring + (s % kKStages) * kKStageBytes, xrow + (int64_t)e0 * esz, bytes, bar);
  };
  if (tid == 0)
    for (int s = 0; s < min(kKStages, n_stages); ++s) issue(s);
  __syncthreads();
  // ---- head (lowest ids first), warp 0, one element per lane
  if (warp == 0 && h0 > 0) {
    float x[8], y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = -INFINITY;
    if (lane < h0) x[0] = load_logit(xrow, p.dtype, lane);
    const uint32_t m = scan8(x, y, invT, may_ovf, -INFINITY, mx, ovf);
    if (m) append(m, y, lane, 0, keys, ids, sh);
  }
  // ---- body stages
  for (int s = 0; s < n_stages; ++s) {
    const int slot = s % kKStages;
    if (tid == 0 && !mbar_wait_bounded(&sh.mbar[slot], (uint32_t)(s / kKStages) & 1u))
      sh.timeout = 1;
    __syncthreads();
    if (sh.timeout) {
      // let the copies still in flight land before the block exits
      if (tid == 0)
        for (int t = s; t < min(s + kKStages, n_stages); ++t)
          mbar_wait_bounded(&sh.mbar[t % kKStages], (uint32_t)(t / kKStages) & 1u);
      break;
    }
    const float thr = sh.thr;
    const int e0 = h0 + s * kKStageElems;
    float x[8], y[8];
    int idb, jump;
    load8(ring + slot * kKStageBytes, min(kKStageElems, h0 + nb - e0), tid, kKThr, f32, e0, x,
          idb, jump);
    const uint32_t m = scan8(x, y, invT, may_ovf, thr, mx, ovf);
    if (m) append(m, y, idb, jump, keys, ids, sh);
    __syncthreads();  // the slot is read and every append of this stage is done
    if (tid == 0 && s + kKStages < n_stages) issue(s + kKStages);
    const int cnt = (int)sh.count;
    if (cnt > trigger && cnt <= kKCap) keep_top_k(cnt, k, keys, ids, tkeys, tids, sh);
  }
  // ---- tail (highest ids last), warp 0
  const int t0 = h0 + nb, nt = V - t0;
  if (!sh.timeout && warp == 0 && nt > 0) {
    float x[8], y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = -INFINITY;
    if (lane < nt) x[0] = load_logit(xrow, p.dtype, t0 + lane);
    const uint32_t m = scan8(x, y, invT, may_ovf, sh.thr, mx, ovf);
    if (m) append(m, y, t0 + lane, 0, keys, ids, sh);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kKThr, 3) q_topk_kernel(KParams p) {
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ KShared sh;
  unsigned char* ring = dyn;
  uint32_t* keys = reinterpret_cast<uint32_t*>(dyn + kKStages * kKStageBytes);
  int32_t* ids = reinterpret_cast<int32_t*>(keys + kKCap);
  uint32_t* tkeys = reinterpret_cast<uint32_t*>(ids + kKCap);
  int32_t* tids = reinterpret_cast<int32_t*>(tkeys + kKSupCap);

  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V, k = p.top_k;
  const bool f32 = (p.dtype == DSPARK_F32);
  const int esz = f32 ? 4 : 2;
  const char* xrow = reinterpret_cast<const char*>(p.x) + (int64_t)row * p.ld * esz;

  // head [0, h0) and tail [h0 + nb, V) by plain loads, the 16-byte aligned
  // body [h0, h0 + nb) by bulk copies
  const uintptr_t rs = reinterpret_cast<uintptr_t>(xrow);
  const uintptr_t a16 = (rs + 15u) & ~(uintptr_t)15u;
  const uintptr_t b16 = (rs + (uintptr_t)V * esz) & ~(uintptr_t)15u;
  int h0 = V, nb = 0;
  if (a16 < b16) {
    h0 = (int)((a16 - rs) / esz);
    nb = (int)((b16 - a16) / esz);
  }
  // every body element is streamed by one warp, from one contiguous range of
  // whole warp stages per warp
  const int b_end = h0 + nb;
  const int per_warp = (nb + kKWarps * kKWStage - 1) / (kKWarps * kKWStage) * kKWStage;
  const int wlo = min(h0 + warp * per_warp, b_end);
  const int whi = min(wlo + per_warp, b_end);
  const int nst_w = (whi - wlo + kKWStage - 1) / kKWStage;
  unsigned char* wring = ring + warp * kKWSlots * kKWStageBytes;

  if (tid == 0) {
    const float T = p.temperature ? p.temperature[row] : 1.0f;
    const float iT = __frcp_rn(T);
    sh.invT = iT;
    sh.bad_T = (!(isfinite(T) && T > 0.0f) || !(isfinite(iT) && iT >= 0x1p-126f)) ? 1 : 0;
    sh.count = 0u;
    sh.n_fin = 0u;
    sh.thr = -INFINITY;
    sh.timeout = 0;
    for (int c = 0; c < kKStages; ++c) mbar_init(&sh.mbar[c], 1);
    for (int c = 0; c < kKWarps * kKWSlots; ++c) mbar_init(&sh.wbar[c], 1);
    mbar_init_fence();
  }
  __syncthreads();
  const bool bad_T = sh.bad_T != 0;
  const float invT = sh.invT;
  const bool may_ovf = invT > 1.0f;  // |x * invT| <= |x| otherwise

  auto issue_w = [&](int t) {
    const int e0 = wlo + t * kKWStage;
    const int ne = min(kKWStage, whi - e0);
    const uint32_t bytes = (uint32_t)ne * (uint32_t)esz;  // a multiple of 16
    uint64_t* bar = &sh.wbar[warp * kKWSlots + t % kKWSlots];
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar, bytes);
    tma_load_bulk(wring + (t % kKWSlots) * kKWStageBytes, xrow + (int64_t)e0 * esz, bytes, bar);
  };
  if (!bad_T && lane == 0)
    for (int t = 0; t < min(kKWSlots, nst_w); ++t) issue_w(t);

  float mx = -INFINITY;
  uint32_t ovf = 0;
  bool fallback = false;
  if (!bad_T) {
    // ---- the filter, from a sample of kKSample elements spread over the
    //      body (64 segments of 32; a prefix would be no sample of rows whose
    //      ids are ordered, as vocabularies often are): y >= the j-th largest
    //      finite y of the sample, j chosen so that about half the buffer is
    //      expected to clear it (j * V / sample elements), and at least
    //      k * sample / V + 8 so that fewer than k is unlikely.  Every finite
    //      element is a candidate when the body is no larger than the sample
    //      or the sample has no finite element.  The sample only sets the
    //      filter: its elements are streamed like the others.
    float thr0 = -INFINITY;  // candidates: y > thr0
    if (nb > kKSample) {
      const int seg = h0 + (((tid >> 2) * (nb / 64)) & ~7) + (tid & 3) * 8;
      (void)DSPARK_CHECK(seg >= h0 && seg + 8 <= h0 + nb);
      float sx[8], sy[8];
      if (f32) {
        const float4* g4 = reinterpret_cast<const float4*>(xrow + (int64_t)seg * 4);
        const float4 a = __ldg(g4), c = __ldg(g4 + 1);
        sx[0] = a.x; sx[1] = a.y; sx[2] = a.z; sx[3] = a.w;
        sx[4] = c.x; sx[5] = c.y; sx[6] = c.z; sx[7] = c.w;
      } else {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(xrow + (int64_t)seg * 2));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sx[2 * i] = __uint_as_float(ww[i] << 16);
          sx[2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
        }
      }
      uint32_t nf = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        sy[i] = __fmul_rn(sx[i], invT);
        const bool fin = sy[i] > -INFINITY && sy[i] < INFINITY;  // NaN: not finite
        keys[i * kKThr + tid] = fin ? float_key(__fadd_rn(sy[i], 0.0f)) : 0u;
        nf += fin ? 1u : 0u;
      }
      nf = warp_reduce(nf, OpAddU32());
      if (lane == 0) atomicAdd(&sh.n_fin, nf);
      __syncthreads();
      const uint32_t n_fin = sh.n_fin;
      if (n_fin > 0u) {
        const uint32_t j_need = (uint32_t)(((int64_t)k * kKSample + V - 1) / V) + 8u;
        const uint32_t j_half = (uint32_t)((int64_t)(kKCap / 2) * kKSample / V);
        const uint32_t j = min(n_fin, max(j_need, j_half));
        uint32_t above, equal;
        const uint32_t T = select_desc(
            kKSample, j, [&](int i) { return keys[i]; }, [&](int i) { return keys[i] != 0u; },
            sh, &above, &equal);
        // y >= t  <=>  y > the float just below t (t is never -0)
        const float t = key_float(T);
        thr0 = (t == 0.0f) ? -0x1p-149f
                           : __int_as_float(__float_as_int(t) + (t > 0.0f ? -1 : 1));
      }
      __syncthreads();  // the sample keys are read: the buffer is free
    }
    // ---- head, warp 0
    if (warp == 0 && h0 > 0) {
      float x[8], y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = -INFINITY;
      if (lane < h0) x[0] = load_logit(xrow, p.dtype, lane);
      const uint32_t m = scan8(x, y, invT, may_ovf, thr0, mx, ovf);
      if (m) append(m, y, lane, 0, keys, ids, sh);
    }
    // ---- the body, one range per warp, no block barrier: each warp waits
    //      for its own copies and refills its own ring
    for (int t = 0; t < nst_w; ++t) {
      const int slot = t % kKWSlots;
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded(&sh.wbar[warp * kKWSlots + slot], (uint32_t)(t / kKWSlots) & 1u)
                 ? 1
                 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();  // lane 0 saw the copy land: the slot is visible to the warp
      if (!ok) {
        if (lane == 0) {
          sh.timeout = 1;
          for (int u = t + 1; u < min(t + kKWSlots, nst_w); ++u)
            mbar_wait_bounded(&sh.wbar[warp * kKWSlots + u % kKWSlots],
                              (uint32_t)(u / kKWSlots) & 1u);
        }
        break;
      }
      const int e0 = wlo + t * kKWStage;
      const int ne = min(kKWStage, whi - e0);
      float x[kKWSub][8];
      int idb[kKWSub], jump;
#pragma unroll
      for (int u = 0; u < kKWSub; ++u)
        load8(wring + slot * kKWStageBytes + u * 256 * esz, ne - 256 * u, lane, 32, f32,
              e0 + 256 * u, x[u], idb[u], jump);
      __syncwarp();
      if (lane == 0 && t + kKWSlots < nst_w) issue_w(t + kKWSlots);
#pragma unroll
      for (int u = 0; u < kKWSub; ++u) {
        float y[8];
        const uint32_t m = scan8(x[u], y, invT, may_ovf, thr0, mx, ovf);
        if (m) append(m, y, idb[u], jump, keys, ids, sh);
      }
    }
    // ---- tail, the last warp
    const int t0 = b_end, nt = V - t0;
    if (warp == kKWarps - 1 && nt > 0) {
      float x[8], y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = -INFINITY;
      if (lane < nt) x[0] = load_logit(xrow, p.dtype, t0 + lane);
      const uint32_t m = scan8(x, y, invT, may_ovf, thr0, mx, ovf);
      if (m) append(m, y, t0 + lane, 0, keys, ids, sh);
    }
    __syncthreads();
    const int cnt = (int)sh.count;
    fallback = !sh.timeout && (cnt > kKCap || (thr0 != -INFINITY && cnt < k));
  }
  if (fallback) {
    // a NaN / +inf row needs no support: refuse it without the second pass
    const float m2 = block_reduce(mx, OpMaxNaN(), sh.redf);
    const uint32_t o2 = block_reduce(ovf, OpOrU32(), sh.red32);
    if (m2 < INFINITY && !o2)
      stream_adaptive(p, xrow, h0, nb, invT, may_ovf, ring, keys, ids, tkeys, tids, sh, mx, ovf);
  }
  __syncthreads();

  // ---- status
  mx = block_reduce(mx, OpMaxNaN(), sh.redf);
  ovf = block_reduce(ovf, OpOrU32(), sh.red32);
  int st = DSPARK_ST_OK;
  const int cnt = (int)sh.count;
  if (bad_T) st = DSPARK_ST_BAD_TEMPERATURE;
  else if (sh.timeout) st = DSPARK_ST_TIMEOUT;
  else if (!(mx < INFINITY) || ovf) st = DSPARK_ST_NONFINITE;  // NaN / +inf / overflow
  else if (cnt == 0) st = DSPARK_ST_ZERO_MASS;
  else if (cnt > kKCap) st = DSPARK_ST_INTERNAL;
  if (st == DSPARK_ST_OK && cnt > k) keep_top_k(cnt, k, keys, ids, tkeys, tids, sh);
  const int ns = min(cnt, k);

  // ---- allocation on the support (the ring is free now), outputs, draw
  uint32_t D = 0;
  if (p.tokens) {
    const int b = row / p.depth, j = row % p.depth;
    const uint32_t req = p.request_ids ? p.request_ids[b] : (uint32_t)b;
    D = draw_u32(p.seed, req, (uint32_t)j, DSPARK_PURPOSE_PROPOSAL) >> 8;
  }
  support_alloc_emit(st, ns, k, keys, ids, ring, sh.sup, p.counts + (int64_t)row * k,
                     p.ids + (int64_t)row * k, p.nnz + row, p.status + row,
                     p.tokens ? p.tokens + row : nullptr, D);
}

}  // namespace

int q_topk_smem_bytes() {
  return kKStages * kKStageBytes + 2 * kKCap * 4 + 2 * kKSupCap * 4;
}

cudaError_t launch_q_topk(const void* x, int dtype, int64_t ld, int n_rows, int V,
                          const float* temperature, int top_k, uint32_t* counts, int32_t* ids,
                          int32_t* nnz, int32_t* status, int32_t* tokens, uint64_t seed,
                          const uint32_t* request_ids, int depth, cudaStream_t stream) {
  KParams p;
  p.x = x;
  p.dtype = dtype;
  p.ld = ld;
  p.V = V;
  p.temperature = temperature;
  p.top_k = top_k;
  p.counts = counts;
  p.ids = ids;
  p.nnz = nnz;
  p.status = status;
  p.tokens = tokens;
  p.seed = seed;
  p.request_ids = request_ids;
  p.depth = depth > 0 ? depth : 1;
  const int smem = q_topk_smem_bytes();
  cudaError_t err =
      cudaFuncSetAttribute(q_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(q_topk_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (err != cudaSuccess) return err;
  q_topk_kernel<<<n_rows, kKThr, smem, stream>>>(p);
  return cudaGetLastError();
}

DSPARK_CHECK_COLLECTOR(q_topk)

}  // namespace dspark
