// debug.cu -- element-wise access to exp_ds / the integer weights and to
// Philox4x32-10 (include/dspark_debug.h).
#define DSPARK_TU 2  // this file's number in the checked build's site codes
#include "common.cuh"
#include "dspark_debug.h"

namespace {

__global__ void exp_weights_kernel(const float* d, int64_t n, float* e_out, uint64_t* E_out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float e = dspark::exp_ds(d[i]);
    if (e_out) e_out[i] = e;
    // the weight as the q kernels compute it: floor(exp_ds(d) * 2^40), exact;
    // the scalar form (top-k and sharded rows) and the packed pair form
    // (dense rows, here with a second lane) must agree, else ~0 is returned
    if (E_out) {
      const float w1 = dspark::weight40(d[i]);
      const float2 w2 = dspark::weight40x2(make_float2(d[i], d[n - 1 - i]));
      const bool same = __float_as_uint(w1) == __float_as_uint(w2.x) &&
                        __float_as_uint(dspark::weight40(d[n - 1 - i])) ==
                            __float_as_uint(w2.y);
      E_out[i] = same ? __float2ull_rz(w1) : ~0ull;
    }
  }
}

// one failing checked site (a comparison that is false for the one thread),
// guarding no access: the checked build's counters must record it
__global__ void check_selftest_kernel(int never) {
  if (!DSPARK_CHECK(threadIdx.x == (unsigned)never)) return;
}

__global__ void alloc_scale_kernel(const uint64_t* S, int64_t n, uint64_t* mk, int32_t* ek,
                                   float* khi, float* klo) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    dspark::AllocScale a = {0ull, 0, 0.0f, 0.0f};
    if (S[i] != 0ull) a = dspark::alloc_scale(S[i]);
    if (mk) mk[i] = a.mk;
    if (ek) ek[i] = a.ek;
    if (khi) khi[i] = a.khi;
    if (klo) klo[i] = a.klo;
  }
}

__global__ void philox_kernel(const uint4* ctr, uint64_t seed, int64_t n, uint4* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = dspark::philox4x32_10(ctr[i], (uint32_t)seed, (uint32_t)(seed >> 32));
}

__global__ void wait_kernel(int which, const uint32_t* count, uint32_t target, int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  bool ok;
  if (which == 2) {
    ok = dspark::wait_count(count, target);
  } else {
    dspark::mbar_init(&bar, 2);
    dspark::mbar_init_fence();
    dspark::mbar_arrive_expect_tx(&bar, 0);
    if (which == 1) dspark::mbar_arrive_expect_tx(&bar, 0);
    ok = dspark::mbar_wait_bounded(&bar, 0);
  }
  *status = ok ? DSPARK_ST_OK : DSPARK_ST_TIMEOUT;
}

int grid_for(int64_t n) {
  const int64_t g = (n + 255) / 256;
  return (int)(g < 152 * 16 ? (g < 1 ? 1 : g) : 152 * 16);
}

}  // namespace

extern "C" {

int dspark_debug_check_selftest(void* stream) {
  check_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(-1);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

int dspark_debug_exp_weights(const float* d, int64_t n, float* e_out, uint64_t* E_out,
                             void* stream) {
  if (n < 0) return DSPARK_ERR_SIZE;
  if (n == 0) return 0;
  if (!d) return DSPARK_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(d) & 3) || (reinterpret_cast<uintptr_t>(e_out) & 3) ||
      (reinterpret_cast<uintptr_t>(E_out) & 7))
    return DSPARK_ERR_ALIGN;
  exp_weights_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(d, n, e_out,
                                                                                   E_out);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

int dspark_debug_alloc_scale(const uint64_t* S, int64_t n, uint64_t* mk_out, int32_t* ek_out,
                             float* khi_out, float* klo_out, void* stream) {
  if (n < 0) return DSPARK_ERR_SIZE;
  if (n == 0) return 0;
  if (!S) return DSPARK_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(S) & 7) || (reinterpret_cast<uintptr_t>(mk_out) & 7) ||
      (reinterpret_cast<uintptr_t>(ek_out) & 3) || (reinterpret_cast<uintptr_t>(khi_out) & 3) ||
      (reinterpret_cast<uintptr_t>(klo_out) & 3))
    return DSPARK_ERR_ALIGN;
  alloc_scale_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      S, n, mk_out, ek_out, khi_out, klo_out);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

int dspark_debug_philox(const uint32_t* ctr, uint64_t seed, int64_t n, uint32_t* out,
                        void* stream) {
  if (n < 0) return DSPARK_ERR_SIZE;
  if (n == 0) return 0;
  if (!ctr || !out) return DSPARK_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(ctr) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
    return DSPARK_ERR_ALIGN;
  philox_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(ctr), seed, n, reinterpret_cast<uint4*>(out));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

int dspark_debug_wait(int32_t which, const uint32_t* count, uint32_t target, int32_t* status,
                      void* stream) {
  if (which < 0 || which > 2) return DSPARK_ERR_ARG;
  if (!status || (which == 2 && !count)) return DSPARK_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(status) & 3) || (reinterpret_cast<uintptr_t>(count) & 3))
    return DSPARK_ERR_ALIGN;
  wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(which, count, target, status);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? 0 : (int)e;
}

}  // extern "C"

namespace dspark {
DSPARK_CHECK_COLLECTOR(debug)
}  // namespace dspark
