// api.cu -- the extern "C" entry points declared in include/dspark.h.  Host
// code only: argument checks (nothing is launched on a bad argument), then
// one kernel launch on the caller's stream.  No allocation, no host sync.
#include <nvtx3/nvToolsExt.h>
#include <cstdint>
#include <cuda_runtime.h>

#include "dspark.h"
#include "dspark_debug.h"

namespace dspark {
cudaError_t launch_q_topk(const void* x, int dtype, int64_t ld, int n_rows, int V,
                          const float* temperature, int top_k, uint32_t* counts, int32_t* ids,
                          int32_t* nnz, int32_t* status, int32_t* tokens, uint64_t seed,
                          const uint32_t* request_ids, int depth, cudaStream_t stream);
cudaError_t launch_q_dense(const void* x, int dtype, int64_t ld, int n_rows, int V,
                           const float* temperature, uint32_t* counts, int32_t* status,
                           int32_t* tokens, uint64_t seed, const uint32_t* request_ids, int depth,
                           cudaStream_t stream);
cudaError_t launch_draft_sample(const uint32_t* counts, const int32_t* ids, const int32_t* nnz,
                                int top_k, int B, int depth, int V, uint64_t seed,
                                const uint32_t* request_ids, int32_t* tokens, int32_t* status,
                                cudaStream_t stream);
cudaError_t launch_verify(int mode, const void* z, int dtype, int64_t ld, int B, int depth, int V,
                          const int32_t* drafts, const uint32_t* counts, const int32_t* ids,
                          const int32_t* nnz, int top_k, uint64_t seed,
                          const uint32_t* request_ids, int32_t* accept_len, int32_t* committed,
                          uint32_t* flags, int32_t* status, cudaStream_t stream);
cudaError_t launch_verify_modes(const void* z, int dtype, int64_t ld, int B, int depth, int V,
                                const int32_t* drafts, const uint32_t* counts, const int32_t* ids,
                                const int32_t* nnz, int top_k, uint64_t seed,
                                const uint32_t* request_ids, int32_t* g_acc, int32_t* g_com,
                                int32_t* g_st, int32_t* r_acc, int32_t* r_com, uint32_t* r_flags,
                                int32_t* r_st, cudaStream_t stream);
int spec_step_schedule(int B, int depth);
int64_t q_sharded_workspace_bytes(int n_rows);
cudaError_t launch_q_sharded(const void* x, int dtype, int64_t ld, int B, int depth, int V,
                             int n_sh, const float* temperature, int top_k, uint64_t seed,
                             const uint32_t* request_ids, uint32_t* counts, int32_t* ids,
                             int32_t* nnz, int32_t* tokens, int32_t* status, void* workspace,
                             cudaStream_t stream);
cudaError_t launch_q_chain(const void* x, int dtype, int64_t ld, int B, int depth, int V,
                           const float* temperature, const float* bias, int64_t bias_ld,
                           int n_bias, const int32_t* anchors, uint64_t seed,
                           const uint32_t* request_ids, uint32_t* counts, int32_t* tokens,
                           int32_t* status, float* margins, cudaStream_t stream);
cudaError_t launch_verify_match(const void* z, int dtype, int64_t ld, int B, int depth, int V,
                                const int32_t* drafts, uint64_t seed,
                                const uint32_t* request_ids, int32_t* accept_len,
                                int32_t* committed, uint32_t* flags, int32_t* status,
                                cudaStream_t stream);
cudaError_t launch_q_pack(const uint32_t* counts, const int32_t* ids, const int32_t* nnz,
                          int top_k, int n_rows, int V, float* q, uint64_t* checksum,
                          cudaStream_t stream);
cudaError_t launch_q_validate(const float* q, const int32_t* ids, const int32_t* nnz, int top_k,
                              int n_rows, int V, const int32_t* tokens, const uint64_t* expect,
                              uint32_t* counts, int32_t* status, cudaStream_t stream);
uint32_t* static_spec_workspace();
cudaError_t launch_spec_step(const void* xd, int d_dtype, int64_t ld_d, const void* xt,
                             int t_dtype, int64_t ld_t, int B, int depth, int V,
                             const float* temperature, uint64_t seed,
                             const uint32_t* request_ids, uint32_t* counts, int32_t* tokens,
                             int32_t* row_status, int32_t* g_acc, int32_t* g_com, int32_t* g_st,
                             int32_t* r_acc, int32_t* r_com, uint32_t* r_flags, int32_t* r_st,
                             uint32_t* workspace, int schedule, cudaStream_t stream);
cudaError_t launch_verify_stats(const uint32_t* flags, int B, uint32_t* stats,
                                cudaStream_t stream);
cudaError_t launch_target_probs(const void* z, int dtype, int64_t ld, int n_rows, int V,
                                float* p_out, int32_t* argmax, int32_t* status,
                                cudaStream_t stream);
#ifdef DSPARK_CHECKED
cudaError_t dspark_check_collect_chain(uint32_t* out);
cudaError_t dspark_check_collect_debug(uint32_t* out);
cudaError_t dspark_check_collect_q_dense(uint32_t* out);
cudaError_t dspark_check_collect_q_topk(uint32_t* out);
cudaError_t dspark_check_collect_q_wire(uint32_t* out);
cudaError_t dspark_check_collect_sample(uint32_t* out);
cudaError_t dspark_check_collect_spec(uint32_t* out);
cudaError_t dspark_check_collect_tp(uint32_t* out);
cudaError_t dspark_check_collect_verify(uint32_t* out);
#endif
}  // namespace dspark

namespace {

// One NVTX range per ABI call, named after the call (a no-op unless a tool
// such as Nsight Systems is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr int kMaxGridRows = (1 << 30) / 8;  // rows per launch (8-CTA clusters)

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int esize(int32_t dtype) { return dtype == DSPARK_F32 ? 4 : 2; }

int check_common(int32_t dtype, int32_t V, int64_t ld) {
  if (dtype != DSPARK_F32 && dtype != DSPARK_BF16) return DSPARK_ERR_DTYPE;
  if (V < 1 || V > DSPARK_MAX_V) return DSPARK_ERR_SIZE;
  if (ld < V) return DSPARK_ERR_SIZE;
  return 0;
}

int check_topk(int32_t top_k, int32_t V) {
  if (top_k < 0 || top_k > V || top_k > DSPARK_MAX_TOPK) return DSPARK_ERR_TOPK;
  return 0;
}

int launch_result(cudaError_t e) { return e == cudaSuccess ? 0 : (int)e; }

}  // namespace

extern "C" {

const char* dspark_version(void) { return "dspark-gb300 0.1 (" DSPARK_QSEM ", sm_103a)"; }

int dspark_checked_status(uint32_t* out) {
  if (!out) return DSPARK_ERR_NULL;
  out[0] = out[1] = 0u;
#ifdef DSPARK_CHECKED
  out[2] = 1u;
  cudaError_t e = cudaSuccess;
  cudaError_t (*collect[])(uint32_t*) = {
      dspark::dspark_check_collect_chain, dspark::dspark_check_collect_debug,
      dspark::dspark_check_collect_q_dense, dspark::dspark_check_collect_q_topk,
      dspark::dspark_check_collect_q_wire, dspark::dspark_check_collect_sample,
      dspark::dspark_check_collect_spec, dspark::dspark_check_collect_tp,
      dspark::dspark_check_collect_verify};
  for (auto fn : collect)
    if (e == cudaSuccess) e = fn(out);
  return e == cudaSuccess ? 0 : (int)e;
#else
  out[2] = 0u;
  return 0;
#endif
}

int dspark_q_build(const void* draft_logits, int32_t dtype, int64_t ld, int32_t n_rows, int32_t V,
                   const float* temperature, int32_t top_k, uint32_t* counts, int32_t* sparse_ids,
                   int32_t* nnz, int32_t* row_status, void* stream) {
  const NvtxRange nvtx_range("dspark_q_build");
  if (int e = check_common(dtype, V, ld)) return e;
  if (int e = check_topk(top_k, V)) return e;
  if (n_rows < 0 || n_rows > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (n_rows == 0) return 0;
  if (!draft_logits || !counts || !row_status) return DSPARK_ERR_NULL;
  if (top_k > 0 && (!sparse_ids || !nnz)) return DSPARK_ERR_NULL;
  if (!aligned(draft_logits, esize(dtype)) || !aligned(counts, 4) || !aligned(row_status, 4) ||
      (temperature && !aligned(temperature, 4)) || (sparse_ids && !aligned(sparse_ids, 4)) ||
      (nnz && !aligned(nnz, 4)))
    return DSPARK_ERR_ALIGN;
  if (top_k == 0)
    return launch_result(dspark::launch_q_dense(draft_logits, dtype, ld, n_rows, V, temperature,
                                                counts, row_status, nullptr, 0ull, nullptr, 1,
                                                static_cast<cudaStream_t>(stream)));
  return launch_result(dspark::launch_q_topk(draft_logits, dtype, ld, n_rows, V, temperature,
                                             top_k, counts, sparse_ids, nnz, row_status, nullptr,
                                             0ull, nullptr, 1, static_cast<cudaStream_t>(stream)));
}

int dspark_q_build_sample(const void* draft_logits, int32_t dtype, int64_t ld, int32_t B,
                          int32_t depth, int32_t V, const float* temperature, int32_t top_k,
                          uint64_t seed, const uint32_t* request_ids, uint32_t* counts,
                          int32_t* sparse_ids, int32_t* nnz, int32_t* draft_tokens,
                          int32_t* row_status, void* stream) {
  const NvtxRange nvtx_range("dspark_q_build_sample");
  if (int e = check_common(dtype, V, ld)) return e;
  if (int e = check_topk(top_k, V)) return e;
  if (depth < 1 || depth > DSPARK_MAX_DEPTH) return DSPARK_ERR_SIZE;
  if (B < 0 || (int64_t)B * depth > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (B == 0) return 0;
  if (!draft_logits || !counts || !row_status || !draft_tokens) return DSPARK_ERR_NULL;
  if (top_k > 0 && (!sparse_ids || !nnz)) return DSPARK_ERR_NULL;
  if (!aligned(draft_logits, esize(dtype)) || !aligned(counts, 4) || !aligned(row_status, 4) ||
      !aligned(draft_tokens, 4) || (temperature && !aligned(temperature, 4)) ||
      (sparse_ids && !aligned(sparse_ids, 4)) || (nnz && !aligned(nnz, 4)) ||
      (request_ids && !aligned(request_ids, 4)))
    return DSPARK_ERR_ALIGN;
  if (top_k == 0)
    return launch_result(dspark::launch_q_dense(draft_logits, dtype, ld, B * depth, V, temperature,
                                                counts, row_status, draft_tokens, seed,
                                                request_ids, depth,
                                                static_cast<cudaStream_t>(stream)));
  return launch_result(dspark::launch_q_topk(draft_logits, dtype, ld, B * depth, V, temperature,
                                             top_k, counts, sparse_ids, nnz, row_status,
                                             draft_tokens, seed, request_ids, depth,
                                             static_cast<cudaStream_t>(stream)));
}

int dspark_draft_sample(const uint32_t* counts, const int32_t* sparse_ids, const int32_t* nnz,
                        int32_t top_k, int32_t B, int32_t depth, int32_t V, uint64_t seed,
                        const uint32_t* request_ids, int32_t* draft_tokens, int32_t* row_status,
                        void* stream) {
  const NvtxRange nvtx_range("dspark_draft_sample");
  if (V < 1 || V > DSPARK_MAX_V) return DSPARK_ERR_SIZE;
  if (depth < 1 || depth > DSPARK_MAX_DEPTH) return DSPARK_ERR_SIZE;
  if (B < 0 || (int64_t)B * depth > (int64_t)(1 << 30)) return DSPARK_ERR_SIZE;
  if (int e = check_topk(top_k, V)) return e;
  if (B == 0) return 0;
  if (!counts || !draft_tokens || !row_status) return DSPARK_ERR_NULL;
  if (top_k > 0 && (!sparse_ids || !nnz)) return DSPARK_ERR_NULL;
  if (!aligned(counts, 4) || !aligned(draft_tokens, 4) || !aligned(row_status, 4) ||
      (request_ids && !aligned(request_ids, 4)) || (sparse_ids && !aligned(sparse_ids, 4)) ||
      (nnz && !aligned(nnz, 4)))
    return DSPARK_ERR_ALIGN;
  return launch_result(dspark::launch_draft_sample(counts, sparse_ids, nnz, top_k, B, depth, V,
                                                   seed, request_ids, draft_tokens, row_status,
                                                   static_cast<cudaStream_t>(stream)));
}

static int check_verify(const void* target_logits, int32_t dtype, int64_t ld, int32_t B,
                        int32_t depth, int32_t V, const int32_t* draft_tokens,
                        const int32_t* accept_len, const int32_t* committed,
                        const int32_t* req_status) {
  if (int e = check_common(dtype, V, ld)) return e;
  if (depth < 1 || depth > DSPARK_MAX_DEPTH) return DSPARK_ERR_SIZE;
  if (B < 0 || B > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (B == 0) return 1;  // nothing to do
  if (!target_logits || !draft_tokens || !accept_len || !committed || !req_status)
    return DSPARK_ERR_NULL;
  if (!aligned(target_logits, esize(dtype)) || !aligned(draft_tokens, 4) ||
      !aligned(accept_len, 4) || !aligned(committed, 4) || !aligned(req_status, 4))
    return DSPARK_ERR_ALIGN;
  return 0;
}

int dspark_verify_greedy(const void* target_logits, int32_t dtype, int64_t ld, int32_t B,
                         int32_t depth, int32_t V, const int32_t* draft_tokens,
                         int32_t* accept_len, int32_t* committed, int32_t* req_status,
                         void* stream) {
  const NvtxRange nvtx_range("dspark_verify_greedy");
  const int e = check_verify(target_logits, dtype, ld, B, depth, V, draft_tokens, accept_len,
                             committed, req_status);
  if (e != 0) return e > 0 ? 0 : e;
  return launch_result(dspark::launch_verify(0, target_logits, dtype, ld, B, depth, V,
                                             draft_tokens, nullptr, nullptr, nullptr, 0, 0ull,
                                             nullptr, accept_len, committed, nullptr, req_status,
                                             static_cast<cudaStream_t>(stream)));
}

int dspark_verify_ratio(const void* target_logits, int32_t dtype, int64_t ld, int32_t B,
                        int32_t depth, int32_t V, const int32_t* draft_tokens,
                        const uint32_t* counts, const int32_t* sparse_ids, const int32_t* nnz,
                        int32_t top_k, uint64_t seed, const uint32_t* request_ids,
                        int32_t* accept_len, int32_t* committed, uint32_t* flags,
                        int32_t* req_status, void* stream) {
  const NvtxRange nvtx_range("dspark_verify_ratio");
  const int e = check_verify(target_logits, dtype, ld, B, depth, V, draft_tokens, accept_len,
                             committed, req_status);
  if (e != 0) return e > 0 ? 0 : e;
  if (int e2 = check_topk(top_k, V)) return e2;
  if (!counts) return DSPARK_ERR_NULL;
  if (top_k > 0 && (!sparse_ids || !nnz)) return DSPARK_ERR_NULL;
  if (!aligned(counts, 4) || (flags && !aligned(flags, 4)) ||
      (request_ids && !aligned(request_ids, 4)) || (sparse_ids && !aligned(sparse_ids, 4)) ||
      (nnz && !aligned(nnz, 4)))
    return DSPARK_ERR_ALIGN;
  return launch_result(dspark::launch_verify(1, target_logits, dtype, ld, B, depth, V,
                                             draft_tokens, counts, sparse_ids, nnz, top_k, seed,
                                             request_ids, accept_len, committed, flags,
                                             req_status, static_cast<cudaStream_t>(stream)));
}

int dspark_verify_match(const void* target_logits, int32_t dtype, int64_t ld, int32_t B,
                        int32_t depth, int32_t V, const int32_t* draft_tokens, uint64_t seed,
                        const uint32_t* request_ids, int32_t* accept_len, int32_t* committed,
                        uint32_t* flags, int32_t* req_status, void* stream) {
  const NvtxRange nvtx_range("dspark_verify_match");
  const int e = check_verify(target_logits, dtype, ld, B, depth, V, draft_tokens, accept_len,
                             committed, req_status);
  if (e != 0) return e > 0 ? 0 : e;
  if ((flags && !aligned(flags, 4)) || (request_ids && !aligned(request_ids, 4)))
    return DSPARK_ERR_ALIGN;
  return launch_result(dspark::launch_verify_match(target_logits, dtype, ld, B, depth, V,
                                                   draft_tokens, seed, request_ids, accept_len,
                                                   committed, flags, req_status,
                                                   static_cast<cudaStream_t>(stream)));
}

int dspark_verify(const void* target_logits, int32_t dtype, int64_t ld, int32_t B, int32_t depth,
                  int32_t V, const int32_t* draft_tokens, const uint32_t* counts,
                  const int32_t* sparse_ids, const int32_t* nnz, int32_t top_k, uint64_t seed,
                  const uint32_t* request_ids, int32_t* greedy_accept_len,
                  int32_t* greedy_committed, int32_t* greedy_status, int32_t* ratio_accept_len,
                  int32_t* ratio_committed, uint32_t* ratio_flags, int32_t* ratio_status,
                  void* stream) {
  const NvtxRange nvtx_range("dspark_verify");
  const bool g = greedy_accept_len || greedy_committed || greedy_status;
  const bool r = ratio_accept_len || ratio_committed || ratio_status;
  if (!g && !r) return DSPARK_ERR_NULL;
  if (g && (!greedy_accept_len || !greedy_committed || !greedy_status)) return DSPARK_ERR_NULL;
  int e = g ? check_verify(target_logits, dtype, ld, B, depth, V, draft_tokens,
                           greedy_accept_len, greedy_committed, greedy_status)
            : check_verify(target_logits, dtype, ld, B, depth, V, draft_tokens, ratio_accept_len,
                           ratio_committed, ratio_status);
  if (e != 0) return e > 0 ? 0 : e;  // > 0: empty batch
  if (r) {
    const int e2 = check_verify(target_logits, dtype, ld, B, depth, V, draft_tokens,
                                ratio_accept_len, ratio_committed, ratio_status);
    if (e2 < 0) return e2;
    if (int e3 = check_topk(top_k, V)) return e3;
    if (!counts) return DSPARK_ERR_NULL;
    if (top_k > 0 && (!sparse_ids || !nnz)) return DSPARK_ERR_NULL;
    if (!aligned(counts, 4) || (ratio_flags && !aligned(ratio_flags, 4)) ||
        (request_ids && !aligned(request_ids, 4)) || (sparse_ids && !aligned(sparse_ids, 4)) ||
        (nnz && !aligned(nnz, 4)))
      return DSPARK_ERR_ALIGN;
  }
  return launch_result(dspark::launch_verify_modes(
      target_logits, dtype, ld, B, depth, V, draft_tokens, r ? counts : nullptr,
      r ? sparse_ids : nullptr, r ? nnz : nullptr, r ? top_k : 0, seed, request_ids,
      g ? greedy_accept_len : nullptr, greedy_committed, greedy_status,
      r ? ratio_accept_len : nullptr, ratio_committed, ratio_flags, ratio_status,
      static_cast<cudaStream_t>(stream)));
}

int dspark_spec_step_schedule(int32_t B, int32_t depth) {
  if (B < 0 || depth < 1 || depth > DSPARK_MAX_DEPTH) return DSPARK_ERR_SIZE;
  return dspark::spec_step_schedule(B, depth);
}

static int spec_step_impl(const void* draft_logits, int32_t draft_dtype, int64_t ld_draft,
                          const void* target_logits, int32_t target_dtype, int64_t ld_target,
                          int32_t B, int32_t depth, int32_t V, const float* temperature,
                          uint64_t seed, const uint32_t* request_ids, uint32_t* counts,
                          int32_t* draft_tokens, int32_t* row_status, int32_t* greedy_accept_len,
                          int32_t* greedy_committed, int32_t* greedy_status,
                          int32_t* ratio_accept_len, int32_t* ratio_committed,
                          uint32_t* ratio_flags, int32_t* ratio_status, uint32_t* workspace,
                          bool static_workspace, int32_t schedule, void* stream) {
  if (int e = check_common(draft_dtype, V, ld_draft)) return e;
  if (int e = check_common(target_dtype, V, ld_target)) return e;
  if (depth < 1 || depth > DSPARK_MAX_DEPTH) return DSPARK_ERR_SIZE;
  if (B < 0 || (int64_t)B * depth > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (schedule < DSPARK_SCHEDULE_AUTO || schedule > DSPARK_SCHEDULE_SEPARATE)
    return DSPARK_ERR_ARG;
  if (B == 0) return 0;
  const bool g = greedy_accept_len || greedy_committed || greedy_status;
  const bool r = ratio_accept_len || ratio_committed || ratio_status;
  if (!draft_logits || !target_logits || !counts || !draft_tokens || !row_status)
    return DSPARK_ERR_NULL;
  if (!workspace && !static_workspace) return DSPARK_ERR_NULL;
  if (!g && !r) return DSPARK_ERR_NULL;
  if (g && (!greedy_accept_len || !greedy_committed || !greedy_status)) return DSPARK_ERR_NULL;
  if (r && (!ratio_accept_len || !ratio_committed || !ratio_status)) return DSPARK_ERR_NULL;
  const void* four[] = {counts, draft_tokens, row_status, greedy_accept_len, greedy_committed,
                        greedy_status, ratio_accept_len, ratio_committed, ratio_flags,
                        ratio_status, temperature, request_ids, workspace};
  for (const void* q : four)
    if (q && !aligned(q, 4)) return DSPARK_ERR_ALIGN;
  if (!aligned(draft_logits, esize(draft_dtype)) || !aligned(target_logits, esize(target_dtype)))
    return DSPARK_ERR_ALIGN;
  if (static_workspace) {
    if (B > DSPARK_SPEC_STATIC_MAX_B) return DSPARK_ERR_SIZE;
    if ((workspace = dspark::static_spec_workspace()) == nullptr) return DSPARK_ERR_DEVICE;
  }
  return launch_result(dspark::launch_spec_step(
      draft_logits, draft_dtype, ld_draft, target_logits, target_dtype, ld_target, B, depth, V,
      temperature, seed, request_ids, counts, draft_tokens, row_status,
      g ? greedy_accept_len : nullptr, greedy_committed, greedy_status,
      r ? ratio_accept_len : nullptr, ratio_committed, ratio_flags, ratio_status, workspace,
      schedule, static_cast<cudaStream_t>(stream)));
}

int dspark_spec_step(const void* draft_logits, int32_t draft_dtype, int64_t ld_draft,
                     const void* target_logits, int32_t target_dtype, int64_t ld_target,
                     int32_t B, int32_t depth, int32_t V, const float* temperature, uint64_t seed,
                     const uint32_t* request_ids, uint32_t* counts, int32_t* draft_tokens,
                     int32_t* row_status, int32_t* greedy_accept_len, int32_t* greedy_committed,
                     int32_t* greedy_status, int32_t* ratio_accept_len, int32_t* ratio_committed,
                     uint32_t* ratio_flags, int32_t* ratio_status, uint32_t* workspace,
                     int32_t schedule, void* stream) {
  const NvtxRange nvtx_range("dspark_spec_step");
  return spec_step_impl(draft_logits, draft_dtype, ld_draft, target_logits, target_dtype,
                        ld_target, B, depth, V, temperature, seed, request_ids, counts,
                        draft_tokens, row_status, greedy_accept_len, greedy_committed,
                        greedy_status, ratio_accept_len, ratio_committed, ratio_flags,
                        ratio_status, workspace, false, schedule, stream);
}

int dspark_spec_step_noalloc(const void* draft_logits, int32_t draft_dtype, int64_t ld_draft,
                             const void* target_logits, int32_t target_dtype, int64_t ld_target,
                             int32_t B, int32_t depth, int32_t V, const float* temperature,
                             uint64_t seed, const uint32_t* request_ids, uint32_t* counts,
                             int32_t* draft_tokens, int32_t* row_status,
                             int32_t* greedy_accept_len, int32_t* greedy_committed,
                             int32_t* greedy_status, int32_t* ratio_accept_len,
                             int32_t* ratio_committed, uint32_t* ratio_flags,
                             int32_t* ratio_status, int32_t schedule, void* stream) {
  const NvtxRange nvtx_range("dspark_spec_step_noalloc");
  return spec_step_impl(draft_logits, draft_dtype, ld_draft, target_logits, target_dtype,
                        ld_target, B, depth, V, temperature, seed, request_ids, counts,
                        draft_tokens, row_status, greedy_accept_len, greedy_committed,
                        greedy_status, ratio_accept_len, ratio_committed, ratio_flags,
                        ratio_status, nullptr, true, schedule, stream);
}

namespace {

// The staging buffer of dspark_spec_step_host: 256-byte aligned segments.
struct HostStaging {
  int64_t counts, draft, target, temperature, request_ids, tokens, row_status, g_acc, g_com,
      g_st, r_acc, r_com, r_flags, r_st, workspace, total;
};

int64_t seg(int64_t* at, int64_t bytes) {
  const int64_t o = *at;
  *at += (bytes + 255) / 256 * 256;
  return o;
}

HostStaging host_staging(int32_t B, int32_t depth, int32_t V, int32_t dd, int32_t td) {
  HostStaging h;
  int64_t at = 0;
  const int64_t rows = (int64_t)B * depth, trows = (int64_t)B * (depth + 1);
  h.counts = seg(&at, rows * V * 4);
  h.draft = seg(&at, rows * V * esize(dd));
  h.target = seg(&at, trows * V * esize(td));
  h.temperature = seg(&at, rows * 4);
  h.request_ids = seg(&at, (int64_t)B * 4);
  h.tokens = seg(&at, rows * 4);
  h.row_status = seg(&at, rows * 4);
  h.g_acc = seg(&at, (int64_t)B * 4);
  h.g_com = seg(&at, trows * 4);
  h.g_st = seg(&at, (int64_t)B * 4);
  h.r_acc = seg(&at, (int64_t)B * 4);
  h.r_com = seg(&at, trows * 4);
  h.r_flags = seg(&at, (int64_t)B * 4);
  h.r_st = seg(&at, (int64_t)B * 4);
  h.workspace = seg(&at, ((int64_t)B + 1) * 4);
  h.total = at;
  return h;
}

}  // namespace

int64_t dspark_spec_step_host_staging_bytes(int32_t B, int32_t depth, int32_t V,
                                            int32_t draft_dtype, int32_t target_dtype) {
  if (B < 0 || depth < 1 || depth > DSPARK_MAX_DEPTH || V < 1 || V > DSPARK_MAX_V) return 0;
  if (check_common(draft_dtype, V, V) || check_common(target_dtype, V, V)) return 0;
  return host_staging(B, depth, V, draft_dtype, target_dtype).total;
}

int dspark_spec_step_host(const void* h_draft_logits, int32_t draft_dtype,
                          const void* h_target_logits, int32_t target_dtype, int32_t B,
                          int32_t depth, int32_t V, const float* h_temperature, uint64_t seed,
                          const uint32_t* h_request_ids, int32_t* h_draft_tokens,
                          int32_t* h_row_status, int32_t* h_greedy_accept_len,
                          int32_t* h_greedy_committed, int32_t* h_greedy_status,
                          int32_t* h_ratio_accept_len, int32_t* h_ratio_committed,
                          uint32_t* h_ratio_flags, int32_t* h_ratio_status, void* staging,
                          int32_t schedule, void* stream) {
  const NvtxRange nvtx_range("dspark_spec_step_host");
  if (int e = check_common(draft_dtype, V, V)) return e;
  if (int e = check_common(target_dtype, V, V)) return e;
  if (depth < 1 || depth > DSPARK_MAX_DEPTH) return DSPARK_ERR_SIZE;
  if (B < 0 || (int64_t)B * depth > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (schedule < DSPARK_SCHEDULE_AUTO || schedule > DSPARK_SCHEDULE_SEPARATE)
    return DSPARK_ERR_ARG;
  if (B == 0) return 0;
  const bool g = h_greedy_accept_len || h_greedy_committed || h_greedy_status;
  const bool r = h_ratio_accept_len || h_ratio_committed || h_ratio_status;
  if (!h_draft_logits || !h_target_logits || !h_draft_tokens || !h_row_status || !staging)
    return DSPARK_ERR_NULL;
  if (!g && !r) return DSPARK_ERR_NULL;
  if (g && (!h_greedy_accept_len || !h_greedy_committed || !h_greedy_status))
    return DSPARK_ERR_NULL;
  if (r && (!h_ratio_accept_len || !h_ratio_committed || !h_ratio_status)) return DSPARK_ERR_NULL;
  if (!aligned(staging, 256)) return DSPARK_ERR_ALIGN;
  const HostStaging h = host_staging(B, depth, V, draft_dtype, target_dtype);
  char* base = static_cast<char*>(staging);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t rows = (int64_t)B * depth, trows = (int64_t)B * (depth + 1);
  auto h2d = [&](int64_t off, const void* src, int64_t bytes) {
    return cudaMemcpyAsync(base + off, src, (size_t)bytes, cudaMemcpyHostToDevice, st);
  };
  auto d2h = [&](void* dst, int64_t off, int64_t bytes) {
    return cudaMemcpyAsync(dst, base + off, (size_t)bytes, cudaMemcpyDeviceToHost, st);
  };
  cudaError_t e = h2d(h.draft, h_draft_logits, rows * V * esize(draft_dtype));
  if (e == cudaSuccess) e = h2d(h.target, h_target_logits, trows * V * esize(target_dtype));
  if (e == cudaSuccess && h_temperature) e = h2d(h.temperature, h_temperature, rows * 4);
  if (e == cudaSuccess && h_request_ids) e = h2d(h.request_ids, h_request_ids, (int64_t)B * 4);
  if (e != cudaSuccess) return launch_result(e);
  auto dp = [&](int64_t off) { return reinterpret_cast<int32_t*>(base + off); };
  const int rc = spec_step_impl(
      base + h.draft, draft_dtype, V, base + h.target, target_dtype, V, B, depth, V,
      h_temperature ? reinterpret_cast<const float*>(base + h.temperature) : nullptr, seed,
      h_request_ids ? reinterpret_cast<const uint32_t*>(base + h.request_ids) : nullptr,
      reinterpret_cast<uint32_t*>(base + h.counts), dp(h.tokens), dp(h.row_status),
      g ? dp(h.g_acc) : nullptr, g ? dp(h.g_com) : nullptr, g ? dp(h.g_st) : nullptr,
      r ? dp(h.r_acc) : nullptr, r ? dp(h.r_com) : nullptr,
      (r && h_ratio_flags) ? reinterpret_cast<uint32_t*>(base + h.r_flags) : nullptr,
      r ? dp(h.r_st) : nullptr, reinterpret_cast<uint32_t*>(base + h.workspace), false, schedule,
      stream);
  if (rc != 0) return rc;
  e = d2h(h_draft_tokens, h.tokens, rows * 4);
  if (e == cudaSuccess) e = d2h(h_row_status, h.row_status, rows * 4);
  if (e == cudaSuccess && g) e = d2h(h_greedy_accept_len, h.g_acc, (int64_t)B * 4);
  if (e == cudaSuccess && g) e = d2h(h_greedy_committed, h.g_com, trows * 4);
  if (e == cudaSuccess && g) e = d2h(h_greedy_status, h.g_st, (int64_t)B * 4);
  if (e == cudaSuccess && r) e = d2h(h_ratio_accept_len, h.r_acc, (int64_t)B * 4);
  if (e == cudaSuccess && r) e = d2h(h_ratio_committed, h.r_com, trows * 4);
  if (e == cudaSuccess && r && h_ratio_flags) e = d2h(h_ratio_flags, h.r_flags, (int64_t)B * 4);
  if (e == cudaSuccess && r) e = d2h(h_ratio_status, h.r_st, (int64_t)B * 4);
  return launch_result(e);
}

int dspark_q_chain_sample(const void* draft_logits, int32_t dtype, int64_t ld, int32_t B,
                          int32_t depth, int32_t V, const float* temperature, const float* bias,
                          int64_t bias_ld, int32_t n_bias, const int32_t* anchors, uint64_t seed,
                          const uint32_t* request_ids, float* workspace, uint32_t* counts,
                          int32_t* draft_tokens, int32_t* row_status, float* margins,
                          void* stream) {
  const NvtxRange nvtx_range("dspark_q_chain_sample");
  if (int e = check_common(dtype, V, ld)) return e;
  if (depth < 1 || depth > DSPARK_MAX_DEPTH) return DSPARK_ERR_SIZE;
  if (B < 0 || (int64_t)B * depth > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (bias && (n_bias < 1 || bias_ld < V)) return DSPARK_ERR_SIZE;
  if (B == 0) return 0;
  // the workspace is no longer used (z is formed in shared memory); it may be NULL
  if (!draft_logits || !anchors || !counts || !draft_tokens || !row_status)
    return DSPARK_ERR_NULL;
  const void* four[] = {anchors, workspace, counts, draft_tokens, row_status, margins,
                        temperature, request_ids, bias};
  for (const void* q : four)
    if (q && !aligned(q, 4)) return DSPARK_ERR_ALIGN;
  if (!aligned(draft_logits, esize(dtype))) return DSPARK_ERR_ALIGN;
  return launch_result(dspark::launch_q_chain(
      draft_logits, dtype, ld, B, depth, V, temperature, bias, bias_ld, bias ? n_bias : 1,
      anchors, seed, request_ids, counts, draft_tokens, row_status, margins,
      static_cast<cudaStream_t>(stream)));
}

int64_t dspark_q_sharded_workspace_bytes(int32_t n_rows) {
  return n_rows < 0 ? 0 : dspark::q_sharded_workspace_bytes(n_rows);
}

int dspark_q_build_sample_sharded(const void* draft_logits, int32_t dtype, int64_t ld, int32_t B,
                                  int32_t depth, int32_t V, int32_t n_shards,
                                  const float* temperature, int32_t top_k, uint64_t seed,
                                  const uint32_t* request_ids, uint32_t* counts,
                                  int32_t* sparse_ids, int32_t* nnz, int32_t* draft_tokens,
                                  int32_t* row_status, void* workspace, void* stream) {
  const NvtxRange nvtx_range("dspark_q_build_sample_sharded");
  if (int e = check_common(dtype, V, ld)) return e;
  if (int e = check_topk(top_k, V)) return e;
  if (depth < 1 || depth > DSPARK_MAX_DEPTH) return DSPARK_ERR_SIZE;
  if (B < 0 || (int64_t)B * depth * 8 > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (n_shards < 1 || n_shards > 8) return DSPARK_ERR_ARG;
  if (B == 0) return 0;
  if (!draft_logits || !counts || !row_status || !workspace) return DSPARK_ERR_NULL;
  if (top_k > 0 && (!sparse_ids || !nnz)) return DSPARK_ERR_NULL;
  if (!aligned(draft_logits, esize(dtype)) || !aligned(counts, 4) || !aligned(row_status, 4) ||
      !aligned(workspace, 16) || (draft_tokens && !aligned(draft_tokens, 4)) ||
      (temperature && !aligned(temperature, 4)) || (request_ids && !aligned(request_ids, 4)) ||
      (sparse_ids && !aligned(sparse_ids, 4)) || (nnz && !aligned(nnz, 4)))
    return DSPARK_ERR_ALIGN;
  return launch_result(dspark::launch_q_sharded(
      draft_logits, dtype, ld, B, depth, V, n_shards, temperature, top_k, seed, request_ids,
      counts, sparse_ids, nnz, draft_tokens, row_status, workspace,
      static_cast<cudaStream_t>(stream)));
}

int dspark_q_pack(const uint32_t* counts, const int32_t* sparse_ids, const int32_t* nnz,
                  int32_t top_k, int32_t n_rows, int32_t V, float* q_out,
                  uint64_t* checksum_out, void* stream) {
  const NvtxRange nvtx_range("dspark_q_pack");
  if (V < 1 || V > DSPARK_MAX_V) return DSPARK_ERR_SIZE;
  if (int e = check_topk(top_k, V)) return e;
  if (n_rows < 0 || n_rows > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (n_rows == 0) return 0;
  if (!counts || !q_out || !checksum_out) return DSPARK_ERR_NULL;
  if (top_k > 0 && (!sparse_ids || !nnz)) return DSPARK_ERR_NULL;
  if (!aligned(counts, 4) || !aligned(q_out, 4) || !aligned(checksum_out, 8) ||
      (sparse_ids && !aligned(sparse_ids, 4)) || (nnz && !aligned(nnz, 4)))
    return DSPARK_ERR_ALIGN;
  return launch_result(dspark::launch_q_pack(counts, top_k > 0 ? sparse_ids : nullptr,
                                             top_k > 0 ? nnz : nullptr, top_k, n_rows, V, q_out,
                                             checksum_out, static_cast<cudaStream_t>(stream)));
}

int dspark_q_validate(const float* q, const int32_t* sparse_ids, const int32_t* nnz,
                      int32_t top_k, int32_t n_rows, int32_t V, const int32_t* tokens,
                      const uint64_t* expect, uint32_t* counts_out, int32_t* row_status,
                      void* stream) {
  const NvtxRange nvtx_range("dspark_q_validate");
  if (V < 1 || V > DSPARK_MAX_V) return DSPARK_ERR_SIZE;
  if (int e = check_topk(top_k, V)) return e;
  if (n_rows < 0 || n_rows > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (n_rows == 0) return 0;
  if (!q || !row_status) return DSPARK_ERR_NULL;
  if (top_k > 0 && (!sparse_ids || !nnz)) return DSPARK_ERR_NULL;
  if (!aligned(q, 4) || !aligned(row_status, 4) || (counts_out && !aligned(counts_out, 4)) ||
      (tokens && !aligned(tokens, 4)) || (expect && !aligned(expect, 8)) ||
      (sparse_ids && !aligned(sparse_ids, 4)) || (nnz && !aligned(nnz, 4)))
    return DSPARK_ERR_ALIGN;
  return launch_result(dspark::launch_q_validate(
      q, top_k > 0 ? sparse_ids : nullptr, top_k > 0 ? nnz : nullptr, top_k, n_rows, V, tokens,
      expect, counts_out, row_status, static_cast<cudaStream_t>(stream)));
}

int dspark_verify_stats(const uint32_t* flags, int32_t B, uint32_t* stats, void* stream) {
  const NvtxRange nvtx_range("dspark_verify_stats");
  if (B < 0 || B > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (!stats || (B > 0 && !flags)) return DSPARK_ERR_NULL;
  if (!aligned(stats, 4) || (flags && !aligned(flags, 4))) return DSPARK_ERR_ALIGN;
  return launch_result(
      dspark::launch_verify_stats(flags, B, stats, static_cast<cudaStream_t>(stream)));
}

int dspark_target_probs(const void* target_logits, int32_t dtype, int64_t ld, int32_t n_rows,
                        int32_t V, float* p_out, int32_t* argmax, int32_t* row_status,
                        void* stream) {
  const NvtxRange nvtx_range("dspark_target_probs");
  if (int e = check_common(dtype, V, ld)) return e;
  if (n_rows < 0 || n_rows > kMaxGridRows) return DSPARK_ERR_SIZE;
  if (n_rows == 0) return 0;
  if (!target_logits || !row_status) return DSPARK_ERR_NULL;
  if (!aligned(target_logits, esize(dtype)) || !aligned(row_status, 4) ||
      (p_out && !aligned(p_out, 4)) || (argmax && !aligned(argmax, 4)))
    return DSPARK_ERR_ALIGN;
  return launch_result(dspark::launch_target_probs(target_logits, dtype, ld, n_rows, V, p_out,
                                                   argmax, row_status,
                                                   static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
