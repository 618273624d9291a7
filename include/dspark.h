/*
 * dspark.h -- C ABI of the GB300 draft-sampling and verification library
 * (libdspark.so, CUDA kernels for sm_103a).
 *
 * What it computes, and where the method is defined:
 *   "PP1 q transport and scheduling design", section "Distribution contract
 *   and precision": the dyadic categorical q (integer counts c_v >= 0 summing
 *   exactly to M = 2^24, q(v) = c_v / M), built from temperature-scaled draft
 *   weights by FP64 floor plus largest remainders with ties to the lowest
 *   token id, optionally on a global top-k support; one token drawn per
 *   position from a uniform 24-bit integer as the first cumulative count
 *   strictly greater than the draw; ratio tests against the target p and a
 *   full-vocabulary residual.  Same page, "Versioned v2 message design": the
 *   validation list, separate RNG domains for proposal, acceptance and
 *   correction/bonus draws, and the commit (accepted count plus the
 *   correction or bonus id).  "DeepSeek-V4.1 DSpark", "State and sampling
 *   contracts": greedy verification accepts while the target argmax equals
 *   the proposal.  "Remote DSpark drafter -- wire and state contract",
 *   section 2: the anchor-as-first block (target row j scores the token
 *   drafted at position j; row `depth` gives the bonus) and lowest-index ties
 *   of the argmax.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless stated otherwise.  The caller owns
 *     every buffer; the library allocates nothing, keeps no state between
 *     calls and never synchronises the host.  `stream` is a cudaStream_t
 *     (NULL = the legacy default stream).  All work is enqueued on `stream`.
 *   - Return value (decided on the host before anything is launched):
 *       0  enqueued;
 *      <0  argument error (one of DSPARK_ERR_*), nothing launched;
 *      >0  the cudaError_t of a failed launch.
 *   - Per-row / per-request device statuses (DSPARK_ST_*) are valid once the
 *     stream has reached the call.  A refused draft row gets all-zero counts
 *     and token -1; a refused request gets accept_len 0 and committed all -1
 *     (the whole unverified proposal is discarded, as the PP1 page asks).
 *   - Logit rows may have any stride `ld` >= V (in elements) and any 4-byte
 *     (fp32) or 2-byte (bf16) alignment; only the V elements of each row are
 *     read.  bf16 logits are widened to fp32 exactly.
 *   - Every integer output is a pure function of the inputs, the seed, the
 *     request id and the row: it does not depend on the batch size, on the
 *     other rows or on the launch shape.
 *   - Random draws: Philox4x32-10 (Salmon et al., SC'11) with key =
 *     (seed low 32 bits, seed high 32 bits) and counter = (request id, row,
 *     purpose, 0); a draw is word 0 of the output.  24-bit draws are word 0
 *     shifted right by 8.  Request ids are request_ids[b] or, if that pointer
 *     is NULL, b.  Callers fold generation and round into seed or request id.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSPARK_QSEM "dyadic24-standard-v1"
#define DSPARK_M 16777216u           /* total mass of every q row, 2^24      */
#define DSPARK_MAX_V 131072          /* largest vocabulary (row length)      */
#define DSPARK_MAX_DEPTH 8           /* draft positions per request          */
#define DSPARK_MAX_TOPK 1024         /* largest sparse support               */

/* logit element types */
#define DSPARK_F32 0
#define DSPARK_BF16 1

/* Philox purposes (word 2 of the counter), fixed in the ABI */
#define DSPARK_PURPOSE_PROPOSAL 0u
#define DSPARK_PURPOSE_ACCEPT 1u
#define DSPARK_PURPOSE_RESIDUAL 2u
#define DSPARK_PURPOSE_BONUS 3u
#define DSPARK_PURPOSE_MATCH 4u       /* the stochastic verifier's draw of row j */

/* host-side argument errors */
#define DSPARK_ERR_NULL (-1)         /* a required pointer is NULL           */
#define DSPARK_ERR_SIZE (-2)         /* V, rows, B, depth, ld out of range   */
#define DSPARK_ERR_DTYPE (-3)        /* unknown dtype                        */
#define DSPARK_ERR_TOPK (-4)         /* top_k < 0, > V or > DSPARK_MAX_TOPK  */
#define DSPARK_ERR_ALIGN (-5)        /* pointer not aligned to its element   */
#define DSPARK_ERR_DEVICE (-6)       /* no usable sm_103 device current      */
#define DSPARK_ERR_ARG (-7)          /* an enumerated argument out of range  */

/* device statuses (per draft row, or per request) */
#define DSPARK_ST_OK 0
#define DSPARK_ST_NONFINITE 1        /* NaN or +inf logit (or y overflowed)  */
#define DSPARK_ST_ZERO_MASS 2        /* no finite logit                      */
#define DSPARK_ST_ALLOC_INCONSISTENT 3 /* remaining tickets out of range     */
#define DSPARK_ST_BAD_TEMPERATURE 4  /* T not finite, <= 0, 1/T not normal   */
#define DSPARK_ST_BAD_Q 5            /* q row mass != M or not canonical     */
#define DSPARK_ST_BAD_DRAFT 6        /* draft id out of range or q(x) == 0   */
#define DSPARK_ST_TIMEOUT 7          /* a bounded wait inside a kernel expired */
#define DSPARK_ST_INTERNAL 8         /* an internal capacity was exceeded    */
#define DSPARK_ST_BAD_CHECKSUM 9     /* a received q row's checksum differs  */

/* verification flags (per request, ratio verification) */
#define DSPARK_FLAG_AMBIG_ACCEPT 1u  /* |u*q - p| <= 1e-6 * q at a tested row */
#define DSPARK_FLAG_NEAR_BOUNDARY 2u /* final draw within 1e-6 (probability
                                        units) of a cumulative boundary     */
#define DSPARK_FLAG_DEGENERATE 4u    /* residual mass was zero: drew from p  */

/*
 * dspark_q_build -- dyadic24-standard-v1 q for n_rows draft rows
 * ("PP1 q transport and scheduling design", Distribution contract and
 * precision: proposal construction and sparse top-k).
 *
 * Per row r (logits at draft_logits + r*ld, V elements, dtype `dtype`):
 *   T = temperature[r] (1.0 if temperature == NULL, a device pointer);
 *   refuse (BAD_TEMPERATURE) unless T is finite and > 0 and RN32(1/T) is a
 *   finite normal float; refuse (NONFINITE) on NaN or +inf logits or a finite
 *   logit whose scaled value overflows; -inf logits are masked.
 *   y_v = RN32(x_v * RN32(1/T)); support = all finite y (top_k == 0) or the
 *   top_k largest y with ties to the lowest id (all finite ones if fewer);
 *   empty support -> ZERO_MASS.  m = max y; E_v = floor(exp_ds(RN32(y_v - m))
 *   * 2^40) with exp_ds the library's deterministic fp32 exponential
 *   (Cody-Waite reduction, degree-7 Taylor polynomial in fma Horner form);
 *   S = sum E_v in uint64; k = RN64(2^24 / RN64(S)); a_v = RN64(E_v * k);
 *   counts = floor(a_v) plus one for the M - sum floor(a_v) support tokens
 *   with the largest a_v - floor(a_v), ties to the lowest id.  Rows where the
 *   remaining tickets fall outside [0, #positive remainders] or the final sum
 *   is not M are refused (ALLOC_INCONSISTENT).
 *
 * Outputs:
 *   top_k == 0: counts[n_rows][V] (row stride V); sparse_ids and nnz unused
 *     (may be NULL).
 *   top_k  > 0: sparse_ids[n_rows][top_k] ascending token ids of the nonzero
 *     counts, counts[n_rows][top_k] the matching counts, nnz[n_rows] their
 *     number; unused slots hold id -1 and count 0.
 *   row_status[n_rows]: DSPARK_ST_*.
 * Limits: 1 <= V <= DSPARK_MAX_V, 1 <= n_rows, ld >= V, 0 <= top_k <=
 * min(V, DSPARK_MAX_TOPK).  Pointers: draft_logits aligned to its element,
 * counts / sparse_ids / nnz / row_status / temperature 4-byte aligned.
 */
int dspark_q_build(const void* draft_logits, int32_t dtype, int64_t ld, int32_t n_rows,
                   int32_t V, const float* temperature, int32_t top_k, uint32_t* counts,
                   int32_t* sparse_ids, int32_t* nnz, int32_t* row_status, void* stream);

/*
 * dspark_q_build_sample -- dspark_q_build of the B*depth draft rows followed
 * by the draft draw of dspark_draft_sample, in one launch: the draw runs on
 * the counts while they are still on chip, so the counts are not read back.
 * Outputs (counts, sparse_ids, nnz, draft_tokens[B*depth], row_status) are
 * exactly those of the two calls in sequence with the same arguments; a
 * refused row gets token -1.  Same limits as the two calls (1 <= depth <=
 * DSPARK_MAX_DEPTH).
 */
int dspark_q_build_sample(const void* draft_logits, int32_t dtype, int64_t ld, int32_t B,
                          int32_t depth, int32_t V, const float* temperature, int32_t top_k,
                          uint64_t seed, const uint32_t* request_ids, uint32_t* counts,
                          int32_t* sparse_ids, int32_t* nnz, int32_t* draft_tokens,
                          int32_t* row_status, void* stream);

/*
 * dspark_draft_sample -- one token per draft row from its q
 * ("PP1 q transport and scheduling design", Distribution contract and
 * precision: the draw is a uniform 24-bit integer compared with exact integer
 * cumulative counts; the token is the first whose cumulative count exceeds
 * it).
 *
 * Row r = b*depth + j (request b, position j): D = Philox(seed; request id,
 * j, PROPOSAL) word 0 >> 8; token = the first id, in ascending order, whose
 * inclusive cumulative count exceeds D.  Counts as written by
 * dspark_q_build (dense [B*depth][V] when top_k == 0, sparse
 * [B*depth][top_k] with sparse_ids and nnz otherwise).  A row whose counts do
 * not sum to M, or whose sparse ids are not strictly ascending in [0, V), is
 * refused (BAD_Q, token -1).
 * Outputs: draft_tokens[B*depth], row_status[B*depth].
 */
int dspark_draft_sample(const uint32_t* counts, const int32_t* sparse_ids, const int32_t* nnz,
                        int32_t top_k, int32_t B, int32_t depth, int32_t V, uint64_t seed,
                        const uint32_t* request_ids, int32_t* draft_tokens, int32_t* row_status,
                        void* stream);

/*
 * dspark_verify_greedy -- greedy verification ("DeepSeek-V4.1 DSpark",
 * State and sampling contracts: greedy verification matches the target
 * argmax; the argmax takes the lowest id among equal maxima).
 *
 * target_logits: B*(depth+1) rows, row b*(depth+1)+j at target_logits +
 * (b*(depth+1)+j)*ld.  draft_tokens[B][depth].  For each request the rows
 * are read in order, stopping at the first row whose argmax differs from the
 * draft: L = first such j (else depth); committed[b][0..L-1] = drafts,
 * committed[b][L] = argmax of row L (the correction, or the bonus when
 * L == depth), committed[b][L+1..depth] = -1; accept_len[b] = L.
 * Rows after the deciding row are not read and not validated.
 * Refusals: a draft id outside [0, V) (BAD_DRAFT); a NaN/+inf in a read row
 * (NONFINITE); a read row with no finite logit (ZERO_MASS).
 * Outputs: accept_len[B], committed[B][depth+1], req_status[B].
 */
int dspark_verify_greedy(const void* target_logits, int32_t dtype, int64_t ld, int32_t B,
                         int32_t depth, int32_t V, const int32_t* draft_tokens,
                         int32_t* accept_len, int32_t* committed, int32_t* req_status,
                         void* stream);

/*
 * dspark_verify_ratio -- standard ratio verification with the dyadic q
 * ("PP1 q transport and scheduling design": ratio tests and full-vocabulary
 * residual sampling with the target p and the defined q; separate
 * acceptance and correction/bonus RNG domains).
 *
 * p_j = softmax of target row j at T = 1 (-inf -> 0).  For j = 0, 1, ...:
 *   c = q_j(x_j) (dense row or sparse lookup); c == 0 -> BAD_DRAFT;
 *   U = Philox(seed; request id, j, ACCEPT) word 0 >> 8;
 *   accept  <=>  U * c < p_j(x_j) * 2^48   (i.e. u < p/q with u = U / 2^24).
 * At the first rejection L < depth the correction is drawn from
 * max(p_L - q_L, 0) over all V tokens with w = Philox(seed; request id, L,
 * RESIDUAL) word 0: t = w/2^32 * Z (Z the residual mass) and the token is the
 * first id whose cumulative residual exceeds t.  If every draft is accepted
 * the bonus is drawn the same way from p_depth with purpose BONUS at row
 * depth.  committed as in dspark_verify_greedy.  Rows after the deciding
 * row are not read.
 * Refusals: draft id outside [0, V) or c == 0 at a tested row (BAD_DRAFT);
 * NONFINITE / ZERO_MASS for a read target row; a sparse q row of a tested
 * position that is not canonical (ids strictly ascending in [0, V), counts
 * > 0, sum M) or a dense residual row whose counts do not sum to M (BAD_Q).
 * p is computed in fp32 on the GPU: a decision with |u*q - p| <= 1e-6*q and a
 * final draw within 1e-6 of a cumulative boundary may differ from exact
 * arithmetic; such requests carry DSPARK_FLAG_* in flags[b] (flags may be
 * NULL).
 * Outputs: accept_len[B], committed[B][depth+1], flags[B], req_status[B].
 */
int dspark_verify_ratio(const void* target_logits, int32_t dtype, int64_t ld, int32_t B,
                        int32_t depth, int32_t V, const int32_t* draft_tokens,
                        const uint32_t* counts, const int32_t* sparse_ids, const int32_t* nnz,
                        int32_t top_k, uint64_t seed, const uint32_t* request_ids,
                        int32_t* accept_len, int32_t* committed, uint32_t* flags,
                        int32_t* req_status, void* stream);

/*
 * dspark_verify_match -- stochastic verification ("DeepSeek-V4.1 DSpark",
 * State and sampling contracts: each row draws from the target's own
 * distribution with independent noise, a matching proposal is accepted and
 * the first mismatch stops verification; it keeps the target distribution
 * and is not the ratio test).
 *
 * p_j = softmax of target row j at T = 1.  For j = 0, 1, ...: the token t_j
 * is drawn from p_j with w = Philox(seed; request id, j, MATCH) word 0 (t =
 * w/2^32 * Z over p's weights, the first id whose cumulative weight exceeds
 * t -- the bonus draw of dspark_verify_ratio); if j < depth and t_j equals
 * draft j the proposal is accepted and row j+1 draws, else L = j and t_j is
 * committed (the correction, or the bonus when L == depth).  committed as in
 * dspark_verify_greedy.  Rows after the deciding row are not read.
 * Refusals: a draft id outside [0, V) (BAD_DRAFT); NONFINITE / ZERO_MASS for
 * a read row.  A draw within 1e-6 of a cumulative boundary sets
 * DSPARK_FLAG_NEAR_BOUNDARY in flags[b] (flags may be NULL).  No q is needed.
 * Outputs: accept_len[B], committed[B][depth+1], flags[B], req_status[B].
 */
int dspark_verify_match(const void* target_logits, int32_t dtype, int64_t ld, int32_t B,
                        int32_t depth, int32_t V, const int32_t* draft_tokens, uint64_t seed,
                        const uint32_t* request_ids, int32_t* accept_len, int32_t* committed,
                        uint32_t* flags, int32_t* req_status, void* stream);

/*
 * dspark_verify -- greedy and/or ratio verification in one pass over the
 * target rows: each output set is exactly that of dspark_verify_greedy /
 * dspark_verify_ratio with the same arguments (same pages and rules).  A
 * request's rows are read until both requested modes have decided.
 * Greedy outputs: greedy_accept_len[B], greedy_committed[B][depth+1],
 * greedy_status[B] -- all three or none; ratio outputs: ratio_accept_len[B],
 * ratio_committed[B][depth+1], ratio_status[B] (all three or none),
 * ratio_flags[B] (may be NULL), with counts / sparse_ids / nnz / top_k /
 * seed / request_ids as in dspark_verify_ratio (ignored without ratio
 * outputs).  At least one mode must be given (DSPARK_ERR_NULL otherwise).
 */
int dspark_verify(const void* target_logits, int32_t dtype, int64_t ld, int32_t B, int32_t depth,
                  int32_t V, const int32_t* draft_tokens, const uint32_t* counts,
                  const int32_t* sparse_ids, const int32_t* nnz, int32_t top_k, uint64_t seed,
                  const uint32_t* request_ids, int32_t* greedy_accept_len,
                  int32_t* greedy_committed, int32_t* greedy_status, int32_t* ratio_accept_len,
                  int32_t* ratio_committed, uint32_t* ratio_flags, int32_t* ratio_status,
                  void* stream);

/*
 * dspark_spec_step -- the whole speculative step in one call, dense q only:
 * dspark_q_build_sample (top_k = 0) of the B*depth draft rows, then
 * dspark_verify_greedy and/or dspark_verify_ratio of the B*(depth+1) target
 * rows with the drafts and q just built ("PP1 q transport and scheduling
 * design", Distribution contract and precision; "DeepSeek-V4.1 DSpark",
 * State and sampling contracts).  Every output is exactly that of the
 * separate calls in sequence on the same stream with the same arguments,
 * whichever schedule runs; both modes share one read of each target row.
 *
 * draft_logits / draft_dtype / ld_draft and target_logits / target_dtype /
 * ld_target as in those calls (either dtype for either side).  q outputs:
 * counts[B*depth][V], draft_tokens[B][depth], row_status[B*depth] (all
 * required).  Greedy outputs: greedy_accept_len[B], greedy_committed[B][depth+1],
 * greedy_status[B] -- all three or none; ratio outputs: ratio_accept_len[B],
 * ratio_committed[B][depth+1], ratio_status[B] (all three or none) and
 * ratio_flags[B] (may be NULL).  At least one mode must be given
 * (DSPARK_ERR_NULL otherwise).  Same limits as the separate calls.
 * workspace: B + 1 words of device memory owned by the caller (required);
 * the one-launch schedule zeroes it on `stream` and keeps the work counter
 * and the finished-row count of each request there, so calls that may
 * overlap need separate workspaces.
 * schedule: DSPARK_SCHEDULE_SEPARATE enqueues dspark_q_build_sample's kernel
 * and dspark_verify's;
 * DSPARK_SCHEDULE_ONE_LAUNCH runs one persistent kernel whose clusters take
 * q rows and verifications from a shared counter, a request's verification
 * waiting (at most 2 s, else DSPARK_ST_TIMEOUT for that request) until its
 * rows are finished; DSPARK_SCHEDULE_AUTO takes the one launch when B >= 2
 * and the B*(depth+1) work items fit in one wave of resident clusters, the
 * two kernels otherwise.  Any other value: DSPARK_ERR_ARG.
 */
#define DSPARK_SCHEDULE_AUTO 0
#define DSPARK_SCHEDULE_ONE_LAUNCH 1
#define DSPARK_SCHEDULE_SEPARATE 2
/* The schedule dspark_spec_step takes for DSPARK_SCHEDULE_AUTO with this
 * B and depth (host only, nothing launched); DSPARK_ERR_SIZE for B < 0 or
 * depth outside [1, DSPARK_MAX_DEPTH]. */
int dspark_spec_step_schedule(int32_t B, int32_t depth);

int dspark_spec_step(const void* draft_logits, int32_t draft_dtype, int64_t ld_draft,
                     const void* target_logits, int32_t target_dtype, int64_t ld_target,
                     int32_t B, int32_t depth, int32_t V, const float* temperature, uint64_t seed,
                     const uint32_t* request_ids, uint32_t* counts, int32_t* draft_tokens,
                     int32_t* row_status, int32_t* greedy_accept_len, int32_t* greedy_committed,
                     int32_t* greedy_status, int32_t* ratio_accept_len, int32_t* ratio_committed,
                     uint32_t* ratio_flags, int32_t* ratio_status, uint32_t* workspace,
                     int32_t schedule, void* stream);

/*
 * dspark_spec_step_noalloc -- dspark_spec_step without the caller's
 * workspace.  The pages have no counterpart: this is a deployment
 * convenience for callers that cannot hand over device memory (for instance
 * while building a CUDA graph around the step).
 *
 * Arguments, outputs and statuses are those of dspark_spec_step, which this
 * call makes with a scratch array of DSPARK_SPEC_STATIC_MAX_B + 1 words
 * that the library holds as a file-scope __device__ variable (one copy per
 * device); nothing is allocated, by this call or any library it calls.
 * - B > DSPARK_SPEC_STATIC_MAX_B: DSPARK_ERR_SIZE, nothing enqueued.
 * - The array's address is looked up with cudaGetSymbolAddress on the first
 *   call on each device and cached; make that first call (any B >= 1)
 *   before capturing a stream into a graph, so that the capture sees no
 *   lookup.  A failed lookup returns DSPARK_ERR_DEVICE.
 * - Every call on a device shares the one array: two calls that may run at
 *   the same time (different streams, host threads or graphs in flight)
 *   race on it and their outputs are undefined.  Order them on one stream,
 *   or use dspark_spec_step with separate workspaces.
 * - What must start at zero (the work counter and the per-request row
 *   counters) is zeroed on `stream` by the one-launch schedule before its
 *   kernel, so a call needs nothing from the one before it.
 */
#define DSPARK_SPEC_STATIC_MAX_B 65535
int dspark_spec_step_noalloc(const void* draft_logits, int32_t draft_dtype, int64_t ld_draft,
                             const void* target_logits, int32_t target_dtype, int64_t ld_target,
                             int32_t B, int32_t depth, int32_t V, const float* temperature,
                             uint64_t seed, const uint32_t* request_ids, uint32_t* counts,
                             int32_t* draft_tokens, int32_t* row_status,
                             int32_t* greedy_accept_len, int32_t* greedy_committed,
                             int32_t* greedy_status, int32_t* ratio_accept_len,
                             int32_t* ratio_committed, uint32_t* ratio_flags,
                             int32_t* ratio_status, int32_t schedule, void* stream);

/*
 * dspark_spec_step_host -- dspark_spec_step on host buffers: the inputs are
 * copied from host memory into the caller's device staging buffer, the step
 * runs there, and the drafts and verification outputs are copied back to
 * host memory.  Copies, kernels and copies are enqueued on `stream` in that
 * order, as cudaMemcpyAsync calls (page-locked host memory keeps them
 * asynchronous; pageable memory works but the host waits for each copy).
 * The pages have no counterpart: this is the path of a caller whose logits
 * are in host memory.
 *
 * Host inputs: h_draft_logits [B*depth][V] and h_target_logits
 * [B*(depth+1)][V], rows contiguous (ld = V), dtypes as dspark_spec_step;
 * h_temperature [B*depth] and h_request_ids [B] may be NULL (T = 1, ids
 * 0..B-1).  Host outputs as dspark_spec_step: h_draft_tokens and
 * h_row_status [B*depth] required, the greedy triple and the ratio triple
 * each all or none (at least one mode), h_ratio_flags [B] may be NULL.
 * staging: dspark_spec_step_host_staging_bytes(B, depth, V, draft_dtype,
 * target_dtype) bytes of device memory, 256-byte aligned, owned by the
 * caller; the step's q counts [B*depth][V] stay at its start (uint32).
 * Overlapping calls need separate staging buffers.  Host argument errors as
 * dspark_spec_step (DSPARK_ERR_ALIGN also for staging); a failed copy or
 * launch returns its CUDA error code (> 0).
 */
int64_t dspark_spec_step_host_staging_bytes(int32_t B, int32_t depth, int32_t V,
                                            int32_t draft_dtype, int32_t target_dtype);
int dspark_spec_step_host(const void* h_draft_logits, int32_t draft_dtype,
                          const void* h_target_logits, int32_t target_dtype, int32_t B,
                          int32_t depth, int32_t V, const float* h_temperature, uint64_t seed,
                          const uint32_t* h_request_ids, int32_t* h_draft_tokens,
                          int32_t* h_row_status, int32_t* h_greedy_accept_len,
                          int32_t* h_greedy_committed, int32_t* h_greedy_status,
                          int32_t* h_ratio_accept_len, int32_t* h_ratio_committed,
                          uint32_t* h_ratio_flags, int32_t* h_ratio_status, void* staging,
                          int32_t schedule, void* stream);

/*
 * dspark_verify_stats -- the verifier's optional statistics, counted from the
 * per-request flags[B] that dspark_verify_ratio, dspark_verify_match,
 * dspark_verify and the whole-step entries write (the numerical-tolerance
 * cases that "PP1 q transport and scheduling design", Distribution contract
 * and precision, asks to be qualified and counted):
 *   stats[0]  requests with DSPARK_FLAG_AMBIG_ACCEPT (an ambiguous decision),
 *   stats[1]  requests with DSPARK_FLAG_NEAR_BOUNDARY (a draw near a
 *             cumulative boundary),
 *   stats[2]  requests with DSPARK_FLAG_DEGENERATE (a zero residual mass).
 * flags: device uint32[B] (may be NULL when B == 0); stats: device
 * uint32[3], overwritten on the stream (zeros for B == 0).  One kernel of one
 * block.  Errors: DSPARK_ERR_SIZE for B < 0 or too large, DSPARK_ERR_NULL,
 * DSPARK_ERR_ALIGN (4-byte alignment); nothing is launched then.
 */
int dspark_verify_stats(const uint32_t* flags, int32_t B, uint32_t* stats, void* stream);

/*
 * dspark_target_probs -- the target distribution p of n_rows logit rows at
 * T = 1 ("PP1 q transport and scheduling design": the full target p after
 * the unchanged target processors, T = 1, top_p = 1), with the argmax
 * (lowest id among maxima).  p_out[n_rows][V] fp32 (may be NULL),
 * argmax[n_rows] (may be NULL), row_status[n_rows] (NONFINITE / ZERO_MASS
 * as above; a refused row gets p = 0 and argmax -1).
 */
int dspark_target_probs(const void* target_logits, int32_t dtype, int64_t ld, int32_t n_rows,
                        int32_t V, float* p_out, int32_t* argmax, int32_t* row_status,
                        void* stream);

/*
 * dspark_q_chain_sample -- the Markov-conditioned draft chain ("Remote DSpark
 * drafter -- wire and state contract", section 2: the sequential Markov step
 * adds the bias row of the previous sampled token, the anchor at step 0;
 * section 6.3: margin = top1 - top2 of (base + Markov) logits at each step).
 *
 * For each request b the rows j = 0 .. depth-1 run in order: z_v =
 * RN32(x_v + bias[prev mod n_bias][v]) (z = x when bias is NULL; prev =
 * anchors[b] at j = 0, else the token drawn at row j-1), then the dense q of
 * z with temperature[b*depth + j] and the draft draw of that row, exactly as
 * dspark_q_build_sample on z.  margins[b*depth + j] (may be NULL): z's
 * largest finite value minus its second largest (0 when they are equal,
 * FLT_MAX with fewer than two finite values, 0 on a refused row).  A row
 * after a refused row is refused with the same status (no token to condition
 * on); an anchor outside [0, V) refuses the request with BAD_DRAFT.
 *
 * draft_logits [B*depth][ld] (fp32 or bf16); bias [n_bias][bias_ld] fp32
 * (bias_ld >= V, n_bias >= 1) or NULL; anchors[B]; workspace: unused (z is
 * formed in shared memory), may be NULL, kept for the argument order of
 * earlier versions; counts [B*depth][V], draft_tokens[B][depth],
 * row_status[B*depth] as in dspark_q_build_sample.
 */
int dspark_q_chain_sample(const void* draft_logits, int32_t dtype, int64_t ld, int32_t B,
                          int32_t depth, int32_t V, const float* temperature, const float* bias,
                          int64_t bias_ld, int32_t n_bias, const int32_t* anchors, uint64_t seed,
                          const uint32_t* request_ids, float* workspace, uint32_t* counts,
                          int32_t* draft_tokens, int32_t* row_status, float* margins,
                          void* stream);

/*
 * dspark_q_build_sample_sharded -- dspark_q_build_sample with the vocabulary
 * split over n_shards emulated ranks on one GPU ("PP1 q transport and
 * scheduling design", Sparse support and vocabulary-sharded TP2 follow-up:
 * all-reduce of the max and the shifted sums, remaining tickets coordinated
 * globally, a global top-k merge of the ranks' local top-k, the leader's one
 * draw choosing the shard by its count mass and then the token inside).
 * Shard s holds ids [s*Vs, min(V, (s+1)*Vs)), Vs = ceil(V / n_shards); each
 * per-rank kernel runs one CTA per (row, shard) and ranks exchange only
 * partials, through the workspace.
 *
 * Arguments and outputs as dspark_q_build_sample (draft_tokens may be NULL:
 * q only); the counts, sparse ids, nnz, tokens and statuses equal that call's
 * bit for bit.  Dense rows: the ranks exchange, for the fraction bin holding
 * the grant threshold, a table of its distinct exact fractions with their
 * counts; a row whose bin holds more than 1024 distinct fractions over all
 * shards is refused with DSPARK_ST_INTERNAL (exact ties of any multiplicity
 * are fine).  Top-k rows: each rank sends at most top_k candidates.
 * n_shards in [1, 8] (DSPARK_ERR_ARG otherwise).
 * workspace: dspark_q_sharded_workspace_bytes(B*depth) bytes of device
 * memory, 16-byte aligned, owned by the caller.
 */
int64_t dspark_q_sharded_workspace_bytes(int32_t n_rows);
int dspark_q_build_sample_sharded(const void* draft_logits, int32_t dtype, int64_t ld, int32_t B,
                                  int32_t depth, int32_t V, int32_t n_shards,
                                  const float* temperature, int32_t top_k, uint64_t seed,
                                  const uint32_t* request_ids, uint32_t* counts,
                                  int32_t* sparse_ids, int32_t* nnz, int32_t* draft_tokens,
                                  int32_t* row_status, void* workspace, void* stream);

/*
 * dspark_q_pack -- the wire form of q rows ("PP1 q transport and scheduling
 * design", Distribution contract and precision: q is sent as little-endian
 * FP32 q(v) = c_v / M, every such value exact; Versioned v2 message design:
 * the per-position reply carries the q values, the sparse ids and a
 * checksum).
 *
 * Dense (top_k == 0): counts[n_rows][V] -> q_out[n_rows][V].  Sparse
 * (top_k > 0): counts[n_rows][top_k] with sparse_ids / nnz as built by
 * dspark_q_build -> q_out[n_rows][top_k] (q = 0 past nnz; the ids are sent
 * as they are).  checksum_out[n_rows]: Fletcher-64 of the row's payload
 * words -- a dense row's V FP32 bit patterns in id order, a sparse row's nnz
 * int32 ids followed by their nnz FP32 bit patterns -- with A = sum w_i and
 * B = sum (n - i) w_i modulo 2^32 - 1, checksum = B << 32 | A.  (The pages
 * ask for a checksum but name none: this is one with published test
 * vectors.)
 */
int dspark_q_pack(const uint32_t* counts, const int32_t* sparse_ids, const int32_t* nnz,
                  int32_t top_k, int32_t n_rows, int32_t V, float* q_out,
                  uint64_t* checksum_out, void* stream);

/*
 * dspark_q_validate -- validation of received q rows before they are used
 * (same sections: the receiver recovers c = q * M, requires an integer,
 * checks the mass in uint64, and refuses the listed malformations).
 *
 * q[n_rows][width] FP32 (width = V dense, top_k sparse), with
 * sparse_ids[n_rows][top_k] and nnz[n_rows] for sparse rows.  tokens[n_rows]
 * (may be NULL): the token proposed from each row, which must have q > 0.
 * expect[n_rows] (may be NULL): the checksums the rows must have.
 * counts_out[n_rows][width] (may be NULL): the recovered counts, all zero
 * for a refused row.  row_status[n_rows], first failing check in this order:
 *   BAD_Q        sparse nnz outside [1, top_k] (the payload's size);
 *   BAD_CHECKSUM the row's checksum differs from expect;
 *   BAD_Q        a value not finite, negative, above 1 or not a multiple of
 *                2^-24; the counts not summing to M; sparse ids not strictly
 *                ascending in [0, V) (duplicates, padding) or a listed zero;
 *   BAD_DRAFT    the proposed token outside [0, V) or with q = 0.
 */
int dspark_q_validate(const float* q, const int32_t* sparse_ids, const int32_t* nnz,
                      int32_t top_k, int32_t n_rows, int32_t V, const int32_t* tokens,
                      const uint64_t* expect, uint32_t* counts_out, int32_t* row_status,
                      void* stream);

/* Library build identifier (static string, host). */
const char* dspark_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
