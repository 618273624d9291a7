/*
 * dspark_debug.h -- element-wise entry points of libdspark.so that expose
 * three building blocks of the q path for exhaustive checks against a
 * reference: the deterministic exponential behind the draft weights, the
 * allocation scale k, and the Philox generator behind every draw.  Same conventions as dspark.h (device
 * pointers, caller-owned buffers, asynchronous on `stream`, 0 / <0 / >0
 * return codes).
 */
#ifndef DSPARK_DEBUG_H
#define DSPARK_DEBUG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * For each d[i] (fp32, d <= 0 is the meaningful range): e_out[i] =
 * exp_ds(d[i]) and E_out[i] = floor(exp_ds(d[i]) * 2^40), the integer weight
 * a draft token at distance d from the row maximum receives
 * ("PP1 q transport and scheduling design", Distribution contract and
 * precision: normalised draft weights; exp_ds is the library's fixed fp32
 * exponential, see dspark_q_build).  Either output may be NULL.  The weight
 * is computed both as the top-k and sharded kernels compute it (one element)
 * and as the dense kernel does (two elements at once, paired here with
 * d[n-1-i]); E_out[i] = ~0 (all ones) if the two ever disagree.
 */
int dspark_debug_exp_weights(const float* d, int64_t n, float* e_out, uint64_t* E_out,
                             void* stream);

/*
 * For each weight sum S[i] >= 1 (u64): the allocation scale
 * k = RN64(2^24 / RN64(S)) ("PP1 q transport and scheduling design",
 * Distribution contract and precision: FP64 floor pass), returned as
 * mk_out[i] * 2^ek_out[i] with mk in [2^52, 2^53), plus khi_out[i] = RN32(k)
 * and klo_out[i] = RN32(k - khi) -- the values the dense q kernel computes
 * with integer arithmetic.  S[i] == 0 gives all-zero outputs.  Any output
 * may be NULL.
 */
int dspark_debug_alloc_scale(const uint64_t* S, int64_t n, uint64_t* mk_out, int32_t* ek_out,
                             float* khi_out, float* klo_out, void* stream);

/*
 * Philox4x32-10 (Salmon et al., SC'11) of n counters: out[i][0..3] =
 * Philox(key = (seed low, seed high), counter = ctr[i][0..3]).
 */
int dspark_debug_philox(const uint32_t* ctr, uint64_t seed, int64_t n, uint32_t* out,
                        void* stream);

/*
 * The library's two bounded waits, run once on one thread so that their
 * time limit can be seen to work (2 s; the kernels that use them report
 * DSPARK_ST_TIMEOUT when it runs out, and the context stays usable):
 *   which = 0: an mbarrier expecting two arrivals gets one, then is waited on
 *              (the wait of every bulk copy into shared memory) -- it never
 *              completes;
 *   which = 1: the same mbarrier gets both arrivals, then is waited on;
 *   which = 2: waits until *count >= target with acquire loads (the fused
 *              step's wait for a request's q rows); count is device memory.
 * *status (device) = DSPARK_ST_OK if the wait ended by its condition,
 * DSPARK_ST_TIMEOUT if it gave up.  Other `which`: DSPARK_ERR_ARG.
 */
int dspark_debug_wait(int32_t which, const uint32_t* count, uint32_t target, int32_t* status,
                      void* stream);

/*
 * dspark_checked_status -- the record of the bounds-checked build.  The
 * library can be built with DSPARK_CHECKED (libdspark_checked.so): every
 * index into a fixed-capacity shared-memory array, every index that comes
 * from data (token ids, sparse ids, histogram bins, table slots, slots taken
 * with an atomic counter) and every output row / element offset is tested
 * against its bound before the access; a failing test skips the access (a
 * load yields a neutral value) and is counted -- no trap, no assert.  This
 * call (host; it synchronises the device) sets out[0] = the failures since
 * the last call, out[1] = the first failing site (source line + 10000 * the
 * source file's number), out[2] = 1 in the checked build and 0 in the normal
 * one (whose out[0], out[1] are 0), and clears the counters.  out is a host
 * array of 3 words.  Returns 0, DSPARK_ERR_NULL, or a CUDA error (> 0).
 */
int dspark_checked_status(uint32_t* out);

/*
 * One kernel of one thread whose single checked site fails (it guards no
 * access): in the checked build the next dspark_checked_status reports one
 * failure at that site; in the normal build it does nothing.
 */
int dspark_debug_check_selftest(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_DEBUG_H */
