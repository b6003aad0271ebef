/*
 * gated_act_testing.h -- test-only entry points of the gated-activation
 * library (libgated_act.so).  Not part of the activation ABI in gated_act.h:
 * these exercise the library's failure handling on purpose and have no use
 * in a model.  Every wait they make run out is bounded; no call leaves a copy
 * in flight, and the CUDA context stays usable.
 */
#ifndef GATED_ACT_TESTING_H
#define GATED_ACT_TESTING_H

#include "gated_act.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Exercise the bounded-wait give-up path of the TMA-rows kernel (for tests of
 * the failure handling).  Runs gelu_and_mul_sparse on contiguous [T, 2d] bf16
 * rows with the TMA-rows geometry, except that every CTA withholds the bulk
 * copy of its first row's up half, so the wait for it runs out after wait_ns
 * (0 < wait_ns <= 1e9).  Each CTA then records bit 0 of the device status,
 * waits (bounded) for the copies it did issue and exits: no copy is left in
 * flight and the context stays usable.  Rows a CTA did not finish are left
 * unwritten.  Needs the 16-byte layout and d <= 32768
 * (GATED_ACT_ERR_VARIANT otherwise).
 */
int gated_act_selftest_wait_timeout(void *out, const void *in, int64_t T,
                                    int64_t d, unsigned long long wait_ns,
                                    cudaStream_t stream);

/*
 * gated_act_selftest_wait_timeout with dynamic rows: the same withheld copy
 * per CTA, with rows taken from `workspace` as in gelu_and_mul_sparse_ws
 * (a zeroed device workspace of gelu_and_mul_sparse_workspace_bytes()).
 * A CTA that gives up still draws row tickets until its first failing one,
 * so the launch hands out its usual number and the workspace is left zeroed
 * for the next call.
 */
int gated_act_selftest_wait_timeout_ws(void *out, const void *in, int64_t T,
                                       int64_t d, unsigned long long wait_ns,
                                       void *workspace, cudaStream_t stream);

/*
 * The same self-test for either bulk-copy geometry: variant is
 * GATED_ACT_VARIANT_TMA_ROWS or GATED_ACT_VARIANT_PIPE_ROWS (the library's
 * choice of CTAs per SM); workspace is null (round-robin rows) or a zeroed
 * workspace (dynamic rows).  In the pipe-rows geometry the consumer warps
 * give up on the withheld copy, vote to stop together and leave their slots
 * unreleased; the producer lane sees that, stops issuing, waits (bounded)
 * for the copies it issued that may still be landing, and, with dynamic
 * rows, draws tickets until its first failing one so the workspace is left
 * zeroed.  Errors as gated_act_selftest_wait_timeout_ws, plus
 * GATED_ACT_ERR_VARIANT for any other variant.
 */
int gated_act_selftest_wait_timeout_ex(void *out, const void *in, int64_t T,
                                       int64_t d, unsigned long long wait_ns,
                                       int variant, void *workspace,
                                       cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GATED_ACT_TESTING_H */
