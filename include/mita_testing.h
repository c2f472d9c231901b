/*
 * mita_testing.h -- test entry points of the MiTA library.
 *
 * The method description has no counterpart of these: they exist so that the
 * device-side error reporting of the operator's kernels can be exercised
 * without faulting, trapping or hanging a GPU.  Each runs one of the
 * library's own kernels (or its bounded wait) on inputs the caller makes,
 * and the kernel reports through the plan's status word exactly as in a
 * forward: mita_get_status() returns the code and clears it.
 */
#ifndef MITA_TESTING_H
#define MITA_TESTING_H

#include "mita.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Run the query-bucketing step of the forward on a caller-made route array
 * (device pointer, [B, H, N] int32, 16-byte aligned) with the plan's
 * workspace, on `stream`.  A route outside [0, m) is skipped before any
 * memory access and sets MITA_ERR_DEVICE in the status word (the check the
 * kernels make on routes they read back).  Returns MITA_ERR_INVALID_ARG for
 * a null or misaligned pointer, MITA_ERR_CUDA if the launch fails. */
int mita_testing_bucket(mita_plan_t plan, const int32_t* route, struct CUstream_st* stream);

/* Launch one block that waits, with the tensor-core kernels' bounded wait,
 * on a shared-memory barrier that nothing arrives on and no copy is in
 * flight for, giving up after `budget_cycles` SM cycles (1 to 2^31) and
 * setting MITA_ERR_TIMEOUT in the status word, then returning.  Returns
 * MITA_ERR_INVALID_ARG for a budget out of range. */
int mita_testing_wait(mita_plan_t plan, long long budget_cycles, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* MITA_TESTING_H */
