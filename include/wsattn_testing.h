/*
 * wsattn_testing.h -- test hooks of libwsattn.so.  Not for production callers.
 *
 * The pages have no counterpart: this entry point exists so that the bounded
 * waits of the kernel (every mbarrier wait gives up after a time limit, raises
 * an abort flag for the block, drains in-flight copies and MMAs, frees Tensor
 * Memory and records a status bit) can be exercised without faulting a GPU.
 */
#ifndef WSATTN_TESTING_H_
#define WSATTN_TESTING_H_

#include "wsattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fmha_fwd_testing -- fmha_fwd with two extra knobs.
 *
 *   inject_fault  0: none (identical to fmha_fwd).
 *                 1: the softmax warps of query tile 0 skip their first
 *                    "P ready" arrival, so the MMA issuer's wait on it runs out;
 *                    the kernel then exits cleanly and the next
 *                    fmha_get_device_status() returns FMHA_ERR_TIMEOUT.
 *                    Outputs are undefined.
 *   wait_limit_s  per-wait time limit in seconds, in (0, 60]; fmha_fwd uses 1.
 *
 * Other arguments, ownership and errors as fmha_fwd; an out-of-range knob is
 * FMHA_ERR_INVALID_ARG.
 */
fmha_status fmha_fwd_testing(const void* q, const void* k, const void* v, void* o, float* lse,
                             int64_t B, int64_t H, int64_t S, int64_t D, int causal, float scale,
                             fmha_dtype dtype, void* stream, int inject_fault,
                             double wait_limit_s);

#ifdef __cplusplus
}
#endif

#endif /* WSATTN_TESTING_H_ */
