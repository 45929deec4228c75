/*
 * wsattn_testing.h -- test hooks of libwsattn.so.  Not for production callers.
 *
 * The pages have no counterpart: these entry points exist so that three
 * properties of the kernel can be tested.  (1) Its bounded waits: every
 * mbarrier wait gives up after a time limit, raises an abort flag for the
 * block, drains in-flight copies and MMAs, frees Tensor Memory and records a
 * status bit -- exercised here without faulting a GPU.  (2) The independence
 * of the result from the online softmax's lazy-rescale threshold.  (3) The
 * key-split units of a short last wave, in every mix with whole units.
 */
#ifndef WSATTN_TESTING_H_
#define WSATTN_TESTING_H_

#include "wsattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fmha_fwd_testing -- fmha_fwd with three extra knobs.
 *
 *   inject_fault  0: none (identical to fmha_fwd).
 *                 1: the softmax warps of query tile 0 skip their first
 *                    "P ready" arrival, so the MMA issuer's wait on it runs out;
 *                    the kernel then exits cleanly and the next
 *                    fmha_get_device_status() returns FMHA_ERR_TIMEOUT.
 *                    Outputs are undefined.
 *   wait_limit_s  per-wait time limit in seconds, in (0, 60]; fmha_fwd uses 1.
 *   tau           lazy-rescale threshold of the online softmax in log2 units,
 *                 in [0, 15] ([0, 8] for FMHA_E4M3); fmha_fwd uses 15 (8 for
 *                 FMHA_E4M3).  The running maximum is raised (and O rescaled)
 *                 only when a block's maximum exceeds it by more than tau, so
 *                 P <= 2^tau (15 keeps P inside the f16 range; E4M3 P is
 *                 stored as 2^(8-tau) P <= 256, inside its range of 448).  The
 *                 result does not depend on tau; 0 gives the classic online
 *                 softmax that rescales whenever the maximum grows.
 *
 * Other arguments, ownership and errors as fmha_fwd; an out-of-range knob is
 * FMHA_ERR_INVALID_ARG.
 */
fmha_status fmha_fwd_testing(const void* q, const void* k, const void* v, void* o, float* lse,
                             int64_t B, int64_t H, int64_t S, int64_t D, int causal, float scale,
                             fmha_dtype dtype, void* stream, int inject_fault,
                             double wait_limit_s, float tau);

/*
 * fmha_fwd_split_testing -- fmha_fwd with the number of key-split units given.
 *
 * Full attention runs on persistent blocks that take (head, 256-row query
 * block) units in index order.  fmha_fwd splits the units of a short last
 * wave: the last split_units units each run as two 128-row halves whose two
 * query tiles take half of the key blocks each, merged in the block
 * (O = sum of each half's O weighted by its share of the softmax sum).  This
 * hook fixes that number, so that tests can compare every mix with the
 * oracle.
 *
 *   split_units  -1: as fmha_fwd.  0: none.  1 .. units: the last split_units
 *                units (units = B * H * ceil(S / 256)).  A positive value
 *                needs causal = 0, D = 128 and an even ceil(S / 128), else
 *                FMHA_ERR_UNSUPPORTED; above units is FMHA_ERR_INVALID_ARG.
 *
 * Other arguments, ownership and errors as fmha_fwd.
 */
fmha_status fmha_fwd_split_testing(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                                   int causal, float scale, fmha_dtype dtype, void* stream,
                                   int64_t split_units);

/*
 * fmha_fwd_split_policy -- how many of the last units fmha_fwd key-splits for
 * this shape on a GPU with n_sm multiprocessors (host arithmetic only; no
 * CUDA call).  Returns 0 where no unit is split (causal, D != 128, an odd
 * ceil(S / 128), or a last wave of more than n_sm / 2 units), and -1 for
 * sizes fmha_fwd would reject or n_sm < 1.
 */
int64_t fmha_fwd_split_policy(int64_t B, int64_t H, int64_t S, int64_t D, int causal, int n_sm);

#ifdef __cplusplus
}
#endif

#endif /* WSATTN_TESTING_H_ */
