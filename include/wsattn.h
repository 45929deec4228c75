/*
 * wsattn.h -- C ABI of the GB300 (sm_103a) fused attention forward library
 * (libwsattn.so).
 *
 * The operation.  Attention as the pages describe it is a loop over key/value
 * blocks with three stages per block: the first tensor-core stage S = Q K^T
 * ("T"), a CUDA-core softmax stage ("C") and the second tensor-core stage
 * O += P V ("U") -- "Tawa: Automatic Warp Specialization for Modern GPUs with
 * Asynchronous References", Section III-D, Algorithm 1 (coarse-grained
 * CUDA/Tensor Core pipeline; attention is its worked example), and the
 * forward-attention experiments of "Optimal Software Pipelining and Warp
 * Specialization for Tensor Core GPUs", Section 6.2 (Figs. 7 and 8: fp16,
 * batch 4, 32 heads, head dim 128, sequence length up to 16384).  The pages
 * name the stages but do not write the formula; this library computes the
 * textbook definition, for every batch b, head h and query row i:
 *
 *     s_ij   = scale * sum_d Q[b,h,i,d] * K[b,h,j,d]
 *     J_i    = {0 .. S-1}, or {0 .. i} when causal (key j visible iff j <= i)
 *     O[b,h,i,:] = sum_{j in J_i} softmax_j(s_i.) * V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_{j in J_i} exp(s_ij)          (natural log)
 *
 * with fp32 accumulation; O is stored in the input dtype, LSE in fp32.
 *
 * FP8.  The same page times multi-head attention in FP8 as well as FP16
 * (Section V-D, Fig. 10: sequence length 1024-16384, batch 4, head dim 128).
 * With dtype FMHA_E4M3, Q, K and V hold E4M3 values (the OCP 8-bit format:
 * 4 exponent bits, 3 mantissa bits, largest finite 448, no infinities), both
 * products run on the 8-bit tensor-core path, P is rounded to E4M3 between
 * the two stages, O is stored in bf16 and LSE in fp32.  The definition above
 * applies to the E4M3 values as given; dequantisation scales are the
 * caller's: fold the Q and K scales into `scale` and multiply O by V's scale
 * (O is linear in V).
 */
#ifndef WSATTN_H_
#define WSATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes.  Every entry point returns one; none aborts the process. */
typedef enum {
  FMHA_OK = 0,
  FMHA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, non-finite or non-positive scale */
  FMHA_ERR_UNSUPPORTED = 2, /* valid but not implemented: D not in {64, 128}, unknown dtype,
                               E4M3 with D != 128 or S not a multiple of 16 */
  FMHA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (see fmha_last_cuda_error) */
  FMHA_ERR_TIMEOUT = 4      /* a device-side wait ran past its limit; outputs are undefined */
} fmha_status;

/* Element type of Q, K, V (and of O: the same, except bf16 for FMHA_E4M3). */
typedef enum { FMHA_F16 = 0, FMHA_BF16 = 1, FMHA_E4M3 = 2 } fmha_dtype;

/*
 * fmha_fwd -- fused attention forward pass, O and LSE, on one GPU.
 *
 *   q, k, v  device pointers, each B*H*S*D elements of `dtype`, contiguous
 *            (B, H, S, D): element (b,h,s,d) at ((b*H + h)*S + s)*D + d.
 *            Read only.  16-byte aligned.  For FMHA_E4M3, v holds V
 *            transposed per (batch, head), contiguous (B, H, D, S): element
 *            (b,h,s,d) of V at ((b*H + h)*D + d)*S + s.
 *   o        device pointer, B*H*S*D elements of `dtype` (bf16 for FMHA_E4M3),
 *            (B, H, S, D) layout.  Written.  16-byte aligned; must not overlap
 *            q, k, v or lse.
 *   lse      device pointer, B*H*S fp32, contiguous (B, H, S).  Written.
 *            4-byte aligned.
 *   B, H, S  batch, heads, sequence length (queries = keys), each >= 1;
 *            B*H < 2^31 and ceil(S/256)*B*H < 2^31.
 *   D        head dimension: 64 or 128 (anything else -> FMHA_ERR_UNSUPPORTED);
 *            128 for FMHA_E4M3, which also needs S % 16 == 0 (the rows of the
 *            transposed V must start on 16-byte boundaries).
 *   causal   0: every key visible; nonzero: key j visible to query i iff j <= i.
 *   scale    softmax scale applied to q.k, finite and > 0 (usually 1/sqrt(D)).
 *   dtype    FMHA_F16, FMHA_BF16 or FMHA_E4M3.
 *   stream   cudaStream_t (as void*) on which the kernel is enqueued; NULL is the
 *            legacy default stream.  Must belong to the current device, which
 *            must hold all five buffers.
 *
 * Ownership: the caller owns every buffer; the library allocates no device or
 * host memory and keeps no pointer after the call returns.
 *
 * Behaviour: arguments are validated on the host before any CUDA call; a bad
 * argument returns FMHA_ERR_INVALID_ARG / FMHA_ERR_UNSUPPORTED with nothing
 * enqueued.  Otherwise one kernel is enqueued and the call returns without
 * waiting for it (FMHA_ERR_CUDA if the launch itself failed).  A device-side
 * timeout is reported by the next fmha_get_device_status().  Safe to call from
 * several host threads on different streams; note that the timeout status is
 * one word per device, shared by every stream and thread (see
 * fmha_get_device_status).
 *
 * Results are deterministic for a given shape on a given GPU model.  With full
 * attention, D = 128 and an even ceil(S/128), the units of a short last wave
 * (at most half the multiprocessors' worth) are computed in two key halves
 * and merged, so the rounding of those rows depends on the multiprocessor
 * count; every result stays within the same bounds of the exact one.
 */
fmha_status fmha_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int64_t B, int64_t H, int64_t S, int64_t D, int causal, float scale,
                     fmha_dtype dtype, void* stream);

/*
 * fmha_fwd_host -- fmha_fwd on host-resident tensors, with the host<->device
 * transfers overlapped with the computation.
 *
 *   q, k, v    host pointers, B*H*S*D elements of `dtype`, in fmha_fwd's
 *              layouts (v transposed per head for FMHA_E4M3).
 *              Page-locked (pinned) memory lets the copies run asynchronously
 *              and overlap; pageable memory works but serialises them.
 *   o, lse     host pointers, outputs in the same layouts as fmha_fwd.
 *   q_dev, k_dev, v_dev, o_dev, lse_dev
 *              caller-owned device staging buffers for q, k, v, o and lse, of
 *              the full sizes (the sizes and alignment rules of fmha_fwd's q,
 *              k, v, o, lse).  Their contents on entry do not matter; on
 *              return they hold the staged inputs and the outputs.
 *   n_chunks   0 for the default (16), else 1..64: the B*H (batch, head)
 *              slices are split into this many contiguous chunks.  The
 *              host-to-device copy of chunk c+1 and the device-to-host copy of
 *              chunk c-1 run on two copy streams while chunk c is computed.
 *              Chunks alternate between `stream` and a second compute stream
 *              of the library, so that a chunk's kernel can start on SMs the
 *              previous chunk's last wave leaves idle.
 *   Other arguments as fmha_fwd.
 *
 * The rows of every (batch, head) slice are independent, so the result is
 * bit-identical to fmha_fwd on the staged device tensors.  The call returns
 * once all work is enqueued; every copy and kernel is complete when `stream`
 * is (synchronise `stream` before reading o and lse).  The library's three
 * streams and a few events are created once per device and host thread and
 * reused; no memory is allocated.  Errors as fmha_fwd (a bad pointer or size is
 * FMHA_ERR_INVALID_ARG before anything is enqueued).
 */
fmha_status fmha_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                          void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev,
                          int64_t B, int64_t H, int64_t S, int64_t D, int causal, float scale,
                          fmha_dtype dtype, int n_chunks, void* stream);

/*
 * fmha_bwd_workspace_bytes -- bytes of device scratch fmha_bwd needs:
 * B*H*S*D + B*H*S fp32 values (a dQ accumulator and the per-row delta).
 * 0 for non-positive sizes.
 */
size_t fmha_bwd_workspace_bytes(int64_t B, int64_t H, int64_t S, int64_t D);

/*
 * fmha_bwd -- backward pass of fmha_fwd: the gradients dQ, dK, dV of a loss L
 * given dO = dL/dO.  The pages schedule this kernel as well ("Optimal Software
 * Pipelining and Warp Specialization for Tensor Core GPUs", Sections 6.3-6.4,
 * FlashAttention backward) without writing it out; it is the chain rule of the
 * definition above, per (batch, head):
 *
 *     P = softmax(scale Q K^T [+ mask]) = exp(scale Q K^T - LSE)   (row-wise)
 *     dV = P^T dO,   dP = dO V^T,   delta_i = dO_i . O_i,
 *     dS = P * (dP - delta),   dQ = scale dS K,   dK = scale dS^T Q.
 *
 *   q, k, v, o, lse   the forward's inputs, output and LSE (layouts as in
 *                     fmha_fwd; lse must come from the same q, k, v, scale,
 *                     causal).  Read only.
 *   d_o               device, (B, H, S, D) `dtype`.  Read only.
 *   dq, dk, dv        device, (B, H, S, D) `dtype`.  Written.
 *   workspace         device scratch of at least fmha_bwd_workspace_bytes()
 *                     bytes, 16-byte aligned, owned by the caller; its contents
 *                     on entry do not matter and are undefined on return.
 *   dtype             FMHA_F16 or FMHA_BF16 (FMHA_E4M3 -> FMHA_ERR_UNSUPPORTED);
 *                     D 64 or 128; other arguments as fmha_fwd.
 *
 * All device pointers 16-byte aligned (lse 4); outputs and workspace must not
 * overlap each other or any input.  Asynchronous on `stream`: a memset and
 * three kernels are enqueued (delta, the warp-specialized backward, the dQ
 * conversion); no memory is allocated.  dQ is accumulated with fp32 atomic
 * additions across key blocks, so its last bits may differ between runs.
 * Errors as fmha_fwd.
 */
fmha_status fmha_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* d_o, void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, int64_t B, int64_t H, int64_t S, int64_t D,
                     int causal, float scale, fmha_dtype dtype, void* stream);

/*
 * fmha_bwd_noalloc -- fmha_bwd without a workspace argument: the dQ
 * accumulator and delta live in a device array of the library (96 MiB, one
 * per device), so the call needs no memory from the caller or an allocator.
 * The pages have no counterpart.  It serves callers that cannot hand the
 * backward a workspace because they may not allocate device memory while
 * they run: a runtime that reserves its whole device-memory budget up front
 * and forbids later cudaMalloc calls, or code inside another library's
 * allocation-free region.
 *
 *   Arguments as fmha_bwd, minus workspace and workspace_bytes.
 *   Capacity: B*H*S*(4*D + 4) bytes must fit in 96 MiB (B*H*S <= 195,084
 *   rows at D = 128, <= 387,166 at D = 64); larger inputs return
 *   FMHA_ERR_UNSUPPORTED before any CUDA call, as do E4M3 inputs.
 *   Races: every call on a device uses the same array, so calls whose work
 *   overlaps in time (different streams, or several host threads) corrupt
 *   each other's dQ; serialise them (one stream, or events).
 *   Set-up: the first call on a device looks up the array's address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.
 * Errors as fmha_bwd.
 */
fmha_status fmha_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                             int64_t B, int64_t H, int64_t S, int64_t D, int causal, float scale,
                             fmha_dtype dtype, void* stream);

/*
 * fmha_bwd_host_scratch_bytes -- bytes of device scratch fmha_bwd_host needs:
 * staging for q, k, v, o, d_o, dq, dk, dv and lse plus fmha_bwd's workspace,
 * each region starting on 256 bytes.  0 for non-positive sizes.
 */
size_t fmha_bwd_host_scratch_bytes(int64_t B, int64_t H, int64_t S, int64_t D);

/*
 * fmha_bwd_host -- fmha_bwd on host-resident tensors, with the host<->device
 * transfers overlapped with the computation (the backward counterpart of
 * fmha_fwd_host; the pages have none).
 *
 *   q, k, v, o, lse, d_o
 *              host pointers, inputs in fmha_bwd's layouts (16-bit only).
 *              Page-locked (pinned) memory lets the copies run asynchronously
 *              and overlap; pageable memory works but serialises them.
 *   dq, dk, dv host pointers, outputs in the same layout.
 *   scratch, scratch_bytes
 *              caller-owned device memory of at least
 *              fmha_bwd_host_scratch_bytes() bytes, 256-byte aligned; its
 *              contents need not be initialised and are overwritten.
 *   n_chunks   0 for the default (16), else 1..64: the B*H (batch, head)
 *              slices are split into this many contiguous chunks; each
 *              chunk's inputs are copied in, its backward pass (delta, the
 *              main kernel, the dQ conversion) runs, and its gradients are
 *              copied back, with the copies on two library streams and the
 *              chunks' work alternating between `stream` and a second
 *              compute stream of the library.
 *   Other arguments as fmha_bwd.
 *
 * Slices are independent, so dK and dV are bit-identical to fmha_bwd on the
 * staged tensors; dQ sums its key blocks' parts in an unspecified order (as
 * in fmha_bwd).  The call returns once all work is enqueued; everything is
 * complete when `stream` is.  Streams and events are those of
 * fmha_fwd_host; no memory is allocated.  Errors as fmha_bwd (a bad pointer
 * or size, or too little scratch, is FMHA_ERR_INVALID_ARG before anything is
 * enqueued).
 */
fmha_status fmha_bwd_host(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                          void* scratch, size_t scratch_bytes, int64_t B, int64_t H, int64_t S,
                          int64_t D, int causal, float scale, fmha_dtype dtype, int n_chunks,
                          void* stream);

/*
 * fmha_get_device_status -- synchronise `stream`, then report and clear the
 * device status word of the current device.  Returns FMHA_ERR_TIMEOUT if any
 * kernel since the previous call abandoned a wait, FMHA_ERR_CUDA if the stream
 * reported an error, FMHA_OK otherwise.
 *
 * Scope: the status word is one per device, shared by every stream and host
 * thread that launches this library's kernels there.  The call waits only for
 * `stream`: a timeout raised by a kernel still running on another stream is
 * not seen yet, and a timeout raised on any stream is reported (and cleared)
 * by whichever caller reads the word first.  Callers on several streams that
 * need per-stream attribution synchronise the device (or every such stream)
 * before this call, and read it from one thread.
 */
fmha_status fmha_get_device_status(void* stream);

/* Static text for a status code. */
const char* fmha_status_str(fmha_status status);

/* Text of the CUDA error behind the calling thread's last FMHA_ERR_CUDA ("" if none). */
const char* fmha_last_cuda_error(void);

/* Library version, (major << 16) | (minor << 8) | patch. */
int fmha_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WSATTN_H_ */
