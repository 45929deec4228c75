// fmha_bwd_sm103.cuh -- the tensor-core forms of the attention backward pass
// that the forward kernel does not use.
//
// With the keys of a 128-key block on the TMEM lanes, the backward pass needs
// five products per 128-row query block.  Three of them have forward forms:
//   S^T  = K Q^T      (issue_qk: both operands K-major)
//   dP^T = V dO^T     (issue_qk)
//   dV  += P^T dO     (issue_pv: P^T from TMEM, dO MN-major)
// The other two take their A operand from one shared-memory tile of dS^T
// (128 keys x 128 queries, 16-bit, two 64-column blocks, 128-byte swizzle):
//   dK  += dS^T Q     A = dS^T read K-major (keys = M, queries = K),
//                     B = Q read MN-major (queries = K rows, head dim = N)
//   dQ   = dS K       A = the same tile read MN-major (queries = M contiguous,
//                     keys = K rows), B = K read MN-major
// Both are 8 steps of K = 16.  Descriptors: K-major steps move 32 bytes along
// a row and every fourth step the next 16 KB column block; MN-major steps move
// 16 rows (2 KB), with the leading byte offset (16 KB) between 64-element
// column blocks.
#pragma once
#include "fmha_fwd_sm103.cuh"

namespace wsa {

template <int D, int ET>
__device__ __forceinline__ void issue_kmaj_mn(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                              bool accumulate) {
  constexpr uint32_t idesc = idesc_f16_ab(ET == kBF16, 128, D, false, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t a_step = (kk >> 2) * ((128 * 128) >> 4) + (kk & 3) * (32 >> 4);
    const uint32_t b_step = kk * ((16 * 128) >> 4);
    mma_ss_warp(d_tmem, sdesc_join(a_lo + a_step, kDescHi), sdesc_join(b_lo + b_step, kDescHi),
                idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int D, int ET>
__device__ __forceinline__ void issue_mn_mn(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                            bool accumulate) {
  constexpr uint32_t idesc = idesc_f16_ab(ET == kBF16, 128, D, true, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t step = kk * ((16 * 128) >> 4);
    mma_ss_warp(d_tmem, sdesc_join(a_lo + step, kDescHi), sdesc_join(b_lo + step, kDescHi),
                idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

}  // namespace wsa
