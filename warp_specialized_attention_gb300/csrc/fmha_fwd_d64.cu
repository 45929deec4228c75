// fmha_fwd_d64.cu -- instantiations of the forward kernel for head dim 64.
#include "fmha_fwd_sm103.cuh"
#include "fmha_launch.h"

namespace wsa {

cudaError_t launch_fwd_d64(bool bf16, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& prm,
                           unsigned grid, cudaStream_t stream) {
  if (bf16)
    return causal ? launch_fmha_fwd<64, kBF16, true>(tq, tk, tv, to, prm, grid, stream)
                  : launch_fmha_fwd<64, kBF16, false>(tq, tk, tv, to, prm, grid, stream);
  return causal ? launch_fmha_fwd<64, kF16, true>(tq, tk, tv, to, prm, grid, stream)
                : launch_fmha_fwd<64, kF16, false>(tq, tk, tv, to, prm, grid, stream);
}

}  // namespace wsa
