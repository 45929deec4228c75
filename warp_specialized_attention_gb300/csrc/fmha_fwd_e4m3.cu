// fmha_fwd_e4m3.cu -- instantiations of the forward kernel for E4M3 inputs
// (head dim 128; V transposed per head; O in bf16).
#include "fmha_fwd_sm103.cuh"
#include "fmha_launch.h"

namespace wsa {

cudaError_t launch_fwd_e4m3(bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tvt, const CUtensorMap& to, const FwdParams& prm, unsigned grid,
                            cudaStream_t stream) {
  return causal ? launch_fmha_fwd<128, kE4M3, true>(tq, tk, tvt, to, prm, grid, stream)
                : launch_fmha_fwd<128, kE4M3, false>(tq, tk, tvt, to, prm, grid, stream);
}

}  // namespace wsa
