// fmha_fwd_ksplit.cu -- instantiations of the forward kernel whose grids end
// in key-split units (full attention, head dim 128: f16, bf16 and E4M3).
#include "fmha_fwd_sm103.cuh"
#include "fmha_launch.h"

namespace wsa {

cudaError_t launch_fwd_ksplit(int et, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& prm,
                              unsigned grid, cudaStream_t stream) {
  if (et == kE4M3) return launch_fmha_fwd<128, kE4M3, false, true>(tq, tk, tv, to, prm, grid, stream);
  if (et == kBF16) return launch_fmha_fwd<128, kBF16, false, true>(tq, tk, tv, to, prm, grid, stream);
  return launch_fmha_fwd<128, kF16, false, true>(tq, tk, tv, to, prm, grid, stream);
}

}  // namespace wsa
