// fmha_launch.h -- host-side launcher declarations shared by the API translation
// unit and the per-head-dim kernel translation units (compiled in parallel).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace wsa {

struct FwdParams;

// Enqueue the forward kernel for one (head dim, dtype, mask) variant.
cudaError_t launch_fwd_d64(bool bf16, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const FwdParams& prm, unsigned grid,
                           cudaStream_t stream);
cudaError_t launch_fwd_d128(bool bf16, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const FwdParams& prm, unsigned grid,
                            cudaStream_t stream);

// E4M3 inputs, head dim 128: tvt maps V transposed, (S, D, B*H).
cudaError_t launch_fwd_e4m3(bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tvt, const FwdParams& prm, unsigned grid,
                            cudaStream_t stream);

}  // namespace wsa
