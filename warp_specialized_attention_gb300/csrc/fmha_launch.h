// fmha_launch.h -- host-side launcher declarations shared by the API translation
// unit and the per-head-dim kernel translation units (compiled in parallel).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace wsa {

struct FwdParams;
struct BwdParams;

// Enqueue the forward kernel for one (head dim, dtype, mask) variant.
// `to` maps O (D, S, B*H) in 16-bit boxes of 64 columns x 32 rows, 128-byte
// swizzle, for the epilogue's TMA stores.
cudaError_t launch_fwd_d64(bool bf16, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& prm,
                           unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_d128(bool bf16, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& prm,
                            unsigned grid, cudaStream_t stream);

// E4M3 inputs, head dim 128: tvt maps V transposed, (S, D, B*H); O is bf16.
cudaError_t launch_fwd_e4m3(bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tvt, const CUtensorMap& to, const FwdParams& prm,
                            unsigned grid, cudaStream_t stream);

// Full attention, head dim 128, with the grid's units from prm.n_whole on
// key-split; et = kF16, kBF16 or kE4M3 (the maps as for the launchers above).
cudaError_t launch_fwd_ksplit(int et, const CUtensorMap& tq, const CUtensorMap& tk,
                              const CUtensorMap& tv, const CUtensorMap& to, const FwdParams& prm,
                              unsigned grid, cudaStream_t stream);

// Backward pass (16-bit, D = 64 or 128): the main kernel over (head, key
// block), the delta pre-pass over rows, and the dQ conversion of n elements.
// tdq maps the fp32 dQ accumulator (D, S, B*H) with 16 x 32 x 1 boxes and the
// 64-byte swizzle.
cudaError_t launch_bwd(int D, bool bf16, bool causal, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdq, const BwdParams& prm, unsigned grid,
                       cudaStream_t stream);
cudaError_t launch_bwd_delta(int D, bool bf16, const void* o, const void* d_o, float* delta,
                             int64_t rows, cudaStream_t stream);
cudaError_t launch_bwd_dq(bool bf16, const float* acc, void* dq, int64_t n, cudaStream_t stream);

// Capacity of the file-scope scratch of the allocation-free backward entry
// point, and its device address (looked up once per device).
constexpr size_t kBwdStaticScratchBytes = size_t{96} << 20;
cudaError_t bwd_static_scratch(void** out);

}  // namespace wsa
