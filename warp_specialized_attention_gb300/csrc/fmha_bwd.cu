// fmha_bwd.cu -- instantiations and launchers of the attention backward pass:
// the delta pre-pass, the warp-specialized dQ/dK/dV kernel and the dQ
// conversion.
#include <atomic>

#include "fmha_bwd_sm103.cuh"
#include "fmha_launch.h"

namespace wsa {

namespace {

// Scratch of the allocation-free backward entry point: the dQ accumulator and
// delta (B*H*S*(4D + 4) bytes) in a file-scope device array, so a call needs
// no memory from anyone.  Every call on this device shares it.
__device__ __align__(256) unsigned char g_bwd_scratch[kBwdStaticScratchBytes];

template <int D, int ET, bool CAUSAL>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdParams& prm,
                         unsigned grid, cudaStream_t stream) {
  auto kern = fmha_bwd_kernel<D, ET, CAUSAL>;
  // Dynamic shared memory above 48 KB is opted into once per device (flags
  // private to this library copy: internal linkage).
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> opted_in[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !opted_in[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BwdCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    // The register split hands out exactly the registers the block is
    // launched with: refuse a build that gave the kernel another count.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kBwdRegLaunch) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < kMaxDevices) opted_in[dev].store(true, std::memory_order_release);
  }
  kern<<<grid, kBwdThreads, BwdCfg<D>::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, prm);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_d(bool bf16, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                         const BwdParams& prm, unsigned grid, cudaStream_t stream) {
  if (bf16)
    return causal ? launch_bwd_t<D, kBF16, true>(tq, tk, tv, tdo, tdq, prm, grid, stream)
                  : launch_bwd_t<D, kBF16, false>(tq, tk, tv, tdo, tdq, prm, grid, stream);
  return causal ? launch_bwd_t<D, kF16, true>(tq, tk, tv, tdo, tdq, prm, grid, stream)
                : launch_bwd_t<D, kF16, false>(tq, tk, tv, tdo, tdq, prm, grid, stream);
}

}  // namespace

cudaError_t bwd_static_scratch(void** out) {
  // looked up once per device (the first call, which should precede any
  // stream capture); later calls only read the cache
  constexpr int kMaxDevices = 64;
  static std::atomic<void*> cache[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = cache[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess) return e;
    cache[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

cudaError_t launch_bwd(int D, bool bf16, bool causal, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdq, const BwdParams& prm, unsigned grid,
                       cudaStream_t stream) {
  return D == 64 ? launch_bwd_d<64>(bf16, causal, tq, tk, tv, tdo, tdq, prm, grid, stream)
                 : launch_bwd_d<128>(bf16, causal, tq, tk, tv, tdo, tdq, prm, grid, stream);
}

cudaError_t launch_bwd_delta(int D, bool bf16, const void* o, const void* d_o, float* delta,
                             int64_t rows, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
  if (D == 64) {
    if (bf16)
      fmha_bwd_delta_kernel<64, kBF16><<<grid, 256, 0, stream>>>(o, d_o, delta, rows);
    else
      fmha_bwd_delta_kernel<64, kF16><<<grid, 256, 0, stream>>>(o, d_o, delta, rows);
  } else {
    if (bf16)
      fmha_bwd_delta_kernel<128, kBF16><<<grid, 256, 0, stream>>>(o, d_o, delta, rows);
    else
      fmha_bwd_delta_kernel<128, kF16><<<grid, 256, 0, stream>>>(o, d_o, delta, rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(bool bf16, const float* acc, void* dq, int64_t n,
                          cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((n / 4 + 255) / 256);
  if (bf16)
    fmha_bwd_dq_kernel<kBF16><<<grid, 256, 0, stream>>>(acc, dq, n);
  else
    fmha_bwd_dq_kernel<kF16><<<grid, 256, 0, stream>>>(acc, dq, n);
  return cudaGetLastError();
}

}  // namespace wsa
