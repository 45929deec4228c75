// probes.cu -- single-purpose kernels that exercise, in isolation, the pieces
// the attention kernel is built from: a 128-byte-swizzled TMA tile load, the
// SMEM x SMEM tcgen05.mma of S = Q K^T (K-major descriptors) and the
// TMEM x SMEM tcgen05.mma of O = P V (P written to TMEM by tcgen05.st, V as an
// MN-major descriptor), each read back with tcgen05.ld.  They call the very
// helpers the attention kernel uses (issue_qk, issue_pv), so a wrong descriptor
// bit shows up here on one tile.  Test-only library: libwsattn_probes.so.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "fmha_bwd_sm103.cuh"
#include "fmha_fwd_sm103.cuh"
#include "wsattn_probes.h"

namespace {

using namespace wsa;

constexpr uint64_t kProbeWaitNs = 1000000000ull;
__device__ int g_probe_status = 0;

struct ProbeSmem {
  uint64_t bar_load;
  uint64_t bar_mma;
  uint32_t tmem_base;
  int abort;
};

// C[128][128] (fp32) = A[128][K] * B[128][K]^T, K = D in {64, 128}.
template <int D, bool BF16>
__global__ void __launch_bounds__(128, 1)
    probe_qk_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                    float* c) {
  extern __shared__ uint8_t raw[];
  const uint32_t raw_addr = smem_u32(raw);
  uint8_t* sm = raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sA = smem_u32(sm), sB = sA + 128 * D * 2;
  ProbeSmem& ctl = *reinterpret_cast<ProbeSmem*>(sm + 2 * 128 * D * 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl.bar_load, 1);
    mbar_init(&ctl.bar_mma, 1);
    ctl.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl.tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* ab = &ctl.abort;
  if (warp == 0) {  // warp-collective issue, as in the attention kernel
    mbar_arrive_expect_tx_warp(&ctl.bar_load, 2 * 128 * D * 2);
    for (int cb = 0; cb < D / 64; ++cb) {
      tma_load_3d_warp(sA + cb * 128 * 128, &ta, &ctl.bar_load, cb * 64, 0, 0, policy_evict_first());
      tma_load_3d_warp(sB + cb * 128 * 128, &tb, &ctl.bar_load, cb * 64, 0, 0, policy_evict_first());
    }
    bool loaded = mbar_wait(&ctl.bar_load, 0, ab, &g_probe_status, 1, kProbeWaitNs);
    if (__all_sync(0xffffffffu, loaded)) {
      tc_fence_after();
      issue_qk<D, BF16 ? kBF16 : kF16>(tmem, sdesc_lo(sA, kLboKMajor), sdesc_lo(sB, kLboKMajor));
    }
    mma_commit_warp(&ctl.bar_mma);
  }
  __syncwarp();
  bool ok = mbar_wait(&ctl.bar_mma, 0, nullptr, &g_probe_status, 2, kProbeWaitNs);
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
    tc_fence_after();
    uint32_t r[128];
    tmem_ld_x128(tmem + (static_cast<uint32_t>(warp * 32) << 16), r);
    const int row = warp * 32 + lane;
    for (int j = 0; j < 128; ++j) c[row * 128 + j] = __uint_as_float(r[j]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// O[128][D] (fp32) = P[128][128] * V[128][D]; P goes to TMEM with tcgen05.st.
template <int D, bool BF16>
__global__ void __launch_bounds__(128, 1)
    probe_pv_kernel(const uint16_t* p, const __grid_constant__ CUtensorMap tv, float* o) {
  extern __shared__ uint8_t raw[];
  const uint32_t raw_addr = smem_u32(raw);
  uint8_t* sm = raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sV = smem_u32(sm);
  ProbeSmem& ctl = *reinterpret_cast<ProbeSmem*>(sm + 128 * D * 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl.bar_load, 1);
    mbar_init(&ctl.bar_mma, 1);
    ctl.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  // P row `row` -> TMEM lane `row`, columns [0,64), two 16-bit values per column
  const int row = warp * 32 + lane;
  uint32_t pk[64];
  const uint32_t* prow = reinterpret_cast<const uint32_t*>(p + row * 128);
  for (int i = 0; i < 64; ++i) pk[i] = prow[i];
  tmem_st_x64(lane_base, pk);
  tc_fence_before();
  __syncthreads();
  volatile int* ab = &ctl.abort;
  if (warp == 0) {  // warp-collective issue, as in the attention kernel
    tc_fence_after();
    mbar_arrive_expect_tx_warp(&ctl.bar_load, 128 * D * 2);
    for (int cb = 0; cb < D / 64; ++cb)
      tma_load_3d_warp(sV + cb * 128 * 128, &tv, &ctl.bar_load, cb * 64, 0, 0, policy_evict_first());
    bool loaded = mbar_wait(&ctl.bar_load, 0, ab, &g_probe_status, 1, kProbeWaitNs);
    if (__all_sync(0xffffffffu, loaded)) {
      tc_fence_after();
      issue_pv<D, BF16 ? kBF16 : kF16>(tmem + 128, tmem, sdesc_lo(sV, kLboV), false);
    }
    mma_commit_warp(&ctl.bar_mma);
  }
  __syncwarp();
  bool ok = mbar_wait(&ctl.bar_mma, 0, nullptr, &g_probe_status, 2, kProbeWaitNs);
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
    tc_fence_after();
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t r[32];
      tmem_ld_x32(lane_base + 128 + ch * 32, r);
      for (int j = 0; j < 32; ++j) o[row * D + ch * 32 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// 8-bit (E4M3) forms.  Both operands K-major, 128 bytes per row, 128-byte
// swizzle: one 16 KB tile of 128 rows x 128 elements.  A K = 32 step moves 32
// bytes along the row, inside one swizzle atom.
constexpr uint32_t kIdescE4m3 = idesc_f16(false, 128, 128, false);  // E4M3 = format 0

// C[128][128] (fp32) = A[128][128] * B[128][128]^T, A and B E4M3.
__global__ void __launch_bounds__(128, 1)
    probe_qk_e4m3_kernel(const __grid_constant__ CUtensorMap ta,
                         const __grid_constant__ CUtensorMap tb, float* c) {
  extern __shared__ uint8_t raw[];
  const uint32_t raw_addr = smem_u32(raw);
  uint8_t* sm = raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sA = smem_u32(sm), sB = sA + 16384;
  ProbeSmem& ctl = *reinterpret_cast<ProbeSmem*>(sm + 2 * 16384);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl.bar_load, 1);
    mbar_init(&ctl.bar_mma, 1);
    ctl.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl.tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* ab = &ctl.abort;
  if (warp == 0) {
    mbar_arrive_expect_tx_warp(&ctl.bar_load, 2 * 16384);
    tma_load_3d_warp(sA, &ta, &ctl.bar_load, 0, 0, 0, policy_evict_first());
    tma_load_3d_warp(sB, &tb, &ctl.bar_load, 0, 0, 0, policy_evict_first());
    bool loaded = mbar_wait(&ctl.bar_load, 0, ab, &g_probe_status, 1, kProbeWaitNs);
    if (__all_sync(0xffffffffu, loaded)) {
      tc_fence_after();
      for (int kk = 0; kk < 4; ++kk)
        mma_ss_f8_warp(tmem, sdesc_join(sdesc_lo(sA, kLboKMajor) + kk * 2, kDescHi),
                       sdesc_join(sdesc_lo(sB, kLboKMajor) + kk * 2, kDescHi), kIdescE4m3,
                       kk > 0 ? 1u : 0u);
    }
    mma_commit_warp(&ctl.bar_mma);
  }
  __syncwarp();
  bool ok = mbar_wait(&ctl.bar_mma, 0, nullptr, &g_probe_status, 2, kProbeWaitNs);
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
    tc_fence_after();
    uint32_t r[128];
    tmem_ld_x128(tmem + (static_cast<uint32_t>(warp * 32) << 16), r);
    const int row = warp * 32 + lane;
    for (int j = 0; j < 128; ++j) c[row * 128 + j] = __uint_as_float(r[j]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// O[128][128] (fp32) = P[128][128] * V[128][128], P and V E4M3.  P goes to
// TMEM with tcgen05.st (four values per column, 32 columns); V arrives
// transposed (vt[d][key]), so the B operand is K-major like the Q K^T forms.
__global__ void __launch_bounds__(128, 1)
    probe_pv_e4m3_kernel(const uint8_t* p, const __grid_constant__ CUtensorMap tvt, float* o) {
  extern __shared__ uint8_t raw[];
  const uint32_t raw_addr = smem_u32(raw);
  uint8_t* sm = raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sV = smem_u32(sm);
  ProbeSmem& ctl = *reinterpret_cast<ProbeSmem*>(sm + 16384);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl.bar_load, 1);
    mbar_init(&ctl.bar_mma, 1);
    ctl.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const int row = warp * 32 + lane;
  uint32_t pk[32];
  const uint32_t* prow = reinterpret_cast<const uint32_t*>(p + row * 128);
  for (int i = 0; i < 32; ++i) pk[i] = prow[i];
  tmem_st_x32_async(lane_base, pk);
  tmem_st_wait();
  tc_fence_before();
  __syncthreads();
  volatile int* ab = &ctl.abort;
  if (warp == 0) {
    tc_fence_after();
    mbar_arrive_expect_tx_warp(&ctl.bar_load, 16384);
    tma_load_3d_warp(sV, &tvt, &ctl.bar_load, 0, 0, 0, policy_evict_first());
    bool loaded = mbar_wait(&ctl.bar_load, 0, ab, &g_probe_status, 1, kProbeWaitNs);
    if (__all_sync(0xffffffffu, loaded)) {
      tc_fence_after();
      for (int kk = 0; kk < 4; ++kk)
        mma_ts_f8_warp(tmem + 128, tmem + kk * 8,
                       sdesc_join(sdesc_lo(sV, kLboKMajor) + kk * 2, kDescHi), kIdescE4m3,
                       kk > 0 ? 1u : 0u);
    }
    mma_commit_warp(&ctl.bar_mma);
  }
  __syncwarp();
  bool ok = mbar_wait(&ctl.bar_mma, 0, nullptr, &g_probe_status, 2, kProbeWaitNs);
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
    tc_fence_after();
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t r[32];
      tmem_ld_x32(lane_base + 128 + ch * 32, r);
      for (int j = 0; j < 32; ++j) o[row * 128 + ch * 32 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// The backward pass's two SS forms on one tile: C[128][D] (fp32) = A B with
// x = the 128 x 128 16-bit tile holding A (MODE 0: A itself, K-major; MODE 1:
// A transposed, read MN-major) and y = B[128][D] (rows = K, read MN-major).
template <int D, bool BF16, int MODE>
__global__ void __launch_bounds__(128, 1)
    probe_bwd_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap ty,
                     float* c) {
  extern __shared__ uint8_t raw[];
  const uint32_t raw_addr = smem_u32(raw);
  uint8_t* sm = raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sX = smem_u32(sm), sY = sX + 128 * 128 * 2;
  ProbeSmem& ctl = *reinterpret_cast<ProbeSmem*>(sm + 128 * 128 * 2 + 128 * D * 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl.bar_load, 1);
    mbar_init(&ctl.bar_mma, 1);
    ctl.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl.tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* ab = &ctl.abort;
  constexpr int kET = BF16 ? kBF16 : kF16;
  if (warp == 0) {
    mbar_arrive_expect_tx_warp(&ctl.bar_load, 128 * 128 * 2 + 128 * D * 2);
    for (int cb = 0; cb < 2; ++cb)
      tma_load_3d_warp(sX + cb * 128 * 128, &tx, &ctl.bar_load, cb * 64, 0, 0, policy_evict_first());
    for (int cb = 0; cb < D / 64; ++cb)
      tma_load_3d_warp(sY + cb * 128 * 128, &ty, &ctl.bar_load, cb * 64, 0, 0, policy_evict_first());
    bool loaded = mbar_wait(&ctl.bar_load, 0, ab, &g_probe_status, 1, kProbeWaitNs);
    if (__all_sync(0xffffffffu, loaded)) {
      tc_fence_after();
      if (MODE == 0)
        issue_kmaj_mn<D, kET>(tmem, sdesc_lo(sX, kLboKMajor), sdesc_lo(sY, kLboV), false);
      else
        issue_mn_mn<D, kET>(tmem, sdesc_lo(sX, kLboV), sdesc_lo(sY, kLboV), false);
    }
    mma_commit_warp(&ctl.bar_mma);
  }
  __syncwarp();
  bool ok = mbar_wait(&ctl.bar_mma, 0, nullptr, &g_probe_status, 2, kProbeWaitNs);
  ok = __all_sync(0xffffffffu, ok);
  if (ok) {
    tc_fence_after();
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int row = warp * 32 + lane;
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t r[32];
      tmem_ld_x32(lane_base + ch * 32, r);
      for (int j = 0; j < 32; ++j) c[row * D + ch * 32 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 128 rows x D 16-bit matrix as a (D, 128, 1) map with the attention kernel's box.
bool encode_tile(CUtensorMap* m, const void* ptr, int D, bool bf16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), 128, 1};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2),
                                 static_cast<cuuint64_t>(128 * D * 2)};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
             const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 128 x 128 E4M3 matrix as a (128, 128, 1) byte map, box 128 x 128 x 1.
bool encode_tile_u8(CUtensorMap* m, const void* ptr) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {128, 128, 1};
  const cuuint64_t strides[2] = {128, 128 * 128};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool BF16>
int run_qk(const void* a, const void* b, float* c) {
  CUtensorMap ta, tb;
  if (!encode_tile(&ta, a, D, BF16) || !encode_tile(&tb, b, D, BF16)) return 3;
  const int smem = 1024 + 2 * 128 * D * 2 + 256;
  auto k = probe_qk_kernel<D, BF16>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 3;
  k<<<1, 128, smem>>>(ta, tb, c);
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}

template <int D, bool BF16>
int run_pv(const void* p, const void* v, float* o) {
  CUtensorMap tv;
  if (!encode_tile(&tv, v, D, BF16)) return 3;
  const int smem = 1024 + 128 * D * 2 + 256;
  auto k = probe_pv_kernel<D, BF16>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 3;
  k<<<1, 128, smem>>>(static_cast<const uint16_t*>(p), tv, o);
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}

int probe_status() {
  int w = 0;
  if (cudaMemcpyFromSymbol(&w, g_probe_status, sizeof(int)) != cudaSuccess) return 3;
  if (w) {
    const int z = 0;
    cudaMemcpyToSymbol(g_probe_status, &z, sizeof(int));
    return 4;
  }
  return 0;
}

template <int D, bool BF16, int MODE>
int run_bwd(const void* x, const void* y, float* c) {
  CUtensorMap tx, ty;
  if (!encode_tile(&tx, x, 128, BF16) || !encode_tile(&ty, y, D, BF16)) return 3;
  const int smem = 1024 + 128 * 128 * 2 + 128 * D * 2 + 256;
  auto k = probe_bwd_kernel<D, BF16, MODE>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 3;
  k<<<1, 128, smem>>>(tx, ty, c);
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}

template <int MODE>
int dispatch_bwd(const void* x, const void* y, float* c, int D, int bf16) {
  if (D == 64) return bf16 ? run_bwd<64, true, MODE>(x, y, c) : run_bwd<64, false, MODE>(x, y, c);
  if (D == 128)
    return bf16 ? run_bwd<128, true, MODE>(x, y, c) : run_bwd<128, false, MODE>(x, y, c);
  return 2;
}

int run_qk_e4m3(const void* a, const void* b, float* c) {
  CUtensorMap ta, tb;
  if (!encode_tile_u8(&ta, a) || !encode_tile_u8(&tb, b)) return 3;
  const int smem = 1024 + 2 * 16384 + 256;
  if (cudaFuncSetAttribute(probe_qk_e4m3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return 3;
  probe_qk_e4m3_kernel<<<1, 128, smem>>>(ta, tb, c);
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}

int run_pv_e4m3(const void* p, const void* vt, float* o) {
  CUtensorMap tv;
  if (!encode_tile_u8(&tv, vt)) return 3;
  const int smem = 1024 + 16384 + 256;
  if (cudaFuncSetAttribute(probe_pv_e4m3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return 3;
  probe_pv_e4m3_kernel<<<1, 128, smem>>>(static_cast<const uint8_t*>(p), tv, o);
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}

}  // namespace

extern "C" {

int wsa_probe_qk(const void* a, const void* b, float* c, int D, int bf16) {
  if (!a || !b || !c || (reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15)
    return 1;
  int r;
  if (D == 64)
    r = bf16 ? run_qk<64, true>(a, b, c) : run_qk<64, false>(a, b, c);
  else if (D == 128)
    r = bf16 ? run_qk<128, true>(a, b, c) : run_qk<128, false>(a, b, c);
  else
    return 2;
  return r ? r : probe_status();
}

int wsa_probe_pv(const void* p, const void* v, float* o, int D, int bf16) {
  if (!p || !v || !o || (reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(v)) & 15)
    return 1;
  int r;
  if (D == 64)
    r = bf16 ? run_pv<64, true>(p, v, o) : run_pv<64, false>(p, v, o);
  else if (D == 128)
    r = bf16 ? run_pv<128, true>(p, v, o) : run_pv<128, false>(p, v, o);
  else
    return 2;
  return r ? r : probe_status();
}

int wsa_probe_qk_e4m3(const void* a, const void* b, float* c) {
  if (!a || !b || !c || (reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15)
    return 1;
  const int r = run_qk_e4m3(a, b, c);
  return r ? r : probe_status();
}

int wsa_probe_pv_e4m3(const void* p, const void* vt, float* o) {
  if (!p || !vt || !o || (reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(vt)) & 15)
    return 1;
  const int r = run_pv_e4m3(p, vt, o);
  return r ? r : probe_status();
}

int wsa_probe_kmaj_mn(const void* a, const void* b, float* c, int D, int bf16) {
  if (!a || !b || !c || (reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15)
    return 1;
  const int r = dispatch_bwd<0>(a, b, c, D, bf16);
  return r ? r : probe_status();
}

int wsa_probe_mn_mn(const void* at, const void* b, float* c, int D, int bf16) {
  if (!at || !b || !c || (reinterpret_cast<uintptr_t>(at) | reinterpret_cast<uintptr_t>(b)) & 15)
    return 1;
  const int r = dispatch_bwd<1>(at, b, c, D, bf16);
  return r ? r : probe_status();
}

}  // extern "C"
