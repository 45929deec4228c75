// fmha_api.cu -- the C ABI of libwsattn.so: argument validation, TMA tensor
// maps, grid choice and launch of the warp-specialized forward kernel, plus the
// device status word that bounded waits report into.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "fmha_bwd_sm103.cuh"
#include "fmha_fwd_sm103.cuh"
#include "fmha_launch.h"
#include "wsattn.h"
#include "wsattn_testing.h"

namespace {

// OR of wsa::kStatusTimeout* bits raised by kernels on this device since the
// last fmha_get_device_status().
__device__ int g_wsa_status = 0;

constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;  // 1 s per wait
constexpr int kMaxDevices = 64;
// Causal unit order: heads are taken in groups whose K and V together fit in
// the 129 MB L2, and the longest query blocks of a group go first.  Larger
// groups give the longest-first order more units to balance; beyond the L2
// size the groups' K and V re-reads start to miss (a sweep of 8 MB to all
// heads: 128 MB is best or within 2 % for causal S = 4096 to 16384).
constexpr int64_t kGroupKvBytes = int64_t{128} << 20;

thread_local char t_last_cuda_error[256] = "";

fmha_status cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "%s: %s (%d)", what,
                cudaGetErrorString(e), static_cast<int>(e));
  return FMHA_ERR_CUDA;
}

// A driver-API failure (the tensor-map encoder), with the driver's own code.
fmha_status drv_fail(CUresult r, const char* what) {
  std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "%s: CUresult %d", what,
                static_cast<int>(r));
  return FMHA_ERR_CUDA;
}

// Makes the current device's primary context current on the calling host
// thread.  The driver-API tensor-map encoder needs a current context, and a
// thread that has not yet made a runtime call (a framework's worker thread,
// for instance) has none; cudaSetDevice initialises and binds it.
fmha_status bind_context() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);
  return e == cudaSuccess ? FMHA_OK : cuda_fail(e, "cudaSetDevice");
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver-entry-point query, so the
// library does not link libcuda and loads on hosts without a GPU driver.
EncodeTiledFn encode_fn(cudaError_t* err) {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                              cudaEnableDefault, &q);
    if (status == cudaSuccess && (q != cudaDriverEntryPointSuccess || f == nullptr))
      status = cudaErrorSymbolNotFound;
    fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  *err = status;
  return fn;
}

// (B*H, rows, cols) tensor viewed as a 3-D map: box = 128 bytes of a row
// (64 16-bit or 128 8-bit elements) x 128 rows x 1 head, 128-byte swizzle.
// Rows past the end read as zeros.  Q, K, V: rows = S, cols = D; the
// transposed E4M3 V: rows = D, cols = S.
CUresult encode_map(EncodeTiledFn enc, CUtensorMap* map, const void* ptr, int dtype, int64_t BH,
                    int64_t rows, int64_t cols) {
  const int64_t eb = dtype == FMHA_E4M3 ? 1 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols * eb),
                                 static_cast<cuuint64_t>(rows * cols * eb)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / eb), 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType t = dtype == FMHA_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                : dtype == FMHA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = enc(map, t, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r;
}

// O (B*H, S, D) in its 16-bit output type for the forward epilogue's TMA
// stores: boxes of 64 columns (128 bytes) x 32 rows (one softmax warp's rows)
// x 1 head, 128-byte swizzle; rows past S are not written.
CUresult encode_o_map(EncodeTiledFn enc, CUtensorMap* map, void* ptr, bool bf16, int64_t BH,
                      int64_t S, int64_t D) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2),
                                 static_cast<cuuint64_t>(S * D * 2)};
  const cuuint32_t box[3] = {64, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         3, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r;
}

// The backward's fp32 dQ accumulator (B*H, S, D): boxes of 32 rows x 16
// columns (64 bytes), 64-byte swizzle, for the kernel's TMA reduce-adds.
CUresult encode_dq_map(EncodeTiledFn enc, CUtensorMap* map, float* ptr, int64_t BH, int64_t S,
                       int64_t D) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 4),
                                 static_cast<cuuint64_t>(S * D * 4)};
  const cuuint32_t box[3] = {16, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r;
}

// Bytes per element of the inputs and of O.
size_t in_bytes(int dtype) { return dtype == FMHA_E4M3 ? 1 : 2; }
constexpr size_t kOutBytes = 2;

// Device address of the status word, looked up once per device.
cudaError_t status_word(int** out) {
  static std::atomic<int*> cache[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cacheable = dev >= 0 && dev < kMaxDevices;
  if (cacheable) {
    *out = cache[dev].load(std::memory_order_acquire);
    if (*out != nullptr) return cudaSuccess;
  }
  e = cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_wsa_status);
  if (e == cudaSuccess && cacheable) cache[dev].store(*out, std::memory_order_release);
  return e;
}

// Heads per group of the causal unit order: as many as keep the group's K and
// V within kGroupKvBytes, then evened out over the groups.
int causal_group_heads(int64_t BH, int64_t S, int64_t D) {
  const int64_t kv_per_head = 2 * S * D * 2;
  const int64_t cap = std::max<int64_t>(1, kGroupKvBytes / kv_per_head);
  const int64_t groups = (BH + cap - 1) / cap;
  return static_cast<int>((BH + groups - 1) / groups);
}

// Streaming multiprocessors of the current device, looked up once per device.
cudaError_t sm_count(int* out) {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cacheable = dev >= 0 && dev < kMaxDevices;
  if (cacheable && (*out = cache[dev].load(std::memory_order_acquire)) > 0) return cudaSuccess;
  e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && cacheable) cache[dev].store(*out, std::memory_order_release);
  return e;
}

// Whether units of this shape may be key-split: full attention under the
// one-issuer schedule (head dim 128), and an even number of key blocks, so
// that each tile of a split unit takes the same number of whole blocks and
// every tile's keys include at least one unmasked key.
bool key_split_allowed(int64_t S, int64_t D, int causal) {
  const int64_t nkv = (S + 127) / 128;
  return !causal && D == 128 && nkv % 2 == 0;
}

// How many of the last units to key-split.  Every full-attention unit costs
// the same, so with U units on n_sm SMs (one block each) the last wave holds
// U mod n_sm units and leaves the other SMs idle.  When that remainder fits
// in half of the SMs, its units are split: each becomes two 128-row halves
// whose two tiles take half of the keys each, so the last wave takes about
// half as long (B4 H32 S1K: 512 units, the last 56 on 152 SMs).
int64_t auto_split_units(int64_t units, int64_t S, int64_t D, int causal, int n_sm) {
  if (!key_split_allowed(S, D, causal) || n_sm <= 0) return 0;
  const int64_t r = units % n_sm;
  return 2 * r <= n_sm ? r : 0;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Sizes, scale and element type (no pointer).
fmha_status validate_sizes(int64_t B, int64_t H, int64_t S, int64_t D, float scale, int dtype) {
  if (B < 1 || H < 1 || S < 1 || D < 1) return FMHA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FMHA_ERR_INVALID_ARG;
  if (dtype != FMHA_F16 && dtype != FMHA_BF16 && dtype != FMHA_E4M3) return FMHA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return FMHA_ERR_UNSUPPORTED;
  if (dtype == FMHA_E4M3 && (D != 128 || S % 16 != 0)) return FMHA_ERR_UNSUPPORTED;
  const int64_t lim = (int64_t{1} << 31) - 1;
  if (B > lim || H > lim || S > lim || B * H > lim) return FMHA_ERR_INVALID_ARG;
  const int64_t nq = (S + 255) / 256;
  if (nq * B * H > lim) return FMHA_ERR_INVALID_ARG;
  return FMHA_OK;
}

fmha_status validate(const void* q, const void* k, const void* v, void* o, float* lse,
                     int64_t B, int64_t H, int64_t S, int64_t D, float scale, int dtype) {
  if (!q || !k || !v || !o || !lse) return FMHA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) & 15u)
    return FMHA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FMHA_ERR_INVALID_ARG;
  const fmha_status vs = validate_sizes(B, H, S, D, scale, dtype);
  if (vs != FMHA_OK) return vs;
  const size_t n = static_cast<size_t>(B * H) * static_cast<size_t>(S) * static_cast<size_t>(D);
  const size_t ib = n * in_bytes(dtype), ob = n * kOutBytes;
  const size_t lb = static_cast<size_t>(B * H * S) * 4;
  if (overlaps(o, ob, q, ib) || overlaps(o, ob, k, ib) || overlaps(o, ob, v, ib) ||
      overlaps(o, ob, lse, lb) || overlaps(lse, lb, q, ib) || overlaps(lse, lb, k, ib) ||
      overlaps(lse, lb, v, ib))
    return FMHA_ERR_INVALID_ARG;
  return FMHA_OK;
}

fmha_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                     int64_t H, int64_t S, int64_t D, int causal, float scale, int dtype,
                     void* stream, int inject, uint64_t wait_limit_ns, float tau = -1.f,
                     int64_t split_units = -1) {
  const fmha_status vs = validate(q, k, v, o, lse, B, H, S, D, scale, dtype);
  if (vs != FMHA_OK) return vs;

  const fmha_status bs = bind_context();
  if (bs != FMHA_OK) return bs;
  cudaError_t e;
  EncodeTiledFn enc = encode_fn(&e);
  if (!enc) return cuda_fail(e, "cuTensorMapEncodeTiled entry point");
  const bool bf16 = dtype == FMHA_BF16, e4m3 = dtype == FMHA_E4M3;
  const int64_t BH = B * H;
  alignas(64) CUtensorMap tq, tk, tv, to;
  CUresult r;
  if ((r = encode_map(enc, &tq, q, dtype, BH, S, D)) != CUDA_SUCCESS ||
      (r = encode_map(enc, &tk, k, dtype, BH, S, D)) != CUDA_SUCCESS ||
      (r = e4m3 ? encode_map(enc, &tv, v, dtype, BH, D, S)
                : encode_map(enc, &tv, v, dtype, BH, S, D)) != CUDA_SUCCESS ||
      (r = encode_o_map(enc, &to, o, bf16 || e4m3, BH, S, D)) != CUDA_SUCCESS)
    return drv_fail(r, "cuTensorMapEncodeTiled");

  int* status = nullptr;
  e = status_word(&status);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");

  wsa::FwdParams prm;
  prm.lse = lse;
  prm.status = status;
  prm.S = static_cast<int>(S);
  prm.n_qblk = static_cast<int>((S + 255) / 256);
  prm.BH = static_cast<int>(BH);
  prm.group_heads = causal ? causal_group_heads(BH, S, D) : 1;
  prm.dynamic = 1;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.wait_limit_ns = wait_limit_ns;
  prm.inject = inject;
  // E4M3 P is stored scaled by 2^(8 - tau), so its largest value is 256 < 448.
  // The default tau = 8 (scale 1) redoes blocks as rarely as the E4M3 range
  // allows; tau = 0 (scale 2^8) keeps smaller P out of the subnormal range at
  // the cost of an exact maximum on nearly every block (1.7x slower).
  if (tau < 0.f) tau = e4m3 ? wsa::kTauDefaultE4m3 : wsa::kTauDefault;
  prm.tau = tau;
  prm.p_shift = e4m3 ? 8.f - tau : 0.f;
  prm.two_pow_tau = std::exp2(tau + prm.p_shift);
  // The last split_units units run as key-split halves: two grid blocks each.
  const int64_t units = prm.n_qblk * BH;
  if (split_units < 0) {
    int n_sm = 0;
    e = sm_count(&n_sm);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(multiprocessor count)");
    split_units = auto_split_units(units, S, D, causal, n_sm);
  }
  if (units + split_units > (int64_t{1} << 31) - 1) split_units = 0;
  prm.n_whole = static_cast<int>(units - split_units);
  const unsigned grid = static_cast<unsigned>(units + split_units);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  e = split_units > 0 ? wsa::launch_fwd_ksplit(e4m3 ? wsa::kE4M3 : bf16 ? wsa::kBF16 : wsa::kF16,
                                               tq, tk, tv, to, prm, grid, st)
      : e4m3          ? wsa::launch_fwd_e4m3(causal != 0, tq, tk, tv, to, prm, grid, st)
      : D == 64       ? wsa::launch_fwd_d64(bf16, causal != 0, tq, tk, tv, to, prm, grid, st)
                      : wsa::launch_fwd_d128(bf16, causal != 0, tq, tk, tv, to, prm, grid, st);
  if (e != cudaSuccess)
    return cuda_fail(e, e == cudaErrorInvalidConfiguration
                            ? "kernel launch (refused: the kernel's register count differs from "
                              "the one its register split assumes)"
                            : "kernel launch");
  return FMHA_OK;
}

// ---------------------------------------------------------------- backward pass

size_t bwd_workspace_bytes(int64_t B, int64_t H, int64_t S, int64_t D) {
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(S);
  return rows * static_cast<size_t>(D) * 4 + rows * 4;  // dQ accumulator + delta, fp32
}

// Argument checks of the backward pass (no CUDA call).
fmha_status bwd_validate(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                         void* workspace, size_t workspace_bytes, int64_t B, int64_t H, int64_t S,
                         int64_t D, float scale, int dtype) {
  if (dtype == FMHA_E4M3) return FMHA_ERR_UNSUPPORTED;
  // q, k, v, o, lse as in the forward (o is an input here)
  const fmha_status vs = validate(q, k, v, const_cast<void*>(o), const_cast<float*>(lse), B, H,
                                  S, D, scale, dtype);
  if (vs != FMHA_OK) return vs;
  if (!d_o || !dq || !dk || !dv || !workspace) return FMHA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(d_o) | reinterpret_cast<uintptr_t>(dq) |
       reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv) |
       reinterpret_cast<uintptr_t>(workspace)) & 15u)
    return FMHA_ERR_INVALID_ARG;
  const int64_t BH = B * H, n_blk = (S + 127) / 128;
  if (n_blk * BH > (int64_t{1} << 31) - 1) return FMHA_ERR_INVALID_ARG;
  const size_t need = bwd_workspace_bytes(B, H, S, D);
  if (workspace_bytes < need) return FMHA_ERR_INVALID_ARG;
  const size_t tb = static_cast<size_t>(BH * S * D) * 2, lb = static_cast<size_t>(BH * S) * 4;
  const void* ins[6] = {q, k, v, o, d_o, lse};
  const size_t in_sz[6] = {tb, tb, tb, tb, tb, lb};
  void* outs[4] = {dq, dk, dv, workspace};
  const size_t out_sz[4] = {tb, tb, tb, need};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlaps(outs[i], out_sz[i], ins[j], in_sz[j])) return FMHA_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j)
      if (overlaps(outs[i], out_sz[i], outs[j], out_sz[j])) return FMHA_ERR_INVALID_ARG;
  }
  return FMHA_OK;
}

// Enqueues the backward pass of BH (batch, head) slices on `st`: clear the
// dQ accumulator, delta, the main kernel, the dQ conversion.  The arguments
// have been checked; dq_acc holds BH*S*D and delta BH*S floats.
fmha_status bwd_enqueue(const void* q, const void* k, const void* v, const void* o,
                        const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                        float* dq_acc, float* delta, int64_t BH, int64_t S, int64_t D, int causal,
                        float scale, int dtype, cudaStream_t st, uint64_t wait_limit_ns) {
  const int64_t n_blk = (S + 127) / 128;
  const fmha_status bs = bind_context();
  if (bs != FMHA_OK) return bs;
  cudaError_t e;
  EncodeTiledFn enc = encode_fn(&e);
  if (!enc) return cuda_fail(e, "cuTensorMapEncodeTiled entry point");
  alignas(64) CUtensorMap tq, tk, tv, tdo;
  CUresult r;
  if ((r = encode_map(enc, &tq, q, dtype, BH, S, D)) != CUDA_SUCCESS ||
      (r = encode_map(enc, &tk, k, dtype, BH, S, D)) != CUDA_SUCCESS ||
      (r = encode_map(enc, &tv, v, dtype, BH, S, D)) != CUDA_SUCCESS ||
      (r = encode_map(enc, &tdo, d_o, dtype, BH, S, D)) != CUDA_SUCCESS)
    return drv_fail(r, "cuTensorMapEncodeTiled");
  int* status = nullptr;
  if ((e = status_word(&status)) != cudaSuccess)
    return cuda_fail(e, "cudaGetSymbolAddress(status)");

  const bool bf16 = dtype == FMHA_BF16;
  alignas(64) CUtensorMap tdq;
  if ((r = encode_dq_map(enc, &tdq, dq_acc, BH, S, D)) != CUDA_SUCCESS)
    return drv_fail(r, "cuTensorMapEncodeTiled(dQ accumulator)");
  if ((e = cudaMemsetAsync(dq_acc, 0, static_cast<size_t>(BH * S * D) * 4, st)) != cudaSuccess)
    return cuda_fail(e, "clear the dQ accumulator");
  if ((e = wsa::launch_bwd_delta(static_cast<int>(D), bf16, o, d_o, delta, BH * S, st)) !=
      cudaSuccess)
    return cuda_fail(e, "delta kernel launch");
  wsa::BwdParams prm;
  prm.lse = lse;
  prm.delta = delta;
  prm.dq_accum = dq_acc;
  prm.dk = dk;
  prm.dv = dv;
  prm.status = status;
  prm.S = static_cast<int>(S);
  prm.n_blk = static_cast<int>(n_blk);
  prm.scale = scale;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.wait_limit_ns = wait_limit_ns;
  if ((e = wsa::launch_bwd(static_cast<int>(D), bf16, causal != 0, tq, tk, tv, tdo, tdq, prm,
                           static_cast<unsigned>(n_blk * BH), st)) != cudaSuccess)
    return cuda_fail(e, e == cudaErrorInvalidConfiguration
                            ? "backward kernel launch (refused: the kernel's register count "
                              "differs from the one its register split assumes)"
                            : "backward kernel launch");
  if ((e = wsa::launch_bwd_dq(bf16, dq_acc, dq, BH * S * D, st)) != cudaSuccess)
    return cuda_fail(e, "dQ conversion launch");
  return FMHA_OK;
}

fmha_status bwd_impl(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, int64_t B, int64_t H, int64_t S,
                     int64_t D, int causal, float scale, int dtype, void* stream,
                     uint64_t wait_limit_ns) {
  const fmha_status vs = bwd_validate(q, k, v, o, lse, d_o, dq, dk, dv, workspace,
                                      workspace_bytes, B, H, S, D, scale, dtype);
  if (vs != FMHA_OK) return vs;
  const int64_t BH = B * H;
  float* dq_acc = static_cast<float*>(workspace);
  float* delta = dq_acc + static_cast<size_t>(BH * S * D);
  return bwd_enqueue(q, k, v, o, lse, d_o, dq, dk, dv, dq_acc, delta, BH, S, D, causal, scale,
                     dtype, static_cast<cudaStream_t>(stream), wait_limit_ns);
}

// Per host thread and device: the two copy streams, a second compute stream
// and the events that chain chunks between them and the caller's stream
// (created on first use).
constexpr int kMaxChunks = 64;
// Chunks of the host-buffer entries when the caller passes 0.  The first
// chunk's copy in and the last chunk's copy out are the exposed transfers, so
// more chunks hide more, but every chunk costs the host a few copies, four
// tensor-map encodes and a launch.  At S16K, end to end: 8 / 16 / 32 chunks
// gave the forward 1511 / 1578 / 1583 TFLOPS and the backward 1067 / 1093 /
// 1121 on one machine, while on another 32 chunks took 13.7 ms per forward
// step against 10.8 ms for 16, its host enqueue falling behind the GPU.
constexpr int kDefaultChunks = 16;
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp = nullptr;
  cudaEvent_t copied[kMaxChunks], computed[kMaxChunks], entry = nullptr, done = nullptr;
};
thread_local HostPipe t_pipe[kMaxDevices];

fmha_status host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "device index");
  HostPipe& hp = t_pipe[dev];
  if (!hp.ready) {
    const unsigned ev_flags = cudaEventDisableTiming;
    if ((e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&hp.comp, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.entry, ev_flags)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.done, ev_flags)) != cudaSuccess)
      return cuda_fail(e, "copy stream/event creation");
    for (int c = 0; c < kMaxChunks; ++c)
      if ((e = cudaEventCreateWithFlags(&hp.copied[c], ev_flags)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&hp.computed[c], ev_flags)) != cudaSuccess)
        return cuda_fail(e, "copy event creation");
    hp.ready = true;
  }
  *out = &hp;
  return FMHA_OK;
}

fmha_status fwd_host_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                          void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev, int64_t B,
                          int64_t H, int64_t S, int64_t D, int causal, float scale, int dtype,
                          int n_chunks, void* stream) {
  if (!q || !k || !v || !o || !lse) return FMHA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FMHA_ERR_INVALID_ARG;
  if (n_chunks < 0 || n_chunks > kMaxChunks) return FMHA_ERR_INVALID_ARG;
  const fmha_status vs = validate(q_dev, k_dev, v_dev, o_dev, lse_dev, B, H, S, D, scale, dtype);
  if (vs != FMHA_OK) return vs;
  const int64_t BH = B * H;
  // one (batch, head) slice of an input, of O and of LSE (V's transposed E4M3
  // slice has the same size as the others)
  const size_t slice = static_cast<size_t>(S * D) * in_bytes(dtype);
  const size_t oslice = static_cast<size_t>(S * D) * kOutBytes, lslice = static_cast<size_t>(S) * 4;
  const size_t in_host = static_cast<size_t>(BH) * slice, o_host = static_cast<size_t>(BH) * oslice;
  if (overlaps(q, in_host, o, o_host) || overlaps(k, in_host, o, o_host) ||
      overlaps(v, in_host, o, o_host) ||
      overlaps(lse, static_cast<size_t>(BH) * lslice, o, o_host))
    return FMHA_ERR_INVALID_ARG;
  const int64_t chunks = std::min<int64_t>(n_chunks == 0 ? kDefaultChunks : n_chunks, BH);

  HostPipe* hp = nullptr;
  const fmha_status ps = host_pipe(&hp);
  if (ps != FMHA_OK) return ps;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  // the copy streams and the second compute stream start after everything
  // already queued on `stream`
  if ((e = cudaEventRecord(hp->entry, st)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hp->h2d, hp->entry, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hp->d2h, hp->entry, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hp->comp, hp->entry, 0)) != cudaSuccess)
    return cuda_fail(e, "stream ordering");
  auto at = [](const void* p, size_t off) {
    return static_cast<void*>(static_cast<char*>(const_cast<void*>(p)) + off);
  };
  // The units that fmha_fwd would key-split on the whole problem (its last
  // ones) are key-split in the chunks that hold them, so that the result is
  // the same bits as fmha_fwd's.
  const int64_t nq = (S + 255) / 256;
  int n_sm = 0;
  if ((e = sm_count(&n_sm)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(multiprocessor count)");
  const int64_t first_split = BH * nq - auto_split_units(BH * nq, S, D, causal, n_sm);
  for (int64_t c = 0; c < chunks; ++c) {
    // chunks alternate between two compute streams, so that one chunk's
    // kernel can start on the SMs that the previous one's last wave leaves
    // idle
    cudaStream_t cs = (c & 1) ? hp->comp : st;
    const int64_t s0 = BH * c / chunks, s1 = BH * (c + 1) / chunks, n = s1 - s0;
    const size_t off = static_cast<size_t>(s0) * slice, bytes = static_cast<size_t>(n) * slice;
    const size_t ooff = static_cast<size_t>(s0) * oslice, obytes = static_cast<size_t>(n) * oslice;
    const size_t loff = static_cast<size_t>(s0) * lslice, lbytes = static_cast<size_t>(n) * lslice;
    if ((e = cudaMemcpyAsync(at(q_dev, off), at(q, off), bytes, cudaMemcpyHostToDevice, hp->h2d)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(at(k_dev, off), at(k, off), bytes, cudaMemcpyHostToDevice, hp->h2d)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(at(v_dev, off), at(v, off), bytes, cudaMemcpyHostToDevice, hp->h2d)) !=
            cudaSuccess ||
        (e = cudaEventRecord(hp->copied[c], hp->h2d)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(cs, hp->copied[c], 0)) != cudaSuccess)
      return cuda_fail(e, "host-to-device copy");
    // one (batch, head) range is a B = 1, H = n problem at offset pointers
    const int64_t split = std::max<int64_t>(0, s1 * nq - std::max(s0 * nq, first_split));
    const fmha_status ks =
        fwd_impl(at(q_dev, off), at(k_dev, off), at(v_dev, off), at(o_dev, ooff),
                 static_cast<float*>(at(lse_dev, loff)), 1, n, S, D, causal, scale, dtype, cs, 0,
                 kDefaultWaitLimitNs, -1.f, split);
    if (ks != FMHA_OK) return ks;
    if ((e = cudaEventRecord(hp->computed[c], cs)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->d2h, hp->computed[c], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(at(o, ooff), at(o_dev, ooff), obytes, cudaMemcpyDeviceToHost, hp->d2h)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(at(lse, loff), at(lse_dev, loff), lbytes, cudaMemcpyDeviceToHost,
                             hp->d2h)) != cudaSuccess)
      return cuda_fail(e, "device-to-host copy");
  }
  // `stream` completes after the last copy back, which follows every chunk's
  // kernel on either compute stream
  if ((e = cudaEventRecord(hp->done, hp->d2h)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(st, hp->done, 0)) != cudaSuccess)
    return cuda_fail(e, "stream ordering");
  return FMHA_OK;
}

// Device scratch of fmha_bwd_host: staged q, k, v, o, d_o, dq, dk, dv, then
// lse, then the backward workspace; every region starts on 256 bytes.
struct BwdHostLayout {
  size_t q, k, v, o, d_o, dq, dk, dv, lse, ws, ws_bytes, total;
};

BwdHostLayout bwd_host_layout(int64_t B, int64_t H, int64_t S, int64_t D) {
  auto up = [](size_t x) { return (x + 255) & ~size_t{255}; };
  const size_t rows = static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(S);
  const size_t tb = up(rows * static_cast<size_t>(D) * 2), lb = up(rows * 4);
  BwdHostLayout L;
  size_t off = 0;
  size_t* tensors[8] = {&L.q, &L.k, &L.v, &L.o, &L.d_o, &L.dq, &L.dk, &L.dv};
  for (size_t* t : tensors) {
    *t = off;
    off += tb;
  }
  L.lse = off;
  off += lb;
  L.ws = off;
  L.ws_bytes = bwd_workspace_bytes(B, H, S, D);
  L.total = off + L.ws_bytes;
  return L;
}

fmha_status bwd_host_impl(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                          void* scratch, size_t scratch_bytes, int64_t B, int64_t H, int64_t S,
                          int64_t D, int causal, float scale, int dtype, int n_chunks,
                          void* stream) {
  if (!q || !k || !v || !o || !lse || !d_o || !dq || !dk || !dv || !scratch)
    return FMHA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FMHA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(scratch) & 255u) return FMHA_ERR_INVALID_ARG;
  if (n_chunks < 0 || n_chunks > kMaxChunks) return FMHA_ERR_INVALID_ARG;
  if (dtype == FMHA_E4M3) return FMHA_ERR_UNSUPPORTED;
  // sizes first, then the layout that depends on them
  const fmha_status sz = validate_sizes(B, H, S, D, scale, dtype);
  if (sz != FMHA_OK) return sz;
  const BwdHostLayout L = bwd_host_layout(B, H, S, D);
  if (scratch_bytes < L.total) return FMHA_ERR_INVALID_ARG;
  char* base = static_cast<char*>(scratch);
  const fmha_status vs = bwd_validate(base + L.q, base + L.k, base + L.v, base + L.o,
                                      reinterpret_cast<float*>(base + L.lse), base + L.d_o,
                                      base + L.dq, base + L.dk, base + L.dv, base + L.ws,
                                      L.ws_bytes, B, H, S, D, scale, dtype);
  if (vs != FMHA_OK) return vs;
  const int64_t BH = B * H;
  // host side: outputs may not overlap the inputs or one another
  const size_t tb = static_cast<size_t>(BH * S * D) * 2, lb = static_cast<size_t>(BH * S) * 4;
  const void* ins[6] = {q, k, v, o, d_o, lse};
  const size_t in_sz[6] = {tb, tb, tb, tb, tb, lb};
  void* outs[3] = {dq, dk, dv};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlaps(outs[i], tb, ins[j], in_sz[j])) return FMHA_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j)
      if (overlaps(outs[i], tb, outs[j], tb)) return FMHA_ERR_INVALID_ARG;
  }
  const int64_t chunks = std::min<int64_t>(n_chunks == 0 ? kDefaultChunks : n_chunks, BH);

  HostPipe* hp = nullptr;
  const fmha_status ps = host_pipe(&hp);
  if (ps != FMHA_OK) return ps;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if ((e = cudaEventRecord(hp->entry, st)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hp->h2d, hp->entry, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hp->d2h, hp->entry, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(hp->comp, hp->entry, 0)) != cudaSuccess)
    return cuda_fail(e, "stream ordering");
  auto at = [](const void* p, size_t off) {
    return static_cast<void*>(static_cast<char*>(const_cast<void*>(p)) + off);
  };
  const size_t slice = static_cast<size_t>(S * D) * 2, lslice = static_cast<size_t>(S) * 4;
  float* dq_acc_all = reinterpret_cast<float*>(base + L.ws);
  float* delta_all = dq_acc_all + static_cast<size_t>(BH * S * D);
  const void* host_in[5] = {q, k, v, o, d_o};
  const size_t dev_in[5] = {L.q, L.k, L.v, L.o, L.d_o};
  void* host_out[3] = {dq, dk, dv};
  const size_t dev_out[3] = {L.dq, L.dk, L.dv};
  for (int64_t c = 0; c < chunks; ++c) {
    // chunks alternate between two compute streams (see fwd_host_impl)
    cudaStream_t cs = (c & 1) ? hp->comp : st;
    const int64_t s0 = BH * c / chunks, s1 = BH * (c + 1) / chunks, n = s1 - s0;
    const size_t off = static_cast<size_t>(s0) * slice, bytes = static_cast<size_t>(n) * slice;
    const size_t loff = static_cast<size_t>(s0) * lslice, lbytes = static_cast<size_t>(n) * lslice;
    for (int i = 0; i < 5; ++i)
      if ((e = cudaMemcpyAsync(base + dev_in[i] + off, at(host_in[i], off), bytes,
                               cudaMemcpyHostToDevice, hp->h2d)) != cudaSuccess)
        return cuda_fail(e, "host-to-device copy");
    if ((e = cudaMemcpyAsync(base + L.lse + loff, at(lse, loff), lbytes, cudaMemcpyHostToDevice,
                             hp->h2d)) != cudaSuccess ||
        (e = cudaEventRecord(hp->copied[c], hp->h2d)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(cs, hp->copied[c], 0)) != cudaSuccess)
      return cuda_fail(e, "host-to-device copy");
    // slices [s0, s1) are a B = 1, H = n problem at offset pointers, with
    // their own part of the dQ accumulator and of delta
    const fmha_status ks = bwd_enqueue(
        base + L.q + off, base + L.k + off, base + L.v + off, base + L.o + off,
        reinterpret_cast<const float*>(base + L.lse + loff), base + L.d_o + off,
        base + L.dq + off, base + L.dk + off, base + L.dv + off,
        dq_acc_all + static_cast<size_t>(s0 * S * D), delta_all + static_cast<size_t>(s0 * S), n,
        S, D, causal, scale, dtype, cs, kDefaultWaitLimitNs);
    if (ks != FMHA_OK) return ks;
    if ((e = cudaEventRecord(hp->computed[c], cs)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->d2h, hp->computed[c], 0)) != cudaSuccess)
      return cuda_fail(e, "stream ordering");
    for (int i = 0; i < 3; ++i)
      if ((e = cudaMemcpyAsync(at(host_out[i], off), base + dev_out[i] + off, bytes,
                               cudaMemcpyDeviceToHost, hp->d2h)) != cudaSuccess)
        return cuda_fail(e, "device-to-host copy");
  }
  if ((e = cudaEventRecord(hp->done, hp->d2h)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(st, hp->done, 0)) != cudaSuccess)
    return cuda_fail(e, "stream ordering");
  return FMHA_OK;
}

}  // namespace

extern "C" {

fmha_status fmha_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                     int64_t H, int64_t S, int64_t D, int causal, float scale, fmha_dtype dtype,
                     void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, S, D, causal, scale, static_cast<int>(dtype), stream, 0,
                  kDefaultWaitLimitNs);
}

fmha_status fmha_fwd_testing(const void* q, const void* k, const void* v, void* o, float* lse,
                             int64_t B, int64_t H, int64_t S, int64_t D, int causal, float scale,
                             fmha_dtype dtype, void* stream, int inject_fault,
                             double wait_limit_s, float tau) {
  if (inject_fault < 0 || inject_fault > 1) return FMHA_ERR_INVALID_ARG;
  if (!(wait_limit_s > 0.0) || wait_limit_s > 60.0) return FMHA_ERR_INVALID_ARG;
  if (!(tau >= 0.f && tau <= (dtype == FMHA_E4M3 ? 8.f : 15.f))) return FMHA_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H, S, D, causal, scale, static_cast<int>(dtype), stream,
                  inject_fault, static_cast<uint64_t>(wait_limit_s * 1e9), tau);
}

int64_t fmha_fwd_split_policy(int64_t B, int64_t H, int64_t S, int64_t D, int causal, int n_sm) {
  if (n_sm < 1 || validate_sizes(B, H, S, D, 1.f, FMHA_F16) != FMHA_OK) return -1;
  return auto_split_units(((S + 255) / 256) * B * H, S, D, causal, n_sm);
}

fmha_status fmha_fwd_split_testing(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                                   int causal, float scale, fmha_dtype dtype, void* stream,
                                   int64_t split_units) {
  if (split_units < -1) return FMHA_ERR_INVALID_ARG;
  if (split_units > 0) {
    const fmha_status vs = validate_sizes(B, H, S, D, scale, static_cast<int>(dtype));
    if (vs != FMHA_OK) return vs;
    if (!key_split_allowed(S, D, causal)) return FMHA_ERR_UNSUPPORTED;
    if (split_units > ((S + 255) / 256) * B * H) return FMHA_ERR_INVALID_ARG;
  }
  return fwd_impl(q, k, v, o, lse, B, H, S, D, causal, scale, static_cast<int>(dtype), stream, 0,
                  kDefaultWaitLimitNs, -1.f, split_units);
}

fmha_status fmha_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                          void* q_dev, void* k_dev, void* v_dev, void* o_dev, float* lse_dev,
                          int64_t B, int64_t H, int64_t S, int64_t D, int causal, float scale,
                          fmha_dtype dtype, int n_chunks, void* stream) {
  return fwd_host_impl(q, k, v, o, lse, q_dev, k_dev, v_dev, o_dev, lse_dev, B, H, S, D, causal, scale,
                       static_cast<int>(dtype), n_chunks, stream);
}

size_t fmha_bwd_host_scratch_bytes(int64_t B, int64_t H, int64_t S, int64_t D) {
  if (B < 1 || H < 1 || S < 1 || D < 1) return 0;
  return bwd_host_layout(B, H, S, D).total;
}

fmha_status fmha_bwd_host(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                          void* scratch, size_t scratch_bytes, int64_t B, int64_t H, int64_t S,
                          int64_t D, int causal, float scale, fmha_dtype dtype, int n_chunks,
                          void* stream) {
  return bwd_host_impl(q, k, v, o, lse, d_o, dq, dk, dv, scratch, scratch_bytes, B, H, S, D,
                       causal, scale, static_cast<int>(dtype), n_chunks, stream);
}

size_t fmha_bwd_workspace_bytes(int64_t B, int64_t H, int64_t S, int64_t D) {
  if (B < 1 || H < 1 || S < 1 || D < 1) return 0;
  return bwd_workspace_bytes(B, H, S, D);
}

fmha_status fmha_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* d_o, void* dq, void* dk, void* dv, void* workspace,
                     size_t workspace_bytes, int64_t B, int64_t H, int64_t S, int64_t D,
                     int causal, float scale, fmha_dtype dtype, void* stream) {
  return bwd_impl(q, k, v, o, lse, d_o, dq, dk, dv, workspace, workspace_bytes, B, H, S, D,
                  causal, scale, static_cast<int>(dtype), stream, kDefaultWaitLimitNs);
}

fmha_status fmha_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                             int64_t B, int64_t H, int64_t S, int64_t D, int causal, float scale,
                             fmha_dtype dtype, void* stream) {
  // host checks first (no CUDA call): the arguments as fmha_bwd takes them,
  // then the capacity of the static scratch, B*H*S rows of (4D + 4) bytes
  // (B*H < 2^31 and S < 2^31 once validated, so the product fits in 64 bits)
  const fmha_status vs = validate(q, k, v, const_cast<void*>(o), const_cast<float*>(lse), B, H,
                                  S, D, scale, static_cast<int>(dtype));
  if (vs != FMHA_OK) return vs;
  if (dtype == FMHA_E4M3) return FMHA_ERR_UNSUPPORTED;
  const int64_t cap_rows = static_cast<int64_t>(wsa::kBwdStaticScratchBytes / (4 * D + 4));
  if (B * H * S > cap_rows) return FMHA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const cudaError_t e = wsa::bwd_static_scratch(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(backward scratch)");
  return bwd_impl(q, k, v, o, lse, d_o, dq, dk, dv, scratch, wsa::kBwdStaticScratchBytes, B, H,
                  S, D, causal, scale, static_cast<int>(dtype), stream, kDefaultWaitLimitNs);
}

fmha_status fmha_get_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_wsa_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "read device status");
  if (word != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_wsa_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear device status");
    return FMHA_ERR_TIMEOUT;
  }
  return FMHA_OK;
}

const char* fmha_status_str(fmha_status s) {
  switch (s) {
    case FMHA_OK: return "ok";
    case FMHA_ERR_INVALID_ARG: return "invalid argument";
    case FMHA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FMHA_ERR_CUDA: return "CUDA error";
    case FMHA_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* fmha_last_cuda_error(void) { return t_last_cuda_error; }

int fmha_version(void) { return (0 << 16) | (1 << 8) | 0; }

}  // extern "C"
