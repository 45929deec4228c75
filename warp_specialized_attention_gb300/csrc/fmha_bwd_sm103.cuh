// fmha_bwd_sm103.cuh -- the tensor-core forms of the attention backward pass
// that the forward kernel does not use.
//
// With the keys of a 128-key block on the TMEM lanes, the backward pass needs
// five products per 128-row query block.  Three of them have forward forms:
//   S^T  = K Q^T      (issue_qk: both operands K-major)
//   dP^T = V dO^T     (issue_qk)
//   dV  += P^T dO     (issue_dv: the forward's P V form, with P^T from TMEM in
//                     two 32-column groups, dO MN-major)
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
#include <type_traits>

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

// dV += P^T dO with P^T from TMEM (TMEM-A form, dO MN-major), the P^T of
// queries 0-63 at columns [0, 32) and of queries 64-127 at [64, 96): each half
// is written by its own warps over S^T columns that only those warps read.
template <int D, int ET>
__device__ __forceinline__ void issue_dv(uint32_t d_tmem, uint32_t p_tmem, uint32_t do_lo,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_f16(ET == kBF16, 128, D, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts_warp(d_tmem, p_tmem + kk * 8 + (kk >= 4 ? 32 : 0),
                sdesc_join(do_lo + kk * ((16 * 128) >> 4), kDescHi), idesc,
                (accumulate || kk > 0) ? 1u : 0u);
}

// ============================================================================ the kernel
//
// Attention backward for one (head, 128-key block) per block of 640 threads:
//   warps 0-7  dS / P: key row 32(w % 4) + lane, query columns 64(w / 4) ..
//              +63 (two warps per SM sub-partition split the block's
//              columns); read S^T and dP^T from TMEM, write P^T (16-bit) over
//              S^T in TMEM and dS^T to shared memory; at the end write dV
//              (w < 4) or dK (w >= 4)
//   warps 8-15 dQ: query row 32(w % 4) + lane, columns D/2 (w - 8) / 4 ..
//              +D/2; read each block's dQ part from TMEM into registers,
//              release the columns, then pass it, scaled, through a 2 KB
//              shared stage to a TMA reduce-add into the fp32 accumulator in
//              global memory (several key blocks add into one row)
//   warp 16    TMEM allocation and the tcgen05.mma issuer
//   warp 17    TMA producer: K, V once; Q, dO per query block; LSE and delta
//   warps 18-19 idle (they complete the producer warpgroup for setmaxnreg)
// Per query block the issuer runs S^T = K Q^T, dP^T = V dO^T, then (once P^T
// and dS^T are in place) dV += P^T dO, dK += dS^T Q and dQ = dS K.  Each
// half of the compute warps writes its P^T over S^T columns only it reads
// (queries 0-63 to columns 0-31, 64-127 to 64-95; issue_dv reads them there).  The
// chain-rule arithmetic is that of the backward oracle:
//   P = exp(scale q.k - LSE), dS = P (dP - delta), delta_i = dO_i . O_i,
//   dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K.
// Synchronisation is the same empty/full mbarrier scheme as the forward (Tawa,
// Section III-B/III-E); every wait is bounded and raises the abort flag.

constexpr float kLog2e = 1.4426950408889634f;
// 20 warps (five whole warpgroups; warps 18 and 19 idle) launched at 96
// registers (61,440 in all).  Register split: the P/dS warpgroups raise their
// limit to 128, the dQ warpgroups lower theirs to 80 and the producer
// warpgroup (MMA, TMA, two idle warps) to 64: 256 x 128 + 256 x 80 + 128 x 64
// = 61,440, exactly the launch's registers.
constexpr int kBwdThreads = 640;
constexpr int kBwdRegLaunch = 96, kBwdRegCompute = 128, kBwdRegDq = 80, kBwdRegProducer = 64;
static_assert(256 * kBwdRegCompute + 256 * kBwdRegDq + 128 * kBwdRegProducer ==
                  kBwdThreads * kBwdRegLaunch,
              "register split");
constexpr int kBwdComputeWarps = 8;  // warps 0-7
constexpr int kBwdDqWarps = 8;       // warps 8-15
constexpr int kBwdWarpMma = 16;
constexpr int kBwdWarpLoad = 17;

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kTile = 128 * D * 2;                // 128 rows x D, 16-bit
  // K, V, two Q buffers, dO, dS^T
  static constexpr int kOffK = 0, kOffV = kTile, kOffQ = 2 * kTile, kOffDO = 4 * kTile;
  static constexpr int kOffDS = 5 * kTile;                 // dS^T, 128 x 128 16-bit
  // dQ stages: one 2 KB tile (32 rows x 16 fp32, 64-byte swizzle) per dQ warp
  static constexpr int kOffDQ = kOffDS + 128 * 128 * 2;
  static constexpr int kDqStage = 32 * 16 * 4;
  static constexpr int kOffStat = kOffDQ + kBwdDqWarps * kDqStage;  // 2 x (LSE*log2e, delta)
  static constexpr int kOffCtl = kOffStat + 2 * 256 * 4;
  static constexpr int kSmemBytes = 1024 + kOffCtl + 256;
  // TMEM columns: S^T (16-bit P^T over columns 0-31 and 64-95 of it), dP^T
  // (dQ reuses it), dV, dK
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 128;
  static constexpr uint32_t kColDV = 256, kColDK = 256 + D;
};

struct BwdCtl {
  uint64_t kv_full;
  uint64_t q_full[2], q_free[2], do_full, do_free;
  uint64_t stat_full[2], stat_free[2];
  uint64_t sd_full;   // S^T and dP^T are in TMEM
  uint64_t p_ready;   // P^T in TMEM and dS^T in shared memory
  uint64_t ds_free;   // the dS^T tile has been read (dK and dQ done)
  uint64_t dq_full, dq_free;
  uint64_t acc_done;  // every MMA of the block is complete
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BwdCtl) <= 256, "control block size");

struct BwdParams {
  const float* lse;    // (B,H,S) natural log-sum-exp of the forward
  const float* delta;  // (B,H,S) dO . O per row
  float* dq_accum;     // (B,H,S,D) fp32, zero before the launch
  void* dk;            // (B,H,S,D) 16-bit
  void* dv;
  int* status;
  int S;
  int n_blk;           // ceil(S / 128)
  float scale;
  float scale_log2;    // scale * log2(e)
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// tcgen05.ld 32 lanes x 32 bits, 16 columns, no wait.
__device__ __forceinline__ void tmem_ld_x16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// tcgen05.wait::ld tied to the 16 destination registers of an async load.
__device__ __forceinline__ void tmem_ld_wait_x16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

template <int D, int ET, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fmha_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  static_assert(ET != kE4M3, "backward: 16-bit inputs");
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  BwdCtl& ctl = *reinterpret_cast<BwdCtl*>(smem + C::kOffCtl);
  float* stats = reinterpret_cast<float*>(smem + C::kOffStat);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.S;
  const int bh = blockIdx.x / p.n_blk;
  const int kb = blockIdx.x - bh * p.n_blk;
  const int qb0 = CAUSAL ? kb : 0;       // query blocks that see this key block
  const int nq = p.n_blk - qb0;          // >= 1
  // The n-th query block of this key block.  Without the mask every key block
  // starts at its own index and wraps around, so that the blocks of a head
  // running side by side add into different dQ rows (with the mask key block
  // kb starts at query block kb, which already spreads them).
  auto qblock = [&](int n) {
    int qb = qb0 + n;
    if (!CAUSAL) {
      qb += kb;
      if (qb >= p.n_blk) qb -= p.n_blk;
    }
    return qb;
  };

  if (threadIdx.x == 0) {
    mbar_init(&ctl.kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.q_full[i], 1);
      mbar_init(&ctl.q_free[i], 1);
    }
    mbar_init(&ctl.do_full, 1);
    mbar_init(&ctl.do_free, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.stat_full[i], 1);
      mbar_init(&ctl.stat_free[i], kBwdComputeWarps);
    }
    mbar_init(&ctl.sd_full, 1);
    mbar_init(&ctl.p_ready, kBwdComputeWarps);
    mbar_init(&ctl.ds_free, 1);
    mbar_init(&ctl.dq_full, 1);
    mbar_init(&ctl.dq_free, kBwdDqWarps);
    mbar_init(&ctl.acc_done, 1);
    mbar_init(&ctl.mma_drain, 1);
    ctl.abort = 0;
    fence_barrier_init();
  }
  if (warp == kBwdWarpMma) {
    tmem_alloc(&ctl.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort;
  const uint32_t sK = sbase + C::kOffK, sV = sbase + C::kOffV, sQ = sbase + C::kOffQ;
  const uint32_t sDO = sbase + C::kOffDO, sDS = sbase + C::kOffDS;
  auto wait = [&](uint64_t* bar, uint32_t parity, int code) {
    bool good = mbar_wait(bar, parity, abort_flag, p.status, code, p.wait_limit_ns);
    return __all_sync(0xffffffffu, good);
  };

  if (warp == kBwdWarpLoad) {
    // ================================================================ TMA producer
    setmaxnreg_dec<kBwdRegProducer>();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_do);
    const uint64_t pol_kv = policy_evict_first(), pol_q = policy_evict_last();
    mbar_arrive_expect_tx_warp(&ctl.kv_full, 2 * C::kTile);
    for (int cb = 0; cb < D / 64; ++cb) {
      tma_load_3d_warp(sK + cb * (128 * 128), &tm_k, &ctl.kv_full, cb * 64, kb * 128, bh, pol_kv);
      tma_load_3d_warp(sV + cb * (128 * 128), &tm_v, &ctl.kv_full, cb * 64, kb * 128, bh, pol_kv);
    }
    int nq_loads = 0, ndo_loads = 0;  // Q and dO tiles issued
    for (int n = 0; n < nq; ++n) {
      const int qb = qblock(n);
      // Q: two buffers, so the next block's Q loads while this one computes
      const int qbuf = n & 1;
      if (n >= 2 && !wait(&ctl.q_free[qbuf], ((n >> 1) - 1) & 1, kStatusTimeoutLoad)) break;
      mbar_arrive_expect_tx_warp(&ctl.q_full[qbuf], C::kTile);
      for (int cb = 0; cb < D / 64; ++cb)
        tma_load_3d_warp(sQ + qbuf * C::kTile + cb * (128 * 128), &tm_q, &ctl.q_full[qbuf],
                         cb * 64, qb * 128, bh, pol_q);
      ++nq_loads;
      if (n >= 1 && !wait(&ctl.do_free, (n - 1) & 1, kStatusTimeoutLoad)) break;
      mbar_arrive_expect_tx_warp(&ctl.do_full, C::kTile);
      for (int cb = 0; cb < D / 64; ++cb)
        tma_load_3d_warp(sDO + cb * (128 * 128), &tm_do, &ctl.do_full, cb * 64, qb * 128, bh,
                         pol_q);
      ++ndo_loads;
      // this block's -LSE (in log2 units) and -delta, negated so that the
      // compute warps add them; rows past S: P = 0
      const int buf = n & 1;
      if (n >= 2 && !wait(&ctl.stat_free[buf], ((n >> 1) - 1) & 1, kStatusTimeoutLoad)) break;
      float* st = stats + buf * 256;
      for (int r = lane; r < 128; r += 32) {
        const int q = qb * 128 + r;
        const size_t idx = static_cast<size_t>(bh) * S + q;
        st[r] = q < S ? -(p.lse[idx] * kLog2e) : -INFINITY;
        st[128 + r] = q < S ? -p.delta[idx] : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.stat_full[buf]);
    }
    // Drain: every issued copy lands before the block may exit.
    mbar_wait(&ctl.kv_full, 0, nullptr, p.status, kStatusTimeoutDrain, p.wait_limit_ns);
    for (int b = 0; b < 2; ++b) {  // loads into buffer b: n = b, b + 2, ...
      const int nb = (nq_loads + 1 - b) >> 1;
      if (nb > 0)
        mbar_wait(&ctl.q_full[b], (nb - 1) & 1, nullptr, p.status, kStatusTimeoutDrain,
                  p.wait_limit_ns);
    }
    if (ndo_loads > 0)
      mbar_wait(&ctl.do_full, (ndo_loads - 1) & 1, nullptr, p.status, kStatusTimeoutDrain,
                p.wait_limit_ns);
    __syncwarp();
  } else if (warp == kBwdWarpMma) {
    // ================================================================ MMA issuer
    setmaxnreg_dec<kBwdRegProducer>();
    const uint32_t k_lo = sdesc_lo(sK, kLboKMajor), v_lo = sdesc_lo(sV, kLboKMajor);
    const uint32_t do_lo = sdesc_lo(sDO, kLboKMajor);
    const uint32_t k_mn = sdesc_lo(sK, kLboV);
    const uint32_t do_mn = sdesc_lo(sDO, kLboV);
    const uint32_t ds_k = sdesc_lo(sDS, kLboKMajor), ds_mn = sdesc_lo(sDS, kLboV);
    bool ok = wait(&ctl.kv_full, 0, kStatusTimeoutMma);
    for (int n = 0; ok && n < nq; ++n) {
      const int qbuf = n & 1;
      const uint32_t q_lo = sdesc_lo(sQ + qbuf * C::kTile, kLboKMajor);
      const uint32_t q_mn = sdesc_lo(sQ + qbuf * C::kTile, kLboV);
      if (!(ok = wait(&ctl.q_full[qbuf], (n >> 1) & 1, kStatusTimeoutMma))) break;
      tc_fence_after();
      issue_qk<D, ET>(tmem + C::kColS, k_lo, q_lo);  // S^T = K Q^T
      // dP^T needs this block's dO (one buffer, loaded once dV of the previous
      // block has read it: S^T runs meanwhile) and takes the columns of the
      // previous block's dQ part
      ok = wait(&ctl.do_full, n & 1, kStatusTimeoutMma) &&
           (n == 0 || wait(&ctl.dq_free, (n - 1) & 1, kStatusTimeoutMma));
      if (!ok) break;
      tc_fence_after();
      issue_qk<D, ET>(tmem + C::kColDP, v_lo, do_lo);  // dP^T = V dO^T
      mma_commit_warp(&ctl.sd_full);
      if (!(ok = wait(&ctl.p_ready, n & 1, kStatusTimeoutMma))) break;
      tc_fence_after();
      issue_dv<D, ET>(tmem + C::kColDV, tmem + C::kColS, do_mn, n > 0);  // dV += P^T dO
      mma_commit_warp(&ctl.do_free);
      issue_kmaj_mn<D, ET>(tmem + C::kColDK, ds_k, q_mn, n > 0);        // dK += dS^T Q
      mma_commit_warp(&ctl.q_free[qbuf]);
      issue_mn_mn<D, ET>(tmem + C::kColDQ, ds_mn, k_mn, false);         // dQ part = dS K
      mma_commit_warp(&ctl.dq_full);
      mma_commit_warp(&ctl.ds_free);
    }
    mma_commit_warp(&ctl.acc_done);
    mma_commit_warp(&ctl.mma_drain);
    mbar_wait(&ctl.mma_drain, 0, nullptr, p.status, kStatusTimeoutDrain, p.wait_limit_ns);
    __syncwarp();
  } else if (warp < kBwdComputeWarps) {
    // ================================================================ P and dS (key rows)
    setmaxnreg_inc<kBwdRegCompute>();
    const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant, column half
    const int r = quad * 32 + lane;               // key row in the block, TMEM lane
    const int key = kb * 128 + r;
    const bool key_ok = key < S;
    const bool key_ok_warp = __all_sync(0xffffffffu, key_ok);
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const float cl2 = p.scale_log2;
    bool ok = true;
    for (int n = 0; ok && n < nq; ++n) {
      const int qb = qblock(n);
      const int buf = n & 1;
      ok = wait(&ctl.stat_full[buf], (n >> 1) & 1, kStatusTimeoutSoftmax) &&
           wait(&ctl.sd_full, n & 1, kStatusTimeoutSoftmax) &&
           (n == 0 || wait(&ctl.ds_free, (n - 1) & 1, kStatusTimeoutSoftmax));
      if (!ok) break;
      tc_fence_after();
      const float* nlse2 = stats + buf * 256;  // -LSE log2(e) per query
      const float* ndl = nlse2 + 128;          // -delta per query
      const bool diag = CAUSAL && qb == kb;
      // no key of any row of this warp is masked: the warp takes the packed
      // path (warp-uniform, the tcgen05 loads and stores are warp-wide)
      const bool plain = key_ok_warp && !diag;
      // four chunks of 16 queries, in one of two instantiations (masked or
      // not) so that each keeps its registers to itself
      auto run_chunks = [&](auto kind) {
        // four chunks of 16 queries; chunk i + 1's S^T and dP^T loads are in
        // flight while chunk i is computed (two register buffers, unrolled so
        // that the buffers are indexed statically)
        uint32_t sv[2][16], dpv[2][16];
        tmem_ld_x16_async(lane_base + C::kColS + half * 64, sv[0]);
        tmem_ld_x16_async(lane_base + C::kColDP + half * 64, dpv[0]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = 4 * half + i;
          const int cur = i & 1;
          tmem_ld_wait_x16(sv[cur]);
          tmem_ld_wait_x16(dpv[cur]);
          if (i < 3) {
            tmem_ld_x16_async(lane_base + C::kColS + (c + 1) * 16, sv[cur ^ 1]);
            tmem_ld_x16_async(lane_base + C::kColDP + (c + 1) * 16, dpv[cur ^ 1]);
          }
          uint32_t pk[8], dk16[8];
          const uint32_t* sc = sv[cur];
          const uint32_t* dpc = dpv[cur];
          if constexpr (decltype(kind)::value) {
            // P = 2^(s c - LSE log2 e) and dS = P (dP - delta), two queries per
            // packed fp32x2 instruction; the same roundings as the masked path
            const uint64_t c2 = f2_pack(cl2, cl2);
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
              // the four queries' statistics: one vector load each (broadcast)
              const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + c * 16 + e);
              const float4 d4 = *reinterpret_cast<const float4*>(ndl + c * 16 + e);
              float x[4];
              f2_unpack(ffma2(f2_pack(__uint_as_float(sc[e]), __uint_as_float(sc[e + 1])), c2,
                              f2_pack(l4.x, l4.y)), x[0], x[1]);
              f2_unpack(ffma2(f2_pack(__uint_as_float(sc[e + 2]), __uint_as_float(sc[e + 3])), c2,
                              f2_pack(l4.z, l4.w)), x[2], x[3]);
              float pp[4];
#pragma unroll
              for (int h = 0; h < 4; ++h) pp[h] = ex2(x[h]);
              const uint64_t dd01 = fmul2(f2_pack(pp[0], pp[1]),
                                          fadd2(f2_pack(__uint_as_float(dpc[e]),
                                                        __uint_as_float(dpc[e + 1])),
                                                f2_pack(d4.x, d4.y)));
              const uint64_t dd23 = fmul2(f2_pack(pp[2], pp[3]),
                                          fadd2(f2_pack(__uint_as_float(dpc[e + 2]),
                                                        __uint_as_float(dpc[e + 3])),
                                                f2_pack(d4.z, d4.w)));
              float dd[4];
              f2_unpack(dd01, dd[0], dd[1]);
              f2_unpack(dd23, dd[2], dd[3]);
              pk[e >> 1] = pack2<ET == kBF16>(pp[0], pp[1]);
              pk[(e >> 1) + 1] = pack2<ET == kBF16>(pp[2], pp[3]);
              dk16[e >> 1] = pack2<ET == kBF16>(dd[0], dd[1]);
              dk16[(e >> 1) + 1] = pack2<ET == kBF16>(dd[2], dd[3]);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + c * 16 + e);
              const float4 d4 = *reinterpret_cast<const float4*>(ndl + c * 16 + e);
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv4[4] = {d4.x, d4.y, d4.z, d4.w};
              float pp[4], dd[4];
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const int qi = c * 16 + e + h;
                const bool vis = key_ok && !(diag && r > qi);
                const float pv = vis ? ex2(fmaf(__uint_as_float(sc[e + h]), cl2, lv[h])) : 0.f;
                pp[h] = pv;
                dd[h] = pv * (__uint_as_float(dpc[e + h]) + dv4[h]);
              }
              pk[e >> 1] = pack2<ET == kBF16>(pp[0], pp[1]);
              pk[(e >> 1) + 1] = pack2<ET == kBF16>(pp[2], pp[3]);
              dk16[e >> 1] = pack2<ET == kBF16>(dd[0], dd[1]);
              dk16[(e >> 1) + 1] = pack2<ET == kBF16>(dd[2], dd[3]);
            }
          }
          // P^T over S^T columns this warp has read: queries 16c.. at column
          // 8c (first half) or 8c + 32 (second half, see issue_dv); below the
          // columns of the load in flight (16c + 16 and up)
          tmem_st_x8_async(lane_base + C::kColS + c * 8 + half * 32, pk);
          // dS^T row r, queries 16c..16c+15: two 16-byte units of the
          // 128-byte-swizzled tile (unit index XOR row % 8)
          const uint32_t cb = c >> 2, u0 = (c & 3) * 2;
          const uint32_t row_addr = sDS + cb * (128 * 128) + r * 128;
          const uint32_t a0 = row_addr + ((u0 ^ (r & 7)) << 4);
          const uint32_t a1 = row_addr + (((u0 + 1) ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "r"(dk16[0]),
                       "r"(dk16[1]), "r"(dk16[2]), "r"(dk16[3])
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a1), "r"(dk16[4]),
                       "r"(dk16[5]), "r"(dk16[6]), "r"(dk16[7])
                       : "memory");
        }
      };
      if (plain)
        run_chunks(std::true_type{});
      else
        run_chunks(std::false_type{});
      tmem_st_wait();
      fence_proxy_async_smem();  // dS^T stores -> visible to the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl.p_ready);
        mbar_arrive(&ctl.stat_free[buf]);
      }
    }
    // ---- epilogue: dV and dK (x scale) in the storage dtype
    if (ok) {
      ok = wait(&ctl.acc_done, 0, kStatusTimeoutSoftmax);
    }
    if (ok) {
      tc_fence_after();
      const size_t row_off = (static_cast<size_t>(bh) * S + (key_ok ? key : 0)) * D * 2;
#pragma unroll 1
      for (int t = half; t < half + 1; ++t) {  // dV from the first half, dK from the second
        uint8_t* out = reinterpret_cast<uint8_t*>(t ? p.dk : p.dv) + row_off;
        const float mul = t ? p.scale : 1.f;
        const uint32_t col = t ? C::kColDK : C::kColDV;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t orr[32];
          tmem_ld_x32(lane_base + col + ch * 32, orr);
          uint32_t pkd[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkd[i] = pack2<ET == kBF16>(__uint_as_float(orr[2 * i]) * mul,
                                        __uint_as_float(orr[2 * i + 1]) * mul);
          if (key_ok) {
            uint4* dst = reinterpret_cast<uint4*>(out + ch * 64);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
          }
        }
      }
    }
  } else if (warp < kBwdComputeWarps + kBwdDqWarps) {
    // ================================================================ dQ (query rows)
    setmaxnreg_dec<kBwdRegDq>();
    constexpr int kCols = D / 2;  // columns of this warp
    const int quad = warp & 3, hc = (warp - kBwdComputeWarps) >> 2;
    const uint32_t t_dq = tmem + (static_cast<uint32_t>(quad * 32) << 16) + C::kColDQ + hc * kCols;
    const uint32_t stage = sbase + C::kOffDQ + (warp - kBwdComputeWarps) * C::kDqStage;
    if (lane == 0) prefetch_tmap(&tm_dq);
    bool ok = true;
    for (int n = 0; ok && n < nq; ++n) {
      if (!(ok = wait(&ctl.dq_full, n & 1, kStatusTimeoutSoftmax))) break;
      tc_fence_after();
      uint32_t r[kCols / 32][32];
#pragma unroll
      for (int ch = 0; ch < kCols / 32; ++ch) tmem_ld_x32_async(t_dq + ch * 32, r[ch]);
#pragma unroll
      for (int ch = 0; ch < kCols / 32; ++ch) tmem_ld_wait_x32(r[ch]);
      // the columns are free for the next block's dP^T
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.dq_free);
      // row q0 + lane of the box: 16 columns per stage, four 16-byte units at
      // unit index XOR (row / 2) % 4 (the 64-byte swizzle)
      // rows past S inside a box are skipped by the copy; boxes wholly past S
      // are not issued
      const int q0 = qblock(n) * 128 + quad * 32;
      if (q0 >= S) continue;
#pragma unroll
      for (int sg = 0; sg < kCols / 16; ++sg) {
        if (lane == 0) bulk_wait_group_read0();  // the stage's previous tile is read
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t a = stage + lane * 64 + ((u ^ ((lane >> 1) & 3)) << 4);
          const uint32_t* f = &r[sg >> 1][(sg & 1) * 16 + 4 * u];
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                       "f"(__uint_as_float(f[0]) * p.scale), "f"(__uint_as_float(f[1]) * p.scale),
                       "f"(__uint_as_float(f[2]) * p.scale), "f"(__uint_as_float(f[3]) * p.scale)
                       : "memory");
        }
        fence_proxy_async_smem();  // the stores -> visible to the bulk copy
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dq, stage, hc * kCols + sg * 16, q0, bh);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group0();  // every reduction has landed
    __syncwarp();
  } else {
    // warps 18 and 19: no role, but every warp of the producer warpgroup takes
    // part in its register release
    setmaxnreg_dec<kBwdRegProducer>();
  }

  // ---- teardown: every role has drained its asynchronous work
  tc_fence_before();
  __syncthreads();
  if (warp == kBwdWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// delta_i = dO_i . O_i in fp32, one warp per row.
template <int D, int ET>
__global__ void __launch_bounds__(256) fmha_bwd_delta_kernel(const void* o, const void* d_o,
                                                             float* delta, int64_t rows) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint32_t* po = reinterpret_cast<const uint32_t*>(o) + row * (D / 2);
  const uint32_t* pd = reinterpret_cast<const uint32_t*>(d_o) + row * (D / 2);
  float acc = 0.f;
#pragma unroll
  for (int i = lane; i < D / 2; i += 32) {
    float a0, a1, b0, b1;
    unpack2<ET == kBF16>(po[i], a0, a1);
    unpack2<ET == kBF16>(pd[i], b0, b1);
    acc = fmaf(a0, b0, fmaf(a1, b1, acc));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) delta[row] = acc;
}

// dq (16-bit) = dq_accum (fp32), four elements per thread.
template <int ET>
__global__ void __launch_bounds__(256) fmha_bwd_dq_kernel(const float* acc, void* dq, int64_t n) {
  const int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (i >= n) return;
  const float4 a = *reinterpret_cast<const float4*>(acc + i);
  uint2 out;
  out.x = pack2<ET == kBF16>(a.x, a.y);
  out.y = pack2<ET == kBF16>(a.z, a.w);
  *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(dq) + i) = out;
}

}  // namespace wsa
