// fmha_fwd_sm103.cuh -- warp-specialized fused attention forward for sm_103a.
//
// One CTA computes 2 query tiles of 128 rows (256 rows) of one (batch, head)
// and streams that head's keys/values in blocks of 128.  Per key block j and
// query tile t the pages' three stages run on three kinds of unit:
//   T : S_t = Q_t K_j^T        tcgen05.mma (SMEM x SMEM -> TMEM, fp32)
//   C : P_t = exp2(S_t*c - m)  CUDA cores + SFU, one softmax warpgroup per tile
//   U : O_t += P_t V_j         tcgen05.mma (TMEM x SMEM -> TMEM, fp32)
// ("Tawa: Automatic Warp Specialization for Modern GPUs with Asynchronous
// References", Section III-D, Algorithm 1: T_j is issued while C_{j-1} and
// U_{j-1} are in flight).  With two query tiles the single tensor-core issuer
// alternates between them, so one tile's softmax overlaps the other tile's
// MMAs -- the two-consumer ping-pong that "Optimal Software Pipelining and Warp
// Specialization for Tensor Core GPUs" rediscovers for Hopper and Blackwell
// (Section 6.2, Figs. 7-8), built here on Tensor Memory instead of registers.
//
// Warp roles (one CTA per SM; 384 threads, except 352 for full attention at
// head dim 64):
//   warps 0-3  softmax + epilogue, query tile 0 (TMEM lanes 0-127)
//   warps 4-7  softmax + epilogue, query tile 1
//   warp  8    TMEM allocator and the tcgen05.mma issuer (of tile 0 at D = 64)
//   warp  9    TMA producer and scheduler: per work unit Q, then K_j / V_j
//              through an SMEM ring
//   warp  10   the tcgen05.mma issuer of tile 1 at D = 64, else idle
//   warp  11   idle
// The two idle warps complete the third warpgroup, so that warps 8-11 can hand
// registers to the softmax warpgroups with setmaxnreg (the register split in
// Cfg).
// The variable-latency TMA loads sit on their own warp and nothing blocking
// shares a warp with the MMA issuer (the warp-specialization rules of the Twill
// page, "core method": variable-latency ops on a dedicated warp, no blocking
// wait beside interruptible ops).
//
// Persistent scheduling.  The grid has one block per work unit (head, 256-row
// query block), but a running block takes further units itself: while it
// streams one unit, its producer warp asks the hardware (cluster launch
// control) to cancel a not-yet-started block and adopts that block's unit.
// So each SM runs one block that moves from unit to unit, the next unit's K/V
// and Q loads overlap the current unit's last blocks and epilogue, and the
// order in which units start is the block-index order, which decode_unit()
// makes longest-first for causal masks.  (Tawa, Section IV-B and Fig. 7(b):
// resident blocks that iterate over tiles, removing relaunch cost and
// overlapping loads, tensor-core work and epilogue; the wave count that a
// one-block-per-tile grid is quantised to is the W of "A Performance Model for
// Warp Specialization Kernels", core formulas.)  No global counter is involved, so a launch needs no
// memory beyond its outputs.  The unit travels from the producer to the other
// roles through a two-slot channel (unit_full / unit_empty); Q tiles are
// reloaded once the previous unit's last Q K^T is done (q_full / q_empty) and
// O_t is overwritten only after the previous epilogue read it (o_empty).
//
// Key-split units.  Full-attention units all cost the same, so a last wave of
// r < #SMs units leaves the other SMs idle for a whole unit.  When r is at most
// half the SMs, the host makes those units key-split: each becomes two grid
// blocks (units), one per 128-row half, and within a half tile 0 takes the
// first h of the 2h key blocks and tile 1 the rest (ring items K_j, K_{h+j},
// V_j, V_{h+j} per step), so the last wave takes half as long.  Tile 1
// then leaves its row statistics (m_1, l_1) in shared memory (merge barrier),
// and tile 0 combines the two tiles: m = max(m_0, m_1), l = l_0 2^(m_0 - m) +
// l_1 2^(m_1 - m), O = (2^(m_0 - m) O_0 + 2^(m_1 - m) O_1) / l -- the online
// softmax's rescaling applied once more, as when two blocks of keys are
// combined -- and frees both O tiles.  (The wave quantisation that this
// shortens is the W of "A Performance Model for Warp Specialization
// Kernels", core formulas.)
//
// Synchronisation is the aref channel of the Tawa page (Section III-B/III-E):
// every ring slot has a full barrier (TMA transaction bytes) and an empty
// barrier (arrived by tcgen05.commit when the MMAs that read the slot finish);
// use number u of a slot waits on parity (u & 1).  Between MMA issuer and
// softmax: s_full[t] (commit after S_t), p_half[t][h] (one arrival per softmax
// warp once P_t of key half h -- keys 64h..64h+63 -- is in TMEM, so the MMA
// multiplies the first half into O_t while the softmax computes the second),
// pva_done[t] (commit after that first half, awaited only by a softmax that
// must rescale O_t mid-block), o_full[t] (commit after the last P_t V).  With
// split P (D = 64) P_t is handed over whole, on p_half[t][1] alone, and
// pvb_done[t] (commit after its P V) tells the softmax when it may rewrite
// the P columns: there each hand-off, vote and wait costs the softmax warp a
// few hundred cycles on a sub-partition shared with the other tile's softmax,
// and whole-block hand-offs measured 6 % faster than half-block ones.
//
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+D),
// O_1 [256+D,256+2D).  At D = 128, P_t overwrites the first columns of S_t
// once the softmax has read S_t into registers: 64 columns of 16-bit P (two
// per column) or 32 of E4M3 P (four per column).  At D = 64, P_t has columns
// of its own after the O tiles (split P, below).
//
// Online softmax with a lazy maximum: the running maximum m (in log2 units of
// the scaled logits) is only raised when a block's maximum exceeds it by more
// than tau, so P <= 2^tau and O_t is rescaled in TMEM only on those rare
// blocks; the result does not depend on tau.  Because m is known before a
// block's S arrives, P is computed against it as S streams out of TMEM, and the
// block is redone in the rare case the rule raises m.  tau = 15 is the largest
// value that keeps every P finite in f16 (2^15 < 65504); the larger tau, the
// rarer a redo: with logits four times as spread as N(0,1) inputs give, tau = 8
// redoes often enough to cost a quarter of the throughput at D = 64.  (tau is a
// kernel parameter so tests can vary it.)
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "ptx.cuh"

namespace wsa {
template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

constexpr int kBM = 128;       // query rows per tile (tcgen05 M)
constexpr int kBN = 128;       // keys per block
constexpr int kWarpMma = 8;    // MMA issuer (of query tile 0 with two issuers) and TMEM allocator
constexpr int kWarpLoad = 9;
constexpr int kWarpMma1 = 10;  // MMA issuer of query tile 1 (with two issuers)
constexpr float kTauDefault = 15.0f;     // lazy-rescale threshold, log2 units (16-bit P)
constexpr float kTauDefaultE4m3 = 8.0f;  // E4M3 P: stored unscaled, <= 2^8 = 256 < 448
constexpr uint32_t kTmemCols = 512;

// Element types: Q, K, V (and P, O) in f16 or bf16; or E4M3 Q, K, V (V
// supplied transposed per head), P in E4M3 and O in bf16.
enum : int { kF16 = 0, kBF16 = 1, kE4M3 = 2 };

// Device status bits (OR-ed into the status word on an abandoned wait).
enum : int {
  kStatusTimeoutLoad = 1,
  kStatusTimeoutMma = 2,
  kStatusTimeoutSoftmax = 4,
  kStatusTimeoutDrain = 8,
};

// Registers per thread that a 12-warp block is launched with (65,536 / 384,
// rounded down to the allocation granularity of 8).
constexpr int kRegLaunch = 168;

template <int D, int ET, bool CAUSAL = false>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(ET != kE4M3 || D == 128, "E4M3 inputs: head dim 128");
  static constexpr int kElemBytes = ET == kE4M3 ? 1 : 2;
  static constexpr int kTileBytes = kBM * D * kElemBytes;  // 128 x D
  static constexpr int kSlotBytes = kBN * D * kElemBytes;
  static constexpr int kStages = kSlotBytes == 16384 ? 8 : 4;  // K/V ring slots
  static constexpr int kBoxElems = 128 / kElemBytes;       // elements per 128-byte row of a box
  static constexpr int kColBlocks = D * kElemBytes / 128;  // 128-byte column blocks of a row
  static constexpr int kQBytes = 2 * kTileBytes;
  static constexpr int kRingOff = kQBytes;
  // O staging for the epilogue's TMA stores: per softmax warp, kStageBoxes
  // boxes of 32 rows x 128 bytes (64 16-bit columns of O), 128-byte swizzle.
  // O rows have kOutColBlocks such boxes; with fewer staging boxes than that
  // (16-bit D = 128, where shared memory holds one box per warp) a box is
  // refilled once the TMA engine has read the previous one.
  static constexpr int kOutColBlocks = D * 2 / 128;
  static constexpr int kStageBoxes = ET == kE4M3 ? 2 : 1;
  static constexpr int kStageBoxBytes = 32 * 128;
  static constexpr int kStageOff = kRingOff + kStages * kSlotBytes;
  // D = 64 leaves 128 TMEM columns free: P_t gets its own 64 columns there
  // (split P), so S_t can be overwritten as soon as the softmax has read it.
  static constexpr bool kSplitP = D == 64 && ET != kE4M3;
  // MMA issuers.  At D = 128 one warp issues both tiles' MMAs in the order
  // P_0 V(j), S_0(j+1), P_1 V(j), S_1(j+1): that order keeps the two tiles
  // half a block period apart, so one tile's softmax runs while the other
  // tile's MMAs do.  With split P (D = 64) the tiles' softmax phases overlap
  // anyway, and one issuer per tile keeps a wait on one tile from holding up
  // the other tile's MMAs.
  static constexpr int kIssuers = kSplitP ? 2 : 1;
  // Register split: 12 warps (three whole warpgroups) launched at 168
  // registers (64,512 in all); the producer warpgroup (warps 8-11: the MMA
  // issuer(s), the TMA warp and idle warps) lowers its limit and the two
  // softmax warpgroups raise theirs by the same total, so the raise never
  // waits on registers that are not there.  D = 128: 104 / 200 (128 x 104 +
  // 256 x 200 = 64,512); measured +1 % (S16K), +6 % (E4M3), +7 % (S1K) and
  // +10-12 % (causal S4K), while a 12-warp launch without the split is slower
  // than 10 warps.  Causal D = 64: 152 / 176, +4 to +7 %; full attention at
  // D = 64 lost 8 % with it and keeps 11 warps.
  static constexpr bool kRegSplit = D == 128 || (kIssuers == 2 && CAUSAL);
  static constexpr int kRegProducer = D == 128 ? 104 : 152;
  static constexpr int kRegSoftmax = D == 128 ? 200 : 176;
  static_assert(!kRegSplit || 128 * kRegProducer + 256 * kRegSoftmax == 384 * kRegLaunch,
                "register split");
  static constexpr int kThreads = kRegSplit ? 384 : kIssuers == 2 ? 352 : 320;  // 12, 11 or 10 warps
  static constexpr int kUnitReaders = 8 + kIssuers;           // softmax warps + issuers
  // Key-split units (full attention, one issuer): both tiles take the same
  // 128 query rows, tile 0 the first half of the key blocks and tile 1 the
  // second; tile 1 leaves its row statistics (m, l) in its staging boxes,
  // which it has no O to store from, for tile 0, which merges the two O tiles.
  static constexpr bool kKeySplit = kIssuers == 1;
  static constexpr int kCtlOff = kStageOff + 8 * kStageBoxes * kStageBoxBytes;
  static constexpr int kSmemBytes = 1024 + kCtlOff + 512;  // + alignment slack + control
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per block");
  static constexpr uint32_t kOCol = 256;                   // O_t at kOCol + t*D
  static constexpr uint32_t kPCol = 256 + 2 * D;           // split P_t at kPCol + 64t
  static_assert(!kSplitP || kPCol + 128 <= 512, "TMEM columns");
};

struct Ctl {
  uint4 clc_answer;        // cluster-launch-control answer (16-byte aligned)
  uint64_t clc_bar;        // its 16 transaction bytes
  uint64_t unit_full[2];   // work-unit channel, loader -> MMA and softmax warps
  uint64_t unit_empty[2];
  int unit_id[2];          // unit index, or -1: no more work
  uint64_t q_full[2];      // [tile]
  uint64_t q_empty[2];     // [tile]: Q_t consumed by the unit's last Q_t K^T
  uint64_t s_full[2];
  uint64_t p_half[2][2];   // [tile][key half]: P of keys 64h..64h+63 is in TMEM
  uint64_t pva_done[2];    // [tile]: the P V of keys 0-63 of the current block is done
  uint64_t pvb_done[2];    // [tile]: ... of keys 64-127 (split P only)
  uint64_t s_free[2];      // [tile]: the softmax has read S_t (split P only)
  uint64_t o_full[2];
  uint64_t o_empty[2];     // [tile]: the epilogue has read O_t out of TMEM
  uint64_t mma_drain[2];
  uint64_t kv_full[8];
  uint64_t kv_empty[2][8]; // [tile][slot]: that tile's MMAs have finished reading the slot
  uint32_t tmem_base;
  int abort;
  uint64_t merge;          // key-split instantiations: tile 1 is done with the unit
                           // (and left its row statistics if the unit is key-split)
};
static_assert(sizeof(Ctl) <= 512, "control block size");

struct FwdParams {
  float* lse;         // (B,H,S) fp32 (O is written through its tensor map)
  int* status;        // device status word
  int S;
  int n_qblk;         // ceil(S / 256)
  int BH;             // B * H
  int group_heads;    // causal unit order: heads per L2 group (>= 1)
  int n_whole;        // full attention: units x >= n_whole are the 128-row halves
                      // of key-split units (n_qblk * BH when none is split)
  int dynamic;        // 1: blocks take further units by cluster launch control
  float scale_log2;   // scale * log2(e)
  uint64_t wait_limit_ns;
  int inject;         // 0 in normal use; 1 drops one softmax arrival (timeout test)
  float tau;          // lazy-rescale threshold (log2 units), 0 <= tau <= 15
  float two_pow_tau;  // 2^(tau + p_shift): the half-sum that proves no raise is due
  float p_shift;      // P is stored as 2^p_shift * exp2(s*c - m): 0 for 16-bit P;
                      // 8 - tau for E4M3, so P <= 256 < 448 and small P stay
                      // out of the E4M3 subnormal range (l carries the same
                      // factor, so O = P V / l is unchanged)
};

// A work unit: one (batch*head) index and one 256-row query block, or, for a
// key-split unit, one 128-row half of it whose keys the two tiles share out.
struct Unit {
  int bh;
  int qb;
  int ks;  // 1: key-split unit
  int r0;  // first query row of tile 0 (of both tiles when ks)
};

template <bool KSPLIT>
__device__ __forceinline__ int tile_row0(const Unit& u, int t) {
  return KSPLIT ? u.r0 + (u.ks ? 0 : t * kBM) : u.qb * 2 * kBM + t * kBM;
}

// Unit index -> (head, query block); the grid has one block per unit and the
// hardware starts (or hands over) blocks in index order, so this fixes the
// order in which units begin.  Full attention: head-major, every unit costs
// the same; the units of the last wave can be split (index n_whole + 2i + h
// is half h of unit n_whole + i), so that a last wave that would leave most
// SMs idle takes half as long.  Causal: unit qb costs 2qb+1 or 2qb+2 key
// blocks, so heads are taken in groups whose K and V fit in L2 together and,
// inside a group, the longest query blocks of all its heads go first
// (longest-processing-time-first list scheduling) -- the schedule that
// shortens the tail, without making K/V of a head leave L2 between its units.
template <bool CAUSAL, bool KSPLIT>
__device__ __forceinline__ Unit decode_unit(int x, const FwdParams& p) {
  Unit u;
  u.ks = 0;
  if (!CAUSAL) {
    int half = 0;
    if (KSPLIT && x >= p.n_whole) {
      const int y = x - p.n_whole;
      x = p.n_whole + (y >> 1);
      half = y & 1;
      u.ks = 1;
    }
    u.bh = x / p.n_qblk;
    u.qb = x - u.bh * p.n_qblk;
    u.r0 = u.qb * 2 * kBM + half * kBM;
    return u;
  }
  const int per_group = p.group_heads * p.n_qblk;
  const int g = x / per_group;
  const int r = x - g * per_group;
  const int gh = min(p.group_heads, p.BH - g * p.group_heads);
  const int level = r / gh;
  u.bh = g * p.group_heads + (r - level * gh);
  u.qb = p.n_qblk - 1 - level;
  u.r0 = u.qb * 2 * kBM;
  return u;
}

// Shared-memory operand descriptors, 128-byte swizzle.  High half: 8-row groups
// 1024 bytes apart.  Low half: start address plus the leading byte offset,
// which K-major operands (Q, K and the transposed 8-bit V: rows of 128 bytes)
// do not use and the MN-major 16-bit V operand of P V uses as the distance
// between its 64-column blocks.
constexpr uint32_t kDescHi = sdesc_hi(1024);
constexpr uint32_t kLboKMajor = 16;
constexpr uint32_t kLboV = kBN * 128;

// S = Q K^T into TMEM: D / K steps of K = 16 (16-bit) or 32 (E4M3) elements,
// 32 bytes within a 128-byte row; every fourth step moves to the next 16 KB
// column block.  Warp-collective.
template <int D, int ET>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_lo, uint32_t k_lo) {
  static_assert(kBM == kBN, "Q and K tiles share one column-block size");
  constexpr int kStep = ET == kE4M3 ? 32 : 16;
  constexpr uint32_t idesc = idesc_f16(ET == kBF16, kBM, kBN, false);
#pragma unroll
  for (int kk = 0; kk < D / kStep; ++kk) {
    const uint32_t step = (kk >> 2) * ((kBM * 128) >> 4) + (kk & 3) * (32 >> 4);
    const uint64_t a = sdesc_join(q_lo + step, kDescHi), b = sdesc_join(k_lo + step, kDescHi);
    if constexpr (ET == kE4M3)
      mma_ss_f8_warp(d_tmem, a, b, idesc, kk > 0 ? 1u : 0u);
    else
      mma_ss_warp(d_tmem, a, b, idesc, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V over keys [64*half, 64*half + 64), P from TMEM (8 columns per
// step).  16-bit: 16 keys per step, V MN-major, 16 rows (2 KB) per step.
// E4M3: 32 keys per step, V transposed (K-major, 128 keys per 128-byte row),
// 32 bytes along the row per step.  Warp-collective.
template <int D, int ET>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_lo,
                                              int half, bool accumulate) {
  if constexpr (ET == kE4M3) {
    constexpr uint32_t idesc = idesc_f16(false, kBM, D, false);
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int kk = half * 2 + k2;
      mma_ts_f8_warp(d_tmem, p_tmem + kk * 8, sdesc_join(v_lo + kk * (32 >> 4), kDescHi), idesc,
                     (accumulate || kk > 0) ? 1u : 0u);
    }
  } else {
    constexpr uint32_t idesc = idesc_f16(ET == kBF16, kBM, D, true);
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const int kk = half * 4 + k4;
      mma_ts_warp(d_tmem, p_tmem + kk * 8, sdesc_join(v_lo + kk * ((16 * 128) >> 4), kDescHi),
                  idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
  }
}

template <int D, int ET>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_lo,
                                         bool accumulate) {
  issue_pv_half<D, ET>(d_tmem, p_tmem, v_lo, 0, accumulate);
  issue_pv_half<D, ET>(d_tmem, p_tmem, v_lo, 1, true);
}

// Raw S values (fp32 bit patterns) of keys with in-block index >= lim_blk
// become -inf (masked).
template <int C0, int N>
__device__ __forceinline__ void mask_keys(uint32_t* s, int lim_blk) {
#pragma unroll
  for (int c = 0; c < N; ++c)
    if (C0 + c >= lim_blk) s[c] = 0xff800000u;
}

template <int N>
__device__ __forceinline__ float row_max(const uint32_t* s) {
  float a = __uint_as_float(s[0]), b = __uint_as_float(s[1]);
#pragma unroll
  for (int c = 2; c + 3 < N; c += 4) {
    a = fmax3(a, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    b = fmax3(b, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
  }
  return fmaxf(fmaxf(a, b), fmaxf(__uint_as_float(s[N - 2]), __uint_as_float(s[N - 1])));
}

// P for 32 keys: p = exp2(s*c - m), rounded to the P type and packed into pk
// (16-bit: two per word, pk[0..15]; E4M3: four per word, pk[0..7]); returns
// the fp32 sum of the 32 values.
template <int ET>
__device__ __forceinline__ float exp_chunk(const uint32_t* s, uint64_t c2, uint64_t negm2,
                                           uint32_t (&pk)[16]) {
  uint64_t acc0 = 0, acc1 = 0;
  float prev_a = 0.f, prev_b = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint64_t x = ffma2(f2_pack(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1])),
                             c2, negm2);
    float a, b;
    f2_unpack(x, a, b);
    a = ex2(a);
    b = ex2(b);
    if (i & 1)
      acc1 = fadd2(acc1, f2_pack(a, b));
    else
      acc0 = fadd2(acc0, f2_pack(a, b));
    if constexpr (ET == kE4M3) {
      if (i & 1)
        pk[i >> 1] = pack4_e4m3(prev_a, prev_b, a, b);
      prev_a = a;
      prev_b = b;
    } else {
      pk[i] = pack2<ET == kBF16>(a, b);
    }
  }
  float s0, s1, s2, s3;
  f2_unpack(acc0, s0, s1);
  f2_unpack(acc1, s2, s3);
  return (s0 + s1) + (s2 + s3);
}

// TMEM columns P takes per 32 keys: 16 (16-bit) or 8 (E4M3).
template <int ET>
constexpr uint32_t kPColsPer32 = ET == kE4M3 ? 8u : 16u;

// Stores the P of 32-key chunk `chunk` of a block at its columns from tP (no
// wait).
template <int ET>
__device__ __forceinline__ void store_p(uint32_t tP, int chunk, const uint32_t (&pk)[16]) {
  if constexpr (ET == kE4M3)
    tmem_st_x8_async(tP + chunk * kPColsPer32<ET>, pk);
  else
    tmem_st_x16_async(tP + chunk * kPColsPer32<ET>, pk);
}

// Loads keys 0-63 of S into lo and 64-127 into hi (waits).
__device__ __forceinline__ void load_s(uint32_t tS, uint32_t (&lo)[64], uint32_t (&hi)[64]) {
  uint32_t(&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&lo[0]);
  uint32_t(&b)[32] = *reinterpret_cast<uint32_t(*)[32]>(&lo[32]);
  uint32_t(&c)[32] = *reinterpret_cast<uint32_t(*)[32]>(&hi[0]);
  uint32_t(&d)[32] = *reinterpret_cast<uint32_t(*)[32]>(&hi[32]);
  tmem_ld_x32_async(tS, a);
  tmem_ld_x32_async(tS + 32, b);
  tmem_ld_x32_async(tS + 64, c);
  tmem_ld_x32_async(tS + 96, d);
  tmem_ld_wait_x32(a);
  tmem_ld_wait_x32(b);
  tmem_ld_wait_x32(c);
  tmem_ld_wait_x32(d);
}

// Keys 0-63 of a block: S columns 0-63 arrive in one TMEM round trip (two
// 32-column loads, one wait; tcgen05.wait::ld waits for every outstanding
// load), then the load of columns 64-95 into hi is put in flight and keys
// 0-63 are exponentiated against m while it lands; P over the first S
// columns (chunks 0, 1).  Returns the sum of P.
template <int ET>
__device__ __forceinline__ float exp_keys_lo(uint32_t (&lo)[64], uint32_t (&hi)[64], uint32_t tS,
                                             uint64_t c2, uint64_t negm2, bool masked,
                                             int lim_blk) {
  uint32_t(&c0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&lo[0]);
  uint32_t(&c1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&lo[32]);
  uint32_t(&c2r)[32] = *reinterpret_cast<uint32_t(*)[32]>(&hi[0]);
  uint32_t pk[16];
  tmem_ld_x32_async(tS, c0);
  tmem_ld_x32_async(tS + 32, c1);
  tmem_ld_wait_x32(c0);
  tmem_ld_wait_x32(c1);
  tmem_ld_x32_async(tS + 64, c2r);
  if (masked) mask_keys<0, 64>(lo, lim_blk);
  float sum = exp_chunk<ET>(c0, c2, negm2, pk);
  store_p<ET>(tS, 0, pk);
  sum += exp_chunk<ET>(c1, c2, negm2, pk);
  store_p<ET>(tS, 1, pk);
  return sum;
}

// Keys 64-127 (the load of 64-95 issued by exp_keys_lo; 96-127 follows it);
// P chunks 2, 3.  Returns the sum of P.
template <int ET>
__device__ __forceinline__ float exp_keys_hi(uint32_t (&hi)[64], uint32_t tS, uint64_t c2,
                                             uint64_t negm2, bool masked, int lim_blk) {
  uint32_t(&c2r)[32] = *reinterpret_cast<uint32_t(*)[32]>(&hi[0]);
  uint32_t(&c3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&hi[32]);
  uint32_t pk[16];
  tmem_ld_wait_x32(c2r);
  tmem_ld_x32_async(tS + 96, c3);
  if (masked) mask_keys<64, 32>(c2r, lim_blk);
  float sum = exp_chunk<ET>(c2r, c2, negm2, pk);
  store_p<ET>(tS, 2, pk);
  tmem_ld_wait_x32(c3);
  if (masked) mask_keys<96, 32>(c3, lim_blk);
  sum += exp_chunk<ET>(c3, c2, negm2, pk);
  store_p<ET>(tS, 3, pk);
  return sum;
}

// P of key half `half` (64 keys already in registers) against m, to its P
// columns from tP (no wait).  Returns the sum of P.
template <int ET>
__device__ __forceinline__ float exp_keys_regs(const uint32_t* s, float cl2, float m, uint32_t tP,
                                               int half) {
  const uint64_t c2 = f2_pack(cl2, cl2), negm2 = f2_pack(-m, -m);
  uint32_t pk[16];
  float sum = exp_chunk<ET>(s, c2, negm2, pk);
  store_p<ET>(tP, 2 * half, pk);
  sum += exp_chunk<ET>(s + 32, c2, negm2, pk);
  store_p<ET>(tP, 2 * half + 1, pk);
  return sum;
}

template <int D, int ET, bool CAUSAL, bool KSPLIT>
__global__ void __launch_bounds__(Cfg<D, ET, CAUSAL>::kThreads, 1)
    fmha_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  using C = Cfg<D, ET, CAUSAL>;
  // KSPLIT: the grid's units from p.n_whole on are key-split (a separate
  // instantiation, so that launches without them run none of its code)
  static_assert(!KSPLIT || (C::kKeySplit && !CAUSAL), "key-split units: full attention, one issuer");
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzle atoms need 1024-byte aligned tiles
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_u32(smem);
  Ctl& ctl = *reinterpret_cast<Ctl*>(smem + C::kCtlOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.S;
  const int nkv_all = (S + kBN - 1) / kBN;
  // key blocks of query tile 0 / tile 1 of query block qb
  auto nkv_tile0 = [&](int qb) { return CAUSAL ? min(nkv_all, 2 * qb + 1) : nkv_all; };
  auto nkv_tile1 = [&](int qb) { return CAUSAL ? min(nkv_all, 2 * qb + 2) : nkv_all; };

  if (threadIdx.x == 0) {
    mbar_init(&ctl.clc_bar, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.unit_full[i], 1);
      mbar_init(&ctl.unit_empty[i], C::kUnitReaders);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&ctl.q_full[t], 1);
      mbar_init(&ctl.q_empty[t], 1);
      mbar_init(&ctl.mma_drain[t], 1);
      mbar_init(&ctl.s_full[t], 1);
      mbar_init(&ctl.p_half[t][0], 4);  // one elected arrival per softmax warp
      mbar_init(&ctl.p_half[t][1], 4);
      mbar_init(&ctl.pva_done[t], 1);
      mbar_init(&ctl.pvb_done[t], 1);
      mbar_init(&ctl.s_free[t], 4);
      mbar_init(&ctl.o_full[t], 1);
      mbar_init(&ctl.o_empty[t], 4);
    }
    mbar_init(&ctl.merge, 4);  // every warp of tile 1 (key-split instantiations)
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&ctl.kv_full[s], 1);
      mbar_init(&ctl.kv_empty[0][s], 1);
      mbar_init(&ctl.kv_empty[1][s], 1);
    }
    ctl.abort = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&ctl.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort;

  const uint32_t sQ = sbase;
  const uint32_t sRing = sbase + C::kRingOff;
  const uint32_t sStage = sbase + C::kStageOff;

  // The k-th unit of this block (k = 0, 1, ...) travels from the loader to the
  // other roles through slot k & 1 of the unit channel; -1 ends the loop.
  auto next_unit = [&](uint32_t k, int code, int* out) {
    bool ok = mbar_wait(&ctl.unit_full[k & 1], (k >> 1) & 1, abort_flag, p.status, code,
                        p.wait_limit_ns);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    *out = *reinterpret_cast<volatile int*>(&ctl.unit_id[k & 1]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl.unit_empty[k & 1]);
    return true;
  };

  if (warp == kWarpLoad) {
    if constexpr (C::kRegSplit) setmaxnreg_dec<C::kRegProducer>();
    // ================================================================ TMA producer
    // The whole warp runs the loop; one elected lane issues each copy.
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    const uint64_t pol_q = policy_evict_first();
    const uint64_t pol_kv = policy_evict_last();
    const uint32_t clc_answer = smem_u32(&ctl.clc_answer);
    uint32_t it = 0;         // ring item: K_j of a unit, then V_j, block after block
    uint32_t nq[2] = {0, 0}; // Q_t loads issued
    // Per ring slot (bit s): which query tiles read the item now in the slot,
    // and the parity of how many items of the slot each tile has read.  A slot
    // is reloaded once every tile that read its previous item has released it
    // (kv_empty[t][slot]); under a causal mask tile 0 skips the unit's last
    // key block, so it neither reads nor releases that block's items.
    uint32_t rd0 = 0, rd1 = 0, par0 = 0, par1 = 0;
    uint32_t asked = 0;      // cancellation requests issued
    uint32_t answered = 0;   // ... and their answers read
    bool ok = true;
    int x = blockIdx.x;
    for (uint32_t k = 0; ok; ++k) {
      ok = mbar_wait(&ctl.unit_empty[k & 1], ((k >> 1) & 1) ^ 1, abort_flag, p.status,
                     kStatusTimeoutLoad, p.wait_limit_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (lane == 0) {
        ctl.unit_id[k & 1] = x;
        mbar_arrive(&ctl.unit_full[k & 1]);
      }
      __syncwarp();
      if (x < 0) break;
      const Unit u = decode_unit<CAUSAL, KSPLIT>(x, p);
      const bool ks = KSPLIT && u.ks;
      // key blocks per tile; a key-split unit loads K_j, K_{h+j}, V_j, V_{h+j}
      // per step j (tile 0 reads key block j, tile 1 key block h + j)
      const int nkv0 = ks ? nkv_all / 2 : nkv_tile0(u.qb);
      const int nkv1 = ks ? nkv_all / 2 : nkv_tile1(u.qb);
      const int per_step = ks ? 4 : 2;
      if (p.dynamic) {
        // ask for the next unit now; the answer is read half-way through this one
        fence_proxy_async_smem();
        mbar_arrive_expect_tx_warp(&ctl.clc_bar, 16);
        clc_try_cancel_warp(clc_answer, &ctl.clc_bar);
        ++asked;
      }
      int x_next = -1;
      for (int j = 0; ok && j < nkv1; ++j) {
        for (int e = 0; e < per_step; ++e) {
          const int kv = ks ? e >> 1 : e;
          const int kb = ks && (e & 1) ? nkv1 + j : j;  // key block
          const uint32_t slot = it % C::kStages, bit = 1u << slot;
          if (rd0 & bit)
            ok = mbar_wait(&ctl.kv_empty[0][slot], (par0 & bit) ? 0u : 1u, abort_flag, p.status,
                           kStatusTimeoutLoad, p.wait_limit_ns);
          if (ok && (rd1 & bit))
            ok = mbar_wait(&ctl.kv_empty[1][slot], (par1 & bit) ? 0u : 1u, abort_flag, p.status,
                           kStatusTimeoutLoad, p.wait_limit_ns);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          if (C::kIssuers == 1 || j < nkv0) {  // one issuer releases every item as tile 0
            rd0 |= bit;
            par0 ^= bit;
          } else {
            rd0 &= ~bit;
          }
          if (C::kIssuers == 2) {
            rd1 |= bit;
            par1 ^= bit;
          }
          mbar_arrive_expect_tx_warp(&ctl.kv_full[slot], C::kSlotBytes);
          if (ET == kE4M3 && kv) {
            // V transposed: one box of 128 keys x 128 rows (d)
            tma_load_3d_warp(sRing + slot * C::kSlotBytes, &tm_v, &ctl.kv_full[slot], kb * kBN, 0,
                             u.bh, pol_kv);
          } else {
            const CUtensorMap* m = kv ? &tm_v : &tm_k;
            for (int cb = 0; cb < C::kColBlocks; ++cb)
              tma_load_3d_warp(sRing + slot * C::kSlotBytes + cb * (kBN * 128), m,
                               &ctl.kv_full[slot], cb * C::kBoxElems, kb * kBN, u.bh, pol_kv);
          }
          ++it;
          if (j == 0 && e == per_step - 1) {
            // Q_t after the first step's K and V: the previous unit's last
            // Q_t K^T frees the tile while this unit's first K/V are in flight.
            for (int t = 0; ok && t < 2; ++t) {
              ok = mbar_wait(&ctl.q_empty[t], (nq[t] & 1) ^ 1, abort_flag, p.status,
                             kStatusTimeoutLoad, p.wait_limit_ns);
              ok = __all_sync(0xffffffffu, ok);
              if (!ok) break;
              mbar_arrive_expect_tx_warp(&ctl.q_full[t], C::kTileBytes);
              for (int cb = 0; cb < C::kColBlocks; ++cb)
                tma_load_3d_warp(sQ + t * C::kTileBytes + cb * (kBM * 128), &tm_q, &ctl.q_full[t],
                                 cb * C::kBoxElems, tile_row0<KSPLIT>(u, t), u.bh, pol_q);
              ++nq[t];
            }
            if (!ok) break;
          }
          if (p.dynamic && j == nkv1 / 2 && e == per_step - 1) {
            ok = mbar_wait(&ctl.clc_bar, answered & 1, abort_flag, p.status, kStatusTimeoutLoad,
                           p.wait_limit_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            x_next = clc_cancelled_x(clc_answer);
            ++answered;
            if (x_next >= 0) {
              // the next unit's Q into L2 while this unit still streams
              const Unit un = decode_unit<CAUSAL, KSPLIT>(x_next, p);
              for (int t = 0; t < 2; ++t)
                for (int cb = 0; cb < C::kColBlocks; ++cb)
                  tma_prefetch_3d_warp(&tm_q, cb * C::kBoxElems, tile_row0<KSPLIT>(un, t), un.bh);
            }
          }
        }
      }
      x = x_next;
    }
    // Drain: every issued copy and request lands before the block may exit.
    if (asked > answered)
      mbar_wait(&ctl.clc_bar, answered & 1, nullptr, p.status, kStatusTimeoutDrain,
                p.wait_limit_ns);
    for (int t = 0; t < 2; ++t)
      if (nq[t] > 0)
        mbar_wait(&ctl.q_full[t], (nq[t] - 1) & 1, nullptr, p.status, kStatusTimeoutDrain,
                  p.wait_limit_ns);
    const uint32_t first = it > (uint32_t)C::kStages ? it - C::kStages : 0u;
    for (uint32_t i = first; i < it; ++i)
      mbar_wait(&ctl.kv_full[i % C::kStages], (i / C::kStages) & 1, nullptr, p.status,
                kStatusTimeoutDrain, p.wait_limit_ns);
    __syncwarp();
  } else if (warp == kWarpMma || (C::kIssuers == 2 && warp == kWarpMma1)) {
    if constexpr (C::kRegSplit) setmaxnreg_dec<C::kRegProducer>();
    // ================================================================ MMA issuers
    // Each issuer warp runs its loop with warp-uniform operands; one elected
    // lane issues every tcgen05.mma and tcgen05.commit.  A commit tracks only
    // the issuing warp's own MMAs: an issuer releases ring slots through
    // kv_empty[i] (i = its index) and the Q tiles of its query tiles through
    // q_empty[t].
    const int issuer = warp == kWarpMma ? 0 : 1;
    auto slot_addr = [&](uint32_t item) { return sRing + (item % C::kStages) * C::kSlotBytes; };
    auto k_lo = [&](uint32_t item) { return sdesc_lo(slot_addr(item), kLboKMajor); };
    auto v_lo = [&](uint32_t item) {
      return sdesc_lo(slot_addr(item), ET == kE4M3 ? kLboKMajor : kLboV);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      const bool good =
          mbar_wait(bar, parity, abort_flag, p.status, kStatusTimeoutMma, p.wait_limit_ns);
      return __all_sync(0xffffffffu, good) != 0;
    };
    auto wait_full = [&](uint32_t item) {
      return wait(&ctl.kv_full[item % C::kStages], (item / C::kStages) & 1);
    };
    auto release = [&](uint32_t item) {
      mma_commit_warp(&ctl.kv_empty[issuer][item % C::kStages]);
    };
    // O_t += P_t V.  P over S: in two key halves, each as soon as its P is in
    // TMEM; the first half's completion is committed for a softmax that has to
    // rescale O_t while computing the second half.  Split P: both halves once
    // all of P is in TMEM.  gj = the tile's block count over all units of this
    // block (P phases).
    auto pv_halves = [&](int t, uint32_t tO, uint32_t tP, uint32_t vlo, uint32_t gj, int j) {
      if constexpr (C::kSplitP) {
        // split P is handed over whole (p_half[t][1])
        if (!wait(&ctl.p_half[t][1], gj & 1)) return false;
        tc_fence_after();
        issue_pv_half<D, ET>(tO, tP, vlo, 0, j > 0);
        issue_pv_half<D, ET>(tO, tP, vlo, 1, true);
        mma_commit_warp(&ctl.pvb_done[t]);
        return true;
      }
      if (!wait(&ctl.p_half[t][0], gj & 1)) return false;
      tc_fence_after();
      issue_pv_half<D, ET>(tO, tP, vlo, 0, j > 0);
      mma_commit_warp(&ctl.pva_done[t]);
      if (!wait(&ctl.p_half[t][1], gj & 1)) return false;
      tc_fence_after();
      issue_pv_half<D, ET>(tO, tP, vlo, 1, true);
      return true;
    };
    bool ok = true;
    uint32_t it = 0;  // ring item of the unit's K_0
    if constexpr (C::kIssuers == 2) {
      // One issuer per query tile (split P).
      const int t = issuer;
      const uint32_t tS = tmem + t * kBM;
      const uint32_t tO = tmem + C::kOCol + t * D;
      const uint32_t tP = tmem + C::kPCol + t * 64;
      const uint32_t q_lo = sdesc_lo(sQ + t * C::kTileBytes, kLboKMajor);
      // S_t = Q_t K^T of ring item ik; after the unit's last one, Q_t is free.
      auto qk = [&](uint32_t ik, bool last) {
        tc_fence_after();
        issue_qk<D, ET>(tS, q_lo, k_lo(ik));
        mma_commit_warp(&ctl.s_full[t]);
        release(ik);
        if (last) mma_commit_warp(&ctl.q_empty[t]);
      };
      uint32_t g = 0;  // key blocks done by this tile over all units of the block
      for (uint32_t k = 0; ok; ++k) {
        int x;
        ok = next_unit(k, kStatusTimeoutMma, &x);
        if (!ok || x < 0) break;
        const Unit u = decode_unit<CAUSAL, KSPLIT>(x, p);
        const int nkv = t ? nkv_tile1(u.qb) : nkv_tile0(u.qb);
        const int nkv1 = nkv_tile1(u.qb);  // the unit's key blocks (ring items / 2)
        // S_t is overwritten only after the softmax has read it
        ok = wait_full(it) && wait(&ctl.q_full[t], k & 1) &&
             (g == 0 || wait(&ctl.s_free[t], (g - 1) & 1));
        if (!ok) break;
        qk(it, nkv == 1);
        // The unit's first P V overwrites O_t: the previous unit's epilogue
        // must have read it.
        ok = wait(&ctl.o_empty[t], (k & 1) ^ 1);
        for (int j = 0; ok && j < nkv; ++j) {
          const uint32_t iv = it + 2 * j + 1, ik = it + 2 * j + 2;
          // The next S_t waits only until the softmax has read this one, so
          // it is computed while the softmax still works on block j.
          if (j + 1 < nkv) {
            ok = wait_full(ik) && wait(&ctl.s_free[t], (g + j) & 1);
            if (!ok) break;
            qk(ik, j + 2 == nkv);
          }
          ok = wait_full(iv) && pv_halves(t, tO, tP, v_lo(iv), g + j, j);
          if (!ok) break;
          release(iv);
          if (j == nkv - 1) mma_commit_warp(&ctl.o_full[t]);
        }
        it += 2 * nkv1;
        g += nkv;
      }
    } else {
      // One issuer for both tiles (P lies over S).  Per block j the issue
      // order is P_0 V(j), S_0(j+1), P_1 V(j), S_1(j+1): each S_t(j+1) follows
      // the P_t V(j) that reads P_t, and the tiles stay half a period apart.
      const uint32_t tS0 = tmem, tS1 = tmem + kBM;
      const uint32_t tO0 = tmem + C::kOCol, tO1 = tmem + C::kOCol + D;
      const uint32_t q0_lo = sdesc_lo(sQ, kLboKMajor);
      const uint32_t q1_lo = sdesc_lo(sQ + C::kTileBytes, kLboKMajor);
      auto free_q = [&]() {  // after the unit's last Q K^T (which is tile 1's)
        mma_commit_warp(&ctl.q_empty[0]);
        mma_commit_warp(&ctl.q_empty[1]);
      };
      uint32_t g0 = 0, g1 = 0;  // key blocks done by tile 0 / tile 1
      // A key-split unit (h key blocks per tile): the same issue order, but
      // each tile reads its own K and V -- ring items 4j + t and 4j + 2 + t of
      // step j -- and each item is released after its tile's MMAs.  (Whole
      // units keep their own loop below: this schedule's issue loop is the
      // critical path, and folding both into one costs whole units 1-3 %.)
      auto run_split_unit = [&](uint32_t k, int h) -> bool {
        bool good = wait_full(it) && wait_full(it + 1) && wait(&ctl.q_full[0], k & 1) &&
                    wait(&ctl.q_full[1], k & 1);
        if (!good) return false;
        tc_fence_after();
        issue_qk<D, ET>(tS0, q0_lo, k_lo(it));
        mma_commit_warp(&ctl.s_full[0]);
        issue_qk<D, ET>(tS1, q1_lo, k_lo(it + 1));
        mma_commit_warp(&ctl.s_full[1]);
        release(it);
        release(it + 1);
        if (h == 1) free_q();
        good = wait(&ctl.o_empty[0], (k & 1) ^ 1) && wait(&ctl.o_empty[1], (k & 1) ^ 1);
        for (int j = 0; good && j < h; ++j) {
          const uint32_t step = it + 4 * j;  // K_j, K_{h+j}, V_j, V_{h+j}
          const bool more = j + 1 < h;
          good = wait_full(step + 2) && pv_halves(0, tO0, tS0, v_lo(step + 2), g0 + j, j);
          if (!good) break;
          if (j == h - 1) mma_commit_warp(&ctl.o_full[0]);
          release(step + 2);
          if (more) {
            if (!(good = wait_full(step + 4))) break;
            tc_fence_after();
            issue_qk<D, ET>(tS0, q0_lo, k_lo(step + 4));
            mma_commit_warp(&ctl.s_full[0]);
            release(step + 4);
          }
          good = wait_full(step + 3) && pv_halves(1, tO1, tS1, v_lo(step + 3), g1 + j, j);
          if (!good) break;
          release(step + 3);
          if (j == h - 1) mma_commit_warp(&ctl.o_full[1]);
          if (more) {
            if (!(good = wait_full(step + 5))) break;
            tc_fence_after();
            issue_qk<D, ET>(tS1, q1_lo, k_lo(step + 5));
            mma_commit_warp(&ctl.s_full[1]);
            release(step + 5);
            if (j + 2 == h) free_q();
          }
        }
        return good;
      };
      for (uint32_t k = 0; ok; ++k) {
        int x;
        ok = next_unit(k, kStatusTimeoutMma, &x);
        if (!ok || x < 0) break;
        const Unit u = decode_unit<CAUSAL, KSPLIT>(x, p);
        if (KSPLIT && u.ks) {
          const int h = nkv_all / 2;
          ok = run_split_unit(k, h);
          it += 4 * h;
          g0 += h;
          g1 += h;
          continue;
        }
        const int nkv0 = nkv_tile0(u.qb), nkv1 = nkv_tile1(u.qb);
        ok = wait_full(it) && wait(&ctl.q_full[0], k & 1) && wait(&ctl.q_full[1], k & 1);
        if (!ok) break;
        tc_fence_after();
        issue_qk<D, ET>(tS0, q0_lo, k_lo(it));
        mma_commit_warp(&ctl.s_full[0]);
        issue_qk<D, ET>(tS1, q1_lo, k_lo(it));
        mma_commit_warp(&ctl.s_full[1]);
        release(it);
        if (nkv1 == 1) free_q();
        // The unit's first P V overwrites O_0 and O_1: the previous unit's
        // epilogue must have read them (waited here, outside the block loop).
        ok = wait(&ctl.o_empty[0], (k & 1) ^ 1) && wait(&ctl.o_empty[1], (k & 1) ^ 1);
        for (int j = 0; ok && j < nkv1; ++j) {
          const uint32_t iv = it + 2 * j + 1, ik = it + 2 * j + 2;
          const bool more = j + 1 < nkv1;
          ok = wait_full(iv);
          if (ok && j < nkv0) {
            ok = pv_halves(0, tO0, tS0, v_lo(iv), g0 + j, j);
            if (ok && j == nkv0 - 1) mma_commit_warp(&ctl.o_full[0]);
          }
          if (ok && more) {
            ok = wait_full(ik);
            tc_fence_after();
            if (ok && j + 1 < nkv0) {
              issue_qk<D, ET>(tS0, q0_lo, k_lo(ik));
              mma_commit_warp(&ctl.s_full[0]);
            }
          }
          ok = ok && pv_halves(1, tO1, tS1, v_lo(iv), g1 + j, j);
          if (!ok) break;
          release(iv);
          if (j == nkv1 - 1) mma_commit_warp(&ctl.o_full[1]);
          if (more) {
            issue_qk<D, ET>(tS1, q1_lo, k_lo(ik));
            mma_commit_warp(&ctl.s_full[1]);
            release(ik);
            if (j + 2 == nkv1) free_q();
          }
        }
        it += 2 * nkv1;
        g0 += nkv0;
        g1 += nkv1;
      }
    }
    // Drain: all issued MMAs complete before TMEM can be released.
    mma_commit_warp(&ctl.mma_drain[issuer]);
    mbar_wait(&ctl.mma_drain[issuer], 0, nullptr, p.status, kStatusTimeoutDrain,
              p.wait_limit_ns);
    __syncwarp();
  } else if (C::kRegSplit && (warp == 11 || (C::kIssuers == 1 && warp == 10))) {
    // the producer warpgroup's warps without a role: every warp of a
    // warpgroup takes part in its register release
    setmaxnreg_dec<C::kRegProducer>();
  } else {
    // ================================================================ softmax tile t
    if constexpr (C::kRegSplit) setmaxnreg_inc<C::kRegSoftmax>();
    const int t = warp >> 2;
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t tS = lane_base + t * kBM;
    const uint32_t tO = lane_base + C::kOCol + t * D;
    const uint32_t tP = C::kSplitP ? lane_base + C::kPCol + t * 64 : tS;  // P_t
    const float cl2 = p.scale_log2;
    // 0 at compile time for 16-bit P (x - 0.f folds to x exactly)
    const float shift = ET == kE4M3 ? p.p_shift : 0.f;
    bool ok = true;
    uint32_t g = 0;  // key blocks done by this tile over all units of the block
    for (uint32_t k = 0; ok; ++k) {
      int x;
      ok = next_unit(k, kStatusTimeoutSoftmax, &x);
      if (!ok || x < 0) break;
      const Unit u = decode_unit<CAUSAL, KSPLIT>(x, p);
      const bool ks = KSPLIT && u.ks;
      const int row = tile_row0<KSPLIT>(u, t) + quad * 32 + lane;
      // key blocks of this tile: a key-split unit gives tile 0 the first half
      // and tile 1 the second
      const int nkv = ks ? nkv_all / 2 : (t ? nkv_tile1(u.qb) : nkv_tile0(u.qb));
      // keys visible to this row, counted from the tile's first key block:
      // [0, lim).  (Tile 0 of a key-split unit ends half-way through the keys;
      // its last block goes through the masking path with nothing to mask.)
      const int lim = (CAUSAL ? min(row + 1, S) : S) - (ks && t ? nkv * kBN : 0);

      float m = -INFINITY;  // running maximum, log2 units of the scaled logits
      float l = 0.f;        // running sum of exp2(s*c - m)
      for (int j = 0; j < nkv; ++j) {
        const uint32_t ph = (g + j) & 1;
        ok = mbar_wait(&ctl.s_full[t], ph, abort_flag, p.status, kStatusTimeoutSoftmax,
                       p.wait_limit_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();

        const bool masked_block = (j == nkv - 1) && (CAUSAL || (S % kBN) != 0);
        const int lim_blk = lim - j * kBN;
        uint32_t lo[64], hi[64];
        // Hands one key half of P to the MMA issuer once its stores have landed.
        auto release = [&](int half) {
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && !(p.inject == 1 && t == 0 && k == 0 && j == 0 && half == 0))
            mbar_arrive(&ctl.p_half[t][half]);
        };
        // Split P: all of P at once, signalled on p_half[t][1] alone.
        auto release_both = [&]() {
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0 && !(p.inject == 1 && t == 0 && k == 0 && j == 0))
            mbar_arrive(&ctl.p_half[t][1]);
        };
        // O_t *= alpha for threads with alpha != 1 (all lanes take part).
        auto rescale_o = [&](float alpha) {
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t orr[32];
            tmem_ld_x32(tO + ch * 32, orr);
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tmem_st_x32(tO + ch * 32, orr);
          }
        };
        // A bounded wait of the whole warp; false ends the block loop.
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
          bool good = mbar_wait(bar, parity, abort_flag, p.status, kStatusTimeoutSoftmax,
                                p.wait_limit_ns);
          good = __all_sync(0xffffffffu, good);
          if (!good) ok = false;
          return good;
        };
        if constexpr (C::kSplitP) {
          // Split P: read all of S_t and hand its columns back to the MMA
          // issuer at once; P_t goes to its own columns once the previous
          // block's P V has finished reading them.
          const uint32_t gj = g + j;
          load_s(tS, lo, hi);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl.s_free[t]);
          if (masked_block) {
            mask_keys<0, 64>(lo, lim_blk);
            mask_keys<64, 64>(hi, lim_blk);
          }
          if (j == 0) m = fmaxf(row_max<64>(lo), row_max<64>(hi)) * cl2;
          // The previous block's P V has read both halves of the P columns
          // (its halves are committed in order, so one wait covers both: each
          // wait costs the softmax warp a few hundred cycles on a sub-partition
          // shared with the other tile's softmax).
          if (gj > 0) {
            if (!wait_all(&ctl.pvb_done[t], (gj - 1) & 1)) break;
            tc_fence_after();  // the P stores below follow the MMAs' reads
          }
          // Both key halves, then one lazy-maximum test for the block (the
          // test of the streaming path below, on registers) and one hand-off
          // of all of P: every vote and release costs the softmax warp a few
          // hundred cycles here.
          float la = exp_keys_regs<ET>(lo, cl2, m - shift, tP, 0);
          float lb = exp_keys_regs<ET>(hi, cl2, m - shift, tP, 1);
          const bool check = j > 0 && (la > p.two_pow_tau || lb > p.two_pow_tau);
          if (__any_sync(0xffffffffu, check)) {
            const float bmax = fmaxf(row_max<64>(lo), row_max<64>(hi)) * cl2;
            const bool raise = check && bmax > m + p.tau;
            if (__any_sync(0xffffffffu, raise)) {
              // O_t holds every earlier block (waited above) and none of this
              // one (its P is not handed over yet): scale it, redo the block
              const float alpha = raise ? ex2(m - bmax) : 1.f;
              if (raise) m = bmax;
              l *= alpha;
              tmem_st_wait();
              la = exp_keys_regs<ET>(lo, cl2, m - shift, tP, 0);
              lb = exp_keys_regs<ET>(hi, cl2, m - shift, tP, 1);
              rescale_o(alpha);
            }
          }
          l += la + lb;
          release_both();
        } else if (j == 0) {
          // First block: no running maximum yet, so take the block maximum first.
          load_s(tS, lo, hi);
          if (masked_block) {
            mask_keys<0, 64>(lo, lim_blk);
            mask_keys<64, 64>(hi, lim_blk);
          }
          m = fmaxf(row_max<64>(lo), row_max<64>(hi)) * cl2;
          l = exp_keys_regs<ET>(lo, cl2, m - shift, tS, 0);
          release(0);
          l += exp_keys_regs<ET>(hi, cl2, m - shift, tS, 1);
          release(1);
        } else {
          // Exponentiate against the running maximum as S arrives from TMEM,
          // one key half at a time.  Every p is at most its half's sum, so a sum
          // <= 2^tau proves that no logit of the half exceeds m by more than
          // tau and its P stands as computed; only a larger sum (rare once m has
          // settled: p <= 1 while the block maximum stays below m) needs the
          // exact maximum of that half.
          uint64_t c2 = f2_pack(cl2, cl2), negm2 = f2_pack(-(m - shift), -(m - shift));
          float la = exp_keys_lo<ET>(lo, hi, tS, c2, negm2, masked_block, lim_blk);
          bool check = la > p.two_pow_tau;
          if (__any_sync(0xffffffffu, check)) {
            const float bmax = row_max<64>(lo) * cl2;
            const bool raise = check && bmax > m + p.tau;
            if (__any_sync(0xffffffffu, raise)) {
              // O_t holds every earlier block (the commit behind s_full[t] was
              // issued after the previous P_t V): scale it, redo keys 0-63.
              const float alpha = raise ? ex2(m - bmax) : 1.f;
              if (raise) m = bmax;
              l *= alpha;
              tmem_st_wait();
              la = exp_keys_regs<ET>(lo, cl2, m - shift, tS, 0);
              rescale_o(alpha);
              negm2 = f2_pack(-(m - shift), -(m - shift));
            }
          }
          l += la;
          release(0);
          const float lb = exp_keys_hi<ET>(hi, tS, c2, negm2, masked_block, lim_blk);
          check = lb > p.two_pow_tau;
          float lhi = lb;
          if (__any_sync(0xffffffffu, check)) {
            const float bmax = row_max<64>(hi) * cl2;
            const bool raise = check && bmax > m + p.tau;
            if (__any_sync(0xffffffffu, raise)) {
              // Keys 0-63 of this block are already being multiplied into O_t:
              // wait for that half of P V, then scale O_t (it now includes them,
              // as does l) and redo keys 64-127 against the raised maximum.
              bool good = mbar_wait(&ctl.pva_done[t], ph, abort_flag, p.status,
                                    kStatusTimeoutSoftmax, p.wait_limit_ns);
              good = __all_sync(0xffffffffu, good);
              if (!good) {
                ok = false;
                break;
              }
              tc_fence_after();
              const float alpha = raise ? ex2(m - bmax) : 1.f;
              if (raise) m = bmax;
              l *= alpha;
              tmem_st_wait();
              lhi = exp_keys_regs<ET>(hi, cl2, m - shift, tS, 1);
              rescale_o(alpha);
            }
          }
          l += lhi;
          release(1);
        }
      }
      g += nkv;

      // ---- epilogue: O / l in the output dtype (the input's, bf16 for E4M3
      // inputs), LSE = ln 2 * (m + log2 l - p_shift).  Per 64-column block of
      // O_t each warp reads its 32 rows out of TMEM in two 32-column loads,
      // scales and packs them into its shared-memory staging box (128-byte
      // swizzle, so the 8 lanes of a quarter-warp store to 8 different 16-byte
      // bank groups), and one lane stores the box with a TMA tensor store:
      // whole 128-byte row segments, no per-row global stores; the store runs
      // while the warp moves on (Tawa, Section IV-B, Fig. 7(b): the epilogue
      // of one tile overlaps the next tile's loads and MMAs).  O_t is released
      // once its last columns are in registers.  Reading all of O_t in one
      // burst instead was 9 % slower on causal workloads, where this tile's
      // epilogue runs beside the other tile's last softmax block.
      if (ok) {
        ok = mbar_wait(&ctl.o_full[t], k & 1, abort_flag, p.status, kStatusTimeoutSoftmax,
                       p.wait_limit_ns);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (!ok) break;
      // (key-split kernels decode the unit again: fewer values live across
      // the block loop)
      const Unit ue = KSPLIT ? decode_unit<CAUSAL, KSPLIT>(x, p) : u;
      const bool kse = KSPLIT && ue.ks;
      // tile 1's warp 4 + quad leaves its rows' statistics in its staging box
      float2* const stat = reinterpret_cast<float2*>(
          smem + C::kStageOff + (4 + quad) * (C::kStageBoxes * C::kStageBoxBytes));
      if (KSPLIT && t == 1) {
        // A key-split unit: hand this row's statistics to tile 0, which
        // merges O_1 into its result and frees O_1.  Every warp of tile 1
        // arrives in every unit, so phase k of the barrier is unit k's.
        if (kse) {
          if (lane == 0) bulk_wait_group_read<0>();  // the box's last store has read it
          __syncwarp();
          stat[lane] = make_float2(m, l);
        }
        __syncwarp();  // the warp's statistics, ordered before lane 0's arrival
        if (lane == 0) mbar_arrive(&ctl.merge);
        if (kse) continue;
      }
      tc_fence_after();
      float inv_l = 1.f / l;
      // Merging a key-split unit: with m = max(m_0, m_1) and
      // l = l_0 2^(m_0 - m) + l_1 2^(m_1 - m), O = w0 O_0 + w1 O_1 where
      // w_t = 2^(m_t - m) / l (then scaled by inv_l = 1).
      float w0 = 0.f, w1 = 0.f;
      if (kse) {
        ok = mbar_wait(&ctl.o_full[1], k & 1, abort_flag, p.status, kStatusTimeoutSoftmax,
                       p.wait_limit_ns) &&
             mbar_wait(&ctl.merge, k & 1, abort_flag, p.status, kStatusTimeoutSoftmax,
                       p.wait_limit_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float2 other = stat[lane];
        const float mx = fmaxf(m, other.x);
        const float a0 = ex2(m - mx), a1 = ex2(other.x - mx);
        m = mx;
        l = l * a0 + other.y * a1;
        const float inv = 1.f / l;
        w0 = a0 * inv;
        w1 = a1 * inv;
        inv_l = 1.f;
      }
      const int row0 = tile_row0<KSPLIT>(ue, t) + quad * 32;  // the warp's first row
      const uint32_t stage = sStage + warp * (C::kStageBoxes * C::kStageBoxBytes);
      // One pass over the 64-column blocks of O; MERGE adds w1 O_1 to w0 O_t.
      auto store_o = [&](auto merge_tag) {
        constexpr bool MERGE = decltype(merge_tag)::value;
#pragma unroll 1
        for (int cb = 0; cb < C::kOutColBlocks; ++cb) {
          const uint32_t box = stage + (cb % C::kStageBoxes) * C::kStageBoxBytes;
          // the box's previous TMA store has finished reading it
          if (lane == 0) bulk_wait_group_read<C::kStageBoxes - 1>();
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t orr[32];
            tmem_ld_x32(tO + cb * 64 + h * 32, orr);
            if (MERGE) {
              uint32_t o1[32];
              tmem_ld_x32(lane_base + C::kOCol + D + cb * 64 + h * 32, o1);  // O_1
#pragma unroll
              for (int i = 0; i < 32; ++i)
                orr[i] = __float_as_uint(
                    fmaf(__uint_as_float(o1[i]), w1, __uint_as_float(orr[i]) * w0));
            }
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const int c = h * 4 + c4;
              uint32_t w4[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                w4[i] = pack2<ET != kF16>(__uint_as_float(orr[c4 * 8 + 2 * i]) * inv_l,
                                          __uint_as_float(orr[c4 * 8 + 2 * i + 1]) * inv_l);
              st_shared_v4(box + lane * 128 + ((c ^ (lane & 7)) << 4), w4[0], w4[1], w4[2], w4[3]);
            }
          }
          fence_proxy_async_smem();  // this lane's writes, visible to the TMA engine
          __syncwarp();
          if (lane == 0) {
            if (row0 < S) tma_store_3d(&tm_o, box, cb * 64, row0, ue.bh);  // rows >= S clipped
            bulk_commit_group();
          }
        }
      };
      if (KSPLIT && kse)
        store_o(BoolTag<KSPLIT>{});
      else
        store_o(BoolTag<false>{});
      // O_t (and O_1 after a merge) has left TMEM: the next unit's first P V
      // may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl.o_empty[t]);
        if (kse) mbar_arrive(&ctl.o_empty[1]);
      }
      if (row < S)
        p.lse[static_cast<size_t>(ue.bh) * S + row] =
            (m + lg2(l) - shift) * 0.69314718055994530942f;
    }
    // every TMA store of O has completed before the block may exit
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  }

  // ---- teardown: every role has drained its asynchronous work
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Dynamic shared memory above 48 KB is opted into once per device.  Internal
// linkage keeps the flags private to each loaded copy of the library (a
// function-local static of an inline template would otherwise become one
// process-wide symbol shared by every copy).
template <int D, int ET, bool CAUSAL, bool KSPLIT = false>
static cudaError_t launch_fmha_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, const FwdParams& prm, unsigned grid,
                            cudaStream_t stream) {
  auto kern = fmha_fwd_kernel<D, ET, CAUSAL, KSPLIT>;
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> opted_in[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices || !opted_in[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<D, ET, CAUSAL>::kSmemBytes);
    if (e != cudaSuccess) return e;
    // The register split hands out exactly the registers the block is
    // launched with; a build that gave the kernel another count would leave
    // setmaxnreg.inc waiting for registers that do not exist, so refuse it.
    if (Cfg<D, ET, CAUSAL>::kRegSplit) {
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != kRegLaunch) return cudaErrorInvalidConfiguration;
    }
    if (dev >= 0 && dev < kMaxDevices) opted_in[dev].store(true, std::memory_order_release);
  }
  kern<<<grid, Cfg<D, ET, CAUSAL>::kThreads, Cfg<D, ET, CAUSAL>::kSmemBytes, stream>>>(tq, tk, tv, to, prm);
  return cudaGetLastError();
}

}  // namespace wsa
