// fa_prefill.cuh -- fused attention forward (prefill) kernel for sm_103a.
//
// A persistent CTA per SM works through items: an item is 256 query rows of
// one (batch, head), as two ping-pong stages of 128 rows (the two-Q-tile
// ping-pong of the B300 G5 page, V21), streamed over the keys in tiles of
// 128.  Items are claimed at run time, heaviest first under causal masking
// (LPT, "The FA5090 Optimization Journey" section 2.7).  Warp roles (16
// warps, 512 threads):
//
//   warps 0-3   softmax, stage 0   one thread per query row (TMEM lane); also
//                                  rescales O when a row's reference max moves
//   warps 4-7   softmax, stage 1
//   warps 8-11  epilogue: O / l to 16 bits, staged in smem, stored by TMA
//               (in the correction-warpgroup form, kCorrWG, they also rescale
//               O for the tiles the softmax warps hand over)
//   warp  12    tcgen05.mma issue (whole warp, one elected lane) + TMEM alloc
//   warp  13    TMA producer (one thread) and item scheduler: claims items,
//               loads each item's Q and then its K/V tiles into a ring; when
//               it runs out of items it lets the next grid on the stream
//               start (programmatic dependent launch)
//   warps 14-15 idle (they complete the fourth warpgroup)
// setmaxnreg gives the softmax warpgroups 176 registers per thread, the
// epilogue 72 and the MMA / producer warpgroup 88.
//
// Launched to overlap the previous grid (PrefillParams::overlap_prev), every
// thread that writes global memory (LSE by the softmax warps, O and the
// split partials by the epilogue warps) first waits for that grid; reads of
// Q, K and V start at once.
//
// Tensor memory (512 columns x 128 lanes): S_s = Q_s K^T at columns s*128
// (fp32), O_s at 256 + s*D (fp32).  Softmax writes P_s as packed 16-bit
// pairs over the first 64 columns of S_s, and PV reads its A operand from
// there (P never touches shared memory).  The next S_s overwrites P_s; the
// MMA warp's elected lane issues PV_s(j) before QK_s(j+1) and the tensor
// core executes one thread's MMAs in issue order.
//
// Issue order of the tensor core: QK_0(0) QK_1(0), then per key tile j
//     PV_0(j)  QK_0(j+1)  PV_1(j)  QK_1(j+1)
// so that each softmax warpgroup has two GEMMs of the other stage to hide
// behind (the aim of the ping-pong on the G5 page); at an item's last tile
// the next item's QK_s(0) take the place of QK_s(j+1), so the tensor core
// goes on while the epilogue warps store the finished item.  K and V occupy
// separate slots of one ring with their own full/empty barriers (the
// decoupled K/V loads of G5 V26), and stage 0's PV never waits for stage 1
// (the PV0 barrier of V30).
//
// Softmax works in the log2 domain with the scale folded into one FFMA
// before ex2 (G5 V33 "log2exp2"; FA5090 section 2.6): t = s*scale*log2(e),
// p = 2^(t - m) against a per-row reference max m.  m is raised only when
// the tile's max exceeds it by more than tau (log2 units); then
// alpha = 2^(m_old - m_new) and the softmax warp multiplies its rows of O by
// alpha before releasing the next PV, skipping it when all 32 rows of the
// warp have alpha == 1 (a warp-uniform vote; the correction merged into the
// softmax warpgroup, G5 V25).  tau = 0 is the identity-only rescale skip of
// the FA5090 page (sections 2.6 and 2.8: skip exactly when the max did not
// change); tau = 8 is FA4's lazy rescale that the same page describes in
// section 3 (p stays <= 2^8, and the final division by l, accumulated
// against the same m, makes the result exact either way).
//
// Causal (bottom-right): key tiles past the last row's diagonal are never
// loaded or computed (FA5090 section 2.7, causal block skip); only tiles that
// cross the diagonal (or the ragged end of the keys) are masked (section
// 2.8, diagonal-only masking).
//
// Every mbarrier wait is bounded by a watchdog; a wait that runs out sets a
// shared abort flag and the device status word, every role leaves its loop,
// in-flight TMA loads and MMAs are drained, TMEM is freed and the CTA exits.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// Items in flight between the producer, which claims them, and the other
// roles, which take them in the same order.
constexpr int kItemRing = 4;
// Warps that take every item: the MMA warp, 8 softmax warps, 4 epilogue warps.
constexpr int kItemTakers = 13;

template <int D>
struct PrefillLayout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kQBytes = kBM * D * 2;    // one stage of Q
  static constexpr int kKVBytes = kBN * D * 2;   // one K or V tile
  static constexpr int kBox = 128 * 64 * 2;      // one TMA box (64 cols)
  static constexpr int kSlots = D == 128 ? 4 : 11;
  static constexpr int kOutWarpBytes = 32 * D * 2;  // one epilogue warp's 32 rows of O
  static constexpr int kOutBox = 32 * 64 * 2;       // one 64-column box of them
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kStages * kQBytes;
  static constexpr int kOffOut = kOffKV + kSlots * kKVBytes;
  static constexpr int kOffMisc = kOffOut + 4 * kOutWarpBytes;
  // mbarrier indices
  static constexpr int Q_FULL = 0;    // [2] Q_s of the current item landed
  static constexpr int Q_EMPTY = 2;   // [2] the item's last QK_s is done: Q_s reusable
  static constexpr int S_FULL = 4;    // [2] S_s = Q_s K^T ready
  static constexpr int PV_READY = 6;  // [2] P_s stored (and O_s rescaled)
  static constexpr int O_READY = 8;   // [2] PV_s done
  static constexpr int ML_FULL = 10;  // [2] the item's 1/l published
  static constexpr int O_FREE = 12;   // [2] the epilogue has read O_s
  static constexpr int DRAIN = 14;
  static constexpr int ITEM_FULL = 15;   // [kItemRing] next item index published
  static constexpr int ITEM_EMPTY = 19;  // [kItemRing] every role has read it
  static constexpr int KV_FULL = 23;            // [kSlots]
  static constexpr int KV_EMPTY = 23 + kSlots;  // [kSlots]
  static constexpr int kNumBars = 23 + 2 * kSlots;
  static constexpr int kOffBars = kOffMisc;
  static constexpr int kOffInvL = kOffBars + ((kNumBars * 8 + 15) / 16) * 16;
  static constexpr int kOffItems = kOffInvL + kStages * kBM * 4;
  static constexpr int kOffTmemSlot = kOffItems + kItemRing * 4;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  // [2][4] correction requests (the correction-warpgroup form): the softmax
  // warp of stage s and TMEM lane quarter q -> the epilogue warp of quarter q
  static constexpr int kOffCorrBars = kOffAbort + 4;
  static constexpr int kMiscBytes = kOffCorrBars + 8 * 8 - kOffMisc;
  static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + align
  static constexpr int kTmemCols = 512;
  static constexpr int kTmemO = 256;  // O_s at column 256 + s*D
  static_assert(kOffCorrBars % 8 == 0, "mbarrier alignment");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// One work item: 256 query rows (two stages) of one (batch, head), over the
// key tiles [t0, t0 + nT1): all of them, unless the keys are split into
// ranges (then `split` numbers the range).
template <bool kSplit>
struct ItemT {
  int bh, row0, nT0, nT1;
  static constexpr int t0 = 0, split = 0;
};
template <>
struct ItemT<true> {
  int bh, row0, nT0, nT1, t0, split;
};

// Register split between warpgroups (setmaxnreg): softmax warpgroups get
// more, the others give theirs back.  The sum over the 512 threads equals
// 512 * 128, the registers the CTA is launched with; the host checks the
// compiled register count before the first launch.
// CTA-pair kernel: 192 for each softmax warpgroup, 64 for the others.
constexpr int kRegsSoftmax = 192;
constexpr int kRegsOther = 64;
static_assert(2 * 128 * kRegsSoftmax + 2 * 128 * kRegsOther == kThreads * 128,
              "register split must equal the launch allocation");
// Single-CTA kernel: 176 for each softmax warpgroup, 72 for the epilogue
// warpgroup and 88 for the MMA / producer warpgroup.  With 64 for both of
// the latter, ptxas spilled in them (4 B stored, 68 B loaded); this split
// compiles without spills and measured 1.4 % faster on causal S4096 and
// 0.7 % on D = 64 (paired, interleaved runs).
constexpr int kRegsSoftmaxSingle = 176;
constexpr int kRegsEpilogueSingle = 72;
constexpr int kRegsControlSingle = 88;
static_assert(128 * (2 * kRegsSoftmaxSingle + kRegsEpilogueSingle + kRegsControlSingle) ==
                  kThreads * 128,
              "register split must equal the launch allocation");

struct Ctl {
  volatile uint32_t* abort;
  unsigned* status;
  unsigned long long timeout;
};

// Back-off between polls, per role.  A warp polling an mbarrier takes issue
// slots from the softmax warps that share its SM sub-partition (each
// sub-partition runs one softmax warp of each stage), and the softmax is on
// the critical path; so every role but the softmax sleeps between polls.
// The MMA warp's sleep is short (it reacts to the softmax's arrivals); the
// producer runs a ring ahead and the epilogue warps wait a whole item.
constexpr unsigned kSleepMmaNs = 32;
constexpr unsigned kSleepProducerNs = 64;
constexpr unsigned kSleepEpilogueNs = 256;

// The slow path of a wait, out of line so that the loops that wait stay
// small: try_wait suspends the thread for a short while before it reports
// "not yet"; the abort flag and the clock are checked every 8th round.
template <unsigned kSleepNs>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity,
                                       volatile uint32_t* abort_flag,
                                       unsigned* status,
                                       unsigned long long timeout) {
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if constexpr (kSleepNs > 0) __nanosleep(kSleepNs);
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 7u) == 0) {
      if (*abort_flag) return false;
      const uint64_t t = globaltimer_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > timeout) {
        *abort_flag = 1u;
        atomicExch(status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Bounded wait; false when the watchdog fired (here or in another role).
template <unsigned kSleepNs = 0>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity,
                                         const Ctl& c) {
  return mbar_try_wait(bar, parity) ||
         wait_slow<kSleepNs>(bar, parity, c.abort, c.status, c.timeout);
}

// Warp-uniform bounded wait (every lane gets the same answer).
template <unsigned kSleepNs = 0>
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity,
                                              const Ctl& c) {
  const bool ok = wait_bar<kSleepNs>(bar, parity, c);
  return __all_sync(0xffffffffu, ok);
}

// Wait used while draining after an abort: time-bounded only.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity,
                                           unsigned long long timeout) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout) return;
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a,
                                             uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a),
               "r"(b), "r"(c), "r"(d)
               : "memory");
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Number of key tiles a stage whose first query row is `row_first` needs.
__device__ __forceinline__ int stage_tiles(int row_first, int Sq, int Skv,
                                           int causal) {
  const int n_all = (Skv + kBN - 1) / kBN;
  if (!causal) return n_all;
  const int last_key = row_first + kBM - 1 + (Skv - Sq);
  if (last_key < 0) return 0;
  return min(n_all, last_key / kBN + 1);
}

// Item idx (0 <= idx < n_items): heaviest first under causal LPT; with
// split keys, the key ranges of one query tile are consecutive items.
template <bool kSplit>
__device__ __forceinline__ ItemT<kSplit> get_item(const PrefillParams& p, int idx) {
  ItemT<kSplit> it;
  int qi = idx;
  if constexpr (kSplit) {
    qi = idx / p.n_splits;
    it.split = idx - qi * p.n_splits;
  }
  int qtile;
  if (p.causal && p.lpt) {
    qtile = p.n_qtiles - 1 - qi / p.BH;
    it.bh = qi % p.BH;
  } else {
    qtile = qi % p.n_qtiles;
    it.bh = qi / p.n_qtiles;
  }
  it.row0 = qtile * kRowsPerCta;
  it.nT0 = stage_tiles(it.row0, p.Sq, p.Skv, p.causal);
  it.nT1 = stage_tiles(it.row0 + kBM, p.Sq, p.Skv, p.causal);
  if constexpr (kSplit) {
    it.t0 = it.split * p.tiles_per_split;
    const int t1 = it.t0 + p.tiles_per_split;
    it.nT0 = max(0, min(it.nT0, t1) - it.t0);
    it.nT1 = max(0, min(it.nT1, t1) - it.t0);
  }
  return it;
}

// Claims the next item for this CTA: a CTA starts with item blockIdx.x and
// then takes items gridDim.x, gridDim.x + 1, ... in the order SMs free up
// (with the heaviest-first numbering, the greedy LPT schedule).  One
// fetch-and-add on the launch's scheduler slot, which starts at zero.
// Returns -1 once every item is claimed.
__device__ __forceinline__ int claim_item(const PrefillParams& p) {
  const unsigned long long ticket = atomicAdd(p.sched, 1ull);
  const unsigned long long idx = gridDim.x + ticket;
  return idx < static_cast<unsigned long long>(p.n_items) ? static_cast<int>(idx) : -1;
}

// The k-th item of this CTA (-1: no more), as published by the producer.
template <unsigned kSleepNs>
__device__ __forceinline__ int take_item(const volatile int* ring, uint32_t full,
                                         uint32_t empty, uint32_t k, const Ctl& c,
                                         bool& ok) {
  const uint32_t slot = k % kItemRing;
  ok = wait_bar_warp<kSleepNs>(full + 8u * slot, (k / kItemRing) & 1, c);
  const int idx = ok ? ring[slot] : -1;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty + 8u * slot);
  return idx;
}

// One key tile of one stage's softmax, for this thread's query row (its TMEM
// lane): load S (128 fp32 columns at tS) into registers, mask keys past the
// ragged end and past the causal diagonal (key0: the tile's first key;
// stage_row0: the first of the 128 rows that share this TMEM quarter's tile;
// row_g: this thread's row), raise the reference max m past the threshold,
// write P = 2^(c*s - m) as packed 16-bit pairs over the first 64 columns of S,
// update the row sum l, and rescale this warp's rows of O (D columns at tO)
// when one of them moved its reference max.  Ends with tcgen05.wait::st.
// kVoteFirst places the warp's vote on that rescale before the exponentials
// rather than after them: the arithmetic is the same, only the instruction
// schedule differs (measured faster for the single-CTA kernel, slower for
// the CTA-pair kernel).  kDefer leaves the rescale to a correction warp: the
// tile writes each row's alpha to column 64 of S (past P) instead, and
// returns true when the warp's rows need it (warp-uniform).
template <int D, bool BF16, bool kVoteFirst = true, bool kDefer = false>
__device__ __forceinline__ bool softmax_tile(uint32_t tS, uint32_t tO, int key0, int stage_row0,
                                             int row_g, const PrefillParams& p, bool may_rescale,
                                             float& m, float& l) {
  const int off = p.Skv - p.Sq;
  const float c = p.scale_log2;
  const float tau = p.rescale_tau;
  uint32_t sr[8][16];
#pragma unroll
  for (int cc = 0; cc < 8; cc += 2) tmem_ld32(tS + cc * 16, sr[cc], sr[cc + 1]);
  tmem_wait_ld();
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) reg_fence16(sr[cc]);

  // mask: ragged key tail, and the causal diagonal
  const bool need_mask =
      (key0 + kBN > p.Skv) || (p.causal && key0 + kBN - 1 > stage_row0 + off);
  if (need_mask) {
    int lim = p.Skv - 1 - key0;
    if (p.causal) lim = min(lim, row_g + off - key0);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc)
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (cc * 16 + e > lim) sr[cc][e] = __float_as_uint(-INFINITY);
  }
  // row max as a shallow tree: 16 independent 8-column maxima, then 3 levels
  float mx[16];
#pragma unroll
  for (int g = 0; g < 16; ++g) {
    const uint32_t* v = &sr[g >> 1][(g & 1) * 8];
    float a = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
    a = fmax3(a, __uint_as_float(v[3]), __uint_as_float(v[4]));
    a = fmax3(a, __uint_as_float(v[5]), __uint_as_float(v[6]));
    mx[g] = fmaxf(a, __uint_as_float(v[7]));
  }
  const float r0 = fmax3(mx[0], mx[1], mx[2]), r1 = fmax3(mx[3], mx[4], mx[5]);
  const float r2 = fmax3(mx[6], mx[7], mx[8]), r3 = fmax3(mx[9], mx[10], mx[11]);
  const float r4 = fmax3(mx[12], mx[13], mx[14]);
  const float t_max = fmaxf(fmax3(r0, r1, r2), fmax3(r3, r4, mx[15])) * c;
  // raise the reference max only past the threshold (m = -inf: always)
  const float m_new = t_max > m + tau ? t_max : m;
  const float m_use = m_new == -INFINITY ? 0.f : m_new;
  const float alpha = m_new == m ? 1.f : ex2_approx(m - m_use);
  const float neg_m = -m_use;
  // O *= alpha when a row of this warp moved its reference max (rare: tau
  // keeps it still).  The caller guarantees that the previous PV into O has
  // completed (the kernels commit S_FULL after it) and passes may_rescale =
  // false on an item's first tile, which has no O to rescale.
  bool rescale = false;
  if constexpr (kVoteFirst)
    rescale = may_rescale && (p.always_rescale || __any_sync(0xffffffffu, alpha != 1.f));
  // p = 2^(s*c - m) in four 32-column pieces: the argument as packed
  // fp32x2 FMAs, the row sum as packed fp32x2 adds; each piece is packed
  // to 16-bit pairs and stored over the first 64 columns of S_s (every S
  // value of this row is already in registers) while the next piece's
  // exponentials run
  float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    uint32_t pk[16];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int col = h * 32 + q * 4;
      uint32_t* v = &sr[col >> 4][col & 15];
      float x0, x1, x2, x3;
      ffma2(x0, x1, __uint_as_float(v[0]), __uint_as_float(v[1]), c, c, neg_m, neg_m);
      ffma2(x2, x3, __uint_as_float(v[2]), __uint_as_float(v[3]), c, c, neg_m, neg_m);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
      const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
      fadd2(l0, l1, l0, l1, p0, p1);
      fadd2(l2, l3, l2, l3, p2, p3);
      pk[2 * q] = pack2<BF16>(p0, p1);
      pk[2 * q + 1] = pack2<BF16>(p2, p3);
    }
    tmem_st16(tS + h * 16, pk);
  }
  l = l * alpha + ((l0 + l1) + (l2 + l3));
  m = m_new;
  if constexpr (!kVoteFirst)
    rescale = may_rescale && (p.always_rescale || __any_sync(0xffffffffu, alpha != 1.f));
  if constexpr (kDefer) {
    // the row's S values are no longer needed: alpha for the correction warp
    if (rescale) tmem_st1(tS + 64, __float_as_uint(alpha));
  } else if (rescale) {
    // the row's S values are no longer needed: all D columns of O in one
    // tensor-memory round trip (each load-and-wait costs ~240 cycles)
    uint32_t v[D / 16][16];
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tO + cc * 32, v[2 * cc], v[2 * cc + 1]);
    tmem_wait_ld();
#pragma unroll
    for (int cc = 0; cc < D / 16; ++cc) {
      reg_fence16(v[cc]);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        v[cc][e] = __float_as_uint(__uint_as_float(v[cc][e]) * alpha);
      tmem_st16(tO + cc * 16, v[cc]);
    }
  }
  tmem_wait_st();
  return rescale;
}

// O_s *= alpha for one warp's 32 rows (the correction-warpgroup form), with
// alpha read from column 64 of S_s where the softmax warp left it: 32
// columns of O per tensor-memory round trip (the correction warp runs with
// the smaller register share).  Ends with tcgen05.wait::st.
template <int D>
__device__ __forceinline__ void correct_rows(uint32_t tS, uint32_t tO) {
  uint32_t a = tmem_ld1(tS + 64);
  tmem_wait_ld();
  asm volatile("" : "+r"(a)::"memory");
  const float alpha = __uint_as_float(a);
#pragma unroll 1
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t v[2][16];
    tmem_ld32(tO + cc * 32, v[0], v[1]);
    tmem_wait_ld();
    reg_fence16(v[0]);
    reg_fence16(v[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int e = 0; e < 16; ++e) v[h][e] = __float_as_uint(__uint_as_float(v[h][e]) * alpha);
      tmem_st16(tO + cc * 32 + h * 16, v[h]);
    }
  }
  tmem_wait_st();
}

// Poll interval of a correction warp (it watches its quarter's requests of
// both stages and its own epilogue barrier).
constexpr unsigned kSleepCorrNs = 32;

// The epilogue's staging of 32 rows x D columns of O (this warp's TMEM lane
// quarter at tO): O * inv_l rounded to 16 bits (zeros when the rows saw no
// key), written to the warp's slice of shared memory as D/64 boxes of 32 rows
// x 128 bytes, 128-byte swizzled, ready for the TMA store.
template <int D, bool BF16>
__device__ __forceinline__ void stage_o_rows(uint32_t tO, bool have_o, float inv_l,
                                             uint32_t stage_buf, int out_box_bytes, int lane) {
  // 32 columns per tensor-memory round trip (a load and its wait take ~240
  // cycles; this read gates the next item's first PV into O)
#pragma unroll 1
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t v[2][16];
    if (have_o) {
      tmem_ld32(tO + cc * 32, v[0], v[1]);
      tmem_wait_ld();
      reg_fence16(v[0]);
      reg_fence16(v[1]);
    } else {  // no visible key: O = 0
#pragma unroll
      for (int e = 0; e < 16; ++e) v[0][e] = v[1][e] = 0u;
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t* x = &v[h >> 1][(h & 1) * 8];
      const int col = cc * 32 + h * 8;  // first column of this 16-byte chunk
      const uint32_t w0 = pack2<BF16>(__uint_as_float(x[0]) * inv_l, __uint_as_float(x[1]) * inv_l);
      const uint32_t w1 = pack2<BF16>(__uint_as_float(x[2]) * inv_l, __uint_as_float(x[3]) * inv_l);
      const uint32_t w2 = pack2<BF16>(__uint_as_float(x[4]) * inv_l, __uint_as_float(x[5]) * inv_l);
      const uint32_t w3 = pack2<BF16>(__uint_as_float(x[6]) * inv_l, __uint_as_float(x[7]) * inv_l);
      const int box = col >> 6, chunk = (col & 63) >> 3;
      st_shared_v4(stage_buf + static_cast<uint32_t>(box * out_box_bytes + lane * 128 +
                                                     ((chunk ^ (lane & 7)) << 4)),
                   w0, w1, w2, w3);
    }
  }
}

// kCorrWG: the correction-warpgroup form.  The softmax warps do not rescale
// O themselves; a warp whose rows moved their reference max hands the tile to
// the epilogue warp of its TMEM lane quarter, which rescales O in tensor
// memory and makes the tile's PV_READY arrival in its place (the dedicated
// correction warpgroup of the B300 G5 page, V21).  Tiles without a rescale
// arrive on PV_READY directly, as in the merged form (G5 V25).
template <int D, bool BF16, bool kSplit, bool kCorrWG = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_prefill_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmO,
                      const PrefillParams p) {
  using L = PrefillLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + L::kOffQ;
  const uint32_t sKV = sbase + L::kOffKV;
  const uint32_t sOut = sbase + L::kOffOut;
  const uint32_t bars = sbase + L::kOffBars;
  float* inv_l_smem = reinterpret_cast<float*>(smem + L::kOffInvL);
  volatile int* item_ring = reinterpret_cast<volatile int*>(smem + L::kOffItems);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem + L::kOffAbort);
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
  auto corr_bar = [&](int s, int q) {
    return sbase + static_cast<uint32_t>(L::kOffCorrBars + 8 * (s * 4 + q));
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- setup (once per CTA; every barrier's phase runs on across items) ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::Q_FULL + s), 1);
      mbar_init(bar(L::Q_EMPTY + s), 1);
      mbar_init(bar(L::S_FULL + s), 1);
      mbar_init(bar(L::PV_READY + s), 4);  // the stage's 4 softmax warps
      mbar_init(bar(L::O_READY + s), 1);
      mbar_init(bar(L::ML_FULL + s), 4);
      mbar_init(bar(L::O_FREE + s), 4);    // the 4 epilogue warps
    }
    mbar_init(bar(L::DRAIN), 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(bar(L::ITEM_FULL + i), 1);
      mbar_init(bar(L::ITEM_EMPTY + i), kItemTakers);
    }
    for (int i = 0; i < L::kSlots; ++i) {
      mbar_init(bar(L::KV_FULL + i), 1);
      mbar_init(bar(L::KV_EMPTY + i), 1);
    }
    if constexpr (kCorrWG)
      for (int i = 0; i < 8; ++i) mbar_init(corr_bar(i >> 2, i & 3), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 13 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};

  const int wg = warp >> 2;
  if (wg < 2) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmaxSingle));
  } else if (wg == 2) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsEpilogueSingle));
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControlSingle));
  }

  if (wg < 2) {
    // =========================== softmax, stage s ===========================
    const int s = wg;
    const int rq = warp & 3;                 // lane quarter of TMEM
    const int r = rq * 32 + lane;            // row within the stage
    const uint32_t t_lane = static_cast<uint32_t>(rq * 32) << 16;
    const uint32_t tS = tmem + t_lane + static_cast<uint32_t>(s * kBN);
    const uint32_t tO = tmem + t_lane + static_cast<uint32_t>(L::kTmemO + s * D);
    uint32_t n_s = 0;  // tiles of this stage so far (S_FULL / O_READY phase)
    bool ok = true;
    bool dep_wait = p.overlap_prev != 0;  // before the first global write

#pragma unroll 1
    for (uint32_t k = 0; ok; ++k) {
      const int idx = take_item<0>(item_ring, bar(L::ITEM_FULL), bar(L::ITEM_EMPTY), k, ctl, ok);
      if (!ok || idx < 0) break;
      const ItemT<kSplit> it = get_item<kSplit>(p, idx);
      const int nT = s == 0 ? it.nT0 : it.nT1;
      const int stage_row0 = it.row0 + s * kBM;
      const int row_g = stage_row0 + r;        // query row
      float m = -INFINITY;  // reference max of c*s (log2 units)
      float l = 0.f;        // running sum of 2^(c*s - m)

#pragma unroll 1
      for (int j = 0; j < nT; ++j, ++n_s) {
        if (!wait_bar_warp(bar(L::S_FULL + s), n_s & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        const bool defer = softmax_tile<D, BF16, true, kCorrWG>(
            tS, tO, (it.t0 + j) * kBN, stage_row0, row_g, p, j > 0, m, l);
        tc_fence_before();
        __syncwarp();
        // a rescale request goes to this quarter's correction warp, which
        // arrives on PV_READY_s in this warp's place
        if (lane == 0) mbar_arrive(kCorrWG && defer ? corr_bar(s, rq) : bar(L::PV_READY + s));
      }
      if (!ok) break;

      // end of the item: LSE straight to global, 1/l to the epilogue warps
      // once the item's last PV_s has completed (then O_s is final)
      if (dep_wait) {
        grid_dependency_wait();
        dep_wait = false;
      }
      if (row_g < p.Sq) {
        const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        if constexpr (kSplit)
          p.part_lse[(static_cast<size_t>(it.split) * p.BH + it.bh) * p.Sq + row_g] = lse;
        else
          p.lse[static_cast<size_t>(it.bh) * p.Sq + row_g] = lse;
      }
      if (nT > 0) {
        if (!wait_bar_warp(bar(L::O_READY + s), (n_s - 1) & 1, ctl)) { ok = false; break; }
        inv_l_smem[s * kBM + r] = l > 0.f ? 1.f / l : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::ML_FULL + s));
      }
    }
    __syncwarp();
  } else if (wg == 2) {
    // =============================== epilogue ===============================
    // Per item and stage: O_s * (1/l), rounded to 16 bits, staged in this
    // warp's 32-row slice of shared memory and written by TMA.  The warp
    // arrives on O_FREE_s as soon as it has read O_s out of tensor memory,
    // which lets the next item's first PV_s overwrite it.
    const int rq = warp & 3;
    const int r = rq * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(rq * 32) << 16;
    const uint32_t stage_buf = sOut + static_cast<uint32_t>(rq * L::kOutWarpBytes);
    uint32_t n_t0 = 0, n_t1 = 0;  // tiles of stage s so far (O_READY phase)
    uint32_t n_e0 = 0, n_e1 = 0;  // ML_FULL phases
    uint32_t n_c[2] = {0u, 0u};   // correction requests served, per stage
    bool ok = true;
    bool dep_wait = p.overlap_prev != 0;  // before the first global write
    // The wait for an item's 1/l (the end of its stage): in the
    // correction-warpgroup form it also serves this quarter's correction
    // requests of both stages, polling without suspending; bounded by the
    // watchdog like every other wait.
    auto epi_wait = [&](uint32_t b, uint32_t par) -> bool {
      if constexpr (!kCorrWG) {
        return wait_bar_warp<kSleepEpilogueNs>(b, par, ctl);
      } else {
        uint64_t t0 = 0;
        for (uint32_t n = 1;; ++n) {
          if (__any_sync(0xffffffffu, mbar_test_wait(b, par))) return true;
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {
            if (__any_sync(0xffffffffu, mbar_test_wait(corr_bar(s2, rq), n_c[s2] & 1))) {
              tc_fence_after();
              correct_rows<D>(tmem + t_lane + static_cast<uint32_t>(s2 * kBN),
                              tmem + t_lane + static_cast<uint32_t>(L::kTmemO + s2 * D));
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(L::PV_READY + s2));
              ++n_c[s2];
              t0 = 0;
            }
          }
          if ((n & 7u) == 0) {
            if (*ctl.abort) return false;
            const uint64_t t = globaltimer_ns();
            if (t0 == 0) {
              t0 = t;
            } else if (t - t0 > ctl.timeout) {
              *ctl.abort = 1u;
              atomicExch(ctl.status, kStatusTimeout);
              return false;
            }
          }
          __nanosleep(kSleepCorrNs);
        }
      }
    };
#pragma unroll 1
    for (uint32_t k = 0; ok; ++k) {
      const int idx = take_item<kSleepEpilogueNs>(item_ring, bar(L::ITEM_FULL),
                                                  bar(L::ITEM_EMPTY), k, ctl, ok);
      if (!ok || idx < 0) break;
      const ItemT<kSplit> it = get_item<kSplit>(p, idx);
      if (dep_wait) {
        grid_dependency_wait();
        dep_wait = false;
      }
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        if (!ok) continue;
        const int nT = s == 0 ? it.nT0 : it.nT1;
        const bool have_o = nT > 0;
        float inv_l = 0.f;
        if (have_o) {
          uint32_t& n_t = s == 0 ? n_t0 : n_t1;
          uint32_t& n_e = s == 0 ? n_e0 : n_e1;
          n_t += static_cast<uint32_t>(nT);
          if (!epi_wait(bar(L::ML_FULL + s), n_e & 1)) { ok = false; continue; }
          ++n_e;
          inv_l = inv_l_smem[s * kBM + r];
          if (!wait_bar_warp<kSleepEpilogueNs>(bar(L::O_READY + s), (n_t - 1) & 1, ctl)) { ok = false; continue; }
          tc_fence_after();
        }
        const uint32_t tO = tmem + t_lane + static_cast<uint32_t>(L::kTmemO + s * D);
        if constexpr (kSplit) {
          // a key range: O / l of this range in fp32, one row per thread
          const int row_g = it.row0 + s * kBM + r;
          float4* prow = reinterpret_cast<float4*>(
              p.part_o + ((static_cast<size_t>(it.split) * p.BH + it.bh) * p.Sq +
                          static_cast<size_t>(row_g)) * D);
#pragma unroll 1
          for (int cc = 0; cc < D / 16; ++cc) {
            uint32_t v[16];
            if (have_o) {
              tmem_ld16(tO + cc * 16, v);
              tmem_wait_ld();
              reg_fence16(v);
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) v[e] = 0u;
            }
            if (row_g < p.Sq) {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                prow[cc * 4 + e] = make_float4(__uint_as_float(v[4 * e]) * inv_l,
                                               __uint_as_float(v[4 * e + 1]) * inv_l,
                                               __uint_as_float(v[4 * e + 2]) * inv_l,
                                               __uint_as_float(v[4 * e + 3]) * inv_l);
            }
          }
          if (have_o) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::O_FREE + s));
          }
          continue;
        }
        // the slice is free once the previous store has read it
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        stage_o_rows<D, BF16>(tO, have_o, inv_l, stage_buf, L::kOutBox, lane);
        if (have_o) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::O_FREE + s));
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int warp_row0 = it.row0 + s * kBM + rq * 32;
        if (lane == 0 && warp_row0 < p.Sq) {
#pragma unroll
          for (int box = 0; box < D / 64; ++box)
            tma_store_3d(&tmO, stage_buf + static_cast<uint32_t>(box * L::kOutBox), box * 64,
                         warp_row0, it.bh);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group0();  // every store has landed before exit
    __syncwarp();
  } else if (warp == 12) {
    // ============================== MMA issuer ==============================
    // the whole warp runs this loop in lockstep; each MMA / commit wrapper
    // elects the issuing lane itself
    {
      constexpr uint32_t kIdescQK = idesc_f16(BF16, false, false, kBM, kBN);
      constexpr uint32_t kIdescPV = idesc_f16(BF16, false, true, kBM, D);
      const uint32_t tS0 = tmem, tS1 = tmem + kBN;
      const uint32_t tO0 = tmem + L::kTmemO, tO1 = tmem + L::kTmemO + D;
      bool issued = false;

      auto slot_of = [&](int fill) { return fill % L::kSlots; };
      auto par_of = [&](int fill) { return static_cast<uint32_t>((fill / L::kSlots) & 1); };
      // QK_s with K from fill fk: one asm block, K = D, both operands K-major
      // in smem; commits S_FULL_s, and Q_EMPTY_s after the item's last QK_s
      auto qk = [&](int s, int fk, bool last_of_stage) {
        const uint64_t da = smem_desc_sw128(sQ + static_cast<uint32_t>(s * L::kQBytes), 16, 1024);
        const uint64_t db = smem_desc_sw128(sKV + static_cast<uint32_t>(slot_of(fk) * L::kKVBytes), 16, 1024);
        if constexpr (D == 128) {
          umma_f16_ss_k128(s == 0 ? tS0 : tS1, da, db, kIdescQK, 0u);
        } else {
          umma_f16_ss_k64(s == 0 ? tS0 : tS1, da, db, kIdescQK, 0u);
        }
        umma_commit(bar(L::S_FULL + s));
        if (last_of_stage) umma_commit(bar(L::Q_EMPTY + s));
      };
      // PV_s: K = 128 keys, A = P_s from tensor memory, B = V MN-major
      auto pv = [&](int s, int fv, bool acc) {
        umma_f16_ts_k128(s == 0 ? tO0 : tO1, s == 0 ? tS0 : tS1,
                         smem_desc_sw128(sKV + static_cast<uint32_t>(slot_of(fv) * L::kKVBytes),
                                         L::kBox, 1024),
                         kIdescPV, acc ? 1u : 0u);
        umma_commit(bar(L::O_READY + s));
      };
      // First QKs of an item whose Q is in buffer phase kq and whose K_0 is
      // fill f (used for the CTA's first item and after an item without keys)
      auto begin = [&](const ItemT<kSplit>& it, int kq, int f) -> bool {
        if (!wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + 0), kq & 1, ctl) ||
            !wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + 1), kq & 1, ctl))
          return false;
        if (it.nT1 > 0 && !wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(f)), par_of(f), ctl)) return false;
        tc_fence_after();
        if (it.nT0 > 0) qk(0, f, it.nT0 == 1); else umma_commit(bar(L::Q_EMPTY + 0));
        if (it.nT1 > 0) {
          qk(1, f, it.nT1 == 1);
          umma_commit(bar(L::KV_EMPTY + slot_of(f)));
        } else {
          umma_commit(bar(L::Q_EMPTY + 1));
        }
        issued = true;
        return true;
      };

      // Tensor-core order within an item: QK_0(0) QK_1(0), then per key tile
      //   PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1)
      // and at an item's last tile the next item's QK_s(0) take the place of
      // QK_s(j+1), so the tensor core moves on while this item's epilogue
      // runs; the next item's PV_s(0) also waits for O_FREE_s.
      uint32_t n_pv0 = 0, n_pv1 = 0;  // PV_s issued so far (PV_READY phase)
      uint32_t n_o0 = 0, n_o1 = 0;    // items so far with a PV_s (O_FREE phase)
      int kq = 0;                     // items begun (Q_FULL phase)
      int fK = 0;                     // fill of the current item's K_0
      bool ok = true;
      const int first = take_item<kSleepMmaNs>(item_ring, bar(L::ITEM_FULL),
                                               bar(L::ITEM_EMPTY), 0, ctl, ok);
      ItemT<kSplit> cur = first >= 0 ? get_item<kSplit>(p, first) : ItemT<kSplit>{0, 0, 0, 0};
      if (ok && first >= 0) ok = begin(cur, 0, 0);
      else ok = false;
#pragma unroll 1
      while (ok) {
        // the next item is taken at this item's last key tile, once the
        // producer has claimed it (it does so after the last K/V fill)
        bool taken = false, has_next = false;
        ItemT<kSplit> nxt{0, 0, 0, 0};
        auto take_next = [&]() {
          if (taken) return;
          taken = true;
          const int nidx = take_item<kSleepMmaNs>(item_ring, bar(L::ITEM_FULL),
                                                  bar(L::ITEM_EMPTY), kq + 1, ctl, ok);
          has_next = ok && nidx >= 0;
          if (has_next) nxt = get_item<kSplit>(p, nidx);
        };
        const int fN = fK + 2 * cur.nT1;  // the next item's K_0
#pragma unroll 1
        for (int j = 0; j < cur.nT1; ++j) {
          const bool last = j + 1 == cur.nT1;
          if (last) {
            take_next();
            if (!ok) break;
          }
          const int fv = fK + 2 * j + 1, fk1 = fK + 2 * j + 2;
          // V_j and PV_READY_0 first, probed together (usually both are
          // complete; the bounded waits only when one is not); K_(j+1) only
          // once PV_0(j) is issued, so that its wait is off the path from
          // the softmax's arrival to the next PV
          bool rdy = mbar_try_wait(bar(L::KV_FULL + slot_of(fv)), par_of(fv));
          if (j < cur.nT0) rdy &= mbar_try_wait(bar(L::PV_READY + 0), n_pv0 & 1);
          if (!__all_sync(0xffffffffu, rdy)) {
            if (!wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(fv)), par_of(fv), ctl)) { ok = false; break; }
            if (j < cur.nT0 && !wait_bar_warp<kSleepMmaNs>(bar(L::PV_READY + 0), n_pv0 & 1, ctl)) { ok = false; break; }
          }
          if (j < cur.nT0) {  // PV_0(j), then QK_0 over P_0(j)
            if (j == 0 && n_o0 > 0 && !wait_bar_warp<kSleepMmaNs>(bar(L::O_FREE + 0), (n_o0 - 1) & 1, ctl)) {
              ok = false;
              break;
            }
            ++n_pv0;
            tc_fence_after();
            pv(0, fv, j > 0);
          }
          if (!last && !wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(fk1)), par_of(fk1), ctl)) {
            ok = false;
            break;
          }
          if (!last) {
            if (j + 1 < cur.nT0) qk(0, fk1, j + 2 == cur.nT0);
          } else if (has_next) {
            if (!wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + 0), (kq + 1) & 1, ctl)) { ok = false; break; }
            if (nxt.nT1 > 0 && !wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(fN)), par_of(fN), ctl)) {
              ok = false;
              break;
            }
            tc_fence_after();
            if (nxt.nT0 > 0) qk(0, fN, nxt.nT0 == 1); else umma_commit(bar(L::Q_EMPTY + 0));
          }
          // PV_1(j), then QK_1 over P_1(j)
          if (!wait_bar_warp<kSleepMmaNs>(bar(L::PV_READY + 1), n_pv1 & 1, ctl)) { ok = false; break; }
          if (j == 0 && n_o1 > 0 && !wait_bar_warp<kSleepMmaNs>(bar(L::O_FREE + 1), (n_o1 - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          ++n_pv1;
          tc_fence_after();
          pv(1, fv, j > 0);
          umma_commit(bar(L::KV_EMPTY + slot_of(fv)));
          if (!last) {
            qk(1, fk1, j + 2 == cur.nT1);
            umma_commit(bar(L::KV_EMPTY + slot_of(fk1)));
          } else if (has_next) {
            if (!wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + 1), (kq + 1) & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            if (nxt.nT1 > 0) {
              qk(1, fN, nxt.nT1 == 1);
              umma_commit(bar(L::KV_EMPTY + slot_of(fN)));
            } else {
              umma_commit(bar(L::Q_EMPTY + 1));
            }
          }
        }
        if (ok) take_next();  // an item without key tiles
        if (!ok || !has_next) break;
        if (cur.nT0 > 0) ++n_o0;
        if (cur.nT1 > 0) ++n_o1;
        if (cur.nT1 == 0) ok = begin(nxt, kq + 1, fN);  // no tile above began it
        ++kq;
        cur = nxt;
        fK = fN;
      }
      if (issued) {  // every MMA issued so far completes before TMEM is freed
        umma_commit(bar(L::DRAIN));
        wait_drain(bar(L::DRAIN), 0, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 13) {
    // ============================== TMA producer =============================
    // Per item: Q_0, K_0, Q_1, V_0, then K_j V_j.  The Q of the next item
    // waits for the current item's last QK on that stage, the K/V ring for
    // the tiles of the previous round of the ring.
    if (lane == 0) {
      int fill = 0;
      int last_fill[L::kSlots];
#pragma unroll
      for (int i = 0; i < L::kSlots; ++i) last_fill[i] = -1;
      int nq[2] = {0, 0};  // Q loads issued per stage
      bool ok = true;
      auto load_q = [&](const ItemT<kSplit>& it, int s) -> bool {
        if (nq[s] > 0 && !wait_bar<kSleepProducerNs>(bar(L::Q_EMPTY + s), (nq[s] - 1) & 1, ctl)) return false;
        mbar_arrive_expect_tx(bar(L::Q_FULL + s), L::kQBytes);
#pragma unroll
        for (int box = 0; box < D / 64; ++box)
          tma_load_3d(sQ + static_cast<uint32_t>(s * L::kQBytes + box * L::kBox), &tmQ,
                      bar(L::Q_FULL + s), box * 64, it.row0 + s * kBM, it.bh);
        ++nq[s];
        return true;
      };
      auto load_kv = [&](const ItemT<kSplit>& it, int kv, int j) -> bool {
        const int slot = fill % L::kSlots;
        const uint32_t par = static_cast<uint32_t>(((fill / L::kSlots) & 1) ^ 1);
        if (!wait_bar<kSleepProducerNs>(bar(L::KV_EMPTY + slot), par, ctl)) return false;
        if (p.test_stall && fill == 2) {  // test hook: withhold the first item's K_1
          ++fill;
          return true;
        }
        mbar_arrive_expect_tx(bar(L::KV_FULL + slot), L::kKVBytes);
        const CUtensorMap* tm = kv == 0 ? &tmK : &tmV;
#pragma unroll
        for (int box = 0; box < D / 64; ++box)
          tma_load_3d(sKV + static_cast<uint32_t>(slot * L::kKVBytes + box * L::kBox), tm,
                      bar(L::KV_FULL + slot), box * 64, (it.t0 + j) * kBN, it.bh);
        last_fill[slot] = fill;
        ++fill;
        return true;
      };
      int idx = static_cast<int>(blockIdx.x);  // the grid never exceeds the items
#pragma unroll 1
      for (uint32_t k = 0; ok; ++k) {
        // publish item k (or the end) once every role has taken item k - 4
        const uint32_t slot = k % kItemRing;
        if (k >= kItemRing &&
            !wait_bar<kSleepProducerNs>(bar(L::ITEM_EMPTY + slot), (k / kItemRing - 1) & 1, ctl)) {
          ok = false;
          break;
        }
        item_ring[slot] = idx;
        mbar_arrive(bar(L::ITEM_FULL + slot));
        if (idx < 0) break;
        const ItemT<kSplit> it = get_item<kSplit>(p, idx);
        ok = load_q(it, 0);
#pragma unroll 1
        for (int j = 0; ok && j < it.nT1; ++j) {
          ok = load_kv(it, 0, j);
          if (ok && j == 0) ok = load_q(it, 1);
          if (ok) ok = load_kv(it, 1, j);
        }
        if (ok && it.nT1 == 0) ok = load_q(it, 1);
        idx = claim_item(p);
        if (idx < 0) grid_launch_dependents();  // the next grid may take the SMs
      }
      // drain: every load issued lands before shared memory goes away
#pragma unroll
      for (int s = 0; s < 2; ++s)
        if (nq[s] > 0) wait_drain(bar(L::Q_FULL + s), (nq[s] - 1) & 1, p.timeout_ns);
#pragma unroll 1
      for (int i = 0; i < L::kSlots; ++i)
        if (last_fill[i] >= 0)
          wait_drain(bar(L::KV_FULL + i), static_cast<uint32_t>((last_fill[i] / L::kSlots) & 1),
                     p.timeout_ns);
    }
    __syncwarp();
  }

  // ---- teardown ----
  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  if (threadIdx.x == 0) {
    // the launch's last CTA clears the scheduler slot (claims are over: a
    // CTA claims only from its producer, which has finished)
    __threadfence();
    if (atomicAdd(&p.sched[1], 1ull) == gridDim.x - 1) {
      p.sched[0] = 0ull;
      p.sched[1] = 0ull;
      __threadfence();
    }
  }
}

}  // namespace fa
