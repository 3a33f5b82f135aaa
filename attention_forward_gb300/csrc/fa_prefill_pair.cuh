// fa_prefill_pair.cuh -- the fused attention forward (prefill) kernel run by
// CTA pairs: a cluster of two CTAs on two SMs whose tensor cores work as one
// (tcgen05 .cta_group::2, M = 256).  Head dimension 128, whole key range.
//
// A pair item is 512 query rows of one (batch, head): two ping-pong stages of
// 256 rows, each split between the CTAs (rank r holds rows 128*r .. 128*r+127
// of the stage).  One MMA of the leader CTA (rank 0) computes a stage's
// S = Q K^T for all 256 rows, with A = Q from both CTAs' shared memory and
// B = K split by keys (rank r loads keys 64*r .. 64*r+63 of each tile); each
// CTA's tensor memory receives S for its own 128 rows.  PV reads P from both
// CTAs' tensor memory and V split by columns (rank r loads columns
// 64*r .. 64*r+63).  Each CTA loads only its half of every K/V tile, so the
// pair reads each tile from L2 once for 512 query rows.  Two cooperating
// CTAs in a cluster are the direction the B300 G5 page ("Flash Attention
// CUDA Kernel optimisation: from 56 to 986 TFLOPS on B300") names at its end
// (section "next steps"); the per-CTA softmax, correction, epilogue and
// scheduling are those of the single-CTA kernel in fa_prefill.cuh (whose
// helpers this file uses).
//
// Roles per CTA (16 warps): softmax 0-7 (stage = warp / 4), epilogue 8-11
// (also the correction warps in the kCorrWG form), warp 12 allocates tensor
// memory for the pair and, in the leader only, issues every MMA, warp 13
// loads this CTA's operands (in the leader it also claims items and
// publishes them to both CTAs; each CTA lets the next grid on the stream
// start once it has no item left, and with overlap_prev waits for the
// previous grid before its first global write, as fa_prefill_kernel does).  Barriers the MMA waits on
// live in the leader and count arrivals from both CTAs; the MMA's commits
// arrive in both CTAs (multicast); the follower's loads signal the leader's
// barriers.
//
// Tail split (non-causal): when the items leave the last round of pairs
// partly idle, the host numbers the last items' key quarters as items of
// their own, so that the last round takes a quarter of an item's time per
// step.  A quarter's softmax warps write its rows' O / l and LSE in fp32 and
// count themselves in; the last of the four merges the rows with LSE weights
// (pair_tail_quarter).  Nothing waits for another quarter.
#pragma once
#include "fa_prefill.cuh"

namespace fa {

constexpr int kPairRows = 512;       // query rows per pair item
constexpr int kPairStageRows = 256;  // per stage, 128 in each CTA
// Takers of each item, both CTAs: leader MMA + 8 softmax + 4 epilogue warps,
// follower 8 softmax + 4 epilogue + producer warps.
constexpr int kPairTakers = 26;

struct PairLayout {
  static constexpr int D = 128;
  static constexpr int kQBytes = kBM * D * 2;   // one stage of this CTA's Q (32 KB)
  static constexpr int kBox = 128 * 64 * 2;     // 128 rows x 64 columns
  static constexpr int kKBox = 64 * 64 * 2;     // 64 keys x 64 columns
  static constexpr int kHalfBytes = 16384;      // this CTA's half of a K or V tile
  static constexpr int kSlots = 8;
  static constexpr int kOutWarpBytes = 32 * D * 2;
  static constexpr int kOutBox = 32 * 64 * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kStages * kQBytes;
  static constexpr int kOffOut = kOffKV + kSlots * kHalfBytes;
  static constexpr int kOffMisc = kOffOut + 4 * kOutWarpBytes;
  // mbarrier indices (L: used in the leader only; B: in both CTAs)
  static constexpr int Q_FULL = 0;     // [2] L: both CTAs' Q_s landed
  static constexpr int Q_EMPTY = 2;    // [2] B: the item's last QK_s is done
  static constexpr int S_FULL = 4;     // [2] B: S_s ready
  static constexpr int PV_READY = 6;   // [2] L: P_s stored in both CTAs (8 warps)
  static constexpr int O_READY = 8;    // [2] B: PV_s done
  static constexpr int ML_FULL = 10;   // [2] B: the item's 1/l published (local)
  static constexpr int O_FREE = 12;    // [2] L: both CTAs' epilogues read O_s (8 warps)
  static constexpr int DRAIN = 14;     // L
  static constexpr int ITEM_FULL = 15;   // [kItemRing] B: item published
  static constexpr int ITEM_EMPTY = 19;  // [kItemRing] L: every taker of both CTAs read it
  static constexpr int KV_FULL = 23;             // [kSlots] L: both halves landed
  static constexpr int KV_EMPTY = 23 + kSlots;   // [kSlots] B: the MMAs that read it are done
  static constexpr int kNumBars = 23 + 2 * kSlots;
  static constexpr int kOffBars = kOffMisc;
  static constexpr int kOffInvL = kOffBars + ((kNumBars * 8 + 15) / 16) * 16;
  static constexpr int kOffItems = kOffInvL + kStages * kBM * 4;
  static constexpr int kOffTmemSlot = kOffItems + kItemRing * 4;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kOffCorrBars = kOffAbort + 4;  // [2][4] L/B: local requests
  static constexpr int kMiscBytes = kOffCorrBars + 8 * 8 - kOffMisc;
  static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + align
  static constexpr int kTmemCols = 512;
  static constexpr int kTmemO = 256;
  static_assert(kOffCorrBars % 8 == 0, "mbarrier alignment");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// One pair item: 512 query rows of one (batch, head) over key tiles
// [t0, t0 + nT1).  The tail-split form also numbers the quarters.
template <bool kTail>
struct PairItemT {
  int bh, row0, nT0, nT1;
  static constexpr int t0 = 0, part = -1, group = 0;
};
template <>
struct PairItemT<true> {
  int bh, row0, nT0, nT1;
  int t0 = 0;     // first key tile (a quarter of a split item)
  int part = -1;  // >= 0: partial index of a quarter (fp32 O / l and LSE to the workspace)
  int group = 0;  // the split item's index among the split ones
};
using PairItem = PairItemT<false>;

// Key quarters of a split item: quarter r covers key tiles
// [r * n / 4, (r + 1) * n / 4), never empty for n >= 4.
constexpr int kTailSplits = 4;

// Key tiles a 256-row stage whose first query row is `row_first` needs.
__device__ __forceinline__ int pair_stage_tiles(int row_first, int Sq, int Skv, int causal) {
  const int n_all = (Skv + kBN - 1) / kBN;
  if (!causal) return n_all;
  const int last_key = row_first + kPairStageRows - 1 + (Skv - Sq);
  if (last_key < 0) return 0;
  return min(n_all, last_key / kBN + 1);
}

// Pair item idx: heaviest first under causal LPT; with kTail, the last
// 4 * tail_items indices are the key quarters of the last tail_items items
// (non-causal launches only).
template <bool kTail>
__device__ __forceinline__ PairItemT<kTail> get_pair_item(const PrefillParams& p, int idx) {
  PairItemT<kTail> it;
  int part = -1, quarter = 0;
  const int tail_first = p.n_items - kTailSplits * p.tail_items;
  if (kTail && p.tail_items > 0 && idx >= tail_first) {
    part = idx - tail_first;
    quarter = part % kTailSplits;
    idx = tail_first + part / kTailSplits;
  }
  int qtile;
  if (p.causal && p.lpt) {
    qtile = p.n_qtiles - 1 - idx / p.BH;
    it.bh = idx % p.BH;
  } else {
    qtile = idx % p.n_qtiles;
    it.bh = idx / p.n_qtiles;
  }
  it.row0 = qtile * kPairRows;
  it.nT0 = pair_stage_tiles(it.row0, p.Sq, p.Skv, p.causal);
  it.nT1 = pair_stage_tiles(it.row0 + kPairStageRows, p.Sq, p.Skv, p.causal);
  if constexpr (kTail) {
    if (part >= 0) {  // non-causal: both stages have the same key tiles
      const int n = it.nT1;
      it.t0 = quarter * n / kTailSplits;
      it.nT0 = it.nT1 = (quarter + 1) * n / kTailSplits - it.t0;
      it.part = part;
      it.group = part / kTailSplits;
    }
  }
  return it;
}

// A warp's arrival at its 32 rows of a split item: returns how many of the
// item's quarters arrived before it (3: this warp merges).  The counter holds
// the launch's epoch above its low byte, so a count left by an earlier launch
// (or an aborted one) reads as zero.  The first compare-and-swap guesses the
// value a completed previous launch leaves (its epoch, four arrivals); each
// failure returns the value to try next and means another arrival landed, so
// the loop ends within four rounds (-1 only as a guard).
__device__ __forceinline__ int tail_arrive(unsigned long long* c, unsigned epoch) {
  unsigned long long old =
      epoch > 1u ? (static_cast<unsigned long long>(epoch - 1u) << 8) | kTailSplits : 0ull;
#pragma unroll 1
  for (int i = 0; i < 64; ++i) {
    const unsigned cnt = (old >> 8) == epoch ? static_cast<unsigned>(old & 0xffull) : 0u;
    const unsigned long long nv = (static_cast<unsigned long long>(epoch) << 8) | (cnt + 1u);
    const unsigned long long prev = atomicCAS(c, old, nv);
    if (prev == old) return static_cast<int>(cnt);
    old = prev;
  }
  return -1;
}

// The fp32 rows of one warp (32 rows of one stage and CTA) in one quarter of
// a split item: [item][quarter][stage][rank][warp] units of 32 x 128 floats,
// each laid out as [column / 4][row][4] so that a warp's 16-byte accesses to
// four columns of its 32 rows are 512 contiguous bytes.
__device__ __forceinline__ size_t tail_unit(int group, int quarter, int s, uint32_t rank, int rq) {
  return ((static_cast<size_t>(group * kTailSplits + quarter) * 2 + s) * 2 + rank) * 4 + rq;
}

// A softmax warp's end of a quarter item (O_s final in tensor memory): its
// rows' O / l to the workspace in fp32 and their LSE beside them, the
// tensor-memory read released to the MMA (O_FREE), then the arrival; the
// quarter that arrives last merges the four quarters' rows, in quarter
// order, into the 16-bit output and the LSE -- the key-range merge of the
// split kernel's combine (weights exp(LSE_r - LSE)).  Returns false only if
// the arrival failed (the status word then holds the error).
template <bool BF16>
__device__ __forceinline__ bool pair_tail_quarter(const PrefillParams& p,
                                                  const PairItemT<true>& it,
                                                  int s, uint32_t rank, int rq, int lane,
                                                  int row_g, uint32_t tO, float m, float l,
                                                  uint32_t o_free_leader) {
  constexpr int D = 128;
  constexpr float kLog2e = 1.4426950408889634f;
  const int quarter = it.part - it.group * kTailSplits;
  const size_t own = tail_unit(it.group, quarter, s, rank, rq);
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  float4* punit = reinterpret_cast<float4*>(p.part_o + own * 32 * D) + lane;
#pragma unroll 1
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t v[2][16];
    tmem_ld32(tO + cc * 32, v[0], v[1]);
    tmem_wait_ld();
    reg_fence16(v[0]);
    reg_fence16(v[1]);
#pragma unroll
    for (int e = 0; e < 8; ++e) {  // columns cc * 32 + 4 e .. + 3
      const uint32_t* x = &v[e >> 2][(e & 3) * 4];
      punit[(cc * 8 + e) * 32] =
          make_float4(__uint_as_float(x[0]) * inv_l, __uint_as_float(x[1]) * inv_l,
                      __uint_as_float(x[2]) * inv_l, __uint_as_float(x[3]) * inv_l);
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster_relaxed(o_free_leader);
  p.part_lse[own * 32 + lane] = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
  __threadfence();  // this lane's partial before the arrival (release)
  __syncwarp();
  int before = 0;
  if (lane == 0) {
    const size_t ctr = ((static_cast<size_t>(it.group) * 2 + s) * 2 + rank) * 4 + rq;
    before = tail_arrive(p.tail_count + ctr, p.tail_epoch);
  }
  before = __shfl_sync(0xffffffffu, before, 0);
  if (before < 0) {
    if (lane == 0) atomicExch(p.status, kStatusTimeout);
    return false;
  }
  if (before != kTailSplits - 1) return true;
  __threadfence();  // every other quarter's partial after the arrival (acquire)

  // merge this lane's row over the quarters
  const size_t u0 = tail_unit(it.group, 0, s, rank, rq);
  constexpr size_t kQStride = 16;  // units from one quarter to the next
  float ls[kTailSplits];
  float M = -INFINITY;
#pragma unroll
  for (int q = 0; q < kTailSplits; ++q) {
    ls[q] = __ldcg(p.part_lse + (u0 + q * kQStride) * 32 + lane);
    M = fmaxf(M, ls[q]);
  }
  const float M_use = M == -INFINITY ? 0.f : M;
  float w[kTailSplits];
  float W = 0.f;
#pragma unroll
  for (int q = 0; q < kTailSplits; ++q) {
    w[q] = ex2_approx((ls[q] - M_use) * kLog2e);
    W += w[q];
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  const bool row_ok = row_g < p.Sq;
  if (row_ok) p.lse[static_cast<size_t>(it.bh) * p.Sq + row_g] = W > 0.f ? M + logf(W) : -INFINITY;
  uint4* orow = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o) +
                                         (static_cast<size_t>(it.bh) * p.Sq + row_g) * D * 2);
  const float4* src = reinterpret_cast<const float4*>(p.part_o + u0 * 32 * D) + lane;
#pragma unroll 1
  for (int cc = 0; cc < D / 32; ++cc) {
    float4 a[kTailSplits][8];
#pragma unroll
    for (int q = 0; q < kTailSplits; ++q)
#pragma unroll
      for (int e = 0; e < 8; ++e)
        a[q][e] = __ldcg(src + (q * kQStride * 32 * D) / 4 + (cc * 8 + e) * 32);
#pragma unroll
    for (int h = 0; h < 4; ++h) {  // 8 columns: one 16-byte store
      float o[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = 0.f;
#pragma unroll
      for (int q = 0; q < kTailSplits; ++q) {
        const float4 x = a[q][2 * h], y = a[q][2 * h + 1];
        o[0] = fmaf(w[q], x.x, o[0]);
        o[1] = fmaf(w[q], x.y, o[1]);
        o[2] = fmaf(w[q], x.z, o[2]);
        o[3] = fmaf(w[q], x.w, o[3]);
        o[4] = fmaf(w[q], y.x, o[4]);
        o[5] = fmaf(w[q], y.y, o[5]);
        o[6] = fmaf(w[q], y.z, o[6]);
        o[7] = fmaf(w[q], y.w, o[7]);
      }
      if (row_ok)
        orow[cc * 4 + h] = make_uint4(pack2<BF16>(o[0] * inv, o[1] * inv),
                                      pack2<BF16>(o[2] * inv, o[3] * inv),
                                      pack2<BF16>(o[4] * inv, o[5] * inv),
                                      pack2<BF16>(o[6] * inv, o[7] * inv));
    }
  }
  return true;
}

// Waits on barriers that another CTA's release-arrive completes (acquire at
// cluster scope); out-of-line slow path as in wait_slow.
template <unsigned kSleepNs>
__device__ __noinline__ bool pair_wait_slow(uint32_t bar, uint32_t parity,
                                            volatile uint32_t* abort_flag, unsigned* status,
                                            unsigned long long timeout) {
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if constexpr (kSleepNs > 0) __nanosleep(kSleepNs);
    if (mbar_try_wait_cluster(bar, parity)) return true;
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

template <unsigned kSleepNs>
__device__ __forceinline__ bool pair_wait_warp(uint32_t bar, uint32_t parity, const Ctl& c) {
  const bool ok = mbar_try_wait_cluster(bar, parity) ||
                  pair_wait_slow<kSleepNs>(bar, parity, c.abort, c.status, c.timeout);
  return __all_sync(0xffffffffu, ok);
}

template <unsigned kSleepNs>
__device__ __forceinline__ bool pair_wait_one(uint32_t bar, uint32_t parity, const Ctl& c) {
  return mbar_try_wait_cluster(bar, parity) ||
         pair_wait_slow<kSleepNs>(bar, parity, c.abort, c.status, c.timeout);
}

// The k-th item of this CTA from its ring (-1: no more); the arrival that
// frees the ring slot goes to the leader's ITEM_EMPTY.  That arrival only has
// to come after this warp's read of the slot, which the leader overwrites
// once it has seen every arrival.  It is made conditional on the value read
// (an index is >= -1, never INT_MIN), so it cannot issue before the read has
// returned, and it is relaxed: a release at cluster scope cost ~1500 cycles
// here, at every item boundary of the softmax and MMA warps.
template <unsigned kSleepNs>
__device__ __forceinline__ int pair_take_item(const volatile int* ring, uint32_t full,
                                              uint32_t empty_leader_cl, uint32_t k,
                                              const Ctl& c, bool& ok) {
  const uint32_t slot = k % kItemRing;
  ok = pair_wait_warp<kSleepNs>(full + 8u * slot, (k / kItemRing) & 1, c);
  const int idx = ok ? ring[slot] : -1;
  __syncwarp();
  if ((threadIdx.x & 31) == 0 && idx != INT_MIN)
    mbar_arrive_cluster_relaxed(empty_leader_cl + 8u * slot);
  return idx;
}

// Distinct sleep values from the single-CTA kernel's, so that no out-of-line
// wait is shared between register regions of different sizes.
constexpr unsigned kPairSleepSoftmaxNs = 1;
constexpr unsigned kPairSleepMmaNs = 33;
constexpr unsigned kPairSleepProducerNs = 65;
constexpr unsigned kPairSleepEpilogueNs = 257;

// kCorrWG: the correction-warpgroup form, as in fa_prefill_kernel: a softmax
// warp whose rows moved their reference max hands the tile to the epilogue
// warp of its lane quarter (same CTA), which rescales O and makes the tile's
// PV_READY arrival on the leader in its place.  kTail: the tail split (an
// instantiation of its own, so that the other forms carry none of its code).
template <bool BF16, bool kCorrWG = false, bool kTail = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK,  // box: 64 keys
                           const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmO,
                           const PrefillParams p) {
  using L = PairLayout;
  using Item = PairItemT<kTail>;
  constexpr int D = L::D;
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
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  // the leader's barriers, as shared::cluster addresses (valid in both CTAs)
  const uint32_t bars_l = mapa_shared(bars, 0);
  auto bar_l = [&](int i) { return bars_l + 8u * static_cast<uint32_t>(i); };

  // ---- setup ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::Q_FULL + s), 1);
      mbar_init(bar(L::Q_EMPTY + s), 1);
      mbar_init(bar(L::S_FULL + s), 1);
      mbar_init(bar(L::PV_READY + s), 8);  // 4 softmax warps of the stage in each CTA
      mbar_init(bar(L::O_READY + s), 1);
      mbar_init(bar(L::ML_FULL + s), 4);
      mbar_init(bar(L::O_FREE + s), 8);    // 4 epilogue warps in each CTA
    }
    mbar_init(bar(L::DRAIN), 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(bar(L::ITEM_FULL + i), 1);
      mbar_init(bar(L::ITEM_EMPTY + i), kPairTakers);
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
    tmem_alloc_pair(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 13 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmO);
  }
  // both CTAs' barriers are initialised before either CTA signals the other's
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};

  const int wg = warp >> 2;
  if (wg < 2) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
  }

  if (wg < 2) {
    // ===================== softmax, stage s, this CTA's rows =====================
    const int s = wg;
    const int rq = warp & 3;
    const int r = rq * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(rq * 32) << 16;
    const uint32_t tS = tmem + t_lane + static_cast<uint32_t>(s * kBN);
    const uint32_t tO = tmem + t_lane + static_cast<uint32_t>(L::kTmemO + s * D);
    uint32_t n_s = 0;
    bool ok = true;
    bool dep_wait = p.overlap_prev != 0;  // before the first global write

#pragma unroll 1
    for (uint32_t k = 0; ok; ++k) {
      const int idx = pair_take_item<kPairSleepSoftmaxNs>(item_ring, bar(L::ITEM_FULL),
                                                          bar_l(L::ITEM_EMPTY), k, ctl, ok);
      if (!ok || idx < 0) break;
      const Item it = get_pair_item<kTail>(p, idx);
      const int nT = s == 0 ? it.nT0 : it.nT1;
      const int stage_row0 = it.row0 + s * kPairStageRows + static_cast<int>(rank) * kBM;
      const int row_g = stage_row0 + r;
      float m = -INFINITY;
      float l = 0.f;

#pragma unroll 1
      for (int j = 0; j < nT; ++j, ++n_s) {
        if (!wait_bar_warp(bar(L::S_FULL + s), n_s & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        // this CTA's rows; the pair's stage may reach one tile further than
        // they need (masked)
        const bool defer = softmax_tile<D, BF16, false, kCorrWG>(
            tS, tO, (it.t0 + j) * kBN, stage_row0, row_g, p, j > 0, m, l);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (kCorrWG && defer)
            mbar_arrive(corr_bar(s, rq));  // the correction warp arrives for us
          else
            mbar_arrive_cluster_relaxed(bar_l(L::PV_READY + s));
        }
      }
      if (!ok) break;

      if (dep_wait) {
        grid_dependency_wait();
        dep_wait = false;
      }
      if constexpr (kTail) {
        if (it.part >= 0) {
          // a key quarter (nT >= 1): this warp writes its rows' partial and
          // perhaps merges; the epilogue only counts the item
          if (!wait_bar_warp(bar(L::O_READY + s), (n_s - 1) & 1, ctl)) { ok = false; break; }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::ML_FULL + s));
          tc_fence_after();
          if (!pair_tail_quarter<BF16>(p, it, s, rank, rq, lane, row_g, tO, m, l,
                                       bar_l(L::O_FREE + s))) {
            *abort_flag = 1u;
            ok = false;
            break;
          }
          continue;
        }
      }
      if (row_g < p.Sq) {
        const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
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
    // ========================= epilogue, this CTA's rows =========================
    const int rq = warp & 3;
    const int r = rq * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(rq * 32) << 16;
    const uint32_t stage_buf = sOut + static_cast<uint32_t>(rq * L::kOutWarpBytes);
    uint32_t n_t0 = 0, n_t1 = 0;
    uint32_t n_e0 = 0, n_e1 = 0;
    uint32_t n_c[2] = {0u, 0u};  // correction requests served, per stage
    bool ok = true;
    bool dep_wait = p.overlap_prev != 0;  // before the first global write
    // as in fa_prefill_kernel: the wait for 1/l serves this quarter's
    // correction requests in the correction-warpgroup form
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
              if (lane == 0) mbar_arrive_cluster_relaxed(bar_l(L::PV_READY + s2));
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
      const int idx = pair_take_item<kPairSleepEpilogueNs>(item_ring, bar(L::ITEM_FULL),
                                                           bar_l(L::ITEM_EMPTY), k, ctl, ok);
      if (!ok || idx < 0) break;
      const Item it = get_pair_item<kTail>(p, idx);
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
          if constexpr (kTail)
            if (it.part >= 0) continue;  // a key quarter: its softmax warps write the rows
          inv_l = inv_l_smem[s * kBM + r];
          if (!wait_bar_warp<kSleepEpilogueNs>(bar(L::O_READY + s), (n_t - 1) & 1, ctl)) { ok = false; continue; }
          tc_fence_after();
        }
        const uint32_t tO = tmem + t_lane + static_cast<uint32_t>(L::kTmemO + s * D);
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        stage_o_rows<D, BF16>(tO, have_o, inv_l, stage_buf, L::kOutBox, lane);
        if (have_o) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster_relaxed(bar_l(L::O_FREE + s));
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int warp_row0 = it.row0 + s * kPairStageRows + static_cast<int>(rank) * kBM + rq * 32;
        if (lane == 0 && warp_row0 < p.Sq) {
#pragma unroll
          for (int box = 0; box < D / 64; ++box)
            tma_store_3d(&tmO, stage_buf + static_cast<uint32_t>(box * L::kOutBox), box * 64,
                         warp_row0, it.bh);
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group0();
    __syncwarp();
  } else if (warp == 12 && leader) {
    // ======================= MMA issuer (leader CTA only) =======================
    // The single-CTA kernel's issue order, with pair MMAs: per item
    // QK_0(0) QK_1(0), then per key tile PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1).
    // Commits arrive in both CTAs.
    {
      constexpr uint16_t kBoth = 3;
      constexpr uint32_t kIdescQK = idesc_f16(BF16, false, false, 2 * kBM, kBN);
      constexpr uint32_t kIdescPV = idesc_f16(BF16, false, true, 2 * kBM, D);
      const uint32_t tS0 = tmem, tS1 = tmem + kBN;
      const uint32_t tO0 = tmem + L::kTmemO, tO1 = tmem + L::kTmemO + D;
      bool issued = false;

      auto slot_of = [&](int fill) { return fill % L::kSlots; };
      auto par_of = [&](int fill) { return static_cast<uint32_t>((fill / L::kSlots) & 1); };
      // QK_s: A = Q_s (2 boxes of 128 rows, +1024 descriptor units apart),
      // B = this CTA's 64 keys of K (2 boxes of 64 rows, +512 units apart)
      auto qk = [&](int s, int fk, bool last_of_stage) {
        const uint64_t da = smem_desc_sw128(sQ + static_cast<uint32_t>(s * L::kQBytes), 16, 1024);
        const uint64_t db = smem_desc_sw128(sKV + static_cast<uint32_t>(slot_of(fk) * L::kHalfBytes), 16, 1024);
        umma_pair_ss_k128<L::kBox / 16, L::kKBox / 16>(s == 0 ? tS0 : tS1, da, db, kIdescQK, 0u);
        umma_commit_pair(bar(L::S_FULL + s), kBoth);
        if (last_of_stage) umma_commit_pair(bar(L::Q_EMPTY + s), kBoth);
      };
      // PV_s: A = P_s from both CTAs' tensor memory, B = this CTA's 64
      // columns of V (one MN-major box)
      auto pv = [&](int s, int fv, bool acc) {
        umma_pair_ts_k128(s == 0 ? tO0 : tO1, s == 0 ? tS0 : tS1,
                          smem_desc_sw128(sKV + static_cast<uint32_t>(slot_of(fv) * L::kHalfBytes),
                                          L::kBox, 1024),
                          kIdescPV, acc ? 1u : 0u);
        umma_commit_pair(bar(L::O_READY + s), kBoth);
      };
      auto begin = [&](const Item& it, int kq, int f) -> bool {
        if (!wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + 0), kq & 1, ctl) ||
            !wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + 1), kq & 1, ctl))
          return false;
        if (it.nT1 > 0 && !wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(f)), par_of(f), ctl)) return false;
        tc_fence_after();
        if (it.nT0 > 0) qk(0, f, it.nT0 == 1); else umma_commit_pair(bar(L::Q_EMPTY + 0), kBoth);
        if (it.nT1 > 0) {
          qk(1, f, it.nT1 == 1);
          umma_commit_pair(bar(L::KV_EMPTY + slot_of(f)), kBoth);
        } else {
          umma_commit_pair(bar(L::Q_EMPTY + 1), kBoth);
        }
        issued = true;
        return true;
      };

      uint32_t n_pv0 = 0, n_pv1 = 0;
      uint32_t n_o0 = 0, n_o1 = 0;
      int kq = 0;
      int fK = 0;
      bool ok = true;
      const int first = pair_take_item<kPairSleepMmaNs>(item_ring, bar(L::ITEM_FULL),
                                                        bar_l(L::ITEM_EMPTY), 0, ctl, ok);
      Item cur = first >= 0 ? get_pair_item<kTail>(p, first) : Item{0, 0, 0, 0};
      if (ok && first >= 0) ok = begin(cur, 0, 0);
      else ok = false;
#pragma unroll 1
      while (ok) {
        bool taken = false, has_next = false;
        Item nxt{0, 0, 0, 0};
        auto take_next = [&]() {
          if (taken) return;
          taken = true;
          const int nidx = pair_take_item<kPairSleepMmaNs>(item_ring, bar(L::ITEM_FULL),
                                                           bar_l(L::ITEM_EMPTY), kq + 1, ctl, ok);
          has_next = ok && nidx >= 0;
          if (has_next) nxt = get_pair_item<kTail>(p, nidx);
        };
        const int fN = fK + 2 * cur.nT1;
#pragma unroll 1
        for (int j = 0; j < cur.nT1; ++j) {
          const bool last = j + 1 == cur.nT1;
          if (last) {
            take_next();
            if (!ok) break;
          }
          const int fv = fK + 2 * j + 1, fk1 = fK + 2 * j + 2;
          bool rdy = mbar_try_wait(bar(L::KV_FULL + slot_of(fv)), par_of(fv));
          if (j < cur.nT0) rdy &= mbar_try_wait_cluster(bar(L::PV_READY + 0), n_pv0 & 1);
          if (!__all_sync(0xffffffffu, rdy)) {
            if (!wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(fv)), par_of(fv), ctl)) { ok = false; break; }
            if (j < cur.nT0 && !pair_wait_warp<kPairSleepMmaNs>(bar(L::PV_READY + 0), n_pv0 & 1, ctl)) { ok = false; break; }
          }
          if (j < cur.nT0) {
            if (j == 0 && n_o0 > 0 && !pair_wait_warp<kPairSleepMmaNs>(bar(L::O_FREE + 0), (n_o0 - 1) & 1, ctl)) {
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
            if (nxt.nT0 > 0) qk(0, fN, nxt.nT0 == 1); else umma_commit_pair(bar(L::Q_EMPTY + 0), kBoth);
          }
          if (!pair_wait_warp<kPairSleepMmaNs>(bar(L::PV_READY + 1), n_pv1 & 1, ctl)) { ok = false; break; }
          if (j == 0 && n_o1 > 0 && !pair_wait_warp<kPairSleepMmaNs>(bar(L::O_FREE + 1), (n_o1 - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          ++n_pv1;
          tc_fence_after();
          pv(1, fv, j > 0);
          umma_commit_pair(bar(L::KV_EMPTY + slot_of(fv)), kBoth);
          if (!last) {
            qk(1, fk1, j + 2 == cur.nT1);
            umma_commit_pair(bar(L::KV_EMPTY + slot_of(fk1)), kBoth);
          } else if (has_next) {
            if (!wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + 1), (kq + 1) & 1, ctl)) { ok = false; break; }
            tc_fence_after();
            if (nxt.nT1 > 0) {
              qk(1, fN, nxt.nT1 == 1);
              umma_commit_pair(bar(L::KV_EMPTY + slot_of(fN)), kBoth);
            } else {
              umma_commit_pair(bar(L::Q_EMPTY + 1), kBoth);
            }
          }
        }
        if (ok) take_next();  // an item without key tiles
        if (!ok || !has_next) break;
        if (cur.nT0 > 0) ++n_o0;
        if (cur.nT1 > 0) ++n_o1;
        if (cur.nT1 == 0) ok = begin(nxt, kq + 1, fN);
        ++kq;
        cur = nxt;
        fK = fN;
      }
      if (issued) {  // every MMA issued so far completes before TMEM is freed
        umma_commit_pair(bar(L::DRAIN), 1);
        wait_drain(bar(L::DRAIN), 0, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 13) {
    // ============================== TMA producers ==============================
    // Both CTAs: per item Q_0, K_0, Q_1, V_0, then K_j V_j -- this CTA's rows
    // of Q and its half of each K/V tile, completion on the leader's
    // barriers (the leader expects both CTAs' bytes).  The leader also claims
    // the items and publishes them to both CTAs.
    if (lane == 0) {
      int fill = 0;
      int last_fill[L::kSlots];
#pragma unroll
      for (int i = 0; i < L::kSlots; ++i) last_fill[i] = -1;
      int nq[2] = {0, 0};
      bool ok = true;
      const int qrow_off = static_cast<int>(rank) * kBM;
      auto load_q = [&](const Item& it, int s) -> bool {
        if (nq[s] > 0 && !wait_bar<kSleepProducerNs>(bar(L::Q_EMPTY + s), (nq[s] - 1) & 1, ctl)) return false;
        if (leader) mbar_arrive_expect_tx(bar(L::Q_FULL + s), 2 * L::kQBytes);
#pragma unroll
        for (int box = 0; box < D / 64; ++box)
          tma_load_3d_pair(sQ + static_cast<uint32_t>(s * L::kQBytes + box * L::kBox), &tmQ,
                           bar_l(L::Q_FULL + s), box * 64,
                           it.row0 + s * kPairStageRows + qrow_off, it.bh);
        ++nq[s];
        return true;
      };
      auto load_kv = [&](const Item& it, int kv, int j) -> bool {
        const int slot = fill % L::kSlots;
        const uint32_t par = static_cast<uint32_t>(((fill / L::kSlots) & 1) ^ 1);
        if (!wait_bar<kSleepProducerNs>(bar(L::KV_EMPTY + slot), par, ctl)) return false;
        if (p.test_stall && fill == 2) {  // test hook: both CTAs withhold the first K_1
          ++fill;
          return true;
        }
        if (leader) mbar_arrive_expect_tx(bar(L::KV_FULL + slot), 2 * L::kHalfBytes);
        const uint32_t dst = sKV + static_cast<uint32_t>(slot * L::kHalfBytes);
        if (kv == 0) {  // keys 64*rank .. of tile j, both 64-column boxes
#pragma unroll
          for (int box = 0; box < D / 64; ++box)
            tma_load_3d_pair(dst + static_cast<uint32_t>(box * L::kKBox), &tmK,
                             bar_l(L::KV_FULL + slot), box * 64,
                             (it.t0 + j) * kBN + static_cast<int>(rank) * 64, it.bh);
        } else {        // columns 64*rank .. of tile j, all 128 keys
          tma_load_3d_pair(dst, &tmV, bar_l(L::KV_FULL + slot), static_cast<int>(rank) * 64,
                           (it.t0 + j) * kBN, it.bh);
        }
        last_fill[slot] = fill;
        ++fill;
        return true;
      };
      const uint32_t ring_f = mapa_shared(smem_u32(const_cast<int*>(item_ring)), 1);
      const uint32_t bars_f = mapa_shared(bars, 1);
      int idx = static_cast<int>(blockIdx.x >> 1);  // the grid never exceeds 2x the items
#pragma unroll 1
      for (uint32_t k = 0; ok; ++k) {
        const uint32_t slot = k % kItemRing;
        if (leader) {
          // publish item k (or the end) to both CTAs once every taker of
          // both has taken item k - 4
          const uint32_t par = (k / kItemRing - 1) & 1;
          if (k >= kItemRing && !mbar_try_wait_cluster(bar(L::ITEM_EMPTY + slot), par) &&
              !pair_wait_slow<kPairSleepProducerNs>(bar(L::ITEM_EMPTY + slot), par, ctl.abort,
                                                    ctl.status, ctl.timeout)) {
            ok = false;
            break;
          }
          item_ring[slot] = idx;
          st_shared_cluster_u32(ring_f + 4u * slot, static_cast<uint32_t>(idx));
          mbar_arrive(bar(L::ITEM_FULL + slot));
          mbar_arrive_cluster(bars_f + 8u * static_cast<uint32_t>(L::ITEM_FULL + slot));
        } else {
          if (!mbar_try_wait_cluster(bar(L::ITEM_FULL + slot), (k / kItemRing) & 1) &&
              !pair_wait_slow<kPairSleepProducerNs>(bar(L::ITEM_FULL + slot), (k / kItemRing) & 1,
                                                    ctl.abort, ctl.status, ctl.timeout)) {
            ok = false;
            break;
          }
          idx = item_ring[slot];
          mbar_arrive_cluster(bar_l(L::ITEM_EMPTY + slot));
        }
        if (idx < 0) {
          grid_launch_dependents();  // the next grid may take the SMs
          break;
        }
        const Item it = get_pair_item<kTail>(p, idx);
        ok = load_q(it, 0);
#pragma unroll 1
        for (int j = 0; ok && j < it.nT1; ++j) {
          ok = load_kv(it, 0, j);
          if (ok && j == 0) ok = load_q(it, 1);
          if (ok) ok = load_kv(it, 1, j);
        }
        if (ok && it.nT1 == 0) ok = load_q(it, 1);
        if (leader) {
          const unsigned long long ticket = atomicAdd(p.sched, 1ull);
          const unsigned long long nidx = (gridDim.x >> 1) + ticket;
          idx = nidx < static_cast<unsigned long long>(p.n_items) ? static_cast<int>(nidx) : -1;
          if (idx >= 0) {
            // the next item's Q (all 512 rows, both CTAs' shares) into L2
            // now: its loads can start only once this item's last QKs have
            // read the Q buffers
            const Item nx = get_pair_item<kTail>(p, idx);
#pragma unroll 1
            for (int rb = 0; rb < kPairRows / kBM; ++rb)
#pragma unroll
              for (int box = 0; box < D / 64; ++box)
                tma_prefetch_l2_3d(&tmQ, box * 64, nx.row0 + rb * kBM, nx.bh);
          }
        }
      }
      // drain (leader): its barriers complete only when both CTAs' loads
      // have landed; the follower exits after the final cluster barrier.
      // After a watchdog abort the follower may have issued loads that the
      // leader never armed; it cannot wait on them (their barrier is the
      // leader's), so it gives them a bounded time to land before exiting.
      if (!leader && *abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 100000ull) __nanosleep(1000);
      }
      if (leader) {
#pragma unroll
        for (int s = 0; s < 2; ++s)
          if (nq[s] > 0) wait_drain(bar(L::Q_FULL + s), (nq[s] - 1) & 1, p.timeout_ns);
#pragma unroll 1
        for (int i = 0; i < L::kSlots; ++i)
          if (last_fill[i] >= 0)
            wait_drain(bar(L::KV_FULL + i), static_cast<uint32_t>((last_fill[i] / L::kSlots) & 1),
                       p.timeout_ns);
      }
    }
    __syncwarp();
  }

  // ---- teardown: both CTAs finish before either frees tensor memory or
  // exits (the leader's MMAs and the follower's loads touch both) ----
  tc_fence_before();
  cluster_sync_all();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, L::kTmemCols);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&p.sched[1], 1ull) == gridDim.x - 1) {
      p.sched[0] = 0ull;
      p.sched[1] = 0ull;
      __threadfence();
    }
  }
}

}  // namespace fa
