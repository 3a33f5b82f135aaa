// fa_prefill_pair64.cuh -- the CTA-pair prefill kernel with 64-key score
// tiles and two score buffers per stage (head dimension 128, whole key range).
//
// The CTA-pair kernel of fa_prefill_pair.cuh keeps P_s in the tensor-memory
// columns of S_s, so the next S_s = Q_s K^T can only be issued after PV_s has
// read P_s: every key tile costs each stage the chain softmax -> PV -> QK ->
// softmax, and the tensor core waits for it.  Here a score tile is 64 keys,
// so S_s needs 64 fp32 columns and each stage gets two of them (S_s0, S_s1:
// 4 x 64 columns, plus O_0 and O_1: 512 columns in all).  P_s(j) is packed
// over the first 32 columns of its own buffer, and QK_s(j+1) writes the other
// one.  The tensor core's order per key tile j becomes
//     QK_0(j+1)  QK_1(j+1)  PV_0(j)  PV_1(j)
// so the next scores are computed while the softmax of tile j runs: between
// S_0(j) ready and PV_0(j) the tensor core has four other GEMMs to do.  The
// price is the QK shape: a 256 x 64 x 16 pair MMA takes 43 cycles on GB300
// against 32 for half of a 256 x 128 x 16 one (measured).
//
// Everything else follows the CTA-pair kernel: a pair item is 512 query rows
// (two stages of 256, 128 in each CTA), the leader's MMA warp issues for
// both CTAs, each CTA loads its half of every K tile (32 keys) and of every V
// tile (64 columns), the softmax and epilogue run per CTA, items are claimed
// heaviest first.
//
// Barrier phases that a waiter checks by parity must never run two phases
// ahead of it: S_FULL and P_READY therefore exist per (stage, buffer), whose
// next completion needs the waiter's own progress; O_READY per stage is only
// waited for by the softmax before a rescale (the previous PV of the stage)
// and by the epilogue at the end of an item.
#pragma once
#include "fa_prefill_pair.cuh"

namespace fa {

constexpr int kP64BN = 64;  // keys per score tile

struct Pair64Layout {
  static constexpr int D = 128;
  static constexpr int kQBytes = kBM * D * 2;   // one stage of this CTA's Q (32 KB)
  static constexpr int kBox = 128 * 64 * 2;     // 128 rows x 64 columns
  static constexpr int kKBox = 32 * 64 * 2;     // this CTA's 32 keys x 64 columns
  static constexpr int kVBox = 64 * 64 * 2;     // 64 keys x this CTA's 64 columns
  static constexpr int kHalfBytes = 8192;       // this CTA's half of a K or V tile
  static constexpr int kSlots = 16;
  static constexpr int kOutWarpBytes = 32 * D * 2;
  static constexpr int kOutBox = 32 * 64 * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kStages * kQBytes;
  static constexpr int kOffOut = kOffKV + kSlots * kHalfBytes;
  static constexpr int kOffMisc = kOffOut + 4 * kOutWarpBytes;
  // mbarrier indices (L: used in the leader only; B: in both CTAs)
  static constexpr int Q_FULL = 0;      // [2] L: both CTAs' Q_s landed
  static constexpr int Q_EMPTY = 2;     // [2] B: the item's last QK_s is done
  static constexpr int S_FULL = 4;      // [2][2] B: S_sb ready (stage s, buffer b)
  static constexpr int P_READY = 8;     // [2][2] L: P_sb stored in both CTAs (8 warps)
  static constexpr int O_READY = 12;    // [2] B: PV_s done
  static constexpr int ML_FULL = 14;    // [2] B: the item's 1/l published (local)
  static constexpr int O_FREE = 16;     // [2] L: both CTAs' epilogues read O_s (8 warps)
  static constexpr int DRAIN = 18;      // L
  static constexpr int ITEM_FULL = 19;  // [kItemRing] B
  static constexpr int ITEM_EMPTY = 23; // [kItemRing] L
  static constexpr int KV_FULL = 27;            // [kSlots] L: both halves landed
  static constexpr int KV_EMPTY = 27 + kSlots;  // [kSlots] B: its readers are done
  static constexpr int kNumBars = 27 + 2 * kSlots;
  static constexpr int kOffBars = kOffMisc;
  static constexpr int kOffInvL = kOffBars + ((kNumBars * 8 + 15) / 16) * 16;
  static constexpr int kOffItems = kOffInvL + kStages * kBM * 4;
  static constexpr int kOffTmemSlot = kOffItems + kItemRing * 4;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kMiscBytes = kOffAbort + 4 - kOffMisc;
  static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + align
  static constexpr int kTmemCols = 512;
  static constexpr int kTmemO = 256;  // O_s at 256 + s*D; S_sb at s*128 + b*64
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Score tiles of 64 keys a 256-row stage whose first query row is
// `row_first` needs.
__device__ __forceinline__ int p64_stage_tiles(int row_first, int Sq, int Skv, int causal) {
  const int n_all = (Skv + kP64BN - 1) / kP64BN;
  if (!causal) return n_all;
  const int last_key = row_first + kPairStageRows - 1 + (Skv - Sq);
  if (last_key < 0) return 0;
  return min(n_all, last_key / kP64BN + 1);
}

__device__ __forceinline__ PairItem get_pair64_item(const PrefillParams& p, int idx) {
  PairItem it;
  int qtile;
  if (p.causal && p.lpt) {
    qtile = p.n_qtiles - 1 - idx / p.BH;
    it.bh = idx % p.BH;
  } else {
    qtile = idx % p.n_qtiles;
    it.bh = idx / p.n_qtiles;
  }
  it.row0 = qtile * kPairRows;
  it.nT0 = p64_stage_tiles(it.row0, p.Sq, p.Skv, p.causal);
  it.nT1 = p64_stage_tiles(it.row0 + kPairStageRows, p.Sq, p.Skv, p.causal);
  return it;
}

// Ring fills of one item, in load order K_0, K_1, V_0, K_2, V_1, ..., V_(n-1)
// (each K one tile ahead of its V, as the tensor core reads them).
__device__ __forceinline__ int p64_fill_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int p64_fill_v(int j, int n) { return j + 1 < n ? 2 * j + 2 : 2 * n - 1; }

// One 64-key tile of one stage's softmax for this thread's query row: as
// softmax_tile, over 64 columns of S at tS; P goes to the first 32 columns
// of the same buffer.  A rescale of this warp's rows of O first waits for
// the stage's previous PV (o_bar, phase parity o_par), which S_FULL no
// longer implies here.  Returns false if that wait ran out (watchdog).
// Ends with tcgen05.wait::st.
template <bool BF16>
__device__ __forceinline__ bool softmax_tile64(uint32_t tS, uint32_t tO, int key0, int stage_row0,
                                               int row_g, const PrefillParams& p, bool may_rescale,
                                               float& m, float& l, uint32_t o_bar, uint32_t o_par,
                                               const Ctl& ctl) {
  constexpr int D = 128;
  const int off = p.Skv - p.Sq;
  const float c = p.scale_log2;
  const float tau = p.rescale_tau;
  uint32_t sr[4][16];
  tmem_ld32(tS, sr[0], sr[1]);
  tmem_ld32(tS + 32, sr[2], sr[3]);
  tmem_wait_ld();
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) reg_fence16(sr[cc]);

  const bool need_mask =
      (key0 + kP64BN > p.Skv) || (p.causal && key0 + kP64BN - 1 > stage_row0 + off);
  if (need_mask) {
    int lim = p.Skv - 1 - key0;
    if (p.causal) lim = min(lim, row_g + off - key0);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (cc * 16 + e > lim) sr[cc][e] = __float_as_uint(-INFINITY);
  }
  float mx[8];
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint32_t* v = &sr[g >> 1][(g & 1) * 8];
    float a = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
    a = fmax3(a, __uint_as_float(v[3]), __uint_as_float(v[4]));
    a = fmax3(a, __uint_as_float(v[5]), __uint_as_float(v[6]));
    mx[g] = fmaxf(a, __uint_as_float(v[7]));
  }
  const float t_max =
      fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(fmax3(mx[3], mx[4], mx[5]), mx[6], mx[7])) * c;
  const float m_new = t_max > m + tau ? t_max : m;
  const float m_use = m_new == -INFINITY ? 0.f : m_new;
  const float alpha = m_new == m ? 1.f : ex2_approx(m - m_use);
  const float neg_m = -m_use;
  float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
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
  const bool rescale =
      may_rescale && (p.always_rescale || __any_sync(0xffffffffu, alpha != 1.f));
  bool ok = true;
  if (rescale) {
    // O_s holds the previous PV_s only once it has completed
    ok = wait_bar_warp(o_bar, o_par, ctl);
    if (ok) {
      tc_fence_after();
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
  }
  tmem_wait_st();
  return ok;
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_prefill_pair64_kernel(const __grid_constant__ CUtensorMap tmQ,
                             const __grid_constant__ CUtensorMap tmK,  // box: 32 keys
                             const __grid_constant__ CUtensorMap tmV,  // box: 64 keys
                             const __grid_constant__ CUtensorMap tmO,
                             const PrefillParams p) {
  using L = Pair64Layout;
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

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t bars_l = mapa_shared(bars, 0);
  auto bar_l = [&](int i) { return bars_l + 8u * static_cast<uint32_t>(i); };

  // ---- setup ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::Q_FULL + s), 1);
      mbar_init(bar(L::Q_EMPTY + s), 1);
      for (int b = 0; b < 2; ++b) {
        mbar_init(bar(L::S_FULL + 2 * s + b), 1);
        mbar_init(bar(L::P_READY + 2 * s + b), 8);  // 4 softmax warps of the stage per CTA
      }
      mbar_init(bar(L::O_READY + s), 1);
      mbar_init(bar(L::ML_FULL + s), 4);
      mbar_init(bar(L::O_FREE + s), 8);
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
    const uint32_t tS = tmem + t_lane + static_cast<uint32_t>(s * 128);
    const uint32_t tO = tmem + t_lane + static_cast<uint32_t>(L::kTmemO + s * D);
    uint32_t n_t = 0;  // tiles of this stage so far: buffer n_t & 1
    bool ok = true;

#pragma unroll 1
    for (uint32_t k = 0; ok; ++k) {
      const int idx = pair_take_item<kPairSleepSoftmaxNs>(item_ring, bar(L::ITEM_FULL),
                                                          bar_l(L::ITEM_EMPTY), k, ctl, ok);
      if (!ok || idx < 0) break;
      const PairItem it = get_pair64_item(p, idx);
      const int nT = s == 0 ? it.nT0 : it.nT1;
      const int stage_row0 = it.row0 + s * kPairStageRows + static_cast<int>(rank) * kBM;
      const int row_g = stage_row0 + r;
      float m = -INFINITY;
      float l = 0.f;

#pragma unroll 1
      for (int j = 0; j < nT; ++j, ++n_t) {
        const uint32_t b = n_t & 1u;
        if (!wait_bar_warp(bar(L::S_FULL + 2 * s + static_cast<int>(b)), (n_t >> 1) & 1u, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (!softmax_tile64<BF16>(tS + b * kP64BN, tO, j * kP64BN, stage_row0, row_g, p, j > 0,
                                  m, l, bar(L::O_READY + s), (n_t - 1u) & 1u, ctl)) {
          ok = false;
          break;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(bar_l(L::P_READY + 2 * s + static_cast<int>(b)));
      }
      if (!ok) break;

      if (row_g < p.Sq) {
        const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        p.lse[static_cast<size_t>(it.bh) * p.Sq + row_g] = lse;
      }
      if (nT > 0) {
        if (!wait_bar_warp(bar(L::O_READY + s), (n_t - 1) & 1, ctl)) { ok = false; break; }
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
    bool ok = true;
#pragma unroll 1
    for (uint32_t k = 0; ok; ++k) {
      const int idx = pair_take_item<kPairSleepEpilogueNs>(item_ring, bar(L::ITEM_FULL),
                                                           bar_l(L::ITEM_EMPTY), k, ctl, ok);
      if (!ok || idx < 0) break;
      const PairItem it = get_pair64_item(p, idx);
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
          if (!wait_bar_warp<kSleepEpilogueNs>(bar(L::ML_FULL + s), n_e & 1, ctl)) { ok = false; continue; }
          ++n_e;
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
    // Per key tile j of an item: QK_0(j+1) QK_1(j+1) (at the item's last tile:
    // the next item's QK_0(0) QK_1(0)), then PV_0(j) PV_1(j).  Commits arrive
    // in both CTAs.
    {
      constexpr uint16_t kBoth = 3;
      constexpr uint32_t kIdescQK = idesc_f16(BF16, false, false, 2 * kBM, kP64BN);
      constexpr uint32_t kIdescPV = idesc_f16(BF16, false, true, 2 * kBM, D);
      bool issued = false;
      uint32_t n_qk[2] = {0u, 0u};  // QK_s issued: buffer n_qk & 1
      uint32_t n_pv[2] = {0u, 0u};  // PV_s issued: buffer n_pv & 1, P_READY phase n_pv >> 1
      uint32_t n_o[2] = {0u, 0u};   // items so far with a PV_s (O_FREE phase)

      auto slot_of = [&](int fill) { return fill % L::kSlots; };
      auto par_of = [&](int fill) { return static_cast<uint32_t>((fill / L::kSlots) & 1); };
      auto kv_wait = [&](int fill) -> bool {
        return wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(fill)), par_of(fill), ctl);
      };
      // QK_s into buffer n_qk[s] & 1, K from fill fk; commits S_FULL_sb, and
      // Q_EMPTY_s after the item's last QK_s
      auto qk = [&](int s, int fk, bool last_of_stage) {
        const uint32_t b = n_qk[s] & 1u;
        const uint64_t da = smem_desc_sw128(sQ + static_cast<uint32_t>(s * L::kQBytes), 16, 1024);
        const uint64_t db =
            smem_desc_sw128(sKV + static_cast<uint32_t>(slot_of(fk) * L::kHalfBytes), 16, 1024);
        umma_pair_ss_k128<L::kBox / 16, L::kKBox / 16>(tmem + static_cast<uint32_t>(s * 128) + b * kP64BN,
                                                       da, db, kIdescQK, 0u);
        umma_commit_pair(bar(L::S_FULL + 2 * s + static_cast<int>(b)), kBoth);
        if (last_of_stage) umma_commit_pair(bar(L::Q_EMPTY + s), kBoth);
        ++n_qk[s];
      };
      // PV_s from buffer n_pv[s] & 1 once its P is stored; V from fill fv
      auto pv = [&](int s, int fv, bool first_of_item) -> bool {
        const uint32_t b = n_pv[s] & 1u;
        if (!pair_wait_warp<kPairSleepMmaNs>(bar(L::P_READY + 2 * s + static_cast<int>(b)),
                                             (n_pv[s] >> 1) & 1u, ctl))
          return false;
        if (first_of_item && n_o[s] > 0 &&
            !pair_wait_warp<kPairSleepMmaNs>(bar(L::O_FREE + s), (n_o[s] - 1) & 1, ctl))
          return false;
        tc_fence_after();
        umma_pair_ts_k64(tmem + L::kTmemO + static_cast<uint32_t>(s * D),
                         tmem + static_cast<uint32_t>(s * 128) + b * kP64BN,
                         smem_desc_sw128(sKV + static_cast<uint32_t>(slot_of(fv) * L::kHalfBytes),
                                         L::kVBox, 1024),
                         kIdescPV, first_of_item ? 0u : 1u);
        umma_commit_pair(bar(L::O_READY + s), kBoth);
        ++n_pv[s];
        return true;
      };
      // an item's first QKs (its Q in buffer phase kq, K_0 at fill f)
      auto first_qks = [&](const PairItem& it, int kq, int f) -> bool {
        if (!wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + 0), kq & 1, ctl) ||
            !wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + 1), kq & 1, ctl))
          return false;
        if (it.nT1 > 0 && !kv_wait(f)) return false;
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

      int kq = 0;
      int fK = 0;
      bool ok = true;
      const int first = pair_take_item<kPairSleepMmaNs>(item_ring, bar(L::ITEM_FULL),
                                                        bar_l(L::ITEM_EMPTY), 0, ctl, ok);
      PairItem cur = first >= 0 ? get_pair64_item(p, first) : PairItem{0, 0, 0, 0};
      if (ok && first >= 0) ok = first_qks(cur, 0, 0);
      else ok = false;
#pragma unroll 1
      while (ok) {
        bool has_next = false;
        PairItem nxt{0, 0, 0, 0};
        const int n = cur.nT1;
        const int fN = fK + 2 * n;  // the next item's K_0
#pragma unroll 1
        for (int j = 0; j < n && ok; ++j) {
          // next scores: this item's tile j + 1, or the next item's first
          if (j + 1 < n) {
            const int fk = fK + p64_fill_k(j + 1);
            if (!kv_wait(fk)) { ok = false; break; }
            tc_fence_after();
            if (j + 1 < cur.nT0) qk(0, fk, j + 2 == cur.nT0);
            qk(1, fk, j + 2 == n);
            umma_commit_pair(bar(L::KV_EMPTY + slot_of(fk)), kBoth);
          } else {
            const int nidx = pair_take_item<kPairSleepMmaNs>(item_ring, bar(L::ITEM_FULL),
                                                             bar_l(L::ITEM_EMPTY), kq + 1, ctl, ok);
            if (!ok) break;
            has_next = nidx >= 0;
            if (has_next) {
              nxt = get_pair64_item(p, nidx);
              if (!first_qks(nxt, kq + 1, fN)) { ok = false; break; }
            }
          }
          // this tile's PVs
          const int fv = fK + p64_fill_v(j, n);
          if (!kv_wait(fv)) { ok = false; break; }
          if (j < cur.nT0 && !pv(0, fv, j == 0)) { ok = false; break; }
          if (!pv(1, fv, j == 0)) { ok = false; break; }
          umma_commit_pair(bar(L::KV_EMPTY + slot_of(fv)), kBoth);
        }
        if (!ok) break;
        if (n == 0) {  // an item without key tiles: take the next one here
          const int nidx = pair_take_item<kPairSleepMmaNs>(item_ring, bar(L::ITEM_FULL),
                                                           bar_l(L::ITEM_EMPTY), kq + 1, ctl, ok);
          if (!ok) break;
          has_next = nidx >= 0;
          if (has_next) {
            nxt = get_pair64_item(p, nidx);
            if (!first_qks(nxt, kq + 1, fN)) { ok = false; break; }
          }
        }
        if (!has_next) break;
        if (cur.nT0 > 0) ++n_o[0];
        if (cur.nT1 > 0) ++n_o[1];
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
    // Per item: Q_0, K_0, Q_1, then K_j V_(j-1) for j = 1 .. n-1, then V_(n-1):
    // this CTA's rows of Q and its half of each K/V tile, completion on the
    // leader's barriers.  The leader claims the items and publishes them.
    if (lane == 0) {
      int fill = 0;
      int last_fill[L::kSlots];
#pragma unroll
      for (int i = 0; i < L::kSlots; ++i) last_fill[i] = -1;
      int nq[2] = {0, 0};
      bool ok = true;
      const int qrow_off = static_cast<int>(rank) * kBM;
      auto load_q = [&](const PairItem& it, int s) -> bool {
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
      auto load_kv = [&](const PairItem& it, int kv, int j) -> bool {
        const int slot = fill % L::kSlots;
        const uint32_t par = static_cast<uint32_t>(((fill / L::kSlots) & 1) ^ 1);
        if (!wait_bar<kSleepProducerNs>(bar(L::KV_EMPTY + slot), par, ctl)) return false;
        if (p.test_stall && fill == 2) {  // test hook: both CTAs withhold the first V_0
          ++fill;
          return true;
        }
        if (leader) mbar_arrive_expect_tx(bar(L::KV_FULL + slot), 2 * L::kHalfBytes);
        const uint32_t dst = sKV + static_cast<uint32_t>(slot * L::kHalfBytes);
        if (kv == 0) {  // keys 32*rank .. of tile j, both 64-column boxes
#pragma unroll
          for (int box = 0; box < D / 64; ++box)
            tma_load_3d_pair(dst + static_cast<uint32_t>(box * L::kKBox), &tmK,
                             bar_l(L::KV_FULL + slot), box * 64,
                             j * kP64BN + static_cast<int>(rank) * (kP64BN / 2), it.bh);
        } else {        // columns 64*rank .. of tile j, all 64 keys
          tma_load_3d_pair(dst, &tmV, bar_l(L::KV_FULL + slot), static_cast<int>(rank) * 64,
                           j * kP64BN, it.bh);
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
        if (idx < 0) break;
        const PairItem it = get_pair64_item(p, idx);
        const int n = it.nT1;
        ok = load_q(it, 0);
        if (ok && n > 0) ok = load_kv(it, 0, 0);
        if (ok) ok = load_q(it, 1);
#pragma unroll 1
        for (int j = 1; ok && j < n; ++j) {
          ok = load_kv(it, 0, j);
          if (ok) ok = load_kv(it, 1, j - 1);
        }
        if (ok && n > 0) ok = load_kv(it, 1, n - 1);
        if (leader) {
          const unsigned long long ticket = atomicAdd(p.sched, 1ull);
          const unsigned long long nidx = (gridDim.x >> 1) + ticket;
          idx = nidx < static_cast<unsigned long long>(p.n_items) ? static_cast<int>(nidx) : -1;
          if (idx >= 0) {
            // the next item's Q (all 512 rows) into L2 now
            const PairItem nx = get_pair64_item(p, idx);
#pragma unroll 1
            for (int rb = 0; rb < kPairRows / kBM; ++rb)
#pragma unroll
              for (int box = 0; box < D / 64; ++box)
                tma_prefetch_l2_3d(&tmQ, box * 64, nx.row0 + rb * kBM, nx.bh);
          }
        }
      }
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

  // ---- teardown ----
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
