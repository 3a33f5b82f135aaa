// fa_prefill_d64x3.cuh -- the fused attention forward (prefill) kernel for
// head dimension 64 with three ping-pong stages.
//
// At D = 64 the two-stage kernel (fa_prefill.cuh) is bound by each stage's
// chain -- S ready, softmax, P stored, PV and the next QK issued, S ready --
// and not by the tensor core: a stage's two GEMMs take half the time they take
// at D = 128 while its softmax takes as long, so one other stage's GEMMs hide
// only part of it.  Here an item is 384 query rows of one (batch, head) as
// three stages of 128 rows, and each softmax warpgroup hides behind the four
// GEMMs of the other two stages (the Q-tile ping-pong of the B300 G5 page,
// V21, taken one stage further).  Tensor memory holds S_s and O_s of three
// stages only with 96-key tiles: S_s at columns 96 s (fp32; P_s as packed
// 16-bit pairs over its first 48 columns, read by PV from there), O_s at
// 288 + 64 s -- 480 of the 512 columns.
//
// Roles (16 warps): softmax of stage s = warp / 4 (warps 0-11, one thread per
// query row), which at the end of an item also writes the stage's O / l in
// 16 bits through its own slice of shared memory and a TMA store (there is no
// separate epilogue warpgroup: its registers went to the third softmax
// warpgroup); warp 12 allocates tensor memory and issues every MMA; warp 13
// is the TMA producer and claims items, heaviest first under causal masking;
// warps 14-15 idle.  Tensor-core issue order per key tile j:
//     PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1) PV_2(j) QK_2(j+1)
// with the next item's QK_s(0) in place of QK_s(j+1) at an item's last tile.
// A stage whose rows all lie past Sq gets no key tiles.  Softmax, masking,
// the lazy rescale (tau), LSE, programmatic-launch waits and the watchdog are
// those of fa_prefill_kernel, whose helpers this file uses.
#pragma once
#include "fa_prefill.cuh"

namespace fa {

// Warps that take every item: 12 softmax warps and the MMA warp.
constexpr int kItemTakers3 = 13;

struct Prefill3Layout {
  static constexpr int D = 64;
  static constexpr int kQBytes = kBM * D * 2;    // one stage of Q (16 KB)
  static constexpr int kKVBytes = kN3 * D * 2;   // one K or V tile (12 KB)
  static constexpr int kSlots = 8;
  static constexpr int kOutWarpBytes = 32 * D * 2;  // a softmax warp's 32 rows of O
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kStages3 * kQBytes;
  static constexpr int kOffOut = kOffKV + kSlots * kKVBytes;
  static constexpr int kOffMisc = kOffOut + 4 * kStages3 * kOutWarpBytes;
  // mbarrier indices, [3] per stage
  static constexpr int Q_FULL = 0;     // Q_s landed
  static constexpr int Q_EMPTY = 3;    // the item's last QK_s is done
  static constexpr int S_FULL = 6;     // S_s ready
  static constexpr int PV_READY = 9;   // P_s stored, O_s rescaled (4 warps)
  static constexpr int O_READY = 12;   // PV_s done
  static constexpr int O_FREE = 15;    // the stage's warps have read O_s (4 warps)
  static constexpr int DRAIN = 18;
  static constexpr int ITEM_FULL = 19;   // [kItemRing]
  static constexpr int ITEM_EMPTY = 23;  // [kItemRing]
  static constexpr int KV_FULL = 27;             // [kSlots]
  static constexpr int KV_EMPTY = 27 + kSlots;   // [kSlots]
  static constexpr int kNumBars = 27 + 2 * kSlots;
  static constexpr int kOffBars = kOffMisc;
  static constexpr int kOffItems = kOffBars + ((kNumBars * 8 + 15) / 16) * 16;
  static constexpr int kOffTmemSlot = kOffItems + kItemRing * 4;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kMiscBytes = kOffAbort + 4 - kOffMisc;
  static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + align
  static constexpr int kTmemCols = 512;
  static constexpr int kTmemO = kStages3 * kN3;  // O_s at column 288 + 64 s
  static_assert(kTmemO + kStages3 * D <= kTmemCols, "tensor memory budget");
  static_assert(kKVBytes % 1024 == 0 && kQBytes % 1024 == 0, "swizzle atom alignment");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Registers per thread after setmaxnreg: the three softmax warpgroups and the
// MMA / producer warpgroup; the sum over the 512 threads equals the 128 per
// thread the CTA is launched with.
constexpr int kRegsSoftmax3 = 144;
constexpr int kRegsControl3 = 80;
static_assert(128 * (3 * kRegsSoftmax3 + kRegsControl3) == kThreads * 128,
              "register split must equal the launch allocation");

struct Item3 {
  int bh, row0;
  int nT[kStages3];
  int nTmax;  // key tiles of the item (the last stage with any)
};

// Key tiles a 128-row stage whose first row is `row_first` needs: none when
// every row lies past Sq; under the causal mask up to the last row's
// diagonal (bottom-right).
__device__ __forceinline__ int stage_tiles3(int row_first, int Sq, int Skv, int causal) {
  if (row_first >= Sq) return 0;
  const int n_all = (Skv + kN3 - 1) / kN3;
  if (!causal) return n_all;
  const int last_key = row_first + kBM - 1 + (Skv - Sq);
  if (last_key < 0) return 0;
  return min(n_all, last_key / kN3 + 1);
}

// Item idx: heaviest first under causal LPT.  The valid stages' tile counts
// never fall with s (causal rows further down see more keys), and the stages
// past Sq come last, so the last stage with tiles has the most.
__device__ __forceinline__ Item3 get_item3(const PrefillParams& p, int idx) {
  Item3 it;
  int qtile;
  if (p.causal && p.lpt) {
    qtile = p.n_qtiles - 1 - idx / p.BH;
    it.bh = idx % p.BH;
  } else {
    qtile = idx % p.n_qtiles;
    it.bh = idx / p.n_qtiles;
  }
  it.row0 = qtile * kRows3;
  it.nTmax = 0;
#pragma unroll
  for (int s = 0; s < kStages3; ++s) {
    it.nT[s] = stage_tiles3(it.row0 + s * kBM, p.Sq, p.Skv, p.causal);
    it.nTmax = max(it.nTmax, it.nT[s]);
  }
  return it;
}

// One 96-key tile of one stage's softmax for this thread's row: the steps of
// softmax_tile (load S, mask, row max, reference max past tau, P = 2^(c s - m)
// packed over the first 48 columns of S, row sum, O *= alpha when a row of
// the warp moved its reference max), for 96 columns and D = 64.  Ends with
// tcgen05.wait::st.
template <bool BF16>
__device__ __forceinline__ void softmax_tile96(uint32_t tS, uint32_t tO, int key0, int stage_row0,
                                               int row_g, const PrefillParams& p,
                                               bool may_rescale, float& m, float& l) {
  constexpr int D = 64;
  const int off = p.Skv - p.Sq;
  const float c = p.scale_log2;
  const float tau = p.rescale_tau;
  uint32_t sr[6][16];
#pragma unroll
  for (int cc = 0; cc < 6; cc += 2) tmem_ld32(tS + cc * 16, sr[cc], sr[cc + 1]);
  tmem_wait_ld();
#pragma unroll
  for (int cc = 0; cc < 6; ++cc) reg_fence16(sr[cc]);

  const bool need_mask =
      (key0 + kN3 > p.Skv) || (p.causal && key0 + kN3 - 1 > stage_row0 + off);
  if (need_mask) {
    int lim = p.Skv - 1 - key0;
    if (p.causal) lim = min(lim, row_g + off - key0);
#pragma unroll
    for (int cc = 0; cc < 6; ++cc)
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (cc * 16 + e > lim) sr[cc][e] = __float_as_uint(-INFINITY);
  }
  // row max: 12 independent 8-column maxima, then a shallow tree
  float mx[12];
#pragma unroll
  for (int g = 0; g < 12; ++g) {
    const uint32_t* v = &sr[g >> 1][(g & 1) * 8];
    float a = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
    a = fmax3(a, __uint_as_float(v[3]), __uint_as_float(v[4]));
    a = fmax3(a, __uint_as_float(v[5]), __uint_as_float(v[6]));
    mx[g] = fmaxf(a, __uint_as_float(v[7]));
  }
  const float r0 = fmax3(mx[0], mx[1], mx[2]), r1 = fmax3(mx[3], mx[4], mx[5]);
  const float r2 = fmax3(mx[6], mx[7], mx[8]), r3 = fmax3(mx[9], mx[10], mx[11]);
  const float t_max = fmaxf(fmaxf(r0, r1), fmaxf(r2, r3)) * c;
  const float m_new = t_max > m + tau ? t_max : m;
  const float m_use = m_new == -INFINITY ? 0.f : m_new;
  const float alpha = m_new == m ? 1.f : ex2_approx(m - m_use);
  const float neg_m = -m_use;
  const bool rescale =
      may_rescale && (p.always_rescale || __any_sync(0xffffffffu, alpha != 1.f));
  float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
  for (int h = 0; h < 3; ++h) {
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
  if (rescale) {
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
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fa_prefill_d64x3_kernel(const __grid_constant__ CUtensorMap tmQ,
                            const __grid_constant__ CUtensorMap tmK,  // box: 96 keys
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmO,
                            const PrefillParams p) {
  using L = Prefill3Layout;
  constexpr int D = L::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + L::kOffQ;
  const uint32_t sKV = sbase + L::kOffKV;
  const uint32_t sOut = sbase + L::kOffOut;
  const uint32_t bars = sbase + L::kOffBars;
  volatile int* item_ring = reinterpret_cast<volatile int*>(smem + L::kOffItems);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem + L::kOffAbort);
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- setup ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages3; ++s) {
      mbar_init(bar(L::Q_FULL + s), 1);
      mbar_init(bar(L::Q_EMPTY + s), 1);
      mbar_init(bar(L::S_FULL + s), 1);
      mbar_init(bar(L::PV_READY + s), 4);
      mbar_init(bar(L::O_READY + s), 1);
      mbar_init(bar(L::O_FREE + s), 4);
    }
    mbar_init(bar(L::DRAIN), 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(bar(L::ITEM_FULL + i), 1);
      mbar_init(bar(L::ITEM_EMPTY + i), kItemTakers3);
    }
    for (int i = 0; i < L::kSlots; ++i) {
      mbar_init(bar(L::KV_FULL + i), 1);
      mbar_init(bar(L::KV_EMPTY + i), 1);
    }
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
  if (wg < kStages3) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax3));
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsControl3));
  }

  if (wg < kStages3) {
    // ================= softmax and output, stage s =================
    const int s = wg;
    const int rq = warp & 3;
    const int r = rq * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(rq * 32) << 16;
    const uint32_t tS = tmem + t_lane + static_cast<uint32_t>(s * kN3);
    const uint32_t tO = tmem + t_lane + static_cast<uint32_t>(L::kTmemO + s * D);
    const uint32_t stage_buf = sOut + static_cast<uint32_t>((s * 4 + rq) * L::kOutWarpBytes);
    uint32_t n_s = 0;  // tiles of this stage so far (S_FULL / O_READY phase)
    bool ok = true;
    bool dep_wait = p.overlap_prev != 0;  // before the first global write

#pragma unroll 1
    for (uint32_t k = 0; ok; ++k) {
      const int idx = take_item<0>(item_ring, bar(L::ITEM_FULL), bar(L::ITEM_EMPTY), k, ctl, ok);
      if (!ok || idx < 0) break;
      const Item3 it = get_item3(p, idx);
      const int nT = it.nT[s];
      const int stage_row0 = it.row0 + s * kBM;
      const int row_g = stage_row0 + r;
      float m = -INFINITY;
      float l = 0.f;

#pragma unroll 1
      for (int j = 0; j < nT; ++j, ++n_s) {
        if (!wait_bar_warp(bar(L::S_FULL + s), n_s & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        softmax_tile96<BF16>(tS, tO, j * kN3, stage_row0, row_g, p, j > 0, m, l);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::PV_READY + s));
      }
      if (!ok) break;

      if (dep_wait) {
        grid_dependency_wait();
        dep_wait = false;
      }
      if (row_g < p.Sq) {
        const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
        p.lse[static_cast<size_t>(it.bh) * p.Sq + row_g] = lse;
      }
      if (stage_row0 >= p.Sq) continue;  // no rows to write (and no tiles)
      // the stage's O / l in 16 bits: this warp's 32 rows through its slice
      // of shared memory and a TMA store
      if (nT > 0) {
        if (!wait_bar_warp(bar(L::O_READY + s), (n_s - 1) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
      }
      if (lane == 0) bulk_wait_group_read0();  // the slice's previous store has read it
      __syncwarp();
      stage_o_rows<D, BF16>(tO, nT > 0, l > 0.f ? 1.f / l : 0.f, stage_buf, L::kOutWarpBytes, lane);
      if (nT > 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::O_FREE + s));
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int warp_row0 = stage_row0 + rq * 32;
      if (lane == 0 && warp_row0 < p.Sq) {
        tma_store_3d(&tmO, stage_buf, 0, warp_row0, it.bh);
        bulk_commit_group();
      }
    }
    if (lane == 0) bulk_wait_group0();  // every store has landed before exit
    __syncwarp();
  } else if (warp == 12) {
    // ============================== MMA issuer ==============================
    {
      constexpr uint32_t kIdescQK = idesc_f16(BF16, false, false, kBM, kN3);
      constexpr uint32_t kIdescPV = idesc_f16(BF16, false, true, kBM, D);
      bool issued = false;
      auto slot_of = [&](int fill) { return fill % L::kSlots; };
      auto par_of = [&](int fill) { return static_cast<uint32_t>((fill / L::kSlots) & 1); };
      auto tS_of = [&](int s) { return tmem + static_cast<uint32_t>(s * kN3); };
      auto tO_of = [&](int s) { return tmem + static_cast<uint32_t>(L::kTmemO + s * D); };
      // QK_s: A = Q_s, B = the 96 keys of fill fk (both K-major, K = 64);
      // commits S_FULL_s, and Q_EMPTY_s after the item's last QK_s
      auto qk = [&](int s, int fk, bool last_of_stage) {
        const uint64_t da = smem_desc_sw128(sQ + static_cast<uint32_t>(s * L::kQBytes), 16, 1024);
        const uint64_t db = smem_desc_sw128(sKV + static_cast<uint32_t>(slot_of(fk) * L::kKVBytes), 16, 1024);
        umma_f16_ss_k64(tS_of(s), da, db, kIdescQK, 0u);
        umma_commit(bar(L::S_FULL + s));
        if (last_of_stage) umma_commit(bar(L::Q_EMPTY + s));
      };
      // PV_s: A = P_s from tensor memory (96 keys), B = V of fill fv, MN-major
      auto pv = [&](int s, int fv, bool acc) {
        // (N = 64 is one 128-byte swizzle width: the leading byte offset,
        // the stride between 64-column boxes, is never used)
        umma_f16_ts_k96(tO_of(s), tS_of(s),
                        smem_desc_sw128(sKV + static_cast<uint32_t>(slot_of(fv) * L::kKVBytes),
                                        16384, 1024),
                        kIdescPV, acc ? 1u : 0u);
        umma_commit(bar(L::O_READY + s));
      };
      // the first QKs of an item (Q in buffer phase kq, K_0 = fill f)
      auto begin = [&](const Item3& it, int kq, int f) -> bool {
        for (int s = 0; s < kStages3; ++s)
          if (!wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + s), kq & 1, ctl)) return false;
        if (it.nTmax > 0 && !wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(f)), par_of(f), ctl))
          return false;
        tc_fence_after();
        for (int s = 0; s < kStages3; ++s) {
          if (it.nT[s] > 0) qk(s, f, it.nT[s] == 1); else umma_commit(bar(L::Q_EMPTY + s));
        }
        if (it.nTmax > 0) umma_commit(bar(L::KV_EMPTY + slot_of(f)));
        issued = true;
        return true;
      };

      uint32_t n_pv[kStages3] = {0u, 0u, 0u};  // PV_s issued (PV_READY phase)
      uint32_t n_o[kStages3] = {0u, 0u, 0u};   // items with a PV_s (O_FREE phase)
      int kq = 0;
      int fK = 0;
      bool ok = true;
      const int first = take_item<kSleepMmaNs>(item_ring, bar(L::ITEM_FULL),
                                               bar(L::ITEM_EMPTY), 0, ctl, ok);
      Item3 cur{};
      if (first >= 0) cur = get_item3(p, first);
      if (ok && first >= 0) ok = begin(cur, 0, 0);
      else ok = false;
#pragma unroll 1
      while (ok) {
        bool taken = false, has_next = false;
        Item3 nxt{};
        auto take_next = [&]() {
          if (taken) return;
          taken = true;
          const int nidx = take_item<kSleepMmaNs>(item_ring, bar(L::ITEM_FULL),
                                                  bar(L::ITEM_EMPTY), kq + 1, ctl, ok);
          has_next = ok && nidx >= 0;
          if (has_next) nxt = get_item3(p, nidx);
        };
        const int fN = fK + 2 * cur.nTmax;  // the next item's K_0
#pragma unroll 1
        for (int j = 0; j < cur.nTmax && ok; ++j) {
          const bool last = j + 1 == cur.nTmax;
          if (last) {
            take_next();
            if (!ok) break;
          }
          const int fv = fK + 2 * j + 1, fk1 = fK + 2 * j + 2;
          if (!wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(fv)), par_of(fv), ctl)) { ok = false; break; }
          bool k_ready = false;   // K_(j+1), or the next item's K_0
          bool nq_ready = false;  // the next item's Q
#pragma unroll
          for (int s = 0; s < kStages3 && ok; ++s) {
            if (j < cur.nT[s]) {  // PV_s(j)
              if (!wait_bar_warp<kSleepMmaNs>(bar(L::PV_READY + s), n_pv[s] & 1, ctl)) { ok = false; break; }
              if (j == 0 && n_o[s] > 0 &&
                  !wait_bar_warp<kSleepMmaNs>(bar(L::O_FREE + s), (n_o[s] - 1) & 1, ctl)) {
                ok = false;
                break;
              }
              ++n_pv[s];
              tc_fence_after();
              pv(s, fv, j > 0);
            }
            if (!last) {  // QK_s(j+1) over P_s(j)
              if (j + 1 < cur.nT[s]) {
                if (!k_ready) {
                  if (!wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(fk1)), par_of(fk1), ctl)) { ok = false; break; }
                  k_ready = true;
                  tc_fence_after();
                }
                qk(s, fk1, j + 2 == cur.nT[s]);
              }
            } else if (has_next) {  // the next item's QK_s(0)
              if (!nq_ready) {
                for (int s2 = 0; s2 < kStages3 && ok; ++s2)
                  ok = wait_bar_warp<kSleepMmaNs>(bar(L::Q_FULL + s2), (kq + 1) & 1, ctl);
                if (!ok) break;
                nq_ready = true;
              }
              if (nxt.nT[s] > 0) {
                if (!k_ready) {
                  if (!wait_bar_warp<kSleepMmaNs>(bar(L::KV_FULL + slot_of(fN)), par_of(fN), ctl)) { ok = false; break; }
                  k_ready = true;
                }
                tc_fence_after();
                qk(s, fN, nxt.nT[s] == 1);
              } else {
                umma_commit(bar(L::Q_EMPTY + s));
              }
            }
          }
          if (!ok) break;
          umma_commit(bar(L::KV_EMPTY + slot_of(fv)));  // every PV of V_j issued
          if (!last) umma_commit(bar(L::KV_EMPTY + slot_of(fk1)));  // every QK of K_(j+1)
          else if (has_next && nxt.nTmax > 0) umma_commit(bar(L::KV_EMPTY + slot_of(fN)));
        }
        if (ok) take_next();  // an item without key tiles
        if (!ok || !has_next) break;
#pragma unroll
        for (int s = 0; s < kStages3; ++s)
          if (cur.nT[s] > 0) ++n_o[s];
        if (cur.nTmax == 0) ok = begin(nxt, kq + 1, fN);  // no tile above began it
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
    // Per item: Q_0, K_0, Q_1, Q_2, V_0, then K_j V_j.
    if (lane == 0) {
      int fill = 0;
      int last_fill[L::kSlots];
#pragma unroll
      for (int i = 0; i < L::kSlots; ++i) last_fill[i] = -1;
      int nq[kStages3] = {0, 0, 0};
      bool ok = true;
      auto load_q = [&](const Item3& it, int s) -> bool {
        if (nq[s] > 0 && !wait_bar<kSleepProducerNs>(bar(L::Q_EMPTY + s), (nq[s] - 1) & 1, ctl)) return false;
        mbar_arrive_expect_tx(bar(L::Q_FULL + s), L::kQBytes);
        tma_load_3d(sQ + static_cast<uint32_t>(s * L::kQBytes), &tmQ, bar(L::Q_FULL + s), 0,
                    it.row0 + s * kBM, it.bh);
        ++nq[s];
        return true;
      };
      auto load_kv = [&](const Item3& it, int kv, int j) -> bool {
        const int slot = fill % L::kSlots;
        const uint32_t par = static_cast<uint32_t>(((fill / L::kSlots) & 1) ^ 1);
        if (!wait_bar<kSleepProducerNs>(bar(L::KV_EMPTY + slot), par, ctl)) return false;
        if (p.test_stall && fill == 2) {  // test hook: withhold the first item's K_1
          ++fill;
          return true;
        }
        mbar_arrive_expect_tx(bar(L::KV_FULL + slot), L::kKVBytes);
        tma_load_3d(sKV + static_cast<uint32_t>(slot * L::kKVBytes), kv == 0 ? &tmK : &tmV,
                    bar(L::KV_FULL + slot), 0, j * kN3, it.bh);
        last_fill[slot] = fill;
        ++fill;
        return true;
      };
      int idx = static_cast<int>(blockIdx.x);  // the grid never exceeds the items
#pragma unroll 1
      for (uint32_t k = 0; ok; ++k) {
        const uint32_t slot = k % kItemRing;
        if (k >= kItemRing &&
            !wait_bar<kSleepProducerNs>(bar(L::ITEM_EMPTY + slot), (k / kItemRing - 1) & 1, ctl)) {
          ok = false;
          break;
        }
        item_ring[slot] = idx;
        mbar_arrive(bar(L::ITEM_FULL + slot));
        if (idx < 0) break;
        const Item3 it = get_item3(p, idx);
        ok = load_q(it, 0);
        if (ok && it.nTmax > 0) ok = load_kv(it, 0, 0);
        if (ok) ok = load_q(it, 1);
        if (ok) ok = load_q(it, 2);
        if (ok && it.nTmax > 0) ok = load_kv(it, 1, 0);
#pragma unroll 1
        for (int j = 1; ok && j < it.nTmax; ++j) {
          ok = load_kv(it, 0, j);
          if (ok) ok = load_kv(it, 1, j);
        }
        idx = claim_item(p);
        if (idx < 0) grid_launch_dependents();  // the next grid may take the SMs
      }
      // drain: every load issued lands before shared memory goes away
#pragma unroll
      for (int s = 0; s < kStages3; ++s)
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
    __threadfence();
    if (atomicAdd(&p.sched[1], 1ull) == gridDim.x - 1) {
      p.sched[0] = 0ull;
      p.sched[1] = 0ull;
      __threadfence();
    }
  }
}

}  // namespace fa
