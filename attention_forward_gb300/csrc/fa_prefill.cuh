// fa_prefill.cuh -- fused attention forward (prefill) kernel for sm_103a.
//
// One CTA owns 256 query rows of one (batch, head) as two ping-pong stages of
// 128 rows (the two-Q-tile ping-pong of the B300 G5 page, V21) and streams
// the keys in tiles of 128.  Warp roles (16 warps, 512 threads):
//
//   warps 0-3   softmax, stage 0   one thread per query row (TMEM lane)
//   warps 4-7   softmax, stage 1
//   warps 8-11  correction: rescales O in TMEM when a row's reference max moved
//   warp  12    tcgen05.mma issue (whole warp, one elected lane) + TMEM alloc
//   warp  13    TMA producer (one thread): Q once, then K/V tiles
//   warps 14-15 idle (they complete the fourth warpgroup)
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
// behind (the aim of the ping-pong on the G5 page).  K and V occupy separate
// slots of one ring with their own full/empty barriers (the decoupled K/V
// loads of G5 V26), and stage 0's PV never waits for stage 1 (the PV0
// barrier of V30).
//
// Softmax works in the log2 domain with the scale folded into one FFMA
// before ex2 (G5 V33 "log2exp2"; "The FA5090 Optimization Journey" section
// 2.6): t = s*scale*log2(e), p = 2^(t - m) against a per-row reference max m.
// m is raised only when the tile's max exceeds it by more than tau (log2
// units); then alpha = 2^(m_old - m_new) and the correction warpgroup
// multiplies O by alpha, skipping any warp whose 32 rows all have alpha == 1
// (a warp-uniform vote).  tau = 0 is the identity-only rescale skip of the
// FA5090 page (sections 2.6 and 2.8: skip exactly when the max did not
// change); tau = 8 is FA4's lazy rescale that the same page describes in
// section 3 (p stays <= 2^8, and the final division by l, accumulated
// against the same m, makes the result exact either way).
//
// Causal (bottom-right): key tiles past the last row's diagonal are never
// loaded or computed (FA5090 section 2.7, causal block skip); only tiles that
// cross the diagonal (or the ragged end of the keys) are masked (section
// 2.8, diagonal-only masking).  CTAs are ordered heaviest-first (LPT,
// section 2.7).
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

template <int D>
struct PrefillLayout {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kQBytes = kBM * D * 2;    // one stage of Q
  static constexpr int kKVBytes = kBN * D * 2;   // one K or V tile
  static constexpr int kBox = 128 * 64 * 2;      // one TMA box (64 cols)
  static constexpr int kSlots = D == 128 ? 5 : 11;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kStages * kQBytes;
  static constexpr int kOffMisc = kOffKV + kSlots * kKVBytes;
  // mbarrier indices
  static constexpr int Q_FULL = 0;    // [2]
  static constexpr int S_FULL = 2;    // [2]
  static constexpr int PV_READY = 4;  // [2] P stored and O rescaled
  static constexpr int A_READY = 6;   // [2]
  static constexpr int O_READY = 8;   // [2]
  static constexpr int DRAIN = 10;
  static constexpr int KV_FULL = 11;            // [kSlots]
  static constexpr int KV_EMPTY = 11 + kSlots;  // [kSlots]
  static constexpr int kNumBars = 11 + 2 * kSlots;
  static constexpr int kOffBars = kOffMisc;
  static constexpr int kOffAlpha = kOffBars + ((kNumBars * 8 + 15) / 16) * 16;
  static constexpr int kOffTmemSlot = kOffAlpha + kStages * kBM * 4;
  static constexpr int kOffAbort = kOffTmemSlot + 4;
  static constexpr int kMiscBytes = kOffAbort + 4 - kOffMisc;
  static constexpr int kSmemBytes = kOffMisc + kMiscBytes + 1024;  // + align
  static constexpr int kTmemCols = 512;
  static constexpr int kTmemO = 256;  // O_s at column 256 + s*D
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Register split between warpgroups (setmaxnreg): softmax warpgroups get
// more, the others give theirs back.  The sum over the 512 threads equals
// 512 * 128, the registers the CTA is launched with; the host checks the
// compiled register count before the first launch.
constexpr int kRegsSoftmax = 192;
constexpr int kRegsOther = 64;
static_assert(2 * 128 * kRegsSoftmax + 2 * 128 * kRegsOther == kThreads * 128,
              "register split must equal the launch allocation");

struct Ctl {
  volatile uint32_t* abort;
  unsigned* status;
  unsigned long long timeout;
};

// try_wait suspends the thread for a while before it reports "not yet", so
// the abort flag and the clock are checked only every 8th round.
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, Ctl c) {
  uint64_t t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 7u) == 0) {
      if (*c.abort) return false;
      const uint64_t t = globaltimer_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > c.timeout) {
        *c.abort = 1u;
        atomicExch(c.status, kStatusTimeout);
        return false;
      }
    }
  }
}

// Bounded wait; false when the watchdog fired (here or in another role).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity,
                                         const Ctl& c) {
  return mbar_try_wait(bar, parity) || wait_slow(bar, parity, c);
}

// Warp-uniform bounded wait (every lane gets the same answer).
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity,
                                              const Ctl& c) {
  const bool ok = wait_bar(bar, parity, c);
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

template <int D, bool BF16>
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
  const uint32_t bars = sbase + L::kOffBars;
  float* alpha_smem = reinterpret_cast<float*>(smem + L::kOffAlpha);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffTmemSlot);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem + L::kOffAbort);
  auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item (heaviest-first for causal) ----
  int qtile, bh;
  if (p.causal && p.lpt) {
    qtile = p.n_qtiles - 1 - static_cast<int>(blockIdx.x) / p.BH;
    bh = static_cast<int>(blockIdx.x) % p.BH;
  } else {
    qtile = static_cast<int>(blockIdx.x) % p.n_qtiles;
    bh = static_cast<int>(blockIdx.x) / p.n_qtiles;
  }
  const int row0 = qtile * kRowsPerCta;
  const int nT0 = stage_tiles(row0, p.Sq, p.Skv, p.causal);
  const int nT1 = stage_tiles(row0 + kBM, p.Sq, p.Skv, p.causal);
  const int n_kv = nT1;  // nT1 >= nT0

  // ---- setup ----
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::Q_FULL + s), 1);
      mbar_init(bar(L::S_FULL + s), 1);
      mbar_init(bar(L::PV_READY + s), 8);  // 4 softmax warps + 4 correction warps
      mbar_init(bar(L::A_READY + s), 4);
      mbar_init(bar(L::O_READY + s), 1);
    }
    mbar_init(bar(L::DRAIN), 1);
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
  if (wg < 2) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
  }

  if (wg < 2) {
    // =========================== softmax, stage s ===========================
    const int s = wg;
    const int rq = warp & 3;                 // lane quarter of TMEM
    const int r = rq * 32 + lane;            // row within the stage
    const int stage_row0 = row0 + s * kBM;
    const int row_g = stage_row0 + r;        // query row
    const int nT = s == 0 ? nT0 : nT1;
    const int off = p.Skv - p.Sq;
    const uint32_t t_lane = static_cast<uint32_t>(rq * 32) << 16;
    const uint32_t tS = tmem + t_lane + static_cast<uint32_t>(s * kBN);
    const uint32_t tO = tmem + t_lane + static_cast<uint32_t>(L::kTmemO + s * D);
    const float c = p.scale_log2;
    const float tau = p.rescale_tau;
    float m = -INFINITY;  // reference max of c*s (log2 units)
    float l = 0.f;        // running sum of 2^(c*s - m)
    bool ok = true;

#pragma unroll 1
    for (int j = 0; j < nT; ++j) {
      if (!wait_bar_warp(bar(L::S_FULL + s), j & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[8][16];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) tmem_ld16(tS + cc * 16, sr[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) reg_fence16(sr[cc]);

      // mask: ragged key tail, and the causal diagonal
      const int key0 = j * kBN;
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
      // p = 2^(s*c - m) in four 32-column pieces: the argument as packed
      // fp32x2 FMAs, the row sum as packed fp32x2 adds; each piece is packed
      // to 16-bit pairs and stored over the first 64 columns of S_s (every S
      // value of this row is already in registers) while the next piece's
      // exponentials run
      float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if (h == 1 && j > 0) {
          // alpha for the correction warpgroup, published once the first
          // piece of P is on its way (it rarely has work: tau keeps the
          // reference max still)
          alpha_smem[s * kBM + r] = alpha;
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::A_READY + s));
        }
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
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::PV_READY + s));
    }

    // ------------------------------ epilogue ------------------------------
    if (ok) {
      const bool have_o = nT > 0;
      // the Q_s buffer becomes the output staging buffer: its TMA load must
      // have landed (a stage with no key tile never waited for it), and the
      // last PV_s must have completed (it also ends every QK_s read of Q_s)
      ok = wait_bar_warp(bar(L::Q_FULL + s), 0, ctl);
      if (ok && have_o) ok = wait_bar_warp(bar(L::O_READY + s), (nT - 1) & 1, ctl);
      if (ok) {
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const uint32_t stage_buf = sQ + static_cast<uint32_t>(s * L::kQBytes);
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
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = cc * 16 + h * 8;  // first column of this chunk
            const uint32_t w0 = pack2<BF16>(__uint_as_float(v[h * 8 + 0]) * inv_l, __uint_as_float(v[h * 8 + 1]) * inv_l);
            const uint32_t w1 = pack2<BF16>(__uint_as_float(v[h * 8 + 2]) * inv_l, __uint_as_float(v[h * 8 + 3]) * inv_l);
            const uint32_t w2 = pack2<BF16>(__uint_as_float(v[h * 8 + 4]) * inv_l, __uint_as_float(v[h * 8 + 5]) * inv_l);
            const uint32_t w3 = pack2<BF16>(__uint_as_float(v[h * 8 + 6]) * inv_l, __uint_as_float(v[h * 8 + 7]) * inv_l);
            const int box = col >> 6, chunk = (col & 63) >> 3;
            const uint32_t addr = stage_buf + static_cast<uint32_t>(
                                                  box * L::kBox + r * 128 + ((chunk ^ (r & 7)) << 4));
            st_shared_v4(addr, w0, w1, w2, w3);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int warp_row0 = stage_row0 + rq * 32;
        if (lane == 0 && warp_row0 < p.Sq) {
#pragma unroll
          for (int box = 0; box < D / 64; ++box)
            tma_store_3d(&tmO, stage_buf + static_cast<uint32_t>(box * L::kBox + rq * 32 * 128),
                         box * 64, warp_row0, bh);
          bulk_commit_group();
          bulk_wait_group0();
        }
        if (row_g < p.Sq) {
          const float lse = l > 0.f ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
          p.lse[static_cast<size_t>(bh) * p.Sq + row_g] = lse;
        }
      }
    }
    __syncwarp();
  } else if (wg == 2) {
    // ============================== correction ==============================
    // For every key tile j of stage s: once softmax has published alpha and
    // PV_s(j-1) has completed, rescale O_s if any row of this warp moved its
    // reference max, then arrive on PV_READY_s (together with the softmax
    // warps' arrival after storing P, that releases PV_s(j)).  Tile 0 has no
    // O to rescale and only arrives.
    const int rq = warp & 3;
    const int r = rq * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(rq * 32) << 16;
#pragma unroll 1
    for (int j = 0; j < n_kv; ++j) {
      bool ok = true;
#pragma unroll 1
      for (int s = 0; s < 2; ++s) {
        if (j >= (s == 0 ? nT0 : nT1)) continue;
        if (j > 0) {
          if (!wait_bar_warp(bar(L::A_READY + s), (j - 1) & 1, ctl)) { ok = false; break; }
          const float alpha = alpha_smem[s * kBM + r];
          if (!wait_bar_warp(bar(L::O_READY + s), (j - 1) & 1, ctl)) { ok = false; break; }
          tc_fence_after();
          if (p.always_rescale || __any_sync(0xffffffffu, alpha != 1.f)) {
            const uint32_t tO = tmem + t_lane + static_cast<uint32_t>(L::kTmemO + s * D);
#pragma unroll 1
            for (int cc = 0; cc < D / 16; cc += 2) {
              uint32_t v0[16], v1[16];
              tmem_ld16(tO + cc * 16, v0);
              tmem_ld16(tO + cc * 16 + 16, v1);
              tmem_wait_ld();
              reg_fence16(v0);
              reg_fence16(v1);
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                v0[e] = __float_as_uint(__uint_as_float(v0[e]) * alpha);
                v1[e] = __float_as_uint(__uint_as_float(v1[e]) * alpha);
              }
              tmem_st16(tO + cc * 16, v0);
              tmem_st16(tO + cc * 16 + 16, v1);
            }
            tmem_wait_st();
          }
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::PV_READY + s));
      }
      if (!ok) break;
    }
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
      bool ok = wait_bar_warp(bar(L::Q_FULL + 0), 0, ctl) &&
                wait_bar_warp(bar(L::Q_FULL + 1), 0, ctl);

      // one asm block per GEMM: K = D for QK (both operands K-major in
      // smem), K = 128 keys for PV (A = P_s from tensor memory, B = V MN-major)
      auto issue_qk = [&](uint32_t d_tmem, uint32_t qbuf, uint32_t kbuf) {
        const uint64_t da = smem_desc_sw128(qbuf, 16, 1024);
        const uint64_t db = smem_desc_sw128(kbuf, 16, 1024);
        if constexpr (D == 128) {
          umma_f16_ss_k128(d_tmem, da, db, kIdescQK, 0u);
        } else {
          umma_f16_ss_k64(d_tmem, da, db, kIdescQK, 0u);
        }
      };
      auto issue_pv = [&](uint32_t d_tmem, uint32_t p_tmem, uint32_t vbuf, bool acc) {
        umma_f16_ts_k128(d_tmem, p_tmem, smem_desc_sw128(vbuf, L::kBox, 1024), kIdescPV,
                         acc ? 1u : 0u);
      };
      auto slot_of = [&](int fill) { return fill % L::kSlots; };
      auto par_of = [&](int fill) { return static_cast<uint32_t>((fill / L::kSlots) & 1); };

      // Tensor-core order: QK_0(0) QK_1(0), then per key tile j
      //   PV_0(j) QK_0(j+1) PV_1(j) QK_1(j+1)
      // Each QK_s(j+1) follows PV_s(j) at once (it overwrites P_s(j)); the
      // wait for K_(j+1) is done earlier, while the softmax of tile j runs.
      if (n_kv > 0) {
        ok = wait_bar_warp(bar(L::KV_FULL + slot_of(0)), par_of(0), ctl);
        if (ok) {
          tc_fence_after();
          if (nT0 > 0) {
            issue_qk(tS0, sQ, sKV + slot_of(0) * L::kKVBytes);
            umma_commit(bar(L::S_FULL + 0));
          }
          issue_qk(tS1, sQ + L::kQBytes, sKV + slot_of(0) * L::kKVBytes);
          umma_commit(bar(L::S_FULL + 1));
          umma_commit(bar(L::KV_EMPTY + slot_of(0)));
          issued = true;
        }
      }
#pragma unroll 1
      for (int j = 0; ok && j < n_kv; ++j) {
        const int fv = 2 * j + 1, fk_next = 2 * j + 2;
        const bool has0 = j < nT0, next = j + 1 < n_kv, next0 = j + 1 < nT0;
        if (next && !wait_bar_warp(bar(L::KV_FULL + slot_of(fk_next)), par_of(fk_next), ctl)) {
          ok = false;
          break;
        }
        if (!wait_bar_warp(bar(L::KV_FULL + slot_of(fv)), par_of(fv), ctl)) { ok = false; break; }
        if (has0) {  // PV_0(j), then QK_0(j+1) over P_0(j)
          if (!wait_bar_warp(bar(L::PV_READY + 0), j & 1, ctl)) { ok = false; break; }
          tc_fence_after();
          issue_pv(tO0, tS0, sKV + slot_of(fv) * L::kKVBytes, j > 0);
          umma_commit(bar(L::O_READY + 0));
          if (next0) {
            issue_qk(tS0, sQ, sKV + slot_of(fk_next) * L::kKVBytes);
            umma_commit(bar(L::S_FULL + 0));
          }
        }
        // PV_1(j), then QK_1(j+1) over P_1(j)
        if (!wait_bar_warp(bar(L::PV_READY + 1), j & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        issue_pv(tO1, tS1, sKV + slot_of(fv) * L::kKVBytes, j > 0);
        umma_commit(bar(L::O_READY + 1));
        umma_commit(bar(L::KV_EMPTY + slot_of(fv)));
        if (next) {
          issue_qk(tS1, sQ + L::kQBytes, sKV + slot_of(fk_next) * L::kKVBytes);
          umma_commit(bar(L::S_FULL + 1));
          umma_commit(bar(L::KV_EMPTY + slot_of(fk_next)));
        }
      }
      if (issued) {  // every MMA issued so far completes before TMEM is freed
        umma_commit(bar(L::DRAIN));
        wait_drain(bar(L::DRAIN), 0, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 13) {
    // ============================== TMA producer =============================
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        mbar_arrive_expect_tx(bar(L::Q_FULL + s), L::kQBytes);
#pragma unroll
        for (int box = 0; box < D / 64; ++box)
          tma_load_3d(sQ + static_cast<uint32_t>(s * L::kQBytes + box * L::kBox), &tmQ,
                      bar(L::Q_FULL + s), box * 64, row0 + s * kBM, bh);
      }
      int fill = 0;
      int last_fill[L::kSlots];
#pragma unroll
      for (int i = 0; i < L::kSlots; ++i) last_fill[i] = -1;
      bool ok = true;
#pragma unroll 1
      for (int j = 0; ok && j < n_kv; ++j) {
#pragma unroll 1
        for (int kv = 0; kv < 2; ++kv, ++fill) {
          const int slot = fill % L::kSlots;
          const uint32_t par = static_cast<uint32_t>(((fill / L::kSlots) & 1) ^ 1);
          if (!wait_bar(bar(L::KV_EMPTY + slot), par, ctl)) { ok = false; break; }
          if (p.test_stall && fill == 2) continue;  // test hook: withhold K_1
          mbar_arrive_expect_tx(bar(L::KV_FULL + slot), L::kKVBytes);
          const CUtensorMap* tm = kv == 0 ? &tmK : &tmV;
#pragma unroll
          for (int box = 0; box < D / 64; ++box)
            tma_load_3d(sKV + static_cast<uint32_t>(slot * L::kKVBytes + box * L::kBox), tm,
                        bar(L::KV_FULL + slot), box * 64, j * kBN, bh);
          last_fill[slot] = fill;
        }
      }
      // drain: every load issued lands before shared memory goes away
      wait_drain(bar(L::Q_FULL + 0), 0, p.timeout_ns);
      wait_drain(bar(L::Q_FULL + 1), 0, p.timeout_ns);
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
}

}  // namespace fa
