// fa_decode.cuh -- attention forward for one query row per head (decode),
// split over the keys.  sm_103a.
//
// With Sq == 1 the work per head is a GEMV: about one FLOP per byte of K/V,
// so the tensor core has nothing to do and the kernel is bound by HBM
// ("The FA5090 Optimization Journey" section 2.3 on decode GEMVs).  Each CTA
// owns one (head, key split).  A producer thread streams the split's K and V
// rows (contiguous in memory) into a shared-memory ring with 1-D TMA bulk
// copies guarded by mbarriers; eight consumer warps each take 8 keys of
// every 64-key tile and keep their own online softmax state (running max m,
// running sum l, fp32 accumulator), in the log2 domain with the scale folded
// into one FFMA before ex2.  At the end the warps merge their states and
// the CTA writes either the final O and LSE (one split) or fp32 partials
// (O_split normalised, LSE_split) that the combine kernel merges with
// weights exp(LSE_split - LSE).  The split-KV scheme and its fp32 workspace
// round trip are the ones "The FA5090 Optimization Journey" section 2.7
// measured on prefill.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

struct DecCtl {
  volatile uint32_t* abort;
  unsigned* status;
  unsigned long long timeout;
};

__device__ __forceinline__ bool dec_wait_slow(uint32_t bar, uint32_t parity,
                                           DecCtl c) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*c.abort) return false;
    if (globaltimer_ns() - t0 > c.timeout) {
      *c.abort = 1u;
      atomicExch(c.status, kStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool dec_wait(uint32_t bar, uint32_t parity,
                                         const DecCtl& c) {
  return mbar_try_wait(bar, parity) || dec_wait_slow(bar, parity, c);
}

__device__ __forceinline__ void dec_wait_drain(uint32_t bar, uint32_t parity,
                                            unsigned long long timeout) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout) return;
  }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2_dec(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <int D>
struct DecodeLayout {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = kDecKeysPerTile * kRowBytes;  // K or V
  static constexpr int kStageBytes = 2 * kTileBytes;              // K + V
  static constexpr int kOffRing = 0;
  static constexpr int kOffBars = kDecStages * kStageBytes;
  static constexpr int kNumBars = 2 * kDecStages + 1;  // full, empty, done
  static constexpr int kOffPart = kOffBars + ((kNumBars * 8 + 15) / 16) * 16;
  // per consumer warp: m, l, then D accumulator values
  static constexpr int kPartFloats = 8 * (2 + D);
  static constexpr int kOffAbort = kOffPart + kPartFloats * 4;
  static constexpr int kSmemBytes = kOffAbort + 16 + 128;  // + align slack
  static constexpr int kDims = D / 32;       // accumulator dims per lane
  static constexpr int kChunks = D / 8 / 4;  // 16-byte K chunks per lane
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kDecThreads + 32, 2)
    fa_decode_kernel(const DecodeParams p) {
  using L = DecodeLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kOffBars;
  auto full_bar = [&](int i) { return bars + 8u * i; };
  auto empty_bar = [&](int i) { return bars + 8u * (kDecStages + i); };
  const uint32_t done_bar = bars + 8u * (2 * kDecStages);
  float* part = reinterpret_cast<float*>(smem + L::kOffPart);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem + L::kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = static_cast<int>(blockIdx.x) % p.BH;
  const int split = static_cast<int>(blockIdx.x) / p.BH;
  const int k_begin = split * p.keys_per_split;
  const int k_end = min(p.Skv, k_begin + p.keys_per_split);
  const int n_keys = max(0, k_end - k_begin);
  const int n_tiles = (n_keys + kDecKeysPerTile - 1) / kDecKeysPerTile;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecStages; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), 8);
    }
    mbar_init(done_bar, 8);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  const DecCtl ctl{abort_flag, p.status, p.timeout_ns};

  const size_t head_off = static_cast<size_t>(bh) * p.Skv * D;

  if (warp == 8) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      const uint8_t* kbase = static_cast<const uint8_t*>(p.k) + (head_off + static_cast<size_t>(k_begin) * D) * 2;
      const uint8_t* vbase = static_cast<const uint8_t*>(p.v) + (head_off + static_cast<size_t>(k_begin) * D) * 2;
      int last_fill[kDecStages];
#pragma unroll
      for (int i = 0; i < kDecStages; ++i) last_fill[i] = -1;
#pragma unroll 1
      for (int t = 0; t < n_tiles; ++t) {
        const int slot = t % kDecStages;
        const uint32_t par = static_cast<uint32_t>(((t / kDecStages) & 1) ^ 1);
        if (!dec_wait(empty_bar(slot), par, ctl)) break;
        const int rows = min(kDecKeysPerTile, n_keys - t * kDecKeysPerTile);
        const uint32_t bytes = static_cast<uint32_t>(rows * L::kRowBytes);
        mbar_arrive_expect_tx(full_bar(slot), 2u * bytes);
        const uint32_t dst = sbase + static_cast<uint32_t>(L::kOffRing + slot * L::kStageBytes);
        const size_t src_off = static_cast<size_t>(t) * L::kTileBytes;
        bulk_load_1d(dst, kbase + src_off, bytes, full_bar(slot));
        bulk_load_1d(dst + L::kTileBytes, vbase + src_off, bytes, full_bar(slot));
        last_fill[slot] = t;
      }
#pragma unroll
      for (int i = 0; i < kDecStages; ++i)
        if (last_fill[i] >= 0)
          dec_wait_drain(full_bar(i), static_cast<uint32_t>((last_fill[i] / kDecStages) & 1),
                         p.timeout_ns);
    }
    __syncwarp();
    return;
  }

  // -------------------------------- consumers --------------------------------
  const int g = lane >> 2;   // key within this warp's 8
  const int r4 = lane & 3;   // quarter of the row this lane reads
  const int key_in_tile = warp * 8 + g;
  const float c = p.scale_log2;
  // q chunks this lane multiplies: chunk index (r4 + 4*i + 4*(g&1)) mod (D/8)
  float qv[L::kChunks][8];
  {
    const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.q) + static_cast<size_t>(bh) * D * 2);
#pragma unroll
    for (int i = 0; i < L::kChunks; ++i) {
      const int ch = (r4 + 4 * i + 4 * (g & 1)) % (D / 8);
      const uint4 w = qrow[ch];
      const float2 a = unpack2<BF16>(w.x), b = unpack2<BF16>(w.y);
      const float2 d2 = unpack2<BF16>(w.z), e = unpack2<BF16>(w.w);
      qv[i][0] = a.x; qv[i][1] = a.y; qv[i][2] = b.x; qv[i][3] = b.y;
      qv[i][4] = d2.x; qv[i][5] = d2.y; qv[i][6] = e.x; qv[i][7] = e.y;
    }
  }
  float m = -INFINITY;   // running max (log2 units), warp-uniform
  float l_lane = 0.f;    // this lane's share of the running sum
  float acc[L::kDims];
#pragma unroll
  for (int d = 0; d < L::kDims; ++d) acc[d] = 0.f;
  bool ok = true;

#pragma unroll 1
  for (int t = 0; t < n_tiles; ++t) {
    const int slot = t % kDecStages;
    const bool got = dec_wait(full_bar(slot), static_cast<uint32_t>((t / kDecStages) & 1), ctl);
    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
    const uint32_t kt = sbase + static_cast<uint32_t>(L::kOffRing + slot * L::kStageBytes);
    const uint32_t vt = kt + L::kTileBytes;
    const int valid = min(kDecKeysPerTile, n_keys - t * kDecKeysPerTile);

    // score of key `key_in_tile`: 4 lanes, D/4 dims each
    float dot = 0.f;
    const uint32_t krow = kt + static_cast<uint32_t>(key_in_tile * L::kRowBytes);
#pragma unroll
    for (int i = 0; i < L::kChunks; ++i) {
      const int ch = (r4 + 4 * i + 4 * (g & 1)) % (D / 8);
      uint32_t w0, w1, w2, w3;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                   : "r"(krow + ch * 16));
      const float2 a = unpack2<BF16>(w0), b = unpack2<BF16>(w1);
      const float2 d2 = unpack2<BF16>(w2), e = unpack2<BF16>(w3);
      dot = fmaf(qv[i][0], a.x, dot); dot = fmaf(qv[i][1], a.y, dot);
      dot = fmaf(qv[i][2], b.x, dot); dot = fmaf(qv[i][3], b.y, dot);
      dot = fmaf(qv[i][4], d2.x, dot); dot = fmaf(qv[i][5], d2.y, dot);
      dot = fmaf(qv[i][6], e.x, dot); dot = fmaf(qv[i][7], e.y, dot);
    }
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
    const float tsc = key_in_tile < valid ? dot * c : -INFINITY;
    float tmax = fmaxf(tsc, __shfl_xor_sync(0xffffffffu, tsc, 4));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
    const float m_new = fmaxf(m, tmax);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = ex2_approx(m - m_use);
    const float pk = ex2_approx(tsc - m_use);
    m = m_new;
    l_lane = l_lane * alpha + (r4 == 0 ? pk : 0.f);
#pragma unroll
    for (int d = 0; d < L::kDims; ++d) acc[d] *= alpha;
    // O += p_g * V[g] for the warp's 8 keys; lane owns dims lane*kDims ...
#pragma unroll
    for (int gg = 0; gg < 8; ++gg) {
      const float pg = __shfl_sync(0xffffffffu, pk, gg * 4);
      // rows past the valid keys hold stale bytes (p = 0 but V may be NaN)
      if (warp * 8 + gg >= valid) continue;
      const uint32_t vrow = vt + static_cast<uint32_t>((warp * 8 + gg) * L::kRowBytes + lane * L::kDims * 2);
      if constexpr (L::kDims == 4) {
        uint32_t w0, w1;
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(vrow));
        const float2 a = unpack2<BF16>(w0), b = unpack2<BF16>(w1);
        acc[0] = fmaf(pg, a.x, acc[0]); acc[1] = fmaf(pg, a.y, acc[1]);
        acc[2] = fmaf(pg, b.x, acc[2]); acc[3] = fmaf(pg, b.y, acc[3]);
      } else {
        uint32_t w0;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w0) : "r"(vrow));
        const float2 a = unpack2<BF16>(w0);
        acc[0] = fmaf(pg, a.x, acc[0]); acc[1] = fmaf(pg, a.y, acc[1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(slot));
  }

  // merge the lanes' sums, publish this warp's state
  float l_w = l_lane;
  l_w += __shfl_xor_sync(0xffffffffu, l_w, 4);
  l_w += __shfl_xor_sync(0xffffffffu, l_w, 8);
  l_w += __shfl_xor_sync(0xffffffffu, l_w, 16);
  if (!ok) return;
  float* mine = part + warp * (2 + D);
  if (lane == 0) { mine[0] = m; mine[1] = l_w; }
#pragma unroll
  for (int d = 0; d < L::kDims; ++d) mine[2 + lane * L::kDims + d] = acc[d];
  __syncwarp();
  if (lane == 0) mbar_arrive(done_bar);
  if (warp != 0) return;

  // warp 0 merges the eight warp states
  const bool got = dec_wait(done_bar, 0, ctl);
  if (!__all_sync(0xffffffffu, got)) return;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < 8; ++w) M = fmaxf(M, part[w * (2 + D)]);
  const float M_use = M == -INFINITY ? 0.f : M;
  float Ls = 0.f;
  float o[L::kDims];
#pragma unroll
  for (int d = 0; d < L::kDims; ++d) o[d] = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float* pw = part + w * (2 + D);
    const float sc = ex2_approx(pw[0] - M_use);
    Ls = fmaf(pw[1], sc, Ls);
#pragma unroll
    for (int d = 0; d < L::kDims; ++d) o[d] = fmaf(pw[2 + lane * L::kDims + d], sc, o[d]);
  }
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
  const float lse = Ls > 0.f ? (M + log2f(Ls)) * 0.69314718055994530942f : -INFINITY;
  if (p.n_splits == 1) {
    uint8_t* orow = static_cast<uint8_t*>(p.o) + static_cast<size_t>(bh) * D * 2;
    if constexpr (L::kDims == 4) {
      uint2 w;
      w.x = pack2_dec<BF16>(o[0] * inv, o[1] * inv);
      w.y = pack2_dec<BF16>(o[2] * inv, o[3] * inv);
      *reinterpret_cast<uint2*>(orow + lane * 8) = w;
    } else {
      *reinterpret_cast<uint32_t*>(orow + lane * 4) = pack2_dec<BF16>(o[0] * inv, o[1] * inv);
    }
    if (lane == 0) p.lse[bh] = lse;
  } else {
    float* po = p.part_o + (static_cast<size_t>(split) * p.BH + bh) * D;
#pragma unroll
    for (int d = 0; d < L::kDims; ++d) po[lane * L::kDims + d] = o[d] * inv;
    if (lane == 0) p.part_lse[static_cast<size_t>(split) * p.BH + bh] = lse;
  }
}

// Merge the splits of each head: one warp per head.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
    fa_decode_combine_kernel(const DecodeParams p) {
  constexpr int kDims = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = static_cast<int>(blockIdx.x) * 8 + warp;
  if (bh >= p.BH) return;
  constexpr float kLog2e = 1.4426950408889634f;
  float M = -INFINITY;
  for (int s = 0; s < p.n_splits; ++s) M = fmaxf(M, p.part_lse[static_cast<size_t>(s) * p.BH + bh]);
  const float M_use = M == -INFINITY ? 0.f : M;
  float W = 0.f;
  float o[kDims];
#pragma unroll
  for (int d = 0; d < kDims; ++d) o[d] = 0.f;
  for (int s = 0; s < p.n_splits; ++s) {
    const float ls = p.part_lse[static_cast<size_t>(s) * p.BH + bh];
    const float w = ex2_approx((ls - M_use) * kLog2e);
    W += w;
    const float* po = p.part_o + (static_cast<size_t>(s) * p.BH + bh) * D;
#pragma unroll
    for (int d = 0; d < kDims; ++d) o[d] = fmaf(w, po[lane * kDims + d], o[d]);
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  uint8_t* orow = static_cast<uint8_t*>(p.o) + static_cast<size_t>(bh) * D * 2;
  if constexpr (kDims == 4) {
    uint2 w;
    w.x = pack2_dec<BF16>(o[0] * inv, o[1] * inv);
    w.y = pack2_dec<BF16>(o[2] * inv, o[3] * inv);
    *reinterpret_cast<uint2*>(orow + lane * 8) = w;
  } else {
    *reinterpret_cast<uint32_t*>(orow + lane * 4) = pack2_dec<BF16>(o[0] * inv, o[1] * inv);
  }
  if (lane == 0) p.lse[bh] = W > 0.f ? M + logf(W) : -INFINITY;
}

}  // namespace fa
