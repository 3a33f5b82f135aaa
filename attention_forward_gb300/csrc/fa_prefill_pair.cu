// fa_prefill_pair.cu -- instantiations and launcher of the CTA-pair prefill
// kernel (head dimension 128, fp16 and bf16, whole key range; merged or
// correction-warpgroup form, and the merged form with the tail split),
// launched with clusters of two CTAs.
#include <mutex>

#include "fa_launch.h"
#include "fa_prefill_pair.cuh"
#include "fa_prefill_pair64.cuh"

namespace fa {
namespace {

template <bool BF16, bool kCorr, bool kTail = false>
cudaError_t set_attrs() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(fa_prefill_pair_kernel<BF16, kCorr, kTail>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, PairLayout::kSmemBytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

// attr must hold 2 entries: the cluster shape, and (overlap) programmatic
// stream serialization: the kernel then overlaps the previous grid on the
// stream and waits for it before its first global write.
cudaLaunchConfig_t pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr,
                               bool overlap = false) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = PairLayout::kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 2 : 1;
  return cfg;
}

template <bool BF16, bool kCorr, bool kTail = false>
cudaError_t launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                   const CUtensorMap& o, const PrefillParams& p, int n_pairs,
                   cudaStream_t stream) {
  cudaError_t e = set_attrs<BF16, kCorr, kTail>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_config(2 * n_pairs, stream, attr, p.overlap_prev != 0);
  return cudaLaunchKernelEx(&cfg, fa_prefill_pair_kernel<BF16, kCorr, kTail>, q, k, v, o, p);
}

// Every form has the same shared memory and threads, so the same number of
// pairs fits; the merged form is queried.
template <bool BF16>
cudaError_t max_pairs(int* n) {
  cudaError_t e = set_attrs<BF16, false>();
  if (e != cudaSuccess) return e;
  e = set_attrs<BF16, true>();
  if (e != cudaSuccess) return e;
  e = set_attrs<BF16, false, true>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_config(2, nullptr, attr);
  return cudaOccupancyMaxActiveClusters(n, fa_prefill_pair_kernel<BF16, false>, &cfg);
}

// Registers per thread of the three forms: their count, or the first that
// is not 128 (the register split assumes 128).
template <bool BF16>
cudaError_t num_regs(int* regs) {
  cudaFuncAttributes a{}, b{}, c{};
  cudaError_t e = cudaFuncGetAttributes(&a, fa_prefill_pair_kernel<BF16, false>);
  if (e != cudaSuccess) return e;
  e = cudaFuncGetAttributes(&b, fa_prefill_pair_kernel<BF16, true>);
  if (e != cudaSuccess) return e;
  e = cudaFuncGetAttributes(&c, fa_prefill_pair_kernel<BF16, false, true>);
  if (e == cudaSuccess)
    *regs = a.numRegs != 128 ? a.numRegs : (b.numRegs != 128 ? b.numRegs : c.numRegs);
  return e;
}

// The 64-key kernel (fa_prefill_pair64.cuh).
template <bool BF16>
cudaError_t set_attrs64() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(fa_prefill_pair64_kernel<BF16>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, Pair64Layout::kSmemBytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

template <bool BF16>
cudaError_t launch64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                     const CUtensorMap& o, const PrefillParams& p, int n_pairs,
                     cudaStream_t stream) {
  cudaError_t e = set_attrs64<BF16>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config(2 * n_pairs, stream, attr);
  cfg.dynamicSmemBytes = Pair64Layout::kSmemBytes;
  return cudaLaunchKernelEx(&cfg, fa_prefill_pair64_kernel<BF16>, q, k, v, o, p);
}

template <bool BF16>
cudaError_t max_pairs64(int* n) {
  cudaError_t e = set_attrs64<BF16>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config(2, nullptr, attr);
  cfg.dynamicSmemBytes = Pair64Layout::kSmemBytes;
  return cudaOccupancyMaxActiveClusters(n, fa_prefill_pair64_kernel<BF16>, &cfg);
}

template <bool BF16>
cudaError_t num_regs64(int* regs) {
  cudaFuncAttributes a{};
  const cudaError_t e = cudaFuncGetAttributes(&a, fa_prefill_pair64_kernel<BF16>);
  if (e == cudaSuccess) *regs = a.numRegs;
  return e;
}

}  // namespace

cudaError_t prefill_pair64_max_pairs(bool bf16, int* n) {
  return bf16 ? max_pairs64<true>(n) : max_pairs64<false>(n);
}

cudaError_t prefill_pair64_num_regs(bool bf16, int* regs) {
  return bf16 ? num_regs64<true>(regs) : num_regs64<false>(regs);
}

cudaError_t launch_prefill_pair64(bool bf16, const CUtensorMap& q, const CUtensorMap& k,
                                  const CUtensorMap& v, const CUtensorMap& o,
                                  const PrefillParams& p, int n_pairs, cudaStream_t stream) {
  return bf16 ? launch64<true>(q, k, v, o, p, n_pairs, stream)
              : launch64<false>(q, k, v, o, p, n_pairs, stream);
}

cudaError_t prefill_pair_max_pairs(bool bf16, int* n) {
  return bf16 ? max_pairs<true>(n) : max_pairs<false>(n);
}

cudaError_t prefill_pair_num_regs(bool bf16, int* regs) {
  return bf16 ? num_regs<true>(regs) : num_regs<false>(regs);
}

cudaError_t launch_prefill_pair(bool bf16, bool corr, const CUtensorMap& q,
                                const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const PrefillParams& p, int n_pairs,
                                cudaStream_t stream) {
  if (p.tail_items > 0)  // the tail split (merged form only)
    return bf16 ? launch<true, false, true>(q, k, v, o, p, n_pairs, stream)
                : launch<false, false, true>(q, k, v, o, p, n_pairs, stream);
  if (corr)
    return bf16 ? launch<true, true>(q, k, v, o, p, n_pairs, stream)
                : launch<false, true>(q, k, v, o, p, n_pairs, stream);
  return bf16 ? launch<true, false>(q, k, v, o, p, n_pairs, stream)
              : launch<false, false>(q, k, v, o, p, n_pairs, stream);
}

}  // namespace fa
