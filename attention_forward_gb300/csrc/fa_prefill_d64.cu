// fa_prefill_d64.cu -- instantiations and launcher of the prefill kernel for
// head dimension 64 (fp16 and bf16; whole key range or split keys; the
// correction-warpgroup form for the whole key range).
#include <mutex>

#include "fa_launch.h"
#include "fa_prefill.cuh"

namespace fa {
namespace {

template <bool BF16, bool kSplit, bool kCorr>
cudaError_t set_smem_attr() {
  // once per (device, kernel)
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(fa_prefill_kernel<64, BF16, kSplit, kCorr>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PrefillLayout<64>::kSmemBytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

template <bool BF16, bool kSplit, bool kCorr = false>
cudaError_t launch(const CUtensorMap& q, const CUtensorMap& k,
                   const CUtensorMap& v, const CUtensorMap& o,
                   const PrefillParams& p, int grid, cudaStream_t stream) {
  cudaError_t e = set_smem_attr<BF16, kSplit, kCorr>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = PrefillLayout<64>::kSmemBytes;
  cfg.stream = stream;
  // overlap with the previous grid on the stream (programmatic dependent
  // launch): the kernel waits for it before its first global write
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.overlap_prev ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fa_prefill_kernel<64, BF16, kSplit, kCorr>, q, k, v, o, p);
}

template <bool BF16, bool kSplit, bool kCorr = false>
cudaError_t num_regs(int* regs) {
  cudaFuncAttributes a{};
  const cudaError_t e = cudaFuncGetAttributes(&a, fa_prefill_kernel<64, BF16, kSplit, kCorr>);
  if (e == cudaSuccess) *regs = a.numRegs;
  return e;
}

}  // namespace

int prefill_smem_bytes_d64() { return PrefillLayout<64>::kSmemBytes; }

// Registers per thread of the three variants (the register split inside the
// kernel assumes the same count for all): that count, or the first one
// that differs from the whole-range variant's.
cudaError_t prefill_num_regs_d64(bool bf16, int* regs) {
  int r0 = 0, r1 = 0, r2 = 0;
  cudaError_t e = bf16 ? num_regs<true, false>(&r0) : num_regs<false, false>(&r0);
  if (e != cudaSuccess) return e;
  e = bf16 ? num_regs<true, true>(&r1) : num_regs<false, true>(&r1);
  if (e != cudaSuccess) return e;
  e = bf16 ? num_regs<true, false, true>(&r2) : num_regs<false, false, true>(&r2);
  if (e != cudaSuccess) return e;
  *regs = r0 == r1 && r0 == r2 ? r0 : (r0 != 128 ? r0 : (r1 != 128 ? r1 : r2));
  return cudaSuccess;
}

cudaError_t launch_prefill_d64(bool bf16, bool corr, const CUtensorMap& q,
                               const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& o, const PrefillParams& p,
                               int grid, cudaStream_t stream) {
  if (p.n_splits > 1)
    return bf16 ? launch<true, true>(q, k, v, o, p, grid, stream)
                : launch<false, true>(q, k, v, o, p, grid, stream);
  if (corr)
    return bf16 ? launch<true, false, true>(q, k, v, o, p, grid, stream)
                : launch<false, false, true>(q, k, v, o, p, grid, stream);
  return bf16 ? launch<true, false>(q, k, v, o, p, grid, stream)
              : launch<false, false>(q, k, v, o, p, grid, stream);
}

}  // namespace fa
