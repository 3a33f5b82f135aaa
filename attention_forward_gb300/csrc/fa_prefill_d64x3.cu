// fa_prefill_d64x3.cu -- instantiations and launcher of the three-stage
// prefill kernel for head dimension 64 (fp16 and bf16; whole key range).
#include <mutex>

#include "fa_launch.h"
#include "fa_prefill_d64x3.cuh"

namespace fa {
namespace {

template <bool BF16>
cudaError_t set_smem_attr() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(fa_prefill_d64x3_kernel<BF16>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Prefill3Layout::kSmemBytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

template <bool BF16>
cudaError_t launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                   const CUtensorMap& o, const PrefillParams& p, int grid, cudaStream_t stream) {
  cudaError_t e = set_smem_attr<BF16>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Prefill3Layout::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.overlap_prev ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, fa_prefill_d64x3_kernel<BF16>, q, k, v, o, p);
}

template <bool BF16>
cudaError_t num_regs(int* regs) {
  cudaFuncAttributes a{};
  const cudaError_t e = cudaFuncGetAttributes(&a, fa_prefill_d64x3_kernel<BF16>);
  if (e == cudaSuccess) *regs = a.numRegs;
  return e;
}

}  // namespace

cudaError_t prefill_d64x3_num_regs(bool bf16, int* regs) {
  return bf16 ? num_regs<true>(regs) : num_regs<false>(regs);
}

cudaError_t launch_prefill_d64x3(bool bf16, const CUtensorMap& q, const CUtensorMap& k,
                                 const CUtensorMap& v, const CUtensorMap& o,
                                 const PrefillParams& p, int grid, cudaStream_t stream) {
  return bf16 ? launch<true>(q, k, v, o, p, grid, stream)
              : launch<false>(q, k, v, o, p, grid, stream);
}

}  // namespace fa
