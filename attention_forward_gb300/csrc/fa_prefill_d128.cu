// fa_prefill_d128.cu -- instantiations and launcher of the prefill kernel for
// head dimension 128 (fp16 and bf16).
#include <mutex>

#include "fa_launch.h"
#include "fa_prefill.cuh"

namespace fa {
namespace {

template <bool BF16>
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
  e = cudaFuncSetAttribute(fa_prefill_kernel<128, BF16>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PrefillLayout<128>::kSmemBytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

template <bool BF16>
cudaError_t launch(const CUtensorMap& q, const CUtensorMap& k,
                   const CUtensorMap& v, const CUtensorMap& o,
                   const PrefillParams& p, int grid, cudaStream_t stream) {
  cudaError_t e = set_smem_attr<BF16>();
  if (e != cudaSuccess) return e;
  fa_prefill_kernel<128, BF16><<<grid, kThreads, PrefillLayout<128>::kSmemBytes,
                                stream>>>(q, k, v, o, p);
  return cudaGetLastError();
}

}  // namespace

int prefill_smem_bytes_d128() { return PrefillLayout<128>::kSmemBytes; }

cudaError_t prefill_num_regs_d128(bool bf16, int* regs) {
  cudaFuncAttributes a{};
  cudaError_t e = bf16 ? cudaFuncGetAttributes(&a, fa_prefill_kernel<128, true>)
                       : cudaFuncGetAttributes(&a, fa_prefill_kernel<128, false>);
  if (e == cudaSuccess) *regs = a.numRegs;
  return e;
}

cudaError_t launch_prefill_d128(bool bf16, const CUtensorMap& q,
                               const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& o, const PrefillParams& p,
                               int grid, cudaStream_t stream) {
  return bf16 ? launch<true>(q, k, v, o, p, grid, stream)
              : launch<false>(q, k, v, o, p, grid, stream);
}

}  // namespace fa
