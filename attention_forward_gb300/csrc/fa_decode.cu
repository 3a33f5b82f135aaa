// fa_decode.cu -- instantiations and launchers of the decode (Sq == 1)
// split-KV kernel and its combine kernel.
#include <mutex>

#include "fa_decode.cuh"
#include "fa_launch.h"

namespace fa {
namespace {

template <int D, bool BF16>
cudaError_t set_smem_attr() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(fa_decode_kernel<D, BF16>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DecodeLayout<D>::kSmemBytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

template <int D, bool BF16>
cudaError_t launch(const DecodeParams& p, int grid, cudaStream_t stream) {
  cudaError_t e = set_smem_attr<D, BF16>();
  if (e != cudaSuccess) return e;
  fa_decode_kernel<D, BF16><<<grid, kDecThreads + 32,
                              DecodeLayout<D>::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t combine(const DecodeParams& p, cudaStream_t stream) {
  fa_decode_combine_kernel<D, BF16><<<(p.BH + 7) / 8, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int decode_smem_bytes(int D) {
  return D == 128 ? DecodeLayout<128>::kSmemBytes : DecodeLayout<64>::kSmemBytes;
}

cudaError_t launch_decode(int D, bool bf16, const DecodeParams& p, int grid,
                          cudaStream_t stream) {
  if (D == 128) return bf16 ? launch<128, true>(p, grid, stream) : launch<128, false>(p, grid, stream);
  return bf16 ? launch<64, true>(p, grid, stream) : launch<64, false>(p, grid, stream);
}

cudaError_t launch_decode_combine(int D, bool bf16, const DecodeParams& p,
                                  cudaStream_t stream) {
  if (D == 128) return bf16 ? combine<128, true>(p, stream) : combine<128, false>(p, stream);
  return bf16 ? combine<64, true>(p, stream) : combine<64, false>(p, stream);
}

}  // namespace fa
