// fa_diag.cu -- device self-check of the exponential the kernels use.
//
// The softmax of every kernel evaluates p = 2^x with the PTX instruction
// ex2.approx.ftz.f32 (the exp2 form of "The FA5090 Optimization Journey",
// section 2.6, which folds log2(e) into the score scale).  Masked scores are
// -inf, so the kernels rely on ex2(-inf) = +0 and on ex2(0) = 1 for the row
// maximum; fa_ex2_approx runs that same instruction (the same wrapper) on
// caller data so that a test can check these values and its accuracy on
// the device.
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_host.h"
#include "sm103_ptx.cuh"

namespace {

__global__ void ex2_kernel(const float* __restrict__ x, float* __restrict__ y, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) y[i] = fa::ex2_approx(x[i]);
}

}  // namespace

extern "C" fa_status_t fa_ex2_approx(const float* x, float* y, int n, fa_stream_t stream) {
  if (!x || !y || n < 1 || n > (1 << 28)) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u))
    return FA_ERR_INVALID_ARG;
  const fa_status_t st = fa::check_device();
  if (st != FA_OK) return st;
  constexpr int kBlock = 256;
  ex2_kernel<<<(n + kBlock - 1) / kBlock, kBlock, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      x, y, n);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
