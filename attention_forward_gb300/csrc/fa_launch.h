// fa_launch.h -- host-side launch entry points of the kernels (internal).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"

namespace fa {

// Dynamic shared memory a prefill CTA needs (bytes).
int prefill_smem_bytes(int D);
// Registers per thread the compiled prefill kernel was built with.
cudaError_t prefill_num_regs(int D, bool bf16, int* regs);
// corr: the correction-warpgroup form (ignored with split keys)
cudaError_t launch_prefill(int D, bool bf16, bool corr, const CUtensorMap& q,
                           const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& o, const PrefillParams& p,
                           int grid, cudaStream_t stream);

// CTA-pair prefill (D = 128, whole key range): registers per thread, the
// number of two-CTA clusters that fit on the device, and the launch (the
// tail-split form when p.tail_items > 0, which excludes corr).
cudaError_t prefill_pair_num_regs(bool bf16, int* regs);
cudaError_t prefill_pair_max_pairs(bool bf16, int* n);
cudaError_t launch_prefill_pair(bool bf16, bool corr, const CUtensorMap& q,
                                const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const PrefillParams& p, int n_pairs,
                                cudaStream_t stream);

// The CTA-pair kernel with 64-key score tiles, two score buffers per stage.
cudaError_t prefill_pair64_num_regs(bool bf16, int* regs);
cudaError_t prefill_pair64_max_pairs(bool bf16, int* n);
cudaError_t launch_prefill_pair64(bool bf16, const CUtensorMap& q, const CUtensorMap& k,
                                  const CUtensorMap& v, const CUtensorMap& o,
                                  const PrefillParams& p, int n_pairs, cudaStream_t stream);

// The three-stage prefill kernel for D = 64 (whole key range; 96-key tiles,
// 384-row items): registers per thread and the launch.
cudaError_t prefill_d64x3_num_regs(bool bf16, int* regs);
cudaError_t launch_prefill_d64x3(bool bf16, const CUtensorMap& q, const CUtensorMap& k,
                                 const CUtensorMap& v, const CUtensorMap& o,
                                 const PrefillParams& p, int grid, cudaStream_t stream);

int decode_smem_bytes(int D);
cudaError_t launch_decode(int D, bool bf16, const DecodeParams& p, int grid,
                          cudaStream_t stream);
cudaError_t launch_decode_combine(int D, bool bf16, const DecodeParams& p,
                                  cudaStream_t stream);

}  // namespace fa
