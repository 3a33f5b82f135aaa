// fa_host.h -- host-side helpers of fa_api.cu that other host translation
// units of the library use (internal; no device code).
#pragma once
#include "../../include/fa.h"

namespace fa {

// The argument checks of fa_fwd and the current device's support check
// (compute capability 10.3, the library's static arrays reachable), in that
// order; launches and allocates nothing.
fa_status_t check_call(const void* q, const void* k, const void* v, const void* o,
                       const void* lse, int B, int H, int Sq, int Skv, int D,
                       float scale, int dtype);

// The current device's support check alone (compute capability 10.3).
fa_status_t check_device();

// Process-unique id of the calling thread's current CUDA context (0 when
// there is none).  Device addresses of the library's static __device__
// arrays belong to the context that loaded the module: after
// cudaDeviceReset the primary context is a new one, with a new id, and every
// cached address must be looked up again.
unsigned long long context_id();

}  // namespace fa
