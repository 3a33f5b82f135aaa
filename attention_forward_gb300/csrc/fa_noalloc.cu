// fa_noalloc.cu -- fa_fwd_decode_static: the decode forward pass for callers
// that cannot allocate device memory.
//
// The split-KV decode needs scratch for its per-split partial results.
// fa_fwd allocates that scratch on its first decode call and fa_fwd_ex takes
// it from the caller; both need a cudaMalloc somewhere.  Some callers cannot
// make one: a host framework that owns every device allocation through its
// own allocator and forbids side allocations, a latency-critical serving loop
// that must never hit cudaMalloc's implicit device synchronisation or its
// run-time failure, or a process whose memory budget is fixed up front.  For
// them the scratch lives in a file-scope __device__ array that is part of
// the library's module image: it is created when the library's module is
// loaded on a GPU and stays there until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fa.h"
#include "fa_host.h"

namespace {

// Capacity of the static decode scratch (FA_DECODE_STATIC_SCRATCH_BYTES).
constexpr size_t kScratchBytes = FA_DECODE_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// The scratch's device address per device, with the context it belongs to.
struct ScratchAddr {
  unsigned long long ctx;
  void* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress: looked up once per device (with that device
// current), and again if the device's context has changed since (after
// cudaDeviceReset the module, and the array with it, is loaded anew).
fa_status_t scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  const unsigned long long ctx = fa::context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchAddr& a = g_scratch[dev];
  if (!a.ptr || a.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) {
      cudaGetLastError();  // leave no pending error behind
      a = ScratchAddr{0, nullptr};
      return FA_ERR_CUDA;
    }
    a = ScratchAddr{ctx, p};
  }
  *out = a.ptr;
  return FA_OK;
}

}  // namespace

extern "C" fa_status_t fa_fwd_decode_static(const void* q, const void* k,
                                            const void* v, void* o, float* lse,
                                            int B, int H, int Skv, int D,
                                            float scale, int dtype,
                                            fa_stream_t stream) {
  // the arguments and the device first (an unsupported device gets
  // FA_ERR_UNSUPPORTED, as from fa_fwd), then the scratch's capacity
  const fa_status_t chk = fa::check_call(q, k, v, o, lse, B, H, 1, Skv, D, scale, dtype);
  if (chk != FA_OK) return chk;
  // the partials of the library's split choice must fit the static array
  const size_t need = fa_workspace_bytes(B, H, 1, Skv, D, 0);
  if (need > kScratchBytes) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const fa_status_t st = scratch_for_current_device(&scratch);
    if (st != FA_OK) return st;
  }
  // the existing decode path, with the static array as its workspace
  return fa_fwd_ex(q, k, v, o, lse, B, H, 1, Skv, D, scale, 0, dtype, 0u, 0,
                   scratch, need > 0 ? kScratchBytes : 0, stream);
}
