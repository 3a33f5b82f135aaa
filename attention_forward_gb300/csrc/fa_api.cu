// fa_api.cu -- the C ABI of libfa_gb300.so (declared in include/fa.h):
// argument validation, device checks, TMA descriptor encoding, workspace
// handling and dispatch to the prefill or decode kernels.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/fa.h"
#include "fa_host.h"
#include "fa_internal.h"
#include "fa_launch.h"

namespace fa {

int prefill_smem_bytes_d128();
int prefill_smem_bytes_d64();
cudaError_t prefill_num_regs_d128(bool bf16, int* regs);
cudaError_t prefill_num_regs_d64(bool bf16, int* regs);
cudaError_t launch_prefill_d128(bool, bool, const CUtensorMap&, const CUtensorMap&,
                                const CUtensorMap&, const CUtensorMap&,
                                const PrefillParams&, int, cudaStream_t);
cudaError_t launch_prefill_d64(bool, bool, const CUtensorMap&, const CUtensorMap&,
                               const CUtensorMap&, const CUtensorMap&,
                               const PrefillParams&, int, cudaStream_t);

int prefill_smem_bytes(int D) {
  return D == 128 ? prefill_smem_bytes_d128() : prefill_smem_bytes_d64();
}
cudaError_t prefill_num_regs(int D, bool bf16, int* regs) {
  return D == 128 ? prefill_num_regs_d128(bf16, regs)
                  : prefill_num_regs_d64(bf16, regs);
}
cudaError_t launch_prefill(int D, bool bf16, bool corr, const CUtensorMap& q,
                           const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& o, const PrefillParams& p,
                           int grid, cudaStream_t stream) {
  return D == 128 ? launch_prefill_d128(bf16, corr, q, k, v, o, p, grid, stream)
                  : launch_prefill_d64(bf16, corr, q, k, v, o, p, grid, stream);
}

}  // namespace fa

namespace {

// Device status word: kernels record FA_ERR_TIMEOUT here.
__device__ unsigned g_status_word;

// Slots of the prefill kernel's item scheduler (see PrefillParams::sched);
// zero at load, and cleared again by the last CTA of every launch.
__device__ unsigned long long g_sched[2 * (fa::kSchedSlots + fa::kGraphSchedSlots)];
// Prefill launches of this process, numbered to pick a scheduler slot: two
// direct launches can share a slot only 1024 launches apart.
std::atomic<unsigned> g_launch_seq{0};
// Prefill launches captured into CUDA graphs: each takes a slot of its own
// (a graph replays with the slot it was captured with, on any stream), out
// of a pool of 4096 that direct launches never use.
std::atomic<unsigned> g_capture_seq{0};

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWatchdogNs = 1000000000ull;
std::atomic<unsigned long long> g_watchdog_ns{kDefaultWatchdogNs};

struct DeviceState {
  bool probed = false;
  unsigned long long ctx_id = 0;  // the context the addresses below belong to
  fa_status_t usable = FA_ERR_UNSUPPORTED;
  int sm_count = 0;
  unsigned* status = nullptr;
  unsigned long long* sched = nullptr;  // g_sched on this device
  bool regs_ok[2][2] = {};  // [D==128][bf16]
  bool regs_checked[2][2] = {};
  // the CTA-pair kernel (D = 128): register check and the number of pairs
  // (two-CTA clusters) that fit on the device at once, per dtype
  bool pair_checked[2] = {};
  int pair_slots[2] = {};  // 0: not usable
  bool pair64_checked[2] = {};
  int pair64_slots[2] = {};  // the 64-key pair kernel; 0: not usable
  bool d64x3_checked[2] = {};
  bool d64x3_ok[2] = {};     // the three-stage D = 64 kernel, per dtype
  // fa_fwd's workspaces for split partials, one per stream handle (calls on
  // one stream run in order; calls on different streams may overlap)
  struct StreamWorkspace {
    cudaStream_t stream;
    void* ptr;
    size_t bytes;
    // the pair kernel's tail-split arrival counters: a block of their own
    // (no other call writes it), zeroed when made, and the epoch of the
    // last launch that used them on this stream
    unsigned long long* tail_ctr = nullptr;
    size_t tail_ctr_n = 0;
    unsigned tail_epoch = 0;
  };
  std::vector<StreamWorkspace> workspaces;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;

fa_status_t get_encoder() {
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? FA_OK : FA_ERR_CUDA;
}

// Current device's state; checks compute capability 10.3 once per context.
// A device whose context changed since the last probe (cudaDeviceReset makes
// a new primary context) is probed again: the static arrays' addresses are
// looked up anew, and the workspaces of the old context, which went away
// with it, are forgotten.
fa_status_t current_device(DeviceState** out, int* dev_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  const unsigned long long ctx = fa::context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (d.probed && d.usable == FA_OK && ctx != d.ctx_id) d = DeviceState{};
  if (!d.probed) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    d.probed = true;
    d.sm_count = sms;
    if (major != 10 || minor != 3) {
      d.usable = FA_ERR_UNSUPPORTED;
    } else {
      void* addr = nullptr;
      void* sched = nullptr;
      if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess ||
          cudaGetSymbolAddress(&sched, g_sched) != cudaSuccess) {
        cudaGetLastError();  // leave no pending error behind
        d.probed = false;
        return FA_ERR_CUDA;
      }
      // the lookup made the device's context current if it was not yet
      d.ctx_id = fa::context_id();
      d.status = static_cast<unsigned*>(addr);
      d.sched = static_cast<unsigned long long*>(sched);
      d.usable = FA_OK;
    }
  }
  if (d.usable != FA_OK) return d.usable;
  *out = &d;
  if (dev_out) *dev_out = dev;
  return FA_OK;
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

fa_status_t validate(const void* q, const void* k, const void* v, const void* o,
                     const void* lse, int B, int H, int Sq, int Skv, int D,
                     float scale, int dtype) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Sq < 1 || Skv < 1) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H >= 65536) return FA_ERR_INVALID_ARG;
  if (Sq > (1 << 24) || Skv > (1 << 24)) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// 3-D view [B*H, S, D] of a [B,H,S,D] tensor; boxes of 64 columns x rows.
fa_status_t encode_3d(CUtensorMap* m, const void* base, int D, int S, int BH,
                      int box_rows, bool bf16) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(S) * D * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = g_encode(
      m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
      const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// The scheduler slot of one prefill launch (see g_launch_seq, g_capture_seq).
unsigned long long* sched_slot(const DeviceState& d, bool captured) {
  const unsigned n = captured
      ? fa::kSchedSlots + g_capture_seq.fetch_add(1) % fa::kGraphSchedSlots
      : g_launch_seq.fetch_add(1) % fa::kSchedSlots;
  return d.sched + 2 * static_cast<size_t>(n);
}

// fa_fwd's workspace for `stream` on this device, grown to `need` bytes.
fa_status_t stream_workspace(DeviceState& d, cudaStream_t stream, size_t need, void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& w : d.workspaces) {
    if (w.stream != stream) continue;
    if (w.bytes < need) {
      cudaFree(w.ptr);  // waits for the work that used it
      w.ptr = nullptr;
      w.bytes = 0;
      if (cudaMalloc(&w.ptr, need) != cudaSuccess) return FA_ERR_CUDA;
      w.bytes = need;
    }
    *out = w.ptr;
    return FA_OK;
  }
  void* ptr = nullptr;
  if (cudaMalloc(&ptr, need) != cudaSuccess) return FA_ERR_CUDA;
  d.workspaces.push_back({stream, ptr, need});
  *out = ptr;
  return FA_OK;
}

// The tail split's memory for `stream`: its partials in the stream's
// workspace (grown to `part_bytes`) and `n_ctr` arrival counters, with the
// launch's epoch.  A new counter block is zeroed on the stream and its
// epochs start again at 1.
fa_status_t stream_tail_state(DeviceState& d, cudaStream_t stream, size_t part_bytes,
                              size_t n_ctr, void** part, unsigned long long** ctr,
                              unsigned* epoch) {
  fa_status_t st = stream_workspace(d, stream, part_bytes, part);
  if (st != FA_OK) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& w : d.workspaces) {
    if (w.stream != stream) continue;
    if (w.tail_ctr_n < n_ctr) {
      if (w.tail_ctr) cudaFree(w.tail_ctr);  // waits for the work that used it
      w.tail_ctr = nullptr;
      w.tail_ctr_n = 0;
      void* p = nullptr;
      if (cudaMalloc(&p, n_ctr * sizeof(unsigned long long)) != cudaSuccess) return FA_ERR_CUDA;
      w.tail_ctr = static_cast<unsigned long long*>(p);
      w.tail_ctr_n = n_ctr;
      if (cudaMemsetAsync(p, 0, n_ctr * sizeof(unsigned long long), stream) != cudaSuccess)
        return FA_ERR_CUDA;
      w.tail_epoch = 0;
    }
    if (++w.tail_epoch == 0) w.tail_epoch = 1;
    *ctr = w.tail_ctr;
    *epoch = w.tail_epoch;
    return FA_OK;
  }
  return FA_ERR_CUDA;  // stream_workspace made the entry
}

// Prefill key splits: only when the (query tile, head) items are fewer than
// the SMs.  Picks the split count with the smallest estimated time, counted
// in key tiles: rounds of one item per SM times the tiles of a range, plus
// eight tiles for the combine kernel and the fp32 partials when split (on
// GB300 a 1024-key item split in two measured slower than unsplit); ties go
// to fewer splits.  An explicit num_splits >= 1 is taken as is (capped at
// the key tiles).
int prefill_splits(int BH, int Sq, int Skv, int sm_count, int num_splits) {
  const long long n_base = static_cast<long long>((Sq + fa::kRowsPerCta - 1) / fa::kRowsPerCta) * BH;
  const int n_tiles = (Skv + fa::kBN - 1) / fa::kBN;
  if (num_splits >= 1) return std::min(num_splits, n_tiles);
  const long long sms = sm_count > 0 ? sm_count : 148;
  if (n_base >= sms) return 1;
  constexpr long long kCombineTiles = 8;
  int best = 1;
  long long best_cost = n_tiles;
  for (int s = 2; s <= std::min(n_tiles, 64); ++s) {
    const int tps = (n_tiles + s - 1) / s;
    const int s_eff = (n_tiles + tps - 1) / tps;
    const long long rounds = (n_base * s_eff + sms - 1) / sms;
    const long long cost = rounds * tps + kCombineTiles;
    if (cost < best_cost) {
      best_cost = cost;
      best = s_eff;
    }
  }
  return best;
}

size_t prefill_ws_bytes(int BH, int Sq, int D, int n_splits) {
  if (n_splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(n_splits) * BH * Sq;
  return ((rows * D * sizeof(float) + 255) / 256) * 256 + ((rows * sizeof(float) + 255) / 256) * 256;
}

// The library runs prefill on CTA pairs where they measured faster than
// single CTAs on GB300: long rows (non-causal from 1024 queries and keys,
// causal from 8192), and at least one 512-row item per pair of SMs.
bool pair_by_default(int BH, int Sq, int Skv, int causal, int sm_count) {
  const long long items = static_cast<long long>(BH) * ((Sq + 511) / 512);
  if (items < (sm_count > 0 ? sm_count / 2 : 76)) return false;
  return causal ? Sq >= 8192 : (Sq >= 1024 && Skv >= 1024);
}

// The CTA-pair kernel's tail split: the pair items of a partly idle last
// round whose key quarters, run as items of their own, fit in at most three
// quarter-rounds (the last round then takes at most three quarters of an
// item's time).  Non-causal only (causal launches run heaviest first and end
// on their lightest items), at least one full round and four key tiles.
int pair_tail_items(long long n_items, long long n_pairs, int causal, int Skv) {
  if (causal || n_pairs <= 0 || n_items <= n_pairs) return 0;
  if ((Skv + fa::kBN - 1) / fa::kBN < 4) return 0;
  const long long rem = n_items % n_pairs;
  if (rem == 0 || 4 * rem > 3 * n_pairs) return 0;
  return static_cast<int>(rem);
}

// fa_fwd's tail-split memory for `tail` items: fp32 O / l and LSE of every
// quarter's 512 rows, and 16 arrival counters (2 stages x 2 CTAs x 4 warps)
// per item.
size_t tail_part_o_bytes(int tail) {
  return ((static_cast<size_t>(tail) * 4 * 512 * 128 * sizeof(float) + 255) / 256) * 256;
}
size_t tail_part_bytes(int tail) {
  return tail_part_o_bytes(tail) + static_cast<size_t>(tail) * 4 * 512 * sizeof(float);
}

// Pairs the pair kernel (or the 64-key one) keeps on the device at once, per
// dtype (0: not usable); checks the kernel's registers on first use.
fa_status_t pair_slots(DeviceState& d, bool bf16, bool k64, int* out) {
  const int ti = bf16 ? 1 : 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!k64 && !d.pair_checked[ti]) {
    int regs = 0, n = 0;
    if (fa::prefill_pair_num_regs(bf16, &regs) != cudaSuccess) return FA_ERR_CUDA;
    if (regs == 128 && fa::prefill_pair_max_pairs(bf16, &n) != cudaSuccess) return FA_ERR_CUDA;
    d.pair_checked[ti] = true;
    d.pair_slots[ti] = regs == 128 ? n : 0;
  }
  if (k64 && !d.pair64_checked[ti]) {
    int regs = 0, n = 0;
    if (fa::prefill_pair64_num_regs(bf16, &regs) != cudaSuccess) return FA_ERR_CUDA;
    if (regs == 128 && fa::prefill_pair64_max_pairs(bf16, &n) != cudaSuccess) return FA_ERR_CUDA;
    d.pair64_checked[ti] = true;
    d.pair64_slots[ti] = regs == 128 ? n : 0;
  }
  *out = k64 ? d.pair64_slots[ti] : d.pair_slots[ti];
  return FA_OK;
}

// Prefill by CTA pairs (FA_FLAG_PAIR, D = 128, whole key range): items of 512
// query rows, a persistent grid of two-CTA clusters.
fa_status_t run_prefill_pair(DeviceState& d, const void* q, const void* k, const void* v,
                             void* o, float* lse, int BH, int Sq, int Skv, float scale,
                             int causal, bool bf16, unsigned flags, bool captured,
                             cudaStream_t stream) {
  const bool k64 = (flags & FA_FLAG_PAIR64) != 0;
  int slots = 0;
  fa_status_t st = pair_slots(d, bf16, k64, &slots);
  if (st != FA_OK) return st;
  if (slots <= 0) return FA_ERR_UNSUPPORTED;
  constexpr int D = 128;
  // a CTA loads half of every key tile (64 of 128 keys, or 32 of 64) and
  // half of every value tile's columns (all of its 128 or 64 keys)
  const int key_tile = k64 ? 64 : fa::kBN;
  CUtensorMap tq, tk, tv, to;
  if ((st = encode_3d(&tq, q, D, Sq, BH, fa::kBM, bf16)) != FA_OK) return st;
  if ((st = encode_3d(&tk, k, D, Skv, BH, key_tile / 2, bf16)) != FA_OK) return st;
  if ((st = encode_3d(&tv, v, D, Skv, BH, key_tile, bf16)) != FA_OK) return st;
  if ((st = encode_3d(&to, o, D, Sq, BH, 32, bf16)) != FA_OK) return st;
  fa::PrefillParams p{};
  p.lse = lse;
  p.status = d.status;
  p.timeout_ns = g_watchdog_ns.load();
  p.BH = BH;
  p.Sq = Sq;
  p.Skv = Skv;
  p.n_qtiles = (Sq + 511) / 512;
  p.causal = causal ? 1 : 0;
  p.lpt = (flags & FA_FLAG_NO_LPT) ? 0 : 1;
  p.always_rescale = (flags & FA_FLAG_ALWAYS_RESCALE) ? 1 : 0;
  p.test_stall = (flags & FA_FLAG_TEST_STALL) ? 1 : 0;
  // the 64-key pair kernel has no programmatic-launch waits: never overlapped
  p.overlap_prev = (flags & FA_FLAG_OVERLAP_PREVIOUS) && !k64 ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.rescale_tau = (flags & FA_FLAG_EXACT_MAX) ? 0.f : 8.f;
  p.n_splits = 1;
  p.tiles_per_split = (Skv + fa::kBN - 1) / fa::kBN;
  const long long n_items = static_cast<long long>(p.n_qtiles) * BH;
  if (n_items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.n_items = static_cast<int>(n_items);
  const int n_pairs = static_cast<int>(std::min<long long>(n_items, slots));
  // the tail split, when asked for (not in the 64-key kernel, not inside a
  // capture: a replay may run on any stream, and the counters' epoch is the
  // launch's)
  const int tail = k64 || captured || !(flags & FA_FLAG_TAIL_SPLIT) ||
                           (flags & FA_FLAG_CORRECTION_WG)
                       ? 0 : pair_tail_items(n_items, n_pairs, causal, Skv);
  if (tail > 0) {
    if (n_items + 3LL * tail > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
    void* part = nullptr;
    if ((st = stream_tail_state(d, stream, tail_part_bytes(tail), static_cast<size_t>(tail) * 16,
                                &part, &p.tail_count, &p.tail_epoch)) != FA_OK)
      return st;
    p.part_o = static_cast<float*>(part);
    p.part_lse = reinterpret_cast<float*>(static_cast<char*>(part) + tail_part_o_bytes(tail));
    p.o = o;
    p.tail_items = tail;
    p.n_items = static_cast<int>(n_items + 3LL * tail);
  }
  p.sched = sched_slot(d, captured);
  const cudaError_t e =
      k64 ? fa::launch_prefill_pair64(bf16, tq, tk, tv, to, p, n_pairs, stream)
          : fa::launch_prefill_pair(bf16, (flags & FA_FLAG_CORRECTION_WG) != 0, tq, tk, tv, to,
                                    p, n_pairs, stream);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

// Prefill at D = 64 by the three-stage kernel (FA_FLAG_D64_THREE_STAGE): items
// of 384 query rows, 96-key tiles, one persistent CTA per SM.
fa_status_t run_prefill_d64x3(DeviceState& d, const void* q, const void* k, const void* v,
                              void* o, float* lse, int BH, int Sq, int Skv, float scale,
                              int causal, bool bf16, unsigned flags, bool captured,
                              cudaStream_t stream) {
  const int ti = bf16 ? 1 : 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!d.d64x3_checked[ti]) {
      int regs = 0;
      if (fa::prefill_d64x3_num_regs(bf16, &regs) != cudaSuccess) return FA_ERR_CUDA;
      d.d64x3_checked[ti] = true;
      d.d64x3_ok[ti] = regs == 128;
    }
    if (!d.d64x3_ok[ti]) return FA_ERR_UNSUPPORTED;
  }
  constexpr int D = 64;
  CUtensorMap tq, tk, tv, to;
  fa_status_t st;
  if ((st = encode_3d(&tq, q, D, Sq, BH, fa::kBM, bf16)) != FA_OK) return st;
  if ((st = encode_3d(&tk, k, D, Skv, BH, fa::kN3, bf16)) != FA_OK) return st;
  if ((st = encode_3d(&tv, v, D, Skv, BH, fa::kN3, bf16)) != FA_OK) return st;
  if ((st = encode_3d(&to, o, D, Sq, BH, 32, bf16)) != FA_OK) return st;
  fa::PrefillParams p{};
  p.lse = lse;
  p.status = d.status;
  p.timeout_ns = g_watchdog_ns.load();
  p.BH = BH;
  p.Sq = Sq;
  p.Skv = Skv;
  p.n_qtiles = (Sq + fa::kRows3 - 1) / fa::kRows3;
  p.causal = causal ? 1 : 0;
  p.lpt = (flags & FA_FLAG_NO_LPT) ? 0 : 1;
  p.always_rescale = (flags & FA_FLAG_ALWAYS_RESCALE) ? 1 : 0;
  p.test_stall = (flags & FA_FLAG_TEST_STALL) ? 1 : 0;
  p.overlap_prev = (flags & FA_FLAG_OVERLAP_PREVIOUS) ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.rescale_tau = (flags & FA_FLAG_EXACT_MAX) ? 0.f : 8.f;
  p.n_splits = 1;
  p.tiles_per_split = (Skv + fa::kN3 - 1) / fa::kN3;
  const long long n_items = static_cast<long long>(p.n_qtiles) * BH;
  if (n_items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.n_items = static_cast<int>(n_items);
  p.sched = sched_slot(d, captured);
  const int grid = static_cast<int>(std::min<long long>(n_items, d.sm_count > 0 ? d.sm_count : 1));
  if (fa::launch_prefill_d64x3(bf16, tq, tk, tv, to, p, grid, stream) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

fa_status_t run_prefill(DeviceState& d, const void* q, const void* k, const void* v,
                        void* o, float* lse, int B, int H, int Sq, int Skv, int D,
                        float scale, int causal, bool bf16, unsigned flags,
                        int num_splits, void* ws, size_t ws_bytes, bool own_ws,
                        bool captured, cudaStream_t stream) {
  fa_status_t st = get_encoder();
  if (st != FA_OK) return st;
  {
    const int di = D == 128 ? 1 : 0, ti = bf16 ? 1 : 0;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!d.regs_checked[di][ti]) {
      // the register split inside the kernel assumes 128 registers/thread
      int regs = 0;
      if (fa::prefill_num_regs(D, bf16, &regs) != cudaSuccess) return FA_ERR_CUDA;
      d.regs_checked[di][ti] = true;
      d.regs_ok[di][ti] = regs == 128;
    }
    if (!d.regs_ok[di][ti]) return FA_ERR_UNSUPPORTED;
  }
  const int BH = B * H;
  if (D == 128 && num_splits <= 1 && !(flags & FA_FLAG_SINGLE_CTA) &&
      ((flags & (FA_FLAG_PAIR | FA_FLAG_PAIR64)) ||
       pair_by_default(BH, Sq, Skv, causal, d.sm_count)))
    return run_prefill_pair(d, q, k, v, o, lse, BH, Sq, Skv, scale, causal, bf16, flags,
                            captured, stream);
  CUtensorMap tq, tk, tv, to;
  if ((st = encode_3d(&tq, q, D, Sq, BH, fa::kBM, bf16)) != FA_OK) return st;
  if ((st = encode_3d(&tk, k, D, Skv, BH, fa::kBN, bf16)) != FA_OK) return st;
  if ((st = encode_3d(&tv, v, D, Skv, BH, fa::kBN, bf16)) != FA_OK) return st;
  if ((st = encode_3d(&to, o, D, Sq, BH, 32, bf16)) != FA_OK) return st;
  fa::PrefillParams p{};
  p.lse = lse;
  p.status = d.status;
  p.timeout_ns = g_watchdog_ns.load();
  p.BH = BH;
  p.Sq = Sq;
  p.Skv = Skv;
  p.n_qtiles = (Sq + fa::kRowsPerCta - 1) / fa::kRowsPerCta;
  p.causal = causal ? 1 : 0;
  p.lpt = (flags & FA_FLAG_NO_LPT) ? 0 : 1;
  p.always_rescale = (flags & FA_FLAG_ALWAYS_RESCALE) ? 1 : 0;
  p.test_stall = (flags & FA_FLAG_TEST_STALL) ? 1 : 0;
  p.overlap_prev = (flags & FA_FLAG_OVERLAP_PREVIOUS) ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.rescale_tau = (flags & FA_FLAG_EXACT_MAX) ? 0.f : 8.f;
  const int n_tiles = (Skv + fa::kBN - 1) / fa::kBN;
  int n_splits = prefill_splits(BH, Sq, Skv, d.sm_count, num_splits);
  if (D == 64 && (flags & FA_FLAG_D64_THREE_STAGE) && n_splits == 1 &&
      !(flags & FA_FLAG_CORRECTION_WG))
    return run_prefill_d64x3(d, q, k, v, o, lse, BH, Sq, Skv, scale, causal, bf16, flags,
                             captured, stream);
  if (n_splits > 1 && static_cast<long long>(BH) * Sq > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.tiles_per_split = (n_tiles + n_splits - 1) / n_splits;
  n_splits = (n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  size_t need = prefill_ws_bytes(BH, Sq, D, n_splits);
  if (need > 0 && !own_ws && num_splits == 0 &&
      (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))) {
    // the library's choice, without room for the partials: no split
    n_splits = 1;
    p.tiles_per_split = n_tiles;
    need = 0;
  }
  p.n_splits = n_splits;
  if (need > 0) {
    if (own_ws) {
      if ((st = stream_workspace(d, stream, need, &ws)) != FA_OK) return st;
    } else if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) {
      return FA_ERR_WORKSPACE;
    }
    const size_t rows = static_cast<size_t>(n_splits) * BH * Sq;
    p.part_o = static_cast<float*>(ws);
    p.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                          ((rows * D * sizeof(float) + 255) / 256) * 256);
  }
  const long long n_items = static_cast<long long>(p.n_qtiles) * BH * n_splits;
  if (n_items > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  p.n_items = static_cast<int>(n_items);
  p.sched = sched_slot(d, captured);
  // persistent: one CTA per SM (the kernel's shared memory allows no second)
  const int grid = static_cast<int>(std::min<long long>(n_items, d.sm_count > 0 ? d.sm_count : 1));
  if (fa::launch_prefill(D, bf16, (flags & FA_FLAG_CORRECTION_WG) != 0, tq, tk, tv, to, p,
                         grid, stream) != cudaSuccess)
    return FA_ERR_CUDA;
  if (n_splits > 1) {
    // merge the key ranges of every (head, query row): the decode combine
    // over BH * Sq rows
    fa::DecodeParams c{};
    c.o = o;
    c.lse = lse;
    c.part_o = p.part_o;
    c.part_lse = p.part_lse;
    c.BH = BH * Sq;
    c.n_splits = n_splits;
    if (fa::launch_decode_combine(D, bf16, c, stream) != cudaSuccess) return FA_ERR_CUDA;
  }
  return FA_OK;
}

// Key split for decode: enough CTAs for many waves over two CTAs per SM,
// at least 256 keys per split, a multiple of the 64-key tile.
int decode_keys_per_split(int BH, int Skv, int sm_count, int num_splits) {
  const int tile = fa::kDecKeysPerTile;
  if (num_splits >= 1) {
    int kps = (Skv + num_splits - 1) / num_splits;
    return ((kps + tile - 1) / tile) * tile;
  }
  const long long slots = 2LL * (sm_count > 0 ? sm_count : 148);
  long long kps = (static_cast<long long>(BH) * Skv + 16 * slots - 1) / (16 * slots);
  kps = ((kps + tile - 1) / tile) * tile;
  if (kps < 256) kps = 256;
  if (kps > 2048) kps = 2048;
  const long long skv_r = ((static_cast<long long>(Skv) + tile - 1) / tile) * tile;
  if (kps > skv_r) kps = skv_r;
  return static_cast<int>(kps);
}

size_t decode_ws_bytes(int BH, int n_splits, int D) {
  if (n_splits <= 1) return 0;
  const size_t po = static_cast<size_t>(n_splits) * BH * D * sizeof(float);
  const size_t pl = static_cast<size_t>(n_splits) * BH * sizeof(float);
  return ((po + 255) / 256) * 256 + ((pl + 255) / 256) * 256;
}

fa_status_t run_decode(DeviceState& d, const void* q, const void* k, const void* v,
                       void* o, float* lse, int BH, int Skv, int D, float scale,
                       bool bf16, int num_splits, void* ws, size_t ws_bytes,
                       bool own_ws, cudaStream_t stream) {
  const int kps = decode_keys_per_split(BH, Skv, d.sm_count, num_splits);
  const int n_splits = (Skv + kps - 1) / kps;
  const size_t need = decode_ws_bytes(BH, n_splits, D);
  if (need > 0) {
    if (own_ws) {
      const fa_status_t wst = stream_workspace(d, stream, need, &ws);
      if (wst != FA_OK) return wst;
    } else {
      if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return FA_ERR_WORKSPACE;
    }
  }
  fa::DecodeParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  if (need > 0) {
    const size_t po = static_cast<size_t>(n_splits) * BH * D * sizeof(float);
    p.part_o = static_cast<float*>(ws);
    p.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + ((po + 255) / 256) * 256);
  }
  p.status = d.status;
  p.timeout_ns = g_watchdog_ns.load();
  p.BH = BH;
  p.Skv = Skv;
  p.n_splits = n_splits;
  p.keys_per_split = kps;
  p.scale_log2 = scale * 1.4426950408889634f;
  const long long grid = static_cast<long long>(BH) * n_splits;
  if (grid > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  if (fa::launch_decode(D, bf16, p, static_cast<int>(grid), stream) != cudaSuccess)
    return FA_ERR_CUDA;
  if (n_splits > 1 && fa::launch_decode_combine(D, bf16, p, stream) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

fa_status_t forward(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int Sq, int Skv, int D, float scale, int causal,
                    int dtype, unsigned flags, int num_splits, void* ws,
                    size_t ws_bytes, bool own_ws, cudaStream_t stream) {
  fa_status_t st = validate(q, k, v, o, lse, B, H, Sq, Skv, D, scale, dtype);
  if (st != FA_OK) return st;
  if (num_splits < 0) return FA_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  if ((st = current_device(&d, nullptr)) != FA_OK) return st;
  // A call captured into a CUDA graph may be replayed on any stream, so it
  // takes a scheduler slot of its own and no library-owned workspace: the
  // shapes the library would split run unsplit (a caller's workspace, passed
  // to fa_fwd_ex, keeps the split).
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return FA_ERR_CUDA;
  const bool captured = cap != cudaStreamCaptureStatusNone;
  if (captured && own_ws) {
    own_ws = false;
    ws = nullptr;
    ws_bytes = 0;
    if (Sq == 1) num_splits = 1;
  }
  const bool bf16 = dtype == FA_BF16;
  // one query row per head: every key is visible (causal or not), and the
  // split-KV decode kernel serves it
  if (Sq == 1 && !(flags & FA_FLAG_TEST_STALL))
    return run_decode(*d, q, k, v, o, lse, B * H, Skv, D, scale, bf16, num_splits, ws,
                      ws_bytes, own_ws, stream);
  return run_prefill(*d, q, k, v, o, lse, B, H, Sq, Skv, D, scale, causal, bf16, flags,
                     num_splits, ws, ws_bytes, own_ws, captured, stream);
}

}  // namespace

namespace fa {

unsigned long long context_id() {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q{};
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!g_ctx_current || !g_ctx_get_id || g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx ||
      g_ctx_get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

fa_status_t check_device() {
  DeviceState* d = nullptr;
  return current_device(&d, nullptr);
}

fa_status_t check_call(const void* q, const void* k, const void* v, const void* o,
                       const void* lse, int B, int H, int Sq, int Skv, int D,
                       float scale, int dtype) {
  const fa_status_t st = validate(q, k, v, o, lse, B, H, Sq, Skv, D, scale, dtype);
  if (st != FA_OK) return st;
  DeviceState* d = nullptr;
  return current_device(&d, nullptr);
}

}  // namespace fa

extern "C" {

fa_status_t fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int Sq, int Skv, int D, float scale, int causal,
                   int dtype, fa_stream_t stream) {
  return forward(q, k, v, o, lse, B, H, Sq, Skv, D, scale, causal, dtype, 0u, 0,
                 nullptr, 0, true, reinterpret_cast<cudaStream_t>(stream));
}

size_t fa_workspace_bytes(int B, int H, int Sq, int Skv, int D, int num_splits) {
  if (B < 1 || H < 1 || Sq < 1 || Skv < 1 || (D != 64 && D != 128) || num_splits < 0)
    return 0;
  int sms = 0;
  if (num_splits == 0) {
    DeviceState* d = nullptr;
    if (current_device(&d, nullptr) == FA_OK) sms = d->sm_count;
  }
  if (Sq > 1) {
    const int n_tiles = (Skv + fa::kBN - 1) / fa::kBN;
    const int s = prefill_splits(B * H, Sq, Skv, sms, num_splits);
    const int tps = (n_tiles + s - 1) / s;
    return prefill_ws_bytes(B * H, Sq, D, (n_tiles + tps - 1) / tps);
  }
  const int kps = decode_keys_per_split(B * H, Skv, sms, num_splits);
  return decode_ws_bytes(B * H, (Skv + kps - 1) / kps, D);
}

fa_status_t fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int Sq, int Skv, int D, float scale, int causal,
                      int dtype, unsigned flags, int num_splits, void* workspace,
                      size_t workspace_bytes, fa_stream_t stream) {
  return forward(q, k, v, o, lse, B, H, Sq, Skv, D, scale, causal, dtype, flags,
                 num_splits, workspace, workspace_bytes, false,
                 reinterpret_cast<cudaStream_t>(stream));
}

size_t fa_host_staging_bytes(int B, int H, int Sq, int Skv, int D) {
  if (B < 1 || H < 1 || Sq < 1 || Skv < 1 || (D != 64 && D != 128)) return 0;
  auto up = [](size_t x) { return ((x + 255) / 256) * 256; };
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t qb = up(BH * Sq * D * 2), kb = up(BH * Skv * D * 2);
  const size_t lb = up(BH * Sq * sizeof(float));
  return qb + 2 * kb + qb + lb + fa_workspace_bytes(B, H, Sq, Skv, D, 0);
}

fa_status_t fa_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                        float* lse_h, int B, int H, int Sq, int Skv, int D, float scale,
                        int causal, int dtype, void* staging, size_t staging_bytes,
                        fa_stream_t stream) {
  fa_status_t st = validate(q_h, k_h, v_h, o_h, lse_h, B, H, Sq, Skv, D, scale, dtype);
  if (st != FA_OK) return st;
  const size_t need = fa_host_staging_bytes(B, H, Sq, Skv, D);
  if (!staging || staging_bytes < need || (reinterpret_cast<uintptr_t>(staging) & 255u))
    return FA_ERR_WORKSPACE;
  auto up = [](size_t x) { return ((x + 255) / 256) * 256; };
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t qn = BH * Sq * D * 2, kn = BH * Skv * D * 2, ln = BH * Sq * sizeof(float);
  char* base = static_cast<char*>(staging);
  char* dq = base;
  char* dk = dq + up(qn);
  char* dv = dk + up(kn);
  char* dO = dv + up(kn);
  char* dl = dO + up(qn);
  char* dws = dl + up(ln);
  const size_t ws_bytes = need - static_cast<size_t>(dws - base);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(dq, q_h, qn, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(dk, k_h, kn, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(dv, v_h, kn, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return FA_ERR_CUDA;
  st = forward(dq, dk, dv, dO, reinterpret_cast<float*>(dl), B, H, Sq, Skv, D, scale,
               causal, dtype, 0u, 0, ws_bytes ? dws : nullptr, ws_bytes, false, s);
  if (st != FA_OK) return st;
  if (cudaMemcpyAsync(o_h, dO, qn, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(lse_h, dl, ln, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

fa_status_t fa_get_device_status(fa_stream_t stream) {
  DeviceState* d = nullptr;
  fa_status_t st = current_device(&d, nullptr);
  if (st != FA_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, d->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return FA_ERR_CUDA;
  return word == 0 ? FA_OK : static_cast<fa_status_t>(word);
}

fa_status_t fa_release_workspaces(void) {
  DeviceState* d = nullptr;
  const fa_status_t st = current_device(&d, nullptr);
  if (st != FA_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  fa_status_t out = FA_OK;
  for (auto& w : d->workspaces) {
    if (cudaFree(w.ptr) != cudaSuccess) out = FA_ERR_CUDA;
    if (w.tail_ctr && cudaFree(w.tail_ctr) != cudaSuccess) out = FA_ERR_CUDA;
  }
  d->workspaces.clear();
  return out;
}

void fa_set_watchdog_ns(unsigned long long ns) {
  g_watchdog_ns.store(ns ? ns : kDefaultWatchdogNs);
}

const char* fa_status_string(fa_status_t status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dim, dtype or device";
    case FA_ERR_CUDA: return "CUDA runtime error";
    case FA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case FA_ERR_TIMEOUT: return "kernel wait timed out";
  }
  return "unknown status";
}

int fa_prefill_uses_pairs(int B, int H, int Sq, int Skv, int D, int causal, unsigned flags,
                          int num_splits) {
  if (B <= 0 || H <= 0 || Sq <= 1 || Skv <= 0 || D != 128 || num_splits > 1 ||
      (flags & FA_FLAG_SINGLE_CTA))
    return 0;
  if (flags & (FA_FLAG_PAIR | FA_FLAG_PAIR64)) return 1;
  int sms = 0;
  DeviceState* d = nullptr;
  if (current_device(&d, nullptr) == FA_OK) sms = d->sm_count;
  return pair_by_default(B * H, Sq, Skv, causal, sms) ? 1 : 0;
}

int fa_prefill_tail_items(int B, int H, int Sq, int Skv, int D, int causal, int dtype,
                          unsigned flags) {
  if (fa_prefill_uses_pairs(B, H, Sq, Skv, D, causal, flags, 0) != 1) return 0;
  if ((flags & (FA_FLAG_PAIR64 | FA_FLAG_CORRECTION_WG)) || !(flags & FA_FLAG_TAIL_SPLIT) ||
      (dtype != FA_F16 && dtype != FA_BF16))
    return 0;
  DeviceState* d = nullptr;
  int slots = 0;
  if (current_device(&d, nullptr) != FA_OK ||
      pair_slots(*d, dtype == FA_BF16, false, &slots) != FA_OK || slots <= 0)
    return 0;
  const long long n_items = static_cast<long long>(B) * H * ((Sq + 511) / 512);
  return pair_tail_items(n_items, std::min<long long>(n_items, slots), causal, Skv);
}

int fa_version(void) { return 10300; }

}  // extern "C"
