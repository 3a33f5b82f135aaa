// fa_internal.h -- parameter blocks and constants shared by the host code and
// the kernels of libfa_gb300.so (not part of the public ABI).
#pragma once
#include <cstdint>

namespace fa {

// Status values written to the device status word (same numbers as
// fa_status_t in include/fa.h).
constexpr unsigned kStatusOk = 0;
constexpr unsigned kStatusTimeout = 5;

// Prefill tiling: a work item is kStages query tiles of kBM rows (two
// ping-pong stages) of one head, walked over the keys in tiles of kBN; a
// persistent CTA per SM takes items in turn.
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kStages = 2;
constexpr int kRowsPerCta = kBM * kStages;
constexpr int kThreads = 512;  // 4 warpgroups
// The three-stage D = 64 kernel: three stages of kBM rows per item, key
// tiles of kN3.
constexpr int kN3 = 96;
constexpr int kStages3 = 3;
constexpr int kRows3 = kStages3 * kBM;

// Dynamic item scheduler: slots of a static device array, one per launch
// (chosen round-robin by the host), two words each: [0] = items claimed,
// [1] = CTAs finished.  Both are zero when a launch starts: the launch's
// last CTA clears them.  kSchedSlots slots rotate among direct launches;
// kGraphSchedSlots more go, one each, to launches captured into CUDA graphs,
// which keep their slot for every replay.
constexpr int kSchedSlots = 1024;
constexpr int kGraphSchedSlots = 4096;

struct PrefillParams {
  float* lse;                 // [B*H, Sq]
  unsigned long long* sched;  // this launch's scheduler slot
  unsigned* status;           // device status word
  unsigned long long timeout_ns;
  int BH;                     // B*H
  int Sq, Skv;
  int n_qtiles;               // ceil(Sq / kRowsPerCta)
  int n_items;                // n_qtiles * BH * n_splits work items
  int causal;
  int lpt;                    // heaviest-first item order (causal only)
  int always_rescale;
  int test_stall;
  float scale_log2;           // scale * log2(e)
  float rescale_tau;          // raise the reference max only past this (log2)
  // split keys (kept after the fields above: the kernel with the whole key
  // range measured about 1% slower with these inserted among them)
  int n_splits;               // key ranges per (query tile, head); 1: no split
  int tiles_per_split;        // key tiles of kBN per range
  float* part_o;              // n_splits > 1: [n_splits, BH*Sq, D] fp32, O / l
  float* part_lse;            // n_splits > 1: [n_splits, BH*Sq] fp32
  // launched to overlap the previous grid on the stream: every thread waits
  // for it before its first global write (reads of Q, K, V may start early)
  int overlap_prev;
  // CTA-pair kernel, last items split by keys (non-causal): the last
  // tail_items of the n_items - 3 * tail_items pair items run as four items
  // each, one per quarter of the key tiles, numbered after the others.  A
  // quarter writes its rows' fp32 O / l and LSE to part_o / part_lse; the
  // last of the four to finish a warp's 32 rows merges them into o and lse.
  // 0: no split.
  int tail_items;
  void* o;                          // [BH, Sq, D] 16-bit (the merged rows)
  unsigned long long* tail_count;   // per (item, stage, rank, warp): epoch << 8 | arrivals
  unsigned tail_epoch;              // this launch's epoch (never 0)
};

// Decode (Sq == 1) split-KV.
constexpr int kDecThreads = 256;     // 8 consumer warps
constexpr int kDecKeysPerTile = 64;  // keys per smem stage
constexpr int kDecStages = 3;        // smem ring depth (two CTAs per SM)

struct DecodeParams {
  const void* q;              // [BH, D]
  const void* k;              // [BH, Skv, D]
  const void* v;              // [BH, Skv, D]
  void* o;                    // [BH, D] (when n_splits == 1)
  float* lse;                 // [BH]    (when n_splits == 1)
  float* part_o;              // [n_splits, BH, D] fp32 (when n_splits > 1)
  float* part_lse;            // [n_splits, BH]
  unsigned* status;
  unsigned long long timeout_ns;
  int BH, Skv;
  int n_splits;
  int keys_per_split;         // multiple of kDecKeysPerTile
  float scale_log2;
};

}  // namespace fa
