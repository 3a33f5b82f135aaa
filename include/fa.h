/*
 * fa.h -- C ABI of the GB300 (sm_103a) fused attention forward library,
 * libfa_gb300.so.
 *
 * Operation (every entry point below computes it):
 *   for each batch b, head h and query row i
 *     O[b,h,i,:]  = sum_j softmax_j(scale * <Q[b,h,i,:], K[b,h,j,:]>) V[b,h,j,:]
 *     LSE[b,h,i]  = ln sum_j exp(scale * <Q[b,h,i,:], K[b,h,j,:]>)
 *   over the visible keys j: all of them, or, when causal, j <= i + (Skv - Sq)
 *   (bottom-right alignment; equal to j <= i when Sq == Skv).  A row with no
 *   visible key gets O = 0 and LSE = -inf.
 *   This is the fused forward pass that "The FA5090 Optimization Journey"
 *   (sections 2.2-2.8) and the B300 G5 page ("Flash Attention CUDA Kernel
 *   optimisation: from 56 to 986 TFLOPS on B300", V21-V36) build: scores and
 *   probabilities stay on chip, an online softmax carries the running row max
 *   and row sum across key tiles.  LSE is the natural-log log-sum-exp of the
 *   scaled scores; the pages do not define it, this library does.
 *
 * Layout and ownership (all device pointers are caller-owned CUDA memory on
 * the current device; the library never frees or keeps them):
 *   q   [B, H, Sq,  D]  contiguous, fp16 or bf16
 *   k   [B, H, Skv, D]  contiguous, same type
 *   v   [B, H, Skv, D]  contiguous, same type
 *   o   [B, H, Sq,  D]  contiguous, same type (written)
 *   lse [B, H, Sq]      contiguous, fp32 (written)
 *   Every pointer must be 16-byte aligned.
 *
 * Supported: D in {64, 128}; dtype FA_F16 or FA_BF16; B*H < 65536;
 * 1 <= Sq, Skv <= 2^24; scale finite and > 0.  A device that is not
 * compute capability 10.3 (sm_103a) is rejected with FA_ERR_UNSUPPORTED.
 *
 * Errors: argument checks are synchronous and happen before anything is
 * launched or allocated; a failed check returns its status and leaves every
 * output untouched.  Launches are asynchronous on `stream`; a launch failure
 * returns FA_ERR_CUDA.  Kernel-side waits are bounded: a wait that exceeds the
 * watchdog limit (default 1 s) makes the kernel stop, release what it holds
 * and record FA_ERR_TIMEOUT in a device status word, which
 * fa_get_device_status() reports.  No entry point prints, throws or aborts.
 *
 * CUDA graphs: fa_fwd, fa_fwd_ex and fa_fwd_host may be called while
 * `stream` is being captured; the graph then replays the same launches, on
 * any stream.  A captured call uses no library-owned workspace, so the
 * shapes fa_fwd would split (few query tiles, or decode) run unsplit there,
 * and FA_FLAG_TAIL_SPLIT is ignored;
 * fa_fwd_ex with a caller workspace keeps the key split, and the workspace is
 * then the graph's to keep.  Each captured prefill takes one of 4096
 * scheduler slots reserved for captures, which direct launches never use:
 * replays of one graph run in stream order, and replays of graphs captured
 * more than 4096 prefill calls apart must not overlap.
 * fa_get_device_status synchronises and cannot be captured;
 * fa_fwd_decode_static's scratch makes overlapping replays race.
 * FA_FLAG_OVERLAP_PREVIOUS has been tested on streams, not inside captures.
 *
 * Device reset: the library keeps, per device, the addresses of its static
 * device arrays and its workspaces.  After cudaDeviceReset (a new primary
 * context) the next call looks the addresses up again and forgets the
 * workspaces, which went away with the old context.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *fa_stream_t;

typedef enum { FA_F16 = 0, FA_BF16 = 1 } fa_dtype_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or scale   */
  FA_ERR_UNSUPPORTED = 2, /* D, dtype or device not supported              */
  FA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed          */
  FA_ERR_WORKSPACE = 4,   /* workspace missing, too small or misaligned    */
  FA_ERR_TIMEOUT = 5      /* a kernel wait ran past the watchdog limit     */
} fa_status_t;

/* fa_fwd_ex flags */
#define FA_FLAG_NO_LPT 0x1u          /* causal: items in plain order instead
                                        of heaviest-first (results are
                                        bitwise identical either way)      */
#define FA_FLAG_ALWAYS_RESCALE 0x2u  /* rescale O on every key tile, not only
                                        when the row max changes (bitwise
                                        identical either way)              */
#define FA_FLAG_EXACT_MAX 0x4u       /* prefill: carry the exact running row
                                        max (rescale O whenever it grows)
                                        instead of raising the reference max
                                        only when a tile's max exceeds it by
                                        more than 8 in log2 units; both are
                                        exact after the final division by
                                        the row sum                         */
#define FA_FLAG_PAIR 0x8u            /* prefill, D = 128, without a key
                                        split: run on CTA pairs (two-CTA
                                        clusters whose tensor cores compute
                                        256-row MMAs together, each CTA
                                        loading half of every K/V tile);
                                        ignored otherwise.  Without this flag
                                        or FA_FLAG_SINGLE_CTA the library
                                        uses pairs for long rows (non-causal
                                        Sq, Skv >= 1024; causal Sq >= 8192)
                                        with at least one 512-row item per
                                        two SMs                             */
#define FA_FLAG_SINGLE_CTA 0x10u     /* prefill: never use CTA pairs        */
#define FA_FLAG_CORRECTION_WG 0x20u  /* prefill over the whole key range: a
                                        dedicated correction warpgroup
                                        rescales O in tensor memory when a
                                        row's max moves (the softmax warps
                                        hand it those tiles) instead of the
                                        softmax warps doing it themselves;
                                        same results, bitwise (measured 5-17 %
                                        slower on GB300; kept for
                                        comparison).  Ignored with split
                                        keys                                */
#define FA_FLAG_PAIR64 0x40u         /* prefill, D = 128, without a key
                                        split: CTA pairs with score tiles of
                                        64 keys and two score buffers per
                                        stage, so that the next tile's
                                        scores are computed while the
                                        softmax of this one runs (measured
                                        slower than the default 128-key
                                        pairs on GB300; kept for
                                        comparison); ignored where
                                        FA_FLAG_PAIR would be               */
#define FA_FLAG_OVERLAP_PREVIOUS 0x80u /* prefill: launch so that the kernel
                                        may start while the previous grid on
                                        `stream` is still running (CUDA
                                        programmatic dependent launch): it
                                        reads q, k, v at once but waits for
                                        that grid before its first write of
                                        o, lse or the workspace.  The caller
                                        guarantees that the work before it
                                        on the stream does not write q, k or
                                        v (e.g. back-to-back calls on
                                        resident inputs).  The library's own
                                        prefill kernels let the next grid
                                        start as soon as their SMs run out
                                        of work items.  Ignored by decode
                                        and FA_FLAG_PAIR64                  */
#define FA_FLAG_TEST_STALL 0x100u    /* test hook: the K/V producer of every
                                        CTA withholds its first item's second
                                        K tile, so the consumers' bounded
                                        waits run out and the kernel reports
                                        FA_ERR_TIMEOUT                      */
#define FA_FLAG_D64_THREE_STAGE 0x400u /* prefill, D = 64, without a key
                                        split and without
                                        FA_FLAG_CORRECTION_WG: the
                                        three-stage kernel (384-row items of
                                        three 128-row stages, 96-key tiles);
                                        ignored otherwise                   */
#define FA_FLAG_TAIL_SPLIT 0x200u    /* CTA pairs, non-causal, without
                                        FA_FLAG_CORRECTION_WG: the tail
                                        split (see fa_fwd).  Measured slower
                                        than without it on GB300 (0.94 on
                                        the B4 H16 S4096 workload); kept
                                        for comparison                      */

/*
 * fa_fwd -- the whole forward pass for one batch, on `stream`.
 * Prefill (Sq > 1): one fused, persistent kernel (one CTA per SM, or one
 * two-CTA cluster per pair of SMs for long rows at D = 128: see
 * FA_FLAG_PAIR); its CTAs claim work items from a counter in a small static
 * device array of the
 * library (1024 slots of 16 bytes, one per launch in turn, cleared by each
 * launch's last CTA), so two prefill launches whose GPU work overlaps must
 * be fewer than 1024 calls apart.  When the (256-row query tile, head)
 * items are fewer than the SMs (short query blocks, few heads), the keys of
 * each item are split into ranges whose fp32 partials a combine kernel
 * merges.  Decode (Sq == 1): split-KV kernel plus combine kernel.
 * Tail split (FA_FLAG_TAIL_SPLIT, fa_fwd_ex only): when the CTA-pair
 * kernel's 512-row items (non-causal, at least 4 key tiles) leave its last
 * round of pairs partly idle, and the quarters of those last items fit in
 * at most three quarter-rounds, each of the last items runs as four items
 * over a quarter of the key tiles; the quarter that finishes last merges
 * their fp32 partials inside the kernel (the key-split merge: weights
 * exp(LSE_r - LSE)), so the rows of those items differ from an unsplit run
 * by rounding only.  Outside a CUDA graph capture, the partials (1 MiB per
 * split item) and arrival counters go to the library's workspace for the
 * stream, as fa_fwd's key splits do.  The
 * partials go to a workspace that the library allocates on the first call
 * that needs one, one per (device, stream handle), and keeps until
 * fa_release_workspaces() or process exit (use fa_fwd_ex to supply your
 * own).  A call that needs a larger workspace than its stream's frees the
 * old one first (cudaFree, which synchronises the device) and allocates
 * the new one.  The cache is keyed on the stream handle: a stream created
 * after another was destroyed may receive the same handle, and would then
 * share that stream's workspace, so call fa_release_workspaces() after
 * destroying streams that fa_fwd used.
 * Returns FA_OK once the work is enqueued.
 */
fa_status_t fa_fwd(const void *q, const void *k, const void *v, void *o,
                   float *lse, int B, int H, int Sq, int Skv, int D,
                   float scale, int causal, int dtype, fa_stream_t stream);

/*
 * fa_workspace_bytes -- bytes of device workspace fa_fwd_ex needs for this
 * shape with `num_splits` key splits (0 = the library's choice); 0 when the
 * shape needs none.  The split-KV partials are fp32 (O, LSE) per split and
 * row: the fp32 workspace round trip that "The FA5090 Optimization Journey"
 * section 2.7 measured (and rejected for prefill at its sizes).  Here the
 * library splits only decode, where one query row per head leaves too few
 * work items to fill the GPU, and prefill whose items are fewer than the
 * SMs.
 */
size_t fa_workspace_bytes(int B, int H, int Sq, int Skv, int D,
                          int num_splits);

/*
 * fa_fwd_ex -- fa_fwd with explicit options.
 *   flags       FA_FLAG_* bits above (0 for the default path)
 *   num_splits  key splits; 0 = the library's choice, 1 = no split.  With
 *               0, a prefill whose workspace is NULL or smaller than
 *               fa_workspace_bytes(..., 0) runs without a split; decode
 *               and an explicit split count need the workspace.
 *   workspace   caller-owned device memory, 256-byte aligned, at least
 *               fa_workspace_bytes(...) bytes; may be NULL when that is 0.
 *               It must not be used by anything else until the work on
 *               `stream` has finished.
 * Allocates nothing.
 */
fa_status_t fa_fwd_ex(const void *q, const void *k, const void *v, void *o,
                      float *lse, int B, int H, int Sq, int Skv, int D,
                      float scale, int causal, int dtype, unsigned flags,
                      int num_splits, void *workspace, size_t workspace_bytes,
                      fa_stream_t stream);

/*
 * fa_host_staging_bytes / fa_fwd_host -- the same operation on HOST buffers.
 * q_h, k_h, v_h, o_h, lse_h are host pointers (pinned memory gives full copy
 * bandwidth; pageable memory works but is slower).  `staging` is caller-owned
 * device memory of at least fa_host_staging_bytes(...) bytes, 256-byte
 * aligned: the library copies Q, K, V into it, runs the forward pass there
 * and copies O and LSE back, all on `stream`.  The call returns once the
 * work is enqueued; the host outputs are valid after the stream synchronises.
 * Allocates nothing.
 */
size_t fa_host_staging_bytes(int B, int H, int Sq, int Skv, int D);
fa_status_t fa_fwd_host(const void *q_h, const void *k_h, const void *v_h,
                        void *o_h, float *lse_h, int B, int H, int Sq,
                        int Skv, int D, float scale, int causal, int dtype,
                        void *staging, size_t staging_bytes,
                        fa_stream_t stream);

/*
 * fa_fwd_decode_static -- the decode pass (one query row per head, Sq = 1)
 * for callers that cannot allocate device memory: host frameworks that own
 * every device allocation and forbid side allocations, serving loops that
 * must not meet cudaMalloc's implicit device synchronisation or its run-time
 * failure, processes with a memory budget fixed up front.  The pages have no
 * counterpart; this is a deployment entry point of this library.
 *   q [B,H,1,D], k and v [B,H,Skv,D], o [B,H,1,D], lse [B,H,1]: caller-owned
 *   device memory as for fa_fwd.  Every key is visible (for one query row the
 *   causal and full masks agree).
 * The split-KV partials go to a static device array of
 * FA_DECODE_STATIC_SCRATCH_BYTES that is part of the library's module: every
 * GPU that loads the library holds it until the process exits.  The partials
 * need n_splits * B * H * (D + 1) * 4 bytes (about, rounded up; n_splits is
 * the library's choice, fa_workspace_bytes(B, H, 1, Skv, D, 0) gives the
 * exact figure); a shape that needs more returns FA_ERR_WORKSPACE before
 * anything is launched.  Nothing in the array has to start at zero.
 * The arguments and the device are checked first, exactly as by fa_fwd
 * (an unsupported device returns FA_ERR_UNSUPPORTED), then the scratch's
 * capacity.  The first call on a device looks up the array's device address
 * (once per device, with that device current, and again after the device's
 * context was reset); make that first call before any stream capture.  Calls share the one array: two calls whose work overlaps on the
 * GPU (different streams, or different host threads) race and corrupt each
 * other's results.  Allocates nothing.
 */
#define FA_DECODE_STATIC_SCRATCH_BYTES (8u << 20)
fa_status_t fa_fwd_decode_static(const void *q, const void *k, const void *v,
                                 void *o, float *lse, int B, int H, int Skv,
                                 int D, float scale, int dtype,
                                 fa_stream_t stream);

/*
 * fa_release_workspaces -- frees the workspaces that fa_fwd keeps for split
 * partials on the current device (one per stream handle it was called
 * with), after synchronising the device.  The next fa_fwd that needs one
 * allocates it again.  Returns FA_ERR_CUDA if the synchronisation or a free
 * failed (the cache is emptied either way).
 */
fa_status_t fa_release_workspaces(void);

/*
 * fa_get_device_status -- synchronises `stream`, then returns and clears the
 * device status word of the current device: FA_OK, or FA_ERR_TIMEOUT if a
 * kernel's bounded wait ran out since the last call.  FA_ERR_CUDA if the
 * synchronisation itself failed.
 */
fa_status_t fa_get_device_status(fa_stream_t stream);

/*
 * fa_ex2_approx -- y[i] = 2^x[i] for i < n, computed on the device by the
 * instruction the softmax of every kernel uses for its exponentials
 * (ex2.approx.ftz.f32: subnormal results flush to +0).  A self-check of the
 * values the kernels rely on: masked scores are -inf and must give +0, the
 * row maximum gives 2^0 = 1 ("The FA5090 Optimization Journey", section 2.6,
 * asserts both on the device).  x and y are device pointers to n fp32
 * values, 4-byte aligned, 1 <= n <= 2^28; asynchronous on `stream`.
 */
fa_status_t fa_ex2_approx(const float *x, float *y, int n, fa_stream_t stream);

/* Watchdog limit for every kernel-side wait, in nanoseconds (default 1e9).
 * Applies to launches made after the call.  0 restores the default. */
void fa_set_watchdog_ns(unsigned long long ns);

/* Static description of a status code (never NULL). */
const char *fa_status_string(fa_status_t status);

/* 1 if fa_fwd / fa_fwd_ex with these arguments runs prefill on CTA pairs
 * (see FA_FLAG_PAIR), else 0 (single-CTA kernel, decode, or arguments fa_fwd
 * would reject).  Reads the current device's SM count; launches nothing. */
int fa_prefill_uses_pairs(int B, int H, int Sq, int Skv, int D, int causal,
                          unsigned flags, int num_splits);

/* Number of 512-row CTA-pair items that fa_fwd_ex with these arguments
 * (outside a capture) splits into key quarters (FA_FLAG_TAIL_SPLIT: see
 * fa_fwd); 0 when there is none.  Reads the current device's SM count
 * and the pair kernel's occupancy; launches nothing. */
int fa_prefill_tail_items(int B, int H, int Sq, int Skv, int D, int causal,
                          int dtype, unsigned flags);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
