// sm103_ptx.cuh -- thin inline-PTX wrappers for the sm_103a features the
// attention kernels use: mbarriers, TMA (tensor and 1-D bulk copies), and the
// 5th-generation tensor core (tcgen05: TMEM allocation, MMA, commit, TMEM
// loads/stores, fences).  Each wrapper is one documented PTX instruction.
#pragma once
#include <cstdint>

namespace fa {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// One lane of the (fully active) warp returns true.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .b32 rx;\n\t.reg .pred px;\n\t"
      "elect.sync rx|px, %1;\n\t"
      "selp.b32 %0, 1, 0, px;\n\t}"
      : "=r"(pred)
      : "r"(0xffffffffu));
  return pred != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar,
                                                      uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// Non-blocking probe: true once the phase with the given parity completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, without suspending the thread (for loops that poll
// several barriers).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------------------ launches

// Programmatic dependent launch: this CTA has no more work to claim, so the
// next grid on the stream (launched with programmatic stream serialization)
// may start once every CTA of this grid has signalled or exited.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Blocks until the grids this one depends on (programmatically) have
// completed and their memory operations are visible; returns at once when
// there is none.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------ proxies

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const void* desc) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(desc))
               : "memory");
}

// 3-D tiled load global -> shared, completion signalled on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* desc,
                                            uint32_t bar, int32_t x, int32_t y,
                                            int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Prefetch a 3-D tile into L2 (no shared memory, no completion signal).
__device__ __forceinline__ void tma_prefetch_l2_3d(const void* desc, int32_t x,
                                                   int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.3d.L2.global [%0, {%1, %2, %3}];" ::"l"(
          reinterpret_cast<uint64_t>(desc)),
      "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 3-D tiled store shared -> global (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const void* desc, uint32_t src,
                                             int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, "
      "%4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(desc)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk store of this thread has read its source.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src,
                                             uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], "
      "[%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// ------------------------------------------------------------ tcgen05

// Allocate `ncols` TMEM columns (power of two >= 32); the TMEM address is
// written to shared memory at `dst`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
          dst),
      "r"(ncols)
      : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile(
      "tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
      "r"(ncols)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The MMA and commit wrappers below are executed by a whole, converged warp:
// elect.sync inside the asm picks the one lane that issues, so the operand
// descriptors, computed identically by every lane, stay warp-uniform.  A
// single divergent lane issuing tcgen05.mma measured ~100 cycles per
// instruction on GB300; the converged form issues faster than the tensor
// core consumes (64 cycles per 128x128x16).

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (fp16/bf16 in, fp32
// accumulate).
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t a_desc,
                                            uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16: A is read from tensor
// memory (row m in lane m, two 16-bit K elements per 32-bit column).
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem,
                                            uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Eight K=16 steps of D (+)= A * B with both operands K-major, 128-byte
// swizzled, in shared memory: the K = 128 contraction of a 64-column-box
// pair.  Step k reads 32 bytes further into each 128-byte row (descriptor
// start + 2 in 16-byte units) for k = 0..3, then the second 64-column box
// (+16384 bytes = +1024 units).  One elect.sync for the whole group; the
// first step overwrites D unless `accumulate`.
__device__ __forceinline__ void umma_f16_ss_k128(uint32_t d_tmem, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t"
      ".reg .b64 a1, a2, a3, a4, a5, a6, a7, b1, b2, b3, b4, b5, b6, b7;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "add.s64 a1, %1, 2;\n\t add.s64 b1, %2, 2;\n\t"
      "add.s64 a2, %1, 4;\n\t add.s64 b2, %2, 4;\n\t"
      "add.s64 a3, %1, 6;\n\t add.s64 b3, %2, 6;\n\t"
      "add.s64 a4, %1, 1024;\n\t add.s64 b4, %2, 1024;\n\t"
      "add.s64 a5, %1, 1026;\n\t add.s64 b5, %2, 1026;\n\t"
      "add.s64 a6, %1, 1028;\n\t add.s64 b6, %2, 1028;\n\t"
      "add.s64 a7, %1, 1030;\n\t add.s64 b7, %2, 1030;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a4, b4, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a5, b5, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a6, b6, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a7, b7, %3, t;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four K=16 steps of D (+)= A * B for a K = 64 contraction (one 64-column
// box): K-major, 128-byte swizzled operands in shared memory.
__device__ __forceinline__ void umma_f16_ss_k64(uint32_t d_tmem, uint64_t a_desc,
                                                uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t"
      ".reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "add.s64 a1, %1, 2;\n\t add.s64 b1, %2, 2;\n\t"
      "add.s64 a2, %1, 4;\n\t add.s64 b2, %2, 4;\n\t"
      "add.s64 a3, %1, 6;\n\t add.s64 b3, %2, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, t;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Eight K=16 steps of D (+)= A * B with A (128 rows x 128 K of 16-bit pairs)
// in tensor memory, 8 columns per step, and B MN-major 128-byte swizzled in
// shared memory, 16 K rows (2048 bytes = 128 descriptor units) per step.
__device__ __forceinline__ void umma_f16_ts_k128(uint32_t d_tmem, uint32_t a_tmem,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t"
      ".reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
      ".reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "add.s32 a1, %1, 8;\n\t  add.s64 b1, %2, 128;\n\t"
      "add.s32 a2, %1, 16;\n\t add.s64 b2, %2, 256;\n\t"
      "add.s32 a3, %1, 24;\n\t add.s64 b3, %2, 384;\n\t"
      "add.s32 a4, %1, 32;\n\t add.s64 b4, %2, 512;\n\t"
      "add.s32 a5, %1, 40;\n\t add.s64 b5, %2, 640;\n\t"
      "add.s32 a6, %1, 48;\n\t add.s64 b6, %2, 768;\n\t"
      "add.s32 a7, %1, 56;\n\t add.s64 b7, %2, 896;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, t;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Six K=16 steps of D (+)= A * B for a K = 96 contraction: A (128 rows x 96
// K of 16-bit pairs) in tensor memory, 8 columns per step; B MN-major
// 128-byte swizzled in shared memory, 16 K rows (2048 bytes = 128
// descriptor units) per step.
__device__ __forceinline__ void umma_f16_ts_k96(uint32_t d_tmem, uint32_t a_tmem,
                                                uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t"
      ".reg .b32 a1, a2, a3, a4, a5;\n\t"
      ".reg .b64 b1, b2, b3, b4, b5;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "add.s32 a1, %1, 8;\n\t  add.s64 b1, %2, 128;\n\t"
      "add.s32 a2, %1, 16;\n\t add.s64 b2, %2, 256;\n\t"
      "add.s32 a3, %1, 24;\n\t add.s64 b3, %2, 384;\n\t"
      "add.s32 a4, %1, 32;\n\t add.s64 b4, %2, 512;\n\t"
      "add.s32 a5, %1, 40;\n\t add.s64 b5, %2, 640;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, t;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by the elected
// lane has completed (the same lane elect.sync picks for the MMAs).
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];\n\t}" ::"r"(bar)
      : "memory");
}

// ------------------------------------------------------------ CTA pairs
// (a cluster of two CTAs whose tensor cores act as one: tcgen05 with
// .cta_group::2, M = 256 with 128 rows in each CTA)

// Rank of this CTA in its cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of the variable at shared address `a` of this
// CTA, in the CTA of cluster rank `rank` (the same offset there).
__device__ __forceinline__ uint32_t mapa_shared(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

// Arrive on an mbarrier of any CTA of the cluster (release, cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cl_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr)
               : "memory");
}

// Arrive on an mbarrier of any CTA of the cluster with relaxed semantics: no
// release fence (a release arrive at cluster scope measured ~1500 cycles).
// For arrivals that publish only tensor-memory accesses the arriving thread
// has already waited for (tcgen05.wait::st / wait::ld, then
// tcgen05.fence::before_thread_sync); the waiter follows its wait with
// tcgen05.fence::after_thread_sync.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cl_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cl_addr)
               : "memory");
}

// As mbar_try_wait, with acquire at cluster scope (for phases completed by
// another CTA's release-arrive).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait_cluster, without suspending the thread.
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// 32-bit store to the shared memory of another CTA of the cluster.
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cl_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cl_addr), "r"(v) : "memory");
}

// Every thread of both CTAs (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// 3-D tiled load into this CTA's shared memory whose completion is signalled
// on `bar_cl`, an mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* desc,
                                                 uint32_t bar_cl, int32_t x, int32_t y,
                                                 int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::"
      "complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar_cl), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// TMEM allocation for a CTA pair: one warp of each CTA executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
      "r"(ncols)
      : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}

// Eight K=16 steps of a pair MMA, D (+)= A * B, both operands K-major and
// 128-byte swizzled in shared memory (the same offsets in both CTAs; A: this
// CTA's 128 rows, B: this CTA's half of N).  The second 64-column box of A
// starts `a_box` descriptor units (16 bytes) after the first, B's `b_box`.
// Issued by the leader CTA's warp (elect.sync inside).
template <int kABox, int kBBox>
__device__ __forceinline__ void umma_pair_ss_k128(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t"
      ".reg .b64 a1, a2, a3, a4, a5, a6, a7, b1, b2, b3, b4, b5, b6, b7;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "add.s64 a1, %1, 2;\n\t add.s64 b1, %2, 2;\n\t"
      "add.s64 a2, %1, 4;\n\t add.s64 b2, %2, 4;\n\t"
      "add.s64 a3, %1, 6;\n\t add.s64 b3, %2, 6;\n\t"
      "add.s64 a4, %1, %5;\n\t add.s64 b4, %2, %6;\n\t"
      "add.s64 a5, a4, 2;\n\t add.s64 b5, b4, 2;\n\t"
      "add.s64 a6, a4, 4;\n\t add.s64 b6, b4, 4;\n\t"
      "add.s64 a7, a4, 6;\n\t add.s64 b7, b4, 6;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a1, b1, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a2, b2, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a3, b3, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a4, b4, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a5, b5, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a6, b6, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], a7, b7, %3, t;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(kABox), "n"(kBBox)
      : "memory");
}

// Eight K=16 steps of a pair MMA with A in tensor memory (each CTA's 128
// rows, 8 columns per step) and B MN-major 128-byte swizzled in shared
// memory, 16 K rows (128 descriptor units) per step.
__device__ __forceinline__ void umma_pair_ts_k128(uint32_t d_tmem, uint32_t a_tmem,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t"
      ".reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
      ".reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "add.s32 a1, %1, 8;\n\t  add.s64 b1, %2, 128;\n\t"
      "add.s32 a2, %1, 16;\n\t add.s64 b2, %2, 256;\n\t"
      "add.s32 a3, %1, 24;\n\t add.s64 b3, %2, 384;\n\t"
      "add.s32 a4, %1, 32;\n\t add.s64 b4, %2, 512;\n\t"
      "add.s32 a5, %1, 40;\n\t add.s64 b5, %2, 640;\n\t"
      "add.s32 a6, %1, 48;\n\t add.s64 b6, %2, 768;\n\t"
      "add.s32 a7, %1, 56;\n\t add.s64 b7, %2, 896;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a1], b1, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a2], b2, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a3], b3, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a4], b4, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a5], b5, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a6], b6, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a7], b7, %3, t;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four K=16 steps of a pair MMA with A in tensor memory (a K = 64
// contraction: 8 columns of packed 16-bit pairs per step) and B MN-major
// 128-byte swizzled in shared memory (16 K rows = 128 descriptor units per
// step).
__device__ __forceinline__ void umma_pair_ts_k64(uint32_t d_tmem, uint32_t a_tmem,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e, t;\n\t"
      ".reg .b32 a1, a2, a3;\n\t"
      ".reg .b64 b1, b2, b3;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.eq.b32 t, 0, 0;\n\t"
      "add.s32 a1, %1, 8;\n\t  add.s64 b1, %2, 128;\n\t"
      "add.s32 a2, %1, 16;\n\t add.s64 b2, %2, 256;\n\t"
      "add.s32 a3, %1, 24;\n\t add.s64 b3, %2, 384;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a1], b1, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a2], b2, %3, t;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [a3], b3, %3, t;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at shared offset `bar` in each CTA of
// `cta_mask` when every pair MMA issued so far by the elected lane has
// completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster."
      "multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Ties 16 registers to this point of the program: placed after
// tcgen05.wait::ld, it keeps the compiler from moving uses of the loaded
// values above the wait (the registers are undefined until then).
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]),
                 "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]),
                 "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns: lane i of the warp gets row
// (taddr.lane + i), registers r[c] = column taddr.col + c.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]),
        "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns in one load: r0 gets columns
// taddr.col + 0..15, r1 columns taddr.col + 16..31 (one instruction instead
// of two tmem_ld16).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r0)[16],
                                          uint32_t (&r1)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]),
        "=r"(r0[6]), "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]),
        "=r"(r0[11]), "=r"(r0[12]), "=r"(r0[13]), "=r"(r0[14]), "=r"(r0[15]),
        "=r"(r1[0]), "=r"(r1[1]), "=r"(r1[2]), "=r"(r1[3]), "=r"(r1[4]), "=r"(r1[5]),
        "=r"(r1[6]), "=r"(r1[7]), "=r"(r1[8]), "=r"(r1[9]), "=r"(r1[10]),
        "=r"(r1[11]), "=r"(r1[12]), "=r"(r1[13]), "=r"(r1[14]), "=r"(r1[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr,
                                          const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
      "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),
      "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// 32 lanes x 32 bit, one column: lane i writes row (taddr.lane + i).
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r)
               : "memory");
}

// 32 lanes x 32 bit, one column (valid after tmem_wait_ld).
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr)
               : "memory");
  return r;
}

// ------------------------------------------------------------ math

// 2^x on the special-function unit (approximate, flush-to-zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (sm_100 family three-input max).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed pair of fp32 fused multiply-adds (one fma.rn.f32x2):
// (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1).
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1,
                                      float b0, float b1, float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// Packed pair of fp32 additions (one add.rn.f32x2).
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1,
                                      float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// ------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor for tcgen05.mma (sm_100 family layout):
// start address, leading / stride byte offsets (all >> 4), version 1, and the
// swizzle mode in bits 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr,
                                                    uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16 with fp32 accumulation.
//   bits 4-5 D format (1 = f32); 7-9 A format, 10-12 B format (0 = f16,
//   1 = bf16); bit 15 A major, bit 16 B major (0 = K-major, 1 = MN-major);
//   bits 17-22 N >> 3; bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, bool a_mn,
                                                 bool b_mn, int M, int N) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((static_cast<uint32_t>(N) >> 3) << 17) |
         ((static_cast<uint32_t>(M) >> 4) << 24);
}

}  // namespace fa
