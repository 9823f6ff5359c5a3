// Inline-PTX wrappers for sm_103a: mbarrier, TMA bulk copies, tcgen05 (TMEM, block-scaled
// MMA, scale-factor copies), and MXFP4 element conversion.
#pragma once

#include <stdint.h>

namespace mxmoe {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- programmatic dependent launch ------------------------------------------
// Lets the next kernel in the stream be scheduled now (its blocks start once
// resources allow and wait in pdl_wait for this grid's memory).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the previous kernel in the stream has completed and its writes are
// visible.  A no-op for kernels launched without the programmatic attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up (returns
// false) when *abort becomes nonzero or after limit_ns; in the latter case it
// sets *abort so that the other roles of the block stop too.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
}

// ---- global-memory ordering ---------------------------------------------------
__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Waits until *p >= target (acquire), bounded like mbar_wait: gives up when *abort
// becomes nonzero or after limit_ns, setting *abort in the latter case.
__device__ __forceinline__ bool wait_counter(const int32_t* p, int target, volatile int* abort,
                                             unsigned long long limit_ns) {
  if (ld_acquire(p) >= target) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    __nanosleep(128);
    if (ld_acquire(p) >= target) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
}

// Orders this thread's generic-proxy global accesses with its async-proxy (TMA)
// accesses to global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory writes before later
// async-proxy (TMA, tensor core) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- L2 cache policies -----------------------------------------------------
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- TMA -------------------------------------------------------------------
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load of a box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int32_t x, int32_t y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Per-thread asynchronous copies global -> shared (no registers involved): 16 bytes
// (both addresses 16-byte aligned, L2 only) or 4 bytes (4-byte aligned).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
               : "memory");
}
// Makes `bar` wait for this thread's earlier cp.async copies: its pending count
// goes up by one now and back down when they have all landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Waits for all of this thread's cp.async copies.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Prefetch of a 2-D box into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const void* tmap, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y)
               : "memory");
}

// Prefetch of a contiguous range into L2 (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_prefetch(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// fp32 reduction into global memory with an L2 eviction policy for the line.
__device__ __forceinline__ void red_add_f32(float* p, float v, uint64_t policy) {
  asm volatile("red.global.add.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(policy)
               : "memory");
}

// ---- tcgen05 ---------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrives once on `bar` when all tcgen05 operations issued so far by this thread
// have completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// Copies a 32-row x 16-byte block of scale factors from shared memory to tensor
// memory, replicated into all four 32-lane quarters.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with MXFP4 operands and UE8M0 scales from tmem.
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with A = E2M1 in the 8-bit-container layout that
// a CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B copy writes, B = E4M3, one UE8M0 scale per
// 32 elements of K for each (K = 32 per instruction).
__device__ __forceinline__ void tc_mma_f8f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: 8-row x 128-byte
// atoms stacked every 1024 bytes.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;              // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;              // descriptor version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}

// Descriptor of a 32-row x 16-byte scale block (rows 16 bytes apart, no swizzle).
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 32;     // stride byte offset: next 8-row core matrix
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor of kind::mxf4 with E2M1 A and B, UE8M0 scales, M = 128,
// K-major operands; sf_id picks the byte pair of the scale registers.
__device__ __forceinline__ uint32_t idesc_mxf4(int N, int sf_id) {
  return ((uint32_t)sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         (1u << 23) | ((uint32_t)(128 >> 4) << 24) | ((uint32_t)sf_id << 29);
}

// Instruction descriptor of kind::mxf8f6f4 with A = E2M1 (format 5), B = E4M3
// (format 0), UE8M0 scales, M = 128, K-major operands; sf_id (0..3) picks the scale
// byte of the four a scale register holds for each row.
__device__ __forceinline__ uint32_t idesc_f8f4(int N, int sf_id) {
  return ((uint32_t)sf_id << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) |
         (1u << 23) | ((uint32_t)(128 >> 4) << 24) | ((uint32_t)sf_id << 29);
}

// 32 lanes x 32 consecutive fp32 columns of tensor memory into registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 16 consecutive fp32 columns of tensor memory into registers.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Starts a load of 32 lanes x 16 consecutive fp32 columns of tensor memory; the
// registers are valid only after tmem_wait_ld on them.
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// Waits for this thread's tensor-memory loads; r is tied to the wait so that no
// use of it moves above it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Stores 32 lanes x 16 consecutive 32-bit columns of tensor memory from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// Waits for this thread's tensor-memory stores.
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- CTA pairs (2-CTA clusters, tcgen05 cta_group::2) -------------------------
// A pair's leader (rank 0) issues the MMAs; each MMA spans both CTAs' shared memory
// (A: 128 rows each, B: N/2 rows each, at the same offsets) and writes each CTA's
// 128 accumulator rows into that CTA's tensor memory.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Every thread of both CTAs: release this CTA's earlier shared-memory writes, wait
// for all threads of the cluster (a hardware barrier, like __syncthreads).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Arrives once on an mbarrier given by its shared::cluster address (either CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}
// One warp of each CTA of the pair, together: the same columns in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Leader only: each CTA's 32-row x 16-byte scale block (same shared offset) into that
// CTA's tensor memory (same address), replicated into all four lane quarters.
__device__ __forceinline__ void tc_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// Leader only: D (+)= A * B^T with M = 256 across the pair (see above), MXFP4 operands
// and UE8M0 scales; each CTA's tensor memory holds its rows' scales and all N of B's.
__device__ __forceinline__ void tc_mma_mxf4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t sfa_tmem,
                                                 uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
// Leader only: arrives once on the mbarrier at a shared::cluster address (this CTA's
// or the peer's) when the pair's earlier tcgen05 operations issued here complete.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar_cluster) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          bar_cluster)
      : "memory");
}
// 2-D tiled load into this CTA's shared memory (dst: its shared-window address) whose
// completion (bytes) is signalled on an mbarrier of either CTA of the pair (given by
// its shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, int32_t x,
                                                 int32_t y, uint32_t bar_cluster, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::"
      "bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
      : "memory");
}
// Instruction descriptor of kind::mxf4 (E2M1 A and B, UE8M0 scales, K-major) for an
// M-row (128 or, across a pair, 256) by N MMA; sf_id picks the scale byte pair.
__device__ __forceinline__ uint32_t idesc_mxf4_m(int M, int N, int sf_id) {
  return ((uint32_t)sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         (1u << 23) | ((uint32_t)(M >> 4) << 24) | ((uint32_t)sf_id << 29);
}

// ---- MXFP4 element math ----------------------------------------------------
// Smallest e with amax <= 6 * 2^e, clamped below at -127 (finite fp32 gives e <= 126).
// amax = 1.m * 2^p: 6 * 2^e = 1.5 * 2^(e+2), so e = p - 2 when 1.m <= 1.5, else p - 1.
__device__ __forceinline__ int mx_scale_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int biased = (int)((b >> 23) & 0xFFu);
  if (biased == 0) return -127;  // zero or subnormal: 6 * 2^-127 already covers it
  const int e = biased - 129 + (((b & 0x7FFFFFu) > 0x400000u) ? 1 : 0);
  return e < -127 ? -127 : e;
}

// 2^-e as an fp32 (e in [-127, 126]).
__device__ __forceinline__ float pow2_neg(int e) {
  return __uint_as_float((uint32_t)(127 - e) << 23);
}

// E2M1 codes of eight scaled values (|v| <= 6) with their signs, element i in bits
// 4i..4i+3 (so element 2j sits in the low nibble of byte j).  The conversion keeps
// each value's sign, so a negative value that rounds to zero gives code 0x8.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// E2M1 byte of two scaled values with their signs, `a` in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float a, float b) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "mov.b16 %0, {t, t};\n\t}"
      : "=h"(r)
      : "f"(b), "f"(a));
  return (uint32_t)r & 0xFFu;
}

// ---- MXFP8 element math ----------------------------------------------------
// Smallest e with amax <= 448 * 2^e, clamped below at -127 (fp32 bit arithmetic:
// amax = 1.m * 2^p needs e >= p - 8, one more when 1.m > 1.75).
__device__ __forceinline__ int mxfp8_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int biased = (int)((b >> 23) & 0xFFu);
  if (biased == 0) return -127;   // zero or subnormal: 448 * 2^-127 already covers it
  const int e = biased - 135 + (((b & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
  return e < -127 ? -127 : e;
}

// Two scaled values (|v| <= 448) to E4M3, round to nearest even; `lo` in bits 0-7.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// Eight scaled values to E4M3 bytes, element i in byte i.
__device__ __forceinline__ uint2 e4m3x8(const float (&v)[8]) {
  return make_uint2(e4m3x2(v[0], v[1]) | (e4m3x2(v[2], v[3]) << 16),
                    e4m3x2(v[4], v[5]) | (e4m3x2(v[6], v[7]) << 16));
}

// ---- NVFP4 element math ------------------------------------------------------
// Value of an unsigned E4M3 byte (sign bit ignored): exponent field 0 holds m/8 *
// 2^-6, otherwise (1 + m/8) * 2^(e-7); built from the fields, exact in fp32.
__device__ __forceinline__ float ue4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  return e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// NVFP4 block scale of a 16-element group: the E4M3 byte nearest to amax / 6
// (correctly rounded fp32 division, then round to nearest even, saturating at 448).
__device__ __forceinline__ uint32_t nvfp4_scale_byte(float amax) {
  return e4m3x2(__fdiv_rn(amax, 6.0f), 0.f) & 0x7Fu;
}

// D[tmem] (+)= A[smem] * B[smem]^T, packed E2M1 operands with one UE4M3 scale per 16
// elements of K for each (K = 64 per instruction: four scales, one 32-bit scale word).
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Instruction descriptor of kind::mxf4nvf4 with E2M1 A and B, UE4M3 scales (scale
// type bit 23 clear), M = 128, K-major operands; the four scales of a step fill the
// whole scale word, so both scale ids are 0.
__device__ __forceinline__ uint32_t idesc_nvf4(int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

}  // namespace ptx
}  // namespace mxmoe
