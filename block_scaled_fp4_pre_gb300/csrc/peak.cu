// FP4 tensor-core throughput probe for sm_103a: the denominator of the layer's
// compute roofline, measured rather than taken from a datasheet.
//
// Each block keeps one 128-row MXFP4 weight tile, one N-row token tile and their
// UE8M0 scale blocks in shared memory (all zero: the values do not change the
// instruction's timing) and issues mma_count tcgen05 block-scaled MMAs of shape
// M=128 x N x K=64 into one TMEM accumulator -- the instruction the layer kernel
// issues, with no global-memory traffic.  The caller times the launch with events.
//
// Pages: "[deepseek-v4] Bump sgl-deep-gemm for packed FP4xFP4 mega-MoE (W4A4)",
// Appendix B (the layer's Compute SOL figure, which needs a compute peak to be read
// against).
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mxmoe {
namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeATile = kBM * kBKBytes;            // 16 KiB
constexpr int kProbeMaxN = 256;

template <int BPS>
__global__ void __launch_bounds__(kProbeThreads, BPS)
    fp4_mma_probe_kernel(int n, long long mma_count, int32_t* flags) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t done_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* a_tile = smem;
  uint8_t* b_tile = a_tile + kProbeATile;
  uint8_t* sf = b_tile + (size_t)n * kBKBytes;
  const int bytes = kProbeATile + n * kBKBytes + 2 * kSFAtomBytes;   // multiple of 16
  for (int i = threadIdx.x * 16; i < bytes; i += kProbeThreads * 16)
    *reinterpret_cast<uint4*>(smem + i) = make_uint4(0u, 0u, 0u, 0u);
  // Tensor-memory columns: the accumulator (n columns, rounded up to 128), then
  // the A and B scale registers, 16 columns each.
  constexpr uint32_t kCols = BPS == 1 ? 512u : 256u;
  const uint32_t acc_cols = n <= 128 ? 128u : 256u;
  if (threadIdx.x < 32) {
    ptx::tmem_alloc(&tmem_base_sh, kCols);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    ptx::mbar_init(&done_bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  ptx::fence_proxy_async_smem();   // the zero fill is read by the tensor core
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (threadIdx.x == 0) {
    const uint32_t sfa = tmem + acc_cols, sfb = sfa + 16;
    const uint32_t s_sf = ptx::smem_addr(sf);
    for (int a = 0; a < 2; ++a) {
      ptx::tc_cp_sf(sfa + a * 4, ptx::desc_sf(s_sf));
      ptx::tc_cp_sf(sfb + a * 4, ptx::desc_sf(s_sf + kSFAtomBytes));
      ptx::tc_cp_sf(sfb + 8 + a * 4, ptx::desc_sf(s_sf + kSFAtomBytes));
    }
    const uint32_t a0 = ptx::smem_addr(a_tile), b0 = ptx::smem_addr(b_tile);
    for (long long i = 0; i < mma_count; ++i) {
      const int s = (int)(i & 3);   // four K=64 steps of one 256-element k-block
      ptx::tc_mma_mxf4(tmem, ptx::desc_sw128(a0 + s * 32), ptx::desc_sw128(b0 + s * 32),
                       ptx::idesc_mxf4(n, (s & 1) * 2), sfa + (s >> 1) * 4, sfb + (s >> 1) * 4,
                       i != 0 ? 1u : 0u);
    }
    ptx::tc_commit(&done_bar);
    if (!ptx::mbar_wait(&done_bar, 0, &abort_flag, kWaitLimitNs)) atomicOr(&flags[0], kErrTimeout);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kCols);
  }
}

// Shared memory requested per block: enough that no more than BPS blocks fit on
// one SM, so that every SM runs exactly BPS of them when blocks = SMs x BPS.
template <int BPS>
constexpr int probe_launch_smem() {
  return BPS == 1 ? 120 * 1024 : 100 * 1024;
}
static_assert(probe_launch_smem<2>() >= 1024 + kProbeATile + kProbeMaxN * kBKBytes + 2 * kSFAtomBytes,
              "probe tiles must fit");

template <int BPS>
cudaError_t launch_probe(int n, int blocks, long long mma_count, int32_t* flags, cudaStream_t st) {
  const size_t smem = probe_launch_smem<BPS>();
  cudaError_t e = cudaFuncSetAttribute(fp4_mma_probe_kernel<BPS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  fp4_mma_probe_kernel<BPS><<<blocks, kProbeThreads, smem, st>>>(n, mma_count, flags);
  return cudaGetLastError();
}

// The same instruction stream in its two-SM form: each 2-CTA cluster issues, from its
// leader, block-scaled MXFP4 MMAs of shape M=256 (128 weight rows in each CTA's shared
// memory) x N x K=64, B split N/2 per CTA, each CTA's 128 accumulator rows in its own
// tensor memory (tcgen05 cta_group::2) -- the form whose operand bytes per FLOP are
// half the single-CTA M=128 ones.  One CTA per SM (the shared-memory request keeps a
// second one off), 512 tensor-memory columns: accumulator, then the scales.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kProbeThreads, 1)
    fp4_mma_probe_pair_kernel(int n, long long mma_count, int32_t* flags) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t done_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* a_tile = smem;
  uint8_t* b_tile = a_tile + kProbeATile;                       // N/2 rows here
  uint8_t* sf = b_tile + (size_t)(kProbeMaxN / 2) * kBKBytes;   // SFA, SFB (two blocks)
  const int bytes = kProbeATile + (kProbeMaxN / 2) * kBKBytes + 3 * kSFAtomBytes;
  for (int i = threadIdx.x * 16; i < bytes; i += kProbeThreads * 16)
    *reinterpret_cast<uint4*>(smem + i) = make_uint4(0u, 0u, 0u, 0u);
  const uint32_t rank = ptx::cluster_ctarank();
  if (threadIdx.x < 32) {
    ptx::tmem_alloc_pair(&tmem_base_sh, 512);
    ptx::tmem_relinquish_pair();
  }
  if (threadIdx.x == 0) {
    ptx::mbar_init(&done_bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  ptx::fence_proxy_async_smem();   // the zero fill is read by the tensor core
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();             // both CTAs' barriers and operands are ready
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (rank == 0 && threadIdx.x == 0) {
    const uint32_t sfa = tmem + 256, sfb = sfa + 8;
    const uint32_t s_sf = ptx::smem_addr(sf);
    for (int a = 0; a < 2; ++a) {
      ptx::tc_cp_sf_pair(sfa + a * 4, ptx::desc_sf(s_sf));
      ptx::tc_cp_sf_pair(sfb + a * 8, ptx::desc_sf(s_sf + kSFAtomBytes));
      ptx::tc_cp_sf_pair(sfb + a * 8 + 4, ptx::desc_sf(s_sf + 2 * kSFAtomBytes));
    }
    const uint32_t a0 = ptx::smem_addr(a_tile), b0 = ptx::smem_addr(b_tile);
    for (long long i = 0; i < mma_count; ++i) {
      const int s = (int)(i & 3);
      ptx::tc_mma_mxf4_pair(tmem, ptx::desc_sw128(a0 + s * 32), ptx::desc_sw128(b0 + s * 32),
                            ptx::idesc_mxf4_m(256, n, (s & 1) * 2), sfa + (s >> 1) * 4,
                            sfb + (s >> 1) * 8, i != 0 ? 1u : 0u);
    }
    const uint32_t bar = ptx::smem_addr(&done_bar);
    ptx::tc_commit_pair(ptx::mapa_shared(bar, 0));
    ptx::tc_commit_pair(ptx::mapa_shared(bar, 1));
  }
  // both CTAs wait for the pair's MMAs before their memory may go
  if (threadIdx.x == 0 && !ptx::mbar_wait(&done_bar, 0, &abort_flag, kWaitLimitNs))
    atomicOr(&flags[0], kErrTimeout);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  if (threadIdx.x < 32) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_fp4_mma_probe_pair(int n, int pairs, long long mma_count, int32_t* flags,
                                      cudaStream_t st) {
  const size_t smem = probe_launch_smem<1>();
  cudaError_t e = cudaFuncSetAttribute(fp4_mma_probe_pair_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  fp4_mma_probe_pair_kernel<<<2 * pairs, kProbeThreads, smem, st>>>(n, mma_count, flags);
  return cudaGetLastError();
}

cudaError_t launch_fp4_mma_probe(int n, int blocks_per_sm, int blocks, long long mma_count,
                                 int32_t* flags, cudaStream_t st) {
  return blocks_per_sm == 1 ? launch_probe<1>(n, blocks, mma_count, flags, st)
                            : launch_probe<2>(n, blocks, mma_count, flags, st);
}

}  // namespace mxmoe
