// MXFP8 producer for sm_103a: bf16 rows -> E4M3 values with one UE8M0 scale per 32
// elements, the scales written either packed four to an int32 along K or directly
// in the 4-D [ceil(rows/128), K/128, 32, 4] int32 layout of the consumer GEMM, with
// padded rows' scales zero (so the live rows' scales are a prefix of a buffer sized
// for more rows).
//
// Pages: SGLang PR #48424, section "DeepGEMM producers write FlashInfer's 128x4 scale
// layout" (the MXFP8 pair, the 4-D scale shape, zeroed padded rows, live rows as a
// prefix under graph replay).
//
// One block covers 128 rows x 128 elements of K, whose scales are exactly one 512-byte
// block of the 4-D layout.  Sixteen threads share a row (16 bytes of bf16 each, so a
// warp reads two whole 256-byte row segments), four consecutive lanes hold one
// 32-element group and reduce its amax with two shuffles.  HBM-bound: 2 bytes read and
// 1 + 1/32 written per element.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mxmoe {
namespace {

constexpr int kRowsPerBlock = 128;
constexpr int kColsPerBlock = 128;
constexpr int kThreads8 = 256;
constexpr unsigned kFull8 = 0xFFFFFFFFu;

using ptx::e4m3x2;
using ptx::mxfp8_exponent;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(kThreads8)
    mxfp8_quantize_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t K,
                          uint8_t* __restrict__ q, uint8_t* __restrict__ sf, int layout) {
  __shared__ alignas(16) uint8_t atom[kRowsPerBlock * 4];   // this block's 128 x 4 scales
  const int t = threadIdx.x;
  const int64_t kc = blockIdx.y;                  // 128-element column block
  const int64_t r0 = (int64_t)blockIdx.x * kRowsPerBlock;
  reinterpret_cast<uint16_t*>(atom)[t] = 0;       // padded rows keep zero scales
  __syncthreads();
  const int c = t & 15;                           // 8-element piece of the row segment
  const int g = c >> 2;                           // its 32-element group (0..3)
  constexpr int kIters = kRowsPerBlock / 16;
  // All of this thread's loads first (eight rows, 16 bytes each), so that they are
  // in flight together.
  uint4 ws[kIters];
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int64_t r = r0 + it * 16 + (t >> 4);
    ws[it] = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows)
      ws[it] = __ldcs(reinterpret_cast<const uint4*>(x + r * K + kc * kColsPerBlock + c * 8));
  }
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int rl = it * 16 + (t >> 4);
    const int64_t r = r0 + rl;
    const bool live = r < rows;
    const int64_t off = r * K + kc * kColsPerBlock + c * 8;
    const uint4 w = ws[it];
    float v[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                  bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(kFull8, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull8, amax, 2));
    const int e = mxfp8_exponent(amax);
    const float s = ptx::pow2_neg(e);             // exact power of two
    if (live) {
      uint2 o;
      o.x = e4m3x2(v[0] * s, v[1] * s) | (e4m3x2(v[2] * s, v[3] * s) << 16);
      o.y = e4m3x2(v[4] * s, v[5] * s) | (e4m3x2(v[6] * s, v[7] * s) << 16);
      *reinterpret_cast<uint2*>(q + off) = o;
      if ((c & 3) == 0) {
        const uint8_t b = (uint8_t)(e + 127);
        if (layout == MOE_SF_128X4)
          atom[(rl & 31) * 16 + (rl >> 5) * 4 + g] = b;
        else
          atom[rl * 4 + g] = b;                   // row-major staging for the packed words
      }
    }
  }
  __syncthreads();
  if (layout == MOE_SF_128X4) {
    if (t < 32)
      reinterpret_cast<uint4*>(sf + ((uint64_t)blockIdx.x * (K / kColsPerBlock) + kc) * 512)[t] =
          reinterpret_cast<const uint4*>(atom)[t];
  } else if (t < kRowsPerBlock && r0 + t < rows) {
    reinterpret_cast<uint32_t*>(sf)[(r0 + t) * (K / kColsPerBlock) + kc] =
        reinterpret_cast<const uint32_t*>(atom)[t];
  }
}

}  // namespace

size_t mxfp8_scale_bytes(int64_t rows_cap, int64_t K, int layout) {
  const int64_t words = K / kColsPerBlock;
  if (layout == MOE_SF_128X4)
    return (size_t)((rows_cap + kRowsPerBlock - 1) / kRowsPerBlock) * (size_t)words * 512;
  return (size_t)rows_cap * (size_t)words * 4;
}

cudaError_t launch_mxfp8_quantize(const void* x, int64_t rows, int64_t K, void* q, void* sf,
                                  int layout, int64_t rows_cap, cudaStream_t st) {
  // Scales of rows no block writes: whole padded 128-row blocks (4-D layout) or
  // rows past the live ones (packed layout).  Either is one contiguous tail.
  const size_t live = layout == MOE_SF_128X4 ? mxfp8_scale_bytes(rows, K, layout)
                                             : (size_t)rows * (size_t)(K / kColsPerBlock) * 4;
  const size_t total = mxfp8_scale_bytes(rows_cap, K, layout);
  if (total > live) {
    cudaError_t e = cudaMemsetAsync(static_cast<uint8_t*>(sf) + live, 0, total - live, st);
    if (e != cudaSuccess) return e;
  }
  if (rows == 0) return cudaSuccess;
  // Row blocks on x (up to 2^23 / 128 = 65536 of them, past grid.y's limit), column
  // blocks on y (K / 128 <= 65535, checked by the caller).
  const dim3 grid((unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)(K / kColsPerBlock));
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  mxfp8_quantize_kernel<<<grid, kThreads8, 0, st>>>(static_cast<const uint16_t*>(x), rows, K,
                                                    static_cast<uint8_t*>(q),
                                                    static_cast<uint8_t*>(sf), layout);
  return cudaGetLastError();
}

}  // namespace mxmoe
