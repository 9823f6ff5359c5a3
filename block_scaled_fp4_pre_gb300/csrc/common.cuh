// Internal definitions shared by the CUDA translation units of libmxmoe.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "mxmoe.h"

namespace mxmoe {

// ---------------------------------------------------------------------------
// Tile geometry of the grouped GEMMs (weights on the MMA M side, tokens on N).
constexpr int kBM = 128;            // weight rows per tile (MMA M)
constexpr int kBN = 128;            // token rows per tile (max MMA N); expert segments are
                                    // padded to multiples of kBN rows
constexpr int kBK = 256;            // FP4 elements per k-block = one 128-byte swizzle row
constexpr int kBKBytes = kBK / 2;   // 128
constexpr int kATileBytes = kBM * kBKBytes;   // 16 KiB
constexpr int kBTileBytes = kBN * kBKBytes;   // 16 KiB
constexpr int kBBoxRows = 32;                 // token rows per TMA box
constexpr int kSFAtomBytes = 512;             // 128 rows x 4 scale bytes
constexpr int kSFStageBytes = 2 * kSFAtomBytes;  // 8 scale columns per k-block
// Narrower token tiles for lighter loads: 32 (decode-sized) or 64 token rows a tile,
// expert segments padded to that many rows, each tile's token scales in 128x4 blocks
// of its own (its rows in the first quarter or half of each block).
constexpr int kBNNarrow = 32;
constexpr int kBNMedium = 64;
// Token tiles of the pair kernel (two SMs share each item, tcgen05 cta_group::2): up
// to kBNPair rows, each starting at a whole 128-row scale block, so a tile spans
// kPairStride workspace rows of which it uses kBNPair.
constexpr int kBNPair = 192;
constexpr int kPairStride = 256;

// Workspace row, from its expert's segment start, of the expert's r-th assignment
// under a dispatch with token tiles of tile_rows rows.
__host__ __device__ __forceinline__ int tile_row_of_rank(int r, int tile_rows) {
  return tile_rows == kBNPair ? (r / kBNPair) * kPairStride + r % kBNPair : r;
}

// Workspace rows of an expert segment holding n assignments: whole tiles (tiles of up
// to 128 rows), or whole kPairStride spans and a last partial tile padded to 128 rows.
__host__ __device__ __forceinline__ int segment_rows(int n, int tile_rows) {
  if (tile_rows == kBNPair) {
    const int rem = n % kBNPair;
    return n / kBNPair * kPairStride + (rem + kBN - 1) / kBN * kBN;
  }
  return (n + tile_rows - 1) / tile_rows * tile_rows;
}

// Device error bits in ws.flags[0].
constexpr int kErrRouting = 1;
constexpr int kErrTimeout = 2;

// Other words of ws.flags: [1] number of token tiles, [2] valid assignments,
// [3] next work item of the layer kernel, [4] blocks of the layer kernel done.
constexpr int kFlagTiles = 1;
constexpr int kFlagValid = 2;
constexpr int kFlagSched = 3;
constexpr int kFlagExit = 4;
constexpr int kFlagBucketTicket = 5;   // blocks of the bucketing kernel done
constexpr int kFlagBucketBad = 6;      // ids outside [0, E) seen by the bucketing kernel

constexpr int kFlagProbe = 8;          // a counter nothing increments (wait probe)

// Assignments (t*k + j) ranked by one block of the bucketing kernel.
constexpr int kBucketChunk = 8192;

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Byte offset of scale column s of row `row` in the 128x4 block layout
// (int32 view [rows/128][Kc/4][32][4]); kc4 = Kc / 4.
__host__ __device__ __forceinline__ size_t sf_atom_offset(size_t row, int s, int kc4) {
  return (((row >> 7) * (size_t)kc4 + (size_t)(s >> 2)) << 9) + ((row & 31) << 4) +
         (((row >> 5) & 3) << 2) + (size_t)(s & 3);
}

// Canonical row (gate 0..I-1, up I..2I-1) of the first weight stored at prepared
// row r under the gran=16 even/odd interleave.
__host__ __device__ __forceinline__ int gate_up_source_row(int r, int I) {
  const int chunk = r >> 5, within = r & 31;
  const int odd = within >> 4;
  const int is_up = (within >> 3) & 1;
  return is_up * I + chunk * 16 + (within & 7) * 2 + odd;
}

// The same under the gran=8 contiguous interleave of FP8 activations: prepared rows
// [gate 0..7, up 0..7, gate 8..15, up 8..15, ...].
__host__ __device__ __forceinline__ int gate_up_source_row8(int r, int I) {
  const int chunk = r >> 4, within = r & 15;
  return (within >> 3) * I + chunk * 8 + (within & 7);
}

// Interleave by activation format: gran=8 when f8, else gran=16.
__host__ __device__ __forceinline__ int gate_up_source_row_for(int r, int I, int f8) {
  return f8 ? gate_up_source_row8(r, I) : gate_up_source_row(r, I);
}

// Byte of token-side scale (row, scale column s) in a workspace of tiles of tile_rows
// rows (32, 64 or 128): the tile of rows tile_rows*t.. owns its scale blocks, with its
// row r in line r % 32, 4-byte word r / 32.  For 128-row tiles this is sf_atom_offset.
__host__ __device__ __forceinline__ size_t sf_tile_offset(size_t row, int s, int kc4,
                                                          int tile_rows) {
  const size_t tile = row / (size_t)tile_rows, r = row % (size_t)tile_rows;
  return ((tile * (size_t)kc4 + (size_t)(s >> 2)) << 9) + ((r & 31) << 4) + ((r >> 5) << 2) +
         (size_t)(s & 3);
}

// ---------------------------------------------------------------------------
// Workspace layout (computed on the host from the dims, passed to kernels).
struct WsLayout {
  int64_t T_cap, A_cap, R_cap, tiles_cap;
  size_t off_header, off_flags, off_counts, off_seg, off_tiles, off_tile_done, off_assign,
      off_local_rank, off_blk_base, off_tile_start,
      off_slot_token, off_slot_assign, off_slot_weight, off_xb, off_xsf, off_xq, off_xs, off_hb,
      off_hsf, off_acc, off_stage_x, off_stage_ids, off_stage_w, off_stage_out, total;
};

struct WsPtrs {
  int32_t* flags;        // error bits and counters, see kFlag*
  int32_t* counts;       // [E]
  int32_t* seg;          // [E+1] first workspace row of each expert (multiples of kBN)
  int4* tiles;           // [tiles_cap] (expert, first row, rows, 0), experts in order
  int32_t* tile_start;   // [E+1] first tile of each expert (exclusive prefix of tiles)
  int32_t* tile_done;    // [tiles_cap] gate/up items finished per token tile
  int32_t* assign_slot;  // [A_cap] workspace row of assignment t*k+j, -1 if skipped
  int32_t* local_rank;   // [A_cap] rank of an assignment among its expert's, in its chunk
  int32_t* blk_base;     // [A_cap/kBucketChunk + 1][E] rows of an expert in earlier chunks
  int32_t* slot_token;   // [R_cap]
  int32_t* slot_assign;  // [R_cap]
  float* slot_weight;    // [R_cap]
  uint8_t* xb;           // [R_cap, H/2] (FP4) or [R_cap, H] (FP8) quantised token rows
  uint8_t* xsf;          // 128x4 blocks of [R_cap, H/32] (H/16 for NVFP4)
  uint8_t* xq;           // [T_cap, H/2] quantised token rows, one per token (pull dispatch)
  uint8_t* xs;           // [T_cap, H/32] their scales, row-major (pull dispatch)
  uint8_t* hb;           // [R_cap, I/2] (FP4) or [R_cap, I] (FP8) requantised intermediate rows
  uint8_t* hsf;          // 128x4 blocks of [R_cap, I/32] (I/16 for NVFP4)
  float* acc;            // [T_cap, H] fp32 combine accumulator, cleared by pre_dispatch
};

struct PrepLayout {
  size_t off_w1c, off_w1s, off_w2c, off_w2s, total;
};

struct Shape {
  int H, I, E, k;
  int f8;   // 1: fp8xfp4 (E4M3 activations, gran=8 interleave)
  int nv;   // 1: nvf4xnvf4 (E4M3 scale per 16 elements); both 0: mxf4xmxf4
};

// Elements per scale of the format: 16 (NVFP4) or 32 (MXFP4, MXFP8).
__host__ __device__ __forceinline__ int sf_group(const Shape& s) { return s.nv ? 16 : 32; }

// Prepared weight codes are stored in k-block tiles: the 128 rows of one weight slab
// over one k-block are contiguous, row after row, so each TMA box of the layer
// kernel reads one contiguous 16 KiB (8 KiB for fp8xfp4) run of memory.  A tile row
// holds one k-block's packed E2M1 bytes: 128 (256 elements) or, for fp8xfp4, whose
// k-blocks are 128 elements, 64.  Byte j of weight row R of a matrix with K elements
// a row sits at ((R / 128 * num_kb + j / kb_bytes) * 128 + R % 128) * kb_bytes +
// j % kb_bytes; a last k-block shorter than the others is zero-padded to full width.
__host__ __device__ __forceinline__ int weight_kb_bytes(const Shape& s) { return s.f8 ? 64 : 128; }
__host__ __device__ __forceinline__ int64_t weight_num_kb(const Shape& s, int64_t K) {
  const int64_t elems = 2 * (int64_t)weight_kb_bytes(s);
  return (K + elems - 1) / elems;
}
// Bytes of the tiled codes of `rows` weight rows (a multiple of 128) of K elements.
__host__ __device__ __forceinline__ int64_t weight_code_bytes(const Shape& s, int64_t rows,
                                                              int64_t K) {
  return rows * weight_num_kb(s, K) * weight_kb_bytes(s);
}

// Launch with programmatic stream serialisation: the kernel may start before the
// previous kernel in the stream finishes and must call ptx::pdl_wait() before it
// touches that kernel's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  cfg.attrs = attr;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Launchers implemented in dispatch.cu / gemm.cu.  Each returns the cudaError_t
// of its launch.
// Bucketing: per-expert counts and segment starts, the tile list, and each
// assignment's rank; the quantiser (or launch_assign_slots) turns ranks into rows.
// tile_rows: kBN (wide tiles), kBNMedium, kBNNarrow or kBNPair.
cudaError_t launch_bucket(const Shape& s, const int32_t* ids, int T, const WsPtrs& ws,
                          int tile_rows, cudaStream_t st);
// Quantise the tokens, give every assignment its row and copy the token there.
// pull: write each token's row once (xq/xs) instead of copying it to its k rows; the
// layer kernel then gathers token rows itself.
// tile_rows: the dispatch's token tiles (rows from tile_row_of_rank; token scales in the
// layout of tiles of min(tile_rows, 128) rows, sf_tile_offset).
cudaError_t launch_quantize_scatter(const Shape& s, const void* x, const int32_t* ids,
                                    const float* tw, int T, const WsPtrs& ws, bool pull,
                                    int tile_rows, cudaStream_t st);
// Rows of all assignments (128-row tiles) and the per-row tables, without quantising
// anything.
cudaError_t launch_assign_slots(const Shape& s, const int32_t* ids, const float* tw, int T,
                                const WsPtrs& ws, cudaStream_t st);
// acc [n] fp32 -> out [n] bf16 (round to nearest even).
cudaError_t launch_convert_out(const float* acc, void* out, int64_t n, cudaStream_t st);
cudaError_t launch_quantize_rows(const float* src, int64_t rows, int K, uint8_t* codes,
                                 uint8_t* sf, cudaStream_t st);
// fp32 rows -> NVFP4 codes and E4M3 scales (one per 16 elements).
cudaError_t launch_quantize_rows_nv(const float* src, int64_t rows, int K, uint8_t* codes,
                                 uint8_t* sf, cudaStream_t st);
cudaError_t launch_prepare(const Shape& s, const uint8_t* w1c, const uint8_t* w1s,
                           const uint8_t* w2c, const uint8_t* w2s, uint8_t* prep,
                           const PrepLayout& pl, cudaStream_t st);

// One block waiting, with the given limit, on an mbarrier no one arrives at and on a
// counter no one increments, through the same bounded waits as the layer kernel.
cudaError_t launch_wait_probe(int32_t* flags, unsigned long long limit_ns, cudaStream_t st);
size_t mxfp8_scale_bytes(int64_t rows_cap, int64_t K, int layout);
cudaError_t launch_mxfp8_quantize(const void* x, int64_t rows, int64_t K, void* q, void* sf,
                                  int layout, int64_t rows_cap, cudaStream_t st);
cudaError_t launch_fp4_mma_probe(int n, int blocks_per_sm, int blocks, long long mma_count,
                                 int32_t* flags, cudaStream_t st);
// M=256 across SM pairs (2-CTA clusters, tcgen05 cta_group::2), `pairs` clusters.
cudaError_t launch_fp4_mma_probe_pair(int n, int pairs, long long mma_count, int32_t* flags,
                                      cudaStream_t st);

// Records the message moe_last_error() returns on this thread.
void set_last_error(const char* msg);

// The layer kernel: gate/up GEMM + SwiGLU + requantisation, then down GEMM +
// weighted combine into the fp32 accumulator, in one persistent launch.  With num_phases == 1
// and gate_up_debug set it runs only the gate/up GEMM and writes raw accumulators.
struct LayerLaunch {
  const uint8_t* w1_codes;   // prepared gate/up codes [E*2I, H/2]
  const uint8_t* w1_sf;      // their scale blocks
  const uint8_t* w2_codes;   // prepared down codes [E*H, I/2]
  const uint8_t* w2_sf;
  int64_t R_cap;
  Shape shape;
  int T;
  int num_phases;
  WsPtrs ws;
  float* gate_up_debug;      // [T*k, 2I] (num_phases == 1)
  int num_sms;
  bool pull;                 // gate/up token rows gathered from ws.xq/xs (pull dispatch)
  int tile_rows;             // token rows a tile: 32, 64, 128 or kBNPair (the dispatch's choice)
};
cudaError_t launch_layer(const LayerLaunch& g, cudaStream_t st);
// The layer on SM pairs (pair.cu): kBNPair-row token tiles, mxf4xmxf4 only, bucketed
// dispatch; pair_shape_ok says whether the shape allows it (H and 2I multiples of 256).
bool pair_shape_ok(const Shape& s);
cudaError_t launch_layer_pair(const LayerLaunch& g, cudaStream_t st);

}  // namespace mxmoe
