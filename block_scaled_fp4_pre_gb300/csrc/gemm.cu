// The expert layer in one persistent kernel for sm_103a (tcgen05 + TMEM + TMA):
//   phase 0  grouped gate/up GEMM (block-scaled FP4 x FP4) -> SwiGLU -> MXFP4
//            requantisation of h
//   phase 1  grouped down GEMM -> top-k weighted combine (fp32 reductions into the
//            workspace accumulator; a small kernel then writes the bf16 output)
// plus a debug mode that runs phase 0 only and writes the raw fp32 accumulators.
//
// Pages: "[deepseek-v4] Bump sgl-deep-gemm for packed FP4xFP4 mega-MoE (W4A4)",
// Appendix B (one fused "mega" layer kernel that streams every touched expert's
// packed FP4 weights and is memory bound at ntok=512, BLOCK_K=256); SGLang PR #48424
// summary (block_m 64 for decode loads); prhub digest of PR #37279 (activation
// "swiglu"; the gran=16 interleave keeps each SwiGLU pair in one 32-row chunk).
//
// Orientation: the weight slab is the MMA's M=128 operand and the expert's tokens
// are the N operand (N = 32..128), so one instruction shape serves a decode load of
// a few tokens per expert as well as a prefill tile of 128 tokens.
//
// Work items are (token tile, 128-row weight slab): first every gate/up item, then
// every down item, each phase ordered expert by expert, then slab by slab, then by
// the expert's token tiles -- so the tiles of a busy expert take a weight slab in
// turn while it is in L2, and the expert's token rows stay in L2 for all its slabs.  Blocks take items from a global
// counter, so all gate/up items are claimed (by running blocks, with no
// dependencies) before any down item is, and a down item's wait for its tile's
// intermediate rows always ends -- whatever number of blocks is resident.  The
// last block to finish resets the counters for the next call.
//
// Roles (192 threads; two persistent blocks per SM, so that one block's MMA issue
// and epilogue overlap the other's -- a single block per SM leaves the stream
// waiting on its one MMA-issuing thread):
//   warp 0      scheduler + TMA producer: weight slab box (128 rows x 128 B), token
//               boxes (32 rows x 128 B each), both operands' 128x4 scale blocks.
//   warp 1      TMEM allocator; lane 0 issues tcgen05.cp (scales) + tcgen05.mma.
//   warps 2-5   epilogue: tcgen05.ld of the fp32 accumulator (lane quarter
//               warp % 4), then the phase's math and global stores.
// Every wait is bounded (kWaitLimitNs); a timeout sets the workspace error flag and
// all roles leave their loops, drain their copies and MMAs, free TMEM and return.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mxmoe {
namespace {

constexpr int kStages = 3;                 // wide token tiles
constexpr int kStagesNarrow = 4;           // 32- and 64-row token tiles
constexpr int kStagesNarrowF8 = 5;         // 32-row tiles, E4M3 tokens: one scale block a stage
constexpr int kMaxStages = kStagesNarrowF8;
constexpr int kThreads = 192;
constexpr int kBlocksPerSM = 2;
constexpr int kTmemCols = 256;             // half of the SM's tensor memory per block
constexpr int kAccCols = kBN;              // one fp32 accumulator of up to 128 columns
constexpr int kSfTmemBase = kAccCols;      // two buffers of scale registers after it

// Tensor-memory columns after the accumulator: two buffers of scale registers (A then
// B; 8 columns an operand, 16 for NVFP4's four scale blocks per k-block), then spare
// columns that hold a copy of the accumulator's first chunks, so that the accumulator
// can go back to the MMA issuer before the math.
template <bool NV>
struct TmemMap {
  static constexpr int kSfCols = NV ? 32 : 16;                // one buffer, A and B
  static constexpr int kSpareCol = kSfTmemBase + 2 * kSfCols;
  static constexpr int kSpareChunks = (kTmemCols - kSpareCol) / 16;
};
static_assert(TmemMap<false>::kSpareChunks == 6 && TmemMap<true>::kSpareChunks == 4,
              "tensor memory layout");
static_assert(kBN / 32 == 4, "row metadata: four registers a lane");
constexpr int kEpiCols = 16;               // accumulator columns per epilogue load
constexpr int kRing = 8;                   // work items in flight inside a block
constexpr unsigned kFull = 0xFFFFFFFFu;

enum LayerMode { kModeLayer = 0, kModeRaw = 1 };

// GLOBAL_TILES: the expert tile table stays in global memory (stage room is short).
template <bool GLOBAL_TILES>
struct __align__(16) SmemTail {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t mma_done;
  uint64_t ring_full[kRing];
  uint64_t ring_empty[kRing];
  int4 ring[kRing];          // (item, first row, rows | slab << 8, tile); item = -1: stop
  uint32_t tmem_base;
  int abort;
  float xchg[2][4][kEpiCols];
  // One chunk of intermediate rows, gathered from the four epilogue warps before
  // it is stored: per column, the item's 64 features (32 code bytes) and their two
  // scale bytes.  Double-buffered across chunks.
  alignas(16) uint8_t hstage[2][kEpiCols][64];   // 32 bytes used for E2M1, 64 for E4M3
  alignas(4) uint8_t sstage[2][kEpiCols][4];      // 2 scale bytes a column (4: NVFP4)
  // first tile of each expert (E <= 1024), see decode_item
  int32_t tile_start[GLOBAL_TILES ? 1 : 1025];
};

// Shared-memory map: kSt stages x (weight box, token boxes, both operands' scale
// blocks: 2 per k-block, 4 for NVFP4, 1 for the 128-element k-blocks of E4M3 tokens),
// then the tail.  Tiles of 32 or 64 rows need a quarter or half of the token room,
// which pays for a fourth stage (a fifth for 32-row tiles of E4M3 tokens, whose weight
// boxes carry half the bytes; NVFP4's larger scale blocks leave 64-row tiles at three).
template <bool NV, int TROWS, bool F8>
struct SmemMap {
  static constexpr int kSt = TROWS == kBN                 ? kStages
                             : TROWS == kBNNarrow && F8    ? kStagesNarrowF8
                             : TROWS == kBNMedium && NV    ? kStages
                                                           : kStagesNarrow;
  static constexpr int kBRows = TROWS;                           // token rows a stage holds
  static constexpr size_t kBSlot = (size_t)kBRows * kBKBytes;
  static constexpr size_t kSF = (size_t)(NV ? 4 : F8 ? 1 : 2) * kSFAtomBytes;
  static constexpr size_t kA = 0;
  static constexpr size_t kB = kA + (size_t)kSt * kATileBytes;
  static constexpr size_t kSFA = kB + (size_t)kSt * kBSlot;
  static constexpr size_t kSFB = kSFA + (size_t)kSt * kSF;
  static constexpr size_t kTail = kSFB + (size_t)kSt * kSF;
  // NVFP4's scale blocks and the fifth 32-row E4M3 stage take the tile table's room
  static constexpr bool kGlobalTiles = NV || (TROWS == kBNNarrow && F8);
  static constexpr size_t kBytes = kTail + sizeof(SmemTail<kGlobalTiles>) + 1024;  // + slack
  // two blocks per SM (228 KiB of shared memory, 1 KiB of it reserved per block)
  static_assert(2 * (kBytes + 1024) <= 228 * 1024, "two blocks per SM");
};

struct PhaseArgs {
  const uint8_t* w_sf;   // weight scale blocks
  const uint8_t* t_sf;   // token-side scale blocks
  int rows_per_expert;   // 2I (gate/up) or H (down)
  int K;                 // H (gate/up) or I (down)
  int m_tiles;           // rows_per_expert / 128
  int num_kb;            // k-blocks of 256 elements (the last may be 128 wide; F8: 128)
  int kc4;               // scale blocks per 128-row group: K/128 (K/64 for NVFP4)
};

struct LayerArgs {
  PhaseArgs ph[2];
  int num_phases;
  int H, I, T, E;
  WsPtrs ws;
  float* gate_up_debug;
};

struct Item {
  int phase, tile, mt, e, ntiles;
};

// Item g of the phase-major, expert-major, slab-major, tile-minor order.
// tile_start[e] is the first tile of expert e (experts without tokens repeat it).
// grp1 > 0 (wide tiles): the down items run in groups of grp1 output slabs -- all
// experts' items of slabs [grp1 * j, grp1 * (j + 1)) before the next group, expert-major
// inside a group -- so that the fp32 accumulator columns a group adds into (tokens x
// grp1 * 128 floats) stay in L2 while each token's k contributions arrive; a token's
// adds to one column otherwise come from experts far apart in the order, after the
// row has left L2.
__device__ __forceinline__ Item decode_item(int g, int n0, int m0, int m1, int E,
                                            const int32_t* __restrict__ tile_start,
                                            int num_tiles = 0, int grp1 = 0) {
  Item it;
  int m = m0;
  int slab0 = 0;   // first slab of the item's group
  it.phase = 0;
  if (g >= n0) {
    g -= n0;
    m = m1;
    it.phase = 1;
    if (grp1 > 0 && grp1 < m1) {
      const int ngrp = (m1 + grp1 - 1) / grp1;
      int j = g / (num_tiles * grp1);
      if (j > ngrp - 1) j = ngrp - 1;
      g -= j * num_tiles * grp1;
      slab0 = j * grp1;
      m = min(grp1, m1 - slab0);
    }
  }
  // last expert e with tile_start[e] * m <= g (that expert has tiles)
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] * m <= g)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int t0 = tile_start[lo];
  it.e = lo;
  it.ntiles = tile_start[lo + 1] - t0;
  const int local = g - t0 * m;
  it.mt = slab0 + local / it.ntiles;
  it.tile = t0 + local % it.ntiles;
  return it;
}

// Output slabs a group of down items spans (wide tiles): 4 x 128 features, so that at
// 16384 tokens the accumulator columns in use are 32 MiB.  Under the grouping the
// intermediate rows of down items are loaded with the normal L2 policy (they are read
// again only by the next group) and the reductions mark accumulator lines evict-last,
// so that the group's accumulator columns, not the intermediate rows, stay in L2.
constexpr int kDownGroup = 4;
constexpr bool kDownRowsNormal = true;
constexpr bool kAccKeep = true;

// silu(g) * u with fast exp and divide (a few ulp; well inside the MXFP4 rounding)
__device__ __forceinline__ float silu_times(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// F8: fp8xfp4 -- E4M3 token and intermediate rows (128 elements a k-block), E2M1
// weights widened to 8-bit containers by their TMA copies (CU_TENSOR_MAP_DATA_TYPE_
// 16U4_ALIGN16B), kind::mxf8f6f4 MMAs, gran=8 gate/up rows.  Otherwise mxf4xmxf4:
// packed E2M1 throughout, 256 elements a k-block, kind::mxf4 MMAs, gran=16.
// NV: nvf4xnvf4 -- as mxf4xmxf4 with one E4M3 scale per 16 elements (four scale
// blocks per k-block and operand), kind::mxf4nvf4 MMAs, NVFP4 requantisation.
// TROWS: token rows a tile (128, or 64 / 32 for lighter loads, with more stages).
template <int MODE, bool PULL, bool F8, bool NV, int TROWS>
__global__ void __launch_bounds__(kThreads, kBlocksPerSM)
    moe_layer_kernel(const __grid_constant__ CUtensorMap tmap_w1,
                     const __grid_constant__ CUtensorMap tmap_x,
                     const __grid_constant__ CUtensorMap tmap_w2,
                     const __grid_constant__ CUtensorMap tmap_h,
                     const __grid_constant__ CUtensorMap tmap_x_full,
                     const __grid_constant__ CUtensorMap tmap_h_full, const LayerArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using SM = SmemMap<NV, TROWS, F8>;
  constexpr int kSt = SM::kSt;
  using TM = TmemMap<NV>;
  SmemTail<SM::kGlobalTiles>* tail = reinterpret_cast<SmemTail<SM::kGlobalTiles>*>(smem + SM::kTail);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kKb = F8 ? 128 : kBK;   // K elements per k-block (128-byte rows either way)
  constexpr int kAtomK = NV ? 64 : 128; // K elements of one scale block (4 scales a row)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      ptx::mbar_init(&tail->full[s], 1);
      ptx::mbar_init(&tail->empty[s], 1);
    }
    ptx::mbar_init(&tail->acc_full, 1);
    ptx::mbar_init(&tail->acc_empty, 128);
    ptx::mbar_init(&tail->mma_done, 1);
    for (int r = 0; r < kRing; ++r) {
      ptx::mbar_init(&tail->ring_full[r], 1);
      // the MMA thread + 4 epilogue warps
      ptx::mbar_init(&tail->ring_empty[r], 5);
    }
    tail->abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmap_w1);
    ptx::prefetch_tmap(&tmap_x);
    ptx::prefetch_tmap(&tmap_w2);
    ptx::prefetch_tmap(&tmap_h);
    ptx::prefetch_tmap(&tmap_x_full);
    ptx::prefetch_tmap(&tmap_h_full);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&tail->tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;
  volatile int* abort_flag = &tail->abort;
  // Set-up above overlaps the previous kernel; its outputs are read only from here on.
  ptx::pdl_launch_dependents();
  if (MODE == kModeLayer && threadIdx.x == 0 && blockIdx.x < args.E * args.ph[0].m_tiles) {
    // While the token dispatch finishes, pull into L2 the gate/up slab this block
    // most likely takes first when every expert has one token tile (decode-sized
    // loads): item b = (expert b / slabs, slab b % slabs).  Only a hint.
    const PhaseArgs& P = args.ph[0];
    const int b = (int)blockIdx.x;
    const int e = b / P.m_tiles, mt = b % P.m_tiles;
    for (int kb = 0; kb < P.num_kb; ++kb)
      ptx::tma_prefetch_2d(&tmap_w1, 0, ((e * P.m_tiles + mt) * P.num_kb + kb) * kBM);
    ptx::bulk_prefetch(P.w_sf + ((size_t)(e * P.m_tiles + mt) * P.kc4) * kSFAtomBytes,
                       (uint32_t)P.kc4 * kSFAtomBytes);
  }
  ptx::pdl_wait();

  const int num_tiles = args.ws.flags[kFlagTiles];
  const int E = args.E;
  const int32_t* tile_start = SM::kGlobalTiles ? args.ws.tile_start : tail->tile_start;
  if (!SM::kGlobalTiles)
    for (int e = threadIdx.x; e <= E; e += blockDim.x) tail->tile_start[e] = args.ws.tile_start[e];
  __syncthreads();
  // Items per token tile and phase: one per weight slab.
  const int m0 = args.ph[0].m_tiles, m1 = args.ph[1].m_tiles;
  const int n0 = num_tiles * m0;
  const int total = n0 + (args.num_phases == 2 ? num_tiles * m1 : 0);
  // A tile's intermediate rows are complete once every gate/up slab has stored its
  // part (one count per slab, from whichever block computed it).
  const int slabs0 = args.ph[0].m_tiles;
  constexpr int kGrp1 = (MODE == kModeLayer && TROWS == kBN) ? kDownGroup : 0;

  if (warp == 0) {
    // ------------------------------------------------- scheduler + producer
    // Lane 0 claims items, hands them on and issues the TMA copies; with PULL the
    // whole warp also gathers the gate/up token rows of each stage (one row per
    // token, written once by the quantiser) with per-thread asynchronous copies.
    const bool leader = lane == 0;
    const uint64_t pol_once = ptx::policy_evict_first();
    const uint64_t pol_shared = ptx::policy_evict_normal();
    const uint64_t pol_t = ptx::policy_evict_last();
    int stage = 0, r = 0;
    uint32_t phase = 0, rph = 0;
    int64_t issued = 0;
    bool ok = true;
    // intermediate rows of down items under the grouped order (see kDownGroup)
    const uint64_t pol_h = (kGrp1 > 0 && kDownRowsNormal) ? pol_shared : pol_t;
    // Items are claimed one ahead so that the claim and the table reads of the
    // next item overlap the loads of the current one.
    int g = 0;
    Item it = {};
    int4 ti = make_int4(0, 0, 0, 0);
    if (leader) {
      g = atomicAdd(&args.ws.flags[kFlagSched], 1);
      if (g < total) {
        it = decode_item(g, n0, m0, m1, E, tile_start, num_tiles, kGrp1);
        ti = args.ws.tiles[it.tile];
      }
    }
    while (true) {
      int item = -1;
      if (leader) {
        item = g < total ? g : -1;
        if (!ptx::mbar_wait(&tail->ring_empty[r], rph ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
        } else {
          tail->ring[r] = make_int4(item, ti.y, ti.z | (it.mt << 8), it.tile);
          ptx::mbar_arrive(&tail->ring_full[r]);
        }
      }
      // the item, to every lane
      ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      item = __shfl_sync(kFull, item, 0);
      if (++r == kRing) {
        r = 0;
        rph ^= 1u;
      }
      if (item < 0) break;
      it.phase = __shfl_sync(kFull, it.phase, 0);
      it.tile = __shfl_sync(kFull, it.tile, 0);
      it.mt = __shfl_sync(kFull, it.mt, 0);
      it.e = __shfl_sync(kFull, it.e, 0);
      it.ntiles = __shfl_sync(kFull, it.ntiles, 0);
      ti.y = __shfl_sync(kFull, ti.y, 0);
      ti.z = __shfl_sync(kFull, ti.z, 0);
      const int g_next = leader ? atomicAdd(&args.ws.flags[kFlagSched], 1) : total;
      Item it_next = {};
      int4 ti_next = make_int4(0, 0, 0, 0);
      const PhaseArgs& P = args.ph[it.phase];
      const CUtensorMap* tw = it.phase ? &tmap_w2 : &tmap_w1;
      const CUtensorMap* tt = it.phase ? &tmap_h : &tmap_x;
      // a full tile's token rows in one box
      const CUtensorMap* tt_full = it.phase ? &tmap_h_full : &tmap_x_full;
      const uint64_t pol_tt = it.phase ? pol_h : pol_t;
      // A slab read by one token tile only is not kept; one shared by several
      // tiles of the expert stays for them.
      const uint64_t pol_w = it.ntiles > 1 ? pol_shared : pol_once;
      const int e = it.e, row0 = ti.y, n = ti.z;
      const int nb = (n + kBBoxRows - 1) / kBBoxRows;
      const int mt = it.mt;   // the item's weight slab
      const int wslab = e * P.m_tiles + mt;   // weight slab over all experts
      const uint8_t* wsf = P.w_sf + ((size_t)wslab * P.kc4) * kSFAtomBytes;
      // the tile's token scale blocks (each tile has blocks of its own)
      const uint8_t* tsf = P.t_sf + ((size_t)(row0 / SM::kBRows) * P.kc4) * kSFAtomBytes;
      // Pulled token rows: lane l gathers rows l, l+32, l+64, l+96 of the tile.
      const bool pulled = PULL && it.phase == 0;
      int tok[kBN / 32];
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i)
        tok[i] = (pulled && lane + 32 * i < n) ? args.ws.slot_token[row0 + lane + 32 * i] : -1;
      if (it.phase == 1) {
        // The down projection reads the intermediate rows that this tile's
        // gate/up items wrote with ordinary stores.
        if (leader) {
          ok = ptx::wait_counter(&args.ws.tile_done[it.tile], slabs0, abort_flag, kWaitLimitNs);
          if (ok) ptx::fence_proxy_async_global();
        }
        ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      for (int kb = 0; kb < P.num_kb; ++kb) {
        if (leader) ok = ptx::mbar_wait(&tail->empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs);
        ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;   // the stage is free for every lane
        if (!ok) break;
        const int kvalid = min(kKb, P.K - kb * kKb);
        const int atoms = kvalid / kAtomK;
        uint64_t* bar = &tail->full[stage];
        uint8_t* b_dst = smem + SM::kB + (size_t)stage * SM::kBSlot;
        if (pulled) {
          // Row i of the tile is token tok's codes [kb*128, kb*128 + kvalid/2) in the
          // 128-byte swizzle (16-byte chunk c of row i at chunk c ^ (i % 8)), and its
          // scales in the 128x4 blocks the scale copy reads.
          uint8_t* sf_dst = smem + SM::kSFB + (size_t)stage * SM::kSF;
          // Lane l copies rows l, l+32, l+64, l+96: only live rows cost anything,
          // which matters for the few-row tiles of decode-sized loads.
          const int chunks = kvalid / 32;
#pragma unroll
          for (int i = 0; i < kBN / 32; ++i) {
            const int row = lane + 32 * i;
            if (tok[i] < 0) continue;
            const uint8_t* src = args.ws.xq + (size_t)tok[i] * (args.H / 2) + (size_t)kb * kBKBytes;
            uint8_t* dst = b_dst + row * kBKBytes;
            for (int c = 0; c < chunks; ++c)
              ptx::cp_async16(dst + ((c ^ (row & 7)) << 4), src + c * 16);
          }
          // Scales: lane l, row l + 32 i, 4 bytes per 128-element block.
#pragma unroll
          for (int i = 0; i < kBN / 32; ++i) {
            const int row = lane + 32 * i;
            if (tok[i] < 0) continue;
            const uint8_t* ssrc = args.ws.xs + (size_t)tok[i] * (args.H / 32) + (size_t)kb * 8;
            for (int a = 0; a < atoms; ++a)
              ptx::cp_async4(sf_dst + a * kSFAtomBytes + (row & 31) * 16 + (row >> 5) * 4,
                             ssrc + a * 4);
          }
          ptx::cp_async_arrive(bar);
          __syncwarp();   // every lane's copies count against the stage before lane 0 arrives
        }
        if (leader) {
          // every byte the TMA lands here: the weight box and scales and, unless
          // pulled, the token rows and their scales.  A widened E2M1 box (F8) counts
          // its packed bytes only: each 16-byte chunk of it gets 8 bytes of data and
          // 8 that the copy leaves untouched.
          const uint32_t bytes =
              (F8 ? kATileBytes / 2 : kATileBytes) + atoms * kSFAtomBytes +
              (pulled ? 0u : (uint32_t)(nb * (kBBoxRows * kBKBytes) + atoms * kSFAtomBytes));
          ptx::mbar_arrive_expect_tx(bar, bytes);
          ptx::tma_load_2d(smem + SM::kA + (size_t)stage * kATileBytes, tw, 0,
                           (wslab * P.num_kb + kb) * kBM, bar, pol_w);
          ptx::bulk_load(smem + SM::kSFA + (size_t)stage * SM::kSF,
                         wsf + (size_t)kb * (kKb / kAtomK) * kSFAtomBytes, atoms * kSFAtomBytes,
                         bar, pol_w);
          if (!pulled) {
            if (nb * kBBoxRows == SM::kBRows) {
              ptx::tma_load_2d(b_dst, tt_full, kb * kBKBytes, row0, bar, pol_tt);
            } else {
              for (int j = 0; j < nb; ++j)
                ptx::tma_load_2d(b_dst + j * kBBoxRows * kBKBytes, tt, kb * kBKBytes,
                                 row0 + j * kBBoxRows, bar, pol_tt);
            }
            ptx::bulk_load(smem + SM::kSFB + (size_t)stage * SM::kSF,
                           tsf + (size_t)kb * (kKb / kAtomK) * kSFAtomBytes, atoms * kSFAtomBytes,
                           bar, pol_tt);
          }
          if (kb == 0 && g_next < total) {
            it_next = decode_item(g_next, n0, m0, m1, E, tile_start, num_tiles, kGrp1);
            ti_next = args.ws.tiles[it_next.tile];
          }
        }
        ++issued;
        if (++stage == kSt) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      g = g_next;
      it = it_next;
      ti = ti_next;
    }
    if (leader && !ok) atomicOr(&args.ws.flags[0], kErrTimeout);
    // Drain: every copy this warp issued must have landed before the block exits
    // (normally they all have, because the MMA consumed them).
    if (PULL) ptx::cp_async_wait_all();
    if (leader) {
      const int64_t first = issued > kSt ? issued - kSt : 0;
      for (int64_t i = first; i < issued; ++i) {
        const int s = (int)(i % kSt);
        const uint32_t par = (uint32_t)((i / kSt) & 1);
        int never = 0;
        ptx::mbar_wait(&tail->full[s], par, &never, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // stage 0's operand and scale descriptors; stage s adds s times a stage's bytes / 16
      const uint64_t da0 = ptx::desc_sw128(ptx::smem_addr(smem + SM::kA));
      const uint64_t db0 = ptx::desc_sw128(ptx::smem_addr(smem + SM::kB));
      const uint64_t dsa0 = ptx::desc_sf(ptx::smem_addr(smem + SM::kSFA));
      const uint64_t dsb0 = ptx::desc_sf(ptx::smem_addr(smem + SM::kSFB));
      const uint32_t sf_t0 = tmem_base + (uint32_t)kSfTmemBase;
      int stage = 0, r = 0;
      uint32_t phase = 0, rph = 0, acc_phase = 0, sfbuf = 0;
      bool ok = true;
      while (true) {
        if (!ptx::mbar_wait(&tail->ring_full[r], rph, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const int4 rec = tail->ring[r];
        ptx::mbar_arrive(&tail->ring_empty[r]);
        if (++r == kRing) {
          r = 0;
          rph ^= 1u;
        }
        const int item = rec.x;
        if (item < 0) break;
        const PhaseArgs& P = args.ph[item < n0 ? 0 : 1];
        // gate/up token rows gathered by per-thread copies (generic proxy) are read
        // by the tensor core (async proxy) after each stage's barrier
        const bool pulled = PULL && item < n0;
        const int n = rec.z & 0xFF;
        const int n_mma = (n + kBBoxRows - 1) / kBBoxRows * kBBoxRows;
        if (!ptx::mbar_wait(&tail->acc_empty, acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // Whole k-blocks take a short path: this one thread issues every
        // tensor-core instruction of the block, and the dependent latency of its own
        // work per k-block paces the stream unless that work is little more than the
        // instructions -- descriptors are stage 0's plus a constant, the two
        // instruction descriptors are set per item, copies and MMAs unrolled.
        const uint32_t id0 = ptx::idesc_mxf4(n_mma, 0), id2 = ptx::idesc_mxf4(n_mma, 2);
        const uint32_t idn = ptx::idesc_nvf4(n_mma);
        const uint32_t if8[4] = {ptx::idesc_f8f4(n_mma, 0), ptx::idesc_f8f4(n_mma, 1),
                                 ptx::idesc_f8f4(n_mma, 2), ptx::idesc_f8f4(n_mma, 3)};
        const int whole_kb = P.K / kKb;
        for (int kb = 0; kb < P.num_kb; ++kb) {
          if (!ptx::mbar_wait(&tail->full[stage], phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          if (pulled) ptx::fence_proxy_async_smem();
          if (kb < whole_kb) {
            const uint32_t sfa_t = sf_t0 + (sfbuf ? (uint32_t)TM::kSfCols : 0u);
            const uint32_t sfb_t = sfa_t + TM::kSfCols / 2;
            const uint64_t dsa = dsa0 + (uint64_t)(stage * (int)(SM::kSF >> 4));
            const uint64_t dsb = dsb0 + (uint64_t)(stage * (int)(SM::kSF >> 4));
            const uint64_t da = da0 + (uint64_t)(stage * (kATileBytes >> 4));
            const uint64_t db = db0 + (uint64_t)(stage * (int)(SM::kBSlot >> 4));
            const uint32_t acc0 = kb != 0 ? 1u : 0u;
            // Four MMAs a k-block, each 32 bytes further along every operand row (+2
            // in a descriptor); scale blocks 512 bytes (+32) apart.
            if constexpr (NV) {
              // four 64-element scale blocks, MMA step s takes block s whole
#pragma unroll
              for (int a = 0; a < 4; ++a) {
                ptx::tc_cp_sf(sfa_t + a * 4, dsa + 32 * a);
                ptx::tc_cp_sf(sfb_t + a * 4, dsb + 32 * a);
              }
#pragma unroll
              for (int s2 = 0; s2 < 4; ++s2)
                ptx::tc_mma_nvf4(tmem_base, da + 2 * s2, db + 2 * s2, idn, sfa_t + s2 * 4,
                                 sfb_t + s2 * 4, s2 == 0 ? acc0 : 1u);
            } else if constexpr (F8) {
              // one scale block: MMA step s takes scale byte s of each row
              ptx::tc_cp_sf(sfa_t, dsa);
              ptx::tc_cp_sf(sfb_t, dsb);
              ptx::tc_mma_f8f4(tmem_base, da, db, if8[0], sfa_t, sfb_t, acc0);
              ptx::tc_mma_f8f4(tmem_base, da + 2, db + 2, if8[1], sfa_t, sfb_t, 1u);
              ptx::tc_mma_f8f4(tmem_base, da + 4, db + 4, if8[2], sfa_t, sfb_t, 1u);
              ptx::tc_mma_f8f4(tmem_base, da + 6, db + 6, if8[3], sfa_t, sfb_t, 1u);
            } else {
              // two 128-element scale blocks, steps 0-1 and 2-3 take byte pairs 0/2
              ptx::tc_cp_sf(sfa_t, dsa);
              ptx::tc_cp_sf(sfb_t, dsb);
              ptx::tc_cp_sf(sfa_t + 4, dsa + 32);
              ptx::tc_cp_sf(sfb_t + 4, dsb + 32);
              ptx::tc_mma_mxf4(tmem_base, da, db, id0, sfa_t, sfb_t, acc0);
              ptx::tc_mma_mxf4(tmem_base, da + 2, db + 2, id2, sfa_t, sfb_t, 1u);
              ptx::tc_mma_mxf4(tmem_base, da + 4, db + 4, id0, sfa_t + 4, sfb_t + 4, 1u);
              ptx::tc_mma_mxf4(tmem_base, da + 6, db + 6, id2, sfa_t + 4, sfb_t + 4, 1u);
            }
            ptx::tc_commit(&tail->empty[stage]);
            sfbuf ^= 1u;
            if (++stage == kSt) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          const int kvalid = min(kKb, P.K - kb * kKb);
          const int atoms = kvalid / kAtomK;
          const uint32_t sfa_t = tmem_base + (uint32_t)(kSfTmemBase + sfbuf * TM::kSfCols);
          const uint32_t sfb_t = sfa_t + TM::kSfCols / 2;
          const uint32_t sa = ptx::smem_addr(smem + SM::kSFA + (size_t)stage * SM::kSF);
          const uint32_t sb = ptx::smem_addr(smem + SM::kSFB + (size_t)stage * SM::kSF);
          for (int a = 0; a < atoms; ++a) {
            ptx::tc_cp_sf(sfa_t + a * 4, ptx::desc_sf(sa + a * kSFAtomBytes));
            ptx::tc_cp_sf(sfb_t + a * 4, ptx::desc_sf(sb + a * kSFAtomBytes));
          }
          const uint32_t a_base = ptx::smem_addr(smem + SM::kA + (size_t)stage * kATileBytes);
          const uint32_t b_base = ptx::smem_addr(smem + SM::kB + (size_t)stage * SM::kBSlot);
          // 32 bytes of K per instruction: 64 packed E2M1 elements, or 32 one-byte ones
          const int steps = kvalid / (F8 ? 32 : 64);
          for (int s = 0; s < steps; ++s) {
            if (NV) {
              // step s (64 elements) takes scale block s whole: four E4M3 scales a row
              ptx::tc_mma_nvf4(tmem_base, ptx::desc_sw128(a_base + s * 32),
                               ptx::desc_sw128(b_base + s * 32), ptx::idesc_nvf4(n_mma),
                               sfa_t + s * 4, sfb_t + s * 4, (kb | s) != 0 ? 1u : 0u);
            } else if (F8) {
              // one 128-element k-block: one scale atom, scale byte s of each row
              ptx::tc_mma_f8f4(tmem_base, ptx::desc_sw128(a_base + s * 32),
                               ptx::desc_sw128(b_base + s * 32), ptx::idesc_f8f4(n_mma, s), sfa_t,
                               sfb_t, (kb | s) != 0 ? 1u : 0u);
            } else {
              const uint32_t idesc = ptx::idesc_mxf4(n_mma, (s & 1) * 2);
              ptx::tc_mma_mxf4(tmem_base, ptx::desc_sw128(a_base + s * 32),
                               ptx::desc_sw128(b_base + s * 32), idesc, sfa_t + (s >> 1) * 4,
                               sfb_t + (s >> 1) * 4, (kb | s) != 0 ? 1u : 0u);
            }
          }
          ptx::tc_commit(&tail->empty[stage]);
          sfbuf ^= 1u;
          if (++stage == kSt) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit(&tail->acc_full);
        acc_phase ^= 1u;
      }
      if (!ok) atomicOr(&args.ws.flags[0], kErrTimeout);
      // Whatever happened, wait until every MMA issued here has finished before
      // the block may release its tensor memory.
      ptx::tc_commit(&tail->mma_done);
      int never = 0;
      ptx::mbar_wait(&tail->mma_done, 0, &never, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int ep_tid = threadIdx.x - 64;
    const uint64_t pol_acc = ptx::policy_evict_last();
    int r = 0, xb = 0;
    uint32_t rph = 0, acc_phase = 0;
    while (true) {
      if (!ptx::mbar_wait(&tail->ring_full[r], rph, abort_flag, kWaitLimitNs)) {
        if (ep_tid == 0) atomicOr(&args.ws.flags[0], kErrTimeout);
        break;
      }
      const int4 rec = tail->ring[r];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tail->ring_empty[r]);
      if (++r == kRing) {
        r = 0;
        rph ^= 1u;
      }
      const int item = rec.x;
      if (item < 0) break;
      const int item_phase = item < n0 ? 0 : 1;
      const int row0 = rec.y, n = rec.z & 0xFF, mt = rec.z >> 8, item_tile = rec.w;
      // Row metadata of a down item, read while the MMAs run: lane l holds rows
      // l, l+32, l+64, l+96 of the tile.
      int tok_r[kBN / 32];
      float w_r[kBN / 32];
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i) {
        tok_r[i] = 0;
        w_r[i] = 0.f;
        if (MODE == kModeLayer && item_phase == 1 && lane + 32 * i < n) {
          tok_r[i] = args.ws.slot_token[row0 + lane + 32 * i];
          w_r[i] = args.ws.slot_weight[row0 + lane + 32 * i];
        }
      }
      if (!ptx::mbar_wait(&tail->acc_full, acc_phase, abort_flag, kWaitLimitNs)) {
        if (ep_tid == 0) atomicOr(&args.ws.flags[0], kErrTimeout);
        break;
      }
      acc_phase ^= 1u;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16);
      const uint32_t tspare = taddr + (uint32_t)TM::kSpareCol;
      // The math of one 16-column chunk, wherever its values were read from.
      auto chunk = [&](const int ci, const float(&v)[kEpiCols]) {
        const int c0 = ci * kEpiCols;
        const int ncol = min(kEpiCols, n - c0);
        if (MODE == kModeRaw) {
          const int m = mt * kBM + q * 32 + lane;
          const int col = gate_up_source_row_for(m, args.I, F8 ? 1 : 0);
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) {
            if (j < ncol) {
              const int a = args.ws.slot_assign[row0 + c0 + j];
              args.gate_up_debug[(size_t)a * 2 * args.I + col] = v[j];
            }
          }
        } else if (item_phase == 0) {
          // Rows of this warp: chunk c of 32 interleaved gate/up rows =
          // [gate even 8 | up even 8 | gate odd 8 | up odd 8] of features c*16..c*16+15
          // (F8, gran=8: [gate 8 | up 8 | gate next 8 | up next 8] of the same features).
          // Either way lane l and lane l^8 hold the gate and up of one feature.
          // Columns go in pairs: gate lanes (0-7, 16-23) compute column 2p from their
          // gate and the up of lane+8, up lanes (8-15, 24-31) column 2p+1 from their up
          // and the gate of lane-8 -- one exchange, and no lane idles.
          const bool up_lane = (lane & 8) != 0;
          float hv[kEpiCols / 2], am[kEpiCols / 2];
#pragma unroll
          for (int p = 0; p < kEpiCols / 2; ++p) {
            const float x = __shfl_xor_sync(kFull, up_lane ? v[2 * p] : v[2 * p + 1], 8);
            const float h = up_lane ? silu_times(x, v[2 * p + 1]) : silu_times(v[2 * p], x);
            hv[p] = h;
            am[p] = fabsf(h);
          }
          // Max |h| of each of the lane's 8 columns over the 16 lanes holding that
          // column (lane bits 0, 1, 2 and 4), as a transposing butterfly: after the
          // steps over bits 0, 1 and 2 each lane keeps one column, p = 4 b0 + 2 b1 + b2
          // (8 shuffles for the 8 columns instead of 32).
          {
            const bool b0 = (lane & 1) != 0, b1 = (lane & 2) != 0, b2 = (lane & 4) != 0;
            float a4[4], a2[2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float send = b0 ? am[i] : am[4 + i];
              const float keep = b0 ? am[4 + i] : am[i];
              a4[i] = fmaxf(keep, __shfl_xor_sync(kFull, send, 1));
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float send = b1 ? a4[i] : a4[2 + i];
              const float keep = b1 ? a4[2 + i] : a4[i];
              a2[i] = fmaxf(keep, __shfl_xor_sync(kFull, send, 2));
            }
            const float send = b2 ? a2[0] : a2[1];
            const float keep = b2 ? a2[1] : a2[0];
            float a1 = fmaxf(keep, __shfl_xor_sync(kFull, send, 4));
            a1 = fmaxf(a1, __shfl_xor_sync(kFull, a1, 16));
            if ((lane & 16) == 0) {
              const int pm = (b0 ? 4 : 0) + (b1 ? 2 : 0) + (b2 ? 1 : 0);
              tail->xchg[xb][q][2 * pm + (up_lane ? 1 : 0)] = a1;
            }
          }
          ptx::named_bar_sync(1, 128);
          const int i_kc4 = args.I / kAtomK;   // scale blocks of an intermediate row
          const size_t hrow_bytes = F8 ? (size_t)args.I : (size_t)args.I / 2;
          // The scale of each column is worked out once, by the lane that holds the
          // column after the butterfly (column 2 pm + up, pm as above), and handed to the
          // lanes that need it with one shuffle per column: that lane's scale byte goes
          // to the staging area directly.
          const int pm = ((lane & 1) << 2) | (lane & 2) | ((lane >> 2) & 1);
          const int cm = 2 * pm + (up_lane ? 1 : 0);
          // 32-feature group = this warp's 16 features + the partner warp's 16 (NVFP4:
          // the 16-feature group is this warp's alone)
          const float am_m = NV ? tail->xchg[xb][q][cm]
                                : fmaxf(tail->xchg[xb][q][cm], tail->xchg[xb][q ^ 1][cm]);
          float mul_m;   // MX: 2^-e; NVFP4: the E4M3 scale's value
          uint32_t sb_m;
          if (NV) {
            sb_m = ptx::nvfp4_scale_byte(am_m);   // E4M3 of amax/6
            mul_m = ptx::ue4m3_value(sb_m);
          } else {
            const int e = F8 ? ptx::mxfp8_exponent(am_m) : ptx::mx_scale_exponent(am_m);
            sb_m = (uint32_t)(e + 127);
            mul_m = ptx::pow2_neg(e);
          }
          if ((lane & 16) == 0) {
            if (NV)
              tail->sstage[xb][cm][q] = (uint8_t)sb_m;
            else if ((q & 1) == 0)
              tail->sstage[xb][cm][q >> 1] = (uint8_t)sb_m;
          }
          uint32_t code[kEpiCols / 2];
#pragma unroll
          for (int p = 0; p < kEpiCols / 2; ++p) {
            // column 2p + up is held by the lane with pm == p and the same up bit
            const int src = ((p >> 2) & 1) | (((p >> 1) & 1) << 1) | ((p & 1) << 2) | (lane & 8);
            const float m = __shfl_sync(kFull, mul_m, src);
            const float qv = NV ? (m > 0.f ? __fdiv_rn(hv[p], m) : copysignf(0.f, hv[p]))
                                : hv[p] * m;
            if (F8) {
              code[p] = ptx::e4m3x2(qv, 0.f) & 0xFFu;
            } else {
              const float qodd = __shfl_down_sync(kFull, qv, 16);
              code[p] = ptx::e2m1x2(qv, qodd);
            }
          }
          if (F8) {
            // one E4M3 byte per lane and column: feature 16q + (l & 7) + 8 * (l >> 4)
            // of the item's 64 (lanes 0-7 and 16-23 column 2p, lanes 8-15 and 24-31
            // column 2p+1)
            const int f = q * 16 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
            for (int p = 0; p < kEpiCols / 2; ++p) {
              const int jc = 2 * p + (up_lane ? 1 : 0);
              tail->hstage[xb][jc][f] = (uint8_t)code[p];
            }
          } else if (lane < 16) {
            // lanes 0-7 (column 2p) and 8-15 (column 2p+1) each hold one of the 8
            // bytes of features c*16..c*16+15 of their column (c = 4*slab + q)
#pragma unroll
            for (int p = 0; p < kEpiCols / 2; ++p) {
              const int jc = 2 * p + (up_lane ? 1 : 0);
              tail->hstage[xb][jc][q * 8 + (lane & 7)] = (uint8_t)code[p];
            }
          }
          ptx::named_bar_sync(1, 128);
          // The chunk's rows, whole: warp q stores columns 4q..4q+3, 16 code bytes a
          // lane (two lanes fill a row's 32-byte sector; F8: four lanes its 64 bytes)
          // and the two scale bytes.
          if (F8) {
            if (lane < 16) {
              const int jc = q * 4 + (lane >> 2);
              if (jc < ncol) {
                const size_t row = (size_t)row0 + c0 + jc;
                const uint4 cv =
                    *reinterpret_cast<const uint4*>(&tail->hstage[xb][jc][(lane & 3) * 16]);
                *reinterpret_cast<uint4*>(args.ws.hb + row * hrow_bytes + (size_t)mt * 64 +
                                          (lane & 3) * 16) = cv;
              }
            } else if (lane < 20) {
              const int jc = q * 4 + (lane - 16);
              if (jc < ncol) {
                const size_t row = (size_t)row0 + c0 + jc;
                const uint16_t sv = *reinterpret_cast<const uint16_t*>(&tail->sstage[xb][jc][0]);
                *reinterpret_cast<uint16_t*>(args.ws.hsf +
                                             sf_tile_offset(row, mt * 2, i_kc4, TROWS)) = sv;
              }
            }
          } else if (lane < 8) {
            const int jc = q * 4 + (lane >> 1);
            if (jc < ncol) {
              const size_t row = (size_t)row0 + c0 + jc;
              const uint4 cv = *reinterpret_cast<const uint4*>(&tail->hstage[xb][jc][(lane & 1) * 16]);
              *reinterpret_cast<uint4*>(args.ws.hb + row * hrow_bytes + (size_t)mt * 32 +
                                        (lane & 1) * 16) = cv;
            }
          } else if (lane < 12) {
            const int jc = q * 4 + (lane - 8);
            if (jc < ncol) {
              const size_t row = (size_t)row0 + c0 + jc;
              if (NV) {   // the item's four scale bytes: one 32-bit word of a scale block
                const uint32_t sv = *reinterpret_cast<const uint32_t*>(&tail->sstage[xb][jc][0]);
                *reinterpret_cast<uint32_t*>(args.ws.hsf +
                                             sf_tile_offset(row, mt * 4, i_kc4, TROWS)) = sv;
              } else {
                const uint16_t sv = *reinterpret_cast<const uint16_t*>(&tail->sstage[xb][jc][0]);
                *reinterpret_cast<uint16_t*>(args.ws.hsf +
                                             sf_tile_offset(row, mt * 2, i_kc4, TROWS)) = sv;
              }
            }
          }
          xb ^= 1;
        } else {
          // Down projection: this warp holds output features mt*128 + q*32 + lane of
          // up to 16 token columns; add them, weighted, into the fp32 accumulator.
          // Column c0+j's row metadata sits in lane (c0+j) % 32, register (c0+j) / 32.
          // Every column's token and weight are fetched before the first reduction, so
          // that the 32 shuffles overlap one another instead of each waiting behind the
          // reduction before it.
          // (the chunk index is a loop variable: select, not index, the register)
          const int hi = ci >> 1;
          const int my_tok = hi == 0 ? tok_r[0] : hi == 1 ? tok_r[1] : hi == 2 ? tok_r[2] : tok_r[3];
          const float my_w = hi == 0 ? w_r[0] : hi == 1 ? w_r[1] : hi == 2 ? w_r[2] : w_r[3];
          int tok_j[kEpiCols];
          float w_j[kEpiCols];
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) {
            const int src = (ci & 1) * kEpiCols + j;
            tok_j[j] = __shfl_sync(kFull, my_tok, src);
            w_j[j] = __shfl_sync(kFull, my_w, src);
          }
          float* const col0 = args.ws.acc + (size_t)mt * kBM + q * 32 + lane;
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) {
            if (j < ncol) {
              float* dst = col0 + (size_t)tok_j[j] * args.H;
              if constexpr (kGrp1 > 0 && kAccKeep)
                ptx::red_add_f32(dst, w_j[j] * v[j], pol_acc);
              else
                atomicAdd(dst, w_j[j] * v[j]);
            }
          }
        }
      };
      const int nch = (n + kEpiCols - 1) / kEpiCols;
      constexpr int kSpareChunks = TM::kSpareChunks;   // 6, or 4 for NVFP4
      const int ncopy = min(nch, kSpareChunks);
      // 1. The first ncopy chunks (up to 96 columns, 64 for NVFP4) into this block's
      //    spare tensor memory, two loads in flight.
#pragma unroll
      for (int ci = 0; ci < kSpareChunks; ci += 2) {
        if (ci < ncopy) {
          uint32_t r0[kEpiCols], r1[kEpiCols];
          const bool two = ci + 1 < ncopy;
          ptx::tmem_ld16_issue(taddr + (uint32_t)(ci * kEpiCols), r0);
          if (two) ptx::tmem_ld16_issue(taddr + (uint32_t)((ci + 1) * kEpiCols), r1);
          ptx::tmem_wait_ld(r0);
          if (two) ptx::tmem_wait_ld(r1);
          ptx::tmem_st16(tspare + (uint32_t)(ci * kEpiCols), r0);
          if (two) ptx::tmem_st16(tspare + (uint32_t)((ci + 1) * kEpiCols), r1);
        }
      }
      // 2. The chunks past the spare area straight from the accumulator: any before
      //    the last two one at a time (NVFP4's smaller spare area), then the last two
      //    both loaded before any math.  Once every accumulator load is done it goes
      //    back to the MMA issuer, so the next item's MMAs run during this item's math.
      constexpr int kLastTwo = kBN / kEpiCols - 2;
      static_assert(kSpareChunks <= kLastTwo, "tensor memory layout");
      bool released = false;
#pragma unroll
      for (int ci = kSpareChunks; ci < kLastTwo; ++ci) {
        if (ci < nch) {
          uint32_t r[kEpiCols];
          ptx::tmem_ld16_issue(taddr + (uint32_t)(ci * kEpiCols), r);
          ptx::tmem_wait_ld(r);
          if (ci + 1 >= nch) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(&tail->acc_empty);
            released = true;
          }
          float v[kEpiCols];
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) v[j] = __uint_as_float(r[j]);
          chunk(ci, v);
        }
      }
      uint32_t rd[2][kEpiCols];
#pragma unroll
      for (int d = 0; d < 2; ++d)
        if (kLastTwo + d < nch)
          ptx::tmem_ld16_issue(taddr + (uint32_t)((kLastTwo + d) * kEpiCols), rd[d]);
#pragma unroll
      for (int d = 0; d < 2; ++d)
        if (kLastTwo + d < nch) ptx::tmem_wait_ld(rd[d]);
      if (!released) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tail->acc_empty);
      }
#pragma unroll
      for (int d = 0; d < 2; ++d) {
        if (kLastTwo + d < nch) {
          float v[kEpiCols];
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) v[j] = __uint_as_float(rd[d][j]);
          chunk(kLastTwo + d, v);
        }
      }
      ptx::tmem_wait_st();
      // 3. The copied chunks; the load of chunk ci+1 runs during the math of ci.  A
      //    rolled loop over pairs of chunks: every unrolled copy of the chunk math
      //    costs instruction-cache room that the epilogue warps then wait on.
      uint32_t ra[kEpiCols], rb[kEpiCols];
      if (ncopy > 0) {
        ptx::tmem_ld16_issue(tspare, ra);
        ptx::tmem_wait_ld(ra);
      }
#pragma unroll 1
      for (int ci = 0; ci < ncopy; ci += 2) {
        const bool m1 = ci + 1 < ncopy, m2 = ci + 2 < ncopy;
        if (m1) ptx::tmem_ld16_issue(tspare + (uint32_t)((ci + 1) * kEpiCols), rb);
        {
          float v[kEpiCols];
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) v[j] = __uint_as_float(ra[j]);
          chunk(ci, v);
        }
        if (m1) ptx::tmem_wait_ld(rb);
        if (m2) ptx::tmem_ld16_issue(tspare + (uint32_t)((ci + 2) * kEpiCols), ra);
        if (m1) {
          float v[kEpiCols];
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) v[j] = __uint_as_float(rb[j]);
          chunk(ci + 1, v);
        }
        if (m2) ptx::tmem_wait_ld(ra);
      }
      if (MODE == kModeLayer && item_phase == 0) {
        // Publish: this item's intermediate rows (and scales) are written.
        // The epilogue threads' stores are ordered before the barrier at block scope;
        // one thread's GPU-scope fence after it then releases them all (fences are
        // cumulative), instead of every thread waiting out a fence of its own.
        ptx::named_bar_sync(2, 128);
        if (ep_tid == 0) {
          __threadfence();
          ptx::fence_proxy_async_global();
          atomicAdd(&args.ws.tile_done[item_tile], 1);
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0) {
    // The last block out resets the scheduler and tile counters for the next call.
    __threadfence();
    if (atomicAdd(&args.ws.flags[kFlagExit], 1) == (int)gridDim.x - 1) {
      args.ws.flags[kFlagSched] = 0;
      args.ws.flags[kFlagExit] = 0;
      for (int t = 0; t < num_tiles; ++t) args.ws.tile_done[t] = 0;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps through the driver entry point (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Row-major uint8 matrix [rows, row_bytes] read in boxes of 128 bytes x box_rows,
// 128-byte swizzle.
cudaError_t make_tmap(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
                      uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// kb_elems: K elements per k-block (256 for packed E2M1 tokens, 128 for E4M3).
// Packed E2M1 matrix [rows, K elements] (K/2 bytes a row), read in boxes of 128
// elements x 128 rows that land one element per byte: each 16 elements' 8 packed
// bytes followed by 8 unused bytes (CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B), the
// operand layout of kind::mxf8f6f4 for E2M1; 128-byte swizzle, 16 KiB a box.
cudaError_t make_tmap_e2m1_wide(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K / 2};
  const cuuint32_t box[2] = {128, kBM};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base),
                         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// atom_k: K elements of one 128x4 scale block (128, or 64 for NVFP4's scale per 16).
PhaseArgs phase_args(const uint8_t* w_sf, const uint8_t* t_sf, int rows_per_expert, int K,
                     int kb_elems, int atom_k) {
  PhaseArgs p;
  p.w_sf = w_sf;
  p.t_sf = t_sf;
  p.rows_per_expert = rows_per_expert;
  p.K = K;
  p.m_tiles = rows_per_expert / kBM;
  p.num_kb = (K + kb_elems - 1) / kb_elems;
  p.kc4 = K / atom_k;
  return p;
}

template <int MODE, bool PULL, bool F8, bool NV, int TROWS>
cudaError_t launch_mode(const LayerLaunch& g, const CUtensorMap* maps, const LayerArgs& a,
                        cudaStream_t st) {
  constexpr size_t kSmemBytes = SmemMap<NV, TROWS, F8>::kBytes;
  static int grid = 0;   // per instantiation, for the device of the first launch
  if (grid == 0) {
    cudaError_t err = cudaFuncSetAttribute(moe_layer_kernel<MODE, PULL, F8, NV, TROWS>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    // two blocks on each SM (the work queue needs no particular number of
    // resident blocks)
    grid = kBlocksPerSM * g.num_sms;
  }
  return launch_pdl(moe_layer_kernel<MODE, PULL, F8, NV, TROWS>, dim3(grid), dim3(kThreads),
                    kSmemBytes, st,
                    maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], a);
}

// The format's instantiation for tiles of TROWS rows.
template <int TROWS>
cudaError_t launch_fmt(const LayerLaunch& g, const CUtensorMap* maps, const LayerArgs& a,
                       cudaStream_t st, bool layer, bool f8, bool nv) {
  if (f8)
    return layer ? launch_mode<kModeLayer, false, true, false, TROWS>(g, maps, a, st)
                 : launch_mode<kModeRaw, false, true, false, TROWS>(g, maps, a, st);
  if (nv)
    return layer ? launch_mode<kModeLayer, false, false, true, TROWS>(g, maps, a, st)
                 : launch_mode<kModeRaw, false, false, true, TROWS>(g, maps, a, st);
  return layer ? launch_mode<kModeLayer, false, false, false, TROWS>(g, maps, a, st)
               : launch_mode<kModeRaw, false, false, false, TROWS>(g, maps, a, st);
}

}  // namespace

cudaError_t launch_layer(const LayerLaunch& g, cudaStream_t st) {
  const Shape& s = g.shape;
  const bool f8 = s.f8 != 0, nv = s.nv != 0;
  if ((f8 || nv) && g.pull) return cudaErrorNotSupported;   // pull: MXFP4 tokens only
  // Activation rows: packed E2M1 (K/2 bytes) or E4M3 (K bytes).
  const uint64_t xrow = f8 ? (uint64_t)s.H : (uint64_t)s.H / 2;
  const uint64_t hrow = f8 ? (uint64_t)s.I : (uint64_t)s.I / 2;
  // Full token tiles come in one box of all their rows (128, 64 or 32).
  const int trows = g.pull ? kBN : g.tile_rows;
  if (trows != kBN && trows != kBNMedium && trows != kBNNarrow) return cudaErrorInvalidValue;
  const uint32_t full_rows = (uint32_t)trows;
  // Weight codes are in k-block tiles: a map row is one slab row's k-block, and the
  // 128 rows of slab w's k-block kb are map rows (w * num_kb + kb) * 128 onwards.
  const uint64_t w1_rows = (uint64_t)s.E * 2 * s.I * weight_num_kb(s, s.H);
  const uint64_t w2_rows = (uint64_t)s.E * s.H * weight_num_kb(s, s.I);
  // TMA row coordinates are 32-bit signed (W1 codes above 256 GiB would overflow them)
  if (w1_rows > 0x7FFFFFFFull || w2_rows > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  CUtensorMap maps[6];
  cudaError_t err;
  if ((err = make_tmap(&maps[4], g.ws.xb, xrow, (uint64_t)g.R_cap, full_rows)) ||
      (err = make_tmap(&maps[5], g.ws.hb, hrow, (uint64_t)g.R_cap, full_rows)) ||
      (err = make_tmap(&maps[1], g.ws.xb, xrow, (uint64_t)g.R_cap, kBBoxRows)) ||
      (err = make_tmap(&maps[3], g.ws.hb, hrow, (uint64_t)g.R_cap, kBBoxRows)))
    return err;
  if (f8) {
    // weights widened from packed E2M1 to one element per byte as they land
    if ((err = make_tmap_e2m1_wide(&maps[0], g.w1_codes, 2 * (uint64_t)weight_kb_bytes(s), w1_rows)) ||
        (err = make_tmap_e2m1_wide(&maps[2], g.w2_codes, 2 * (uint64_t)weight_kb_bytes(s), w2_rows)))
      return err;
  } else if ((err = make_tmap(&maps[0], g.w1_codes, kBKBytes, w1_rows, kBM)) ||
             (err = make_tmap(&maps[2], g.w2_codes, kBKBytes, w2_rows, kBM))) {
    return err;
  }
  LayerArgs a;
  const int kb_elems = f8 ? 128 : kBK;
  const int atom_k = nv ? 64 : 128;
  a.ph[0] = phase_args(g.w1_sf, g.ws.xsf, 2 * s.I, s.H, kb_elems, atom_k);
  a.ph[1] = phase_args(g.w2_sf, g.ws.hsf, s.H, s.I, kb_elems, atom_k);
  a.num_phases = g.num_phases;
  a.H = s.H;
  a.I = s.I;
  a.T = g.T;
  a.E = s.E;
  a.ws = g.ws;
  a.gate_up_debug = g.gate_up_debug;
  const bool layer = g.num_phases == 2;
  if (g.pull)
    return layer ? launch_mode<kModeLayer, true, false, false, kBN>(g, maps, a, st)
                 : launch_mode<kModeRaw, true, false, false, kBN>(g, maps, a, st);
  if (trows == kBNNarrow) return launch_fmt<kBNNarrow>(g, maps, a, st, layer, f8, nv);
  if (trows == kBNMedium) return launch_fmt<kBNMedium>(g, maps, a, st, layer, f8, nv);
  return launch_fmt<kBN>(g, maps, a, st, layer, f8, nv);
}

}  // namespace mxmoe
