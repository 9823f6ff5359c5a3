// The expert layer on SM pairs, for loads with many tokens per expert (sm_103a,
// tcgen05 cta_group::2 + TMEM + TMA), W4A4 MXFP4 only:
//   phase 0  grouped gate/up GEMM -> SwiGLU -> MXFP4 requantisation of h
//   phase 1  grouped down GEMM -> top-k weighted combine into the fp32 accumulator
// plus the raw mode of the gate/up GEMM (fp32 accumulators out, no SwiGLU).
//
// Pages: "[deepseek-v4] Bump sgl-deep-gemm for packed FP4xFP4 mega-MoE (W4A4)",
// Appendix B (the fused layer kernel, whose Compute SOL is the second roof beside its
// Memory SOL once the token count grows); prhub digest of SGLang PR #37279
// (activation "swiglu", the gran=16 interleave keeping each SwiGLU pair in one
// 32-row chunk).
//
// Why pairs.  At large loads the single-block kernel (gemm.cu) stages one 128-row
// weight slab and one 128-row token tile per k-block for 2*128*128*256 FLOPs, and its
// operand stream from L2 is bound by the bytes each SM can hold in flight.  Here a
// 2-CTA cluster on two SMs issues one M=256 MMA over both CTAs' shared memory: each
// CTA stages its own 128-row weight slab (one of the item's two) and half of a
// 192-row token tile, and receives 128 x 192 accumulators -- 1.6 times the FLOPs per
// staged byte, with no multicast.  Two 192-column accumulators fit one SM's tensor
// memory with the scale registers, so an item's MMAs never wait for the previous
// item's epilogue to read its accumulator.
// Measured on GB300 it is slower than the single-block kernel (T=16384: 2.25 against
// 1.64 ms): the staged bytes turned out not to bind, the MMA issuer does.  One thread
// issues every tensor-core instruction of a pair -- a k-block's copies, MMAs and
// commits plus the stage round trip, ~900 cycles whatever the MMA's N -- for two SMs,
// where the single-block kernel has two issuers on every SM.  So the layer uses this
// kernel only when asked (MOE_TILES_PAIR).
//
// Items are (token tile <= 192 rows, pair of 128-row weight slabs), first every
// gate/up item, then every down item, each phase expert by expert, slab pair by slab
// pair, then by the expert's token tiles.  Cluster c takes items c, c + C, c + 2C, ...
// (C clusters, all resident), so both CTAs of a pair know the sequence without
// talking; every gate/up item of a tile precedes its down items in every cluster's
// sequence, so a down item's bounded wait for its tile's intermediate rows ends.
// Token tiles start at whole 128-row scale blocks (kPairStride-row spans, see
// tile_row_of_rank), so a tile's token scales are one or two whole blocks.
//
// Roles (320 threads, one CTA per SM, one pair per two SMs):
//   warp 0      lane 0: items into the CTA's ring; TMA loads of this CTA's weight slab,
//               its half of the token rows, the slab's scale blocks and the whole
//               tile's token scale blocks, all completing on the LEADER's stage
//               barrier (TMA .cta_group::2).
//   warp 1      allocates tensor memory in both CTAs (cta_group::2); on the leader,
//               lane 0 issues the scale copies and MMAs for the pair and commits them
//               to the stage, accumulator and exit barriers of both CTAs.
//   warps 2-9   epilogue: warp w reads lane quarter w % 4 of its CTA's accumulator,
//               the 16-column chunks c with c % 2 == (w - 2) / 4.
// Every wait is bounded (kWaitLimitNs); a timeout sets the workspace error flag and
// each role leaves its loop; both CTAs meet at a cluster barrier before the tensor
// memory is freed.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mxmoe {
namespace {

constexpr int kStages = 7;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kTmemCols = 512;
constexpr int kAccCols = kBNPair;                 // 128 lanes x up to 192 fp32 columns
constexpr int kAccBufs = 2;
// Scale registers after the two accumulators, two buffers: A (this CTA's 128 rows) 4
// columns per 128-element scale block, B (up to 192 token rows, two 128-row blocks) 8
// columns per scale block (block b of rows at +4b).
constexpr int kSfaCols = 8;
constexpr int kSfCols = kSfaCols + 16;
constexpr int kSfBase = kAccBufs * kAccCols;
static_assert(kSfBase + 2 * kSfCols <= kTmemCols, "tensor memory layout");
constexpr int kEpiCols = 16;
constexpr int kMaxChunks = kBNPair / kEpiCols;    // 12 column chunks an item
constexpr int kBoxRows = 16;                      // token rows of a partial-tile TMA box
constexpr int kHalfRows = kBNPair / 2;            // token rows a CTA stages (full tile)
constexpr int kBSlot = kHalfRows * kBKBytes;      // 12 KiB
constexpr int kRing = 8;
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kSfaBytes = 2 * kSFAtomBytes;       // one k-block of one 128-row slab
constexpr int kSfbBytes = 2 * kSfaBytes;          // one k-block of two 128-row blocks

enum PairMode { kModeLayer = 0, kModeRaw = 1 };

// Shared memory: kStages x (weight box, token half-tile, weight scales, token
// scales), then the tail.
constexpr size_t kSmA = 0;
constexpr size_t kSmB = kSmA + (size_t)kStages * kATileBytes;
constexpr size_t kSmSfa = kSmB + (size_t)kStages * kBSlot;
constexpr size_t kSmSfb = kSmSfa + (size_t)kStages * kSfaBytes;
constexpr size_t kSmTail = kSmSfb + (size_t)kStages * kSfbBytes;

struct __align__(16) PairTail {
  uint64_t full[kStages];    // leader: both CTAs' loads of a stage landed
  uint64_t empty[kStages];   // each CTA: the pair's MMAs are done with its stage
  uint64_t acc_full[kAccBufs];    // each CTA: the item's accumulator is complete
  uint64_t acc_empty[kAccBufs];   // leader: all 16 epilogue warps have read it
  uint64_t mma_done;         // leader: every MMA it issued has finished
  uint64_t ring_full[kRing];
  uint64_t ring_empty[kRing];
  int4 ring[kRing];          // (item, first row, rows | slab pair << 16, tile); item -1: stop
  uint32_t tmem_base;
  int abort;
  float xchg[2][2][4][kEpiCols];                 // [half][buffer][quarter][column]
  alignas(16) uint8_t hstage[2][2][kEpiCols][32];
  alignas(4) uint8_t sstage[2][2][kEpiCols][2];
  int32_t tile_start[1025];  // first tile of each expert (E <= 1024), see decode_pair_item
};
constexpr size_t kSmemBytes = kSmTail + sizeof(PairTail) + 1024;   // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");

struct PairPhase {
  int m_pairs;   // slab pairs per expert: rows_per_expert / 256
  int K;         // reduction length: H (gate/up) or I (down)
  int num_kb;    // k-blocks of 256 elements (the last may be 128 wide)
  int kc4;       // 128x4 scale blocks per 128-row group: K / 128
};

struct PairArgs {
  PairPhase ph[2];
  int num_phases;
  int H, I, E;
  WsPtrs ws;
  float* gate_up_debug;
};

struct PairItem {
  int phase, tile, mp, e;
};

// Item g of the phase-major, expert-major, slab-pair-major, tile-minor order;
// tile_start[e] (shared memory) is expert e's first tile (experts without tokens
// repeat it).
__device__ __forceinline__ PairItem decode_pair_item(int g, int n0, int m0, int m1, int E,
                                                     const int32_t* __restrict__ tile_start) {
  PairItem it;
  int m = m0;
  it.phase = 0;
  if (g >= n0) {
    g -= n0;
    m = m1;
    it.phase = 1;
  }
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] * m <= g)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int t0 = tile_start[lo];
  const int ntiles = tile_start[lo + 1] - t0;
  it.e = lo;
  const int local = g - t0 * m;
  it.mp = local / ntiles;
  it.tile = t0 + local % ntiles;
  return it;
}

__device__ __forceinline__ float silu_times(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Tensor maps: weight codes (128-row boxes of k-block tiles), token/intermediate rows
// (one map per half-tile height 16, 32, .., 96 rows, so that a stage's token rows are
// one copy), and every scale region viewed as 256-byte rows (4-row boxes: two
// 512-byte scale blocks).  Each copy costs the issuing SM's TMA unit about the same
// whatever its size, so fewer, larger boxes keep more bytes in flight.
constexpr int kHalfSizes = kHalfRows / kBoxRows;   // 6
struct PairMaps {
  CUtensorMap w[2], wsf[2], tsf[2], t[2][kHalfSizes];
};

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    moe_pair_kernel(const __grid_constant__ PairMaps maps, const PairArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  PairTail* tail = reinterpret_cast<PairTail*>(smem + kSmTail);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = (int)cluster_id(), npairs = (int)cluster_count();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&tail->full[s], 1);
      ptx::mbar_init(&tail->empty[s], 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      ptx::mbar_init(&tail->acc_full[b], 1);
      ptx::mbar_init(&tail->acc_empty[b], 2 * kEpiWarps);
    }
    ptx::mbar_init(&tail->mma_done, 1);
    for (int r = 0; r < kRing; ++r) {
      ptx::mbar_init(&tail->ring_full[r], 1);
      ptx::mbar_init(&tail->ring_empty[r], kEpiWarps + (leader ? 1 : 0));
    }
    tail->abort = 0;
    ptx::fence_mbar_init();
    for (int p = 0; p < 2; ++p) {
      ptx::prefetch_tmap(&maps.w[p]);
      for (int h = 0; h < kHalfSizes; ++h) ptx::prefetch_tmap(&maps.t[p][h]);
      ptx::prefetch_tmap(&maps.wsf[p]);
      ptx::prefetch_tmap(&maps.tsf[p]);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&tail->tmem_base, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // Both CTAs' barriers exist before either signals the other's.
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = tail->tmem_base;
  volatile int* abort_flag = &tail->abort;
  ptx::pdl_launch_dependents();
  ptx::pdl_wait();

  const int num_tiles = args.ws.flags[kFlagTiles];
  const int E = args.E;
  const int32_t* tile_start = tail->tile_start;
  for (int e = threadIdx.x; e <= E; e += blockDim.x) tail->tile_start[e] = args.ws.tile_start[e];
  __syncthreads();
  const int m0 = args.ph[0].m_pairs, m1 = args.ph[1].m_pairs;
  const int n0 = num_tiles * m0;
  const int total = n0 + (args.num_phases == 2 ? num_tiles * m1 : 0);
  // A tile's intermediate rows are complete once each gate/up slab of it has been
  // stored: one count per CTA and item, 2 * m0 in all.
  const int slabs0 = 2 * m0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_once = ptx::policy_evict_first();
      const uint64_t pol_shared = ptx::policy_evict_normal();
      const uint64_t pol_t = ptx::policy_evict_last();
      const uint32_t full0 = ptx::mapa_shared(ptx::smem_addr(&tail->full[0]), 0);
      const uint32_t s_a = ptx::smem_addr(smem + kSmA), s_b = ptx::smem_addr(smem + kSmB);
      const uint32_t s_sfa = ptx::smem_addr(smem + kSmSfa), s_sfb = ptx::smem_addr(smem + kSmSfb);
      int stage = 0, r = 0;
      uint32_t phase = 0, rph = 0;
      int64_t issued = 0;
      bool ok = true;
      // Items are decoded one ahead: the next item's table reads overlap the loads of
      // the current one.
      PairItem it = {};
      int4 ti = make_int4(0, 0, 0, 0);
      if (pair < total) {
        it = decode_pair_item(pair, n0, m0, m1, E, tile_start);
        ti = args.ws.tiles[it.tile];
      }
      for (int g = pair;; g += npairs) {
        const bool live = g < total;
        if (!ptx::mbar_wait(&tail->ring_empty[r], rph ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tail->ring[r] = live ? make_int4(g, ti.y, ti.z | (it.mp << 16), it.tile)
                             : make_int4(-1, 0, 0, 0);
        ptx::mbar_arrive(&tail->ring_full[r]);
        if (++r == kRing) {
          r = 0;
          rph ^= 1u;
        }
        if (!live) break;
        const PairPhase& P = args.ph[it.phase];
        const int row0 = ti.y, n = ti.z;
        const int nmma = (n + 31) / 32 * 32;       // MMA N: a multiple of 32, <= 192
        const int half = nmma / 2;                 // token rows this CTA stages
        const int nblk = nmma > kBN ? 2 : 1;       // 128-row token scale blocks
        const int wslab = it.e * (2 * P.m_pairs) + it.mp * 2 + (int)rank;
        const int brow = row0 + (int)rank * half;
        const CUtensorMap* tw = &maps.w[it.phase];
        const CUtensorMap* twsf = &maps.wsf[it.phase];
        const CUtensorMap* ttsf = &maps.tsf[it.phase];
        const CUtensorMap* tb = &maps.t[it.phase][half / kBoxRows - 1];   // half rows a box
        // A pair of slabs read by one token tile only is not kept; one shared by
        // several tiles of the expert stays for them.
        const int ntiles = tile_start[it.e + 1] - tile_start[it.e];
        const int g_next = g + npairs;
        PairItem it_next = {};
        int4 ti_next = make_int4(0, 0, 0, 0);
        const uint64_t pol_w = ntiles > 1 ? pol_shared : pol_once;
        // Both CTAs' bytes of a stage, all counted on the leader's barrier.
        const uint32_t bytes =
            2u * (uint32_t)(kATileBytes + kSfaBytes + half * kBKBytes + nblk * kSfaBytes);
        if (it.phase == 1) {
          // the down projection reads intermediate rows stored with ordinary stores
          ok = ptx::wait_counter(&args.ws.tile_done[it.tile], slabs0, abort_flag, kWaitLimitNs);
          if (!ok) break;
          ptx::fence_proxy_async_global();
        }
        // Coordinates of k-block 0; each k-block adds one tile (128 map rows) to the
        // weight box, 128 bytes to the token box and two scale blocks (4 rows) to both
        // scale boxes.
        int wy = wslab * P.num_kb * kBM;
        int sfay = wslab * P.kc4 * 2;
        int sfby = (row0 / kBN) * P.kc4 * 2;
        int bx = 0;
        const int sfb_next = P.kc4 * 2;   // the tile's second scale block, in 256-byte rows
        for (int kb = 0; kb < P.num_kb; ++kb) {
          if (!ptx::mbar_wait(&tail->empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t bar = full0 + (uint32_t)stage * 8u;
          if (leader) ptx::mbar_arrive_expect_tx(&tail->full[stage], bytes);
          ptx::tma_load_2d_pair(s_a + (uint32_t)stage * kATileBytes, tw, 0, wy, bar, pol_w);
          // the slab's two scale blocks of this k-block: 1 KiB = four 256-byte rows
          ptx::tma_load_2d_pair(s_sfa + (uint32_t)stage * kSfaBytes, twsf, 0, sfay, bar, pol_w);
          ptx::tma_load_2d_pair(s_b + (uint32_t)stage * kBSlot, tb, bx, brow, bar, pol_t);
          // the whole tile's token scale blocks (every CTA's MMA reads all N columns)
          const uint32_t d_sfb = s_sfb + (uint32_t)stage * kSfbBytes;
          ptx::tma_load_2d_pair(d_sfb, ttsf, 0, sfby, bar, pol_t);
          if (nblk == 2) ptx::tma_load_2d_pair(d_sfb + kSfaBytes, ttsf, 0, sfby + sfb_next, bar, pol_t);
          wy += kBM;
          sfay += 4;
          sfby += 4;
          bx += kBKBytes;
          if (kb == 0 && g_next < total) {
            it_next = decode_pair_item(g_next, n0, m0, m1, E, tile_start);
            ti_next = args.ws.tiles[it_next.tile];
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        it = it_next;
        ti = ti_next;
      }
      if (!ok) atomicOr(&args.ws.flags[0], kErrTimeout);
      // Drain: the pair's MMAs are done reading this CTA's last stages (they commit to
      // each CTA's stage barriers) before the block may leave.
      const int64_t first = issued > kStages ? issued - kStages : 0;
      for (int64_t i = first; i < issued; ++i) {
        int never = 0;
        ptx::mbar_wait(&tail->empty[(int)(i % kStages)], (uint32_t)((i / kStages) & 1), &never,
                       kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      const uint32_t empty_l = ptx::mapa_shared(ptx::smem_addr(&tail->empty[0]), 0);
      const uint32_t empty_p = ptx::mapa_shared(ptx::smem_addr(&tail->empty[0]), 1);
      const uint32_t accf_l = ptx::mapa_shared(ptx::smem_addr(&tail->acc_full[0]), 0);
      const uint32_t accf_p = ptx::mapa_shared(ptx::smem_addr(&tail->acc_full[0]), 1);
      // stage 0's operand descriptors; stage s adds s times a stage's bytes / 16
      const uint64_t da0 = ptx::desc_sw128(ptx::smem_addr(smem + kSmA));
      const uint64_t db0 = ptx::desc_sw128(ptx::smem_addr(smem + kSmB));
      const uint64_t dsa0 = ptx::desc_sf(ptx::smem_addr(smem + kSmSfa));
      const uint64_t dsb0 = ptx::desc_sf(ptx::smem_addr(smem + kSmSfb));
      const uint32_t sf_t0 = tmem_base + (uint32_t)kSfBase;
      int stage = 0, r = 0;
      uint32_t phase = 0, rph = 0, sfbuf = 0;
      int items = 0;   // items issued so far: accumulator buffer items % 2
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
        if (rec.x < 0) break;
        const PairPhase& P = args.ph[rec.x < n0 ? 0 : 1];
        const int n = rec.z & 0xFFFF;
        const int nmma = (n + 31) / 32 * 32;
        const int nblk = nmma > kBN ? 2 : 1;
        const int ab = items & 1;
        const uint32_t use = (uint32_t)(items >> 1);   // earlier uses of this buffer
        // the epilogue of this buffer's previous item has read it
        if (!ptx::mbar_wait(&tail->acc_empty[ab], (use & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // This one thread issues every tensor-core instruction of the pair, so its own
        // work per k-block is kept to the instructions themselves: descriptors advance
        // with the stage, the two instruction descriptors are set per item, and a
        // whole k-block's copies and MMAs are unrolled.
        const uint32_t d_tmem = tmem_base + (uint32_t)(ab * kAccCols);
        const uint32_t id0 = ptx::idesc_mxf4_m(2 * kBM, nmma, 0);
        const uint32_t id2 = ptx::idesc_mxf4_m(2 * kBM, nmma, 2);
        const int whole_kb = P.K / kBK;   // a last k-block of 128 elements follows these
        for (int kb = 0; kb < P.num_kb; ++kb) {
          if (!ptx::mbar_wait(&tail->full[stage], phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sfa_t = sf_t0 + (sfbuf ? (uint32_t)kSfCols : 0u);
          const uint32_t sfb_t = sfa_t + kSfaCols;
          const uint64_t da = da0 + (uint64_t)(stage * (kATileBytes >> 4));
          const uint64_t db = db0 + (uint64_t)(stage * (kBSlot >> 4));
          const uint64_t dsa = dsa0 + (uint64_t)(stage * (kSfaBytes >> 4));
          const uint64_t dsb = dsb0 + (uint64_t)(stage * (kSfbBytes >> 4));
          const uint32_t acc0 = kb != 0 ? 1u : 0u;
          // scale block a of B's 128-row block b: smem dsb + (b * 1024 + a * 512) / 16,
          // tensor memory sfb_t + 8 a + 4 b; A's atom a: dsa + a * 512 / 16, sfa_t + 4 a
          ptx::tc_cp_sf_pair(sfa_t, dsa);
          ptx::tc_cp_sf_pair(sfb_t, dsb);
          if (nblk == 2) ptx::tc_cp_sf_pair(sfb_t + 4, dsb + 64);
          if (kb < whole_kb) {
            ptx::tc_cp_sf_pair(sfa_t + 4, dsa + 32);
            ptx::tc_cp_sf_pair(sfb_t + 8, dsb + 32);
            if (nblk == 2) ptx::tc_cp_sf_pair(sfb_t + 12, dsb + 96);
          }
          // K = 64 per MMA (32 bytes of each operand row: +2 in a descriptor)
          ptx::tc_mma_mxf4_pair(d_tmem, da, db, id0, sfa_t, sfb_t, acc0);
          ptx::tc_mma_mxf4_pair(d_tmem, da + 2, db + 2, id2, sfa_t, sfb_t, 1u);
          if (kb < whole_kb) {
            ptx::tc_mma_mxf4_pair(d_tmem, da + 4, db + 4, id0, sfa_t + 4, sfb_t + 8, 1u);
            ptx::tc_mma_mxf4_pair(d_tmem, da + 6, db + 6, id2, sfa_t + 4, sfb_t + 8, 1u);
          }
          ptx::tc_commit_pair(empty_l + (uint32_t)stage * 8u);
          ptx::tc_commit_pair(empty_p + (uint32_t)stage * 8u);
          sfbuf ^= 1u;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit_pair(accf_l + (uint32_t)ab * 8u);
        ptx::tc_commit_pair(accf_p + (uint32_t)ab * 8u);
        ++items;
      }
      if (!ok) atomicOr(&args.ws.flags[0], kErrTimeout);
      // Whatever happened, every MMA issued here finishes before the pair's memory goes.
      ptx::tc_commit_pair(ptx::mapa_shared(ptx::smem_addr(&tail->mma_done), 0));
      int never = 0;
      ptx::mbar_wait(&tail->mma_done, 0, &never, kWaitLimitNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                 // 0..7
    const int q = warp & 3;                  // tensor-memory lane quarter of this warp
    const int hh = ew >> 2;                  // chunk parity: chunks hh, hh + 2, ...
    const int ep_tid = threadIdx.x - 64;     // 0..255
    const uint32_t acc_empty_l = ptx::mapa_shared(ptx::smem_addr(&tail->acc_empty[0]), 0);
    int r = 0, xb = 0, items = 0;
    uint32_t rph = 0;
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
      const int row0 = rec.y, n = rec.z & 0xFFFF, mp = rec.z >> 16, item_tile = rec.w;
      const int slab = mp * 2 + (int)rank;   // this CTA's 128-row weight slab of the expert
      const int ab = items & 1;
      const uint32_t use = (uint32_t)(items >> 1);
      ++items;
      const int nch = (n + kEpiCols - 1) / kEpiCols;
      // Down items: row metadata of this warp's chunks (ci = hh + 2k covers columns
      // 32k + 16hh .. +15), read while the MMAs run: lane 16hh + j holds column
      // 32k + 16hh + j in register k.
      int tok_r[kMaxChunks / 2];
      float w_r[kMaxChunks / 2];
#pragma unroll
      for (int k = 0; k < kMaxChunks / 2; ++k) {
        const int col = 32 * k + lane;
        tok_r[k] = 0;
        w_r[k] = 0.f;
        if (MODE == kModeLayer && item_phase == 1 && (lane >> 4) == hh && col < n) {
          tok_r[k] = args.ws.slot_token[row0 + col];
          w_r[k] = args.ws.slot_weight[row0 + col];
        }
      }
      if (!ptx::mbar_wait(&tail->acc_full[ab], use & 1u, abort_flag, kWaitLimitNs)) {
        if (ep_tid == 0) atomicOr(&args.ws.flags[0], kErrTimeout);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t taddr =
          tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * kAccCols);
      // Chunk ci = hh + 2k of this warp (k: its index among the warp's chunks).
      auto chunk = [&](const int ci, const int k, const float(&v)[kEpiCols]) {
        const int c0 = ci * kEpiCols;
        const int ncol = min(kEpiCols, n - c0);
        if (MODE == kModeRaw) {
          const int m = slab * kBM + q * 32 + lane;
          const int col = gate_up_source_row(m, args.I);
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) {
            if (j < ncol) {
              const int a = args.ws.slot_assign[row0 + c0 + j];
              args.gate_up_debug[(size_t)a * 2 * args.I + col] = v[j];
            }
          }
        } else if (item_phase == 0) {
          // Warp rows: [gate even 8 | up even 8 | gate odd 8 | up odd 8] of features
          // (slab * 4 + q) * 16 ..+15; lane l and l ^ 8 hold one feature's gate and up.
          // Gate lanes compute column 2p, up lanes column 2p+1: one exchange each.
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
          // steps over bits 0, 1 and 2 each lane keeps one column, p = 4 b0 + 2 b1 + b2.
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
          float a1;
          {
            const float send = b2 ? a2[0] : a2[1];
            const float keep = b2 ? a2[1] : a2[0];
            a1 = fmaxf(keep, __shfl_xor_sync(kFull, send, 4));
          }
          a1 = fmaxf(a1, __shfl_xor_sync(kFull, a1, 16));
          if ((lane & 16) == 0) {
            const int pm = (b0 ? 4 : 0) + (b1 ? 2 : 0) + (b2 ? 1 : 0);
            tail->xchg[hh][xb][q][2 * pm + (up_lane ? 1 : 0)] = a1;
          }
          ptx::named_bar_sync(1 + hh, 128);
          const int i_kc4 = args.I / 128;
          // Each column's scale once, by the lane holding the column after the
          // butterfly (column 2 pm + up), shuffled to the lanes that need it; that
          // lane stages the scale byte.  32-feature group: this warp's 16 features
          // and the partner quarter's.
          const int pm = ((lane & 1) << 2) | (lane & 2) | ((lane >> 2) & 1);
          const int cm = 2 * pm + (up_lane ? 1 : 0);
          const float am_m = fmaxf(tail->xchg[hh][xb][q][cm], tail->xchg[hh][xb][q ^ 1][cm]);
          const int e_m = ptx::mx_scale_exponent(am_m);
          const float mul_m = ptx::pow2_neg(e_m);
          if ((lane & 16) == 0 && (q & 1) == 0) tail->sstage[hh][xb][cm][q >> 1] = (uint8_t)(e_m + 127);
          uint32_t code[kEpiCols / 2];
#pragma unroll
          for (int p = 0; p < kEpiCols / 2; ++p) {
            const int src = ((p >> 2) & 1) | (((p >> 1) & 1) << 1) | ((p & 1) << 2) | (lane & 8);
            const float qv = hv[p] * __shfl_sync(kFull, mul_m, src);
            const float qodd = __shfl_down_sync(kFull, qv, 16);
            code[p] = ptx::e2m1x2(qv, qodd);
          }
          if (lane < 16) {
#pragma unroll
            for (int p = 0; p < kEpiCols / 2; ++p) {
              const int jc = 2 * p + (up_lane ? 1 : 0);
              tail->hstage[hh][xb][jc][q * 8 + (lane & 7)] = (uint8_t)code[p];
            }
          }
          ptx::named_bar_sync(1 + hh, 128);
          // The chunk's rows, whole: warp q stores columns 4q..4q+3, 16 code bytes a
          // lane (two lanes a row's 32 bytes) and the two scale bytes.
          if (lane < 8) {
            const int jc = q * 4 + (lane >> 1);
            if (jc < ncol) {
              const size_t row = (size_t)row0 + c0 + jc;
              const uint4 cv =
                  *reinterpret_cast<const uint4*>(&tail->hstage[hh][xb][jc][(lane & 1) * 16]);
              *reinterpret_cast<uint4*>(args.ws.hb + row * (size_t)(args.I / 2) +
                                        (size_t)slab * 32 + (lane & 1) * 16) = cv;
            }
          } else if (lane < 12) {
            const int jc = q * 4 + (lane - 8);
            if (jc < ncol) {
              const size_t row = (size_t)row0 + c0 + jc;
              const uint16_t sv = *reinterpret_cast<const uint16_t*>(&tail->sstage[hh][xb][jc][0]);
              *reinterpret_cast<uint16_t*>(args.ws.hsf + sf_atom_offset(row, slab * 2, i_kc4)) = sv;
            }
          }
          xb ^= 1;
        } else {
          // Down projection: this warp holds output features slab*128 + q*32 + lane of
          // up to 16 token columns; add them, weighted, into the fp32 accumulator.
          // Every column's token and weight first, so the shuffles overlap.
          const int my_tok = tok_r[k];
          const float my_w = w_r[k];
          int tok_j[kEpiCols];
          float w_j[kEpiCols];
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) {
            const int src = hh * kEpiCols + j;
            tok_j[j] = __shfl_sync(kFull, my_tok, src);
            w_j[j] = __shfl_sync(kFull, my_w, src);
          }
          float* const col0 = args.ws.acc + (size_t)slab * kBM + q * 32 + lane;
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j)
            if (j < ncol) atomicAdd(col0 + (size_t)tok_j[j] * args.H, w_j[j] * v[j]);
        }
      };
      // This warp's chunks, each load issued one chunk ahead of its math; once the
      // last load has landed the buffer goes back to the MMA issuer (one arrival per
      // warp on the leader's barrier; the next item already runs on the other buffer).
      uint32_t ra[kEpiCols], rb[kEpiCols];
      if (hh < nch) ptx::tmem_ld16_issue(taddr + (uint32_t)(hh * kEpiCols), ra);
      bool released = false;
#pragma unroll
      for (int k = 0; k < kMaxChunks / 2; ++k) {
        const int ci = hh + 2 * k;
        if (ci >= nch) break;
        uint32_t(&cur)[kEpiCols] = (k & 1) ? rb : ra;
        uint32_t(&nxt)[kEpiCols] = (k & 1) ? ra : rb;
        ptx::tmem_wait_ld(cur);
        if (ci + 2 < nch) {
          ptx::tmem_ld16_issue(taddr + (uint32_t)((ci + 2) * kEpiCols), nxt);
        } else {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive_cluster(acc_empty_l + (uint32_t)ab * 8u);
          released = true;
        }
        float v[kEpiCols];
#pragma unroll
        for (int j = 0; j < kEpiCols; ++j) v[j] = __uint_as_float(cur[j]);
        chunk(ci, k, v);
      }
      if (!released) {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(acc_empty_l + (uint32_t)ab * 8u);
      }
      if (MODE == kModeLayer && item_phase == 0) {
        // Publish: this CTA's slab of the tile's intermediate rows is written.
        // The epilogue threads' stores are ordered before the barrier at block scope;
        // one thread's GPU-scope fence after it then releases them all (fences are
        // cumulative), instead of every thread waiting out a fence of its own.
        ptx::named_bar_sync(3, 2 * 128);
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
  // Neither CTA leaves, nor frees its tensor memory, while the pair may still use it.
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0) {
    // The last CTA out resets the tile counters for the next call.
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
// Host side.
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

// uint8 matrix [rows, row_bytes] read in boxes of box_x bytes x box_rows rows.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
                     uint32_t box_x, uint32_t box_rows, bool swizzle128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_x, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A scale region of `bytes` bytes (a multiple of 1024) as 256-byte rows, read four rows
// (two 512-byte scale blocks) at a time.
cudaError_t make_sf_map(CUtensorMap* m, const void* base, uint64_t bytes) {
  return make_map(m, base, 256, bytes / 256, 256, 4, false);
}

template <int MODE>
cudaError_t launch_pair_mode(const LayerLaunch& g, const PairMaps& maps, const PairArgs& a,
                             cudaStream_t st) {
  static int clusters = 0;   // per instantiation, for the device of the first launch
  if (clusters == 0) {
    cudaError_t err = cudaFuncSetAttribute(moe_pair_kernel<MODE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    // Every cluster must be resident at once (a down item waits for other clusters'
    // gate/up items), so the grid is at most what the device holds together.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    int c = 0;
    err = cudaOccupancyMaxActiveClusters(&c, moe_pair_kernel<MODE>, &cfg);
    if (err != cudaSuccess) return err;
    if (c < 1) return cudaErrorInvalidConfiguration;
    clusters = c < g.num_sms / 2 ? c : g.num_sms / 2;
  }
  return launch_pdl(moe_pair_kernel<MODE>, dim3(2 * clusters), dim3(kThreads), kSmemBytes, st,
                    maps, a);
}

}  // namespace

bool pair_shape_ok(const Shape& s) {
  return !s.f8 && !s.nv && s.H % (2 * kBM) == 0 && (2 * s.I) % (2 * kBM) == 0;
}

cudaError_t launch_layer_pair(const LayerLaunch& g, cudaStream_t st) {
  const Shape& s = g.shape;
  if (!pair_shape_ok(s) || g.pull) return cudaErrorNotSupported;
  const uint64_t xrow = (uint64_t)s.H / 2, hrow = (uint64_t)s.I / 2;
  const uint64_t w1_rows = (uint64_t)s.E * 2 * s.I * weight_num_kb(s, s.H);
  const uint64_t w2_rows = (uint64_t)s.E * s.H * weight_num_kb(s, s.I);
  if (w1_rows > 0x7FFFFFFFull || w2_rows > 0x7FFFFFFFull) return cudaErrorInvalidValue;
  // scale regions: weights' 128x4 blocks (sizes as laid out by the prepared blob), the
  // workspace's token and intermediate blocks (128-row tiles)
  const uint64_t w1sf = (uint64_t)s.E * 2 * s.I * (s.H / 32);
  const uint64_t w2sf = (uint64_t)s.E * s.H * (s.I / 32);
  const uint64_t xsf = (uint64_t)g.R_cap * (s.H / 32);
  const uint64_t hsf = (uint64_t)g.R_cap * (s.I / 32);
  PairMaps maps;
  cudaError_t err;
  if ((err = make_map(&maps.w[0], g.w1_codes, kBKBytes, w1_rows, kBKBytes, kBM, true)) ||
      (err = make_map(&maps.w[1], g.w2_codes, kBKBytes, w2_rows, kBKBytes, kBM, true)) ||

      (err = make_sf_map(&maps.wsf[0], g.w1_sf, w1sf)) ||
      (err = make_sf_map(&maps.wsf[1], g.w2_sf, w2sf)) ||
      (err = make_sf_map(&maps.tsf[0], g.ws.xsf, xsf)) ||
      (err = make_sf_map(&maps.tsf[1], g.ws.hsf, hsf)))
    return err;
  for (int h = 0; h < kHalfSizes; ++h) {
    const uint32_t rows = (uint32_t)((h + 1) * kBoxRows);
    if ((err = make_map(&maps.t[0][h], g.ws.xb, xrow, (uint64_t)g.R_cap, kBKBytes, rows, true)) ||
        (err = make_map(&maps.t[1][h], g.ws.hb, hrow, (uint64_t)g.R_cap, kBKBytes, rows, true)))
      return err;
  }
  PairArgs a;
  for (int p = 0; p < 2; ++p) {
    const int rows = p == 0 ? 2 * s.I : s.H;
    const int K = p == 0 ? s.H : s.I;
    a.ph[p].m_pairs = rows / (2 * kBM);
    a.ph[p].K = K;
    a.ph[p].num_kb = (K + kBK - 1) / kBK;
    a.ph[p].kc4 = K / 128;
  }
  a.num_phases = g.num_phases;
  a.H = s.H;
  a.I = s.I;
  a.E = s.E;
  a.ws = g.ws;
  a.gate_up_debug = g.gate_up_debug;
  return g.num_phases == 2 ? launch_pair_mode<kModeLayer>(g, maps, a, st)
                           : launch_pair_mode<kModeRaw>(g, maps, a, st);
}

}  // namespace mxmoe
