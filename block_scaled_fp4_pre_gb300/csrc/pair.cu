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
// 256-row token tile, and receives 128 x 256 accumulators -- twice the FLOPs per
// staged byte, with no multicast.
//
// Items are (token tile <= 256 rows, pair of 128-row weight slabs), first every
// gate/up item, then every down item, each phase expert by expert, slab pair by slab
// pair, then by the expert's token tiles.  Cluster c takes items c, c + C, c + 2C, ...
// (C clusters, all resident), so both CTAs of a pair know the sequence without
// talking; every gate/up item of a tile precedes its down items in every cluster's
// sequence, so a down item's bounded wait for its tile's intermediate rows ends.
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
//               columns [128h, 128h + 128) with h = (w - 2) / 4.
// Every wait is bounded (kWaitLimitNs); a timeout sets the workspace error flag and
// each role leaves its loop; both CTAs meet at a cluster barrier before the tensor
// memory is freed.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mxmoe {
namespace {

constexpr int kStages = 6;
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kTmemCols = 512;
constexpr int kAccCols = kBNPair;                 // 128 lanes x up to 256 fp32 columns
// Scale registers after the accumulator, two buffers: A (this CTA's 128 rows) 4
// columns per 128-element scale block, B (up to 256 token rows = two 128-row blocks)
// 8 columns per scale block (block b of rows at +4b).
constexpr int kSfaCols = 8;
constexpr int kSfCols = kSfaCols + 16;
constexpr int kSfBase = kAccCols;
constexpr int kSpareBase = kSfBase + 2 * kSfCols;  // copies of accumulator chunks
constexpr int kEpiCols = 16;
constexpr int kSpareChunks = 6;                   // per column half (96 columns)
static_assert(kSpareBase + 2 * kSpareChunks * kEpiCols <= kTmemCols, "tensor memory layout");
constexpr int kBoxRows = 16;                      // token rows of a partial-tile TMA box
constexpr int kRing = 8;
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kSfaBytes = 2 * kSFAtomBytes;       // one k-block of one 128-row slab
constexpr int kSfbBytes = 2 * kSfaBytes;          // one k-block of two 128-row blocks

enum PairMode { kModeLayer = 0, kModeRaw = 1 };

// Shared memory: kStages x (weight box, token half-tile, weight scales, token
// scales), then the tail.
constexpr size_t kSmA = 0;
constexpr size_t kSmB = kSmA + (size_t)kStages * kATileBytes;
constexpr size_t kSmSfa = kSmB + (size_t)kStages * kBTileBytes;
constexpr size_t kSmSfb = kSmSfa + (size_t)kStages * kSfaBytes;
constexpr size_t kSmTail = kSmSfb + (size_t)kStages * kSfbBytes;

struct __align__(16) PairTail {
  uint64_t full[kStages];    // leader: both CTAs' loads of a stage landed
  uint64_t empty[kStages];   // each CTA: the pair's MMAs are done with its stage
  uint64_t acc_full;         // each CTA: the item's accumulator is complete
  uint64_t acc_empty;        // leader: all 16 epilogue warps have read it
  uint64_t mma_done;         // leader: every MMA it issued has finished
  uint64_t ring_full[kRing];
  uint64_t ring_empty[kRing];
  int4 ring[kRing];          // (item, first row, rows | slab pair << 16, tile); item -1: stop
  uint32_t tmem_base;
  int abort;
  float xchg[2][2][4][kEpiCols];                 // [half][buffer][quarter][column]
  alignas(16) uint8_t hstage[2][2][kEpiCols][32];
  alignas(4) uint8_t sstage[2][2][kEpiCols][2];
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
// tile_start[e] is expert e's first tile (experts without tokens repeat it).
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
    if (__ldg(&tile_start[mid]) * m <= g)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int t0 = __ldg(&tile_start[lo]);
  const int ntiles = __ldg(&tile_start[lo + 1]) - t0;
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
// (a whole 128-row half-tile, or 16-row boxes), and every scale region viewed as
// 256-byte rows (4-row boxes: two 512-byte scale blocks).
struct PairMaps {
  CUtensorMap w[2], t128[2], t16[2], wsf[2], tsf[2];
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
    ptx::mbar_init(&tail->acc_full, 1);
    ptx::mbar_init(&tail->acc_empty, 2 * kEpiWarps);
    ptx::mbar_init(&tail->mma_done, 1);
    for (int r = 0; r < kRing; ++r) {
      ptx::mbar_init(&tail->ring_full[r], 1);
      ptx::mbar_init(&tail->ring_empty[r], kEpiWarps + (leader ? 1 : 0));
    }
    tail->abort = 0;
    ptx::fence_mbar_init();
    for (int p = 0; p < 2; ++p) {
      ptx::prefetch_tmap(&maps.w[p]);
      ptx::prefetch_tmap(&maps.t128[p]);
      ptx::prefetch_tmap(&maps.t16[p]);
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
  const int32_t* tile_start = args.ws.tile_start;
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
      int stage = 0, r = 0;
      uint32_t phase = 0, rph = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int g = pair;; g += npairs) {
        const bool live = g < total;
        PairItem it = {};
        int4 ti = make_int4(0, 0, 0, 0);
        if (live) {
          it = decode_pair_item(g, n0, m0, m1, E, tile_start);
          ti = args.ws.tiles[it.tile];
        }
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
        const int nmma = (n + 31) / 32 * 32;       // MMA N: a multiple of 32, <= 256
        const int half = nmma / 2;                 // token rows this CTA stages
        const int nblk = nmma > kBN ? 2 : 1;       // 128-row token scale blocks
        const int wslab = it.e * (2 * P.m_pairs) + it.mp * 2 + (int)rank;
        const int brow = row0 + (int)rank * half;
        const CUtensorMap* tw = &maps.w[it.phase];
        const CUtensorMap* twsf = &maps.wsf[it.phase];
        const CUtensorMap* ttsf = &maps.tsf[it.phase];
        // A pair of slabs read by one token tile only is not kept; one shared by
        // several tiles of the expert stays for them.
        const int ntiles = __ldg(&tile_start[it.e + 1]) - __ldg(&tile_start[it.e]);
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
        for (int kb = 0; kb < P.num_kb; ++kb) {
          if (!ptx::mbar_wait(&tail->empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const uint32_t bar = full0 + (uint32_t)stage * 8u;
          if (leader) ptx::mbar_arrive_expect_tx(&tail->full[stage], bytes);
          ptx::tma_load_2d_pair(smem + kSmA + (size_t)stage * kATileBytes, tw, 0,
                                (wslab * P.num_kb + kb) * kBM, bar, pol_w);
          // the slab's two scale blocks of this k-block: 1 KiB = four 256-byte rows
          ptx::tma_load_2d_pair(smem + kSmSfa + (size_t)stage * kSfaBytes, twsf, 0,
                                (wslab * P.kc4 + 2 * kb) * 2, bar, pol_w);
          uint8_t* b_dst = smem + kSmB + (size_t)stage * kBTileBytes;
          if (half == kBN) {
            ptx::tma_load_2d_pair(b_dst, &maps.t128[it.phase], kb * kBKBytes, brow, bar, pol_t);
          } else {
            for (int j = 0; j < half / kBoxRows; ++j)
              ptx::tma_load_2d_pair(b_dst + j * kBoxRows * kBKBytes, &maps.t16[it.phase],
                                    kb * kBKBytes, brow + j * kBoxRows, bar, pol_t);
          }
          // the whole tile's token scale blocks (every CTA's MMA reads all N columns)
          for (int b = 0; b < nblk; ++b)
            ptx::tma_load_2d_pair(smem + kSmSfb + (size_t)stage * kSfbBytes + b * kSfaBytes, ttsf,
                                  0, ((row0 / kBN + b) * P.kc4 + 2 * kb) * 2, bar, pol_t);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
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
      const uint32_t accf_l = ptx::mapa_shared(ptx::smem_addr(&tail->acc_full), 0);
      const uint32_t accf_p = ptx::mapa_shared(ptx::smem_addr(&tail->acc_full), 1);
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
        if (rec.x < 0) break;
        const PairPhase& P = args.ph[rec.x < n0 ? 0 : 1];
        const int n = rec.z & 0xFFFF;
        const int nmma = (n + 31) / 32 * 32;
        const int nblk = nmma > kBN ? 2 : 1;
        if (!ptx::mbar_wait(&tail->acc_empty, acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        for (int kb = 0; kb < P.num_kb; ++kb) {
          if (!ptx::mbar_wait(&tail->full[stage], phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int kvalid = min(kBK, P.K - kb * kBK);
          const int atoms = kvalid / 128;
          const uint32_t sfa_t = tmem_base + (uint32_t)(kSfBase + sfbuf * kSfCols);
          const uint32_t sfb_t = sfa_t + kSfaCols;
          const uint32_t sa = ptx::smem_addr(smem + kSmSfa + (size_t)stage * kSfaBytes);
          const uint32_t sb = ptx::smem_addr(smem + kSmSfb + (size_t)stage * kSfbBytes);
          for (int a = 0; a < atoms; ++a) {
            ptx::tc_cp_sf_pair(sfa_t + a * 4, ptx::desc_sf(sa + a * kSFAtomBytes));
            for (int b = 0; b < nblk; ++b)
              ptx::tc_cp_sf_pair(sfb_t + a * 8 + b * 4,
                                 ptx::desc_sf(sb + b * kSfaBytes + a * kSFAtomBytes));
          }
          const uint32_t a_base = ptx::smem_addr(smem + kSmA + (size_t)stage * kATileBytes);
          const uint32_t b_base = ptx::smem_addr(smem + kSmB + (size_t)stage * kBTileBytes);
          const int steps = kvalid / 64;   // K = 64 per MMA
          for (int s = 0; s < steps; ++s)
            ptx::tc_mma_mxf4_pair(tmem_base, ptx::desc_sw128(a_base + s * 32),
                                  ptx::desc_sw128(b_base + s * 32),
                                  ptx::idesc_mxf4_m(2 * kBM, nmma, (s & 1) * 2),
                                  sfa_t + (s >> 1) * 4, sfb_t + (s >> 1) * 8,
                                  (kb | s) != 0 ? 1u : 0u);
          ptx::tc_commit_pair(empty_l + (uint32_t)stage * 8u);
          ptx::tc_commit_pair(empty_p + (uint32_t)stage * 8u);
          sfbuf ^= 1u;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::tc_commit_pair(accf_l);
        ptx::tc_commit_pair(accf_p);
        acc_phase ^= 1u;
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
    const int hh = ew >> 2;                  // column half: tile columns [128 hh, 128 hh + 128)
    const int ep_tid = threadIdx.x - 64;     // 0..255
    const uint32_t acc_empty_l = ptx::mapa_shared(ptx::smem_addr(&tail->acc_empty), 0);
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
      const int row0 = rec.y, n = rec.z & 0xFFFF, mp = rec.z >> 16, item_tile = rec.w;
      const int slab = mp * 2 + (int)rank;   // this CTA's 128-row weight slab of the expert
      const int cbase = hh * kBN;            // first tile column of this half
      const int nh = max(0, min(kBN, n - cbase));
      const int hrow0 = row0 + cbase;        // workspace row of this half's column 0
      // Down items: the half's row metadata, read while the MMAs run (lane l holds
      // columns l, l+32, l+64, l+96).
      int tok_r[kBN / 32];
      float w_r[kBN / 32];
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i) {
        tok_r[i] = 0;
        w_r[i] = 0.f;
        if (MODE == kModeLayer && item_phase == 1 && lane + 32 * i < nh) {
          tok_r[i] = args.ws.slot_token[hrow0 + lane + 32 * i];
          w_r[i] = args.ws.slot_weight[hrow0 + lane + 32 * i];
        }
      }
      if (!ptx::mbar_wait(&tail->acc_full, acc_phase, abort_flag, kWaitLimitNs)) {
        if (ep_tid == 0) atomicOr(&args.ws.flags[0], kErrTimeout);
        break;
      }
      acc_phase ^= 1u;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)cbase;
      const uint32_t tspare = tmem_base + ((uint32_t)(q * 32) << 16) +
                              (uint32_t)(kSpareBase + hh * kSpareChunks * kEpiCols);
      auto chunk = [&](const int ci, const float(&v)[kEpiCols]) {
        const int c0 = ci * kEpiCols;
        const int ncol = min(kEpiCols, nh - c0);
        if (MODE == kModeRaw) {
          const int m = slab * kBM + q * 32 + lane;
          const int col = gate_up_source_row(m, args.I);
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) {
            if (j < ncol) {
              const int a = args.ws.slot_assign[hrow0 + c0 + j];
              args.gate_up_debug[(size_t)a * 2 * args.I + col] = v[j];
            }
          }
        } else if (item_phase == 0) {
          // Warp rows: [gate even 8 | up even 8 | gate odd 8 | up odd 8] of features
          // (slab * 4 + q) * 16 ..+15; lane l and l ^ 8 hold one feature's gate and up.
          // Gate lanes compute column 2p, up lanes column 2p+1: one exchange each.
          const bool up_lane = (lane & 8) != 0;
          float hv[kEpiCols / 2];
#pragma unroll
          for (int p = 0; p < kEpiCols / 2; ++p) {
            const float x = __shfl_xor_sync(kFull, up_lane ? v[2 * p] : v[2 * p + 1], 8);
            const float h = up_lane ? silu_times(x, v[2 * p + 1]) : silu_times(v[2 * p], x);
            hv[p] = h;
            float a = fabsf(h);
            a = fmaxf(a, __shfl_xor_sync(kFull, a, 1));
            a = fmaxf(a, __shfl_xor_sync(kFull, a, 2));
            a = fmaxf(a, __shfl_xor_sync(kFull, a, 4));
            a = fmaxf(a, __shfl_xor_sync(kFull, a, 16));
            if ((lane & 23) == 0) tail->xchg[hh][xb][q][2 * p + (up_lane ? 1 : 0)] = a;
          }
          ptx::named_bar_sync(1 + hh, 128);
          const int i_kc4 = args.I / 128;
          float amax[kEpiCols / 2];
#pragma unroll
          for (int p = 0; p < kEpiCols / 2; ++p) {
            const int jc = 2 * p + (up_lane ? 1 : 0);
            // 32-feature group: this warp's 16 features and the partner quarter's
            amax[p] = fmaxf(tail->xchg[hh][xb][q][jc], tail->xchg[hh][xb][q ^ 1][jc]);
          }
          uint32_t code[kEpiCols / 2];
          int ex[kEpiCols / 2];
#pragma unroll
          for (int p = 0; p < kEpiCols / 2; ++p) {
            ex[p] = ptx::mx_scale_exponent(amax[p]);
            const float qv = hv[p] * ptx::pow2_neg(ex[p]);
            const float qodd = __shfl_down_sync(kFull, qv, 16);
            code[p] = ptx::e2m1x2(qv, qodd);
          }
          if (lane < 16) {
#pragma unroll
            for (int p = 0; p < kEpiCols / 2; ++p) {
              const int jc = 2 * p + (up_lane ? 1 : 0);
              tail->hstage[hh][xb][jc][q * 8 + (lane & 7)] = (uint8_t)code[p];
              if ((lane & 7) == 0 && (q & 1) == 0)
                tail->sstage[hh][xb][jc][q >> 1] = (uint8_t)(ex[p] + 127);
            }
          }
          ptx::named_bar_sync(1 + hh, 128);
          // The chunk's rows, whole: warp q stores columns 4q..4q+3, 16 code bytes a
          // lane (two lanes a row's 32 bytes) and the two scale bytes.
          if (lane < 8) {
            const int jc = q * 4 + (lane >> 1);
            if (jc < ncol) {
              const size_t row = (size_t)hrow0 + c0 + jc;
              const uint4 cv =
                  *reinterpret_cast<const uint4*>(&tail->hstage[hh][xb][jc][(lane & 1) * 16]);
              *reinterpret_cast<uint4*>(args.ws.hb + row * (size_t)(args.I / 2) +
                                        (size_t)slab * 32 + (lane & 1) * 16) = cv;
            }
          } else if (lane < 12) {
            const int jc = q * 4 + (lane - 8);
            if (jc < ncol) {
              const size_t row = (size_t)hrow0 + c0 + jc;
              const uint16_t sv = *reinterpret_cast<const uint16_t*>(&tail->sstage[hh][xb][jc][0]);
              *reinterpret_cast<uint16_t*>(args.ws.hsf + sf_atom_offset(row, slab * 2, i_kc4)) = sv;
            }
          }
          xb ^= 1;
        } else {
          // Down projection: this warp holds output features slab*128 + q*32 + lane of
          // up to 16 token columns; add them, weighted, into the fp32 accumulator.
          const int my_tok = tok_r[ci >> 1];
          const float my_w = w_r[ci >> 1];
          const size_t feat = (size_t)slab * kBM + q * 32 + lane;
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) {
            const int src = (ci & 1) * kEpiCols + j;
            const int tok = __shfl_sync(kFull, my_tok, src);
            const float wt = __shfl_sync(kFull, my_w, src);
            if (j < ncol) atomicAdd(args.ws.acc + (size_t)tok * args.H + feat, wt * v[j]);
          }
        }
      };
      const int nch = (nh + kEpiCols - 1) / kEpiCols;
      const int ncopy = min(nch, kSpareChunks);
      // 1. The first chunks of this half into spare tensor memory, two loads in flight.
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
      // 2. The last two chunks straight into registers; then the accumulator goes back
      //    to the MMA issuer (one arrival per warp, on the leader's barrier), so the
      //    next item's MMAs run during this item's math.
      constexpr int kLastTwo = kBN / kEpiCols - 2;
      static_assert(kSpareChunks == kLastTwo, "tensor memory layout");
      uint32_t rd[2][kEpiCols];
#pragma unroll
      for (int d = 0; d < 2; ++d)
        if (kLastTwo + d < nch)
          ptx::tmem_ld16_issue(taddr + (uint32_t)((kLastTwo + d) * kEpiCols), rd[d]);
#pragma unroll
      for (int d = 0; d < 2; ++d)
        if (kLastTwo + d < nch) ptx::tmem_wait_ld(rd[d]);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(acc_empty_l);
#pragma unroll
      for (int d = 0; d < 2; ++d) {
        if (kLastTwo + d < nch) {
          float v[kEpiCols];
#pragma unroll
          for (int j = 0; j < kEpiCols; ++j) v[j] = __uint_as_float(rd[d][j]);
          chunk(kLastTwo + d, v);
        }
      }
      // 3. The copied chunks; the load of chunk ci+1 runs during the math of ci.
      uint32_t ra[kEpiCols], rb[kEpiCols];
      if (ncopy > 0) {
        ptx::tmem_ld16_issue(tspare, ra);
        ptx::tmem_wait_ld(ra);
      }
#pragma unroll
      for (int ci = 0; ci < kSpareChunks; ++ci) {
        if (ci >= ncopy) break;
        uint32_t(&cur)[kEpiCols] = (ci & 1) ? rb : ra;
        uint32_t(&nxt)[kEpiCols] = (ci & 1) ? ra : rb;
        const bool more = ci + 1 < ncopy;
        if (more) ptx::tmem_ld16_issue(tspare + (uint32_t)((ci + 1) * kEpiCols), nxt);
        float v[kEpiCols];
#pragma unroll
        for (int j = 0; j < kEpiCols; ++j) v[j] = __uint_as_float(cur[j]);
        chunk(ci, v);
        if (more) ptx::tmem_wait_ld(nxt);
      }
      if (MODE == kModeLayer && item_phase == 0) {
        // Publish: this CTA's slab of the tile's intermediate rows is written.
        __threadfence();
        ptx::named_bar_sync(3, 2 * 128);
        if (ep_tid == 0) {
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
      (err = make_map(&maps.t128[0], g.ws.xb, xrow, (uint64_t)g.R_cap, kBKBytes, kBN, true)) ||
      (err = make_map(&maps.t128[1], g.ws.hb, hrow, (uint64_t)g.R_cap, kBKBytes, kBN, true)) ||
      (err = make_map(&maps.t16[0], g.ws.xb, xrow, (uint64_t)g.R_cap, kBKBytes, kBoxRows, true)) ||
      (err = make_map(&maps.t16[1], g.ws.hb, hrow, (uint64_t)g.R_cap, kBKBytes, kBoxRows, true)) ||
      (err = make_sf_map(&maps.wsf[0], g.w1_sf, w1sf)) ||
      (err = make_sf_map(&maps.wsf[1], g.w2_sf, w2sf)) ||
      (err = make_sf_map(&maps.tsf[0], g.ws.xsf, xsf)) ||
      (err = make_sf_map(&maps.tsf[1], g.ws.hsf, hsf)))
    return err;
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
