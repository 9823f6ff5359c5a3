// pre_dispatch (quantise + bucket), weight preparation, MXFP4 quantisation of fp32
// rows, and the fp32 -> bf16 output conversion.
//
// Pages: prhub digest of SGLang PR #37279, section 实现拆解 items 3-4 (pre_dispatch
// writes E2M1 codes and group_size=32 scales plus the routing copies; the weight
// transform and the gran=16 interleave for MXFP4 activations); SGLang PR #48424,
// "DeepGEMM producers write FlashInfer's 128x4 scale layout" (scale blocks).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mxmoe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

// ---------------------------------------------------------------------------
// Bucketing.  Block b ranks the assignments a = t*k + j of chunk b (kBucketChunk of
// them, ascending a, i.e. ascending t then j) among those of the same expert:
// warp w owns a contiguous run of the chunk, walked 32 at a time; lanes holding the
// same expert are found with one ballot per bit of the expert id, the lowest of
// them advances the warp's count for that expert, and a scan over warps turns the
// counts into each warp's base.  Each block publishes its per-expert totals; the
// last block to finish scans them over blocks (bases of later chunks) and over
// experts (segment sizes from segment_rows -- whole tiles of tile_rows rows, or for
// the pair kernel kPairStride-row spans -- and the tile list).  Row of an assignment =
// segment start + tile_row_of_rank(its chunk's base + its rank in the chunk).

// Lanes whose key equals this lane's key (keys < 2^nbits): one ballot per bit, which
// measured faster here than __match_any_sync.
__device__ __forceinline__ unsigned peers_of(int key, int nbits) {
  unsigned m = kFull;
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (key >> b) & 1;
    const unsigned bal = __ballot_sync(kFull, bit);
    m &= bit ? bal : ~bal;
  }
  return m;
}

__global__ void __launch_bounds__(1024) bucket_kernel(const int32_t* __restrict__ ids, int T,
                                                      int k, int E, WsPtrs ws, int tile_rows) {
  extern __shared__ int32_t sh[];
  int32_t* cnt = sh;                        // [32][E] per-warp counts, then bases
  int32_t* key_sh = cnt + 32 * E;           // [kBucketChunk] expert id, E if invalid
  int32_t* tot = key_sh + kBucketChunk;     // [E]   tokens per expert (all chunks)
  int32_t* seg = tot + E;                   // [E+1] segment starts
  int32_t* tst = seg + E + 1;               // [E+1] tile starts
  __shared__ int32_t bad;
  __shared__ int32_t is_last;

  ptx::pdl_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int A = T * k;
  const int c0 = blockIdx.x * kBucketChunk;
  const int len = min(kBucketChunk, A - c0);
  // per-warp runs are whole multiples of 32 so that every round is one aligned chunk
  const int per = ((len + 32 * 32 - 1) / (32 * 32)) * 32;
  const int w0 = min(len, warp * per), w1 = min(len, w0 + per);
  int nbits = 1;
  while ((1 << nbits) <= E + 1) ++nbits;  // keys 0..E+1

  for (int i = tid; i < 32 * E; i += blockDim.x) cnt[i] = 0;
  for (int i = tid; i < len; i += blockDim.x) {
    const int e = ids[c0 + i];
    key_sh[i] = (e >= 0 && e < E) ? e : E;
  }
  if (tid == 0) bad = 0;
  __syncthreads();

  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const int key = i < w1 ? key_sh[i] : E + 1;
    const unsigned peers = peers_of(key, nbits);
    if ((peers & lt_mask) == 0) {  // lowest lane of its group
      if (key < E)
        cnt[warp * E + key] += __popc(peers);
      else if (key == E)
        atomicAdd(&bad, __popc(peers));
    }
  }
  __syncthreads();

  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += c;
    }
    if (gridDim.x == 1) {
      ws.blk_base[e] = 0;
      tot[e] = run;
    } else {
      ws.blk_base[(size_t)blockIdx.x * E + e] = run;  // this chunk's total, for now
    }
  }
  __syncthreads();

  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const int key = i < w1 ? key_sh[i] : E + 1;
    const unsigned peers = peers_of(key, nbits);
    const int rank = __popc(peers & lt_mask);
    if (key < E) ws.local_rank[c0 + i] = cnt[warp * E + key] + rank;
    __syncwarp();
    if (key < E && rank == 0) cnt[warp * E + key] += __popc(peers);
    __syncwarp();
  }

  int bad_all;
  if (gridDim.x == 1) {
    __syncthreads();
    bad_all = bad;
  } else {
    // Publish this chunk's totals; the last block to finish does the global scans.
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      if (bad) atomicAdd(&ws.flags[kFlagBucketBad], bad);
      is_last = atomicAdd(&ws.flags[kFlagBucketTicket], 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    const int nblk = gridDim.x;
    for (int e = tid; e < E; e += blockDim.x) {
      int run = 0;
      for (int b = 0; b < nblk; ++b) {
        int32_t* p = ws.blk_base + (size_t)b * E + e;
        const int c = __ldcg(p);
        *p = run;
        run += c;
      }
      tot[e] = run;
    }
    __syncthreads();
    bad_all = __ldcg(&ws.flags[kFlagBucketBad]);
  }

  // Exclusive scans over experts of the padded rows and the tiles: warp w scans
  // experts 32w..32w+31 (E <= 1024), then warp 0 scans the 32 warp totals.
  __shared__ int32_t wsum_rows[32], wsum_tiles[32];
  int ir = 0, it = 0, rows = 0, tiles = 0;
  {
    const int e = warp * 32 + lane;
    const int n = e < E ? tot[e] : 0;
    tiles = (n + tile_rows - 1) / tile_rows;
    rows = segment_rows(n, tile_rows);   // every tile starts at row 0 of a scale block
    ir = rows;
    it = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vr = __shfl_up_sync(kFull, ir, o), vt = __shfl_up_sync(kFull, it, o);
      if (lane >= o) {
        ir += vr;
        it += vt;
      }
    }
    if (lane == 31) {
      wsum_rows[warp] = ir;
      wsum_tiles[warp] = it;
    }
  }
  __syncthreads();
  if (warp == 0) {
    int br = wsum_rows[lane], bt = wsum_tiles[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vr = __shfl_up_sync(kFull, br, o), vt = __shfl_up_sync(kFull, bt, o);
      if (lane >= o) {
        br += vr;
        bt += vt;
      }
    }
    wsum_rows[lane] = br - wsum_rows[lane];    // exclusive bases of the warps
    wsum_tiles[lane] = bt - wsum_tiles[lane];
    if (lane == 31) {
      seg[E] = br;
      tst[E] = bt;
    }
  }
  __syncthreads();
  {
    const int e = warp * 32 + lane;
    if (e < E) {
      seg[e] = wsum_rows[warp] + ir - rows;
      tst[e] = wsum_tiles[warp] + it - tiles;
    }
  }
  __syncthreads();

  for (int e = tid; e <= E; e += blockDim.x) ws.tile_start[e] = tst[e];
  for (int e = tid; e < E; e += blockDim.x) {
    const int n = tot[e];
    ws.counts[e] = n;
    ws.seg[e] = seg[e];
    for (int i = 0, r = 0; r < n; ++i, r += tile_rows) {
      ws.tiles[tst[e] + i] =
          make_int4(e, seg[e] + tile_row_of_rank(r, tile_rows), min(tile_rows, n - r), 0);
      ws.tile_done[tst[e] + i] = 0;
    }
  }
  if (tid == 0) {
    ws.seg[E] = seg[E];
    ws.flags[kFlagTiles] = tst[E];
    ws.flags[kFlagValid] = A - bad_all;
    ws.flags[kFlagSched] = 0;
    ws.flags[kFlagExit] = 0;
    ws.flags[kFlagBucketTicket] = 0;
    ws.flags[kFlagBucketBad] = 0;
    if (bad_all) atomicOr(&ws.flags[0], kErrRouting);
  }
}

// Row of assignment a (or -1 for an id outside [0, E)), and the per-row tables, for a
// dispatch with token tiles of tile_rows rows.
__device__ __forceinline__ int assign_slot(int a, int k, int E, const int32_t* __restrict__ ids,
                                           const float* __restrict__ tw, const WsPtrs& ws,
                                           int tile_rows) {
  const int e = ids[a];
  int slot = -1;
  if (e >= 0 && e < E) {
    const int rank = ws.blk_base[(size_t)(a / kBucketChunk) * E + e] + ws.local_rank[a];
    slot = ws.seg[e] + tile_row_of_rank(rank, tile_rows);
    ws.slot_token[slot] = a / k;
    ws.slot_assign[slot] = a;
    ws.slot_weight[slot] = tw[a];
  }
  ws.assign_slot[a] = slot;
  return slot;
}

__global__ void assign_slots_kernel(const int32_t* __restrict__ ids, const float* __restrict__ tw,
                                    int A, int k, int E, WsPtrs ws) {
  ptx::pdl_wait();
  for (int a = blockIdx.x * blockDim.x + threadIdx.x; a < A; a += gridDim.x * blockDim.x)
    assign_slot(a, k, E, ids, tw, ws, kBN);
}

// ---------------------------------------------------------------------------
// Quantise one token row per block and scatter it to the token's k workspace rows.
// A thread owns 8 consecutive elements; 4 adjacent threads form one 32-group.
// The row is quantised into shared memory (and the token's fp32 combine row
// cleared) while the bucketing kernel may still be running; the block then waits
// for it, gives the token's k assignments their rows and copies the row to each.
// Token row formats of pre_dispatch.
enum TokenFormat { kTokMxfp4 = 0, kTokMxfp8 = 1, kTokNvfp4 = 2 };

// FMT kTokMxfp8: one E4M3 byte per element, scale rule amax <= 448 * 2^e (fp8xfp4);
// kTokNvfp4: packed E2M1 with an E4M3 scale per 16 elements (nvf4xnvf4); kTokMxfp4:
// packed E2M1, amax <= 6 * 2^e per 32.
template <int FMT>
__global__ void __launch_bounds__(256) quantize_scatter_kernel(const __nv_bfloat16* __restrict__ x,
                                                               const int32_t* __restrict__ ids,
                                                               const float* __restrict__ tw,
                                                               int H, int k, int E, WsPtrs ws,
                                                               bool pull, int tile_rows) {
  constexpr bool F8 = FMT == kTokMxfp8, NV = FMT == kTokNvfp4;
  constexpr int kBytesPer8 = F8 ? 8 : 4;                // code bytes of 8 elements
  constexpr int kGroup = NV ? 16 : 32;                  // elements per scale
  extern __shared__ __align__(16) uint8_t qsh[];       // [row codes | H/kGroup scales]
  __shared__ int32_t slots[32];
  const int row_bytes_q = H / 8 * kBytesPer8;
  uint8_t* codes_sh = qsh;
  uint8_t* sf_sh = qsh + row_bytes_q;
  const int t = blockIdx.x, tid = threadIdx.x;
  ptx::pdl_launch_dependents();
  {
    // The down projection adds this token's k contributions into its fp32 row.
    float4* acc = reinterpret_cast<float4*>(ws.acc + (size_t)t * H);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = tid; i < H / 4; i += blockDim.x) acc[i] = z;
  }
  // Every lane of a warp runs every round (the shuffles below need all 32): H is a
  // multiple of 128, so a round can end mid-warp (H = 384: lanes 16-31 of warp 1 are
  // past the row); those lanes work on zeros and store nothing.
  for (int round0 = 0; round0 < H; round0 += blockDim.x * 8) {
    const int base = round0 + tid * 8;
    const bool live = base < H;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (live) raw = *reinterpret_cast<const uint4*>(x + (size_t)t * H + base);
    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(p2[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    if (NV) {
      // 16-element group = this lane and its neighbour: scale = E4M3(amax / 6),
      // elements fp32(x / scale) (signed zeros when the scale is zero)
      const uint32_t sb = ptx::nvfp4_scale_byte(amax);
      const float sc = ptx::ue4m3_value(sb);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = sc > 0.f ? __fdiv_rn(v[i], sc) : copysignf(0.f, v[i]);
      const uint32_t c8 = ptx::e2m1x8(v);
      if (!live) continue;
      *reinterpret_cast<uint32_t*>(codes_sh + base / 2) = c8;
      if ((tid & 1) == 0) sf_sh[base / 16] = (uint8_t)sb;
      continue;
    }
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    const int e = F8 ? ptx::mxfp8_exponent(amax) : ptx::mx_scale_exponent(amax);
    const float inv = ptx::pow2_neg(e);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] *= inv;
    const uint8_t sb = (uint8_t)(e + 127);
    if (F8) {
      const uint2 c8 = ptx::e4m3x8(v);
      if (!live) continue;
      *reinterpret_cast<uint2*>(codes_sh + base) = c8;
      if ((tid & 3) == 0) sf_sh[base / 32] = sb;
      continue;
    }
    const uint32_t c8 = ptx::e2m1x8(v);
    if (!live) continue;
    if (pull) {
      // the token's one row, gathered by the layer kernel for each of its experts
      *reinterpret_cast<uint32_t*>(ws.xq + (size_t)t * (H / 2) + base / 2) = c8;
      if ((tid & 3) == 0) ws.xs[(size_t)t * (H / 32) + base / 32] = sb;
    } else {
      *reinterpret_cast<uint32_t*>(codes_sh + base / 2) = c8;
      if ((tid & 3) == 0) sf_sh[base / 32] = sb;
    }
  }
  ptx::pdl_wait();
  if (tid < k) slots[tid] = assign_slot(t * k + tid, k, E, ids, tw, ws, tile_rows);
  if (pull) return;
  __syncthreads();
  const int nsf = H / kGroup;      // scale bytes of a row
  const int kc4 = nsf / 4;
  const int sf_rows = tile_rows > kBN ? kBN : tile_rows;   // pair tiles: whole 128-row blocks
  const size_t row_bytes = (size_t)row_bytes_q;
  for (int j = 0; j < k; ++j) {
    const int slot = slots[j];
    if (slot < 0) continue;
    uint4* dst = reinterpret_cast<uint4*>(ws.xb + (size_t)slot * row_bytes);
    for (int i = tid; i < row_bytes_q / 16; i += blockDim.x)   // 16-byte chunks of the row
      dst[i] = reinterpret_cast<const uint4*>(codes_sh)[i];
    for (int i = tid; i < nsf; i += blockDim.x)
      ws.xsf[sf_tile_offset((size_t)slot, i, kc4, sf_rows)] = sf_sh[i];
  }
}

// fp32 rows -> canonical MXFP4 codes/scales.  A thread owns 8 elements.
__global__ void quantize_rows_kernel(const float* __restrict__ src, int64_t n_threads,
                                     uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // n_threads is a multiple of 4, so a 4-lane group is either wholly in range or
  // wholly past the end; lanes past the end work on a clamped copy and store nothing.
  const int64_t ic = i < n_threads ? i : n_threads - 1;
  const int64_t elem = ic * 8;
  const float4 a = *reinterpret_cast<const float4*>(src + elem);
  const float4 b = *reinterpret_cast<const float4*>(src + elem + 4);
  float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
  const int e = ptx::mx_scale_exponent(amax);
  const float inv = ptx::pow2_neg(e);
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] *= inv;
  const uint32_t c = ptx::e2m1x8(v);
  if (i < n_threads) {
    reinterpret_cast<uint32_t*>(codes)[ic] = c;
    if ((ic & 3) == 0) sf[elem / 32] = (uint8_t)(e + 127);
  }
}

// fp32 rows -> canonical NVFP4 codes/scales (one E4M3 scale per 16 elements).  A
// thread owns 8 elements; a lane pair shares a group.
__global__ void quantize_rows_nv_kernel(const float* __restrict__ src, int64_t n_threads,
                                        uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // n_threads is even, so a lane pair is wholly in range or wholly past the end
  const int64_t ic = i < n_threads ? i : n_threads - 1;
  const int64_t elem = ic * 8;
  const float4 a = *reinterpret_cast<const float4*>(src + elem);
  const float4 b = *reinterpret_cast<const float4*>(src + elem + 4);
  float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
  amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
  const uint32_t sb = ptx::nvfp4_scale_byte(amax);
  const float sc = ptx::ue4m3_value(sb);
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = sc > 0.f ? __fdiv_rn(v[j], sc) : copysignf(0.f, v[j]);
  const uint32_t c = ptx::e2m1x8(v);
  if (i < n_threads) {
    reinterpret_cast<uint32_t*>(codes)[ic] = c;
    if ((ic & 1) == 0) sf[elem / 16] = (uint8_t)sb;
  }
}

// Canonical codes [E*rows, row_bytes] -> k-block tiles (the layout of
// weight_code_bytes), with the optional gate/up interleave (interleave: 0 none, 16 or
// 8 the granule): 16 bytes per thread, written in tile order.  Bytes past a row's
// end (a short last k-block) are zero.
__global__ void tile_codes_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                  int64_t total_chunks, int row_bytes, int kb_bytes, int num_kb,
                                  int rows_per_expert, int I, int interleave) {
  const int cpr = kb_bytes / 16;   // 16-byte chunks a tile row
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < total_chunks;
       c += (int64_t)gridDim.x * blockDim.x) {
    const int part = (int)(c % cpr);
    const int64_t trow = c / cpr;                     // tile row, over all tiles
    const int64_t tile = trow >> 7;
    const int kb = (int)(tile % num_kb);
    const int64_t row = (tile / num_kb) * 128 + (trow & 127);   // weight row over E*rows
    const int64_t e = row / rows_per_expert;
    const int r = (int)(row % rows_per_expert);
    const int sr = interleave ? gate_up_source_row_for(r, I, interleave == 8) : r;
    const int j = kb * kb_bytes + part * 16;          // byte of the row
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (j < row_bytes)
      v = *reinterpret_cast<const uint4*>(src + ((size_t)e * rows_per_expert + sr) *
                                                    (size_t)row_bytes + j);
    reinterpret_cast<uint4*>(dst)[c] = v;
  }
}

// Canonical scales [E*rows, Kc] -> 128x4 blocks, one int32 (4 scale columns of one
// row) per thread, written in block order.
__global__ void scale_blocks_kernel(const uint8_t* __restrict__ src, uint32_t* __restrict__ dst,
                                    int64_t total_words, int rows_per_expert, int Kc, int I,
                                    int interleave) {
  const int kc4 = Kc / 4;
  for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < total_words;
       w += (int64_t)gridDim.x * blockDim.x) {
    // word index = ((rb * kc4 + kb) * 32 + i) * 4 + q
    const int q = (int)(w & 3);
    const int i = (int)((w >> 2) & 31);
    const int64_t blk = w >> 7;
    const int kb = (int)(blk % kc4);
    const int64_t rb = blk / kc4;                       // 128-row block over E*rows
    const int64_t row = rb * 128 + q * 32 + i;          // row over E*rows
    const int64_t e = row / rows_per_expert;
    const int r = (int)(row % rows_per_expert);
    const int sr = interleave ? gate_up_source_row_for(r, I, interleave == 8) : r;
    const uint8_t* s = src + ((size_t)e * rows_per_expert + sr) * (size_t)Kc + 4 * kb;
    dst[w] = (uint32_t)s[0] | ((uint32_t)s[1] << 8) | ((uint32_t)s[2] << 16) |
             ((uint32_t)s[3] << 24);
  }
}

// acc fp32 -> bf16, 8 elements per thread.
__global__ void convert_out_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ out,
                                   int64_t n8) {
  ptx::pdl_wait();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4* a4 = reinterpret_cast<const float4*>(acc) + 2 * i;
    const float4 a = a4[0];
    const float4 b = a4[1];
    __nv_bfloat162 o[4] = {__floats2bfloat162_rn(a.x, a.y), __floats2bfloat162_rn(a.z, a.w),
                           __floats2bfloat162_rn(b.x, b.y), __floats2bfloat162_rn(b.z, b.w)};
    reinterpret_cast<uint4*>(out)[i] = *reinterpret_cast<const uint4*>(o);
  }
}

__global__ void wait_probe_kernel(int32_t* flags, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
    // phase 0 of `bar` never completes: nothing arrives on it
    const bool got_bar = ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns);
    abort_flag = 0;
    const bool got_count = ptx::wait_counter(&flags[kFlagProbe], 1, &abort_flag, limit_ns);
    if (!got_bar && !got_count) atomicOr(&flags[0], kErrTimeout);
  }
}

// Blocks for a grid-stride loop over `work` items, capped at `cap`.
unsigned grid_for(int64_t work, int block, int64_t cap) {
  int64_t g = (work + block - 1) / block;
  if (g > cap) g = cap;
  return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_bucket(const Shape& s, const int32_t* ids, int T, const WsPtrs& ws,
                          int tile_rows, cudaStream_t st) {
  const size_t smem = ((size_t)35 * s.E + kBucketChunk + 2) * sizeof(int32_t);
  cudaError_t err = cudaFuncSetAttribute(bucket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  const int A = T * s.k;
  bucket_kernel<<<(A + kBucketChunk - 1) / kBucketChunk, 1024, smem, st>>>(ids, T, s.k, s.E, ws,
                                                                            tile_rows);
  return cudaGetLastError();
}

cudaError_t launch_quantize_scatter(const Shape& s, const void* x, const int32_t* ids,
                                    const float* tw, int T, const WsPtrs& ws, bool pull,
                                    int tile_rows, cudaStream_t st) {
  const size_t smem = (size_t)(s.f8 ? s.H : s.H / 2) + s.H / sf_group(s);
  auto kern = s.f8   ? quantize_scatter_kernel<kTokMxfp8>
              : s.nv ? quantize_scatter_kernel<kTokNvfp4>
                     : quantize_scatter_kernel<kTokMxfp4>;
  if (smem > 48 * 1024) {   // wide rows (H up to 65536) need the opt-in limit
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(kern, dim3(T), dim3(256), smem, st, reinterpret_cast<const __nv_bfloat16*>(x),
                    ids, tw, s.H, s.k, s.E, ws, pull, tile_rows);
}

cudaError_t launch_assign_slots(const Shape& s, const int32_t* ids, const float* tw, int T,
                                const WsPtrs& ws, cudaStream_t st) {
  const int A = T * s.k;
  return launch_pdl(assign_slots_kernel, dim3(grid_for(A, 256, 4096)), dim3(256), 0, st, ids, tw,
                    A, s.k, s.E, ws);
}

cudaError_t launch_convert_out(const float* acc, void* out, int64_t n, cudaStream_t st) {
  const int64_t n8 = n / 8;
  return launch_pdl(convert_out_kernel, dim3(grid_for(n8, 256, 4096)), dim3(256), 0, st, acc,
                    reinterpret_cast<__nv_bfloat16*>(out), n8);
}

cudaError_t launch_wait_probe(int32_t* flags, unsigned long long limit_ns, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(flags, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const float* src, int64_t rows, int K, uint8_t* codes,
                                 uint8_t* sf, cudaStream_t st) {
  const int64_t n_threads = rows * (int64_t)K / 8;
  const int64_t blocks = (n_threads + 255) / 256;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  quantize_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(src, n_threads, codes, sf);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows_nv(const float* src, int64_t rows, int K, uint8_t* codes,
                                    uint8_t* sf, cudaStream_t st) {
  const int64_t n_threads = rows * (int64_t)K / 8;
  const int64_t blocks = (n_threads + 255) / 256;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  quantize_rows_nv_kernel<<<(unsigned)blocks, 256, 0, st>>>(src, n_threads, codes, sf);
  return cudaGetLastError();
}

cudaError_t launch_prepare(const Shape& s, const uint8_t* w1c, const uint8_t* w1s,
                           const uint8_t* w2c, const uint8_t* w2s, uint8_t* prep,
                           const PrepLayout& pl, cudaStream_t st) {
  const int64_t E = s.E, H = s.H, I = s.I;
  const int gran = s.f8 ? 8 : 16;   // gate/up interleave of the activation format
  const int kbb = weight_kb_bytes(s);
  {  // W1 codes: interleaved rows, k-block tiles
    const int64_t total = weight_code_bytes(s, E * 2 * I, H) / 16;
    tile_codes_kernel<<<grid_for(total, 256, 16384), 256, 0, st>>>(
        w1c, prep + pl.off_w1c, total, (int)(H / 2), kbb, (int)weight_num_kb(s, H), (int)(2 * I),
        (int)I, gran);
  }
  {  // W1 scales: interleaved rows, 128x4 blocks
    const int64_t words = E * 2 * I * (H / sf_group(s)) / 4;
    scale_blocks_kernel<<<grid_for(words, 256, 16384), 256, 0, st>>>(
        w1s, reinterpret_cast<uint32_t*>(prep + pl.off_w1s), words, (int)(2 * I),
        (int)(H / sf_group(s)), (int)I, gran);
  }
  {  // W2 codes: rows unchanged, k-block tiles
    const int64_t total = weight_code_bytes(s, E * H, I) / 16;
    tile_codes_kernel<<<grid_for(total, 256, 16384), 256, 0, st>>>(
        w2c, prep + pl.off_w2c, total, (int)(I / 2), kbb, (int)weight_num_kb(s, I), (int)H,
        (int)I, 0);
  }
  {  // W2 scales: 128x4 blocks
    const int64_t words = E * H * (I / sf_group(s)) / 4;
    scale_blocks_kernel<<<grid_for(words, 256, 16384), 256, 0, st>>>(
        w2s, reinterpret_cast<uint32_t*>(prep + pl.off_w2s), words, (int)H,
        (int)(I / sf_group(s)), (int)I, 0);
  }
  return cudaGetLastError();
}

}  // namespace mxmoe
