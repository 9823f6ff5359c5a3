// C ABI of libmxmoe (declared in include/mxmoe.h): argument checks, workspace and
// prepared-weight layouts, the workspace registry, launches, debug readback and
// timing hooks.  No entry point here allocates device memory.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "mxmoe.h"

using namespace mxmoe;

namespace {

thread_local std::string g_err;

moe_status fail(moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t kAlign = 1024;
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool dims_equal(const moe_dims& a, const moe_dims& b) {
  return a.hidden == b.hidden && a.inter == b.inter && a.num_experts == b.num_experts &&
         a.topk == b.topk && a.max_tokens == b.max_tokens && a.mma_type == b.mma_type;
}

// Bytes of one quantised activation row of K elements: packed E2M1 (two per byte)
// for mxf4xmxf4, one E4M3 byte each for fp8xfp4.
int64_t act_row_bytes(const moe_dims& d, int64_t K) {
  return d.mma_type == MOE_MMA_FP8xFP4 ? K : K / 2;
}

// Scale bytes of one row of K elements: one E4M3 byte per 16 for nvf4xnvf4, one
// UE8M0 byte per 32 otherwise.
int64_t sf_row_bytes(const moe_dims& d, int64_t K) {
  return d.mma_type == MOE_MMA_NVF4xNVF4 ? K / 16 : K / 32;
}

WsLayout ws_layout(const moe_dims& d) {
  WsLayout L;
  const int64_t H = d.hidden, I = d.inter, E = d.num_experts, k = d.topk;
  L.T_cap = d.max_tokens;
  L.A_cap = L.T_cap * k;
  // Segments of the pair dispatch take up to 4/3 of their rows plus a 128-row tail
  // (segment_rows); every other dispatch at most its rows plus 127.
  L.R_cap = (int64_t)align_up((size_t)((L.A_cap * kPairStride + kBNPair - 1) / kBNPair), kBN) +
            (int64_t)kBN * E;
  L.tiles_cap = L.A_cap / kBNNarrow + E + 1;   // enough for narrow tiles too
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, kAlign);
    return at;
  };
  L.off_header = take(256);
  L.off_flags = take(64 * sizeof(int32_t));
  L.off_counts = take((size_t)E * 4);
  L.off_seg = take((size_t)(E + 1) * 4);
  L.off_tiles = take((size_t)L.tiles_cap * 16);
  L.off_tile_done = take((size_t)L.tiles_cap * 4);
  L.off_tile_start = take((size_t)(E + 1) * 4);
  L.off_assign = take((size_t)L.A_cap * 4);
  L.off_local_rank = take((size_t)L.A_cap * 4);
  L.off_blk_base = take((size_t)(L.A_cap / kBucketChunk + 1) * E * 4);
  L.off_slot_token = take((size_t)L.R_cap * 4);
  L.off_slot_assign = take((size_t)L.R_cap * 4);
  L.off_slot_weight = take((size_t)L.R_cap * 4);
  L.off_xb = take((size_t)L.R_cap * act_row_bytes(d, H));
  // scale blocks of wide tiles, or of narrow ones (a quarter of each block used)
  L.off_xsf = take((size_t)L.R_cap * sf_row_bytes(d, H) * 4);
  L.off_xq = take((size_t)L.T_cap * H / 2);
  L.off_xs = take((size_t)L.T_cap * H / 32);
  L.off_hb = take((size_t)L.R_cap * act_row_bytes(d, I));
  L.off_hsf = take((size_t)L.R_cap * sf_row_bytes(d, I) * 4);
  L.off_acc = take((size_t)L.T_cap * H * 4);
  L.off_stage_x = take((size_t)L.T_cap * H * 2);
  L.off_stage_ids = take((size_t)L.A_cap * 4);
  L.off_stage_w = take((size_t)L.A_cap * 4);
  L.off_stage_out = take((size_t)L.T_cap * H * 2);
  L.total = o;
  return L;
}

WsPtrs ws_ptrs(void* ws, const WsLayout& L) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  WsPtrs p;
  p.flags = reinterpret_cast<int32_t*>(b + L.off_flags);
  p.counts = reinterpret_cast<int32_t*>(b + L.off_counts);
  p.seg = reinterpret_cast<int32_t*>(b + L.off_seg);
  p.tiles = reinterpret_cast<int4*>(b + L.off_tiles);
  p.tile_done = reinterpret_cast<int32_t*>(b + L.off_tile_done);
  p.tile_start = reinterpret_cast<int32_t*>(b + L.off_tile_start);
  p.assign_slot = reinterpret_cast<int32_t*>(b + L.off_assign);
  p.local_rank = reinterpret_cast<int32_t*>(b + L.off_local_rank);
  p.blk_base = reinterpret_cast<int32_t*>(b + L.off_blk_base);
  p.slot_token = reinterpret_cast<int32_t*>(b + L.off_slot_token);
  p.slot_assign = reinterpret_cast<int32_t*>(b + L.off_slot_assign);
  p.slot_weight = reinterpret_cast<float*>(b + L.off_slot_weight);
  p.xb = b + L.off_xb;
  p.xsf = b + L.off_xsf;
  p.xq = b + L.off_xq;
  p.xs = b + L.off_xs;
  p.hb = b + L.off_hb;
  p.hsf = b + L.off_hsf;
  p.acc = reinterpret_cast<float*>(b + L.off_acc);
  return p;
}

Shape shape_of(const moe_dims& d) {
  return Shape{d.hidden, d.inter, d.num_experts, d.topk, d.mma_type == MOE_MMA_FP8xFP4 ? 1 : 0,
               d.mma_type == MOE_MMA_NVF4xNVF4 ? 1 : 0};
}

// Codes in k-block tiles (weight_code_bytes), then the scales in 128x4 blocks.
PrepLayout prep_layout(const moe_dims& d) {
  PrepLayout P;
  const size_t H = d.hidden, I = d.inter, E = d.num_experts;
  const Shape s = shape_of(d);
  size_t o = 0;
  P.off_w1c = o;
  o = align_up(o + (size_t)weight_code_bytes(s, (int64_t)(E * 2 * I), (int64_t)H), kAlign);
  P.off_w1s = o;
  o = align_up(o + E * 2 * I * (size_t)sf_row_bytes(d, (int64_t)H), kAlign);
  P.off_w2c = o;
  o = align_up(o + (size_t)weight_code_bytes(s, (int64_t)(E * H), (int64_t)I), kAlign);
  P.off_w2s = o;
  o = align_up(o + E * H * (size_t)sf_row_bytes(d, (int64_t)I), kAlign);
  P.total = o;
  return P;
}

// Workspaces initialised by moe_workspace_init, with the dims they were laid out for
// and whether their accumulator holds a fresh pre_dispatch (cleared rows, no sums
// yet): moe_pre_dispatch sets it, moe_forward consumes it.
struct WsState {
  moe_dims dims;
  bool dispatched;
  int dispatch_mode;   // MOE_DISPATCH_*
  int tile_mode;       // MOE_TILES_*
  int tile_rows;       // the last pre_dispatch's token rows a tile (32, 64 or 128)
};
std::mutex g_reg_mu;
std::map<const void*, WsState> g_registry;

// Dispatch mode of a registered workspace (bucketed copies if unknown).
int dispatch_mode(const void* ws) {
  std::lock_guard<std::mutex> lk(g_reg_mu);
  auto it = g_registry.find(ws);
  return it == g_registry.end() ? MOE_DISPATCH_BUCKETED : it->second.dispatch_mode;
}

// Marks the workspace's pre_dispatch as consumed; returns whether it was fresh.
bool take_dispatch(const void* ws) {
  std::lock_guard<std::mutex> lk(g_reg_mu);
  auto it = g_registry.find(ws);
  if (it == g_registry.end()) return false;
  const bool fresh = it->second.dispatched;
  it->second.dispatched = false;
  return fresh;
}

void mark_dispatched(const void* ws, int tile_rows) {
  std::lock_guard<std::mutex> lk(g_reg_mu);
  auto it = g_registry.find(ws);
  if (it != g_registry.end()) {
    it->second.dispatched = true;
    it->second.tile_rows = tile_rows;
  }
}

// Token rows a tile of a workspace's last pre_dispatch (128 if unknown).
int tile_rows_of(const void* ws) {
  std::lock_guard<std::mutex> lk(g_reg_mu);
  auto it = g_registry.find(ws);
  return it == g_registry.end() ? kBN : it->second.tile_rows;
}

int tile_mode(const void* ws) {
  std::lock_guard<std::mutex> lk(g_reg_mu);
  auto it = g_registry.find(ws);
  return it == g_registry.end() ? MOE_TILES_AUTO : it->second.tile_mode;
}

// Token rows a tile: as asked for, or (auto) by the experts' average rows: up to 16,
// 32-row tiles (decode-sized loads); up to 64, 64-row tiles; else 128.  Smaller tiles
// keep more weight bytes in flight but stream an expert's weights once per tile, so
// each size wins where few experts need more than one tile.  The pull dispatch
// gathers into 128-row tiles only.
int choose_tile_rows(const moe_dims& d, int32_t T, int mode, bool pull) {
  const bool pair_ok = !pull && pair_shape_ok(shape_of(d));
  if (pull || mode == MOE_TILES_WIDE) return kBN;
  if (mode == MOE_TILES_NARROW) return kBNNarrow;
  if (mode == MOE_TILES_MEDIUM) return kBNMedium;
  if (mode == MOE_TILES_PAIR) return pair_ok ? kBNPair : kBN;
  const int64_t rows = (int64_t)T * d.topk, E = d.num_experts;
  return rows <= 16 * E ? kBNNarrow : rows <= 64 * E ? kBNMedium : kBN;
}

// Token rows of a 128x4 scale block's tile in the layout of a dispatch with tiles of
// tile_rows rows (pair tiles are two whole 128-row blocks).
int sf_layout_rows(int tile_rows) { return tile_rows > kBN ? kBN : tile_rows; }

cudaError_t launch_any_layer(const LayerLaunch& g, cudaStream_t st) {
  return g.tile_rows == kBNPair ? launch_layer_pair(g, st) : launch_layer(g, st);
}

// Timing hooks.
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
struct ProfSum {
  double ms = 0.0;
  int launches = 0;
  const char* name = nullptr;
};
std::map<std::string, ProfSum> g_prof_done;

struct ProfScope {
  const char* name;
  cudaStream_t st;
  cudaEvent_t a = nullptr;
  ProfScope(const char* n, cudaStream_t s) : name(n), st(s) {
    if (!g_prof_on) return;
    if (cudaEventCreate(&a) == cudaSuccess)
      cudaEventRecord(a, st);
    else
      a = nullptr;
  }
  ~ProfScope() {
    if (!a) return;
    cudaEvent_t b = nullptr;
    if (cudaEventCreate(&b) == cudaSuccess) {
      cudaEventRecord(b, st);
      std::lock_guard<std::mutex> lk(g_prof_mu);
      g_prof.push_back({name, a, b});
    } else {
      cudaEventDestroy(a);
    }
  }
};

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

moe_status check_dims(const moe_dims* d) {
  if (!d) return fail(MOE_ERR_INVALID_ARG, "dims is NULL");
  if (d->mma_type != MOE_MMA_MXF4xMXF4 && d->mma_type != MOE_MMA_FP8xFP4 &&
      d->mma_type != MOE_MMA_NVF4xNVF4)
    return fail(MOE_ERR_UNSUPPORTED,
                "mma_type %d: MOE_MMA_MXF4xMXF4, MOE_MMA_FP8xFP4 and MOE_MMA_NVF4xNVF4 are built",
                d->mma_type);
  if (d->hidden < 256 || d->hidden % 128 != 0 || d->hidden > 65536)
    return fail(MOE_ERR_INVALID_ARG, "hidden %d must be a multiple of 128 in [256, 65536]",
                d->hidden);
  if (d->inter < 128 || d->inter % 128 != 0 || d->inter > 65536)
    return fail(MOE_ERR_INVALID_ARG, "inter %d must be a multiple of 128 in [128, 65536]",
                d->inter);
  if (d->num_experts < 1 || d->num_experts > 1024)
    return fail(MOE_ERR_INVALID_ARG, "num_experts %d outside [1, 1024]", d->num_experts);
  if (d->topk < 1 || d->topk > 32 || d->topk > d->num_experts)
    return fail(MOE_ERR_INVALID_ARG, "topk %d outside [1, min(num_experts, 32)]", d->topk);
  if (d->max_tokens < 1 || d->max_tokens > 65536)
    return fail(MOE_ERR_INVALID_ARG, "max_tokens %d outside [1, 65536]", d->max_tokens);
  return MOE_OK;
}

moe_status check_ws(const moe_dims* d, const void* ws, size_t ws_bytes) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  const size_t need = ws_layout(*d).total;
  if (ws_bytes < need)
    return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  std::lock_guard<std::mutex> lk(g_reg_mu);
  auto it = g_registry.find(ws);
  if (it == g_registry.end())
    return fail(MOE_ERR_WORKSPACE_MISMATCH,
                "workspace %p was not initialised by moe_workspace_init", ws);
  if (!dims_equal(it->second.dims, *d))
    return fail(MOE_ERR_WORKSPACE_MISMATCH,
                "workspace %p was initialised for other dims or mma_type", ws);
  return MOE_OK;
}

moe_status check_tokens(const moe_dims* d, int32_t T) {
  if (T < 0 || T > d->max_tokens)
    return fail(MOE_ERR_INVALID_ARG, "num_tokens %d outside [0, max_tokens=%d]", T,
                d->max_tokens);
  return MOE_OK;
}

__global__ void write_header_kernel(int32_t* hdr, moe_dims d, unsigned long long total) {
  hdr[0] = 0x454F4D58;  // "XMOE"
  hdr[1] = 1;           // layout version
  hdr[2] = d.hidden;
  hdr[3] = d.inter;
  hdr[4] = d.num_experts;
  hdr[5] = d.topk;
  hdr[6] = d.max_tokens;
  hdr[7] = d.mma_type;
  *reinterpret_cast<unsigned long long*>(hdr + 8) = total;
}

moe_status pre_dispatch_impl(const moe_dims* d, const void* x, const int32_t* ids,
                             const float* tw, int32_t T, void* ws, cudaStream_t st) {
  const WsLayout L = ws_layout(*d);
  const WsPtrs p = ws_ptrs(ws, L);
  const Shape s = shape_of(*d);
  const bool pull = dispatch_mode(ws) == MOE_DISPATCH_PULL;
  const int tile_rows = choose_tile_rows(*d, T, tile_mode(ws), pull);
  cudaError_t e;
  {
    ProfScope ps("bucket", st);
    e = launch_bucket(s, ids, T, p, tile_rows, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "bucket kernel");
  {
    ProfScope ps("quantize_scatter", st);
    e = launch_quantize_scatter(s, x, ids, tw, T, p, pull, tile_rows, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "quantize kernel");
  mark_dispatched(ws, tile_rows);
  return MOE_OK;
}

LayerLaunch layer_launch(const moe_dims* d, const void* prepared, void* ws, int32_t T) {
  const WsLayout L = ws_layout(*d);
  const PrepLayout P = prep_layout(*d);
  const uint8_t* prep = static_cast<const uint8_t*>(prepared);
  LayerLaunch g;
  g.w1_codes = prep + P.off_w1c;
  g.w1_sf = prep + P.off_w1s;
  g.w2_codes = prep + P.off_w2c;
  g.w2_sf = prep + P.off_w2s;
  g.R_cap = L.R_cap;
  g.shape = shape_of(*d);
  g.T = T;
  g.num_phases = 2;
  g.ws = ws_ptrs(ws, L);
  g.gate_up_debug = nullptr;
  g.num_sms = sm_count();
  g.pull = dispatch_mode(ws) == MOE_DISPATCH_PULL;
  g.tile_rows = tile_rows_of(ws);
  return g;
}

moe_status forward_impl(const moe_dims* d, const void* prepared, void* ws, void* out, int32_t T,
                        cudaStream_t st) {
  LayerLaunch g = layer_launch(d, prepared, ws, T);
  if (g.num_sms <= 0) return fail(MOE_ERR_CUDA, "no CUDA device");
  cudaError_t e;
  if (!take_dispatch(ws)) {
    // A second forward on the same pre_dispatch: its rows still hold the first
    // call's sums, so clear them before adding again.
    e = cudaMemsetAsync(g.ws.acc, 0, (size_t)T * d->hidden * sizeof(float), st);
    if (e != cudaSuccess) return cuda_fail(e, "accumulator clear");
  }
  {
    ProfScope ps("layer", st);
    e = launch_any_layer(g, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "layer kernel");
  {
    ProfScope ps("convert_out", st);
    e = launch_convert_out(g.ws.acc, out, (int64_t)T * d->hidden, st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "output conversion");
  return MOE_OK;
}

}  // namespace

void mxmoe::set_last_error(const char* msg) { g_err = msg; }

extern "C" {

const char* moe_last_error(void) { return g_err.c_str(); }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_WORKSPACE_MISMATCH: return "MOE_ERR_WORKSPACE_MISMATCH";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_ROUTING: return "MOE_ERR_ROUTING";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

moe_status moe_validate_dims(const moe_dims* dims) { return check_dims(dims); }

size_t moe_prepared_weights_size(const moe_dims* dims) {
  if (check_dims(dims) != MOE_OK) return 0;
  return prep_layout(*dims).total;
}

size_t moe_workspace_size(const moe_dims* dims) {
  if (check_dims(dims) != MOE_OK) return 0;
  return ws_layout(*dims).total;
}

moe_status moe_workspace_init(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream) {
  moe_status s = check_dims(dims);
  if (s) return s;
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  const WsLayout L = ws_layout(*dims);
  if (ws_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE_TOO_SMALL, "workspace has %zu bytes, needs %zu", ws_bytes,
                L.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, L.total, st);
  if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
  write_header_kernel<<<1, 1, 0, st>>>(static_cast<int32_t*>(ws), *dims,
                                       (unsigned long long)L.total);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "workspace header");
  std::lock_guard<std::mutex> lk(g_reg_mu);
  g_registry[ws] = WsState{*dims, false, MOE_DISPATCH_BUCKETED, MOE_TILES_AUTO, kBN};
  return MOE_OK;
}

moe_status moe_workspace_set_dispatch(void* ws, int32_t mode) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if (mode != MOE_DISPATCH_BUCKETED && mode != MOE_DISPATCH_PULL)
    return fail(MOE_ERR_INVALID_ARG, "unknown dispatch mode %d", mode);
  std::lock_guard<std::mutex> lk(g_reg_mu);
  auto it = g_registry.find(ws);
  if (it == g_registry.end())
    return fail(MOE_ERR_WORKSPACE_MISMATCH, "workspace %p was not initialised", ws);
  if (mode == MOE_DISPATCH_PULL && it->second.dims.mma_type != MOE_MMA_MXF4xMXF4)
    return fail(MOE_ERR_UNSUPPORTED, "pull dispatch is built for mxf4xmxf4 only");
  it->second.dispatch_mode = mode;
  it->second.dispatched = false;   // a pre_dispatch in the new mode must come first
  return MOE_OK;
}

moe_status moe_workspace_set_tiles(void* ws, int32_t mode) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if (mode != MOE_TILES_AUTO && mode != MOE_TILES_WIDE && mode != MOE_TILES_NARROW &&
      mode != MOE_TILES_MEDIUM && mode != MOE_TILES_PAIR)
    return fail(MOE_ERR_INVALID_ARG, "unknown tile mode %d", mode);
  std::lock_guard<std::mutex> lk(g_reg_mu);
  auto it = g_registry.find(ws);
  if (it == g_registry.end())
    return fail(MOE_ERR_WORKSPACE_MISMATCH, "workspace %p was not initialised", ws);
  it->second.tile_mode = mode;
  it->second.dispatched = false;   // a pre_dispatch in the new mode must come first
  return MOE_OK;
}

moe_status moe_quantize_mxfp4(const float* src, int64_t rows, int32_t K, uint8_t* codes,
                              uint8_t* scales, void* stream) {
  if (rows < 0 || K <= 0 || K % 32 != 0)
    return fail(MOE_ERR_INVALID_ARG, "rows %lld / K %d: need rows >= 0 and K %% 32 == 0",
                (long long)rows, K);
  if (rows == 0) return MOE_OK;
  if (!src || !codes || !scales) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(src, 16) || !aligned(codes, 4))
    return fail(MOE_ERR_INVALID_ARG, "src must be 16-byte and codes 4-byte aligned");
  cudaError_t e =
      launch_quantize_rows(src, rows, K, codes, scales, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize kernel");
  return MOE_OK;
}

moe_status moe_quantize_nvfp4(const float* src, int64_t rows, int32_t K, uint8_t* codes,
                              uint8_t* scales, void* stream) {
  if (rows < 0 || K <= 0 || K % 16 != 0)
    return fail(MOE_ERR_INVALID_ARG, "rows %lld / K %d: need rows >= 0 and K %% 16 == 0",
                (long long)rows, K);
  if (rows == 0) return MOE_OK;
  if (!src || !codes || !scales) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(src, 16) || !aligned(codes, 4))
    return fail(MOE_ERR_INVALID_ARG, "src must be 16-byte and codes 4-byte aligned");
  cudaError_t e =
      launch_quantize_rows_nv(src, rows, K, codes, scales, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize kernel");
  return MOE_OK;
}

moe_status moe_prepare_weights(const moe_dims* dims, const uint8_t* w1c, const uint8_t* w1s,
                               const uint8_t* w2c, const uint8_t* w2s, void* prepared,
                               size_t prepared_bytes, void* stream) {
  moe_status s = check_dims(dims);
  if (s) return s;
  if (!w1c || !w1s || !w2c || !w2s || !prepared)
    return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(w1c, 16) || !aligned(w2c, 16) || !aligned(prepared, 256))
    return fail(MOE_ERR_INVALID_ARG,
                "weight codes must be 16-byte aligned and the prepared blob 256-byte aligned");
  const PrepLayout P = prep_layout(*dims);
  if (prepared_bytes < P.total)
    return fail(MOE_ERR_INVALID_ARG, "prepared blob has %zu bytes, needs %zu", prepared_bytes,
                P.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_prepare(shape_of(*dims), w1c, w1s, w2c, w2s,
                                 static_cast<uint8_t*>(prepared), P, st);
  if (e != cudaSuccess) return cuda_fail(e, "weight preparation");
  return MOE_OK;
}

moe_status moe_pre_dispatch(const moe_dims* dims, const void* x, const int32_t* ids,
                            const float* tw, int32_t T, void* ws, size_t ws_bytes, void* stream) {
  moe_status s = check_dims(dims);
  if (s) return s;
  if ((s = check_tokens(dims, T))) return s;
  if ((s = check_ws(dims, ws, ws_bytes))) return s;
  if (T == 0) return MOE_OK;
  if (!x || !ids || !tw) return fail(MOE_ERR_INVALID_ARG, "NULL input pointer");
  if (!aligned(x, 16) || !aligned(ids, 4) || !aligned(tw, 4))
    return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned, ids/weights 4-byte aligned");
  return pre_dispatch_impl(dims, x, ids, tw, T, ws, static_cast<cudaStream_t>(stream));
}

moe_status moe_forward(const moe_dims* dims, const void* prepared, void* ws, size_t ws_bytes,
                       void* out, int32_t T, void* stream) {
  moe_status s = check_dims(dims);
  if (s) return s;
  if ((s = check_tokens(dims, T))) return s;
  if ((s = check_ws(dims, ws, ws_bytes))) return s;
  if (T == 0) return MOE_OK;
  if (!prepared || !out) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(prepared, 256) || !aligned(out, 16))
    return fail(MOE_ERR_INVALID_ARG, "prepared must be 256-byte and out 16-byte aligned");
  return forward_impl(dims, prepared, ws, out, T, static_cast<cudaStream_t>(stream));
}

// Device address of a host buffer the GPU can access directly (page-locked, e.g.
// cudaHostAlloc / cudaHostRegister), 16-byte aligned; nullptr otherwise.
void* device_alias(const void* host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    (void)cudaGetLastError();   // not a CUDA-known pointer: not an error here
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer || !aligned(a.devicePointer, 16))
    return nullptr;
  return a.devicePointer;
}

moe_status moe_run_host(const moe_dims* dims, const void* prepared, void* ws, size_t ws_bytes,
                        const void* x_host, const int32_t* ids_host, const float* tw_host,
                        void* out_host, int32_t T, void* stream) {
  moe_status s = check_dims(dims);
  if (s) return s;
  if ((s = check_tokens(dims, T))) return s;
  if ((s = check_ws(dims, ws, ws_bytes))) return s;
  if (T == 0) return MOE_OK;
  if (!prepared || !x_host || !ids_host || !tw_host || !out_host)
    return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(prepared, 256)) return fail(MOE_ERR_INVALID_ARG, "prepared not 256-byte aligned");
  const WsLayout L = ws_layout(*dims);
  uint8_t* b = static_cast<uint8_t*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t xbytes = (size_t)T * dims->hidden * 2, abytes = (size_t)T * dims->topk * 4;
  cudaError_t e;
  // Page-locked inputs are read by the dispatch kernels straight from host memory,
  // and a page-locked output buffer is written by the bf16 conversion directly;
  // other buffers go through staging copies.
  const void* x_dev = device_alias(x_host);
  const void* ids_dev = device_alias(ids_host);
  const void* tw_dev = device_alias(tw_host);
  void* out_dev = device_alias(out_host);
  if (!x_dev) {
    if ((e = cudaMemcpyAsync(b + L.off_stage_x, x_host, xbytes, cudaMemcpyHostToDevice, st)))
      return cuda_fail(e, "input copy");
    x_dev = b + L.off_stage_x;
  }
  if (!ids_dev) {
    if ((e = cudaMemcpyAsync(b + L.off_stage_ids, ids_host, abytes, cudaMemcpyHostToDevice, st)))
      return cuda_fail(e, "input copy");
    ids_dev = b + L.off_stage_ids;
  }
  if (!tw_dev) {
    if ((e = cudaMemcpyAsync(b + L.off_stage_w, tw_host, abytes, cudaMemcpyHostToDevice, st)))
      return cuda_fail(e, "input copy");
    tw_dev = b + L.off_stage_w;
  }
  s = pre_dispatch_impl(dims, x_dev, static_cast<const int32_t*>(ids_dev),
                        static_cast<const float*>(tw_dev), T, ws, st);
  if (s) return s;
  s = forward_impl(dims, prepared, ws, out_dev ? out_dev : b + L.off_stage_out, T, st);
  if (s) return s;
  if (!out_dev &&
      (e = cudaMemcpyAsync(out_host, b + L.off_stage_out, xbytes, cudaMemcpyDeviceToHost, st)))
    return cuda_fail(e, "output copy");
  if ((e = cudaStreamSynchronize(st))) return cuda_fail(e, "stream synchronize");
  return MOE_OK;
}

moe_status moe_check(void* ws, void* stream) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  moe_dims d;
  {
    std::lock_guard<std::mutex> lk(g_reg_mu);
    auto it = g_registry.find(ws);
    if (it == g_registry.end())
      return fail(MOE_ERR_WORKSPACE_MISMATCH, "workspace %p was not initialised", ws);
    d = it->second.dims;
  }
  const WsLayout L = ws_layout(d);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int32_t flag = 0;
  int32_t* dflag = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + L.off_flags);
  if ((e = cudaMemcpy(&flag, dflag, sizeof(flag), cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "flag read");
  if ((e = cudaMemset(dflag, 0, sizeof(int32_t)))) return cuda_fail(e, "flag clear");
  if (flag & kErrTimeout) return fail(MOE_ERR_TIMEOUT, "a device wait ran past its limit");
  if (flag & kErrRouting)
    return fail(MOE_ERR_ROUTING, "topk ids outside [0, num_experts) were skipped");
  return MOE_OK;
}

moe_status moe_read_dispatch(const moe_dims* dims, const void* ws, int32_t T, int32_t* counts_host,
                             int32_t* assign_host, uint8_t* xc_host, uint8_t* xs_host,
                             int32_t* slot_token_host) {
  moe_status s = check_dims(dims);
  if (s) return s;
  if ((s = check_tokens(dims, T))) return s;
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  const WsLayout L = ws_layout(*dims);
  const uint8_t* b = static_cast<const uint8_t*>(ws);
  const int E = dims->num_experts, k = dims->topk, H = dims->hidden;
  const int64_t A = (int64_t)T * k;
  cudaError_t e = cudaDeviceSynchronize();
  if (e) return cuda_fail(e, "synchronize");
  if (counts_host &&
      (e = cudaMemcpy(counts_host, b + L.off_counts, (size_t)E * 4, cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "counts read");
  std::vector<int32_t> assign((size_t)A);
  if (A &&
      (e = cudaMemcpy(assign.data(), b + L.off_assign, (size_t)A * 4, cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "assign read");
  if (assign_host) std::memcpy(assign_host, assign.data(), (size_t)A * 4);
  std::vector<int32_t> seg((size_t)E + 1);
  if ((e = cudaMemcpy(seg.data(), b + L.off_seg, (size_t)(E + 1) * 4, cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "seg read");
  const int64_t R = seg[E];
  if (R < 0 || R > L.R_cap) return fail(MOE_ERR_CUDA, "corrupt segment table");
  if (slot_token_host) {
    std::vector<int32_t> st((size_t)R);
    if (R && (e = cudaMemcpy(st.data(), b + L.off_slot_token, (size_t)R * 4,
                             cudaMemcpyDeviceToHost)))
      return cuda_fail(e, "slot read");
    for (int64_t a = 0; a < A; ++a)
      slot_token_host[a] = (assign[a] >= 0 && assign[a] < R) ? st[assign[a]] : -1;
  }
  if ((xc_host || xs_host) && dispatch_mode(ws) == MOE_DISPATCH_PULL) {
    // one row per token; an assignment's row is its token's
    std::vector<uint8_t> codes((size_t)T * H / 2), sf((size_t)T * H / 32);
    if (T && (e = cudaMemcpy(codes.data(), b + L.off_xq, codes.size(), cudaMemcpyDeviceToHost)))
      return cuda_fail(e, "codes read");
    if (T && (e = cudaMemcpy(sf.data(), b + L.off_xs, sf.size(), cudaMemcpyDeviceToHost)))
      return cuda_fail(e, "scales read");
    for (int64_t a = 0; a < A; ++a) {
      const bool ok = assign[a] >= 0 && assign[a] < R;
      const int64_t t = a / k;
      if (xc_host) {
        if (ok)
          std::memcpy(xc_host + a * (H / 2), codes.data() + (size_t)t * H / 2, (size_t)H / 2);
        else
          std::memset(xc_host + a * (H / 2), 0, (size_t)H / 2);
      }
      if (xs_host) {
        if (ok)
          std::memcpy(xs_host + a * (H / 32), sf.data() + (size_t)t * H / 32, (size_t)H / 32);
        else
          std::memset(xs_host + a * (H / 32), 0, (size_t)H / 32);
      }
    }
  } else if (xc_host || xs_host) {
    const size_t rb = (size_t)act_row_bytes(*dims, H);
    const int sfb = (int)sf_row_bytes(*dims, H);
    const int tr = sf_layout_rows(tile_rows_of(ws));
    std::vector<uint8_t> codes((size_t)R * rb), sf((size_t)R * sfb * (kBN / tr));
    if (R && (e = cudaMemcpy(codes.data(), b + L.off_xb, codes.size(), cudaMemcpyDeviceToHost)))
      return cuda_fail(e, "codes read");
    if (R && (e = cudaMemcpy(sf.data(), b + L.off_xsf, sf.size(), cudaMemcpyDeviceToHost)))
      return cuda_fail(e, "scales read");
    for (int64_t a = 0; a < A; ++a) {
      const int32_t r = assign[a];
      const bool ok = r >= 0 && r < R;
      if (xc_host) {
        if (ok)
          std::memcpy(xc_host + a * rb, codes.data() + (size_t)r * rb, rb);
        else
          std::memset(xc_host + a * rb, 0, rb);
      }
      if (xs_host)
        for (int g = 0; g < sfb; ++g)
          xs_host[a * sfb + g] = ok ? sf[sf_tile_offset((size_t)r, g, sfb / 4, tr)] : 0;
    }
  }
  return MOE_OK;
}

moe_status moe_read_intermediate(const moe_dims* dims, const void* ws, int32_t T,
                                 uint8_t* hc_host, uint8_t* hs_host) {
  moe_status s = check_dims(dims);
  if (s) return s;
  if ((s = check_tokens(dims, T))) return s;
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  const WsLayout L = ws_layout(*dims);
  const uint8_t* b = static_cast<const uint8_t*>(ws);
  const int E = dims->num_experts, k = dims->topk, I = dims->inter;
  const int64_t A = (int64_t)T * k;
  cudaError_t e = cudaDeviceSynchronize();
  if (e) return cuda_fail(e, "synchronize");
  std::vector<int32_t> assign((size_t)A), seg((size_t)E + 1);
  if (A &&
      (e = cudaMemcpy(assign.data(), b + L.off_assign, (size_t)A * 4, cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "assign read");
  if ((e = cudaMemcpy(seg.data(), b + L.off_seg, (size_t)(E + 1) * 4, cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "seg read");
  const int64_t R = seg[E];
  if (R < 0 || R > L.R_cap) return fail(MOE_ERR_CUDA, "corrupt segment table");
  const size_t rb = (size_t)act_row_bytes(*dims, I);
  const int sfb = (int)sf_row_bytes(*dims, I);
  const int tr = sf_layout_rows(tile_rows_of(ws));
  std::vector<uint8_t> codes((size_t)R * rb), sf((size_t)R * sfb * (kBN / tr));
  if (R && (e = cudaMemcpy(codes.data(), b + L.off_hb, codes.size(), cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "codes read");
  if (R && (e = cudaMemcpy(sf.data(), b + L.off_hsf, sf.size(), cudaMemcpyDeviceToHost)))
    return cuda_fail(e, "scales read");
  for (int64_t a = 0; a < A; ++a) {
    const int32_t r = assign[a];
    const bool ok = r >= 0 && r < R;
    if (hc_host) {
      if (ok)
        std::memcpy(hc_host + a * rb, codes.data() + (size_t)r * rb, rb);
      else
        std::memset(hc_host + a * rb, 0, rb);
    }
    if (hs_host)
      for (int g = 0; g < sfb; ++g)
        hs_host[a * sfb + g] = ok ? sf[sf_tile_offset((size_t)r, g, sfb / 4, tr)] : 0;
  }
  return MOE_OK;
}

moe_status moe_debug_gate_up(const moe_dims* dims, const void* prepared, void* ws,
                             size_t ws_bytes, float* gate_up, int32_t T, void* stream) {
  moe_status s = check_dims(dims);
  if (s) return s;
  if ((s = check_tokens(dims, T))) return s;
  if ((s = check_ws(dims, ws, ws_bytes))) return s;
  if (T == 0) return MOE_OK;
  if (!prepared || !gate_up) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned(prepared, 256)) return fail(MOE_ERR_INVALID_ARG, "prepared not 256-byte aligned");
  LayerLaunch g = layer_launch(dims, prepared, ws, T);
  if (g.num_sms <= 0) return fail(MOE_ERR_CUDA, "no CUDA device");
  g.num_phases = 1;
  g.gate_up_debug = gate_up;
  cudaError_t e = launch_any_layer(g, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gate/up GEMM (raw)");
  return MOE_OK;
}

moe_status moe_debug_wait_probe(void* ws, int64_t limit_ns, void* stream) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if (limit_ns < 1000 || limit_ns > 1000000000)
    return fail(MOE_ERR_INVALID_ARG, "limit_ns %lld outside [1 us, 1 s]", (long long)limit_ns);
  moe_dims d;
  {
    std::lock_guard<std::mutex> lk(g_reg_mu);
    auto it = g_registry.find(ws);
    if (it == g_registry.end())
      return fail(MOE_ERR_WORKSPACE_MISMATCH, "workspace %p was not initialised", ws);
    d = it->second.dims;
  }
  int32_t* flags = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + ws_layout(d).off_flags);
  cudaError_t e = launch_wait_probe(flags, (unsigned long long)limit_ns,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait probe");
  return MOE_OK;
}

size_t moe_mxfp8_scale_bytes(int64_t rows_cap, int64_t K, int32_t layout) {
  if (rows_cap < 0 || K <= 0 || K % 128 || (layout != MOE_SF_PACKED && layout != MOE_SF_128X4))
    return 0;
  return mxfp8_scale_bytes(rows_cap, K, layout);
}

moe_status moe_mxfp8_quantize(const void* x, int64_t rows, int64_t K, void* q, void* sf,
                              int32_t layout, int64_t rows_cap, void* stream) {
  constexpr int64_t kMax = (int64_t)1 << 23;
  constexpr int64_t kMaxK = (int64_t)65535 * 128;   // one grid row of blocks per 128 columns
  if (K <= 0 || K % 128 || K > kMaxK)
    return fail(MOE_ERR_INVALID_ARG,
                "K = %lld: must be a positive multiple of 128, at most 65535 * 128",
                (long long)K);
  if (rows < 0 || rows > rows_cap || rows_cap > kMax)
    return fail(MOE_ERR_INVALID_ARG, "rows = %lld, rows_cap = %lld: need 0 <= rows <= rows_cap <= 2^23",
                (long long)rows, (long long)rows_cap);
  if (layout != MOE_SF_PACKED && layout != MOE_SF_128X4)
    return fail(MOE_ERR_INVALID_ARG, "unknown scale layout %d", layout);
  if (!sf || !aligned(sf, 16)) return fail(MOE_ERR_INVALID_ARG, "sf must be a 16-byte aligned pointer");
  if (rows > 0 && (!x || !q || !aligned(x, 16) || !aligned(q, 16)))
    return fail(MOE_ERR_INVALID_ARG, "x and q must be 16-byte aligned pointers");
  cudaError_t e = launch_mxfp8_quantize(x, rows, K, q, sf, layout, rows_cap,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mxfp8 quantize");
  return MOE_OK;
}

moe_status moe_fp4_mma_probe(void* ws, int32_t n, int32_t blocks_per_sm, int32_t blocks,
                             int64_t mma_count, void* stream) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if (n != 32 && n != 64 && n != 128 && n != 256)
    return fail(MOE_ERR_INVALID_ARG, "n = %d: must be 32, 64, 128 or 256", n);
  if (blocks_per_sm != 1 && blocks_per_sm != 2)
    return fail(MOE_ERR_INVALID_ARG, "blocks_per_sm = %d: must be 1 or 2", blocks_per_sm);
  if (blocks_per_sm == 2 && n > 128)
    return fail(MOE_ERR_INVALID_ARG, "n = %d needs the whole tensor memory: blocks_per_sm = 1", n);
  if (blocks < 1 || blocks > 65536)
    return fail(MOE_ERR_INVALID_ARG, "blocks = %d outside [1, 65536]", blocks);
  if (mma_count < 1 || mma_count > ((int64_t)1 << 20))
    return fail(MOE_ERR_INVALID_ARG, "mma_count = %lld outside [1, 2^20]", (long long)mma_count);
  moe_dims d;
  {
    std::lock_guard<std::mutex> lk(g_reg_mu);
    auto it = g_registry.find(ws);
    if (it == g_registry.end())
      return fail(MOE_ERR_WORKSPACE_MISMATCH, "workspace %p was not initialised", ws);
    d = it->second.dims;
  }
  int32_t* flags = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + ws_layout(d).off_flags);
  cudaError_t e = launch_fp4_mma_probe(n, blocks_per_sm, blocks, (long long)mma_count, flags,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fp4 mma probe");
  return MOE_OK;
}

moe_status moe_fp4_mma_probe_pair(void* ws, int32_t n, int32_t pairs, int64_t mma_count,
                                  void* stream) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
  if (n < 32 || n > 256 || n % 32 != 0)
    return fail(MOE_ERR_INVALID_ARG, "n = %d: must be a multiple of 32 in [32, 256]", n);
  if (pairs < 1 || pairs > 32768)
    return fail(MOE_ERR_INVALID_ARG, "pairs = %d outside [1, 32768]", pairs);
  if (mma_count < 1 || mma_count > ((int64_t)1 << 20))
    return fail(MOE_ERR_INVALID_ARG, "mma_count = %lld outside [1, 2^20]", (long long)mma_count);
  moe_dims d;
  {
    std::lock_guard<std::mutex> lk(g_reg_mu);
    auto it = g_registry.find(ws);
    if (it == g_registry.end())
      return fail(MOE_ERR_WORKSPACE_MISMATCH, "workspace %p was not initialised", ws);
    d = it->second.dims;
  }
  int32_t* flags = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + ws_layout(d).off_flags);
  cudaError_t e = launch_fp4_mma_probe_pair(n, pairs, (long long)mma_count, flags,
                                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "fp4 mma pair probe");
  return MOE_OK;
}

moe_status moe_profile_enable(int32_t on) {
  g_prof_on = on != 0;
  return MOE_OK;
}

int32_t moe_profile_read(const char** names_out, float* ms_out, int32_t* launches_out,
                         int32_t max_kernels) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof);
  }
  for (auto& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess &&
        cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      std::lock_guard<std::mutex> lk(g_prof_mu);
      ProfSum& sum = g_prof_done[r.name];
      sum.ms += ms;
      sum.launches += 1;
      sum.name = r.name;
    }
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  std::lock_guard<std::mutex> lk(g_prof_mu);
  int32_t n = 0;
  for (auto& kv : g_prof_done) {
    if (n >= max_kernels) break;
    if (names_out) names_out[n] = kv.second.name;
    if (ms_out) ms_out[n] = (float)kv.second.ms;
    if (launches_out) launches_out[n] = kv.second.launches;
    ++n;
  }
  return n;
}

void moe_profile_reset(void) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof);
    g_prof_done.clear();
  }
  for (auto& r : recs) {
    cudaEventSynchronize(r.b);
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
}

int32_t moe_device_sm_count(void) { return sm_count(); }

}  // extern "C"
