// moe_bucket_noalloc: the routing/bucketing step with its scratch in a fixed device
// array that the library owns, for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc on the path that routes tokens: runtimes that
// plan every device buffer up front and forbid allocation afterwards, and
// latency-critical threads for which cudaMalloc's implicit device-wide
// synchronisation is unacceptable.  They pass only their inputs and outputs; the
// bucketing kernels' other buffers (segment starts, tile list and tile counters,
// per-chunk ranks and bases, per-row slot tables, flags) live in g_bucket_scratch
// below.  The kernels are the ones moe_pre_dispatch launches; only where their
// scratch lives differs.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "mxmoe.h"

namespace mxmoe {
namespace {

// Limits of the static scratch: at most 8192 assignments (num_tokens * topk, one
// chunk of the bucketing kernel) and 256 experts per call.
constexpr int64_t kMaxAssignments = 8192;
constexpr int64_t kMaxExperts = 256;
constexpr int64_t kMaxRows = kMaxAssignments + (int64_t)kBN * kMaxExperts;
constexpr int64_t kMaxTiles = kMaxAssignments / kBN + kMaxExperts + 1;

constexpr size_t align256(size_t v) { return (v + 255) / 256 * 256; }
constexpr size_t kOffFlags = 0;
constexpr size_t kOffSeg = kOffFlags + align256(64 * sizeof(int32_t));
constexpr size_t kOffTiles = kOffSeg + align256((kMaxExperts + 1) * sizeof(int32_t));
constexpr size_t kOffTileDone = kOffTiles + align256(kMaxTiles * sizeof(int4));
constexpr size_t kOffTileStart = kOffTileDone + align256(kMaxTiles * sizeof(int32_t));
constexpr size_t kOffLocalRank = kOffTileStart + align256((kMaxExperts + 1) * sizeof(int32_t));
constexpr size_t kOffBlkBase = kOffLocalRank + align256(kMaxAssignments * sizeof(int32_t));
constexpr size_t kOffSlotToken = kOffBlkBase + align256(kMaxExperts * sizeof(int32_t));
constexpr size_t kOffSlotAssign = kOffSlotToken + align256(kMaxRows * sizeof(int32_t));
constexpr size_t kOffSlotWeight = kOffSlotAssign + align256(kMaxRows * sizeof(int32_t));
constexpr size_t kScratchBytes = kOffSlotWeight + align256(kMaxRows * sizeof(float));  // ~0.5 MiB

// Every GPU that loads the library holds this array until the process exits.  All
// calls share it: it keeps the previous call's contents, and calls that overlap on
// the GPU (different streams, or different host threads on one device) race on it.
static __device__ __align__(256) unsigned char g_bucket_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// Per device: the array's device address and the context it was looked up in.  A
// device reset (cudaDeviceReset) or a rebuilt primary context reloads the module, so
// the address is looked up again whenever the current context is not the recorded one.
unsigned char* g_scratch_dev[kMaxDevices] = {};
void* g_scratch_ctx[kMaxDevices] = {};

typedef int (*CtxGetCurrentFn)(void**);   // cuCtxGetCurrent, through the runtime's entry point

// The current driver context (nullptr if it cannot be read).
void* current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static bool looked = false;
  if (!looked) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
    looked = true;
  }
  void* ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

// Device address of g_bucket_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, with that device current: once per device and context (the
// first call on a device, or the first after its context was rebuilt).
cudaError_t scratch_address(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  void* ctx = current_context();
  if (!g_scratch_dev[dev] || ctx == nullptr || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bucket_scratch);   // makes the device's context current
    if (e != cudaSuccess) return e;
    g_scratch_dev[dev] = static_cast<unsigned char*>(p);
    g_scratch_ctx[dev] = current_context();
  }
  *out = g_scratch_dev[dev];
  return cudaSuccess;
}

moe_status fail(moe_status s, const char* msg) {
  set_last_error(msg);
  return s;
}

}  // namespace
}  // namespace mxmoe

extern "C" moe_status moe_bucket_noalloc(const moe_dims* dims, const int32_t* topk_ids_dev,
                                         const float* topk_weights_dev, int32_t num_tokens,
                                         int32_t* counts_dev, int32_t* assign_slot_dev,
                                         void* stream) {
  using namespace mxmoe;
  // Bucketing reads only the expert count, top-k and mma_type of the dims.
  if (!dims) return fail(MOE_ERR_INVALID_ARG, "moe_bucket_noalloc: dims is NULL");
  if (dims->mma_type != MOE_MMA_MXF4xMXF4 && dims->mma_type != MOE_MMA_FP8xFP4 &&
      dims->mma_type != MOE_MMA_NVF4xNVF4)
    return fail(MOE_ERR_UNSUPPORTED, "moe_bucket_noalloc: unknown mma_type");
  if (dims->num_experts < 1)
    return fail(MOE_ERR_INVALID_ARG, "moe_bucket_noalloc: num_experts < 1");
  if (dims->topk < 1 || dims->topk > 32 || dims->topk > dims->num_experts)
    return fail(MOE_ERR_INVALID_ARG, "moe_bucket_noalloc: topk outside [1, min(num_experts, 32)]");
  if (num_tokens < 0) return fail(MOE_ERR_INVALID_ARG, "num_tokens < 0");
  if (dims->num_experts > kMaxExperts)
    return fail(MOE_ERR_INVALID_ARG, "moe_bucket_noalloc: num_experts above its limit of 256");
  if ((int64_t)num_tokens * dims->topk > kMaxAssignments)
    return fail(MOE_ERR_INVALID_ARG,
                "moe_bucket_noalloc: num_tokens * topk above its limit of 8192 assignments");
  if (num_tokens == 0) return MOE_OK;
  if (!topk_ids_dev || !topk_weights_dev || !counts_dev || !assign_slot_dev)
    return fail(MOE_ERR_INVALID_ARG, "moe_bucket_noalloc: NULL pointer");
  if ((reinterpret_cast<uintptr_t>(topk_ids_dev) | reinterpret_cast<uintptr_t>(topk_weights_dev) |
       reinterpret_cast<uintptr_t>(counts_dev) | reinterpret_cast<uintptr_t>(assign_slot_dev)) & 3)
    return fail(MOE_ERR_INVALID_ARG, "moe_bucket_noalloc: pointers must be 4-byte aligned");

  unsigned char* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The error flags are OR-ed into; everything else the kernel reads it writes first.
  e = cudaMemsetAsync(base + kOffFlags, 0, 64 * sizeof(int32_t), st);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));

  WsPtrs p = {};
  p.flags = reinterpret_cast<int32_t*>(base + kOffFlags);
  p.counts = counts_dev;
  p.seg = reinterpret_cast<int32_t*>(base + kOffSeg);
  p.tiles = reinterpret_cast<int4*>(base + kOffTiles);
  p.tile_done = reinterpret_cast<int32_t*>(base + kOffTileDone);
  p.tile_start = reinterpret_cast<int32_t*>(base + kOffTileStart);
  p.local_rank = reinterpret_cast<int32_t*>(base + kOffLocalRank);
  p.blk_base = reinterpret_cast<int32_t*>(base + kOffBlkBase);
  p.assign_slot = assign_slot_dev;
  p.slot_token = reinterpret_cast<int32_t*>(base + kOffSlotToken);
  p.slot_assign = reinterpret_cast<int32_t*>(base + kOffSlotAssign);
  p.slot_weight = reinterpret_cast<float*>(base + kOffSlotWeight);
  const Shape shape{dims->hidden, dims->inter, dims->num_experts, dims->topk};
  e = launch_bucket(shape, topk_ids_dev, num_tokens, p, kBN, st);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  e = launch_assign_slots(shape, topk_ids_dev, topk_weights_dev, num_tokens, p, st);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  return MOE_OK;
}
