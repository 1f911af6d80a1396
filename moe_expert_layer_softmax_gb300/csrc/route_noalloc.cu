// moe_route_noalloc: the routing call for callers that cannot provide a
// workspace buffer.
//
// moe_route needs `ws` (error word, per-block expert histograms, per-route
// ranks).  Some callers have no way to obtain that device memory: plugins
// hosted by a framework that owns all device memory and offers them no
// allocator, hosts that work inside a fixed device-memory budget handed out up
// front, and latency-critical loops that must not enter cudaMalloc because it
// can synchronise the whole device and stall other streams.  This variant keeps its scratch in
// one file-scope device array instead, so the caller passes only inputs and
// outputs and nothing is ever allocated.
//
// Rules of use:
//   - The array holds at most kNoAllocScratchBytes (2 MiB); shapes that need
//     more are rejected with MOE_ERR_SCRATCH_LIMIT before any work is queued.
//     Every GPU that loads this library keeps the array until the process ends.
//   - The first call on a device looks up the array's device address (with that
//     device current) and caches it; moe_init drops the cached address, so the
//     first call after a moe_init (e.g. after a device reset) looks it up
//     again.  Make that first call before any stream capture begins.
//   - All calls on a device share the one array and it keeps what the last call
//     left there.  Each call clears the error word itself; the histograms and
//     ranks are fully rewritten.  Calls whose work overlaps on the GPU (e.g. on
//     two streams at once) race on the array: serialise them.
#include <mutex>

#include "moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;

// The shared scratch: [error word (256 B) | block histograms | route ranks].
static __device__ __align__(256) uint8_t g_route_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev] = {};
std::mutex g_scratch_mutex;

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

// Device address of g_route_scratch on the current device (looked up once).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// moe_init calls this: after a device reset the module is loaded again and the
// array may sit at another address, so the cached one must not be reused.
void noalloc_forget_device(int dev) {
  if (dev < 0 || dev >= kMaxDev) return;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  g_scratch_addr[dev] = nullptr;
}

}  // namespace moe

using namespace moe;

extern "C" MOE_API int moe_route_noalloc(const moe_shape_t* s, const void* x, const void* w_router,
                                         const float* logit_bias, float* logits,
                                         int32_t* topk_idx, float* gates, int32_t* counts,
                                         int32_t* offsets, int32_t* tile_offsets,
                                         int32_t* slot_of_route, int32_t* route_of_slot,
                                         int32_t* dev_error, void* stream) {
  // Same shape and pointer rules as moe_route (no workspace argument).
  int64_t rows_max = 0;
  int rc = moe_rows_max(s, &rows_max);
  if (rc != MOE_OK) return rc;
  const void* must[] = {logits, topk_idx, gates, counts, offsets, tile_offsets, slot_of_route,
                        route_of_slot};
  for (const void* p : must) {
    if (p == nullptr) return MOE_ERR_INVALID;
    if (!aligned16(p)) return MOE_ERR_ALIGN;
  }
  if (w_router != nullptr) {
    if (x == nullptr) return MOE_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_ALIGN;
  }
  if ((logit_bias != nullptr && !aligned16(logit_bias)) ||
      (dev_error != nullptr && !aligned16(dev_error)))
    return MOE_ERR_ALIGN;

  const int nb = (s->T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  const size_t hist_off = 256;
  const size_t rank_off = hist_off + round256((size_t)nb * s->n_experts * 4);
  const size_t need = rank_off + round256((size_t)s->T * s->top_k * 4);
  if (need > kNoAllocScratchBytes) return MOE_ERR_SCRATCH_LIMIT;

  const DeviceInfo* di = device_info();
  if (di == nullptr || !di->ready) return MOE_ERR_NOT_INIT;
  void* base = nullptr;
  rc = scratch_address(&base);
  if (rc != MOE_OK) return rc;
  uint8_t* b = static_cast<uint8_t*>(base);
  int32_t* err = reinterpret_cast<int32_t*>(b);
  int32_t* hist = reinterpret_cast<int32_t*>(b + hist_off);
  int32_t* rank = reinterpret_cast<int32_t*>(b + rank_off);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (cudaMemsetAsync(err, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
  // the same kernels as moe_route, on the static scratch
  if (launch_route(s->T, s->d_model, s->n_experts, s->top_k, rows_max, x, w_router, logit_bias,
                   logits, topk_idx, gates, counts, offsets, tile_offsets, slot_of_route,
                   route_of_slot, err, hist, rank, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (dev_error != nullptr &&
      cudaMemcpyAsync(dev_error, err, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
