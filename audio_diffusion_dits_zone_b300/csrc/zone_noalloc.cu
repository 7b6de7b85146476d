// prism_zone_shapes_noalloc: the zone-shape step for callers that cannot hand the
// library any device memory of its own.
//
// prism_zone_shapes needs a scratch workspace (per-zone partial statistics) that
// the caller allocates.  Some callers cannot do that at the point of the call:
// hosts whose device memory is owned entirely by another allocator (a framework's
// caching pool, an inference engine that plans every byte up front) and plugin or
// callback hooks that are not allowed to allocate while they run (an allocation
// there can block on the device or fail in the middle of a step).  This entry point
// gives them the same result with no workspace argument: the scratch lives in the
// fixed-size device array below, which is part of the library image and is held by
// every GPU that loads the library until the process exits.
//
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.  The scratch
// array is shared by every call on a device and keeps what the last call left in
// it; no word of it needs to start at zero, because each call writes every scratch
// word before it reads it.  Two calls whose work overlaps on the GPU (different
// streams, no ordering between them) race on the array and must not be issued.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

// Room for the partial statistics of up to (zones x channel chunks) = 87,000
// zone-chunk pairs, e.g. a 2K grid (700 zones) with 5,120 feature channels.
constexpr size_t kScratchBytes = (size_t)1 << 20;

static __device__ __align__(256) unsigned char g_zone_scratch[kScratchBytes];

// Device address of g_zone_scratch on the current device.  The host-side symbol is
// only a stand-in for the array, so the address is looked up with
// cudaGetSymbolAddress the first time a device is used (with that device current)
// and cached; later calls on that device reuse it.
cudaError_t scratch_on_current_device(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_zone_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int prism_zone_shapes_noalloc(const void* feat, int32_t feat_dtype, int64_t feat_ld, int32_t C,
                                         const float* a2v, int32_t T, int32_t H, int32_t W, int32_t zt, int32_t zh,
                                         int32_t zw, const int32_t* shapes, int32_t n_shapes, int32_t* zone_shape,
                                         int32_t* perm, void* stream) {
  // Argument checks and the scratch size, exactly as the workspace entry point computes them.
  size_t need = 0;
  int rc = prism_zone_shapes(feat, feat_dtype, feat_ld, C, a2v, T, H, W, zt, zh, zw, shapes, n_shapes, zone_shape,
                             perm, nullptr, &need, stream);
  if (rc != PRISM_OK) return rc;
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "prism_zone_shapes_noalloc: this grid needs %zu bytes of zone scratch, more than the %zu built into "
             "the library; call prism_zone_shapes with a workspace instead",
             need, kScratchBytes);
    return prism::report_error(PRISM_EUNSUPPORTED, msg);
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "prism_zone_shapes_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
    return prism::report_error(PRISM_ECUDA, msg);
  }
  size_t cap = kScratchBytes;
  return prism_zone_shapes(feat, feat_dtype, feat_ld, C, a2v, T, H, W, zt, zh, zw, shapes, n_shapes, zone_shape,
                           perm, scratch, &cap, stream);
}
