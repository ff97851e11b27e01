// nvfp4_quantize for callers that cannot allocate device memory.
//
// nvfp4_quantize needs a small scratch buffer when it computes the outer
// scales itself: one partial maximum per amax block, plus one slot per matrix
// for the scale.  Some callers have no way to provide it: code embedded in a
// host runtime that owns every device allocation and hands out none, or code
// that must not allocate once it is running (inside a long-lived service loop
// with a fixed memory budget).  This entry point uses a fixed scratch array
// that lives in the library's own device memory instead.
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace nvm {

// The fixed scratch: 512 KiB of fp32.  Every GPU that loads the library holds
// it until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[131072];

// Device address of the scratch on the current device.  Looked up once per
// device, with that device current, on the first call made on it; host
// threads that race on that first lookup store the same address, and the
// atomic makes the race well-defined.  In host code the array's name is only
// a stand-in for it, never a device address.
static float *noalloc_scratch() {
  static std::atomic<float *> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  float *p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    void *a = nullptr;
    if (cudaGetSymbolAddress(&a, g_noalloc_scratch) != cudaSuccess) return nullptr;
    p = static_cast<float *>(a);
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace nvm

extern "C" int nvfp4_quantize_noalloc(const void *x, int64_t batch, int64_t rows, int64_t cols,
                                      const int32_t *group_offsets, int32_t num_groups, const float *outer_scale_in,
                                      float *outer_scale_out, uint8_t *codes, uint8_t *scales, nv_stream_t stream) {
  // the same argument and shape checks as nvfp4_quantize, before the limit,
  // so that a bad call reports the same error through both entry points
  const int chk = nvm::quantize_check_args(x, batch, rows, cols, group_offsets, num_groups, codes, scales);
  if (chk != NV_OK) return chk;
  void *ws = nullptr;
  size_t ws_bytes = 0;
  if (!outer_scale_in && rows > 0 && cols > 0) {  // the amax pass needs the scratch
    const size_t need = nvfp4moe_quantize_workspace_bytes(batch, rows, cols);
    if (need > sizeof(nvm::g_noalloc_scratch)) return NV_ERR_WORKSPACE;
    ws = nvm::noalloc_scratch();
    if (!ws) return NV_ERR_CUDA;
    ws_bytes = sizeof(nvm::g_noalloc_scratch);
  }
  return nvfp4_quantize(x, batch, rows, cols, group_offsets, num_groups, outer_scale_in, outer_scale_out, codes,
                        scales, ws, ws_bytes, stream);
}
