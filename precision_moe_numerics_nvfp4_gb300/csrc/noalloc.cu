// nvfp4_quantize for callers that cannot allocate device memory.
//
// nvfp4_quantize needs a small scratch buffer when it computes the outer
// scales itself: one partial maximum per amax block, plus one slot per matrix
// for the scale.  Some callers have no way to provide it: code embedded in a
// host runtime that owns every device allocation and hands out none, or code
// that must not allocate once it is running (inside a long-lived service loop
// with a fixed memory budget).  This entry point uses a fixed scratch array
// that lives in the library's own device memory instead.
#include "common.cuh"
#include "launch.h"

namespace nvm {

// The fixed scratch: 512 KiB of fp32.  Every GPU that loads the library holds
// it until the process exits.
static __device__ __align__(256) float g_noalloc_scratch[131072];

// Device address of the scratch on the current device.  Looked up once per
// device, with that device current, on the first call made on it.
static float *noalloc_scratch() {
  static float *cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<float *>(p);
  }
  return cache[dev];
}

}  // namespace nvm

extern "C" int nvfp4_quantize_noalloc(const void *x, int64_t batch, int64_t rows, int64_t cols,
                                      const int32_t *group_offsets, int32_t num_groups, const float *outer_scale_in,
                                      float *outer_scale_out, uint8_t *codes, uint8_t *scales, nv_stream_t stream) {
  void *ws = nullptr;
  size_t ws_bytes = 0;
  if (!outer_scale_in) {  // the amax pass needs the scratch
    const size_t need = nvfp4moe_quantize_workspace_bytes(batch, rows, cols);
    if (need > sizeof(nvm::g_noalloc_scratch)) return NV_ERR_WORKSPACE;
    ws = nvm::noalloc_scratch();
    if (!ws) return NV_ERR_CUDA;
    ws_bytes = sizeof(nvm::g_noalloc_scratch);
  }
  return nvfp4_quantize(x, batch, rows, cols, group_offsets, num_groups, outer_scale_in, outer_scale_out, codes,
                        scales, ws, ws_bytes, stream);
}
