// Library-wide entry points of the C ABI: status names, version, device info.
#include <mutex>

#include "common.cuh"

namespace tl {

int num_sms() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace tl

extern "C" const char* tl_status_string(tl_status status) {
  switch (status) {
    case TL_OK: return "TL_OK";
    case TL_ERR_INVALID_ARG: return "TL_ERR_INVALID_ARG: a null pointer, bad size or misaligned pointer";
    case TL_ERR_UNSUPPORTED: return "TL_ERR_UNSUPPORTED: valid arguments, but not a shape or dtype this build runs";
    case TL_ERR_CUDA: return "TL_ERR_CUDA: a CUDA call or kernel launch failed";
    case TL_ERR_WORKSPACE: return "TL_ERR_WORKSPACE: workspace missing or too small";
  }
  return "unknown tl_status";
}

extern "C" int32_t tl_version(void) { return 1 * 10000 + 0 * 100 + 0; }
