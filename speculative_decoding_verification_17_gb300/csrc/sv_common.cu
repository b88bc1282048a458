// sv_common.cu — library-wide C ABI helpers: version, status names, last CUDA error.
#include <atomic>

#include <cuda_runtime.h>

#include "specverify.h"
#include "sv_host.h"

namespace {
thread_local int g_last_cuda_error = 0;
}

namespace sv {
sv_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return SV_ERR_CUDA;
}

// SMs of the current device (queried once per device; 152 if the query fails).
int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load();
    if (c > 0) return c;
  }
  int c = 0;
  if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
    c = 152;
  if (dev >= 0 && dev < 64) cache[dev].store(c);
  return c;
}
}  // namespace sv

extern "C" int sv_version(void) { return 10000 * 0 + 100 * 1 + 0; }

extern "C" const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARG: return "invalid argument";
    case SV_ERR_UNSUPPORTED: return "unsupported";
    case SV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SV_ERR_CUDA: return "CUDA error";
    case SV_ERR_TIMEOUT: return "timeout";
  }
  return "unknown status";
}

extern "C" int sv_last_cuda_error(void) { return g_last_cuda_error; }
