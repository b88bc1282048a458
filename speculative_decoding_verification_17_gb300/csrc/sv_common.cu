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

// Zero n16 16-byte words at p. The launch that follows on the stream (a segment kernel,
// launched with programmatic serialization) may start its CTAs at once: they stream their
// rows meanwhile and wait in griddepcontrol.wait before they touch what this clears.
__global__ void clear_kernel(uint4* p, long long n16) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

sv_status launch_clear(void* p, size_t bytes, cudaStream_t st) {
  const long long n16 = (long long)(bytes / 16);
  if (n16 <= 0) return SV_OK;
  if (!SV_CLEAR_KERNEL) {  // a build may compare against a plain memset
    const cudaError_t e = cudaMemsetAsync(p, 0, bytes, st);
    return e == cudaSuccess ? SV_OK : cuda_fail(e);
  }
  constexpr int kClearThreads = 256;
  long long blocks = (n16 + 4 * kClearThreads - 1) / (4 * kClearThreads);
  blocks = blocks < 1 ? 1 : (blocks > 1024 ? 1024 : blocks);
  clear_kernel<<<(unsigned)blocks, kClearThreads, 0, st>>>(static_cast<uint4*>(p), n16);
  return launch_status();
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
