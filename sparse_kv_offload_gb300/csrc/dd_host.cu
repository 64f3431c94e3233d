// Host-side helpers shared by the launchers: the per-launch driver calls a
// decode step would otherwise repeat (opt-in shared memory of a kernel).
#include <mutex>

#include "dd_common.cuh"

namespace dd {

namespace {

struct SmemEntry {
  const void *func;
  int device;
  size_t bytes;
};

std::mutex g_smem_mu;
SmemEntry g_smem[256];
int g_smem_n = 0;

}  // namespace

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device, calling the runtime only when the limit grows.
cudaError_t set_dyn_smem(const void *func, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;   // below the default limit: nothing to opt in to
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_smem_mu);
  for (int i = 0; i < g_smem_n; ++i)
    if (g_smem[i].func == func && g_smem[i].device == dev) {
      if (g_smem[i].bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
      if (e == cudaSuccess) g_smem[i].bytes = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && g_smem_n < 256) g_smem[g_smem_n++] = {func, dev, bytes};
  return e;
}

}  // namespace dd
