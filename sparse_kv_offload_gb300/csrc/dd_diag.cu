// Diagnostics: the library's bounded device waits, run on something nothing
// will ever signal, so that a test can watch a wait run out and report
// DD_ERR_TIMEOUT while the context stays usable.  No fault, trap or
// unbounded loop is involved: each wait gives up after ~2 s by itself.
#include "dd_common.cuh"

namespace dd {

// kind 0: an mbarrier that no thread arrives on and no copy completes
//         (the waits of the attention kernel's pipeline and of the
//         selection's landmark ring);
// kind 1: a look-back word that no unit publishes (the selection's sum over
//         the earlier units).
__global__ void k_selftest_wait(int kind, const unsigned long long *word, int32_t *status) {
  __shared__ __align__(8) uint64_t bar;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x != 0) return;
  if (kind == 0) {
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_wait(smem_u32(&bar), 0, status);   // records DD_ERR_TIMEOUT when it gives up
  } else {
    bool ok = true;
    wait_published(word, 1u, globaltimer_ns(), &ok);
    if (!ok) set_status(status, DD_ERR_TIMEOUT);
  }
}

cudaError_t launch_selftest_wait(int kind, const unsigned long long *word, int32_t *status, cudaStream_t s) {
  return launch_k(k_selftest_wait, dim3(1), dim3(32), 0, s, kind, word, status);
}

}  // namespace dd
