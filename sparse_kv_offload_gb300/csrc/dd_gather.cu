// Host -> HBM gather of the missing chunks (zero-copy kernel variant).
//
// DualDecoder §5.4, GPU-side sparse KV assembly: only the selected KV blocks
// move from host memory into a GPU staging region, where they are laid out
// for attention; the gather on the GPU side avoids the many small host-side
// copies of a CPU gather (§6.4, Fig. 19).  Here one warp copies one chunk of
// K or V (cs rows x 256 bytes, contiguous in both the host tensor and the
// staging slot) with 16-byte loads issued over the host link, eight in
// flight per lane before the stores.
#include "dd_common.cuh"

namespace dd {

constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) k_gather(
    const uint4 *__restrict__ Kh, const uint4 *__restrict__ Vh, const int32_t *__restrict__ miss_list,
    const int32_t *__restrict__ miss_count, uint4 *__restrict__ Kst, uint4 *__restrict__ Vst, int64_t max_misses,
    int64_t n_chunks_total, int vec_per_chunk, int32_t *map_out, int32_t *status) {
  pdl_wait();
  pdl_trigger();
  if (load_status(status) != 0) return;
  const int64_t M = min((int64_t)*miss_count, max_misses);
  const int lane = threadIdx.x & 31;
  const int64_t gw = ((int64_t)blockIdx.x * kGatherThreads + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * kGatherThreads) >> 5;
  for (int64_t w = gw; w < 2 * M; w += nw) {
    const int64_t m = w >> 1;
    const int half = (int)(w & 1);
    const int32_t packed = miss_list[m];
    if (packed < 0 || packed >= n_chunks_total) {
      if (lane == 0) set_status(status, DD_ERR_DEVICE_CHECK);
      continue;
    }
    if (map_out && half == 0 && lane == 0) map_out[packed] = (int32_t)m;   // prefetch map: chunk -> slot
    const uint4 *src = (half ? Vh : Kh) + (int64_t)packed * vec_per_chunk;
    uint4 *dst = (half ? Vst : Kst) + m * vec_per_chunk;
    for (int i0 = 0; i0 < vec_per_chunk; i0 += 256) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * 32 + lane;
        v[u] = (i < vec_per_chunk) ? ldg_nc(src + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * 32 + lane;
        if (i < vec_per_chunk) dst[i] = v[u];
      }
    }
  }
}

cudaError_t launch_gather(const uint4 *Kh, const uint4 *Vh, const int32_t *miss_list, const int32_t *miss_count,
                          uint4 *Kst, uint4 *Vst, int64_t max_misses, int64_t n_chunks_total, int cs,
                          int32_t *status, int sm_count, cudaStream_t s, int32_t *map_out, int ctas_per_sm) {
  if (max_misses == 0) return cudaSuccess;
  // persistent grid: enough warps to keep the host link busy, never more
  // than the largest possible miss count needs
  const int64_t want_warps = 2 * max_misses;
  int64_t blocks = (want_warps * 32 + kGatherThreads - 1) / kGatherThreads;
  const int64_t cap = (int64_t)sm_count * ctas_per_sm;
  if (blocks > cap) blocks = cap;
  return launch_k(k_gather, dim3((unsigned)blocks), dim3(kGatherThreads), 0, s, Kh, Vh, miss_list, miss_count, Kst,
                  Vst, max_misses, n_chunks_total, cs * kVecPerRow, map_out, status);
}

}  // namespace dd
