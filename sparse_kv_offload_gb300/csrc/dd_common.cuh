// Shared device helpers of libdd (CUDA path only).
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "dd.h"

namespace dd {

constexpr int kD = 128;          // head dimension the kernels are built for
constexpr int kVecPerRow = 16;   // uint4 (8 x bf16) per row of d = 128
constexpr int kMaxNq = 8;
constexpr int kMaxC = 16384;
constexpr int kMaxNQV = 64;      // n_q * G query vectors per KV head

// Record a device-side error; the first error wins.
__device__ __forceinline__ void set_status(int32_t *status, int32_t code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ int32_t load_status(const int32_t *status) {
  return *reinterpret_cast<const volatile int32_t *>(status);
}

// bf16 pair in one 32-bit word -> two floats (exact)
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 &v, float f[8]) {
  f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
  f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
  f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
  f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// fp32 -> bf16 bits, round to nearest even (finite inputs; NaN kept quiet)
__device__ __forceinline__ uint32_t f2bf(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (u >> 16) | 0x40u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return u >> 16;
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  return f2bf(lo) | (f2bf(hi) << 16);
}

__device__ __forceinline__ uint4 ldg_nc(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

}  // namespace dd

// Host-side launch helpers, defined in dd_api.cu
namespace dd {
struct Ctx;
cudaError_t launch_build_landmarks(const uint4 *K, uint4 *lm, int64_t n_chunks, int cs, cudaStream_t s);
cudaError_t launch_score(const uint4 *q, const uint4 *lm, float *scores, int B, int n_q, int Hq, int Hkv,
                         int C, cudaStream_t s);
cudaError_t launch_topk(const float *scores, int32_t *sel, int rows, int C, int k, cudaStream_t s);
cudaError_t launch_union(const int32_t *sel, const int32_t *resident_slot, int32_t *union_idx,
                         int32_t *union_slot, uint8_t *union_qmask, int32_t *union_cnt,
                         int32_t *unit_miss, int units, int n_q, int Hkv, int k, int C, int umax,
                         int64_t hot_slots, int32_t *status, cudaStream_t s);
cudaError_t launch_assign(const int32_t *sel, const int32_t *union_idx, int32_t *union_slot,
                          const int32_t *union_cnt, const int32_t *unit_miss, int32_t *miss_list,
                          int32_t *miss_count, int32_t *attn_slot, int units, int n_q, int Hkv, int k,
                          int C, int umax, int64_t max_misses, int32_t *status, cudaStream_t s);
cudaError_t launch_gather(const uint4 *Kh, const uint4 *Vh, const int32_t *miss_list,
                          const int32_t *miss_count, uint4 *Kst, uint4 *Vst, int64_t max_misses,
                          int64_t n_chunks_total, int cs, int32_t *status, int sm_count, cudaStream_t s);
}  // namespace dd
