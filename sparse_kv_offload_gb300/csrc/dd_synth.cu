// Device implementation of the seeded synthetic-input generator (see
// include/dd_synth.h for the definition).  Integer SplitMix64 words, an exact
// Irwin-Hall(12) fp32 normal, separately rounded fp32 multiply and add, and
// round-to-nearest-even to bf16 -- the same bits as the host generator.
#include "dd_common.cuh"
#include "dd_synth.h"

namespace dd {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t stream_key(uint64_t seed, uint64_t tid) {
  return sm64_mix((seed << 32) + tid + kGamma);
}

__device__ __forceinline__ float ih_normal(uint64_t key, uint64_t idx) {
  uint32_t s = 0;
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const uint64_t w = sm64_mix(key + (3ull * idx + (uint64_t)r + 1ull) * kGamma);
    s += (uint32_t)(w & 0xFFFFu) + (uint32_t)((w >> 16) & 0xFFFFu) + (uint32_t)((w >> 32) & 0xFFFFu) +
         (uint32_t)(w >> 48);
  }
  return __int2float_rn((int)s - 393210) * 0x1p-16f;
}

__global__ void k_synth_kv(uint16_t *__restrict__ dst, int64_t n, uint64_t key, int Hkv, int L, int cs,
                           const float *__restrict__ bias, const float *__restrict__ u_hat,
                           const int32_t *__restrict__ chunk_map) {
  const int C = L / cs;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(e & 127);
    int64_t unit, t;
    if (chunk_map) {
      const int64_t row = e >> 7;               // row of the slot pool
      const int64_t slot = row / cs;
      const int r = (int)(row - slot * cs);
      const int32_t packed = chunk_map[slot];
      unit = packed / C;
      t = (int64_t)(packed - unit * C) * cs + r;
    } else {
      const int64_t row = e >> 7;
      unit = row / L;
      t = row - unit * L;
    }
    const uint64_t idx = ((uint64_t)unit * L + (uint64_t)t) * 128ull + (uint64_t)i;
    float x = ih_normal(key, idx);
    if (bias) x = __fadd_rn(x, __fmul_rn(bias[unit * C + t / cs], u_hat[unit * 128 + i]));
    dst[e] = (uint16_t)f2bf(x);
  }
}

struct NoiseKeys {
  uint64_t key[8];   // stream key of the noise of query j (j >= 1)
  float scale[8];    // fp32 scale of that noise
};

__global__ void k_synth_q(uint16_t *__restrict__ dst, int64_t n, int n_q, int Hq, uint64_t key_real,
                          const NoiseKeys nk) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(e & 127);
    const int64_t row = e >> 7;                 // (b, j, h)
    const int h = (int)(row % Hq);
    const int64_t bj = row / Hq;
    const int j = (int)(bj % n_q);
    const int64_t b = bj / n_q;
    const uint64_t idx = ((uint64_t)b * Hq + (uint64_t)h) * 128ull + (uint64_t)i;
    const uint32_t real = f2bf(ih_normal(key_real, idx));
    if (j == 0) {
      dst[e] = (uint16_t)real;
    } else {
      const float x = __fadd_rn(__uint_as_float(real << 16), __fmul_rn(nk.scale[j], ih_normal(nk.key[j], idx)));
      dst[e] = (uint16_t)f2bf(x);
    }
  }
}

static bool valid_kv_dims(const dd_dims *d) {
  return d && d->B >= 0 && d->Hkv > 0 && d->d == 128 && d->cs > 0 && d->L > 0 && d->L % d->cs == 0;
}

static int grid_for(int64_t n) {
  int64_t b = (n + 255) / 256;
  return (int)(b > 65536 ? 65536 : (b < 1 ? 1 : b));
}

}  // namespace dd

extern "C" dd_status dd_synth_kv(const dd_dims *dims, uint64_t seed, int32_t tensor_id, const float *chunk_bias,
                                 const float *u_hat, const int32_t *chunk_map, int64_t n_slots, void *dst,
                                 dd_stream_t stream) {
  using namespace dd;
  if (!valid_kv_dims(dims) || dst == nullptr || (chunk_bias == nullptr) != (u_hat == nullptr) || n_slots < 0)
    return DD_ERR_INVALID_ARG;
  const int64_t n = chunk_map ? n_slots * dims->cs * 128 : (int64_t)dims->B * dims->Hkv * dims->L * 128;
  if (n == 0) return DD_OK;
  void *dptr = dst;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, dst) == cudaSuccess && a.type == cudaMemoryTypeHost && a.devicePointer)
    dptr = a.devicePointer;
  cudaGetLastError();
  k_synth_kv<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(static_cast<uint16_t *>(dptr), n,
                                                            stream_key(seed, (uint64_t)tensor_id), dims->Hkv,
                                                            dims->L, dims->cs, chunk_bias, u_hat, chunk_map);
  return cudaGetLastError() == cudaSuccess ? DD_OK : DD_ERR_CUDA;
}

extern "C" dd_status dd_synth_queries(const dd_dims *dims, uint64_t seed, int32_t layer, const float *spec_scale,
                                      void *dst, dd_stream_t stream) {
  using namespace dd;
  if (!dims || dst == nullptr || spec_scale == nullptr || dims->d != 128 || dims->n_q < 1 || dims->n_q > 8 ||
      dims->Hq <= 0 || dims->B < 0)
    return DD_ERR_INVALID_ARG;
  const int64_t n = (int64_t)dims->B * dims->n_q * dims->Hq * 128;
  if (n == 0) return DD_OK;
  NoiseKeys nk = {};
  for (int j = 1; j < dims->n_q; ++j) {
    nk.key[j] = stream_key(seed, (uint64_t)(8 + j + 64 * layer));
    nk.scale[j] = spec_scale[j];
  }
  k_synth_q<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(static_cast<uint16_t *>(dst), n, dims->n_q, dims->Hq,
                                                           stream_key(seed, (uint64_t)(3 + 64 * layer)), nk);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DD_OK : DD_ERR_CUDA;
}
