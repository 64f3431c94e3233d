// Landmark build and dual-query landmark scoring.
//
// DualDecoder §2.2 / §4.1: chunk landmarks are built once before decoding and
// the retrieval index of a step comes from the query and the landmarks; §5.2:
// the output token and the speculative token are scored in one pass.
#include "dd_common.cuh"

namespace dd {

// ---------------------------------------------------------------------------
// a0: lm[chunk, i] = bf16(sum_{t<cs} K[chunk*cs+t, i] / cs), fp32 sum in order t.
// 16 threads per chunk, each owning 8 coordinates (one 16-byte vector per row).
// K may be device memory or pinned host memory read over the host link.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_build_landmarks(const uint4 *__restrict__ K, uint4 *__restrict__ lm,
                                                          int64_t n_chunks, int cs) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t chunk = gid >> 4;
  const int part = (int)(gid & 15);
  if (chunk >= n_chunks) return;
  const uint4 *src = K + chunk * cs * kVecPerRow + part;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int t0 = 0; t0 < cs; t0 += 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = (t0 + u < cs) ? src[(int64_t)(t0 + u) * kVecPerRow] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (t0 + u < cs) {
        float f[8];
        unpack8(v[u], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
      }
    }
  }
  const float fcs = (float)cs;
  uint4 o;
  o.x = pack_bf2(__fdiv_rn(acc[0], fcs), __fdiv_rn(acc[1], fcs));
  o.y = pack_bf2(__fdiv_rn(acc[2], fcs), __fdiv_rn(acc[3], fcs));
  o.z = pack_bf2(__fdiv_rn(acc[4], fcs), __fdiv_rn(acc[5], fcs));
  o.w = pack_bf2(__fdiv_rn(acc[6], fcs), __fdiv_rn(acc[7], fcs));
  lm[chunk * kVecPerRow + part] = o;
}

cudaError_t launch_build_landmarks(const uint4 *K, uint4 *lm, int64_t n_chunks, int cs, cudaStream_t s) {
  if (n_chunks == 0) return cudaSuccess;
  const int64_t threads = n_chunks * 16;
  const int64_t blocks = (threads + 255) / 256;
  k_build_landmarks<<<(unsigned)blocks, 256, 0, s>>>(K, lm, n_chunks, cs);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// a1: scores[b,j,g,c] = qsum[b,j,g,:] . lm[b,g,c,:] with qsum the fp32 sum of
// the group's G query heads.  One CTA scores kTile landmarks of one (b,g) for
// all NQ queries, so every landmark byte is read once.  16 lanes share one
// landmark row (one 16-byte load each) and reduce with shuffles; each thread
// keeps kPass landmark loads in flight before using them.
// ---------------------------------------------------------------------------
constexpr int kScoreThreads = 256;
constexpr int kPass = 8;                                  // landmark rows in flight per thread
constexpr int kRowsPerPass = kScoreThreads / 16;          // 16
constexpr int kTile = kPass * kRowsPerPass;               // 128 landmarks per CTA

template <int NQ>
__global__ void __launch_bounds__(kScoreThreads) k_score(const uint4 *__restrict__ q, const uint4 *__restrict__ lm,
                                                         float *__restrict__ scores, int Hq, int Hkv, int C) {
  __shared__ float sc[NQ][kTile];
  const int unit = blockIdx.x;
  const int b = unit / Hkv, g = unit - b * Hkv;
  const int G = Hq / Hkv;
  const int tid = threadIdx.x;
  const int part = tid & 15;
  const int sub = tid >> 4;
  const int c0 = blockIdx.y * kTile;

  // issue the landmark loads first
  uint4 v[kPass];
  const uint4 *base = lm + (int64_t)unit * C * kVecPerRow + part;
#pragma unroll
  for (int p = 0; p < kPass; ++p) {
    const int c = c0 + p * kRowsPerPass + sub;
    v[p] = (c < C) ? ldg_nc(base + (int64_t)c * kVecPerRow) : make_uint4(0, 0, 0, 0);
  }

  // this lane's 8 coordinates of each query's group sum
  float qs[NQ][8];
#pragma unroll
  for (int j = 0; j < NQ; ++j) {
#pragma unroll
    for (int e = 0; e < 8; ++e) qs[j][e] = 0.f;
    for (int h = g * G; h < (g + 1) * G; ++h) {
      float f[8];
      unpack8(q[((int64_t)(b * NQ + j) * Hq + h) * kVecPerRow + part], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) qs[j][e] += f[e];
    }
  }

#pragma unroll
  for (int p = 0; p < kPass; ++p) {
    float f[8];
    unpack8(v[p], f);
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc = fmaf(qs[j][e], f[e], acc);
      acc += __shfl_xor_sync(0xffffffffu, acc, 8);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      if (part == 0) sc[j][p * kRowsPerPass + sub] = acc;
    }
  }
  __syncthreads();
  for (int i = tid; i < NQ * kTile; i += kScoreThreads) {
    const int j = i / kTile, cc = i - j * kTile;
    const int c = c0 + cc;
    if (c < C) scores[((int64_t)(b * NQ + j) * Hkv + g) * C + c] = sc[j][cc];
  }
}

cudaError_t launch_score(const uint4 *q, const uint4 *lm, float *scores, int B, int n_q, int Hq, int Hkv, int C,
                         cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  dim3 grid(B * Hkv, (C + kTile - 1) / kTile);
  switch (n_q) {
#define DD_SCORE_CASE(N) \
  case N: k_score<N><<<grid, kScoreThreads, 0, s>>>(q, lm, scores, Hq, Hkv, C); break;
    DD_SCORE_CASE(1) DD_SCORE_CASE(2) DD_SCORE_CASE(3) DD_SCORE_CASE(4)
    DD_SCORE_CASE(5) DD_SCORE_CASE(6) DD_SCORE_CASE(7) DD_SCORE_CASE(8)
#undef DD_SCORE_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace dd
