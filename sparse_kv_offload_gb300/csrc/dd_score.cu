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
  pdl_wait();
  pdl_trigger();
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
  return launch_k(k_build_landmarks, dim3((unsigned)blocks), dim3(256), 0, s, K, lm, n_chunks, cs);
}

// ---------------------------------------------------------------------------
// a1: scores[b,j,g,c] = qsum[b,j,g,:] . lm[b,g,c,:] with qsum the fp32 sum of
// the group's G query heads.  One CTA scores kTilesPerCta tiles of kTile
// landmarks of one (b,g) for all NQ queries, so every landmark byte is read
// once.  16 lanes share one landmark row (one 16-byte load each); each
// thread holds kPass rows of a tile and the loads of the next tile are in
// flight while the current one is reduced.  The 16-lane reduction of the
// kPass*NQ partial dots is a butterfly that halves the value set at every
// step (8+4+2+1 shuffles per 16 dots), leaving dot (lane position) in each
// lane.
// ---------------------------------------------------------------------------
constexpr int kScoreThreads = 256;
constexpr int kPass = 8;                                  // landmark rows per thread per tile
constexpr int kRowsPerPass = kScoreThreads / 16;          // 16
constexpr int kTile = kPass * kRowsPerPass;               // 128 landmarks per tile
constexpr int kTilesPerCta = 4;

// Butterfly over the 16 lanes sharing a row: x[0..15] in every lane ->
// lane `part` returns the 16-lane sum of x[part].
__device__ __forceinline__ float butterfly16(float (&x)[16], int part) {
  float y[8], z[4], w[2];
  const bool b3 = part & 8, b2 = part & 4, b1 = part & 2, b0 = part & 1;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = b3 ? x[i] : x[i + 8];
    const float keep = b3 ? x[i + 8] : x[i];
    y[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b2 ? y[i] : y[i + 4];
    const float keep = b2 ? y[i + 4] : y[i];
    z[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b1 ? z[i] : z[i + 2];
    const float keep = b1 ? z[i + 2] : z[i];
    w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  const float send = b0 ? w[0] : w[1];
  const float keep = b0 ? w[1] : w[0];
  return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

template <int NQ>
__global__ void __launch_bounds__(kScoreThreads) k_score(const uint4 *__restrict__ q, const uint4 *__restrict__ lm,
                                                         float *__restrict__ scores, int Hq, int Hkv, int C) {
  constexpr int kVals = kPass * NQ;                       // partial dots per lane per tile
  constexpr int kChunks = (kVals + 15) / 16;
  __shared__ float sc[NQ][kTile];
  pdl_wait();
  pdl_trigger();
  const int unit = blockIdx.x;
  const int b = unit / Hkv, g = unit - b * Hkv;
  const int G = Hq / Hkv;
  const int tid = threadIdx.x;
  const int part = tid & 15;
  const int sub = tid >> 4;
  const int cta_c0 = blockIdx.y * kTile * kTilesPerCta;
  const uint4 *base = lm + (int64_t)unit * C * kVecPerRow + part;

  uint4 v[kPass], nv[kPass];
#pragma unroll
  for (int p = 0; p < kPass; ++p) {
    const int c = cta_c0 + p * kRowsPerPass + sub;
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

  for (int t = 0; t < kTilesPerCta; ++t) {
    const int c0 = cta_c0 + t * kTile;
    if (c0 >= C) break;
    if (t + 1 < kTilesPerCta) {
#pragma unroll
      for (int p = 0; p < kPass; ++p) {
        const int c = c0 + kTile + p * kRowsPerPass + sub;
        nv[p] = (c < C) ? ldg_nc(base + (int64_t)c * kVecPerRow) : make_uint4(0, 0, 0, 0);
      }
    }
    // partial dots: value a = p*NQ + j
    float x[kChunks * 16];
#pragma unroll
    for (int a = kVals; a < kChunks * 16; ++a) x[a] = 0.f;
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      float f[8];
      unpack8(v[p], f);
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(qs[j][e], f[e], acc);
        x[p * NQ + j] = acc;
      }
    }
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
      float xs[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) xs[i] = x[ch * 16 + i];
      const float r = butterfly16(xs, part);
      const int a = ch * 16 + part;
      if (a < kVals) sc[a % NQ][(a / NQ) * kRowsPerPass + sub] = r;
    }
    __syncthreads();
    for (int i = tid; i < NQ * kTile; i += kScoreThreads) {
      const int j = i / kTile, cc = i - j * kTile;
      const int c = c0 + cc;
      if (c < C) scores[((int64_t)(b * NQ + j) * Hkv + g) * C + c] = sc[j][cc];
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < kPass; ++p) v[p] = nv[p];
  }
}

cudaError_t launch_score(const uint4 *q, const uint4 *lm, float *scores, int B, int n_q, int Hq, int Hkv, int C,
                         cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  dim3 grid(B * Hkv, (C + kTile * kTilesPerCta - 1) / (kTile * kTilesPerCta));
  switch (n_q) {
#define DD_SCORE_CASE(N) \
  case N: return launch_k(k_score<N>, grid, dim3(kScoreThreads), 0, s, q, lm, scores, Hq, Hkv, C);
    DD_SCORE_CASE(1) DD_SCORE_CASE(2) DD_SCORE_CASE(3) DD_SCORE_CASE(4)
    DD_SCORE_CASE(5) DD_SCORE_CASE(6) DD_SCORE_CASE(7) DD_SCORE_CASE(8)
#undef DD_SCORE_CASE
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dd
