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
// a0, second landmark kind (OasisKV Methodology, Quest-style summaries): the
// coordinate-wise minimum and maximum key of each chunk, lm2[chunk][0][:] and
// lm2[chunk][1][:].  The extremes are taken on order keys of the bf16 bit
// patterns (-0 below +0), two 16-bit keys per 32-bit word with the SIMD
// min/max instructions, so the result is exact and unique.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t bf2_order_key(uint32_t w) {
  const uint32_t neg = ((w >> 15) & 0x00010001u) * 0xFFFFu;   // 0xFFFF in each negative half
  return w ^ (neg | 0x80008000u);
}

__device__ __forceinline__ uint32_t bf2_from_order_key(uint32_t k) {
  const uint32_t neg = ((~k >> 15) & 0x00010001u) * 0xFFFFu;  // halves whose key top bit is clear
  return k ^ (neg | 0x80008000u);
}

__global__ void __launch_bounds__(256) k_build_minmax(const uint4 *__restrict__ K, uint4 *__restrict__ lm2,
                                                       int64_t n_chunks, int cs) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t chunk = gid >> 4;
  const int part = (int)(gid & 15);
  if (chunk >= n_chunks) return;
  const uint4 *src = K + chunk * cs * kVecPerRow + part;
  uint4 lo = make_uint4(~0u, ~0u, ~0u, ~0u), hi = make_uint4(0, 0, 0, 0);
  for (int t0 = 0; t0 < cs; t0 += 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = (t0 + u < cs) ? src[(int64_t)(t0 + u) * kVecPerRow] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (t0 + u < cs) {
        const uint32_t kx = bf2_order_key(v[u].x), ky = bf2_order_key(v[u].y);
        const uint32_t kz = bf2_order_key(v[u].z), kw = bf2_order_key(v[u].w);
        lo.x = __vminu2(lo.x, kx); hi.x = __vmaxu2(hi.x, kx);
        lo.y = __vminu2(lo.y, ky); hi.y = __vmaxu2(hi.y, ky);
        lo.z = __vminu2(lo.z, kz); hi.z = __vmaxu2(hi.z, kz);
        lo.w = __vminu2(lo.w, kw); hi.w = __vmaxu2(hi.w, kw);
      }
    }
  }
  uint4 *dst = lm2 + chunk * 2 * kVecPerRow + part;
  dst[0] = make_uint4(bf2_from_order_key(lo.x), bf2_from_order_key(lo.y), bf2_from_order_key(lo.z),
                      bf2_from_order_key(lo.w));
  dst[kVecPerRow] = make_uint4(bf2_from_order_key(hi.x), bf2_from_order_key(hi.y), bf2_from_order_key(hi.z),
                               bf2_from_order_key(hi.w));
}

cudaError_t launch_build_minmax(const uint4 *K, uint4 *lm2, int64_t n_chunks, int cs, cudaStream_t s) {
  if (n_chunks == 0) return cudaSuccess;
  const int64_t blocks = (n_chunks * 16 + 255) / 256;
  return launch_k(k_build_minmax, dim3((unsigned)blocks), dim3(256), 0, s, K, lm2, n_chunks, cs);
}

// ---------------------------------------------------------------------------
// a1: scores[b,j,g,c] = qsum[b,j,g,:] . lm[b,g,c,:] with qsum the fp32 sum of
// the group's G query heads (mean landmarks), or
// sum_i max(qsum_i * min_i, qsum_i * max_i) (min/max landmarks: the largest
// value qsum . k can take over any key k inside the chunk's box).  One CTA
// scores kTilesPerCta tiles of landmarks of one (b,g) for all NQ queries, so
// every landmark byte is read once.  16 lanes share one landmark (one
// 16-byte load per vector each); each thread holds kPass landmarks of a tile
// (8, or 4 of the twice as large min/max ones) and the loads of the next tile
// are in flight while the current one is reduced.  The 16-lane reduction of
// the kPass*NQ partial dots is a butterfly that halves the value set at every
// step (8+4+2+1 shuffles per 16 dots), leaving dot (lane position) in each
// lane.
// ---------------------------------------------------------------------------
constexpr int kScoreThreads = 256;
constexpr int kRowsPerPass = kScoreThreads / 16;          // 16
constexpr int kTilesPerCta = 4;
__host__ __device__ constexpr int score_pass(bool mm) { return mm ? 4 : 8; }
__host__ __device__ constexpr int score_tile(bool mm) { return score_pass(mm) * kRowsPerPass; }

template <int NQ, bool MM>
__global__ void __launch_bounds__(kScoreThreads) k_score(const uint4 *__restrict__ q, const uint4 *__restrict__ lm,
                                                         float *__restrict__ scores, int Hq, int Hkv, int C) {
  constexpr int kPass = score_pass(MM);
  constexpr int kTile = score_tile(MM);
  constexpr int kVecs = MM ? 2 : 1;                       // vectors per landmark
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
  const uint4 *base = lm + (int64_t)unit * C * kVecs * kVecPerRow + part;

  uint4 v[kPass][kVecs], nv[kPass][kVecs];
#pragma unroll
  for (int p = 0; p < kPass; ++p) {
    const int c = cta_c0 + p * kRowsPerPass + sub;
#pragma unroll
    for (int e = 0; e < kVecs; ++e)
      v[p][e] = (c < C) ? ldg_nc(base + ((int64_t)c * kVecs + e) * kVecPerRow) : make_uint4(0, 0, 0, 0);
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
#pragma unroll
        for (int e = 0; e < kVecs; ++e)
          nv[p][e] = (c < C) ? ldg_nc(base + ((int64_t)c * kVecs + e) * kVecPerRow) : make_uint4(0, 0, 0, 0);
      }
    }
    // partial dots: value a = p*NQ + j
    float x[kChunks * 16];
#pragma unroll
    for (int a = kVals; a < kChunks * 16; ++a) x[a] = 0.f;
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      float f[8], fh[8];
      unpack8(v[p][0], f);
      if (MM) unpack8(v[p][kVecs - 1], fh);
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        float acc = 0.f;
        if (MM) {
#pragma unroll
          for (int e = 0; e < 8; ++e) acc += fmaxf(qs[j][e] * f[e], qs[j][e] * fh[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = fmaf(qs[j][e], f[e], acc);
        }
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
    for (int p = 0; p < kPass; ++p)
#pragma unroll
      for (int e = 0; e < kVecs; ++e) v[p][e] = nv[p][e];
  }
}

template <bool MM>
static cudaError_t launch_score_t(const uint4 *q, const uint4 *lm, float *scores, int B, int n_q, int Hq, int Hkv,
                                  int C, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const int per_cta = score_tile(MM) * kTilesPerCta;
  dim3 grid(B * Hkv, (C + per_cta - 1) / per_cta);
  switch (n_q) {
#define DD_SCORE_CASE(N) \
  case N: return launch_k(k_score<N, MM>, grid, dim3(kScoreThreads), 0, s, q, lm, scores, Hq, Hkv, C);
    DD_SCORE_CASE(1) DD_SCORE_CASE(2) DD_SCORE_CASE(3) DD_SCORE_CASE(4)
    DD_SCORE_CASE(5) DD_SCORE_CASE(6) DD_SCORE_CASE(7) DD_SCORE_CASE(8)
#undef DD_SCORE_CASE
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_score(const uint4 *q, const uint4 *lm, float *scores, int B, int n_q, int Hq, int Hkv, int C,
                         cudaStream_t s) {
  return launch_score_t<false>(q, lm, scores, B, n_q, Hq, Hkv, C, s);
}

cudaError_t launch_score_minmax(const uint4 *q, const uint4 *lm2, float *scores, int B, int n_q, int Hq, int Hkv,
                                int C, cudaStream_t s) {
  return launch_score_t<true>(q, lm2, scores, B, n_q, Hq, Hkv, C, s);
}

}  // namespace dd
