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
  // no early trigger: the scoring kernel reads landmarks before its
  // dependency wait, so a kernel that writes them releases its dependents
  // only when it exits
  pdl_wait();
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
  pdl_wait();   // no early trigger (see k_build_landmarks)
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
// a1 on the CUDA cores, for min/max landmarks: scores[b,j,g,c] =
// sum_i max(qsum_i * min_i, qsum_i * max_i) with qsum the fp32 sum of the
// group's G query heads (the largest value qsum . k can take over any key k
// inside the chunk's box), which is not a product the tensor cores can take.
// (The kernel also holds the mean-landmark form qsum . lm, which mean
// landmarks no longer use: they are scored on the tensor cores,
// dd_score_tc.cu.)
//
// The landmarks of all (b,g) units lie end to end in HBM, and scoring reads
// each of their bytes once, so the kernel is a stream: two CTAs per SM each
// take an equal contiguous span of landmark rows (a multiple of a ring stage)
// and pull it through a ring of kScoreStages 32 KB shared-memory stages with
// 1-D bulk copies (one thread issues; completion on an mbarrier per stage,
// bounded waits).  A stage never crosses a unit boundary, so every stage
// scores against one unit's group sums (rebuilt when the unit changes).
// 16 lanes share one landmark row (one 16-byte shared-memory load per
// vector each) and every thread scores kPass rows of a stage for all NQ
// queries; the 16-lane reduction of the kPass*NQ partial dots is a butterfly
// that halves the value set at every step (8+4+2+1 shuffles per 16 dots),
// leaving dot (lane position) in each lane.  Each (row, query) sum therefore
// has one fixed order: an fmaf chain over the lane's 8 coordinates, then the
// xor-8/4/2/1 tree over the 16 lanes.  A stage's scores are gathered in
// shared memory and written out as contiguous runs of each query row.
// ---------------------------------------------------------------------------
constexpr int kScoreThreads = 256;
constexpr int kScoreRowsPerPass = kScoreThreads / 16;     // 16 landmark rows per pass
constexpr int kScoreStages = 3;
constexpr int kScoreCtasPerSm = 2;   // two issuers per SM: one streams while the other scores
constexpr int kScoreStageBytes = 32 * 1024;
__host__ __device__ constexpr int score_stage_rows(bool mm) { return kScoreStageBytes / (mm ? 512 : 256); }
__host__ __device__ constexpr size_t score_smem(int n_q, bool mm) {
  return (size_t)kScoreStages * kScoreStageBytes + 2 * (size_t)n_q * score_stage_rows(mm) * 4;
}

template <int NQ, bool MM>
__global__ void __launch_bounds__(kScoreThreads, kScoreCtasPerSm) k_score(const uint4 *__restrict__ q, const uint4 *__restrict__ lm,
                                                            float *__restrict__ scores, int Hq, int Hkv, int C,
                                                            int64_t total_rows, int64_t rows_per_cta,
                                                            int32_t *status, unsigned long long *trace) {
  constexpr int kVecs = MM ? 2 : 1;                       // vectors per landmark
  constexpr int kRowBytes = 256 * kVecs;
  constexpr int kStageRows = score_stage_rows(MM);       // 128 or 64
  constexpr int kPass = kStageRows / kScoreRowsPerPass;   // rows per thread per stage: 8 or 4
  constexpr int kVals = kPass * NQ;                       // partial dots per lane per stage
  constexpr int kChunks = (kVals + 15) / 16;
  extern __shared__ __align__(128) unsigned char ssm[];
  unsigned char *ring = ssm;
  float *outb = reinterpret_cast<float *>(ssm + kScoreStages * kScoreStageBytes);   // [2][NQ][kStageRows]
  __shared__ __align__(8) uint64_t bar[kScoreStages];
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < kScoreStages; ++i) mbar_init(smem_u32(&bar[i]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int64_t lo = (int64_t)blockIdx.x * rows_per_cta;
  const int span = (int)((lo + rows_per_cta < total_rows ? lo + rows_per_cta : total_rows) - lo);
  const unsigned char *src = reinterpret_cast<const unsigned char *>(lm) + lo * kRowBytes;
  const int unit0 = (int)(lo / C), c_first = (int)(lo - (int64_t)unit0 * C);
  // a stage: up to kStageRows rows, within the span and within one unit; the
  // issuing thread and the consumers walk the same sequence with their own
  // cursors (row offset in the span, chunk index in the unit)
  auto stage_rows = [&](int done, int c) { return min(min(kStageRows, span - done), C - c); };
  int i_done = 0, i_c = c_first, st_issue = 0;   // issuing thread only
  auto issue = [&]() {
    const int n = stage_rows(i_done, i_c);
    const int rb = st_issue % kScoreStages;
    const uint32_t b = smem_u32(&bar[rb]);
    mbar_arrive_expect_tx(b, (uint32_t)n * kRowBytes);
    bulk_load(smem_u32(ring + rb * kScoreStageBytes), src + (int64_t)i_done * kRowBytes, (uint32_t)n * kRowBytes, b);
    i_done += n;
    i_c += n;
    if (i_c == C) i_c = 0;
    ++st_issue;
  };
  // The landmarks are not written by the kernel this one may overlap (the
  // landmark builders release their dependents only at exit), so the first
  // ring stages are requested before the dependency wait: the stream's ramp
  // overlaps the previous kernel's tail.  The queries and the score rows wait.
  if (tid == 0)
    while (st_issue < kScoreStages && i_done < span) issue();
  pdl_wait();
  pdl_trigger();
  // the step's critical path: from the end of the kernel before this one
  if (trace && tid == 0) trace_start(trace);

  const int part = tid & 15, sub = tid >> 4;
  const int G = Hq / Hkv;
  float qs[NQ][8];
  int unit = unit0, c0 = c_first, done = 0, st = 0;
  bool fresh = true;   // the group sums of `unit` are still to be built
  for (; done < span; ++st) {
    const int n = stage_rows(done, c0);
    const int b = unit / Hkv, g = unit - b * Hkv;
    if (fresh) {   // this lane's 8 coordinates of each query's group sum
      fresh = false;
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
    }
    const int rb = st % kScoreStages;
    const bool ok = mbar_wait(smem_u32(&bar[rb]), (uint32_t)(st / kScoreStages) & 1u, status);
    const unsigned char *stage = ring + rb * kScoreStageBytes;
    float *out = outb + (st & 1) * NQ * kStageRows;
    float x[kChunks * 16];
#pragma unroll
    for (int a = kVals; a < kChunks * 16; ++a) x[a] = 0.f;
#pragma unroll
    for (int p = 0; p < kPass; ++p) {
      const int row = p * kScoreRowsPerPass + sub;
      const bool live = ok && row < n;
      const uint4 *v = reinterpret_cast<const uint4 *>(stage + row * kRowBytes) + part;
      float f[8], fh[8];
      unpack8(live ? v[0] : make_uint4(0, 0, 0, 0), f);
      if (MM) unpack8(live ? v[kVecPerRow * (kVecs - 1)] : make_uint4(0, 0, 0, 0), fh);
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
      const float s = butterfly16(xs, part);
      const int a = ch * 16 + part;
      if (a < kVals) out[(a % NQ) * kStageRows + (a / NQ) * kScoreRowsPerPass + sub] = s;
    }
    // stage rb consumed by every warp (and the scores of this stage are in
    // `out`); a timed-out wait anywhere ends the CTA's loop on every thread
    if (__syncthreads_or(!ok)) break;
    if (tid == 0 && i_done < span) issue();
    // the other half of the double-buffered `out` is written only after the
    // next barrier, which every thread reaches after these stores
    float *dst = scores + ((int64_t)(b * NQ) * Hkv + g) * C + c0;
#pragma unroll
    for (int i = tid; i < NQ * kStageRows; i += kScoreThreads) {
      const int j = i / kStageRows, cc = i % kStageRows;
      if (cc < n) dst[(int64_t)j * Hkv * C + cc] = out[i];
    }
    done += n;
    c0 += n;
    if (c0 == C) {
      c0 = 0;
      ++unit;
      fresh = true;
    }
  }
  // after a timed-out wait: let the copies still in flight land (bounded) before the CTA exits
  if (done < span && tid == 0)
    for (int s2 = st + 1; s2 < st_issue; ++s2)
      mbar_wait(smem_u32(&bar[s2 % kScoreStages]), (uint32_t)(s2 / kScoreStages) & 1u, status);
  if (trace) {
    __syncthreads();
    if (tid == 0) trace_end(trace);
  }
}

template <bool MM>
static cudaError_t launch_score_t(const uint4 *q, const uint4 *lm, float *scores, int B, int n_q, int Hq, int Hkv,
                                  int C, int sm_count, int32_t *status, unsigned long long *trace, cudaStream_t s) {
  const int64_t total = (int64_t)B * Hkv * C;
  if (total == 0) return cudaSuccess;
  constexpr int kStageRows = score_stage_rows(MM);
  const int64_t stages = (total + kStageRows - 1) / kStageRows;
  const int64_t slots = (int64_t)kScoreCtasPerSm * (sm_count > 0 ? sm_count : 1);
  const int64_t ctas = slots < stages ? slots : stages;
  const int64_t per = (stages + ctas - 1) / ctas * kStageRows;   // rows per CTA, whole stages
  const int grid = (int)((total + per - 1) / per);
  const size_t smem = score_smem(n_q, MM);
  switch (n_q) {
#define DD_SCORE_CASE(N)                                                                                         \
  case N: {                                                                                                       \
    cudaError_t e = set_dyn_smem((const void *)k_score<N, MM>, smem);                                         \
    if (e != cudaSuccess) return e;                                                                               \
    return launch_k(k_score<N, MM>, dim3(grid), dim3(kScoreThreads), smem, s, q, lm, scores, Hq, Hkv, C, total,   \
                    per, status, trace);                                                                          \
  }
    DD_SCORE_CASE(1) DD_SCORE_CASE(2) DD_SCORE_CASE(3) DD_SCORE_CASE(4)
    DD_SCORE_CASE(5) DD_SCORE_CASE(6) DD_SCORE_CASE(7) DD_SCORE_CASE(8)
#undef DD_SCORE_CASE
    default: return cudaErrorInvalidValue;
  }
}

// mean landmarks: a product of the landmark rows with the query vectors, on
// the tensor cores (dd_score_tc.cu)
cudaError_t launch_score(const uint4 *q, const uint4 *lm, float *scores, int B, int n_q, int Hq, int Hkv, int C,
                         int sm_count, int32_t *status, cudaStream_t s, unsigned long long *trace) {
  return launch_score_tc(q, lm, scores, B, n_q, Hq, Hkv, C, sm_count, status, s, trace);
}

cudaError_t launch_score_minmax(const uint4 *q, const uint4 *lm2, float *scores, int B, int n_q, int Hq, int Hkv,
                                int C, int sm_count, int32_t *status, cudaStream_t s, unsigned long long *trace) {
  return launch_score_t<true>(q, lm2, scores, B, n_q, Hq, Hkv, C, sm_count, status, trace, s);
}

}  // namespace dd
