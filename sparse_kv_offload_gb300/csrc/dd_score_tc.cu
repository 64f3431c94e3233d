// a1 with mean landmarks on the fifth-generation tensor cores (tcgen05).
//
// DualDecoder §4.1 scores every chunk by its landmark (the mean key) against
// the step's queries; OasisKV summary / Methodology rank the blocks of each KV
// head.  For a (request b, KV head g) unit the scores of its n_q queries are
//
//   scores[b,j,g,c] = sum over the G query heads h of group g of q[b,j,h,:] . lm[b,g,c,:]
//
// a product of the unit's C landmark rows with its NQ = n_q * G query vectors
// (K = 128), followed by a sum over each query's G columns.  With several
// queries per request (a real one plus drafts) the CUDA-core scoring spends
// more issue slots on the products than the stream takes to arrive; here the
// products run on the tensor cores and the kernel is a stream of the
// landmarks:
//
//   tiles      128 landmark rows (M), both 64-column halves by two 2-D TMA
//              boxes into a five-stage ring (128-byte swizzle, K-major A);
//              each CTA takes an equal contiguous span of all units' tiles,
//              the first stages requested before the dependency wait
//   queries    the unit's NQ vectors by two 4-D TMA boxes (rows j*G + h, the
//              B operand, K-major), double-buffered by unit parity and freed
//              by a tcgen05.commit when the next unit begins
//   MMA        one thread: eight K = 16 steps per tile, M = 128, N = NQ rounded
//              up to 16, fp32 accumulators in tensor memory (two buffers)
//   epilogue   four warps, one tensor-memory lane (one landmark row) per
//              thread: the NQ columns by tcgen05.ld, the G columns of each
//              query summed in head order in fp32, the scores stored as runs
//              of consecutive chunks
//
// Products of bf16 values are exact in fp32; each per-head dot product is
// accumulated in fp32 by the tensor core and the G heads are then added in
// fp32, which keeps every score within the fp32 accumulation bound of the
// exact value (min/max landmarks are not a product and stay on the CUDA cores
// in dd_score.cu).
#include "dd_tc.cuh"

namespace dd {

namespace {

constexpr int kScRows = 128;                 // landmark rows per tile (M)
constexpr int kScHalf = kScRows * 128;       // a 64-column half of a tile, 16 KiB
constexpr int kScTile = 2 * kScHalf;         // 32 KiB
constexpr int kScStages = 5;
constexpr int kScQHalf = 64 * 128;           // a 64-column half of a query tile (up to 64 vectors)
constexpr int kScThreads = 192;              // TMA warp, MMA warp, four epilogue warps
constexpr int kScTmemCols = 128;             // two accumulators of up to 64 columns

// [ring][query tiles: 2 units x 2 halves][mbarriers: full, empty per stage;
// acc_full[2], acc_empty[2], q_free[2], mma_done]
constexpr size_t kScSmem = 1024 + (size_t)kScStages * kScTile + 4 * (size_t)kScQHalf + (2 * kScStages + 7) * 8;

// NQP: query vectors rounded up to 16 (N of the MMA, accumulator columns);
// GT: the group size G when known at compile time (the epilogue's column sums
// then unroll to G - 1 adds per query), 0 for any G
template <int NQP, int GT>
__global__ void __launch_bounds__(kScThreads, 1)
    k_score_tc(const __grid_constant__ CUtensorMap tm_lm, const __grid_constant__ CUtensorMap tm_q,
               float *__restrict__ scores, int n_q, int G, int Hkv, int C, int64_t total_tiles,
               int32_t *status, unsigned long long *trace) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *ring = smem;
  uint8_t *qbuf = ring + kScStages * kScTile;
  uint64_t *bars = reinterpret_cast<uint64_t *>(qbuf + 4 * kScQHalf);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kScStages);
  const uint32_t afull0 = smem_u32(bars + 2 * kScStages), aempty0 = smem_u32(bars + 2 * kScStages + 2);
  const uint32_t qfree0 = smem_u32(bars + 2 * kScStages + 4), mmadone = smem_u32(bars + 2 * kScStages + 6);
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tpu = (C + kScRows - 1) / kScRows;   // tiles per unit
  // CTA c takes tiles [c T / n, (c + 1) T / n) of all T: spans differ by one
  // tile at most, and every SM holds one CTA (a selection CTA launched early
  // then finds room for exactly one of its own beside it on each SM)
  const int64_t t0 = (int64_t)blockIdx.x * total_tiles / gridDim.x;
  const int64_t t1 = ((int64_t)blockIdx.x + 1) * total_tiles / gridDim.x;
  if (t0 >= t1) return;
  const int n = (int)(t1 - t0);
  const int NQ = n_q * G;

  if (tid == 0) {
    for (int i = 0; i < kScStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(afull0 + 8 * i, 1);
      mbar_init(aempty0 + 8 * i, 4);   // one arrival per epilogue warp
      mbar_init(qfree0 + 8 * i, 1);
    }
    mbar_init(mmadone, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kScTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA issue
    if (lane == 0) {
      // the landmarks are not written by the kernels this one may overlap: the
      // first stages' boxes go out before the dependency wait (their bytes
      // expected now, the arrival once the unit's queries are issued too)
      const int pre = n < kScStages ? n : kScStages;
      for (int s = 0; s < pre; ++s) {
        const int64_t t = t0 + s;
        const int u = (int)(t / tpu), i = (int)(t - (int64_t)u * tpu);
        const int row0 = u * C + i * kScRows;
        const uint32_t bar = full0 + 8 * s, dst = smem_u32(ring + s * kScTile);
        mbar_expect_tx(bar, (uint32_t)kScTile);
        tma_load_2d(dst, &tm_lm, 0, row0, bar);
        tma_load_2d(dst + kScHalf, &tm_lm, 64, row0, bar);
      }
      pdl_wait();
      pdl_trigger();
      if (trace) trace_start(trace);
      int run = 0, prev = -1;
      for (int s = 0; s < n; ++s) {
        const int slot = s % kScStages;
        const int64_t t = t0 + s;
        const int u = (int)(t / tpu), i = (int)(t - (int64_t)u * tpu);
        if (s >= kScStages && !mbar_wait(empty0 + 8 * slot, ((s / kScStages) - 1) & 1, status)) break;
        const bool first = u != prev;
        prev = u;
        // the query tile of unit number run (this CTA's) is reused two units
        // later, once every product that read it is done
        if (first && run >= 2 && !mbar_wait(qfree0 + 8 * (run & 1), ((run >> 1) - 1) & 1, status)) break;
        const uint32_t bar = full0 + 8 * slot;
        mbar_arrive_expect_tx(bar, (first ? (uint32_t)NQ * 256u : 0u) + (s >= pre ? (uint32_t)kScTile : 0u));
        if (first) {
          const int b = u / Hkv, g = u - b * Hkv;
          const uint32_t qd = smem_u32(qbuf + (run & 1) * 2 * kScQHalf);
          tma_load_4d(qd, &tm_q, 0, g * G, 0, b, bar);
          tma_load_4d(qd + kScQHalf, &tm_q, 64, g * G, 0, b, bar);
          ++run;
        }
        if (s >= pre) {
          const uint32_t dst = smem_u32(ring + slot * kScTile);
          tma_load_2d(dst, &tm_lm, 0, u * C + i * kScRows, bar);
          tma_load_2d(dst + kScHalf, &tm_lm, 64, u * C + i * kScRows, bar);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kScRows, NQP, 0, 0);
      int run = 0, prev = -1;
      uint32_t qb = smem_u32(qbuf);
      for (int s = 0; s < n; ++s) {
        const int slot = s % kScStages;
        if (!mbar_wait(full0 + 8 * slot, (s / kScStages) & 1, status)) break;
        const int u = (int)((t0 + s) / tpu);
        if (u != prev) {
          prev = u;
          if (run > 0) tc_commit(qfree0 + 8 * ((run - 1) & 1));   // the previous unit's query tile, once read
          qb = smem_u32(qbuf + (run & 1) * 2 * kScQHalf);
          ++run;
        }
        const int buf = s & 1;
        if (s >= 2 && !mbar_wait(aempty0 + 8 * buf, ((s >> 1) - 1) & 1, status)) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(ring + slot * kScTile);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc_mma(tmem + buf * 64, smem_desc_sw128(a0 + (ks >> 2) * kScHalf + (ks & 3) * 32, 16, 1024),
                 smem_desc_sw128(qb + (ks >> 2) * kScQHalf + (ks & 3) * 32, 16, 1024), idesc, ks > 0);
        tc_commit(empty0 + 8 * slot);
        tc_commit(afull0 + 8 * buf);
      }
      // every product issued has completed before the tensor memory is freed
      tc_commit(mmadone);
      mbar_wait(mmadone, 0, status);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- epilogue
    pdl_wait();   // the score rows are written after the dependency wait
    const int q4 = warp & 3, row = 32 * q4 + lane;   // this thread's tensor-memory lane: landmark row of the tile
    for (int s = 0; s < n; ++s) {
      const int buf = s & 1;
      if (!mbar_wait(afull0 + 8 * buf, (s >> 1) & 1, status)) break;
      tc_fence_after();
      float v[NQP];
#pragma unroll
      for (int c = 0; c < NQP / 16; ++c) tmem_ld32x32b_x16(tmem + ((uint32_t)(32 * q4) << 16) + buf * 64 + 16 * c, v + 16 * c);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty0 + 8 * buf);
      const int64_t t = t0 + s;
      const int u = (int)(t / tpu), i = (int)(t - (int64_t)u * tpu);
      const int c = i * kScRows + row;
      if (c < C) {
        const int b = u / Hkv, g = u - b * Hkv;
        float *dst = scores + ((int64_t)b * n_q * Hkv + g) * C + c;   // query j at + j * Hkv * C
        if (GT > 0) {
#pragma unroll
          for (int j = 0; j < NQP / (GT > 0 ? GT : 1); ++j)
            if (j < n_q) {
              float acc = v[j * GT];   // the query's G columns, in head order
#pragma unroll
              for (int h = 1; h < GT; ++h) acc += v[j * GT + h];
              dst[(int64_t)j * Hkv * C] = acc;
            }
        } else {
          for (int j = 0; j < n_q; ++j) {
            float acc = 0.f;
#pragma unroll
            for (int h = 0; h < NQP; ++h)   // the query's G columns, in head order
              if (h >= j * G && h < (j + 1) * G) acc += v[h];
            dst[(int64_t)j * Hkv * C] = acc;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kScTmemCols) : "memory");
  }
  if (trace && tid == 0) trace_end(trace);
}

}  // namespace

cudaError_t launch_score_tc(const void *q, const void *lm, float *scores, int B, int n_q, int Hq, int Hkv, int C,
                            int sm_count, int32_t *status, cudaStream_t s, unsigned long long *trace) {
  const int64_t units = (int64_t)B * Hkv;
  if (units == 0 || C == 0) return cudaSuccess;
  const int G = Hq / Hkv, NQ = n_q * G;
  if (NQ > 64) return cudaErrorInvalidValue;
  CUtensorMap tlm, tq;
  if (!make_pool_map(&tlm, lm, units * C, kScRows) || !make_q_map(&tq, q, B, n_q, Hq, G)) return cudaErrorInvalidValue;
  const int64_t total = units * ((C + kScRows - 1) / kScRows);
  const int grid = (int)(sm_count > 0 && sm_count < total ? sm_count : total);
  const int P = (NQ + 15) / 16;
#define DD_SCORE_TC(NQP, GT)                                                                                   \
  do {                                                                                                          \
    cudaError_t e = set_dyn_smem((const void *)k_score_tc<NQP, GT>, kScSmem);                                  \
    if (e != cudaSuccess) return e;                                                                             \
    return launch_k(k_score_tc<NQP, GT>, dim3(grid), dim3(kScThreads), kScSmem, s, tlm, tq, scores, n_q, G,     \
                    Hkv, C, total, status, trace);                                                              \
  } while (0)
  // the common group sizes with their column sums unrolled, any other G generically
  if (G == 8) {
    if (P == 1) DD_SCORE_TC(16, 8);
    if (P == 2) DD_SCORE_TC(32, 8);
    if (P == 3) DD_SCORE_TC(48, 8);
    DD_SCORE_TC(64, 8);
  }
  if (G == 4) {
    if (P == 1) DD_SCORE_TC(16, 4);
    DD_SCORE_TC(32, 4);
  }
  if (P == 1) DD_SCORE_TC(16, 0);
  if (P == 2) DD_SCORE_TC(32, 0);
  if (P == 3) DD_SCORE_TC(48, 0);
  DD_SCORE_TC(64, 0);
#undef DD_SCORE_TC
}

}  // namespace dd
