// Split-K GQA decode attention over the deduplicated union of the queries'
// selected chunks.
//
// DualDecoder §5.2: the output token and the speculative token attend in one
// pass instead of two.  Adaptive DHiSparse Fig. 3 / OasisKV Methodology: the
// normal and draft queries share the HBM working set, but query j only sees
// the chunks it picked.  Every union row is streamed from HBM once and serves
// all NQ = n_q*G query vectors of its KV head; rows of a chunk a query did not
// pick are masked for that query (the chunk's query mask).
//
// Work split ("stream-K"): the unions of all (request, KV head) units are
// laid end to end (chunk_off = exclusive prefix of the union sizes) and each
// persistent CTA takes an equal contiguous slice of that sequence (two CTAs
// per SM for up to 16 query vectors per KV head, so that one's producer
// issues copies while the other's does its per-stage bookkeeping or waits on
// a fresh slice's tables).  A slice covers a few units ("runs").  At the end
// of a run the consumer warps that share an m-tile merge their states in
// shared memory.  A unit that lies inside one slice is then complete and its
// outputs are written at once.  For a unit shared by several CTAs the CTA
// writes one partial (running max, sum and accumulator per query vector) into
// slot CTA + unit -- slices are ordered like the units, so no two (CTA, unit)
// pairs share a slot and n_cta + units slots suffice -- and counts itself in
// on the unit's arrival counter; the CTA that arrives last merges the unit's
// partials (stream-K fix-up), so the outputs leave the same kernel.  Only a
// slice's first run can continue a unit begun earlier without being its last
// run; when the gather is not fused, that run's count (and merge) is left to
// the otherwise idle second producer warp, so the consumers never wait on a
// GPU-scope round trip in the middle of their slice.
//
// Data movement: the issuing producer warp streams 64-row tiles of K and V
// into shared memory with 2-D TMA loads (cp.async.bulk.tensor, 128-byte
// swizzle, one box per chunk and 64-column half) from the hot pool or the
// staging buffer, and each run's query vectors with bulk copies, all
// completing on mbarriers; it runs ahead across run boundaries with kStages
// tiles in flight.  When the gather is fused in, the other producer warp
// copies the slice's missing chunks from pinned host memory into staging
// ahead of it.  Math: consumer warps own 16 query vectors (one m16 tile) and
// 16- or 32-row slices of each tile; S = Q.K^T and O += P.V run on the tensor
// cores (mma.sync m16n8k16 bf16, fp32 accumulate) with an online softmax in
// fp32; P is split into bf16 hi + lo parts so the PV product keeps ~16
// significant bits.  The work is bound by HBM or the host link: the MMAs only
// keep the arithmetic under the memory time.
#include <cuda.h>
#include <mutex>
#include <cudaTypedefs.h>

#include "dd_attn.cuh"

namespace dd {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of (row, 16-byte column group cg in 0..15) inside a stage's
// K or V region: two 64-column halves, 128-byte rows, TMA 128B swizzle
// (16-byte chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t swz(int row, int cg) {
  return (uint32_t)((cg >> 3) * kHalfBytes + row * 128 + ((((cg & 7) ^ (row & 7))) << 4));
}

// ----------------------------------------------------------------- the kernel
// Registers per thread: the register file holds `ctas` CTAs (their threads
// rounded up to a multiple of 128); at most 224.
__host__ __device__ constexpr int attn_max_regs(int threads, int ctas) {
  return (65536 / ((ctas * threads + 127) / 128 * 128)) / 8 * 8 > 224
             ? 224
             : (65536 / ((ctas * threads + 127) / 128 * 128)) / 8 * 8;
}

// Producer warps: warp 0 issues the stages' metadata and every tile copy
// (TMA); in the fused gather warp 1 copies the slice's missing chunks from
// host memory into staging ahead of it, otherwise it counts the first run's
// partial in (the finisher).  Measured on the 16-request 32K
// layer, the host link moved the most with about 16 KB of 16-byte loads in
// flight per SM (2 x 8 per lane of one warp in each of two CTAs now; with
// one CTA per SM, 2 warps x 8 beat 1 x 16, 2 x 16, 4 x 16 and 1 x 4).
__host__ __device__ constexpr int producers_for(int) { return 2; }

template <int MT, int WPM>
__global__ void __maxnreg__(attn_max_regs((MT * WPM + producers_for(MT * WPM)) * 32, ctas_per_sm(MT)))
    k_attn(const __grid_constant__ CUtensorMap tm_khot, const __grid_constant__ CUtensorMap tm_vhot,
           const __grid_constant__ CUtensorMap tm_kst, const __grid_constant__ CUtensorMap tm_vst,
           const AttnParams p) {
  constexpr int kConsumers = MT * WPM;
  constexpr int kProducers = producers_for(kConsumers);
  constexpr int kStages = stages_for(MT);
  constexpr int kRowsPerWarp = kStageRows / WPM;      // 16, 32 or 64
  constexpr int kBlocks = kRowsPerWarp >= 32 ? kRowsPerWarp / 32 : 1;   // 16-row warps: half A only
  constexpr int kQBytes = 16 * MT * kQStride;

  extern __shared__ uint8_t smem_raw[];
  // the 128-byte swizzle pattern is anchored at 1024-byte shared-memory boundaries
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *stages = smem;                                                    // [kStages][64 KiB]
  uint8_t *qsm = stages + kStages * kStageBytes;                             // [kStages][16*MT][272 B]
  StageMeta *meta = reinterpret_cast<StageMeta *>(qsm + kStages * kQBytes);  // [kStages]
  uint64_t *bars = reinterpret_cast<uint64_t *>(meta + kStages);             // full[kStages], empty[kStages]

  __shared__ int s_fix;   // this CTA finished the last part of the unit whose run just ended
  __shared__ int s_ready; // fused gather: missing chunks of this slice already in staging, in slice order
  __shared__ int s_pub;   // partials the consumers handed to the finisher warp (one per m-tile and run)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_ready = 0;
    s_pub = 0;
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  // self-planned slice of the concatenated unions (the same split the fix-up assumes)
  const int total = p.chunk_off[p.units];
  const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
  const int lo = min(total, (int)blockIdx.x * per), hi = min(total, lo + per);
  if (lo >= hi) return;
  if (load_status(p.status) != 0) return;

  if (warp >= kConsumers) {
    attn_producer_warp<kStages>(p, &tm_khot, &tm_vhot, &tm_kst, &tm_vst, lo, hi, per, warp - kConsumers, stages,
                                qsm, kQBytes, meta, full0, empty0, &s_ready, &s_pub, MT);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int mt = warp / WPM, wq = warp - mt * WPM;
  const int gr = lane >> 2, tq = lane & 3;
  const int qv0 = mt * 16 + gr, qv1 = qv0 + 8;
  const int j0 = qv0 < p.NQ ? qv0 / p.G : 31;
  const int j1 = qv1 < p.NQ ? qv1 / p.G : 31;
  const float sl2 = p.scale_log2;
  const int rows_per_chunk_shift = 31 - __clz(p.cs);     // cs is a power of two

  uint32_t qa[8][4];
  float o[16][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int s = 0;; ++s) {
    const int buf = s % kStages;
    if (!mbar_wait(full0 + 8 * buf, (s / kStages) & 1, p.status)) break;
    const int m_nch = meta[buf].nch, m_flags = meta[buf].flags, m_unit = meta[buf].unit;
    const int m_uoff = meta[buf].uoff, m_ucnt = meta[buf].ucnt;
    const uint8_t *m_qm = meta[buf].qm;
    if (m_flags & kFirst) {
      // this run's query vectors from shared memory (padded rows: no bank conflicts)
      const uint8_t *qb = qsm + buf * kQBytes;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int c0 = (ks * 16 + 2 * tq) * 2, c1 = c0 + 16;
        qa[ks][0] = qv0 < p.NQ ? *reinterpret_cast<const uint32_t *>(qb + qv0 * kQStride + c0) : 0u;
        qa[ks][1] = qv1 < p.NQ ? *reinterpret_cast<const uint32_t *>(qb + qv1 * kQStride + c0) : 0u;
        qa[ks][2] = qv0 < p.NQ ? *reinterpret_cast<const uint32_t *>(qb + qv0 * kQStride + c1) : 0u;
        qa[ks][3] = qv1 < p.NQ ? *reinterpret_cast<const uint32_t *>(qb + qv1 * kQStride + c1) : 0u;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
    }
    const uint32_t kbase = smem_u32(stages + buf * kStageBytes);
    const uint32_t vbase = kbase + 2 * kHalfBytes;
#pragma unroll
    for (int blk = 0; blk < kBlocks; ++blk) {
      // 32 rows: halves A (rows row0..row0+15) and B (row0+16..row0+31), each
      // inside one chunk; a half outside the stage or with an empty mask is
      // skipped in both products (its shared memory may hold stale bytes)
      const int row0 = wq * kRowsPerWarp + blk * 32;
      const int ciA = row0 >> rows_per_chunk_shift, ciB = (row0 + 16) >> rows_per_chunk_shift;
      const uint32_t qmA = ciA < m_nch ? m_qm[ciA] : 0u;
      const uint32_t qmB = (kRowsPerWarp >= 32 && ciB < m_nch) ? m_qm[ciB] : 0u;
      if ((qmA | qmB) == 0) continue;
      const bool okA0 = (qmA >> j0) & 1u, okA1 = (qmA >> j1) & 1u;
      const bool okB0 = (qmB >> j0) & 1u, okB1 = (qmB >> j1) & 1u;

      // S = Q K^T: n8 tiles 0,1 from half A, 2,3 from half B
      float sc[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
      {
        const int mi = lane >> 3, r = lane & 7;
        const int krow = row0 + (mi >> 1) * 8 + r;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t cg = swz(krow, ks * 2 + (mi & 1));
          if (qmA) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + cg, b0, b1, b2, b3);
            mma_bf16(sc[0], qa[ks], b0, b1);
            mma_bf16(sc[1], qa[ks], b2, b3);
          }
          if (qmB) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + cg + 16 * 128, b0, b1, b2, b3);
            mma_bf16(sc[2], qa[ks], b0, b1);
            mma_bf16(sc[3], qa[ks], b2, b3);
          }
        }
      }
      // scale to log2 units and mask (rows gr and gr+8 of the m-tile)
      float x[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const bool o0 = n < 2 ? okA0 : okB0, o1 = n < 2 ? okA1 : okB1;
        x[n][0] = o0 ? sc[n][0] * sl2 : -INFINITY;
        x[n][1] = o0 ? sc[n][1] * sl2 : -INFINITY;
        x[n][2] = o1 ? sc[n][2] * sl2 : -INFINITY;
        x[n][3] = o1 ? sc[n][3] * sl2 : -INFINITY;
      }
      float mx0 = fmaxf(fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1])),
                        fmaxf(fmaxf(x[2][0], x[2][1]), fmaxf(x[3][0], x[3][1])));
      float mx1 = fmaxf(fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3])),
                        fmaxf(fmaxf(x[2][2], x[2][3]), fmaxf(x[3][2], x[3][3])));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float base0 = mn0 == -INFINITY ? 0.f : mn0;
      const float base1 = mn1 == -INFINITY ? 0.f : mn1;
      // rescale the accumulator only when some row's maximum moved
      if (__any_sync(0xffffffffu, mn0 != m0 || mn1 != m1)) {
        const float a0 = exp2f(m0 - base0), a1 = exp2f(m1 - base1);
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          o[i][0] *= a0;
          o[i][1] *= a0;
          o[i][2] *= a1;
          o[i][3] *= a1;
        }
      }
      m0 = mn0;
      m1 = mn1;
      float pr[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        pr[n][0] = exp2f(x[n][0] - base0);
        pr[n][1] = exp2f(x[n][1] - base0);
        pr[n][2] = exp2f(x[n][2] - base1);
        pr[n][3] = exp2f(x[n][3] - base1);
      }
      l0 += ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1])) + ((pr[2][0] + pr[2][1]) + (pr[3][0] + pr[3][1]));
      l1 += ((pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3])) + ((pr[2][2] + pr[2][3]) + (pr[3][2] + pr[3][3]));
      // P as the A operand of two k16 steps (halves A and B), split into bf16 hi + lo
      uint32_t ph[2][4], pl[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float v[4][2] = {{pr[2 * h][0], pr[2 * h][1]}, {pr[2 * h][2], pr[2 * h][3]},
                               {pr[2 * h + 1][0], pr[2 * h + 1][1]}, {pr[2 * h + 1][2], pr[2 * h + 1][3]}};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t hi = cvt_bf16x2(v[i][0], v[i][1]);
          ph[h][i] = hi;
          pl[h][i] = cvt_bf16x2(v[i][0] - bf_lo(hi), v[i][1] - bf_hi(hi));
        }
      }
      // O += P V: V fragments by transposed ldmatrix, two 8-column tiles per load
      {
        const int mi = lane >> 3, r = lane & 7;
        const int vrow = row0 + (mi & 1) * 8 + r;
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          const uint32_t cg = swz(vrow, dp * 2 + (mi >> 1));
          if (qmA) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(vbase + cg, v0, v1, v2, v3);
            mma_bf16(o[2 * dp], ph[0], v0, v1);
            mma_bf16(o[2 * dp + 1], ph[0], v2, v3);
            mma_bf16(o[2 * dp], pl[0], v0, v1);
            mma_bf16(o[2 * dp + 1], pl[0], v2, v3);
          }
          if (qmB) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(vbase + cg + 16 * 128, v0, v1, v2, v3);
            mma_bf16(o[2 * dp], ph[1], v0, v1);
            mma_bf16(o[2 * dp + 1], ph[1], v2, v3);
            mma_bf16(o[2 * dp], pl[1], v0, v1);
            mma_bf16(o[2 * dp + 1], pl[1], v2, v3);
          }
        }
      }
    }
    if (m_flags & kLast) {
      // the run is over: first merge the WPM warps of each m-tile, which hold
      // the same query rows over different key rows, into warp wq = 0.  Lane
      // l of partner warps holds the same (row, column) elements, so each
      // round is elementwise: warps [h, 2h) put their state into slots of the
      // stage just consumed (released only after the last round), warps
      // [0, h) rescale both to the larger maximum and add.
      if constexpr (WPM > 1) {
        static_assert(MT * (WPM / 2) * kMergeFloats * 32 * 4 <= kStageBytes, "merge slots exceed a stage");
        float *xs = reinterpret_cast<float *>(stages + buf * kStageBytes);
#pragma unroll
        for (int h = WPM / 2; h >= 1; h /= 2) {
          // every warp is done with the stage's tiles (first round) or with the last round's slots
          asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
          if (wq >= h && wq < 2 * h) {
            float *d = xs + (mt * h + wq - h) * (kMergeFloats * 32) + lane;
#pragma unroll
            for (int i = 0; i < 16; ++i)
#pragma unroll
              for (int e = 0; e < 4; ++e) d[(4 * i + e) * 32] = o[i][e];
            d[64 * 32] = m0;
            d[65 * 32] = m1;
            d[66 * 32] = l0;
            d[67 * 32] = l1;
          }
          asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
          if (wq < h) {
            const float *d = xs + (mt * h + wq) * (kMergeFloats * 32) + lane;
            const float mb0 = d[64 * 32], mb1 = d[65 * 32];
            const float M0 = fmaxf(m0, mb0), M1 = fmaxf(m1, mb1);
            const float sa0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M0), sb0 = mb0 == -INFINITY ? 0.f : exp2f(mb0 - M0);
            const float sa1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M1), sb1 = mb1 == -INFINITY ? 0.f : exp2f(mb1 - M1);
            l0 = l0 * sa0 + d[66 * 32] * sb0;
            l1 = l1 * sa1 + d[67 * 32] * sb1;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              o[i][0] = o[i][0] * sa0 + d[(4 * i + 0) * 32] * sb0;
              o[i][1] = o[i][1] * sa0 + d[(4 * i + 1) * 32] * sb0;
              o[i][2] = o[i][2] * sa1 + d[(4 * i + 2) * 32] * sb1;
              o[i][3] = o[i][3] * sa1 + d[(4 * i + 3) * 32] * sb1;
            }
            m0 = M0;
            m1 = M1;
          }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");   // the slots are read
        // order the slots' generic writes before the tile copies that refill the stage
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * buf);
      // CTAs c0..c1 hold parts of the unit.  A unit inside this slice (c0 ==
      // c1) is complete here: without tail rows its rows of each m-tile are
      // written straight from warp wq = 0.  Otherwise warp wq = 0 publishes
      // the CTA's partial into slot CTA + unit, and the CTA counts itself in
      // on the unit's arrival counter: here, or -- for the slice's first run
      // when it continues an earlier CTA's unit and is not the slice's last run
      // and the gather is not fused -- by the finisher warp, so that these
      // warps go straight on with the next run.
      const int c0 = m_uoff / per, c1 = (m_uoff + m_ucnt - 1) / per;
      const bool direct = c0 == c1 && p.k_tail == nullptr;
      const bool handoff = c0 != c1 && p.kh == nullptr && m_uoff < lo && !(m_flags & kEnd);
      if (wq == 0) {
        float lq0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
        lq0 += __shfl_xor_sync(0xffffffffu, lq0, 2);
        float lq1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
        lq1 += __shfl_xor_sync(0xffffffffu, lq1, 2);
        if (direct) {
          const int b = m_unit / p.Hkv, g = m_unit - b * p.Hkv;
          if (qv0 < p.NQ) {
            const int h = g * p.G + (qv0 - j0 * p.G);
            const float inv = lq0 > 0.f ? 1.f / lq0 : 0.f;
            float *dst = p.out + ((int64_t)(b * p.n_q + j0) * p.Hq + h) * 128 + 2 * tq;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              *reinterpret_cast<float2 *>(dst + i * 8) = make_float2(o[i][0] * inv, o[i][1] * inv);
          }
          if (qv1 < p.NQ) {
            const int h = g * p.G + (qv1 - j1 * p.G);
            const float inv = lq1 > 0.f ? 1.f / lq1 : 0.f;
            float *dst = p.out + ((int64_t)(b * p.n_q + j1) * p.Hq + h) * 128 + 2 * tq;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              *reinterpret_cast<float2 *>(dst + i * 8) = make_float2(o[i][2] * inv, o[i][3] * inv);
          }
        } else {
          const int64_t pbase = ((int64_t)blockIdx.x + m_unit) * p.NQ;
          if (qv0 < p.NQ) {
            float *dst = p.part_o + (pbase + qv0) * 128 + 2 * tq;
#pragma unroll
            for (int i = 0; i < 16; ++i) *reinterpret_cast<float2 *>(dst + i * 8) = make_float2(o[i][0], o[i][1]);
            if (tq == 0) *reinterpret_cast<float2 *>(p.part_ml + (pbase + qv0) * 2) = make_float2(m0, lq0);
          }
          if (qv1 < p.NQ) {
            float *dst = p.part_o + (pbase + qv1) * 128 + 2 * tq;
#pragma unroll
            for (int i = 0; i < 16; ++i) *reinterpret_cast<float2 *>(dst + i * 8) = make_float2(o[i][2], o[i][3]);
            if (tq == 0) *reinterpret_cast<float2 *>(p.part_ml + (pbase + qv1) * 2) = make_float2(m1, lq1);
          }
          if (handoff) {
            // the m-tile's partial is written: hand it to the finisher warp
            __syncwarp();
            if (lane == 0) asm volatile("red.release.cta.shared.add.u32 [%0], 1;" ::"r"(smem_u32(&s_pub)) : "memory");
          }
        }
      }
      // the next stage starts a new run, which reloads the queries and
      // restarts the accumulators, so none of them stays live through the
      // fix-up below
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) qa[ks][0] = qa[ks][1] = qa[ks][2] = qa[ks][3] = 0u;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
      if (!direct && !handoff) {
        // stream-K fix-up: the CTA that counts itself in last merges the
        // unit's partials (a unit inside one CTA needs no count).  The
        // barrier orders the CTA's partial before thread 0's count, and
        // thread 0's acquire before every thread's reads of the partials.
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");   // consumer warps only
        if (tid == 0) s_fix = c0 == c1 || atom_add_acq_rel_gpu(p.arrive + m_unit, 1) + 1 == c1 - c0 + 1;
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
        if (s_fix) fixup_unit(p, m_unit, c0, c1, kConsumers * 32, tid);
      }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * buf);
    }
    if (m_flags & kEnd) break;
  }
  if (p.trace) {
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");   // every consumer warp is done
    if (tid == 0) trace_end(p.trace);
  }
}

// --------------------------------------------------------------- plan
// Stand-alone plan for direct attention calls (the resolver builds the same
// plan itself inside a step): one CTA per unit.  A unit with an empty union
// gets zero outputs here, since no slice visits it.
constexpr int kPlanThreads = 256;

__global__ void __launch_bounds__(kPlanThreads) k_attn_plan(
    const int32_t *__restrict__ union_cnt, const int32_t *__restrict__ union_slot,
    const uint8_t *__restrict__ union_qmask, const int32_t *__restrict__ miss_count, AttnPlanOut po, float *out,
    int units, int umax, int n_q, int Hq, int Hkv, int64_t hot_slots, int64_t max_misses, int cs, int32_t *status,
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ k_tail, const uint16_t *__restrict__ v_tail,
    float scale_log2) {
  __shared__ int scratch[33];
  pdl_wait();
  pdl_trigger();
  const int unit = blockIdx.x;
  int before = 0, all = 0;
  for (int u = threadIdx.x; u < units; u += kPlanThreads) {
    int c = union_cnt[u];
    if (c < 0 || c > umax) {
      if (u == unit) set_status(status, DD_ERR_DEVICE_CHECK);
      c = c < 0 ? 0 : umax;
    }
    all += c;
    if (u < unit) before += c;
  }
  const int off = block_sum(before, scratch);
  const int total = block_sum(all, scratch);
  const int U = min(max(union_cnt[unit], 0), umax);
  const int64_t ubase = (int64_t)unit * umax;
  attn_plan_unit(po, unit, units, off, U, total, union_slot + ubase, union_qmask + ubase, nullptr, 0,
                 min((int64_t)*miss_count, max_misses), hot_slots, cs, status);
  if (U == 0) {
    // no slice visits this unit: its output is the attention over the tail
    // rows alone (rows 0..j for query j), or zero without them
    const int G = Hq / Hkv, b = unit / Hkv, g = unit - b * Hkv;
    for (int e = threadIdx.x; e < n_q * G * 128; e += kPlanThreads) {
      const int qv = e >> 7, col = e & 127, j = qv / G, h = g * G + (qv - j * G);
      float M = -INFINITY, L = 0.f, acc = 0.f;
      if (k_tail) {
        const uint16_t *qr = q + ((int64_t)(b * n_q + j) * Hq + h) * 128;
        for (int t = 0; t <= j; ++t) {
          const int64_t trow = ((int64_t)(b * n_q + t) * Hkv + g) * 128;
          float x = 0.f;
          for (int c = 0; c < 128; ++c)
            x = fmaf(__uint_as_float((uint32_t)qr[c] << 16), __uint_as_float((uint32_t)k_tail[trow + c] << 16), x);
          const float s2 = x * scale_log2, Mn = fmaxf(M, s2);
          const float a = M == -INFINITY ? 0.f : exp2f(M - Mn), w = exp2f(s2 - Mn);
          L = L * a + w;
          acc = acc * a + w * __uint_as_float((uint32_t)v_tail[trow + col] << 16);
          M = Mn;
        }
      }
      out[((int64_t)(b * n_q + j) * Hq + h) * 128 + col] = L > 0.f ? acc / L : 0.f;
    }
  }
}

// --------------------------------------------------------------- host side
struct AttnShape {
  int mt, wpm, threads;
  size_t smem;
};

AttnShape attn_shape(int NQ) {
  AttnShape s;
  s.mt = (NQ + 15) / 16;
  s.wpm = s.mt == 1 ? 4 : (s.mt == 4 ? 1 : 2);
  s.threads = (s.mt * s.wpm + producers_for(s.mt * s.wpm)) * 32;
  const int ns = stages_for(s.mt);
  s.smem = 1024 + (size_t)ns * kStageBytes + (size_t)ns * 16 * s.mt * kQStride + ns * sizeof(StageMeta) + 2 * ns * 8 + 16;
  return s;
}

// ctas_per_sm persistent CTAs per SM; partial slot CTA + unit for every
// (CTA, unit) pair that shares chunks.
AttnPlan attn_plan(int units, int umax, int NQ, int sm_count) {
  AttnPlan pl;
  pl.n_cta = sm_count > 0 ? ctas_per_sm(attn_shape(NQ).mt) * sm_count : 1;
  pl.part_o_floats = ((int64_t)pl.n_cta + units) * NQ * 128;
  pl.part_ml_floats = ((int64_t)pl.n_cta + units) * NQ * 2;
  pl.flat_entries = (int64_t)units * umax;
  return pl;
}

template <int MT, int WPM>
static cudaError_t launch_attn_t(int n_cta, const AttnShape &sh, const CUtensorMap &a, const CUtensorMap &b,
                                 const CUtensorMap &c, const CUtensorMap &d, const AttnParams &p, cudaStream_t s) {
  cudaError_t e = set_dyn_smem((const void *)k_attn<MT, WPM>, sh.smem);
  if (e != cudaSuccess) return e;
  return launch_k(k_attn<MT, WPM>, dim3(n_cta), dim3(sh.threads), sh.smem, s, a, b, c, d, p);
}

cudaError_t launch_attn(const void *q, const void *Khot, const void *Vhot, const void *Kst, const void *Vst,
                        const int32_t *union_slot, const uint8_t *union_qmask, const int32_t *union_cnt,
                        const int32_t *miss_count, float softmax_scale, float *out, const AttnPlan &plan,
                        const AttnScratch &scr, bool plan_ready, const void *kh_dev, const void *vh_dev,
                        int32_t *status, int B, int n_q, int Hq, int Hkv, int cs, int umax, int64_t hot_slots,
                        int64_t max_misses, cudaStream_t s, const void *k_tail, const void *v_tail,
                        unsigned long long *trace) {
  const int units = B * Hkv;
  if (units == 0) return cudaSuccess;
  const int G = Hq / Hkv, NQ = n_q * G;
  const AttnShape sh = attn_shape(NQ);

  CUtensorMap tkh, tvh, tks, tvs;
  const bool has_hot = hot_slots > 0 && Khot && Vhot;
  const bool has_st = max_misses > 0 && Kst && Vst;
  // a map must always be valid; unused ones point at a small dummy pool
  if (!(has_hot ? make_pool_map(&tkh, Khot, hot_slots * cs, cs) : make_pool_map(&tkh, scr.dummy_pool, cs, cs)))
    return cudaErrorInvalidValue;
  if (!(has_hot ? make_pool_map(&tvh, Vhot, hot_slots * cs, cs) : make_pool_map(&tvh, scr.dummy_pool, cs, cs)))
    return cudaErrorInvalidValue;
  if (!(has_st ? make_pool_map(&tks, Kst, max_misses * cs, cs) : make_pool_map(&tks, scr.dummy_pool, cs, cs)))
    return cudaErrorInvalidValue;
  if (!(has_st ? make_pool_map(&tvs, Vst, max_misses * cs, cs) : make_pool_map(&tvs, scr.dummy_pool, cs, cs)))
    return cudaErrorInvalidValue;

  cudaError_t e = cudaSuccess;
  const bool tail = k_tail && v_tail;
  const uint16_t *kt = tail ? static_cast<const uint16_t *>(k_tail) : nullptr;
  const uint16_t *vt = tail ? static_cast<const uint16_t *>(v_tail) : nullptr;
  const float scale_log2 = softmax_scale * 1.4426950408889634f;
  if (!plan_ready) {
    const AttnPlanOut po = {scr.chunk_off, scr.flat};
    e = launch_k(k_attn_plan, dim3(units), dim3(kPlanThreads), 0, s, union_cnt, union_slot, union_qmask, miss_count,
                 po, out, units, umax, n_q, Hq, Hkv, has_hot ? hot_slots : 0, has_st ? max_misses : 0, cs, status,
                 static_cast<const uint16_t *>(q), kt, vt, scale_log2);
    if (e != cudaSuccess) return e;
  }

  AttnParams p;
  p.q = static_cast<const uint16_t *>(q);
  p.chunk_off = scr.chunk_off;
  p.flat = scr.flat;
  const bool fused = kh_dev && vh_dev && has_st;
  p.kh = fused ? static_cast<const uint4 *>(kh_dev) : nullptr;
  p.vh = fused ? static_cast<const uint4 *>(vh_dev) : nullptr;
  p.kst = fused ? static_cast<uint4 *>(const_cast<void *>(Kst)) : nullptr;
  p.vst = fused ? static_cast<uint4 *>(const_cast<void *>(Vst)) : nullptr;
  p.out = out;
  p.part_o = scr.part_o;
  p.part_ml = scr.part_ml;
  p.status = status;
  p.arrive = scr.chunk_off + units + 1;   // the planner zeroed these counters
  p.k_tail = kt;
  p.v_tail = vt;
  p.trace = trace;
  p.n_q = n_q; p.Hq = Hq; p.Hkv = Hkv; p.G = G; p.NQ = NQ; p.cs = cs; p.umax = umax; p.units = units;
  p.scale_log2 = scale_log2;

  // up to 16 query vectors per KV head: mma.sync consumers, two CTAs per SM;
  // more: tcgen05 with the accumulators in tensor memory, one CTA per SM
  if (sh.mt == 1) return launch_attn_t<1, 4>(plan.n_cta, sh, tkh, tvh, tks, tvs, p, s);
  if (sh.mt > 4) return cudaErrorInvalidValue;
  CUtensorMap tq;
  if (!make_q_map(&tq, q, B, n_q, Hq, G)) return cudaErrorInvalidValue;
  return launch_attn_tc(plan.n_cta, tkh, tvh, tks, tvs, tq, p, s);
}

}  // namespace dd
