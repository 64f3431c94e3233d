// Split-K GQA decode attention over the deduplicated union of the queries'
// selected chunks.
//
// DualDecoder §5.2: the output token and the speculative token attend in one
// pass instead of two.  Adaptive DHiSparse Fig. 3 / OasisKV Methodology: the
// normal and draft queries share the HBM working set, but query j only sees
// the chunks it picked.  Here one work item is a segment of the union of one
// (request, KV head): every union row is streamed from HBM once and serves
// all NQ = n_q*G query vectors of that KV head; rows of a chunk a query did
// not select are masked for that query (the chunk's query mask).
//
// Data movement: a producer warp stages 128-row tiles of K and V into shared
// memory with 2-D TMA loads (cp.async.bulk.tensor, 128-byte swizzle, one box
// per chunk and per 64-column half) completing on mbarriers; kStages tiles
// are in flight.  Math: consumer warps own 16 query vectors (one m16 tile)
// and 16-row slices of the tile; S = Q.K^T and O += P.V run on the tensor
// cores (mma.sync m16n8k16 bf16, fp32 accumulate) with an online softmax in
// fp32; P is split into bf16 hi + lo parts so the PV product keeps ~16
// significant bits.  Work is HBM-bound: the MMAs only keep the arithmetic
// below the memory time.  Partial (max, sum, acc) per segment go to a
// workspace and a combine kernel merges the segments.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "dd_common.cuh"

namespace dd {

constexpr int kStageRows = 128;
constexpr int kHalfBytes = kStageRows * 128;          // 128 rows x 64 bf16
constexpr int kStageBytes = 4 * kHalfBytes;           // K lo, K hi, V lo, V hi
// Tiles in flight: three, except for four m-tiles where the merge buffer
// leaves room for two within the 227 KiB of shared memory.
__host__ __device__ constexpr int stages_for(int mt) { return mt >= 4 ? 2 : 3; }
constexpr int kMergeStride = 136;                     // padded fp32 row of the merge buffer
constexpr int kMaxChunksPerStage = kStageRows / 16;   // cs >= 16

struct AttnParams {
  const uint32_t *q;          // bf16 pairs [B,n_q,Hq,64]
  const int32_t *union_slot;
  const uint8_t *union_qmask;
  const int32_t *union_cnt;
  const int32_t *miss_count;
  float *part_o;              // [units, max_seg, NQ, 128]
  float *part_ml;             // [units, max_seg, NQ, 2]
  int32_t *status;
  int n_q, Hq, Hkv, G, NQ, cs, umax, seg_chunks, max_seg;
  int has_hot;
  int64_t hot_slots, max_misses;
  float scale_log2;           // softmax scale * log2(e)
};

// ----------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: gives up after ~2 s, records DD_ERR_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && globaltimer_ns() - t0 > 2000000000ull) {
      set_status(status, DD_ERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

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

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) { return pack_bf2(lo, hi); }

// ----------------------------------------------------------------- the kernel
template <int MT, int WPM>
__global__ void __launch_bounds__((MT * WPM + 1) * 32, 1)
    k_attn(const __grid_constant__ CUtensorMap tm_khot, const __grid_constant__ CUtensorMap tm_vhot,
           const __grid_constant__ CUtensorMap tm_kst, const __grid_constant__ CUtensorMap tm_vst,
           const AttnParams p) {
  constexpr int kConsumers = MT * WPM;
  constexpr int kStages = stages_for(MT);
  constexpr int kRowsPerWarp = kStageRows / WPM;      // 16, 32 or 64
  constexpr int kGroups = kRowsPerWarp / 16;

  const int unit = blockIdx.x;
  const int seg = blockIdx.y;
  const int U = p.union_cnt[unit];
  const int seg_begin = seg * p.seg_chunks;
  if (seg_begin >= U) return;
  if (load_status(p.status) != 0) return;
  const int nch_seg = min(p.seg_chunks, U - seg_begin);
  const int chunks_per_stage = kStageRows / p.cs;
  const int n_stages = (nch_seg + chunks_per_stage - 1) / chunks_per_stage;

  extern __shared__ uint8_t smem_raw[];
  // the 128-byte swizzle pattern is anchored at 1024-byte shared-memory boundaries
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *stages = smem;
  float *merge = reinterpret_cast<float *>(smem + kStages * kStageBytes);               // [MT][16][136]
  float *wml = merge + MT * 16 * kMergeStride;                                           // [MT][WPM][16][2]
  uint8_t *meta = reinterpret_cast<uint8_t *>(wml + MT * WPM * 16 * 2);                  // [kStages][8]
  uint64_t *bars = reinterpret_cast<uint64_t *>(meta + kStages * kMaxChunksPerStage);    // full[kStages], empty[kStages]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumers);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int b = unit / p.Hkv, gkv = unit - b * p.Hkv;
  const int64_t ubase = (int64_t)unit * p.umax + seg_begin;

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int64_t m_valid = min((int64_t)*p.miss_count, p.max_misses);
      const uint32_t box_bytes = (uint32_t)p.cs * 128u;
      for (int s = 0; s < n_stages; ++s) {
        const int buf = s % kStages;
        if (s >= kStages && !mbar_wait(empty0 + 8 * buf, ((s / kStages) - 1) & 1, p.status)) break;
        const int c0 = s * chunks_per_stage;
        const int nch = min(chunks_per_stage, nch_seg - c0);
        uint32_t bytes = 0;
        for (int i = 0; i < kMaxChunksPerStage; ++i) {
          uint8_t qm = 0;
          if (i < nch) {
            const int32_t slot = p.union_slot[ubase + c0 + i];
            qm = p.union_qmask[ubase + c0 + i];
            const bool hot_ok = slot >= 0 && p.has_hot && slot < p.hot_slots;
            const bool st_ok = slot < 0 && (-(int64_t)slot - 1) < m_valid;
            if (!hot_ok && !st_ok) {
              set_status(p.status, DD_ERR_DEVICE_CHECK);
              qm = 0;
            }
            if (qm) bytes += 4 * box_bytes;
          }
          meta[buf * kMaxChunksPerStage + i] = qm;
        }
        mbar_arrive_expect_tx(full0 + 8 * buf, bytes);
        const uint32_t sbase = smem_u32(stages + buf * kStageBytes);
        for (int i = 0; i < nch; ++i) {
          if (!meta[buf * kMaxChunksPerStage + i]) continue;
          const int32_t slot = p.union_slot[ubase + c0 + i];
          const CUtensorMap *mk = slot >= 0 ? &tm_khot : &tm_kst;
          const CUtensorMap *mv = slot >= 0 ? &tm_vhot : &tm_vst;
          const int y = (int)((slot >= 0 ? (int64_t)slot : (-(int64_t)slot - 1)) * p.cs);
          const uint32_t roff = (uint32_t)(i * p.cs * 128);
          const uint32_t bar = full0 + 8 * buf;
          tma_load_2d(sbase + 0 * kHalfBytes + roff, mk, 0, y, bar);
          tma_load_2d(sbase + 1 * kHalfBytes + roff, mk, 64, y, bar);
          tma_load_2d(sbase + 2 * kHalfBytes + roff, mv, 0, y, bar);
          tma_load_2d(sbase + 3 * kHalfBytes + roff, mv, 64, y, bar);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int mt = warp / WPM, wq = warp - mt * WPM;
    const int gr = lane >> 2, tq = lane & 3;
    const int qv0 = mt * 16 + gr, qv1 = qv0 + 8;
    const int j0 = qv0 < p.NQ ? qv0 / p.G : 31;
    const int j1 = qv1 < p.NQ ? qv1 / p.G : 31;

    // Q A-fragments for the 8 k-steps over d
    uint32_t qa[8][4];
    {
      const uint32_t *q0 = qv0 < p.NQ
          ? p.q + ((int64_t)(b * p.n_q + j0) * p.Hq + gkv * p.G + (qv0 % p.G)) * 64 : nullptr;
      const uint32_t *q1 = qv1 < p.NQ
          ? p.q + ((int64_t)(b * p.n_q + j1) * p.Hq + gkv * p.G + (qv1 % p.G)) * 64 : nullptr;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa[ks][0] = q0 ? q0[ks * 8 + tq] : 0u;
        qa[ks][1] = q1 ? q1[ks * 8 + tq] : 0u;
        qa[ks][2] = q0 ? q0[ks * 8 + 4 + tq] : 0u;
        qa[ks][3] = q1 ? q1[ks * 8 + 4 + tq] : 0u;
      }
    }

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float sl2 = p.scale_log2;

    for (int s = 0; s < n_stages; ++s) {
      const int buf = s % kStages;
      if (!mbar_wait(full0 + 8 * buf, (s / kStages) & 1, p.status)) break;
      const uint32_t kbase = smem_u32(stages + buf * kStageBytes);
      const uint32_t vbase = kbase + 2 * kHalfBytes;
#pragma unroll
      for (int grp = 0; grp < kGroups; ++grp) {
        const int row0 = wq * kRowsPerWarp + grp * 16;
        const uint32_t qm = meta[buf * kMaxChunksPerStage + row0 / p.cs];
        if (qm == 0) continue;
        const bool ok0 = (qm >> j0) & 1u, ok1 = (qm >> j1) & 1u;

        // S = Q K^T for 16 rows: two n8 tiles
        float sc[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
        {
          const int mi = lane >> 3, r = lane & 7;
          const int krow = row0 + (mi >> 1) * 8 + r;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + swz(krow, ks * 2 + (mi & 1)), b0, b1, b2, b3);
            mma_bf16(sc[0], qa[ks], b0, b1);
            mma_bf16(sc[1], qa[ks], b2, b3);
          }
        }
        // scale to log2 units, mask, online softmax (rows gr and gr+8)
        float x[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          x[n][0] = ok0 ? sc[n][0] * sl2 : -INFINITY;
          x[n][1] = ok0 ? sc[n][1] * sl2 : -INFINITY;
          x[n][2] = ok1 ? sc[n][2] * sl2 : -INFINITY;
          x[n][3] = ok1 ? sc[n][3] * sl2 : -INFINITY;
        }
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float base0 = mn0 == -INFINITY ? 0.f : mn0;
        const float base1 = mn1 == -INFINITY ? 0.f : mn1;
        const float a0 = exp2f(m0 - base0), a1 = exp2f(m1 - base1);
        m0 = mn0;
        m1 = mn1;
        float pr[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          pr[n][0] = exp2f(x[n][0] - base0);
          pr[n][1] = exp2f(x[n][1] - base0);
          pr[n][2] = exp2f(x[n][2] - base1);
          pr[n][3] = exp2f(x[n][3] - base1);
        }
        l0 = l0 * a0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
        l1 = l1 * a1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          o[i][0] *= a0;
          o[i][1] *= a0;
          o[i][2] *= a1;
          o[i][3] *= a1;
        }
        // P as the A operand (k = the 16 rows), split into bf16 hi and lo
        uint32_t ph[4], pl[4];
        {
          const float v[4][2] = {{pr[0][0], pr[0][1]}, {pr[0][2], pr[0][3]}, {pr[1][0], pr[1][1]}, {pr[1][2], pr[1][3]}};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t h = pack_bf16x2_rn(v[i][0], v[i][1]);
            ph[i] = h;
            pl[i] = pack_bf16x2_rn(v[i][0] - bf_lo(h), v[i][1] - bf_hi(h));
          }
        }
        // O += P V: V fragments by transposed ldmatrix, two 8-column tiles per load
        {
          const int mi = lane >> 3, r = lane & 7;
          const int vrow = row0 + (mi & 1) * 8 + r;
#pragma unroll
          for (int dp = 0; dp < 8; ++dp) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(vbase + swz(vrow, dp * 2 + (mi >> 1)), v0, v1, v2, v3);
            mma_bf16(o[2 * dp], ph, v0, v1);
            mma_bf16(o[2 * dp], pl, v0, v1);
            mma_bf16(o[2 * dp + 1], ph, v2, v3);
            mma_bf16(o[2 * dp + 1], pl, v2, v3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * buf);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    if (tq == 0) {
      float *w = wml + ((mt * WPM + wq) * 16) * 2;
      w[gr * 2 + 0] = m0;
      w[gr * 2 + 1] = l0;
      w[(gr + 8) * 2 + 0] = m1;
      w[(gr + 8) * 2 + 1] = l1;
    }
    // stash this warp's state in registers for the merge below
    // (o, m0, m1 stay live across the barriers)
    __syncthreads();
    // common max over the WPM warps of this m-tile, per row
    float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
    for (int w2 = 0; w2 < WPM; ++w2) {
      const float *w = wml + ((mt * WPM + w2) * 16) * 2;
      M0 = fmaxf(M0, w[gr * 2]);
      M1 = fmaxf(M1, w[(gr + 8) * 2]);
    }
    for (int w2 = 0; w2 < WPM; ++w2) {
      const float *w = wml + ((mt * WPM + w2) * 16) * 2;
      if (M0 != -INFINITY) L0 += w[gr * 2 + 1] * exp2f(w[gr * 2] - M0);
      if (M1 != -INFINITY) L1 += w[(gr + 8) * 2 + 1] * exp2f(w[(gr + 8) * 2] - M1);
    }
    const float f0 = M0 == -INFINITY ? 0.f : exp2f(m0 - M0);
    const float f1 = M1 == -INFINITY ? 0.f : exp2f(m1 - M1);
    float *acc = merge + mt * 16 * kMergeStride;
    for (int w2 = 0; w2 < WPM; ++w2) {
      if (wq == w2) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = i * 8 + 2 * tq;
          float *r0p = acc + gr * kMergeStride + col;
          float *r1p = acc + (gr + 8) * kMergeStride + col;
          if (w2 == 0) {
            r0p[0] = o[i][0] * f0; r0p[1] = o[i][1] * f0;
            r1p[0] = o[i][2] * f1; r1p[1] = o[i][3] * f1;
          } else {
            r0p[0] += o[i][0] * f0; r0p[1] += o[i][1] * f0;
            r1p[0] += o[i][2] * f1; r1p[1] += o[i][3] * f1;
          }
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32));
    }
    // write this m-tile's partial: rows of valid query vectors
    const int64_t pbase = ((int64_t)unit * p.max_seg + seg) * p.NQ;
    for (int e = wq * 32 + lane; e < 16 * 128; e += WPM * 32) {
      const int r = e >> 7, col = e & 127;
      const int qv = mt * 16 + r;
      if (qv < p.NQ) p.part_o[(pbase + qv) * 128 + col] = acc[r * kMergeStride + col];
    }
    if (wq == 0 && tq == 0) {
      if (qv0 < p.NQ) { p.part_ml[(pbase + qv0) * 2] = M0; p.part_ml[(pbase + qv0) * 2 + 1] = L0; }
      if (qv1 < p.NQ) { p.part_ml[(pbase + qv1) * 2] = M1; p.part_ml[(pbase + qv1) * 2 + 1] = L1; }
    }
    return;
  }
  // producer warp joins the consumers' first barrier
  __syncthreads();
}

// --------------------------------------------------------------- combine
__global__ void __launch_bounds__(128) k_attn_combine(const float *__restrict__ part_o,
                                                      const float *__restrict__ part_ml,
                                                      const int32_t *__restrict__ union_cnt, float *__restrict__ out,
                                                      const int32_t *status, int n_q, int Hq, int Hkv, int G, int NQ,
                                                      int seg_chunks, int max_seg) {
  if (load_status(status) != 0) return;
  const int unit = blockIdx.x, qv = blockIdx.y, col = threadIdx.x;
  const int U = union_cnt[unit];
  const int nseg = min(max_seg, (U + seg_chunks - 1) / seg_chunks);
  const int64_t pbase = (int64_t)unit * max_seg * NQ + qv;
  float M = -INFINITY;
  for (int s = 0; s < nseg; ++s) M = fmaxf(M, part_ml[(pbase + (int64_t)s * NQ) * 2]);
  float L = 0.f, acc = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < nseg; ++s) {
      const int64_t i = pbase + (int64_t)s * NQ;
      const float ms = part_ml[i * 2];
      if (ms == -INFINITY) continue;
      const float w = exp2f(ms - M);
      L += w * part_ml[i * 2 + 1];
      acc += w * part_o[i * 128 + col];
    }
  }
  const int b = unit / Hkv, g = unit - b * Hkv;
  const int j = qv / G, h = g * G + (qv - j * G);
  out[((int64_t)(b * n_q + j) * Hq + h) * 128 + col] = L > 0.f ? acc / L : 0.f;
}

// --------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// A [rows, 128] bf16 pool viewed as 2-D, boxes of cs rows x 64 columns.
static bool make_pool_map(CUtensorMap *map, const void *base, int64_t rows, int cs) {
  auto enc = tensor_map_encoder();
  if (!enc || base == nullptr || rows <= 0) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, (cuuint32_t)cs};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct AttnShape {
  int mt, wpm, threads;
  size_t smem;
};

AttnShape attn_shape(int NQ) {
  AttnShape s;
  s.mt = (NQ + 15) / 16;
  s.wpm = s.mt == 1 ? 8 : (s.mt == 4 ? 2 : 4);
  s.threads = (s.mt * s.wpm + 1) * 32;
  const int ns = stages_for(s.mt);
  s.smem = 1024 + (size_t)ns * kStageBytes + (size_t)s.mt * 16 * kMergeStride * 4 +
           (size_t)s.mt * s.wpm * 16 * 2 * 4 + ns * kMaxChunksPerStage + 2 * ns * 8 + 16;
  return s;
}

int attn_seg_chunks(int NQ, int cs) {
  const int mt = (NQ + 15) / 16;
  return (512 * mt) / cs;
}

template <int MT, int WPM>
static cudaError_t launch_attn_t(dim3 grid, const AttnShape &sh, const CUtensorMap &a, const CUtensorMap &b,
                                 const CUtensorMap &c, const CUtensorMap &d, const AttnParams &p, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(k_attn<MT, WPM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sh.smem);
  if (e != cudaSuccess) return e;
  k_attn<MT, WPM><<<grid, sh.threads, sh.smem, s>>>(a, b, c, d, p);
  return cudaGetLastError();
}

cudaError_t launch_attn(const void *q, const void *Khot, const void *Vhot, const void *Kst, const void *Vst,
                        const int32_t *union_slot, const uint8_t *union_qmask, const int32_t *union_cnt,
                        const int32_t *miss_count, float softmax_scale, float *out, float *part_o, float *part_ml,
                        int32_t *status, int B, int n_q, int Hq, int Hkv, int cs, int umax, int64_t hot_slots,
                        int64_t max_misses, const void *dummy_pool, cudaStream_t s) {
  const int units = B * Hkv;
  if (units == 0) return cudaSuccess;
  const int G = Hq / Hkv, NQ = n_q * G;
  const AttnShape sh = attn_shape(NQ);
  const int seg_chunks = attn_seg_chunks(NQ, cs);
  const int max_seg = (umax + seg_chunks - 1) / seg_chunks;

  CUtensorMap tkh, tvh, tks, tvs;
  const bool has_hot = hot_slots > 0 && Khot && Vhot;
  const bool has_st = max_misses > 0 && Kst && Vst;
  // a map must always be valid; unused ones point at a small dummy pool
  if (!(has_hot ? make_pool_map(&tkh, Khot, hot_slots * cs, cs) : make_pool_map(&tkh, dummy_pool, cs, cs)))
    return cudaErrorInvalidValue;
  if (!(has_hot ? make_pool_map(&tvh, Vhot, hot_slots * cs, cs) : make_pool_map(&tvh, dummy_pool, cs, cs)))
    return cudaErrorInvalidValue;
  if (!(has_st ? make_pool_map(&tks, Kst, max_misses * cs, cs) : make_pool_map(&tks, dummy_pool, cs, cs)))
    return cudaErrorInvalidValue;
  if (!(has_st ? make_pool_map(&tvs, Vst, max_misses * cs, cs) : make_pool_map(&tvs, dummy_pool, cs, cs)))
    return cudaErrorInvalidValue;

  AttnParams p;
  p.q = static_cast<const uint32_t *>(q);
  p.union_slot = union_slot;
  p.union_qmask = union_qmask;
  p.union_cnt = union_cnt;
  p.miss_count = miss_count;
  p.part_o = part_o;
  p.part_ml = part_ml;
  p.status = status;
  p.n_q = n_q; p.Hq = Hq; p.Hkv = Hkv; p.G = G; p.NQ = NQ; p.cs = cs; p.umax = umax;
  p.seg_chunks = seg_chunks; p.max_seg = max_seg;
  p.has_hot = has_hot ? 1 : 0;
  p.hot_slots = has_hot ? hot_slots : 0;
  p.max_misses = has_st ? max_misses : 0;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;

  dim3 grid(units, max_seg);
  cudaError_t e;
  switch (sh.mt) {
    case 1: e = launch_attn_t<1, 8>(grid, sh, tkh, tvh, tks, tvs, p, s); break;
    case 2: e = launch_attn_t<2, 4>(grid, sh, tkh, tvh, tks, tvs, p, s); break;
    case 3: e = launch_attn_t<3, 4>(grid, sh, tkh, tvh, tks, tvs, p, s); break;
    case 4: e = launch_attn_t<4, 2>(grid, sh, tkh, tvh, tks, tvs, p, s); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  k_attn_combine<<<dim3(units, NQ), 128, 0, s>>>(part_o, part_ml, union_cnt, out, status, n_q, Hq, Hkv, G, NQ,
                                                 seg_chunks, max_seg);
  return cudaGetLastError();
}

}  // namespace dd
