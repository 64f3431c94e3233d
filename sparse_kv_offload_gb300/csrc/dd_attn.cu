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

#include "dd_common.cuh"

namespace dd {

// Persistent CTAs per SM: two for one m-tile (16 query vectors), one for
// more, whose consumers need the registers of a whole SM (two CTAs would cap
// them at 128 per thread and spill).
__host__ __device__ constexpr int ctas_per_sm(int mt) { return mt == 1 ? 2 : 1; }
constexpr int kStageRows = 64;
constexpr int kHalfBytes = kStageRows * 128;          // 64 rows x 64 bf16
constexpr int kStageBytes = 4 * kHalfBytes;           // K lo, K hi, V lo, V hi
constexpr int kMaxChunksPerStage = kStageRows / 16;   // cs >= 16
constexpr int kQStride = 272;                         // bytes per staged query vector (256 + pad)
constexpr int kCopyBatch = 8;                         // fused gather: 16-byte host loads in flight per copier lane
constexpr int kMergeFloats = 68;                       // a lane's run state: 64 accumulator elements, m0, m1, l0, l1

// Tiles in flight per CTA: three for one m-tile (two CTAs share an SM's
// 228 KiB), four for more (one CTA per SM, beside its staged queries).
__host__ __device__ constexpr int stages_for(int mt) { return mt == 1 ? 3 : 4; }

enum : int32_t { kFirst = 1, kLast = 2, kEnd = 4 };

// 16-byte aligned: the mbarriers that follow the per-stage records in shared
// memory need 8-byte alignment whatever the number of chunks per stage
struct alignas(16) StageMeta {
  int32_t unit, nch, flags, uoff, ucnt, pad;   // uoff/ucnt: the unit's range in the concatenated unions
  uint8_t qm[kMaxChunksPerStage];
};
static_assert(sizeof(StageMeta) % 8 == 0, "mbarriers follow the stage records");

struct AttnParams {
  const uint16_t *q;          // bf16 [B,n_q,Hq,128]
  const int32_t *chunk_off;   // [units+1] exclusive prefix of the union sizes
  const int4 *flat;           // per chunk of the concatenated unions: {pool row code, query mask, host chunk, 0}
  const uint4 *kh, *vh;       // fused gather: device view of the pinned host K/V (null: staging comes by TMA)
  uint4 *kst, *vst;           // fused gather: staging buffers the host chunks are also written to
  float *out;                 // fp32 [B,n_q,Hq,128]
  float *part_o;              // [gridDim + units, NQ, 128], slot = CTA + unit
  float *part_ml;             // [gridDim + units, NQ, 2]
  int32_t *status;
  int32_t *arrive;            // [units] CTAs that have finished a part of each unit (zeroed by the planner)
  unsigned long long *trace;  // optional [2][kTraceSlots]: per-SM earliest start, latest end (ns)
  const uint16_t *k_tail, *v_tail;   // bf16 [B,n_q,Hkv,128] the step's own new rows, or null
  int n_q, Hq, Hkv, G, NQ, cs, umax, units;
  float scale_log2;           // softmax scale * log2(e)
};

// pool row code of a chunk in the flat table: first hot-pool row as is,
// staging row r as -2 - r, -1 = not loaded

// Largest unit u with chunk_off[u] <= x (the unit whose union holds chunk x),
// found by one warp: 32 probes per round (two rounds up to 1024 units).
// Invariant: off[lo] <= x; the answer lies in [lo, lo + n).
__device__ __forceinline__ int unit_of_chunk_warp(const int32_t *off, int units, int x) {
  const int lane = threadIdx.x & 31;
  int lo = 0, n = units;
  while (n > 1) {
    const int step = (n + 31) / 32;
    const int idx = lo + lane * step;
    const bool le = lane * step < n && off[idx] <= x;
    const unsigned m = __ballot_sync(0xffffffffu, le);   // lane 0 always set
    const int l = 31 - __clz(m);
    lo += l * step;
    n = min(step, n - l * step);
  }
  return lo;
}


// ----------------------------------------------------------------- PTX helpers
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

// Stream-K arrival count: adds one with release (the CTA's published
// partials, ordered before it by a barrier, become visible with it) and
// acquire (the other CTAs' partials are visible to whoever reads them after
// this thread, through a barrier) semantics at GPU scope.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t *p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// two fp32 -> packed bf16x2 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}


// ------------------------------------------------------------ stream-K fix-up
// Run by the consumer warps of the CTA that finished the last part of `unit`
// (every other CTA whose slice covered part of it has published its partials
// before counting itself in).  Thread (query vector, 8 columns): merges the
// partials of CTAs c0..c1 in order, then, when the
// step's own rows are given, its tail rows: query j of the unit also attends
// to the new rows of tokens 0..j (DualDecoder §5.2: the tokens of a step
// follow one another along the sequence under a causal mask).
__device__ __forceinline__ void fixup_unit(const AttnParams &p, int unit, int c0, int c1, int n_threads, int ctid) {
  const int lane = threadIdx.x & 31;
  const int n_parts = c1 - c0 + 1;
  const int b = unit / p.Hkv, g = unit - b * p.Hkv;
  for (int w0 = (ctid >> 5) * 32; w0 < p.NQ * 16; w0 += n_threads) {   // warp-uniform
    const int w = w0 + lane;
    const bool act = w < p.NQ * 16;
    const int qv = act ? (w >> 4) : 0, cg = w & 15;
    const int j = qv / p.G, h = g * p.G + (qv - j * p.G);
    float M = -INFINITY, L = 0.f, acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int i0 = 0; i0 < n_parts; i0 += 4) {
      float ms[4], ls[4];
      float4 oa[4], ob[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int i = i0 + t;
        const bool ok = act && i < n_parts;
        const int64_t k = ((int64_t)c0 + i + unit) * p.NQ + qv;
        const float4 *src = reinterpret_cast<const float4 *>(p.part_o + k * 128 + cg * 8);
        ms[t] = ok ? p.part_ml[k * 2] : -INFINITY;
        ls[t] = ok ? p.part_ml[k * 2 + 1] : 0.f;
        oa[t] = ok ? src[0] : make_float4(0.f, 0.f, 0.f, 0.f);
        ob[t] = ok ? src[1] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (ms[t] == -INFINITY) continue;
        const float Mn = fmaxf(M, ms[t]);
        const float a = M == -INFINITY ? 0.f : exp2f(M - Mn), wt = exp2f(ms[t] - Mn);
        const float o8[8] = {oa[t].x, oa[t].y, oa[t].z, oa[t].w, ob[t].x, ob[t].y, ob[t].z, ob[t].w};
        L = L * a + wt * ls[t];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = acc[e] * a + wt * o8[e];
        M = Mn;
      }
    }
    if (p.k_tail) {
      float qf[8];
      unpack8(act ? *reinterpret_cast<const uint4 *>(p.q + ((int64_t)(b * p.n_q + j) * p.Hq + h) * 128 + cg * 8)
                  : make_uint4(0, 0, 0, 0),
              qf);
#pragma unroll
      for (int t = 0; t < kMaxNq; ++t) {
        const bool use = act && t <= j;
        const int64_t trow = ((int64_t)(b * p.n_q + t) * p.Hkv + g) * 128 + cg * 8;
        float x = 0.f;
        if (use) {
          float kf[8];
          unpack8(*reinterpret_cast<const uint4 *>(p.k_tail + trow), kf);
#pragma unroll
          for (int e = 0; e < 8; ++e) x = fmaf(qf[e], kf[e], x);
        }
        // the 16 lanes of this query vector hold its 128 columns
        x += __shfl_xor_sync(0xffffffffu, x, 8);
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        if (use) {
          float vf[8];
          unpack8(*reinterpret_cast<const uint4 *>(p.v_tail + trow), vf);
          const float s2 = x * p.scale_log2;
          const float Mn = fmaxf(M, s2);
          const float a = M == -INFINITY ? 0.f : exp2f(M - Mn), wt = exp2f(s2 - Mn);
          L = L * a + wt;
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] = acc[e] * a + wt * vf[e];
          M = Mn;
        }
      }
    }
    if (act) {
      float4 *dst = reinterpret_cast<float4 *>(p.out + ((int64_t)(b * p.n_q + j) * p.Hq + h) * 128 + cg * 8);
      dst[0] = make_float4(L > 0.f ? acc[0] / L : 0.f, L > 0.f ? acc[1] / L : 0.f, L > 0.f ? acc[2] / L : 0.f,
                           L > 0.f ? acc[3] / L : 0.f);
      dst[1] = make_float4(L > 0.f ? acc[4] / L : 0.f, L > 0.f ? acc[5] / L : 0.f, L > 0.f ? acc[6] / L : 0.f,
                           L > 0.f ? acc[7] / L : 0.f);
    }
  }
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
    // ------------------------------------------------------------ producers
    const bool fused = p.kh != nullptr;
    const int pw = warp - kConsumers;
    if (pw > 0) {
      if (!fused && pw == 1) {
        // finisher warp (the gather is not fused, so this warp copies
        // nothing): the stream-K count of the slice's first run when that run
        // continues a unit begun by an earlier CTA and is not the slice's last
        // run.  Only the first run can be such a run (every later one starts
        // inside the slice).  The consumers publish that run's partial and go
        // on with the next run; this warp counts the CTA in on the unit and,
        // when it arrives last, merges the unit, off the consumers' path.
        const int u = unit_of_chunk_warp(p.chunk_off, p.units, lo);
        const int off_u = p.chunk_off[u], end_u = p.chunk_off[u + 1];
        if (off_u < lo && end_u < hi) {
          const int c0 = off_u / per, c1 = (end_u - 1) / per;
          bool ok = true;
          const uint64_t t0 = globaltimer_ns();
          for (uint32_t it = 0;; ++it) {   // the partials of every m-tile, published with release
            int n;
            asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(n) : "r"(smem_u32(&s_pub)) : "memory");
            if (n >= MT) break;
            __nanosleep(64);
            if ((it & 15u) == 15u && globaltimer_ns() - t0 > 2000000000ull) {
              ok = false;
              break;
            }
          }
          if (!ok) {
            if (lane == 0) set_status(p.status, DD_ERR_TIMEOUT);
            return;
          }
          int last = 0;
          if (lane == 0) last = atom_add_acq_rel_gpu(p.arrive + u, 1) + 1 == c1 - c0 + 1;
          if (__shfl_sync(0xffffffffu, last, 0)) fixup_unit(p, u, c0, c1, 32, lane);
        }
      }
      if (fused && pw == 1) {
        // fused gather, copier warp: every missing chunk of the slice, in
        // slice order, from pinned host memory into its staging rows, as far
        // ahead of the issuing warp as the link allows.  The batch's missing
        // chunks are numbered k = 0..n-1 (lane k holds chunk k's host index
        // and staging row) and their elements walked as one sequence,
        // kCopyBatch loads per lane in flight.  Whenever chunks complete, all
        // lanes fence (GPU scope, then the generic -> async proxy fence, as
        // the issuing warp reads staging by TMA) and lane 0 publishes how
        // many of the slice's misses are in place (s_ready, release).
        const int vec = p.cs * 16;   // uint4 per chunk, K or V
        int done = 0;                // misses of the slice copied so far
        for (int xb = lo; xb < hi; xb += 32) {
          const int4 e = (xb + lane < hi) ? p.flat[xb + lane] : make_int4(-1, 0, -1, 0);
          const unsigned mm = __ballot_sync(0xffffffffu, e.x < -1 && e.y != 0 && e.z >= 0);
          const int n_miss = __popc(mm);
          if (n_miss == 0) continue;
          int my_pos = 0;   // batch position of missing chunk number `lane`
          {
            unsigned m2 = mm;
            for (int k = 0; k < lane && m2; ++k) m2 &= m2 - 1;
            my_pos = m2 ? __ffs(m2) - 1 : 0;
          }
          const int my_host = __shfl_sync(0xffffffffu, e.z, my_pos);
          const int my_row = __shfl_sync(0xffffffffu, e.x, my_pos);
          const int total_e = n_miss * 2 * vec;
          int published = 0;
#pragma unroll 1
          for (int e0 = 0; e0 < total_e; e0 += 32 * kCopyBatch) {
            uint4 v[kCopyBatch];
#pragma unroll
            for (int t = 0; t < kCopyBatch; ++t) {
              const int eu = e0 + t * 32;                       // warp-uniform
              const int k = eu / (2 * vec);
              const int host = __shfl_sync(0xffffffffu, my_host, k & 31);
              const int el = eu - k * 2 * vec + lane;           // within the chunk: K then V
              const uint4 *src = el >= vec ? p.vh + (int64_t)host * vec + (el - vec) : p.kh + (int64_t)host * vec + el;
              v[t] = eu < total_e ? ldg_nc(src) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int t = 0; t < kCopyBatch; ++t) {
              const int eu = e0 + t * 32;
              const int k = eu / (2 * vec);
              const int row = __shfl_sync(0xffffffffu, my_row, k & 31);
              if (eu >= total_e) continue;
              const int el = eu - k * 2 * vec + lane;
              const int kv = el >= vec, r = kv ? el - vec : el;
              (kv ? p.vst : p.kst)[(int64_t)(-2 - row) * 16 + r] = v[t];   // -2 - row: first staging row
            }
            // chunks whose every element precedes e0 + 32 * kCopyBatch are complete
            const int complete = min(n_miss, (e0 + 32 * kCopyBatch) / (2 * vec));
            if (complete > published) {
              __threadfence();
              asm volatile("fence.proxy.async.global;" ::: "memory");
              __syncwarp();
              if (lane == 0)
                asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_u32(&s_ready)), "r"(done + complete)
                             : "memory");
              published = complete;
            }
          }
          done += n_miss;
        }
      }
      return;
    }
    // issuing warp: streams the flat chunk table of this slice in batches of
    // 32 (the next batch already in flight) and cuts it into stages that never
    // cross a unit boundary; lane i of `bnd` holds the end of unit ubase + i
    const int chunks_per_stage = kStageRows / p.cs;
    const uint32_t box_bytes = (uint32_t)p.cs * 128u;
    const int u0 = unit_of_chunk_warp(p.chunk_off, p.units, lo);
    int ubase = u0;
    int bnd = (ubase + 1 + lane <= p.units) ? p.chunk_off[ubase + 1 + lane] : 0x7FFFFFFF;
    int ustart = p.chunk_off[u0];
    int x0 = lo;
    int4 cur = (x0 + lane < hi) ? p.flat[x0 + lane] : make_int4(-1, 0, -1, 0);
    int4 nxt = (x0 + 32 + lane < hi) ? p.flat[x0 + 32 + lane] : make_int4(-1, 0, -1, 0);
    if (p.trace && lane == 0) trace_start(p.trace);   // before this CTA's first copy
    int missed = 0;   // fused gather: missing chunks met so far, in slice order (lane 0)
    int s = 0, u = u0, x = lo;
    bool first = true, alive = true;
    while (x < hi && alive) {
      if (u - ubase >= 32) {
        ubase = u;
        bnd = (ubase + 1 + lane <= p.units) ? p.chunk_off[ubase + 1 + lane] : 0x7FFFFFFF;
      }
      const int end_u = __shfl_sync(0xffffffffu, bnd, u - ubase);
      if (x >= end_u) {   // unit u finished (or empty): next unit, new run
        ++u;
        ustart = end_u;
        first = true;
        continue;
      }
      const int stop = min(min(end_u, hi), x0 + 32);
      const int nch = min(chunks_per_stage, stop - x);
      const bool last = x + nch == min(end_u, hi);
      const bool end = x + nch == hi;
      const int b = u / p.Hkv, g = u - b * p.Hkv;
      {
          int32_t rows[kMaxChunksPerStage], hosts[kMaxChunksPerStage];
          uint32_t qms[kMaxChunksPerStage];
#pragma unroll
          for (int i = 0; i < kMaxChunksPerStage; ++i) {
            rows[i] = __shfl_sync(0xffffffffu, cur.x, (x - x0 + i) & 31);
            qms[i] = (uint32_t)__shfl_sync(0xffffffffu, cur.y, (x - x0 + i) & 31);
            hosts[i] = __shfl_sync(0xffffffffu, cur.z, (x - x0 + i) & 31);
          }
          const int buf = s % kStages;
          if (lane == 0) {
            if (s >= kStages && !mbar_wait(empty0 + 8 * buf, ((s / kStages) - 1) & 1, p.status)) {
              alive = false;
            } else {
              StageMeta &m = meta[buf];
              m.unit = u;
              m.nch = nch;
              m.flags = (first ? kFirst : 0) | (last ? kLast : 0) | (end ? kEnd : 0);
              m.uoff = ustart;
              m.ucnt = end_u - ustart;
              uint32_t bytes = first ? (uint32_t)p.NQ * 256u : 0u;
#pragma unroll
              for (int i = 0; i < kMaxChunksPerStage; ++i) {
                const uint8_t q8 = (i < nch && rows[i] != -1) ? (uint8_t)qms[i] : 0;
                m.qm[i] = q8;
                if (q8) bytes += 4 * box_bytes;
              }
              const uint32_t bar = full0 + 8 * buf;
              mbar_arrive_expect_tx(bar, bytes);
              if (first) {
                const uint32_t qdst = smem_u32(qsm + buf * kQBytes);
                for (int qv = 0; qv < p.NQ; ++qv) {
                  const int j = qv / p.G, h = g * p.G + (qv - j * p.G);
                  bulk_load(qdst + qv * kQStride, p.q + ((int64_t)(b * p.n_q + j) * p.Hq + h) * 128, 256u, bar);
                }
              }
              const uint32_t sbase = smem_u32(stages + buf * kStageBytes);
#pragma unroll
              for (int i = 0; i < kMaxChunksPerStage; ++i) {
                if (i >= nch || rows[i] == -1 || qms[i] == 0) continue;
                if (fused && rows[i] < -1 && hosts[i] >= 0) {
                  // a missing chunk: staged by the copier warp; wait until it is in place (bounded)
                  const int ord = missed++;
                  const uint64_t t0 = globaltimer_ns();
                  for (uint32_t it = 0;; ++it) {
                    int ready;
                    asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(ready) : "r"(smem_u32(&s_ready))
                                 : "memory");
                    if (ready > ord) break;
                    if ((it & 63u) == 63u && globaltimer_ns() - t0 > 2000000000ull) {
                      set_status(p.status, DD_ERR_TIMEOUT);
                      alive = false;
                      break;
                    }
                  }
                  if (!alive) break;
                  asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                const bool hot = rows[i] >= 0;
                const CUtensorMap *mk = hot ? &tm_khot : &tm_kst;
                const CUtensorMap *mv = hot ? &tm_vhot : &tm_vst;
                const int y = hot ? rows[i] : -2 - rows[i];
                const uint32_t roff = (uint32_t)(i * p.cs * 128);
                tma_load_2d(sbase + 0 * kHalfBytes + roff, mk, 0, y, bar);
                tma_load_2d(sbase + 1 * kHalfBytes + roff, mk, 64, y, bar);
                tma_load_2d(sbase + 2 * kHalfBytes + roff, mv, 0, y, bar);
                tma_load_2d(sbase + 3 * kHalfBytes + roff, mv, 64, y, bar);
              }
            }
          }
          alive = __shfl_sync(0xffffffffu, alive, 0);
          if (!alive) break;
          first = false;
          ++s;
      }
      x += nch;
      if (x == x0 + 32) {   // batch used up: the prefetched one becomes current
        x0 += 32;
        cur = nxt;
        nxt = (x0 + 32 + lane < hi) ? p.flat[x0 + 32 + lane] : make_int4(-1, 0, -1, 0);
      }
    }
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
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// A [rows, 128] bf16 pool viewed as 2-D, boxes of cs rows x 64 columns.  A
// descriptor depends on nothing but (base, rows, cs), so the last few are
// kept: a decode loop cycles through the same pools step after step.
static bool make_pool_map(CUtensorMap *map, const void *base, int64_t rows, int cs) {
  struct Entry {
    const void *base;
    int64_t rows;
    int cs;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int n = 0, next = 0;
  if (base == nullptr || rows <= 0) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
      if (cache[i].base == base && cache[i].rows == rows && cache[i].cs == cs) {
        *map = cache[i].map;
        return true;
      }
  }
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, (cuuint32_t)cs};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(mu);
  cache[next] = {base, rows, cs, *map};
  next = (next + 1) % 32;
  if (n < 32) ++n;
  return true;
}

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

  switch (sh.mt) {
    case 1: e = launch_attn_t<1, 4>(plan.n_cta, sh, tkh, tvh, tks, tvs, p, s); break;
    case 2: e = launch_attn_t<2, 2>(plan.n_cta, sh, tkh, tvh, tks, tvs, p, s); break;
    case 3: e = launch_attn_t<3, 2>(plan.n_cta, sh, tkh, tvh, tks, tvs, p, s); break;
    case 4: e = launch_attn_t<4, 1>(plan.n_cta, sh, tkh, tvh, tks, tvs, p, s); break;
    default: return cudaErrorInvalidValue;
  }
  return e;
}

}  // namespace dd
