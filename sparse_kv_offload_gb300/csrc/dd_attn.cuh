// Shared device code of the two sparse attention kernels (dd_attn.cu with
// mma.sync consumers, dd_attn_tc.cu with tcgen05 consumers): the tile ring's
// layout and stage records, the kernel parameters, the producer warps (tile
// copies by TMA, the fused gather's copier, the stream-K finisher) and the
// stream-K fix-up.  The work split and the protocols are described at the top
// of dd_attn.cu.
#ifndef DD_ATTN_CUH_
#define DD_ATTN_CUH_

#include "dd_tc.cuh"

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

// stage flags: first / last stage of a run, last stage of the slice, every chunk slot loaded
enum : int32_t { kFirst = 1, kLast = 2, kEnd = 4, kFull = 8 };

// 16-byte aligned: the mbarriers that follow the per-stage records in shared
// memory need 8-byte alignment whatever the number of chunks per stage
struct alignas(16) StageMeta {
  int32_t unit, nch, flags, uoff, ucnt, pad;   // uoff/ucnt: the unit's range in the concatenated unions
  uint8_t qm[kMaxChunksPerStage];
  uint64_t rows_of[kMaxNq];   // bit t: row t of the stage was loaded and picked by query j
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
// 2^x by the PTX ex2.approx instruction (results below 2^-126 flushed to 0;
// 2^-inf = 0); the attention tests hold it to the oracle's tolerance
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// The producer warps of a CTA (pw = 0: issuing warp; pw = 1: the copier of
// the fused gather, or the finisher when the gather is not fused).  The tile
// ring has kStages stages of kStageBytes, each run's query vectors go to a
// q_bytes slot per stage (kQStride bytes per vector), and the finisher waits
// for n_pub hand-offs of the consumers' partial.  With a query tensor map
// (tm_q: q viewed as [B][n_q][Hq][128] bf16, boxes of 64 x G x n_q), a run's
// query vectors come instead by two TMA boxes straight into the 128B-swizzled
// query tile of the run's parity at qsm (2 x kHalfBytes each, rows j*G + h);
// before the tile of run r >= 2 is overwritten, the issuing warp waits on
// q_free[r & 1], which the MMA issuer arrives on (tcgen05.commit) when run
// r - 1 begins, i.e. once every MMA that read run r - 2's queries is done.
// With n_issue > 1 issuing
// warps, each walks the whole slice and issues the stages s with
// s % n_issue == issue_idx: a stage costs its issuing warp a few thousand
// cycles (the record, the mbarrier and one TMA instruction per 2 KiB box),
// which one warp cannot hide behind the stages of a single CTA per SM.  The
// fused gather keeps one issuing warp (it meets the misses in slice order).
template <int kStages>
__device__ __forceinline__ void attn_producer_warp(const AttnParams &p, const CUtensorMap *tm_khot,
                                                   const CUtensorMap *tm_vhot, const CUtensorMap *tm_kst,
                                                   const CUtensorMap *tm_vst, int lo, int hi, int per, int pw,
                                                   uint8_t *stages, uint8_t *qsm, int q_bytes, StageMeta *meta,
                                                   uint32_t full0, uint32_t empty0, int *s_ready, int *s_pub,
                                                   int n_pub, int issue_idx = 0, int n_issue = 1,
                                                   const CUtensorMap *tm_q = nullptr, uint32_t qfree0 = 0) {
  const int lane = threadIdx.x & 31;
  const bool fused = p.kh != nullptr;
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
          asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(n) : "r"(smem_u32(s_pub)) : "memory");
          if (n >= n_pub) break;
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
              asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_u32(s_ready)), "r"(done + complete)
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
  if (p.trace && lane == 0 && issue_idx == 0) trace_start(p.trace);   // before this CTA's first copy
  int missed = 0;   // fused gather: missing chunks met so far, in slice order
  int s = 0, u = u0, x = lo;
  int run = 0;   // runs begun before this stage
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
    if (s % n_issue != issue_idx) {   // another issuing warp's stage
      run += first;
      first = false;
      ++s;
    } else {
        int32_t rows[kMaxChunksPerStage];   // the stage's chunks, for its record (lane 0)
        uint32_t qms[kMaxChunksPerStage];
#pragma unroll
        for (int i = 0; i < kMaxChunksPerStage; ++i) {
          rows[i] = __shfl_sync(0xffffffffu, cur.x, (x - x0 + i) & 31);
          qms[i] = (uint32_t)__shfl_sync(0xffffffffu, cur.y, (x - x0 + i) & 31);
        }
        const int buf = s % kStages;
        const uint32_t bar = full0 + 8 * buf;
        uint32_t bytes = 0;   // the stage's copies (lane 0)
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
            bytes = first ? (uint32_t)p.NQ * 256u : 0u;
            bool full = true;
#pragma unroll
            for (int i = 0; i < kMaxChunksPerStage; ++i) {
              const uint8_t q8 = (i < nch && rows[i] != -1) ? (uint8_t)qms[i] : 0;
              m.qm[i] = q8;
              if (q8) bytes += 4 * box_bytes;
              if (i * p.cs < kStageRows && !q8) full = false;
            }
            if (full) m.flags |= kFull;
          }
        }
        alive = __shfl_sync(0xffffffffu, alive, 0);
        if (!alive) break;
        if (lane < kMaxNq) {
          // the stage's rows each query sees (lane j: query j)
          uint64_t rm = 0;
#pragma unroll
          for (int i = 0; i < kMaxChunksPerStage; ++i)
            if (i < nch && rows[i] != -1 && ((qms[i] >> lane) & 1u))
              rm |= (p.cs == 64 ? ~0ull : ((1ull << p.cs) - 1ull)) << (i * p.cs);
          meta[buf].rows_of[lane] = rm;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(bar, bytes);   // the record is written; no copy has been issued yet
        // the copies themselves, spread over the lanes: the run's query vectors,
        // and lane i the four boxes of the stage's chunk i
        if (first && tm_q != nullptr) {
          if (lane == 0) {
            if (run >= 2 && !mbar_wait(qfree0 + 8 * (run & 1), ((run >> 1) - 1) & 1, p.status)) alive = false;
            if (alive) {
              const uint32_t qdst = smem_u32(qsm) + (uint32_t)(run & 1) * 2u * kHalfBytes;
              tma_load_4d(qdst, tm_q, 0, g * p.G, 0, b, bar);
              tma_load_4d(qdst + kHalfBytes, tm_q, 64, g * p.G, 0, b, bar);
            }
          }
          alive = __shfl_sync(0xffffffffu, alive, 0);
          if (!alive) break;
        } else if (first) {
          const uint32_t qdst = smem_u32(qsm + buf * q_bytes);
          for (int qv = lane; qv < p.NQ; qv += 32) {
            const int j = qv / p.G, h = g * p.G + (qv - j * p.G);
            bulk_load(qdst + qv * kQStride, p.q + ((int64_t)(b * p.n_q + j) * p.Hq + h) * 128, 256u, bar);
          }
        }
        const int my_row = __shfl_sync(0xffffffffu, cur.x, (x - x0 + lane) & 31);
        const uint32_t my_qm = (uint32_t)__shfl_sync(0xffffffffu, cur.y, (x - x0 + lane) & 31);
        const int my_host = __shfl_sync(0xffffffffu, cur.z, (x - x0 + lane) & 31);
        const bool mine = lane < kMaxChunksPerStage && lane < nch && my_row != -1 && my_qm != 0u;
        // fused gather: a missing chunk is staged by the copier warp, in slice
        // order; its lane waits (bounded) until the copier has passed it
        const unsigned miss = __ballot_sync(0xffffffffu, mine && fused && my_row < -1 && my_host >= 0);
        bool ok = true;
        if ((miss >> lane) & 1u) {
          const int ord = missed + __popc(miss & ((1u << lane) - 1u));
          const uint64_t t0 = globaltimer_ns();
          for (uint32_t it = 0;; ++it) {
            int ready;
            asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(ready) : "r"(smem_u32(s_ready)) : "memory");
            if (ready > ord) break;
            if ((it & 63u) == 63u && globaltimer_ns() - t0 > 2000000000ull) {
              set_status(p.status, DD_ERR_TIMEOUT);
              ok = false;
              break;
            }
          }
          if (ok) asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        missed += __popc(miss);
        if (mine && ok) {
          const uint32_t sbase = smem_u32(stages + buf * kStageBytes);
          const bool hot = my_row >= 0;
          const CUtensorMap *mk = hot ? tm_khot : tm_kst;
          const CUtensorMap *mv = hot ? tm_vhot : tm_vst;
          const int y = hot ? my_row : -2 - my_row;
          const uint32_t roff = (uint32_t)(lane * p.cs * 128);
          tma_load_2d(sbase + 0 * kHalfBytes + roff, mk, 0, y, bar);
          tma_load_2d(sbase + 1 * kHalfBytes + roff, mk, 64, y, bar);
          tma_load_2d(sbase + 2 * kHalfBytes + roff, mv, 0, y, bar);
          tma_load_2d(sbase + 3 * kHalfBytes + roff, mv, 64, y, bar);
        }
        alive = __all_sync(0xffffffffu, ok);
        if (!alive) break;
        run += first;
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

// tcgen05 attention (dd_attn_tc.cu) for more than 16 query vectors per KV
// head: one persistent CTA per SM of attn_tc_threads() threads.
cudaError_t launch_attn_tc(int n_cta, const CUtensorMap &khot, const CUtensorMap &vhot, const CUtensorMap &kst,
                           const CUtensorMap &vst, const CUtensorMap &q, const AttnParams &p, cudaStream_t s);
int attn_tc_threads();

}  // namespace dd

#endif  // DD_ATTN_CUH_
