// Sparse GQA decode attention on the fifth-generation tensor cores (tcgen05),
// for more than 16 query vectors per KV head.
//
// Same work split, tile ring, producer warps and stream-K protocol as the
// mma.sync kernel in dd_attn.cu (DualDecoder §5.2 co-batched attention over
// the deduplicated union; Adaptive DHiSparse Fig. 3: every query over its own
// selection).  What changes is the math.  With 17-64 query vectors the
// mma.sync consumers need a whole SM's registers for their accumulators, so
// only six consumer warps fit and they stall on the MMA dependency chains;
// here the accumulators live in tensor memory and one thread issues the MMAs:
//
//   S = Q K^T   tcgen05.mma, M = 64 query vectors (rows >= NQ unused), N = the
//               64 rows of a stage, K = 128; A (queries) and B (the stage's K
//               tile, as TMA left it) both K-major with the 128-byte swizzle;
//               fp32 in tensor memory, double-buffered (64 columns each).
//   softmax     warps 0-7, four threads per query vector (the M = 64 layout
//               puts row r in tensor-memory lane 32*(r/16) + r%16; warps w
//               and w + 4 share a lane quarter and take the two halves of
//               each row, and the 16x32bx2 access splits a half between lanes
//               t and t + 16 of a warp); online softmax in the log2 domain with a
//               lazy reference: the accumulator is rescaled only when a row's
//               maximum grows by more than 2^8.  P is written to shared memory
//               as bf16 hi + lo parts, both by truncation on the integer
//               pipes (the PV product keeps ~14 significant bits).
//   O += P V    tcgen05.mma, M = 64, N = 128, K = 64 rows in four K = 16 steps;
//               A = P (K-major), B = the stage's V tile read MN-major (its
//               64-column halves 8 KiB apart); fp32 accumulator in tensor
//               memory (128 columns).  Completion of each stage's PV releases
//               the stage to the producer (tcgen05.commit on its mbarrier).
//
// At the end of a run the softmax warps read O from tensor memory and write
// the outputs, or a partial for the stream-K fix-up (dd_attn.cuh).
#include "dd_attn.cuh"

namespace dd {

namespace {

// Eight softmax warps, two per tensor-memory lane quarter.  (Sixteen, four
// per quarter with half the columns each, ran the fully resident 32B-class
// layer's attention at 151 us against 121: at 640 threads a thread gets 96
// registers and the kernel spills.)
constexpr int kTcSoftmaxWarps = 8;
constexpr int kTcColGroups = kTcSoftmaxWarps / 4;                  // warps sharing a lane quarter: column groups
constexpr int kTcThreads = (kTcSoftmaxWarps + 4) * 32;             // + 2 issuing warps, copier / finisher, MMA warp
constexpr int kTcM = 64;                                           // query vectors per MMA (M)
constexpr int kTcTmemCols = 256;                                   // S: 2 x 64 columns, O: 128 columns
constexpr int kTcTileBytes = kTcM * 128;                           // a 64-row, 128-byte-row swizzled tile
constexpr float kRescaleLog2 = 8.f;                                // lazy rescale threshold (log2 units)

// 16x32bx2 tensor-memory access, 32 columns per thread: threads 0-15 of the
// warp read lanes 0-15 of its lane quarter at columns [c, c + 32), threads
// 16-31 the same lanes at columns [c + kSplit, c + kSplit + 32).
#define DD_R32(r) "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), \
    "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),      \
    "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),    \
    "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define DD_W32(r) "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), \
    "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),     \
    "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),    \
    "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])

template <int kSplit>
__device__ __forceinline__ void tmem_ld32_split(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], %33;"
      : DD_R32(r)
      : "r"(taddr), "n"(kSplit));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <int kSplit>
__device__ __forceinline__ void tmem_ld16_split(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], %17;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr), "n"(kSplit));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <int kSplit>
__device__ __forceinline__ void tmem_st32_split(uint32_t taddr, const float *v) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %1, {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};" ::"r"(taddr),
      "n"(kSplit), DD_W32(r)
      : "memory");
}
template <int kSplit>
__device__ __forceinline__ void tmem_ld8_split(uint32_t taddr, float *v) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr), "n"(kSplit));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

template <int kSplit>
__device__ __forceinline__ void tmem_st16_split(uint32_t taddr, const float *v) {
  uint32_t r[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %1, {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17};"
      ::"r"(taddr), "n"(kSplit), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
      "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// A thread's columns of S (kCols = 16 or 8) or O (32 or 16), in the 16x32bx2
// layout: threads 0-15 at [c, c + kCols), threads 16-31 at [c + kCols, c + 2 kCols).
template <int kCols>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float *v) {
  if constexpr (kCols == 32) tmem_ld32_split<32>(taddr, v);
  else if constexpr (kCols == 16) tmem_ld16_split<16>(taddr, v);
  else tmem_ld8_split<8>(taddr, v);
}
template <int kCols>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float *v) {
  if constexpr (kCols == 32) tmem_st32_split<32>(taddr, v);
  else tmem_st16_split<16>(taddr, v);
}
#undef DD_R32
#undef DD_W32

// Shared-memory plan, 1024-byte aligned parts:
//   tile ring  [kStages][32 KiB]  K lo, K hi, V lo, V hi halves of 64 rows
//   Q tiles    [2 runs][2 halves][64 rows][128 B]   the queries of runs of
//              each parity (A of S), written by TMA with the 128-byte swizzle
//   P          [2 buffers][hi, lo][64 rows][128 B]   (A of O += P V)
//   stage records, then the mbarriers:
//     full[kStages], empty[kStages], s_full[2], pv_done[2], p_ready, q_free[2], mma_done
size_t tc_smem_bytes(int stages) {
  return 1024 + (size_t)stages * kStageBytes + 4 * kTcTileBytes + 4 * kTcTileBytes +
         (size_t)stages * sizeof(StageMeta) + (size_t)(2 * stages + 8) * 8;
}

template <int kStages>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap tm_khot, const __grid_constant__ CUtensorMap tm_vhot,
              const __grid_constant__ CUtensorMap tm_kst, const __grid_constant__ CUtensorMap tm_vst,
              const __grid_constant__ CUtensorMap tm_q, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *stages = smem;
  uint8_t *qtile = stages + kStages * kStageBytes;
  uint8_t *pbuf = qtile + 4 * kTcTileBytes;
  StageMeta *meta = reinterpret_cast<StageMeta *>(pbuf + 4 * kTcTileBytes);
  uint64_t *bars = reinterpret_cast<uint64_t *>(meta + kStages);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);
  const uint32_t sfull0 = smem_u32(bars + 2 * kStages), pvdone0 = smem_u32(bars + 2 * kStages + 2);
  const uint32_t pready = smem_u32(bars + 2 * kStages + 4), qfree0 = smem_u32(bars + 2 * kStages + 5);
  const uint32_t mmadone = smem_u32(bars + 2 * kStages + 7);

  __shared__ int s_fix, s_ready, s_pub;
  __shared__ uint32_t s_tmem;
  // per column group of each row: the stage maxima, and at a run end the row
  // sums (the same words: a run end reads the sums before a barrier that every
  // thread passes before it writes the next stage's maxima)
  __shared__ float s_red[kTcColGroups][kTcM];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // The V halves of the tile ring start zeroed: rows of chunk slots that a
  // stage does not load keep older tile data, which is then finite (P is
  // exactly 0 there, and a 0 x Inf product would reach the whole row of O).
  for (int i = tid * 16; i < kStages * 2 * kHalfBytes; i += kTcThreads * 16)
    *reinterpret_cast<uint4 *>(stages + (i / (2 * kHalfBytes)) * kStageBytes + 2 * kHalfBytes + i % (2 * kHalfBytes)) =
        make_uint4(0, 0, 0, 0);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);   // released by the commit after the stage's PV
    }
    for (int i = 2 * kStages; i < 2 * kStages + 8; ++i) mbar_init(smem_u32(bars + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_ready = 0;
    s_pub = 0;
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int total = p.chunk_off[p.units];
  const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
  const int lo = min(total, (int)blockIdx.x * per), hi = min(total, lo + per);
  if (lo >= hi) return;
  if (load_status(p.status) != 0) return;

  // tensor memory: allocated by warp 0, freed by it once the MMA and softmax warps are done
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kTcTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t tmem_o = tmem + 2 * kTcM;   // O: columns 128..255

  if (warp >= kTcSoftmaxWarps) {
    // warps 8 and 9 issue the stages alternately and warp 10 finishes; when
    // the gather is fused, warp 8 issues every stage and warp 9 copies (warp
    // 10 has nothing to do).  Warp 11 issues the MMAs.
    const int pw = warp - kTcSoftmaxWarps;
    if (pw < 3) {
      const bool fused = p.kh != nullptr;
      if (pw == 0 || (pw == 1 && !fused))
        attn_producer_warp<kStages>(p, &tm_khot, &tm_vhot, &tm_kst, &tm_vst, lo, hi, per, 0, stages, qtile, 0, meta,
                                    full0, empty0, &s_ready, &s_pub, 1, pw, fused ? 1 : 2, &tm_q, qfree0);
      else if (pw == (fused ? 1 : 2))
        attn_producer_warp<kStages>(p, &tm_khot, &tm_vhot, &tm_kst, &tm_vst, lo, hi, per, 1, stages, qtile, 0, meta,
                                    full0, empty0, &s_ready, &s_pub, 1);
      return;
    }
    // ---------------------------------------------------------------- MMA warp
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(kTcM, kStageRows, 0, 0);
      const uint32_t id_o = idesc_bf16(kTcM, 128, 0, 1);
      const uint32_t qt = smem_u32(qtile), pb = smem_u32(pbuf), st0 = smem_u32(stages);
      // O += P V of stage t: P from buffer t & 1, V of ring slot t % kStages; the
      // first of a run overwrites O.  Its completion frees the ring slot and the
      // P buffer.
      auto issue_pv = [&](int t, bool first) -> bool {
        if (!mbar_wait(pready, t & 1, p.status)) return false;
        tc_fence_after();
        const uint32_t pa = pb + (t & 1) * 2 * kTcTileBytes;
        const uint32_t vb = st0 + (t % kStages) * kStageBytes + 2 * kHalfBytes;
#pragma unroll
        for (int ks = 0; ks < kStageRows / 16; ++ks) {
          const uint64_t b = smem_desc_sw128(vb + ks * 16 * 128, kHalfBytes, 1024);
          tc_mma(tmem_o, smem_desc_sw128(pa + ks * 32, 16, 1024), b, id_o, !(first && ks == 0));
          tc_mma(tmem_o, smem_desc_sw128(pa + kTcTileBytes + ks * 32, 16, 1024), b, id_o, 1);
        }
        tc_commit(empty0 + 8 * (t % kStages));
        tc_commit(pvdone0 + 8 * (t & 1));
        return true;
      };
      int run = 0, pend = -1;
      uint32_t qrun = qt;
      bool pend_first = false, ok = true;
      for (int s = 0; ok; ++s) {
        const int b = s % kStages;
        if (!mbar_wait(full0 + 8 * b, (s / kStages) & 1, p.status)) break;
        const int flags = meta[b].flags;
        if (flags & kFirst) {
          // a new run, its queries in the Q tile of its parity (they came with
          // this stage); every MMA issued so far, among them the last that
          // read the previous run's queries, frees that run's tile once done
          if (run > 0) tc_commit(qfree0 + 8 * ((run - 1) & 1));
          qrun = qt + (uint32_t)(run & 1) * 2u * kTcTileBytes;
          ++run;
        }
        tc_fence_after();
        // S(s) into buffer s & 1 (the softmax warps are done with S(s - 2): P(s - 2) is ready)
        const uint32_t kb = st0 + b * kStageBytes;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
          tc_mma(tmem + (s & 1) * kTcM, smem_desc_sw128(qrun + (ks >> 2) * kTcTileBytes + (ks & 3) * 32, 16, 1024),
                 smem_desc_sw128(kb + off, 16, 1024), id_s, ks > 0);
        }
        tc_commit(sfull0 + 8 * (s & 1));
        if (pend >= 0 && !(ok = issue_pv(pend, pend_first))) break;
        pend = s;
        pend_first = (flags & kFirst) != 0;
        if (flags & kEnd) {
          ok = issue_pv(pend, pend_first);
          break;
        }
      }
      // every MMA issued has completed before the tensor memory is freed
      tc_commit(mmadone);
      mbar_wait(mmadone, 0, p.status);
    }
    __syncwarp();
    tc_fence_before();
    asm volatile("bar.sync 2, %0;" ::"r"((kTcSoftmaxWarps + 1) * 32) : "memory");
    return;
  }

  // -------------------------------------------------------------- softmax warps
  // Row r = 16 * (warp & 3) + (lane & 15) is query vector r.  The
  // kTcColGroups warps w, w + 4, ... read the same tensor-memory lane quarter
  // and take the row's columns in as many groups (warp >> 2); inside a warp
  // the 16x32bx2 access gives lanes t and t + 16 the two halves of a group:
  // kSCols columns of S and kOCols of O each.
  constexpr int kSCols = kTcM / (2 * kTcColGroups), kOCols = 128 / (2 * kTcColGroups);
  const int wq = warp & 3, wc = warp >> 2, sub = lane >> 4;
  const int row = 16 * wq + (lane & 15);
  const int col0 = (2 * wc + sub) * kSCols;      // this thread's S columns [col0, col0 + kSCols)
  const int ocol = (2 * wc + sub) * kOCols;      // and O columns
  const bool active = row < p.NQ;
  const int j = active ? row / p.G : 0;
  const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
  const float sl2 = p.scale_log2;
  const int slots = kStageRows / p.cs;           // chunk slots per stage
  float m_ref = -INFINITY, l = 0.f;              // l: this thread's part of the row sum
  for (int s = 0;; ++s) {
    const int b = s % kStages;
    if (!mbar_wait(full0 + 8 * b, (s / kStages) & 1, p.status)) break;
    const int m_nch = meta[b].nch, m_flags = meta[b].flags, m_unit = meta[b].unit;
    const int m_uoff = meta[b].uoff, m_ucnt = meta[b].ucnt;
    uint32_t qm4 = 0;   // the stage's four query masks, one byte each
#pragma unroll
    for (int i = 0; i < kMaxChunksPerStage; ++i) qm4 |= (uint32_t)meta[b].qm[i] << (8 * i);
    if (m_flags & kFirst) {   // a new run (its queries came by TMA with the stage)
      m_ref = -INFINITY;
      l = 0.f;
    }
    if (!mbar_wait(sfull0 + 8 * (s & 1), (s >> 1) & 1, p.status)) break;
    tc_fence_after();
    float x[kSCols];
    tmem_ld_cols<kSCols>(tmem + lane_base + (s & 1) * kTcM + 2 * kSCols * wc, x);
    // the stage's rows query j sees (loaded and picked)
    const uint32_t cm = active ? (uint32_t)(meta[b].rows_of[j] >> col0) & ((1u << kSCols) - 1u) : 0u;
    // (raw scores here; the scale is applied to the maximum and inside the
    // exponent: x -> x * scale is increasing, so max(x) * scale is the maximum
    // of the scaled scores exactly)
#pragma unroll
    for (int t = 0; t < kSCols; ++t) x[t] = ((cm >> t) & 1u) ? x[t] : -INFINITY;
    float pm = x[0];
#pragma unroll
    for (int t = 1; t < kSCols; ++t) pm = fmaxf(pm, x[t]);
    pm *= sl2;
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));   // this warp's group of the row
    if (sub == 0) s_red[wc][row] = pm;
    // One barrier with an OR reduction both exchanges the halves' maxima and
    // takes the group's vote on a rescale (a row's maximum exceeds its
    // reference by more than 2^8 iff one of its halves does).  Before P(s)
    // goes into buffer s & 1, PV(s - 2) (its last reader) must be done;
    // before any row of O is rescaled, PV(s - 1) too.  Every softmax thread
    // waits on the same barrier, so a wait that runs out stops the whole
    // group at one place.
    uint32_t group_rescale;
    asm volatile(
        "{\n .reg .pred q, r;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred r, 1, %2, q;\n selp.u32 %0, 1, 0, r;\n}\n"
        : "=r"(group_rescale)
        : "r"((uint32_t)(pm > m_ref + kRescaleLog2)), "r"(kTcSoftmaxWarps * 32)
        : "memory");
    float mx = pm;
#pragma unroll
    for (int c = 0; c < kTcColGroups; ++c) mx = fmaxf(mx, s_red[c][row]);
    float factor = 1.f;
    if (mx > m_ref + kRescaleLog2) {
      if (m_ref != -INFINITY) factor = exp2f(m_ref - mx);
      m_ref = mx;
    }
    const int wait_for = group_rescale ? s - 1 : s - 2;
    if (wait_for >= 0 && !mbar_wait(pvdone0 + 8 * (wait_for & 1), (wait_for >> 1) & 1, p.status)) break;
    tc_fence_after();
    if (__any_sync(0xffffffffu, factor != 1.f)) {
      // the accumulator moves to the new reference, before PV(s): this
      // thread's columns of O
      float o[kOCols];
      tmem_ld_cols<kOCols>(tmem_o + lane_base + 2 * kOCols * wc, o);
#pragma unroll
      for (int i = 0; i < kOCols; ++i) o[i] *= factor;
      tmem_st_cols<kOCols>(tmem_o + lane_base + 2 * kOCols * wc, o);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      l *= factor;
    }
    if (active) {
      // p = 2^(x - ref) as bf16 hi + lo parts, both truncations: hi keeps the
      // top 8 significant bits, lo = p - hi (exact in fp32) the next 8, so
      // hi + lo carries p to ~2^-14 relative
      uint8_t *ph = pbuf + (s & 1) * 2 * kTcTileBytes + row * 128;
      const float nbase = m_ref == -INFINITY ? -INFINITY : -m_ref;   // an all-masked row: every p is 0
      float gsum[kSCols / 8];
#pragma unroll
      for (int c2 = 0; c2 < kSCols / 8; ++c2) {
        float e[8];
        uint32_t hb[8], lb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          e[i] = ex2_approx(fmaf(x[c2 * 8 + i], sl2, nbase));
          hb[i] = __float_as_uint(e[i]) & 0xFFFF0000u;
          lb[i] = __float_as_uint(e[i] - __uint_as_float(hb[i]));
        }
        gsum[c2] = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
        const uint4 h = make_uint4(__byte_perm(hb[0], hb[1], 0x7632), __byte_perm(hb[2], hb[3], 0x7632),
                                   __byte_perm(hb[4], hb[5], 0x7632), __byte_perm(hb[6], hb[7], 0x7632));
        const uint4 lw = make_uint4(__byte_perm(lb[0], lb[1], 0x7632), __byte_perm(lb[2], lb[3], 0x7632),
                                    __byte_perm(lb[4], lb[5], 0x7632), __byte_perm(lb[6], lb[7], 0x7632));
        const int c8 = (col0 >> 3) + c2;   // 16-byte chunk of the row (tokens 8 c8 .. 8 c8 + 7)
        const uint32_t off = (uint32_t)((c8 ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(ph + off) = h;
        *reinterpret_cast<uint4 *>(ph + kTcTileBytes + off) = lw;
      }
#pragma unroll
      for (int c2 = 0; c2 < kSCols / 8; ++c2) l += gsum[c2];
    }
    // V rows of chunk slots this stage did not load: zero (their P is 0)
    if (!(m_flags & kFull))
    for (int i = 0; i < slots; ++i) {
      if (((qm4 >> (8 * i)) & 0xFFu) != 0u && i < m_nch) continue;
      uint8_t *vb = stages + b * kStageBytes + 2 * kHalfBytes + i * p.cs * 128;
      for (int e = tid * 16; e < p.cs * 128; e += kTcSoftmaxWarps * 32 * 16) {
        *reinterpret_cast<uint4 *>(vb + e) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(vb + kHalfBytes + e) = make_uint4(0, 0, 0, 0);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"r"(kTcSoftmaxWarps * 32) : "memory");
    if (tid == 0) mbar_arrive(pready);

    if (m_flags & kLast) {
      // the run's O is final once PV(s) completed
      if (!mbar_wait(pvdone0 + 8 * (s & 1), (s >> 1) & 1, p.status)) break;
      tc_fence_after();
      const float lh = l + __shfl_xor_sync(0xffffffffu, l, 16);
      if (sub == 0) s_red[wc][row] = lh;
      asm volatile("bar.sync 1, %0;" ::"r"(kTcSoftmaxWarps * 32) : "memory");
      float lrow = 0.f;
#pragma unroll
      for (int c = 0; c < kTcColGroups; ++c) lrow += s_red[c][row];
      asm volatile("bar.sync 1, %0;" ::"r"(kTcSoftmaxWarps * 32) : "memory");   // the sums are read
      const int c0 = m_uoff / per, c1 = (m_uoff + m_ucnt - 1) / per;
      const bool direct = c0 == c1 && p.k_tail == nullptr;
      const bool handoff = c0 != c1 && p.kh == nullptr && m_uoff < lo && !(m_flags & kEnd);
      const int bb = m_unit / p.Hkv, g = m_unit - bb * p.Hkv;
      float *dst = nullptr;
      float inv = 1.f;
      if (active) {
        if (direct) {
          const int h = g * p.G + (row - j * p.G);
          dst = p.out + ((int64_t)(bb * p.n_q + j) * p.Hq + h) * 128 + ocol;
          inv = lrow > 0.f ? 1.f / lrow : 0.f;
        } else {
          const int64_t k = ((int64_t)blockIdx.x + m_unit) * p.NQ + row;
          dst = p.part_o + k * 128 + ocol;
          if (wc == 0 && sub == 0) *reinterpret_cast<float2 *>(p.part_ml + k * 2) = make_float2(m_ref, lrow);
        }
      }
      {
        float o[kOCols];
        tmem_ld_cols<kOCols>(tmem_o + lane_base + 2 * kOCols * wc, o);
        if (active) {
#pragma unroll
          for (int i = 0; i < kOCols; i += 4)
            *reinterpret_cast<float4 *>(dst + i) = make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
        }
      }
      tc_fence_before();   // O is read before the next run's first PV overwrites it
      m_ref = -INFINITY;
      l = 0.f;
      if (handoff) {
        // the partial is written: hand it to the finisher warp
        asm volatile("bar.sync 1, %0;" ::"r"(kTcSoftmaxWarps * 32) : "memory");
        if (tid == 0) asm volatile("red.release.cta.shared.add.u32 [%0], 1;" ::"r"(smem_u32(&s_pub)) : "memory");
      } else if (!direct) {
        asm volatile("bar.sync 1, %0;" ::"r"(kTcSoftmaxWarps * 32) : "memory");
        if (tid == 0) s_fix = c0 == c1 || atom_add_acq_rel_gpu(p.arrive + m_unit, 1) + 1 == c1 - c0 + 1;
        asm volatile("bar.sync 1, %0;" ::"r"(kTcSoftmaxWarps * 32) : "memory");
        if (s_fix) fixup_unit(p, m_unit, c0, c1, kTcSoftmaxWarps * 32, tid);
      }
    }
    if (m_flags & kEnd) break;
  }
  tc_fence_before();
  asm volatile("bar.sync 2, %0;" ::"r"((kTcSoftmaxWarps + 1) * 32) : "memory");
  if (p.trace) {
    asm volatile("bar.sync 1, %0;" ::"r"(kTcSoftmaxWarps * 32) : "memory");
    if (tid == 0) trace_end(p.trace);
  }
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols) : "memory");
  }
}

}  // namespace


cudaError_t launch_attn_tc(int n_cta, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &c,
                           const CUtensorMap &d, const CUtensorMap &tq, const AttnParams &p, cudaStream_t s) {
  // five stages when they fit beside the kernel's static shared memory in the
  // per-block limit, else four
  static int five = -1;
  if (five < 0) {
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, (const void *)k_attn_tc<5>);
    if (e != cudaSuccess) return e;
    five = tc_smem_bytes(5) + fa.sharedSizeBytes <= (size_t)optin ? 1 : 0;
  }
  const size_t smem = tc_smem_bytes(five ? 5 : 4);
  const void *fn = five ? (const void *)k_attn_tc<5> : (const void *)k_attn_tc<4>;
  cudaError_t e = set_dyn_smem(fn, smem);
  if (e != cudaSuccess) return e;
  return five ? launch_k(k_attn_tc<5>, dim3(n_cta), dim3(kTcThreads), smem, s, a, b, c, d, tq, p)
              : launch_k(k_attn_tc<4>, dim3(n_cta), dim3(kTcThreads), smem, s, a, b, c, d, tq, p);
}

int attn_tc_threads() { return kTcThreads; }

}  // namespace dd
