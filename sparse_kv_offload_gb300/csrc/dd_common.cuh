// Shared device helpers of libdd (CUDA path only).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "dd.h"

namespace dd {

constexpr int kD = 128;          // head dimension the kernels are built for
constexpr int kVecPerRow = 16;   // uint4 (8 x bf16) per row of d = 128
constexpr int kMaxNq = 8;
constexpr int kMaxC = 16384;
constexpr int kMaxNQV = 64;      // n_q * G query vectors per KV head

// Record a device-side error; the first error wins.
__device__ __forceinline__ void set_status(int32_t *status, int32_t code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ int32_t load_status(const int32_t *status) {
  return *reinterpret_cast<const volatile int32_t *>(status);
}

// bf16 pair in one 32-bit word -> two floats (exact)
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 &v, float f[8]) {
  f[0] = bf_lo(v.x); f[1] = bf_hi(v.x);
  f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
  f[4] = bf_lo(v.z); f[5] = bf_hi(v.z);
  f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// fp32 -> bf16 bits, round to nearest even (finite inputs; NaN kept quiet)
__device__ __forceinline__ uint32_t f2bf(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (u >> 16) | 0x40u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return u >> 16;
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  return f2bf(lo) | (f2bf(hi) << 16);
}

__device__ __forceinline__ uint4 ldg_nc(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

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

// ---------------------------------------------------------------------------
// mbarriers (shared memory) with a bounded wait
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

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

// Bounded wait until a 64-bit word carries `epoch` in its top 30 bits (the
// look-back words of the fused selection).  Returns the word; sets *ok to
// false and stops waiting ~2 s after t0 (the caller records DD_ERR_TIMEOUT).
__device__ __forceinline__ unsigned long long wait_published(const unsigned long long *word, uint32_t epoch,
                                                             uint64_t t0, bool *ok) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(word) : "memory");
  for (uint32_t it = 0; *ok && (w >> 34) != epoch; ++it) {
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(word) : "memory");
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > 2000000000ull) *ok = false;
  }
  return w;
}

// Optional in-step timing (dd_step_args.trace): one pair of words per SM so
// that only the CTAs sharing an SM contend; the reader takes the minimum of
// the starts and the maximum of the ends over the kTraceSlots slots.
constexpr int kTraceSlots = DD_TRACE_SLOTS;
__device__ __forceinline__ int trace_slot() {
  uint32_t id;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
  return (int)(id & (kTraceSlots - 1));
}
// Out of line: called once per CTA, they should not add to the register
// pressure of the kernels' main loops.
static __device__ __noinline__ void trace_start(unsigned long long *t) {   // t: this kernel's [2][kTraceSlots]
  atomicMin(t + trace_slot(), (unsigned long long)globaltimer_ns());
}
static __device__ __noinline__ void trace_end(unsigned long long *t) {
  atomicMax(t + kTraceSlots + trace_slot(), (unsigned long long)globaltimer_ns());
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier (16-byte
// aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialization (launch_k below): its CTAs may become
// resident while the previous kernel in the stream is still finishing, so the
// launch and the shared-memory set-up overlap that kernel's tail.  Each kernel
// therefore calls pdl_wait() unconditionally, before its first global-memory
// access and before any early return: the wait returns once every earlier
// kernel in the stream has completed and its writes are visible, which also
// keeps the completion order transitive along the chain.  pdl_trigger() lets
// the next kernel's CTAs launch early; it is issued right after the wait.
// One exception: the scoring kernel requests its first landmark tiles before
// its wait (landmarks are an input of the step, not an output of the kernel
// before it), so the landmark builders skip pdl_trigger and release their
// dependents only at exit.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// block-wide exclusive scan of one int per thread (blockDim a multiple of 32)
// ---------------------------------------------------------------------------
__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// `scratch` holds 33 ints of shared memory.  Returns the exclusive prefix and
// the block total; ends with a barrier so scratch can be reused.
__device__ __forceinline__ int block_excl_scan(int v, int *scratch, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int incl = warp_incl_scan(v);
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int x = lane < nw ? scratch[lane] : 0;
    const int xi = warp_incl_scan(x);
    if (lane < nw) scratch[lane] = xi - x;
    if (lane == 31) scratch[32] = xi;
  }
  __syncthreads();
  const int r = scratch[warp] + incl - v;
  *total = scratch[32];
  __syncthreads();
  return r;
}

// block-wide sum of one int per thread (blockDim a multiple of 32; scratch 33 ints)
__device__ __forceinline__ int block_sum(int v, int *scratch) {
  int tot;
  block_excl_scan(v, scratch, &tot);
  return tot;
}

// Work plan of the attention kernel (dd_attn.cu), built per (b, g) unit by
// the resolver or by the attention's own plan kernel.  The unions of all
// units are laid end to end: chunk x of that sequence is position
// x - chunk_off[u] of unit u's union.  The attention kernel plans itself
// from it: persistent CTA c takes chunks [c*per, (c+1)*per) with
// per = ceil(chunk_off[units] / number of CTAs).
struct AttnPlanOut {
  int32_t *chunk_off;   // [units + 1] exclusive prefix of the union sizes, then [units] arrival counters
                        // of the attention's stream-K fix-up, which the planner zeroes
  int4 *flat;           // [units * umax] per chunk: {first pool row (hot) | -2 - row (staging) | -1, query mask,
                        //  host chunk (b*Hkv+g)*C + c for staging chunks | -1, 0}
};

// One CTA, all threads: the plan entries that belong to `unit`.
__device__ __forceinline__ void attn_plan_unit(const AttnPlanOut &po, int unit, int units, int off, int U, int total,
                                               const int32_t *uslot, const uint8_t *uqm, const int32_t *uidx,
                                               int C, int64_t m_valid, int64_t hot_slots, int cs, int32_t *status) {
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int i = tid; i < U; i += nt) {
    const int32_t slot = uslot[i];
    uint32_t qm = uqm[i];
    const bool hot_ok = slot >= 0 && slot < hot_slots;
    const bool st_ok = slot < 0 && (-(int64_t)slot - 1) < m_valid;
    int32_t row = -1;
    if (!hot_ok && !st_ok) {
      set_status(status, DD_ERR_DEVICE_CHECK);
      qm = 0;
    } else if (qm) {
      const int32_t r = (int32_t)((slot >= 0 ? (int64_t)slot : (-(int64_t)slot - 1)) * cs);
      row = slot >= 0 ? r : -2 - r;
    }
    const int host = (uidx && slot < 0 && row != -1) ? unit * C + uidx[i] : -1;
    po.flat[off + i] = make_int4(row, (int)qm, host, 0);
  }
  if (tid == 0) {
    po.chunk_off[unit] = off;
    po.chunk_off[units + 1 + unit] = 0;   // arrival counter of the attention's fix-up
    if (unit == units - 1) po.chunk_off[units] = total;
  }
}

}  // namespace dd

// Host-side launch helpers, defined with their kernels
namespace dd {
struct Ctx;
// dynamic shared-memory opt-in of a kernel on the current device, cached (dd_host.cu)
cudaError_t set_dyn_smem(const void *func, size_t bytes);
cudaError_t launch_build_landmarks(const uint4 *K, uint4 *lm, int64_t n_chunks, int cs, cudaStream_t s);
cudaError_t launch_score_tc(const void *q, const void *lm, float *scores, int B, int n_q, int Hq, int Hkv, int C,
                            int sm_count, int32_t *status, cudaStream_t s, unsigned long long *trace);
cudaError_t launch_score(const uint4 *q, const uint4 *lm, float *scores, int B, int n_q, int Hq, int Hkv,
                         int C, int sm_count, int32_t *status, cudaStream_t s, unsigned long long *trace = nullptr);
cudaError_t launch_build_minmax(const uint4 *K, uint4 *lm2, int64_t n_chunks, int cs, cudaStream_t s);
cudaError_t launch_score_minmax(const uint4 *q, const uint4 *lm2, float *scores, int B, int n_q, int Hq, int Hkv,
                                int C, int sm_count, int32_t *status, cudaStream_t s,
                                unsigned long long *trace = nullptr);
cudaError_t launch_topk(const float *scores, int32_t *sel, int rows, int C, int k, cudaStream_t s);
// outputs and state of the fused selection kernel (dd_select.cu)
struct SelectOut {
  const float *scores;            // [B,n_q,Hkv,C] input: the scoring kernel's rows
  int32_t *sel;                   // [B,n_q,Hkv,k] or null
  int32_t *attn_slot;             // [B,n_q,Hkv,k] or null
  const int32_t *resident_slot;   // [B,Hkv,C]
  int32_t *union_idx, *union_slot;
  uint8_t *union_qmask;
  int32_t *union_cnt, *unit_miss, *miss_list, *miss_count;
  int32_t *chunk_off;             // attention plan: [units + 1], then [units] fix-up counters
  int4 *flat;                     // attention plan: [units * umax]
  unsigned long long *lb_word;    // look-back: [units] {epoch:30, union count:17, miss count:17}
  int32_t *ticket;                // [3] next unit, CTAs done, look-back epoch of the next launch (never 0)
  // [16 * units] every unit's union and miss offsets {epoch:32, offset:32}
  // (words 16u and 16u + 1), written by the last CTA to arrive when all of
  // the launch's CTAs are resident at once; null: the look-back over the
  // earlier units instead
  unsigned long long *lb_pref;
  int units, Hq, Hkv, C, k, umax, cs;
  int64_t hot_slots, max_misses;
  int32_t *status;
  unsigned long long *trace;      // optional [2][kTraceSlots]: per-SM earliest start, latest end (ns)
  int sm_count;                   // SMs of the device (two CTAs per SM when the units outnumber them)
  bool after_tc_score;            // launched behind the tensor-core scoring kernel (one CTA on every SM)
  // scoring folded in (mean landmarks): the landmarks as a 2-D tensor map
  // ([units * C, 128] bf16, boxes of 128 rows x 64 columns), the queries, the
  // score rows when asked for, the scoring phase's timing words
  CUtensorMap tm_lm;
  const uint16_t *q16;
  float *scores_out;
  unsigned long long *trace_score;
};
size_t fused_select_smem(int n_q, int C, int k);
cudaError_t launch_select_fused(const SelectOut &o, int n_q, cudaStream_t s);
// the ring stages of the kernel with the scoring folded in for this step (0:
// the two-kernel path: units not filling one wave of SMs, or too large)
int score_select_stages(int units, int sm_count, int n_q, int C, int k);
cudaError_t launch_score_select(const SelectOut &o, int n_q, int stages, cudaStream_t s);
cudaError_t launch_selftest_wait(int kind, const unsigned long long *word, int32_t *status, cudaStream_t s);
cudaError_t launch_topk_mass(const float *scores, int32_t *sel, int32_t *sel_cnt, int rows, int C, int k_max,
                             int k_min, float gamma, float tau_log2e, cudaStream_t s);
cudaError_t launch_union(const int32_t *sel, const int32_t *resident_slot, int32_t *union_idx,
                         int32_t *union_slot, uint8_t *union_qmask, int32_t *union_cnt,
                         int32_t *unit_miss, int units, int n_q, int Hkv, int k, int C, int umax,
                         int64_t hot_slots, int32_t *status, cudaStream_t s, int sel_rows = 0);
cudaError_t launch_assign(const int32_t *sel, const int32_t *union_idx, int32_t *union_slot,
                          const uint8_t *union_qmask, const int32_t *union_cnt, const int32_t *unit_miss,
                          int32_t *miss_list, int32_t *miss_count, int32_t *attn_slot, int units, int n_q, int Hkv,
                          int k, int C, int umax, int64_t max_misses, int64_t hot_slots, int cs,
                          const AttnPlanOut *plan, int32_t *status, cudaStream_t s);
// attention: launch plan (persistent CTAs, partial slots) and scratch
struct AttnPlan {
  int n_cta;
  int64_t part_o_floats, part_ml_floats, flat_entries;
};
struct AttnScratch {
  float *part_o, *part_ml;
  int32_t *chunk_off;         // [units + 1], then [units] fix-up counters
  int4 *flat;                 // [units * umax]
  const void *dummy_pool;     // >= 64 rows x 256 B, a valid base for unused tensor maps
};
AttnPlan attn_plan(int units, int umax, int NQ, int sm_count);
cudaError_t launch_attn(const void *q, const void *Khot, const void *Vhot, const void *Kst, const void *Vst,
                        const int32_t *union_slot, const uint8_t *union_qmask, const int32_t *union_cnt,
                        const int32_t *miss_count, float softmax_scale, float *out, const AttnPlan &plan,
                        const AttnScratch &scr, bool plan_ready, const void *kh_dev, const void *vh_dev,
                        int32_t *status, int B, int n_q, int Hq, int Hkv, int cs, int umax, int64_t hot_slots,
                        int64_t max_misses, cudaStream_t s, const void *k_tail = nullptr,
                        const void *v_tail = nullptr, unsigned long long *trace = nullptr);
cudaError_t launch_update_residency(int32_t step, int32_t cap, int S, int units, const int32_t *union_idx,
                                    const int32_t *union_slot, const int32_t *union_cnt, const int32_t *miss_count,
                                    int64_t max_misses, const uint4 *Kst, const uint4 *Vst, int32_t *resident_slot,
                                    int32_t *slot_chunk, int32_t *last_used, uint4 *Khot, uint4 *Vhot,
                                    int32_t *admitted, int C, int umax, int cs, int32_t *status, cudaStream_t s);
cudaError_t launch_gather(const uint4 *Kh, const uint4 *Vh, const int32_t *miss_list,
                          const int32_t *miss_count, uint4 *Kst, uint4 *Vst, int64_t max_misses,
                          int64_t n_chunks_total, int cs, int32_t *status, int sm_count, cudaStream_t s,
                          int32_t *map_out = nullptr, int ctas_per_sm = 8);
}  // namespace dd
