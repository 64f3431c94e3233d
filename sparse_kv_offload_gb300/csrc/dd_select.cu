// Per-row top-k chunk selection and the cross-query union / residency resolver.
//
// OasisKV summary, Methodology: blocks are ranked independently for every KV
// head and the top-K kept.  Adaptive DHiSparse, Figs. 2 and 3: the selections
// of all queries of a request are resolved together (hot pool first, host for
// the rest), so a chunk wanted by several queries crosses the host link a
// single time; attention still uses each query's own top-k.
#include <algorithm>
#include <mutex>

#include "dd_tc.cuh"

namespace dd {

// Order-preserving map fp32 -> uint32: larger float, larger key.  -0 maps to
// +0's key; NaN maps to 0, below every number.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// a2: one CTA per (b, j, g) row.  Radix select (4 passes of 8 bits, most
// significant first) finds the k-th largest key T and how many keys equal to
// T are needed; a scan over the row in chunk order then emits every key > T
// and the lowest-index keys == T, which yields the (score desc, index asc)
// top-k listed in ascending chunk order.
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 512;

// Radix select over the order keys of one row: the k-th largest key T and how
// many keys equal to T belong to the top k (the lowest chunks first).
__device__ __forceinline__ void radix_threshold(const uint32_t *keys, int C, int k, int *hist, uint32_t *s_prefix,
                                                int *s_remaining, uint32_t &T, int &need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, pmask = 0;
  int remaining = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    for (int i = tid; i < C; i += kTopkThreads) {
      const uint32_t key = keys[i];
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l down to 248-8l (descending digit order)
      int cnt[8], s = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cnt[e] = hist[255 - 8 * lane - e];
        s += cnt[e];
      }
      const int incl = warp_incl_scan(s);
      const int excl = incl - s;
      if (excl < remaining && remaining <= incl) {
        int r = remaining - excl;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (r > 0 && r <= cnt[e]) {
            *s_prefix = prefix | ((uint32_t)(255 - 8 * lane - e) << shift);
            *s_remaining = r;
            r = 0;
          } else if (r > 0) {
            r -= cnt[e];
          }
        }
      }
    }
    __syncthreads();
    prefix = *s_prefix;
    remaining = *s_remaining;
    pmask |= 0xFFu << shift;
    __syncthreads();
  }
  T = prefix;
  need = remaining;
}

// Writes the top-k chunks of the row (every key > T, and the `need` lowest
// chunks with key == T) to dst in ascending chunk order.
__device__ __forceinline__ void emit_topk(const uint32_t *keys, int C, uint32_t T, int need, int *scratch,
                                          int32_t *dst) {
  const int tid = threadIdx.x;
  const int per = (C + kTopkThreads - 1) / kTopkThreads;
  const int lo = min(C, tid * per), hi = min(C, lo + per);
  int eq_local = 0;
  for (int c = lo; c < hi; ++c) eq_local += (keys[c] == T);
  int tot;
  const int eq_before = block_excl_scan(eq_local, scratch, &tot);
  int take = 0;
  {
    int er = eq_before;
    for (int c = lo; c < hi; ++c) {
      const uint32_t key = keys[c];
      if (key > T) ++take;
      else if (key == T) { take += (er < need); ++er; }
    }
  }
  int pos = block_excl_scan(take, scratch, &tot);
  int er = eq_before;
  for (int c = lo; c < hi; ++c) {
    const uint32_t key = keys[c];
    bool t = key > T;
    if (key == T) { t = er < need; ++er; }
    if (t) dst[pos++] = c;
  }
}

__global__ void __launch_bounds__(kTopkThreads) k_topk(const float *__restrict__ scores, int32_t *__restrict__ sel,
                                                       int C, int k) {
  extern __shared__ uint32_t keys[];
  __shared__ int hist[256];
  __shared__ int scratch[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  pdl_wait();
  pdl_trigger();

  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const float *src = scores + (int64_t)row * C;
  for (int i = tid; i < C; i += kTopkThreads) keys[i] = order_key(src[i]);
  uint32_t T;
  int need;
  radix_threshold(keys, C, k, hist, &s_prefix, &s_remaining, T, need);
  emit_topk(keys, C, T, need, scratch, sel + (int64_t)row * k);
}

cudaError_t launch_topk(const float *scores, int32_t *sel, int rows, int C, int k, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const size_t smem = (size_t)C * sizeof(uint32_t);
  if (smem > 48 * 1024) {   // the opt-in is per device, so ask on every launch that needs it
    cudaError_t e = set_dyn_smem((const void *)k_topk, smem);
    if (e != cudaSuccess) return e;
  }
  return launch_k(k_topk, dim3(rows), dim3(kTopkThreads), smem, s, scores, sel, C, k);
}

// ---------------------------------------------------------------------------
// a2 with a coverage budget (MOIRA: per request, layer, KV head and step, the
// smallest set of chunks whose estimated attention mass reaches gamma).  One
// CTA per row: the top k_max chunks by radix select as above; their scores
// sorted by (score desc, chunk asc) with a bitonic sort in shared memory;
// masses w = exp2((s - max s) * tau_log2e) and Z = the sum over the whole
// row, both in fp32 in a fixed order (per-thread sequential sums, then a
// fixed tree), so the result is the same on every run; k_row = 1 + the
// number of sorted prefixes below gamma * Z, clamped to [k_min, k_max].  The
// row is written as its k_row chunks ascending, then -1.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_sum_f(float v, float *scratchf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) scratchf[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < nw; ++w) t += scratchf[w];
    scratchf[32] = t;
  }
  __syncthreads();
  const float r = scratchf[32];
  __syncthreads();
  return r;
}

__device__ __forceinline__ float block_max_f(float v, float *scratchf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) scratchf[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = -INFINITY;
    for (int w = 0; w < nw; ++w) t = fmaxf(t, scratchf[w]);
    scratchf[32] = t;
  }
  __syncthreads();
  const float r = scratchf[32];
  __syncthreads();
  return r;
}

// exclusive scan of one float per thread in thread order (fixed order); total in *total
__device__ __forceinline__ float block_excl_scan_f(float v, float *scratchf, float *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) scratchf[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < nw; ++w) {
      const float x = scratchf[w];
      scratchf[w] = t;
      t += x;
    }
    scratchf[32] = t;
  }
  __syncthreads();
  const float r = scratchf[warp] + incl - v;
  *total = scratchf[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kTopkThreads) k_topk_mass(const float *__restrict__ scores,
                                                            int32_t *__restrict__ sel, int32_t *__restrict__ sel_cnt,
                                                            int C, int k_max, int k_min, float gamma,
                                                            float tau_log2e) {
  extern __shared__ unsigned long long smem_ull[];
  __shared__ int hist[256];
  __shared__ int scratch[33];
  __shared__ float scratchf[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  pdl_wait();
  pdl_trigger();
  int k_pow = 1;
  while (k_pow < k_max) k_pow <<= 1;
  const int W = (C + 31) >> 5;
  unsigned long long *skey = smem_ull;                                      // [k_pow]
  uint32_t *keys = reinterpret_cast<uint32_t *>(skey + k_pow);              // [C]
  int32_t *list = reinterpret_cast<int32_t *>(keys + C);                    // [k_max]
  uint32_t *bits = reinterpret_cast<uint32_t *>(list + k_max);              // [W]

  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const float *src = scores + (int64_t)row * C;
  float mx = -INFINITY;
  for (int i = tid; i < C; i += kTopkThreads) {
    const float v = src[i];
    keys[i] = order_key(v);
    mx = fmaxf(mx, v);
  }
  for (int i = tid; i < W; i += kTopkThreads) bits[i] = 0u;
  mx = block_max_f(mx, scratchf);
  uint32_t T;
  int need;
  radix_threshold(keys, C, k_max, hist, &s_prefix, &s_remaining, T, need);
  emit_topk(keys, C, T, need, scratch, list);

  // Z over the whole row, sequential per thread, then the fixed tree
  float z = 0.f;
  for (int i = tid; i < C; i += kTopkThreads) z += exp2f((src[i] - mx) * tau_log2e);
  const float Z = block_sum_f(z, scratchf);   // its barriers also publish `list`

  for (int r = tid; r < k_pow; r += kTopkThreads) {
    unsigned long long key = ~0ull;
    if (r < k_max) {
      const int c = list[r];
      key = ((unsigned long long)(~keys[c]) << 32) | (unsigned long long)(uint32_t)c;
    }
    skey[r] = key;
  }
  __syncthreads();
  for (int kk = 2; kk <= k_pow; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < k_pow; i += kTopkThreads) {
        const int x = i ^ j;
        if (x > i) {
          const unsigned long long a = skey[i], b = skey[x];
          if ((a > b) == ((i & kk) == 0)) {
            skey[i] = b;
            skey[x] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  // prefix masses of the sorted list: thread t owns a contiguous segment
  const int per = (k_max + kTopkThreads - 1) / kTopkThreads;
  const int r0 = min(k_max, tid * per), r1 = min(k_max, r0 + per);
  float seg = 0.f;
  for (int r = r0; r < r1; ++r) seg += exp2f((src[(uint32_t)skey[r]] - mx) * tau_log2e);
  float tot;
  float run = block_excl_scan_f(seg, scratchf, &tot);
  const float target = gamma * Z;
  int below = 0;
  for (int r = r0; r < r1; ++r) {
    run += exp2f((src[(uint32_t)skey[r]] - mx) * tau_log2e);
    below += run < target;
  }
  const int n_below = block_sum(below, scratch);
  const int k_row = max(k_min, min(k_max, n_below + 1));
  for (int r = tid; r < k_row; r += kTopkThreads) {
    const uint32_t c = (uint32_t)skey[r];
    atomicOr(&bits[c >> 5], 1u << (c & 31));
  }
  __syncthreads();
  // the chosen chunks in ascending order (list is ascending), then padding
  int32_t *dst = sel + (int64_t)row * k_max;
  int take = 0;
  for (int r = r0; r < r1; ++r) {
    const int c = list[r];
    take += (bits[c >> 5] >> (c & 31)) & 1u;
  }
  int itot;
  int pos = block_excl_scan(take, scratch, &itot);
  for (int r = r0; r < r1; ++r) {
    const int c = list[r];
    if ((bits[c >> 5] >> (c & 31)) & 1u) dst[pos++] = c;
  }
  for (int r = k_row + tid; r < k_max; r += kTopkThreads) dst[r] = -1;
  if (tid == 0 && sel_cnt) sel_cnt[row] = k_row;
}

cudaError_t launch_topk_mass(const float *scores, int32_t *sel, int32_t *sel_cnt, int rows, int C, int k_max,
                             int k_min, float gamma, float tau_log2e, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  int k_pow = 1;
  while (k_pow < k_max) k_pow <<= 1;
  const size_t smem = (size_t)k_pow * 8 + (size_t)C * 4 + (size_t)k_max * 4 + (size_t)((C + 31) / 32) * 4;
  if (smem > 48 * 1024) {
    cudaError_t e = set_dyn_smem((const void *)k_topk_mass, smem);
    if (e != cudaSuccess) return e;
  }
  return launch_k(k_topk_mass, dim3(rows), dim3(kTopkThreads), smem, s, scores, sel, sel_cnt, C, k_max, k_min,
                  gamma, tau_log2e);
}

// ---------------------------------------------------------------------------
// a3, pass 1 (one CTA per (b,g)): per-query bitmaps of the selections, their
// union listed in ascending chunk order with the query mask of each chunk,
// residency lookup, and the (b,g)-local ordinal of every miss, stored as
// -(local+1) in union_slot until pass 2 adds the global offset.
// ---------------------------------------------------------------------------
constexpr int kUnionThreads = 512;
constexpr int kMaxWords = kMaxC / 32;

// The union of one unit's n_q selection rows (row j at selb + j * jstride,
// device or shared memory) and its residency lookup; `qbits` (n_q * W words)
// and `missw` (W words) are shared scratch.  All threads of the CTA.
__device__ __forceinline__ void union_unit(const int32_t *selb, int64_t jstride, int unit, int n_q, int k, int C,
                                           int umax, int64_t hot_slots, const int32_t *__restrict__ resident_slot,
                                           int32_t *__restrict__ union_idx, int32_t *__restrict__ union_slot,
                                           uint8_t *__restrict__ union_qmask, int32_t *__restrict__ union_cnt,
                                           int32_t *__restrict__ unit_miss, uint32_t *qbits, uint32_t *missw,
                                           int *scratch, int32_t *status) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int W = (C + 31) >> 5;
  for (int i = tid; i < n_q * W; i += nt) qbits[i] = 0u;
  __syncthreads();
  for (int i = tid; i < n_q * k; i += nt) {
    const int j = i / k, r = i - j * k;
    const int c = selb[j * jstride + r];
    if (c == -1) continue;   // padding of a row shorter than k (coverage budgets)
    if (c < 0 || c >= C) {
      set_status(status, DD_ERR_DEVICE_CHECK);
      continue;
    }
    atomicOr(&qbits[j * W + (c >> 5)], 1u << (c & 31));
  }
  __syncthreads();

  const int per = (W + nt - 1) / nt;
  const int w0 = min(W, tid * per), w1 = min(W, w0 + per);
  const int32_t *rs_unit = resident_slot + (int64_t)unit * C;
  int cnt_u = 0, cnt_m = 0;
  for (int w = w0; w < w1; ++w) {
    uint32_t ub = 0;
    for (int j = 0; j < n_q; ++j) ub |= qbits[j * W + w];
    uint32_t mb = 0, rest = ub;
    while (rest) {
      const int bit = __ffs(rest) - 1;
      rest &= rest - 1;
      const int32_t rs = rs_unit[w * 32 + bit];
      if (rs >= hot_slots) set_status(status, DD_ERR_DEVICE_CHECK);
      if (rs < 0 || rs >= hot_slots) mb |= 1u << bit;
    }
    missw[w] = mb;
    cnt_u += __popc(ub);
    cnt_m += __popc(mb);
  }
  int total;
  const int excl = block_excl_scan((cnt_u << 16) | cnt_m, scratch, &total);
  int upos = excl >> 16, mpos = excl & 0xFFFF;
  const int64_t ubase = (int64_t)unit * umax;
  for (int w = w0; w < w1; ++w) {
    uint32_t ub = 0;
    for (int j = 0; j < n_q; ++j) ub |= qbits[j * W + w];
    const uint32_t mb = missw[w];
    while (ub) {
      const int bit = __ffs(ub) - 1;
      ub &= ub - 1;
      const int c = w * 32 + bit;
      uint32_t qm = 0;
      for (int j = 0; j < n_q; ++j) qm |= ((qbits[j * W + w] >> bit) & 1u) << j;
      union_idx[ubase + upos] = c;
      union_qmask[ubase + upos] = (uint8_t)qm;
      if ((mb >> bit) & 1u) {
        union_slot[ubase + upos] = -(mpos + 1);
        ++mpos;
      } else {
        union_slot[ubase + upos] = rs_unit[c];
      }
      ++upos;
    }
  }
  if (tid == 0) {
    union_cnt[unit] = total >> 16;
    unit_miss[unit] = total & 0xFFFF;
  }
}

__global__ void __launch_bounds__(kUnionThreads) k_union(
    const int32_t *__restrict__ sel, const int32_t *__restrict__ resident_slot, int32_t *__restrict__ union_idx,
    int32_t *__restrict__ union_slot, uint8_t *__restrict__ union_qmask, int32_t *__restrict__ union_cnt,
    int32_t *__restrict__ unit_miss, int n_q, int sel_rows, int Hkv, int k, int C, int umax, int64_t hot_slots,
    int32_t *status) {
  __shared__ uint32_t qbits[kMaxNq * kMaxWords];
  __shared__ uint32_t missw[kMaxWords];
  __shared__ int scratch[33];
  pdl_wait();
  pdl_trigger();
  const int unit = blockIdx.x;
  const int b = unit / Hkv, g = unit - b * Hkv;
  union_unit(sel + ((int64_t)b * sel_rows * Hkv + g) * k, (int64_t)Hkv * k, unit, n_q, k, C, umax, hot_slots,
             resident_slot, union_idx, union_slot, union_qmask, union_cnt, unit_miss, qbits, missw, scratch, status);
}

cudaError_t launch_union(const int32_t *sel, const int32_t *resident_slot, int32_t *union_idx, int32_t *union_slot,
                         uint8_t *union_qmask, int32_t *union_cnt, int32_t *unit_miss, int units, int n_q, int Hkv,
                         int k, int C, int umax, int64_t hot_slots, int32_t *status, cudaStream_t s, int sel_rows) {
  if (units == 0) return cudaSuccess;
  return launch_k(k_union, dim3(units), dim3(kUnionThreads), 0, s, sel, resident_slot, union_idx, union_slot,
                  union_qmask, union_cnt, unit_miss, n_q, sel_rows > 0 ? sel_rows : n_q, Hkv, k, C, umax, hot_slots,
                  status);
}

// ---------------------------------------------------------------------------
// The selection of a step after scoring, in one kernel, one CTA (512
// threads) per (b,g) unit, when a unit's n_q score rows fit in shared memory:
//  a2  the unit's score rows (just written by the scoring kernel, so read
//      from L2) become order keys in shared memory; the top-k of every row
//      comes from one radix select over all rows at once (per-row
//      histograms, warp j settles row j);
//  a3  the union and residency lookup read the selections from shared
//      memory; the global miss ordinals and union offsets (sums over the
//      earlier units) come from a look-back: each CTA takes its unit from a
//      ticket counter, so it only ever waits for units whose CTAs are
//      already running, publishes its union and miss counts, and sums the
//      counts of all earlier units as they are published; every wait is
//      bounded (DD_ERR_TIMEOUT).  The CTA then writes its union lists with
//      global slots, its miss-list entries and its part of the attention
//      plan; the last unit writes the totals.
// Selections and per-entry slots go to device memory only when asked for.
// ---------------------------------------------------------------------------
constexpr int kFusedThreads = 512;

constexpr int kLookBatch = 8;   // look-back words per lane in flight (256 units per round)
constexpr int kPrefStride = 16;  // 64-bit words between two units' offset pairs: a 128-byte line each

// fetch-and-add at GPU scope with no ordering: the words it counts carry
// their launch's epoch, so a reader re-polls a word it sees too early instead
// of every writer paying for a GPU-wide fence
__device__ __forceinline__ int atom_add_relaxed(int32_t *p, int v) {
  int r;
  asm volatile("atom.relaxed.gpu.global.add.s32 %0, [%1], %2;" : "=r"(r) : "l"(p), "r"(v) : "memory");
  return r;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

constexpr size_t kSelectMaxSmem = 216 * 1024;   // dynamic shared memory (beside the static ~8 KB)

// dynamic shared memory of the fused kernel: [union scratch, (NQ + 4) words
// per 32 chunks][keys, NQ*C][selections, NQ*k]; 0 when it does not fit
size_t fused_select_smem(int n_q, int C, int k) {
  const size_t W = (size_t)(C + 31) / 32;
  const size_t bytes = ((size_t)n_q + 4) * W * 4 + (size_t)n_q * C * 4 + (size_t)n_q * k * 4;
  return bytes <= kSelectMaxSmem ? bytes : 0;
}

// No two of the kernel's CTAs should share an SM while there are SMs enough
// for one unit each: a CTA that shares one runs at part speed, and every later
// unit waits for it in the look-back.  Behind the tensor-core scoring, which
// holds one CTA and ~198 KB of shared memory on every SM, a CTA of up to
// kSelectCoSmem bytes launched early fits beside it once per SM and no
// twice: it then waits at its dependency wait, already resident, and starts
// the moment the scores are in.  Otherwise (larger rows, or behind the
// min/max scoring) it asks for kSelectMinSmem, one CTA per SM.  With more
// units than SMs, two CTAs per SM (kSelectMinSmem2 each) run all units in one
// wave instead of two.
constexpr size_t kSelectMinSmem = 120 * 1024;
constexpr size_t kSelectMinSmem2 = 100 * 1024;
constexpr size_t kSelectCoSmem = 20 * 1024;

// ---------------------------------------------------------------------------
// Scoring folded into the selection, on the tensor cores (mean landmarks;
// taken when the units fill most SMs in one wave, one CTA per SM).  The CTA
// streams its own unit's C landmark rows through a ring of 128-row tiles (two
// 2-D TMA boxes a tile, the first stages requested before the dependency
// wait) and scores them as a product with the unit's n_q group-summed
// queries, each fp32 group sum split into three bf16 parts (hi + mid + lo
// equals it exactly, so each part's product is exact in fp32 and the three
// add up to the fp32 dot product within fp32 accumulation): M = 128
// landmarks, N = 3 n_q rounded up to 16, K = 128, fp32 accumulators in
// tensor memory (two buffers).  Warps 0-3 read their lane (one landmark) and
// write the order keys straight into the key rows; warp 4 issues the tile
// copies, warp 5 the MMAs, warps 6-15 build the query tile.  The kernel
// boundary, the round trip of the score rows through L2 and the rows' load
// disappear from the step; the selection then runs as below.
// ---------------------------------------------------------------------------
constexpr int kFsRows = 128;                 // landmark rows per tile (M)
constexpr int kFsHalf = kFsRows * 128;       // a 64-column half of a tile, 16 KiB
constexpr int kFsTile = 2 * kFsHalf;         // 32 KiB
constexpr int kFsMaxStages = 5;
constexpr int kFsQHalf = 32 * 128;           // a 64-column half of the query tile (3 n_q <= 24 rows, 32 kept)
constexpr int kFsTmemCols = 64;              // two accumulators of up to 32 columns

// where the kernel with scoring folded in keeps its parts: the key rows,
// selections and the unit's residency row, then (1024-aligned) the query tile
// and the ring, which the selection's union scratch reuses once the scores
// are in
__host__ __device__ inline size_t fs_head_bytes(int nq, int C, int k) {
  return (((size_t)nq * C + (size_t)nq * k + (size_t)C) * 4 + 1023) & ~(size_t)1023;   // + the residency row
}
size_t score_select_tc_smem(int n_q, int C, int k, int stages) {
  const size_t W = (size_t)(C + 31) / 32;
  const size_t tail = std::max((size_t)2 * kFsQHalf + (size_t)stages * kFsTile, ((size_t)n_q + 4) * W * 4);
  return 1024 + fs_head_bytes(n_q, C, k) + tail;   // + the alignment of the dynamic base
}

// bf16 of x rounded to nearest even, and its value as a float
__device__ __forceinline__ uint16_t bf16_rn_bits(float x) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
  return h;
}

// Besides the key rows, the epilogue warps take the segment maxima of the
// selection's lower bound as the keys go by (segments of S chunks: lanes of a
// warp hold 32 consecutive chunks) into s_lo / s_hi, and warps 6-15, once the
// query tile is built, load the unit's residency row into rs_all.
template <int NQ>
__device__ __forceinline__ void fused_tc_score(const SelectOut &o, int unit, int b, int g, uint32_t *keys,
                                               uint8_t *qtile, uint8_t *ring, uint64_t *bars, uint32_t tmem,
                                               int n_stages, int S, uint32_t *s_lo, uint32_t *s_hi,
                                               int32_t *rs_all) {
  constexpr int NB = 3 * NQ;                           // B rows: the hi, mid, lo parts of each query's sum
  constexpr int NQP = NB <= 16 ? 16 : 32;              // N of the MMA
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = o.C, Hq = o.Hq, Hkv = o.Hkv, G = Hq / Hkv;
  const int nt = (C + kFsRows - 1) / kFsRows;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kFsMaxStages);
  const uint32_t afull0 = smem_u32(bars + 2 * kFsMaxStages), aempty0 = smem_u32(bars + 2 * kFsMaxStages + 2);
  const uint32_t mmadone = smem_u32(bars + 2 * kFsMaxStages + 4);
  const int row_base = unit * C;
  const int pre = nt < n_stages ? nt : n_stages;
  if (warp == 4 && lane == 0) {
    // the landmarks are not written by the kernels this one may overlap: the
    // first stages go out before the dependency wait (bytes expected now,
    // the arrivals after it)
    for (int s = 0; s < pre; ++s) {
      const uint32_t bar = full0 + 8 * s, dst = smem_u32(ring + s * kFsTile);
      mbar_expect_tx(bar, (uint32_t)kFsTile);
      tma_load_2d(dst, &o.tm_lm, 0, row_base + s * kFsRows, bar);
      tma_load_2d(dst + kFsHalf, &o.tm_lm, 64, row_base + s * kFsRows, bar);
    }
  }
  pdl_wait();
  pdl_trigger();
  if (o.trace_score && tid == 0) trace_start(o.trace_score);
  if (warp >= 6) {
    // ------------------------------------------------ the query tile (B)
    // row 3j + p: part p of query j's fp32 group sum (heads in order);
    // column i at the 128-byte-swizzled place of a K-major tile
    for (int e = tid - 192; e < NQP * 128; e += kFusedThreads - 192) {
      const int r = e >> 7, i = e & 127;
      uint16_t v = 0;
      if (r < NB) {
        const int j = r / 3, part = r - 3 * j;
        float sum = 0.f;
        for (int h = g * G; h < (g + 1) * G; ++h)
          sum += __uint_as_float((uint32_t)o.q16[((int64_t)(b * NQ + j) * Hq + h) * 128 + i] << 16);
        const uint16_t hi = bf16_rn_bits(sum);
        const float r1 = sum - __uint_as_float((uint32_t)hi << 16);
        const uint16_t mid = bf16_rn_bits(r1);
        const float r2 = r1 - __uint_as_float((uint32_t)mid << 16);
        v = part == 0 ? hi : (part == 1 ? mid : bf16_rn_bits(r2));
      }
      const int half = i >> 6, cc = i & 63;
      *reinterpret_cast<uint16_t *>(qtile + half * kFsQHalf + r * 128 + ((((cc >> 3) ^ (r & 7))) << 4) + (cc & 7) * 2) = v;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("bar.arrive 3, %0;" ::"r"(kFusedThreads - 160) : "memory");   // warps 5-15
    const int32_t *rs_unit = o.resident_slot + (int64_t)unit * C;
    for (int c = tid - 192; c < C; c += kFusedThreads - 192) rs_all[c] = rs_unit[c];
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA
    asm volatile("bar.sync 3, %0;" ::"r"(kFusedThreads - 160) : "memory");   // the query tile is written
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kFsRows, NQP, 0, 0), qb = smem_u32(qtile);
      for (int s = 0; s < nt; ++s) {
        const int slot = s % n_stages, buf = s & 1;
        if (!mbar_wait(full0 + 8 * slot, (s / n_stages) & 1, o.status)) break;
        if (s >= 2 && !mbar_wait(aempty0 + 8 * buf, ((s >> 1) - 1) & 1, o.status)) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(ring + slot * kFsTile);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc_mma(tmem + buf * 32, smem_desc_sw128(a0 + (ks >> 2) * kFsHalf + (ks & 3) * 32, 16, 1024),
                 smem_desc_sw128(qb + (ks >> 2) * kFsQHalf + (ks & 3) * 32, 16, 1024), idesc, ks > 0);
        tc_commit(empty0 + 8 * slot);
        tc_commit(afull0 + 8 * buf);
      }
      tc_commit(mmadone);
      mbar_wait(mmadone, 0, o.status);
    }
    __syncwarp();
  } else if (warp == 4) {
    // ------------------------------------------------------- tile copies
    if (lane == 0)
      for (int s = 0; s < nt; ++s) {
        const int slot = s % n_stages;
        if (s >= n_stages && !mbar_wait(empty0 + 8 * slot, ((s / n_stages) - 1) & 1, o.status)) break;
        const uint32_t bar = full0 + 8 * slot;
        if (s < pre) {
          mbar_arrive(bar);
        } else {
          const uint32_t dst = smem_u32(ring + slot * kFsTile);
          mbar_arrive_expect_tx(bar, (uint32_t)kFsTile);
          tma_load_2d(dst, &o.tm_lm, 0, row_base + s * kFsRows, bar);
          tma_load_2d(dst + kFsHalf, &o.tm_lm, 64, row_base + s * kFsRows, bar);
        }
      }
  } else {
    // ---------------------------------------------- epilogue, warps 0-3
    const int row = 32 * warp + lane;   // this thread's tensor-memory lane: landmark row of a tile
    uint32_t mn[NQ], mx[NQ];            // over the segments this lane leads
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      mn[j] = 0xFFFFFFFFu;
      mx[j] = 0u;
    }
    for (int s = 0; s < nt; ++s) {
      const int buf = s & 1;
      if (!mbar_wait(afull0 + 8 * buf, (s >> 1) & 1, o.status)) break;
      tc_fence_after();
      float v[NQP];
#pragma unroll
      for (int c = 0; c < NQP / 16; ++c) tmem_ld32x32b_x16(tmem + ((uint32_t)(32 * warp) << 16) + buf * 32 + 16 * c, v + 16 * c);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(aempty0 + 8 * buf);
      const int c = s * kFsRows + row;
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        const float sc = (v[3 * j] + v[3 * j + 1]) + v[3 * j + 2];
        const uint32_t key = c < C ? order_key(sc) : 0u;
        if (c < C) {
          keys[j * C + c] = key;
          if (o.scores_out) o.scores_out[((int64_t)(b * NQ + j) * Hkv + g) * C + c] = sc;
        }
        uint32_t m = key;
        for (int off = 1; off < S; off <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
        if ((lane & (S - 1)) == 0 && c < C) {
          mn[j] = min(mn[j], m);
          mx[j] = max(mx[j], m);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        mn[j] = min(mn[j], __shfl_xor_sync(0xffffffffu, mn[j], off));
        mx[j] = max(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], off));
      }
      if (lane == 0 && mx[j] >= mn[j]) {   // the warp led at least one segment
        atomicMin(&s_lo[j], mn[j]);
        atomicMax(&s_hi[j], mx[j]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();   // every key row is in place; the tensor memory is no longer read
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kFsTmemCols) : "memory");
  }
  if (o.trace_score && tid == 0) trace_end(o.trace_score);
}

template <int NQ, bool kScore>
__global__ void __launch_bounds__(kFusedThreads, kScore ? 1 : 2)
    k_select_fused(const __grid_constant__ SelectOut o, int n_stages) {
  extern __shared__ __align__(128) unsigned char fsm_raw[];
  __shared__ int hist[NQ][256];
  __shared__ int scratch[33];
  __shared__ int s_unit, s_uoff, s_moff, s_last;
  __shared__ uint32_t s_epoch;
  __shared__ __align__(8) uint64_t s_bars[2 * kFsMaxStages + 5];   // scoring folded in: full, empty, acc full/empty, done
  __shared__ uint32_t s_tmem;
  // With the scoring folded in, the ticket and the first landmark stages come
  // before the dependency wait (the selection launched two kernels earlier
  // has finished: the kernel in between waited for it before it released
  // this one, so the counters are reset); everything it writes comes after.
  if (!kScore) {
    pdl_wait();
    pdl_trigger();
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    if (o.trace && !kScore) trace_start(o.trace);
    s_unit = atomicAdd(o.ticket, 1);                       // units in the order their CTAs start
    // this launch's look-back epoch; the previous launch's last CTA advanced it
    s_epoch = *reinterpret_cast<volatile uint32_t *>(o.ticket + 2);
    if (kScore) {
      for (int i = 0; i < 2 * kFsMaxStages + 5; ++i)
        mbar_init(smem_u32(&s_bars[i]), i == 2 * kFsMaxStages + 2 || i == 2 * kFsMaxStages + 3 ? 4 : 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  }
  if (kScore && warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "r"(kFsTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (kScore) tc_fence_before();
  __syncthreads();
  if (kScore) tc_fence_after();
  const int unit = s_unit;
  const uint32_t epoch = s_epoch;
  const int C = o.C, k = o.k, Hkv = o.Hkv;
  const int b = unit / Hkv, g = unit - b * Hkv;
  const int W = (C + 31) >> 5;
  uint32_t *keys, *qbits;
  int32_t *sel_s;
  uint8_t *tail = nullptr;
  if (kScore) {
    uint8_t *base = fsm_raw + ((1024u - (smem_u32(fsm_raw) & 1023u)) & 1023u);
    keys = reinterpret_cast<uint32_t *>(base);                       // [NQ][C]
    sel_s = reinterpret_cast<int32_t *>(keys + NQ * C);              // [NQ][k]
    tail = base + fs_head_bytes(NQ, C, k);                           // query tile + ring, then the union scratch
    qbits = reinterpret_cast<uint32_t *>(tail);
  } else {
    qbits = reinterpret_cast<uint32_t *>(fsm_raw);                   // [NQ][W]
    keys = qbits + (NQ + 4) * W;
    sel_s = reinterpret_cast<int32_t *>(keys + NQ * C);
  }
  uint32_t *ubw = qbits + NQ * W, *mbw = ubw + W;
  int *upre = reinterpret_cast<int *>(mbw + W), *mpre = upre + W;

  // ---- a2: the top k of every row (score descending, lower chunk first among
  // equal scores), as one bitmap per row.  The row is split into at least k
  // aligned segments of S chunks (S a power of two, at most 32); the smallest
  // segment maximum t is a lower bound on the row's k-th largest key, since
  // every segment holds a key >= t.  Only keys >= t take part in a radix
  // select whose 8-bit digits are taken relative to the low end of the
  // current key range (first pass: [t, row maximum], digit width sized to
  // it), so the few keys left spread over the bins.  A pass ends the row when
  // the boundary bin holds exactly the keys still needed; after the last
  // digit the remaining ties go to the lowest chunks.
  // per row: the current key range [lo, lo + w], its digit shift, keys still needed
  __shared__ uint32_t s_lo[NQ], s_hi[NQ], s_w[NQ];
  __shared__ int s_shift[NQ], s_rem[NQ], s_state[NQ];   // state 0: running, 1: keys >= lo, 2: ties at lo
  int S = 32;
  while (S > 1 && (C + S - 1) / S < k) S >>= 1;
  if (tid < NQ) {
    s_lo[tid] = 0xFFFFFFFFu;
    s_hi[tid] = 0u;
  }
  __syncthreads();
  if (kScore) {
    fused_tc_score<NQ>(o, unit, b, g, keys, tail, tail + 2 * kFsQHalf, s_bars, s_tmem, n_stages, S, s_lo, s_hi,
                       sel_s + NQ * k);
    if (o.trace && tid == 0) trace_start(o.trace);
  }
  {
    // every row's scores of a 4 x 512-chunk slab in flight at once
    const float *rows = kScore ? nullptr : o.scores + ((int64_t)(b * NQ) * Hkv + g) * C;   // row j at + j * Hkv * C
    uint32_t mn[NQ], mx[NQ];   // over the segments this thread takes
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      mn[j] = 0xFFFFFFFFu;
      mx[j] = 0u;
    }
    if (!kScore)   // with the scoring folded in the key rows are written already
    for (int c0 = warp * 32; c0 < C; c0 += 4 * kFusedThreads) {   // warp-uniform
      float v[NQ][4];
#pragma unroll
      for (int j = 0; j < NQ; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = c0 + e * kFusedThreads + lane;
          v[j][e] = c < C ? rows[(int64_t)j * Hkv * C + c] : 0.f;
        }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = c0 + e * kFusedThreads + lane;
#pragma unroll
        for (int j = 0; j < NQ; ++j)
          if (c < C) keys[j * C + c] = order_key(v[j][e]);
      }
    }
    __syncthreads();
    // segment maxima from shared memory, one segment of S keys per thread and
    // row (independent loads instead of a shuffle chain per key; the read
    // order is rotated by the thread so that a warp's 32 segments hit
    // different banks); with the scoring folded in they were taken already
    const int nseg = kScore ? 0 : (C + S - 1) / S;
#pragma unroll
    for (int j = 0; j < NQ; ++j)
      for (int sg = tid; sg < nseg; sg += kFusedThreads) {
        const uint32_t *kr = keys + j * C + sg * S;
        uint32_t m = 0u;
        if (sg * S + S <= C) {
#pragma unroll 8
          for (int i = 0; i < S; ++i) m = max(m, kr[(i + tid) & (S - 1)]);
        } else {
          for (int i = 0; i < C - sg * S; ++i) m = max(m, kr[i]);
        }
        mn[j] = min(mn[j], m);
        mx[j] = max(mx[j], m);
      }
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        mn[j] = min(mn[j], __shfl_xor_sync(0xffffffffu, mn[j], off));
        mx[j] = max(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], off));
      }
      if (lane == 0 && mx[j] >= mn[j]) {   // the warp led at least one segment
        atomicMin(&s_lo[j], mn[j]);
        atomicMax(&s_hi[j], mx[j]);
      }
    }
  }
  __syncthreads();
  if (tid < NQ) {
    const uint32_t d = s_hi[tid] - s_lo[tid];
    s_w[tid] = d;
    s_shift[tid] = d ? max(0, 24 - __clz(d)) : 0;   // w >> shift < 256
    s_rem[tid] = k;
    s_state[tid] = 0;
  }
  for (int pass = 0; pass < 5; ++pass) {
    for (int i = tid; i < NQ * 256; i += kFusedThreads) (&hist[0][0])[i] = 0;
    __syncthreads();
    for (int j = 0; j < NQ; ++j) {
      if (s_state[j] != 0) continue;
      const uint32_t lo = s_lo[j], w = s_w[j];
      const int sh = s_shift[j];
      for (int c0 = tid; c0 < C; c0 += 4 * kFusedThreads) {   // four keys in flight
        uint32_t kk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) kk[e] = c0 + e * kFusedThreads < C ? keys[j * C + c0 + e * kFusedThreads] : 0u;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c0 + e * kFusedThreads < C && kk[e] >= lo && kk[e] - lo <= w) atomicAdd(&hist[j][(kk[e] - lo) >> sh], 1);
      }
    }
    __syncthreads();
    if (warp < NQ && s_state[warp] == 0) {
      // lane l owns bins 255-8l down to 248-8l (descending digit order)
      int cnt[8], sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cnt[e] = hist[warp][255 - 8 * lane - e];
        sum += cnt[e];
      }
      const int incl = warp_incl_scan(sum);
      const int rem = s_rem[warp];
      int above = incl - sum;
      if (above < rem && rem <= incl) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (above < rem && rem <= above + cnt[e]) {
            const int sh = s_shift[warp];
            const uint32_t lo = s_lo[warp] + ((uint32_t)(255 - 8 * lane - e) << sh);
            const int r = rem - above;
            s_lo[warp] = lo;
            s_rem[warp] = r;
            if (cnt[e] == r) {
              s_state[warp] = 1;
            } else if (sh == 0) {
              s_state[warp] = 2;
            } else {   // the boundary bin [lo, lo + 2^sh - 1] becomes the range
              const uint32_t w = (1u << sh) - 1u;
              s_w[warp] = w;
              s_shift[warp] = max(0, 24 - __clz(w));
            }
          }
          above += cnt[e];
        }
      }
    }
    __syncthreads();
    bool more = false;
#pragma unroll
    for (int j = 0; j < NQ; ++j) more |= s_state[j] == 0;
    if (!more) break;
  }
  // bitmaps: every warp builds whole 32-chunk words with a ballot; a row with
  // ties at its last key is walked in chunk order by warp 0
  for (int j = 0; j < NQ; ++j) {
    const uint32_t lo = s_lo[j];
    if (s_state[j] == 1) {
      for (int c0 = warp * 32; c0 < C; c0 += kFusedThreads) {
        const int c = c0 + lane;
        const unsigned w = __ballot_sync(0xffffffffu, c < C && keys[j * C + c] >= lo);
        if (lane == 0) qbits[j * W + (c0 >> 5)] = w;
      }
    } else if (warp == 0) {
      if (s_state[j] != 2 && lane == 0) set_status(o.status, DD_ERR_DEVICE_CHECK);
      const int rem = s_rem[j];
      int run = 0;
      for (int c0 = 0; c0 < C; c0 += 32) {
        const int c = c0 + lane;
        const uint32_t key = c < C ? keys[j * C + c] : 0u;
        const bool eq = c < C && key == lo;
        const unsigned be = __ballot_sync(0xffffffffu, eq);
        const bool take = key > lo || (eq && run + __popc(be & ((1u << lane) - 1u)) < rem);
        const unsigned w = __ballot_sync(0xffffffffu, c < C && take);
        if (lane == 0) qbits[j * W + (c0 >> 5)] = w;
        run += __popc(be);
      }
    }
  }
  __syncthreads();
  if (o.sel || o.attn_slot) {
    // the selections in ascending chunk order, from the bitmaps (row j has k bits)
    for (int j = 0; j < NQ; ++j) {
      const uint32_t w = tid < W ? qbits[j * W + tid] : 0u;
      int tot;
      int pos = block_excl_scan(__popc(w), scratch, &tot);
      uint32_t rest = w;
      while (rest) {
        const int bit = __ffs(rest) - 1;
        rest &= rest - 1;
        if (pos < k) sel_s[j * k + pos] = tid * 32 + bit;
        ++pos;
      }
      if (tid == 0 && tot != k) set_status(o.status, DD_ERR_DEVICE_CHECK);
    }
    __syncthreads();
  }
  if (o.sel) {
    for (int i = tid; i < NQ * k; i += kFusedThreads) {
      const int j = i / k, r = i - j * k;
      o.sel[((int64_t)(b * NQ + j) * Hkv + g) * k + r] = sel_s[i];
    }
  }

  // ---- a3: union words, then the residency of every union chunk (one
  // lookup per chunk, all of them in flight at once, kept in shared memory
  // where the keys were), then one union word per thread (W <= 512)
  // (with the scoring folded in the whole row is in shared memory already)
  const int32_t *rs_unit = kScore ? sel_s + NQ * k : o.resident_slot + (int64_t)unit * C;
  int32_t *rs_s = kScore ? sel_s + NQ * k : reinterpret_cast<int32_t *>(keys);   // [C], valid for union chunks
  if (tid < W) {
    uint32_t ub = 0;
#pragma unroll
    for (int j = 0; j < NQ; ++j) ub |= qbits[j * W + tid];
    ubw[tid] = ub;
    mbw[tid] = 0u;
  }
  __syncthreads();
  for (int c0 = tid; c0 < C; c0 += 4 * kFusedThreads) {
    int32_t rs[4];
    bool in[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = c0 + e * kFusedThreads;
      in[e] = c < C && ((ubw[c >> 5] >> (c & 31)) & 1u);
      rs[e] = in[e] ? rs_unit[c] : -1;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!in[e]) continue;
      const int c = c0 + e * kFusedThreads;
      rs_s[c] = rs[e];
      if (rs[e] >= o.hot_slots) set_status(o.status, DD_ERR_DEVICE_CHECK);
      if (rs[e] < 0 || rs[e] >= o.hot_slots) atomicOr(&mbw[c >> 5], 1u << (c & 31));
    }
  }
  __syncthreads();
  int cu = 0, cm = 0;
  if (tid < W) {
    cu = __popc(ubw[tid]);
    cm = __popc(mbw[tid]);
  }
  int tot;
  const int ex = block_excl_scan((cu << 16) | cm, scratch, &tot);   // unions never exceed C <= 16384
  if (tid < W) {
    upre[tid] = ex >> 16;
    mpre[tid] = ex & 0xFFFF;
  }
  const int U = tot >> 16, M = tot & 0xFFFF;

  // Every unit publishes one 64-bit word {epoch:30, union count:17, miss
  // count:17} as soon as it has its counts (counts never exceed C <= 16384,
  // and a single aligned 64-bit store is seen whole, so the word is its own
  // message).
  const unsigned long long my_word =
      ((unsigned long long)epoch << 34) | ((unsigned long long)U << 17) | (unsigned long long)M;
  if (o.lb_pref) {
    // Every unit's CTA is resident at once (the host checked the occupancy),
    // so each may wait for all of them: a CTA publishes its word and counts
    // itself in; the CTA that arrives last reads every word (re-polling one
    // not yet seen with this launch's epoch), sums the counts in unit order,
    // publishes every unit's union and miss offsets as words {epoch:32,
    // offset:32}, each unit's pair on a cache line of its own, and resets
    // the counters for the next launch; the others wait for their own pair.
    // One round trip per CTA on the shared lines, instead of a look-back load
    // of every earlier word by every CTA, which queued at the few L2 lines
    // holding the words.
    if (tid == 0) {
      st_relaxed_u64(&o.lb_word[unit], my_word);
      s_last = atom_add_relaxed(o.ticket + 1, 1) == o.units - 1;
    }
    __syncthreads();
    if (s_last) {
      if (warp == 0) {
        const unsigned long long tag = (unsigned long long)epoch << 32;
        bool ok = true;
        const uint64_t t0 = globaltimer_ns();
        int carry_u = 0, carry_m = 0;   // counts of the units before this batch of words
        for (int base = 0; base < o.units; base += 32 * kLookBatch) {
          unsigned long long w8[kLookBatch];
          int su = 0, sm = 0;
#pragma unroll
          for (int t = 0; t < kLookBatch; ++t) {   // lane l: units base + 8l .. base + 8l + 7
            const int idx = base + lane * kLookBatch + t;
            w8[t] = idx < o.units ? ld_relaxed_u64(&o.lb_word[idx]) : (unsigned long long)epoch << 34;
          }
#pragma unroll
          for (int t = 0; t < kLookBatch; ++t) {
            const int idx = base + lane * kLookBatch + t;
            if ((w8[t] >> 34) != epoch) w8[t] = wait_published(&o.lb_word[idx], epoch, t0, &ok);
            su += (int)((w8[t] >> 17) & 0x1FFFFull);
            sm += (int)(w8[t] & 0x1FFFFull);
          }
          if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) set_status(o.status, DD_ERR_TIMEOUT);
            break;
          }
          const int iu = warp_incl_scan(su), im = warp_incl_scan(sm);
          int eu = carry_u + iu - su, em = carry_m + im - sm;
#pragma unroll
          for (int t = 0; t < kLookBatch; ++t) {
            const int idx = base + lane * kLookBatch + t;
            if (idx < o.units) {
              st_relaxed_u64(&o.lb_pref[(int64_t)idx * kPrefStride], tag | (uint32_t)eu);
              st_relaxed_u64(&o.lb_pref[(int64_t)idx * kPrefStride + 1], tag | (uint32_t)em);
              if (idx == unit) {
                s_uoff = eu;
                s_moff = em;
              }
            }
            eu += (int)((w8[t] >> 17) & 0x1FFFFull);
            em += (int)(w8[t] & 0x1FFFFull);
          }
          carry_u += __shfl_sync(0xffffffffu, iu, 31);
          carry_m += __shfl_sync(0xffffffffu, im, 31);
        }
        if (lane == 0) {   // every CTA has taken its ticket, read the epoch and arrived
          const uint32_t next = (epoch + 1u) & 0x3FFFFFFFu;
          o.ticket[0] = 0;
          o.ticket[1] = 0;
          o.ticket[2] = (int32_t)(next == 0u ? 1u : next);
        }
      }
    } else if (tid == 0) {
      const uint64_t t0 = globaltimer_ns();
      unsigned long long wu = 0, wm = 0;
      for (uint32_t it = 0;; ++it) {
        wu = ld_relaxed_u64(&o.lb_pref[(int64_t)unit * kPrefStride]);
        wm = ld_relaxed_u64(&o.lb_pref[(int64_t)unit * kPrefStride + 1]);
        if ((wu >> 32) == epoch && (wm >> 32) == epoch) break;
        if ((it & 63u) == 63u && globaltimer_ns() - t0 > 2000000000ull) {
          set_status(o.status, DD_ERR_TIMEOUT);
          break;
        }
      }
      s_uoff = (int)(uint32_t)wu;
      s_moff = (int)(uint32_t)wm;
    }
  } else if (warp == 0) {
    // look-back over the earlier units: sum all of the predecessors'
    // counts: each lane loads its strided share of their words at once and
    // re-polls only those not yet published; one round trip after the
    // slowest predecessor, no chain
    const unsigned long long ep = (unsigned long long)epoch << 34;
    if (lane == 0) st_relaxed_u64(&o.lb_word[unit], my_word);
    int su = 0, sm = 0;
    bool ok = true;
    const uint64_t t0 = globaltimer_ns();
    for (int base = 0; base < unit; base += 32 * kLookBatch) {
      unsigned long long w8[kLookBatch];
#pragma unroll
      for (int t = 0; t < kLookBatch; ++t) {
        const int idx = base + t * 32 + lane;
        w8[t] = idx < unit ? ld_relaxed_u64(&o.lb_word[idx]) : ep;
      }
#pragma unroll
      for (int t = 0; t < kLookBatch; ++t) {
        const int idx = base + t * 32 + lane;
        if ((w8[t] >> 34) != epoch) w8[t] = wait_published(&o.lb_word[idx], epoch, t0, &ok);
        su += (int)((w8[t] >> 17) & 0x1FFFFull);
        sm += (int)(w8[t] & 0x1FFFFull);
      }
      if (!__all_sync(0xffffffffu, ok)) break;
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
      su += __shfl_xor_sync(0xffffffffu, su, sh);
      sm += __shfl_xor_sync(0xffffffffu, sm, sh);
    }
    if (!__all_sync(0xffffffffu, ok) && lane == 0) set_status(o.status, DD_ERR_TIMEOUT);
    if (lane == 0) {
      s_uoff = su;
      s_moff = sm;
    }
  }
  // the lists that need no offset, while warp 0 finds the offsets: the
  // union's chunks and query masks, the resident chunks' slots
  const int64_t ubase = (int64_t)unit * o.umax;
  if (warp > 0) {
    for (int wi = tid - 32; wi < W; wi += kFusedThreads - 32) {
      uint32_t rest = ubw[wi];
      const uint32_t mb = mbw[wi];
      int up = upre[wi];
      while (rest) {
        const int bit = __ffs(rest) - 1;
        rest &= rest - 1;
        const int c = wi * 32 + bit;
        uint32_t qm = 0;
        for (int j = 0; j < NQ; ++j) qm |= ((qbits[j * W + wi] >> bit) & 1u) << j;
        o.union_idx[ubase + up] = c;
        o.union_qmask[ubase + up] = (uint8_t)qm;
        if (!((mb >> bit) & 1u)) o.union_slot[ubase + up] = rs_s[c];
        ++up;
      }
    }
    if (o.attn_slot) {
      for (int i = tid - 32; i < NQ * k; i += kFusedThreads - 32) {
        const int j = i / k, r = i - j * k, c = sel_s[i];
        const bool miss = c >= 0 && c < C && ((mbw[c >> 5] >> (c & 31)) & 1u);
        if (!miss) o.attn_slot[((int64_t)(b * NQ + j) * Hkv + g) * k + r] = c >= 0 && c < C ? rs_s[c] : INT32_MIN;
      }
    }
    if (tid == 32) {
      o.union_cnt[unit] = U;
      o.unit_miss[unit] = M;
      o.chunk_off[o.units + 1 + unit] = 0;   // arrival counter of the attention's fix-up
    }
  }
  __syncthreads();
  const int uoff = s_uoff, moff = s_moff;

  // the attention plan's entries and the misses' slots and list
  if (tid < W) {
    uint32_t rest = ubw[tid];
    const uint32_t mb = mbw[tid];
    int up = upre[tid], mp = mpre[tid];
    while (rest) {
      const int bit = __ffs(rest) - 1;
      rest &= rest - 1;
      const int c = tid * 32 + bit;
      uint32_t qm = 0;
      for (int j = 0; j < NQ; ++j) qm |= ((qbits[j * W + tid] >> bit) & 1u) << j;
      int32_t row, host = -1;
      if ((mb >> bit) & 1u) {
        const int64_t m = (int64_t)moff + mp++;
        o.union_slot[ubase + up] = -(int32_t)(m + 1);
        if (m < o.max_misses) {
          o.miss_list[m] = unit * C + c;
          row = -2 - (int32_t)(m * o.cs);
          host = unit * C + c;
        } else {
          row = -1;   // beyond the staging capacity: the last unit reports it
          qm = 0;
        }
      } else {
        row = rs_s[c] * o.cs;
      }
      o.flat[uoff + up] = make_int4(row, (int)qm, host, 0);
      ++up;
    }
  }
  if (o.attn_slot && M > 0) {
    for (int i = tid; i < NQ * k; i += kFusedThreads) {
      const int j = i / k, r = i - j * k, c = sel_s[i];
      if (c >= 0 && c < C && ((mbw[c >> 5] >> (c & 31)) & 1u)) {
        const int w = c >> 5;
        const uint32_t low = (1u << (c & 31)) - 1u;
        o.attn_slot[((int64_t)(b * NQ + j) * Hkv + g) * k + r] =
            -(int32_t)((int64_t)moff + mpre[w] + __popc(mbw[w] & low) + 1);
      }
    }
  }
  if (tid == 0) {
    o.chunk_off[unit] = uoff;
    if (unit == o.units - 1) {
      o.chunk_off[o.units] = uoff + U;
      *o.miss_count = moff + M;
      if ((int64_t)moff + M > o.max_misses) set_status(o.status, DD_ERR_CAPACITY);
    }
    // the last CTA to finish resets the ticket counters and advances the
    // epoch (30 bits, never 0: zeroed words carry epoch 0) for the next launch;
    // every CTA of this launch has read the epoch by then.  Kept on the device,
    // so replaying a captured step in a CUDA graph stays correct.  (With
    // every CTA resident, the last to arrive at the offsets did it.)
    if (!o.lb_pref) {
      __threadfence();
      if (atomicAdd(o.ticket + 1, 1) == o.units - 1) {
        uint32_t next = (epoch + 1u) & 0x3FFFFFFFu;
        o.ticket[0] = 0;
        o.ticket[1] = 0;
        o.ticket[2] = (int32_t)(next == 0u ? 1u : next);
        __threadfence();
      }
    }
  }
  if (o.trace) {
    __syncthreads();
    if (tid == 0) trace_end(o.trace);
  }
}

// Whether a grid of `units` CTAs of the kernel fits on the device at once
// (blocks per SM at this shared memory x SMs), cached per kernel and size.
static bool all_resident(const void *func, size_t smem, int units, int sm_count) {
  struct Entry {
    const void *func;
    size_t smem;
    int dev, per_sm;
  };
  static Entry cache[32];
  static int n_cache = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  int per_sm = -1;
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].func == func && cache[i].smem == smem && cache[i].dev == dev) per_sm = cache[i].per_sm;
  if (per_sm < 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, kFusedThreads, smem) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    if (n_cache < 32) cache[n_cache++] = Entry{func, smem, dev, per_sm};
  }
  return (int64_t)units <= (int64_t)per_sm * sm_count;
}

cudaError_t launch_select_fused(const SelectOut &o, int n_q, cudaStream_t s) {
  if (o.units == 0) return cudaSuccess;
  size_t smem = fused_select_smem(n_q, o.C, o.k);
  if (smem == 0) return cudaErrorInvalidValue;
  const size_t floor_bytes = o.units > o.sm_count ? kSelectMinSmem2 : kSelectMinSmem;
  if (!(o.units <= o.sm_count && o.after_tc_score && smem <= kSelectCoSmem) && smem < floor_bytes)
    smem = floor_bytes;
  switch (n_q) {
#define DD_FUSED_CASE(N)                                                                                      \
  case N: {                                                                                                    \
    cudaError_t e = set_dyn_smem((const void *)k_select_fused<N, false>, smem);                               \
    if (e != cudaSuccess) return e;                                                                            \
    SelectOut oo = o;                                                                                          \
    if (!all_resident((const void *)k_select_fused<N, false>, smem, o.units, o.sm_count)) oo.lb_pref = nullptr; \
    return launch_k(k_select_fused<N, false>, dim3(o.units), dim3(kFusedThreads), smem, s, oo, 0);            \
  }
    DD_FUSED_CASE(1) DD_FUSED_CASE(2) DD_FUSED_CASE(3) DD_FUSED_CASE(4)
    DD_FUSED_CASE(5) DD_FUSED_CASE(6) DD_FUSED_CASE(7) DD_FUSED_CASE(8)
#undef DD_FUSED_CASE
    default: return cudaErrorInvalidValue;
  }
}

// Folding the scoring in pays when one CTA per SM streams one unit and the
// units fill most SMs in one wave (3/4 of them or more): a unit's landmarks
// then stream at one SM's share of HBM, and the scoring kernel's boundary,
// the score rows' round trip and their load leave the step.  With fewer
// units the idle SMs' share of the bandwidth is lost, with more a second wave
// follows; the scoring kernel then streams over every SM instead.
int score_select_stages(int units, int sm_count, int n_q, int C, int k) {
  if (units > sm_count || 4 * units < 3 * sm_count) return 0;
  for (int st = kFsMaxStages; st >= 3; --st)
    if (score_select_tc_smem(n_q, C, k, st) <= kSelectMaxSmem) return st;
  return 0;
}

cudaError_t launch_score_select(const SelectOut &o, int n_q, int stages, cudaStream_t s) {
  if (o.units == 0) return cudaSuccess;
  if (stages < 1 || stages > kFsMaxStages) return cudaErrorInvalidValue;
  const size_t smem = score_select_tc_smem(n_q, o.C, o.k, stages);
  switch (n_q) {
#define DD_SS_CASE(N)                                                                                         \
  case N: {                                                                                                    \
    cudaError_t e = set_dyn_smem((const void *)k_select_fused<N, true>, smem);                                \
    if (e != cudaSuccess) return e;                                                                            \
    SelectOut oo = o;                                                                                          \
    if (!all_resident((const void *)k_select_fused<N, true>, smem, o.units, o.sm_count)) oo.lb_pref = nullptr; \
    return launch_k(k_select_fused<N, true>, dim3(o.units), dim3(kFusedThreads), smem, s, oo, stages);        \
  }
    DD_SS_CASE(1) DD_SS_CASE(2) DD_SS_CASE(3) DD_SS_CASE(4)
    DD_SS_CASE(5) DD_SS_CASE(6) DD_SS_CASE(7) DD_SS_CASE(8)
#undef DD_SS_CASE
    default: return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------------------
// a3, pass 2 (one CTA per (b,g)): global miss ordinals = misses of all
// earlier (b,g) units + the local ordinal, written to the miss list and the
// union slots; then every selection entry looks up its encoded slot.
// ---------------------------------------------------------------------------
constexpr int kAssignThreads = 256;

__global__ void __launch_bounds__(kAssignThreads) k_assign(
    const int32_t *__restrict__ sel, const int32_t *__restrict__ union_idx, int32_t *__restrict__ union_slot,
    const uint8_t *__restrict__ union_qmask, const int32_t *__restrict__ union_cnt,
    const int32_t *__restrict__ unit_miss, int32_t *__restrict__ miss_list, int32_t *__restrict__ miss_count,
    int32_t *__restrict__ attn_slot, int units, int n_q, int Hkv, int k, int C, int umax, int64_t max_misses,
    int64_t hot_slots, int cs, AttnPlanOut po, int with_plan, int32_t *status) {
  __shared__ int scratch[33];
  pdl_wait();
  pdl_trigger();
  const int unit = blockIdx.x;
  const int b = unit / Hkv, g = unit - b * Hkv;
  const int tid = threadIdx.x;
  // misses and union sizes of the earlier units, and of all units
  int before_m = 0, all_m = 0, before_c = 0, all_c = 0;
  for (int u = tid; u < units; u += kAssignThreads) {
    const int m = unit_miss[u], c = union_cnt[u];
    all_m += m;
    all_c += c;
    if (u < unit) {
      before_m += m;
      before_c += c;
    }
  }
  const int offset = block_sum(before_m, scratch);
  const int total_m = block_sum(all_m, scratch);
  const int off_c = with_plan ? block_sum(before_c, scratch) : 0;
  const int total_c = with_plan ? block_sum(all_c, scratch) : 0;

  const int cnt = union_cnt[unit];
  const int64_t ubase = (int64_t)unit * umax;
  bool over = false;
  for (int u = tid; u < cnt; u += kAssignThreads) {
    const int32_t s = union_slot[ubase + u];
    if (s < 0) {
      const int64_t m = (int64_t)offset + (-(int64_t)s - 1);
      if (m < max_misses) miss_list[m] = unit * C + union_idx[ubase + u];
      else over = true;
      union_slot[ubase + u] = (int32_t)(-(m + 1));
    }
  }
  if (over) set_status(status, DD_ERR_CAPACITY);
  if (unit == units - 1 && tid == 0) *miss_count = total_m;
  __syncthreads();
  if (with_plan)
    attn_plan_unit(po, unit, units, off_c, cnt, total_c, union_slot + ubase, union_qmask + ubase, union_idx + ubase,
                   C, min((int64_t)total_m, max_misses), hot_slots, cs, status);
  if (attn_slot == nullptr) return;
  for (int i = tid; i < n_q * k; i += kAssignThreads) {
    const int j = i / k, r = i - j * k;
    const int64_t si = ((int64_t)(b * n_q + j) * Hkv + g) * k + r;
    const int c = sel[si];
    int lo = 0, hi = cnt - 1, found = -1;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      const int v = union_idx[ubase + mid];
      if (v == c) { found = mid; break; }
      if (v < c) lo = mid + 1; else hi = mid - 1;
    }
    attn_slot[si] = found >= 0 ? union_slot[ubase + found] : INT32_MIN;
  }
}

cudaError_t launch_assign(const int32_t *sel, const int32_t *union_idx, int32_t *union_slot,
                          const uint8_t *union_qmask, const int32_t *union_cnt, const int32_t *unit_miss,
                          int32_t *miss_list, int32_t *miss_count, int32_t *attn_slot, int units, int n_q, int Hkv,
                          int k, int C, int umax, int64_t max_misses, int64_t hot_slots, int cs,
                          const AttnPlanOut *plan, int32_t *status, cudaStream_t s) {
  if (units == 0) return cudaSuccess;
  AttnPlanOut po = {};
  if (plan) po = *plan;
  return launch_k(k_assign, dim3(units), dim3(kAssignThreads), 0, s, sel, union_idx, union_slot, union_qmask,
                  union_cnt, unit_miss, miss_list, miss_count, attn_slot, units, n_q, Hkv, k, C, umax, max_misses,
                  hot_slots, cs, po, plan ? 1 : 0, status);
}

}  // namespace dd
