// Residency update of the per-(request, KV head) hot pools after a step.
//
// OasisKV summary, Methodology (delta selection and capped eviction): chunks
// of the selection that are already resident cost no traffic; resident
// chunks outside the selection are ranked by the step they were last
// selected in; every admitted non-resident chunk is paired with one eviction
// target, least recently used first; at most `cap` pairs per step and KV
// head, which bounds the transfer to cap * H chunk entries.  Adaptive
// DHiSparse Fig. 3 (3): promoted rows are copied from the staging arena into
// the hot cache.
//
// One CTA per unit u = b*Hkv + g, owning pool slots u*S .. u*S+S-1:
//   1. resident chunks of the union: last_used = step (never evicted);
//   2. targets = free slots (slot_chunk < 0) by slot, then the other
//      resident slots by (last_used, slot) -- one bitonic sort of 64-bit
//      keys {class, last_used, slot} in shared memory;
//   3. the union's missing chunks, in ascending chunk order, take the first
//      A = min(cap, misses, targets) targets in order; for each pair the old
//      chunk leaves the map, the new one enters it, and its K/V rows are
//      copied from staging slot m (union_slot = -(m+1)) into the pool slot.
#include "dd_common.cuh"

namespace dd {

constexpr int kResThreads = 512;
constexpr int kMaxSlotsPerUnit = 4096;

__global__ void __launch_bounds__(kResThreads) k_update_residency(
    int32_t step, int32_t cap, int S, const int32_t *__restrict__ union_idx, const int32_t *__restrict__ union_slot,
    const int32_t *__restrict__ union_cnt, const int32_t *__restrict__ miss_count, int64_t max_misses,
    const uint4 *__restrict__ Kst, const uint4 *__restrict__ Vst, int32_t *__restrict__ resident_slot,
    int32_t *__restrict__ slot_chunk, int32_t *__restrict__ last_used, uint4 *__restrict__ Khot,
    uint4 *__restrict__ Vhot, int32_t *__restrict__ admitted, int C, int umax, int cs, int32_t *status) {
  __shared__ unsigned long long keys[kMaxSlotsPerUnit];
  __shared__ uint8_t in_union[kMaxSlotsPerUnit];
  __shared__ int scratch[33];
  pdl_wait();
  pdl_trigger();
  if (load_status(status) != 0) return;
  const int u = blockIdx.x, tid = threadIdx.x;
  const int64_t base = (int64_t)u * S;
  int32_t *sc = slot_chunk + base;
  int32_t *lu = last_used + base;
  int32_t *rs = resident_slot + (int64_t)u * C;
  const int32_t *ui = union_idx + (int64_t)u * umax;
  const int32_t *us = union_slot + (int64_t)u * umax;
  const int U = min(max(union_cnt[u], 0), umax);
  const int64_t m_valid = min((int64_t)*miss_count, max_misses);

  for (int t = tid; t < S; t += kResThreads) in_union[t] = 0;
  __syncthreads();
  // 1. union residents: refreshed and protected; count the misses
  int my_miss = 0;
  for (int i = tid; i < U; i += kResThreads) {
    const int32_t sl = us[i];
    if (sl >= 0) {
      const int64_t t = sl - base;
      if (t < 0 || t >= S) {
        set_status(status, DD_ERR_DEVICE_CHECK);
        continue;
      }
      in_union[t] = 1;
      lu[t] = step;
    } else {
      ++my_miss;
    }
  }
  const int n_miss = block_sum(my_miss, scratch);   // ends with a barrier: in_union complete

  // 2. eviction keys, sorted ascending: class 0 free, 1 evictable (by last_used), 2 protected
  int n_pow = 1;
  while (n_pow < S) n_pow <<= 1;
  int my_targets = 0;
  for (int t = tid; t < n_pow; t += kResThreads) {
    unsigned long long key = ~0ull;
    if (t < S) {
      const int32_t c = sc[t];
      const unsigned long long cls = in_union[t] ? 2ull : (c < 0 ? 0ull : 1ull);
      const unsigned long long age = cls == 1 ? (unsigned long long)((uint32_t)lu[t] ^ 0x80000000u) : 0ull;
      key = (cls << 62) | (age << 16) | (unsigned long long)t;
      my_targets += cls < 2;
    }
    keys[t] = key;
  }
  const int n_targets = block_sum(my_targets, scratch);
  for (int k = 2; k <= n_pow; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < n_pow; i += kResThreads) {
        const int x = i ^ j;
        if (x > i) {
          const unsigned long long a = keys[i], b = keys[x];
          if ((a > b) == ((i & k) == 0)) {
            keys[i] = b;
            keys[x] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  const int A = max(0, min(min(cap, n_miss), n_targets));

  // 3. the r-th missing chunk of the union (ascending chunk order) takes target r
  int carry = 0;   // misses in the earlier batches
  for (int i0 = 0; i0 < U; i0 += kResThreads) {
    const int i = i0 + tid;
    const bool miss = i < U && us[i] < 0;
    int tot;
    const int rank = carry + block_excl_scan(miss ? 1 : 0, scratch, &tot);
    carry += tot;
    if (miss && rank < A) {
      const int t = (int)(keys[rank] & 0xFFFFull);
      const int32_t c = ui[i];
      const int64_t m = -(int64_t)us[i] - 1;
      if (c < 0 || c >= C || m >= m_valid) {
        set_status(status, DD_ERR_DEVICE_CHECK);
        continue;
      }
      const int32_t old = sc[t];
      if (old >= 0 && old < C) rs[old] = -1;
      rs[c] = (int32_t)(base + t);
      sc[t] = c;
      lu[t] = step;
    }
  }
  if (tid == 0 && admitted) admitted[u] = A;
  __syncthreads();

  // copy the admitted chunks' K and V rows from staging into their pool slots;
  // every thread walks the union in the same order to find pair r
  const int vec = cs * kVecPerRow;
  for (int i = 0, rank = 0; i < U && rank < A; ++i) {
    const int32_t sl = us[i];
    if (sl >= 0) continue;
    const int t = (int)(keys[rank] & 0xFFFFull);
    const int64_t m = -(int64_t)sl - 1;
    ++rank;
    if (m >= m_valid) continue;
    const uint4 *ks = Kst + m * vec, *vs = Vst + m * vec;
    uint4 *kd = Khot + (base + t) * vec, *vd = Vhot + (base + t) * vec;
    for (int e = tid; e < vec; e += kResThreads) {
      kd[e] = ks[e];
      vd[e] = vs[e];
    }
  }
}

cudaError_t launch_update_residency(int32_t step, int32_t cap, int S, int units, const int32_t *union_idx,
                                    const int32_t *union_slot, const int32_t *union_cnt, const int32_t *miss_count,
                                    int64_t max_misses, const uint4 *Kst, const uint4 *Vst, int32_t *resident_slot,
                                    int32_t *slot_chunk, int32_t *last_used, uint4 *Khot, uint4 *Vhot,
                                    int32_t *admitted, int C, int umax, int cs, int32_t *status, cudaStream_t s) {
  if (units == 0) return cudaSuccess;
  return launch_k(k_update_residency, dim3(units), dim3(kResThreads), 0, s, step, cap, S, union_idx, union_slot,
                  union_cnt, miss_count, max_misses, Kst, Vst, resident_slot, slot_chunk, last_used, Khot, Vhot,
                  admitted, C, umax, cs, status);
}

}  // namespace dd
