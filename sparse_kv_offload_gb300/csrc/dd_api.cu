// C ABI of libdd: context, argument checks, the per-stage entry points and
// the one-layer step with its two-buffer ping-pong (DualDecoder §5.4,
// Fig. 11: one staging buffer serves the current layer's attention while the
// other receives a later layer's chunks; CUDA events order the copy into a
// buffer after the attention that last read it, and the attention after the
// copy).
#include <math.h>
#include <string.h>

#include <vector>

#include "dd_tc.cuh"

struct dd_ctx {
  dd_dims dims;
  int C, G, NQ, umax, units, device, sm_count;
  int64_t max_misses, hot_slots;
  // device workspace
  void *ws = nullptr;
  int32_t *status = nullptr;
  float *scores = nullptr;
  int32_t *sel = nullptr, *union_idx = nullptr, *union_slot = nullptr, *union_cnt = nullptr;
  uint8_t *union_qmask = nullptr;
  int32_t *unit_miss = nullptr, *miss_list = nullptr, *miss_count = nullptr, *attn_slot = nullptr;
  float *part_o = nullptr, *part_ml = nullptr;
  int32_t *chunk_off = nullptr;
  int4 *flat = nullptr;
  unsigned long long *lb_word = nullptr;        // fused selection: look-back words, ticket
  unsigned long long *lb_pref = nullptr;        // fused selection: offsets by the last CTA
  unsigned long long *diag_word = nullptr;      // a word nothing publishes (bounded-wait self-test)
  int32_t *ticket = nullptr;
  void *dummy_pool = nullptr;
  dd::AttnPlan plan;
  // host side
  int32_t *h_miss = nullptr;          // pinned: [1 + max_misses]
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t released[2] = {nullptr, nullptr};   // attention finished reading staging buffer p
  cudaStream_t released_on[2] = {nullptr, nullptr};
  cudaEvent_t ready = nullptr;                    // miss list available to the copy stream / copies done
  bool used[2] = {false, false};
  int64_t launches = 0;
  // recent host -> device pointer translations for pinned host memory
  static constexpr int kViews = 16;
  const void *view_host[kViews] = {};
  const void *view_dev[kViews] = {};
  int view_next = 0;
};

namespace {

using dd::kD;

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

inline dd_status cuda_ok(cudaError_t e) {
  if (e == cudaSuccess) return DD_OK;
  g_last_cuda_error = e;
  return DD_ERR_CUDA;
}

#define DD_TRY(expr)                       \
  do {                                     \
    const dd_status _s = (expr);           \
    if (_s != DD_OK) return _s;            \
  } while (0)

#define DD_CUDA(expr) DD_TRY(cuda_ok(expr))

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dd_status check_dims(const dd_dims *d) {
  if (!d) return DD_ERR_INVALID_ARG;
  if (d->B < 0 || d->Hq <= 0 || d->Hkv <= 0 || d->Hq % d->Hkv) return DD_ERR_INVALID_ARG;
  if (d->d != kD) return DD_ERR_INVALID_ARG;
  if (d->cs != 16 && d->cs != 32 && d->cs != 64) return DD_ERR_INVALID_ARG;
  if (d->L <= 0 || d->L % d->cs) return DD_ERR_INVALID_ARG;
  const int C = d->L / d->cs;
  if (C > dd::kMaxC || d->k < 1 || d->k > C) return DD_ERR_INVALID_ARG;
  if (d->n_q < 1 || d->n_q > dd::kMaxNq) return DD_ERR_INVALID_ARG;
  if (d->n_q * (d->Hq / d->Hkv) > dd::kMaxNQV) return DD_ERR_INVALID_ARG;
  if ((int64_t)d->B * d->Hkv * C >= (int64_t(1) << 31)) return DD_ERR_INVALID_ARG;
  return DD_OK;
}

// Device-visible address of a K/V pointer: device memory as is, pinned host
// memory through its mapped device address.  Pageable memory is refused.
dd_status device_view(const void *p, const void **out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return DD_ERR_INVALID_ARG;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *out = p;
    return DD_OK;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    *out = a.devicePointer;
    return DD_OK;
  }
  return DD_ERR_INVALID_ARG;
}

// Device view of a pinned host pointer, from the context's small cache of
// recent translations (a decode loop cycles through a few layers' K and V).
dd_status cached_view(dd_ctx *c, const void *h, const void **d) {
  for (int i = 0; i < dd_ctx::kViews; ++i)
    if (c->view_host[i] == h && h != nullptr) {
      *d = c->view_dev[i];
      return DD_OK;
    }
  DD_TRY(device_view(h, d));
  c->view_host[c->view_next] = h;
  c->view_dev[c->view_next] = *d;
  c->view_next = (c->view_next + 1) % dd_ctx::kViews;
  return DD_OK;
}

dd_status host_kv_views(dd_ctx *c, const void *Kh, const void *Vh, const void **kd, const void **vd) {
  DD_TRY(cached_view(c, Kh, kd));
  return cached_view(c, Vh, vd);
}

// Landmark scoring of all n_q queries (mean or min/max landmarks), with the
// step's optional timing words.
dd_status score_impl(dd_ctx *c, const void *q, const void *lm, float *scores, bool minmax,
                     unsigned long long *trace, dd_stream_t stream) {
  if (!c) return DD_ERR_INVALID_ARG;
  if (c->units == 0) return DD_OK;
  if (!q || !lm || !scores || !aligned16(q) || !aligned16(lm)) return DD_ERR_INVALID_ARG;
  c->launches += 1;
  const dd_dims &d = c->dims;
  return cuda_ok(minmax ? dd::launch_score_minmax(static_cast<const uint4 *>(q), static_cast<const uint4 *>(lm),
                                                  scores, d.B, d.n_q, d.Hq, d.Hkv, c->C, c->sm_count, c->status,
                                                  (cudaStream_t)stream, trace)
                        : dd::launch_score(static_cast<const uint4 *>(q), static_cast<const uint4 *>(lm), scores, d.B,
                                           d.n_q, d.Hq, d.Hkv, c->C, c->sm_count, c->status, (cudaStream_t)stream,
                                           trace));
}

template <typename T>
T *carve(uint8_t *&cur, int64_t n) {
  T *p = reinterpret_cast<T *>(cur);
  const int64_t bytes = ((n * (int64_t)sizeof(T)) + 255) & ~int64_t(255);
  cur += bytes;
  return p;
}

}  // namespace

extern "C" {

const char *dd_status_str(dd_status s) {
  switch (s) {
    case DD_OK: return "ok";
    case DD_ERR_INVALID_ARG: return "invalid argument";
    case DD_ERR_CUDA: return "CUDA runtime error";
    case DD_ERR_CAPACITY: return "more missing chunks than the staging capacity";
    case DD_ERR_TIMEOUT: return "a bounded device wait ran out";
    case DD_ERR_DEVICE_CHECK: return "an index read on the device was out of range";
  }
  return "unknown status";
}

dd_status dd_create(const dd_dims *dims, int64_t max_misses, int64_t hot_slots, dd_ctx **out) {
  if (!out) return DD_ERR_INVALID_ARG;
  *out = nullptr;
  DD_TRY(check_dims(dims));
  // pool rows are addressed with 32-bit coordinates
  if (max_misses < 0 || hot_slots < 0 || max_misses * dims->cs >= (int64_t(1) << 31) ||
      hot_slots * dims->cs >= (int64_t(1) << 31))
    return DD_ERR_INVALID_ARG;
  dd_ctx *c = new dd_ctx();
  c->dims = *dims;
  c->C = dims->L / dims->cs;
  c->G = dims->Hq / dims->Hkv;
  c->NQ = dims->n_q * c->G;
  c->umax = dims->n_q * dims->k < c->C ? dims->n_q * dims->k : c->C;
  c->units = dims->B * dims->Hkv;
  c->max_misses = max_misses;
  c->hot_slots = hot_slots;
  auto fail = [&](dd_status s) {
    dd_destroy(c);
    return s;
  };
  if (cuda_ok(cudaGetDevice(&c->device)) != DD_OK ||
      cuda_ok(cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device)) != DD_OK)
    return fail(DD_ERR_CUDA);

  const int64_t B = dims->B, Hkv = dims->Hkv, n_q = dims->n_q, k = dims->k, C = c->C;
  const int64_t units = c->units;
  c->plan = dd::attn_plan(c->units, c->umax, c->NQ, c->sm_count);
  int64_t bytes = 0;
  auto add = [&](int64_t n, int64_t sz) { bytes += ((n * sz) + 255) & ~int64_t(255); };
  add(1, 4);                                   // status
  add(B * n_q * Hkv * C, 4);                   // scores
  add(B * n_q * Hkv * k, 4);                   // sel
  add(units * c->umax, 4);                     // union_idx
  add(units * c->umax, 4);                     // union_slot
  add(units * c->umax, 1);                     // union_qmask
  add(units, 4);                               // union_cnt
  add(units, 4);                               // unit_miss
  add(max_misses > 0 ? max_misses : 1, 4);     // miss_list
  add(1, 4);                                   // miss_count
  add(B * n_q * Hkv * k, 4);                   // attn_slot
  add(c->plan.part_o_floats, 4);               // part_o
  add(c->plan.part_ml_floats, 4);              // part_ml
  add(2 * units + 1, 4);                       // chunk_off + fix-up counters
  add(c->plan.flat_entries, 16);               // flat chunk table
  add(64 * 128, 2);                            // dummy pool (64 rows)
  add(units, 8);                               // look-back words
  add(16 * units, 8);                          // union and miss offsets by the last CTA (a line per unit)
  add(3, 4);                                   // ticket counters + look-back epoch
  add(1, 8);                                   // self-test word
  if (cudaMalloc(&c->ws, bytes) != cudaSuccess) return fail(DD_ERR_CUDA);
  uint8_t *cur = static_cast<uint8_t *>(c->ws);
  c->status = carve<int32_t>(cur, 1);
  c->scores = carve<float>(cur, B * n_q * Hkv * C);
  c->sel = carve<int32_t>(cur, B * n_q * Hkv * k);
  c->union_idx = carve<int32_t>(cur, units * c->umax);
  c->union_slot = carve<int32_t>(cur, units * c->umax);
  c->union_qmask = carve<uint8_t>(cur, units * c->umax);
  c->union_cnt = carve<int32_t>(cur, units);
  c->unit_miss = carve<int32_t>(cur, units);
  c->miss_list = carve<int32_t>(cur, max_misses > 0 ? max_misses : 1);
  c->miss_count = carve<int32_t>(cur, 1);
  c->attn_slot = carve<int32_t>(cur, B * n_q * Hkv * k);
  c->part_o = carve<float>(cur, c->plan.part_o_floats);
  c->part_ml = carve<float>(cur, c->plan.part_ml_floats);
  c->chunk_off = carve<int32_t>(cur, 2 * units + 1);
  c->flat = carve<int4>(cur, c->plan.flat_entries);
  c->dummy_pool = carve<uint16_t>(cur, 64 * 128);
  c->lb_word = carve<unsigned long long>(cur, units);
  c->lb_pref = carve<unsigned long long>(cur, 16 * units);
  c->ticket = carve<int32_t>(cur, 3);
  c->diag_word = carve<unsigned long long>(cur, 1);
  if (cudaMemset(c->ws, 0, bytes) != cudaSuccess) return fail(DD_ERR_CUDA);
  const int32_t first_epoch = 1;   // look-back words start zeroed, i.e. with epoch 0
  if (cudaMemcpy(c->ticket + 2, &first_epoch, sizeof(first_epoch), cudaMemcpyHostToDevice) != cudaSuccess)
    return fail(DD_ERR_CUDA);
  if (cudaMallocHost(reinterpret_cast<void **>(&c->h_miss), (size_t)(1 + (max_misses > 0 ? max_misses : 1)) * 4) !=
      cudaSuccess)
    return fail(DD_ERR_CUDA);
  if (cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking) != cudaSuccess) return fail(DD_ERR_CUDA);
  for (int p = 0; p < 2; ++p) {
    if (cudaEventCreateWithFlags(&c->released[p], cudaEventDisableTiming) != cudaSuccess)
      return fail(DD_ERR_CUDA);
  }
  if (cudaEventCreateWithFlags(&c->ready, cudaEventDisableTiming) != cudaSuccess) return fail(DD_ERR_CUDA);
  *out = c;
  return DD_OK;
}

dd_status dd_destroy(dd_ctx *c) {
  if (!c) return DD_ERR_INVALID_ARG;
  if (c->copy_stream) cudaStreamSynchronize(c->copy_stream);
  for (int p = 0; p < 2; ++p) {
    if (c->released[p]) cudaEventDestroy(c->released[p]);
  }
  if (c->ready) cudaEventDestroy(c->ready);
  if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
  if (c->h_miss) cudaFreeHost(c->h_miss);
  if (c->ws) cudaFree(c->ws);
  delete c;
  return DD_OK;
}

int64_t dd_launch_count(const dd_ctx *c) { return c ? c->launches : -1; }

const char *dd_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "" : cudaGetErrorString(g_last_cuda_error);
}

dd_status dd_get_status(dd_ctx *c, int32_t *device_status) {
  if (!c || !device_status) return DD_ERR_INVALID_ARG;
  DD_CUDA(cudaDeviceSynchronize());
  DD_CUDA(cudaMemcpy(device_status, c->status, 4, cudaMemcpyDeviceToHost));
  DD_CUDA(cudaMemset(c->status, 0, 4));
  return DD_OK;
}

dd_status dd_build_landmarks(dd_ctx *c, const void *K, void *lm, dd_stream_t stream) {
  if (!c) return DD_ERR_INVALID_ARG;
  if (c->units == 0) return DD_OK;
  if (!K || !lm || !aligned16(K) || !aligned16(lm)) return DD_ERR_INVALID_ARG;
  const void *kd;
  DD_TRY(device_view(K, &kd));
  c->launches += 1;
  return cuda_ok(dd::launch_build_landmarks(static_cast<const uint4 *>(kd), static_cast<uint4 *>(lm),
                                            (int64_t)c->units * c->C, c->dims.cs, (cudaStream_t)stream));
}

dd_status dd_score_landmarks(dd_ctx *c, const void *q, const void *lm, float *scores, dd_stream_t stream) {
  return score_impl(c, q, lm, scores, false, nullptr, stream);
}

dd_status dd_build_landmarks_minmax(dd_ctx *c, const void *K, void *lm2, dd_stream_t stream) {
  if (!c) return DD_ERR_INVALID_ARG;
  if (c->units == 0) return DD_OK;
  if (!K || !lm2 || !aligned16(K) || !aligned16(lm2)) return DD_ERR_INVALID_ARG;
  const void *kd;
  DD_TRY(device_view(K, &kd));
  c->launches += 1;
  return cuda_ok(dd::launch_build_minmax(static_cast<const uint4 *>(kd), static_cast<uint4 *>(lm2),
                                         (int64_t)c->units * c->C, c->dims.cs, (cudaStream_t)stream));
}

dd_status dd_score_landmarks_minmax(dd_ctx *c, const void *q, const void *lm2, float *scores, dd_stream_t stream) {
  return score_impl(c, q, lm2, scores, true, nullptr, stream);
}

dd_status dd_select_topk(dd_ctx *c, const float *scores, int32_t *sel, dd_stream_t stream) {
  if (!c) return DD_ERR_INVALID_ARG;
  if (c->units == 0) return DD_OK;
  if (!scores || !sel) return DD_ERR_INVALID_ARG;
  c->launches += 1;
  return cuda_ok(dd::launch_topk(scores, sel, c->dims.B * c->dims.n_q * c->dims.Hkv, c->C, c->dims.k,
                                 (cudaStream_t)stream));
}

dd_status dd_select_topk_mass(dd_ctx *c, const float *scores, int32_t *sel, int32_t *sel_cnt, float gamma,
                              int32_t k_min, float softmax_scale, dd_stream_t stream) {
  if (!c) return DD_ERR_INVALID_ARG;
  if (!(gamma > 0.f) || k_min < 1 || k_min > c->dims.k || c->dims.k > 4096) return DD_ERR_INVALID_ARG;
  if (c->units == 0) return DD_OK;
  if (!scores || !sel) return DD_ERR_INVALID_ARG;
  // one query head's logit scale: the score sums the group's G dot products
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)kD);
  const float tau_log2e = scale / (float)c->G * 1.4426950408889634f;
  c->launches += 1;
  return cuda_ok(dd::launch_topk_mass(scores, sel, sel_cnt, c->dims.B * c->dims.n_q * c->dims.Hkv, c->C, c->dims.k,
                                      k_min, gamma, tau_log2e, (cudaStream_t)stream));
}

static dd_status resolve_impl(dd_ctx *c, const int32_t *sel, const int32_t *resident_slot, int32_t *union_idx,
                              int32_t *union_slot, uint8_t *union_qmask, int32_t *union_cnt, int32_t *miss_list,
                              int32_t *miss_count, int32_t *attn_slot, bool with_plan, dd_stream_t stream) {
  if (!c) return DD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (c->units == 0) return miss_count ? cuda_ok(cudaMemsetAsync(miss_count, 0, 4, s)) : DD_OK;
  if (!sel || !resident_slot || !union_idx || !union_slot || !union_qmask || !union_cnt || !miss_list ||
      !miss_count)
    return DD_ERR_INVALID_ARG;
  const dd_dims &d = c->dims;
  DD_CUDA(dd::launch_union(sel, resident_slot, union_idx, union_slot, union_qmask, union_cnt, c->unit_miss, c->units,
                           d.n_q, d.Hkv, d.k, c->C, c->umax, c->hot_slots, c->status, s));
  const dd::AttnPlanOut po = {c->chunk_off, c->flat};
  DD_CUDA(dd::launch_assign(sel, union_idx, union_slot, union_qmask, union_cnt, c->unit_miss, miss_list, miss_count,
                            attn_slot, c->units, d.n_q, d.Hkv, d.k, c->C, c->umax, c->max_misses, c->hot_slots, d.cs,
                            with_plan ? &po : nullptr, c->status, s));
  c->launches += 2;
  return DD_OK;
}

dd_status dd_resolve_union(dd_ctx *c, const int32_t *sel, const int32_t *resident_slot, int32_t *union_idx,
                           int32_t *union_slot, uint8_t *union_qmask, int32_t *union_cnt, int32_t *miss_list,
                           int32_t *miss_count, int32_t *attn_slot, dd_stream_t stream) {
  return resolve_impl(c, sel, resident_slot, union_idx, union_slot, union_qmask, union_cnt, miss_list, miss_count,
                      attn_slot, false, stream);
}

// MEMCPY mode: miss list to the host, then one copy per run of consecutive
// chunks (consecutive ordinals whose packed indices are consecutive are
// contiguous in both the host tensor and the staging buffer).
static dd_status gather_memcpy(dd_ctx *c, const void *Kh, const void *Vh, const int32_t *miss_list,
                               const int32_t *miss_count, void *Kst, void *Vst, cudaStream_t s) {
  DD_CUDA(cudaMemcpyAsync(c->h_miss, miss_count, 4, cudaMemcpyDeviceToHost, s));
  DD_CUDA(cudaStreamSynchronize(s));
  int64_t M = c->h_miss[0];
  if (M < 0) return DD_ERR_DEVICE_CHECK;
  if (M > c->max_misses) M = c->max_misses;   // the resolver already flagged DD_ERR_CAPACITY
  if (M == 0) return DD_OK;
  DD_CUDA(cudaMemcpyAsync(c->h_miss + 1, miss_list, (size_t)M * 4, cudaMemcpyDeviceToHost, s));
  DD_CUDA(cudaStreamSynchronize(s));
  const int64_t chunk_bytes = (int64_t)c->dims.cs * kD * 2;
  const int64_t n_total = (int64_t)c->units * c->C;
  const int32_t *ml = c->h_miss + 1;
  // the whole list is checked before the first copy is queued, so an error
  // leaves nothing in flight on the copy stream
  for (int64_t i = 0; i < M; ++i)
    if (ml[i] < 0 || ml[i] >= n_total) return DD_ERR_DEVICE_CHECK;
  DD_CUDA(cudaEventRecord(c->ready, s));
  DD_CUDA(cudaStreamWaitEvent(c->copy_stream, c->ready, 0));
  int64_t m = 0;
  while (m < M) {
    int64_t run = 1;
    while (m + run < M && ml[m + run] == ml[m] + run) ++run;
    const int64_t src = (int64_t)ml[m] * chunk_bytes, dst = m * chunk_bytes;
    DD_CUDA(cudaMemcpyAsync(static_cast<uint8_t *>(Kst) + dst, static_cast<const uint8_t *>(Kh) + src,
                            (size_t)(run * chunk_bytes), cudaMemcpyDefault, c->copy_stream));
    DD_CUDA(cudaMemcpyAsync(static_cast<uint8_t *>(Vst) + dst, static_cast<const uint8_t *>(Vh) + src,
                            (size_t)(run * chunk_bytes), cudaMemcpyDefault, c->copy_stream));
    m += run;
  }
  DD_CUDA(cudaEventRecord(c->ready, c->copy_stream));
  DD_CUDA(cudaStreamWaitEvent(s, c->ready, 0));
  return DD_OK;
}

dd_status dd_gather_kv(dd_ctx *c, const void *Kh, const void *Vh, const int32_t *miss_list, const int32_t *miss_count,
                       void *Kst, void *Vst, dd_gather_mode mode, dd_stream_t stream) {
  if (!c) return DD_ERR_INVALID_ARG;
  if (mode != DD_GATHER_ZEROCOPY && mode != DD_GATHER_MEMCPY && mode != DD_GATHER_KERNEL) return DD_ERR_INVALID_ARG;
  if (c->units == 0) return DD_OK;
  if (!Kh || !Vh || !miss_list || !miss_count) return DD_ERR_INVALID_ARG;
  if (c->max_misses > 0 && (!Kst || !Vst || !aligned16(Kst) || !aligned16(Vst))) return DD_ERR_INVALID_ARG;
  if (!aligned16(Kh) || !aligned16(Vh)) return DD_ERR_INVALID_ARG;
  if (c->units == 0 || c->max_misses == 0) return DD_OK;
  cudaStream_t s = (cudaStream_t)stream;
  if (mode == DD_GATHER_MEMCPY) {
    int32_t st = 0;
    DD_CUDA(cudaMemcpyAsync(&c->h_miss[0], c->status, 4, cudaMemcpyDeviceToHost, s));
    DD_CUDA(cudaStreamSynchronize(s));
    st = c->h_miss[0];
    if (st != 0) return DD_OK;   // a device error is pending: no work, as the kernels do
    return gather_memcpy(c, Kh, Vh, miss_list, miss_count, Kst, Vst, s);
  }
  const void *kd, *vd;
  DD_TRY(host_kv_views(c, Kh, Vh, &kd, &vd));
  c->launches += 1;
  return cuda_ok(dd::launch_gather(static_cast<const uint4 *>(kd), static_cast<const uint4 *>(vd), miss_list,
                                   miss_count, static_cast<uint4 *>(Kst), static_cast<uint4 *>(Vst), c->max_misses,
                                   (int64_t)c->units * c->C, c->dims.cs, c->status, c->sm_count, s));
}

dd_status dd_prefetch_kv(dd_ctx *c, const int32_t *sel, int32_t sel_rows, int32_t first_row, int32_t n_pred,
                         const void *Kh, const void *Vh, void *Kpf, void *Vpf, int32_t *pf_map, int32_t *pf_count,
                         int32_t ctas_per_sm, dd_stream_t stream) {
  if (!c || n_pred < 1 || n_pred > c->dims.n_q || sel_rows < 1 || first_row < 0 || first_row + n_pred > sel_rows)
    return DD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (c->units == 0) return pf_count ? cuda_ok(cudaMemsetAsync(pf_count, 0, 4, s)) : DD_OK;
  if (!sel || !Kh || !Vh || !pf_map || !aligned16(Kh) || !aligned16(Vh)) return DD_ERR_INVALID_ARG;
  const int32_t *sel_pred = sel + (int64_t)first_row * c->dims.Hkv * c->dims.k;
  if (c->max_misses > 0 && (!Kpf || !Vpf || !aligned16(Kpf) || !aligned16(Vpf))) return DD_ERR_INVALID_ARG;
  if (ctas_per_sm <= 0 || ctas_per_sm > 8) ctas_per_sm = 8;
  const dd_dims &d = c->dims;
  int32_t *cnt = pf_count ? pf_count : c->miss_count;
  const void *kd, *vd;
  DD_TRY(host_kv_views(c, Kh, Vh, &kd, &vd));
  // nothing is resident for the resolver: every predicted chunk gets a slot
  DD_CUDA(cudaMemsetAsync(pf_map, 0xFF, (size_t)c->units * c->C * sizeof(int32_t), s));
  DD_CUDA(dd::launch_union(sel_pred, pf_map, c->union_idx, c->union_slot, c->union_qmask, c->union_cnt, c->unit_miss,
                           c->units, n_pred, d.Hkv, d.k, c->C, c->umax, 0, c->status, s, sel_rows));
  DD_CUDA(dd::launch_assign(sel_pred, c->union_idx, c->union_slot, c->union_qmask, c->union_cnt, c->unit_miss,
                            c->miss_list, cnt, nullptr, c->units, n_pred, d.Hkv, d.k, c->C, c->umax, c->max_misses, 0,
                            d.cs, nullptr, c->status, s));
  c->launches += 2;
  if (c->max_misses == 0) return DD_OK;
  c->launches += 1;
  return cuda_ok(dd::launch_gather(static_cast<const uint4 *>(kd), static_cast<const uint4 *>(vd), c->miss_list, cnt,
                                   static_cast<uint4 *>(Kpf), static_cast<uint4 *>(Vpf), c->max_misses,
                                   (int64_t)c->units * c->C, d.cs, c->status, c->sm_count, s, pf_map, ctas_per_sm));
}

static dd_status attn_impl(dd_ctx *c, const void *q, const void *Khot, const void *Vhot, const void *Kst,
                           const void *Vst, const int32_t *union_slot, const uint8_t *union_qmask,
                           const int32_t *union_cnt, const int32_t *miss_count, float softmax_scale, float *out,
                           bool plan_ready, const void *kh_dev, const void *vh_dev, const void *k_tail,
                           const void *v_tail, dd_stream_t stream, unsigned long long *trace = nullptr) {
  if (!c) return DD_ERR_INVALID_ARG;
  if (c->units == 0) return DD_OK;
  if ((k_tail == nullptr) != (v_tail == nullptr)) return DD_ERR_INVALID_ARG;
  if (!q || !union_slot || !union_qmask || !union_cnt || !miss_count || !out || !aligned16(q))
    return DD_ERR_INVALID_ARG;
  if (c->hot_slots > 0 && (!Khot || !Vhot || !aligned16(Khot) || !aligned16(Vhot))) return DD_ERR_INVALID_ARG;
  if (c->max_misses > 0 && (!Kst || !Vst || !aligned16(Kst) || !aligned16(Vst))) return DD_ERR_INVALID_ARG;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)kD);
  const dd_dims &d = c->dims;
  c->launches += plan_ready ? 1 : 2;   // the attention (and its plan kernel)
  const dd::AttnScratch scr = {c->part_o, c->part_ml, c->chunk_off, c->flat, c->dummy_pool};
  return cuda_ok(dd::launch_attn(q, Khot, Vhot, Kst, Vst, union_slot, union_qmask, union_cnt, miss_count, scale, out,
                                 c->plan, scr, plan_ready, kh_dev, vh_dev, c->status, d.B, d.n_q, d.Hq, d.Hkv, d.cs,
                                 c->umax, c->hot_slots, c->max_misses, (cudaStream_t)stream, k_tail, v_tail,
                                 trace));
}

dd_status dd_sparse_attn_decode(dd_ctx *c, const void *q, const void *Khot, const void *Vhot, const void *Kst,
                                const void *Vst, const void *K_tail, const void *V_tail, const int32_t *union_slot,
                                const uint8_t *union_qmask, const int32_t *union_cnt, const int32_t *miss_count,
                                float softmax_scale, float *out, dd_stream_t stream) {
  return attn_impl(c, q, Khot, Vhot, Kst, Vst, union_slot, union_qmask, union_cnt, miss_count, softmax_scale, out,
                   false, nullptr, nullptr, K_tail, V_tail, stream);
}

dd_status dd_update_residency(dd_ctx *c, int32_t step, int32_t cap, int32_t slots_per_unit,
                              const int32_t *union_idx, const int32_t *union_slot, const int32_t *union_cnt,
                              const int32_t *miss_count, const void *Kst, const void *Vst, int32_t *resident_slot,
                              int32_t *slot_chunk, int32_t *last_used, void *Khot, void *Vhot, int32_t *admitted,
                              dd_stream_t stream) {
  if (!c || step < 0 || cap < 0 || slots_per_unit < 1 || slots_per_unit > 4096) return DD_ERR_INVALID_ARG;
  if (c->units == 0) return DD_OK;
  if ((int64_t)c->units * slots_per_unit != c->hot_slots) return DD_ERR_INVALID_ARG;
  if (!resident_slot || !slot_chunk || !last_used || !Khot || !Vhot || !aligned16(Khot) || !aligned16(Vhot))
    return DD_ERR_INVALID_ARG;
  if (c->max_misses > 0 && (!Kst || !Vst || !aligned16(Kst) || !aligned16(Vst))) return DD_ERR_INVALID_ARG;
  if (!union_idx) union_idx = c->union_idx;
  if (!union_slot) union_slot = c->union_slot;
  if (!union_cnt) union_cnt = c->union_cnt;
  if (!miss_count) miss_count = c->miss_count;
  c->launches += 1;
  return cuda_ok(dd::launch_update_residency(
      step, cap, slots_per_unit, c->units, union_idx, union_slot, union_cnt, miss_count, c->max_misses,
      static_cast<const uint4 *>(Kst), static_cast<const uint4 *>(Vst), resident_slot, slot_chunk, last_used,
      static_cast<uint4 *>(Khot), static_cast<uint4 *>(Vhot), admitted, c->C, c->umax, c->dims.cs, c->status,
      (cudaStream_t)stream));
}

dd_status dd_selftest_bounded_wait(dd_ctx *c, int32_t kind, dd_stream_t stream) {
  if (!c || (kind != 0 && kind != 1)) return DD_ERR_INVALID_ARG;
  c->launches += 1;
  return cuda_ok(dd::launch_selftest_wait(kind, c->diag_word, c->status, (cudaStream_t)stream));
}

int32_t dd_step_folds_scoring(const dd_dims *d, int32_t sm_count, dd_landmark_kind lm_kind, float mass_gamma) {
  if (!d || check_dims(d) != DD_OK || lm_kind != DD_LM_MEAN || !(mass_gamma <= 0.f)) return 0;
  const int C = d->L / d->cs;
  if (dd::fused_select_smem(d->n_q, C, d->k) == 0) return 0;
  return dd::score_select_stages(d->B * d->Hkv, sm_count, d->n_q, C, d->k);
}

dd_status dd_step(dd_ctx *c, const dd_step_args *a, dd_stream_t stream) {
  if (!c || !a || a->layer < 0) return DD_ERR_INVALID_ARG;
  if (a->lm_kind != DD_LM_MEAN && a->lm_kind != DD_LM_MINMAX) return DD_ERR_INVALID_ARG;
  if ((a->K_tail == nullptr) != (a->V_tail == nullptr)) return DD_ERR_INVALID_ARG;
  if (a->mass_gamma > 0.f && (a->mass_k_min < 1 || a->mass_k_min > c->dims.k || c->dims.k > 4096))
    return DD_ERR_INVALID_ARG;
  if (c->units == 0) return DD_OK;
  if (!a->q || !a->lm || !a->Kh || !a->Vh || !a->resident_slot || !a->out) return DD_ERR_INVALID_ARG;
  const int p = a->layer & 1;
  if (c->max_misses > 0 && (!a->Kst[p] || !a->Vst[p])) return DD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned long long *trace = reinterpret_cast<unsigned long long *>(a->trace);
  float *scores = a->scores ? a->scores : c->scores;
  int32_t *sel = a->sel ? a->sel : c->sel;
  int32_t *union_idx = a->union_idx ? a->union_idx : c->union_idx;
  int32_t *union_slot = a->union_slot ? a->union_slot : c->union_slot;
  uint8_t *union_qmask = a->union_qmask ? a->union_qmask : c->union_qmask;
  int32_t *union_cnt = a->union_cnt ? a->union_cnt : c->union_cnt;
  int32_t *miss_list = a->miss_list ? a->miss_list : c->miss_list;
  int32_t *miss_count = a->miss_count ? a->miss_count : c->miss_count;
  int32_t *attn_slot = a->attn_slot ? a->attn_slot : c->attn_slot;

  auto mark = [&](int i) -> dd_status {
    return a->stage_events[i] ? cuda_ok(cudaEventRecord((cudaEvent_t)a->stage_events[i], s)) : DD_OK;
  };
  DD_TRY(mark(0));
  const dd_dims &d = c->dims;
  // Top-k, union, residency, global ordinals and the attention plan run in
  // one kernel per (b,g) when a unit's score rows fit in shared memory (fixed
  // k only), and as separate stage kernels otherwise.  The scoring streams
  // every landmark once over all SMs before it, except when mean landmarks'
  // units fill most SMs in one wave: the selection kernel then streams and
  // scores its own unit on the tensor cores.
  const bool fused = a->mass_gamma <= 0.f && dd::fused_select_smem(d.n_q, c->C, d.k) > 0;
  const int ss_stages = a->q && a->lm && aligned16(a->q) && aligned16(a->lm)
                            ? dd_step_folds_scoring(&d, c->sm_count, a->lm_kind, a->mass_gamma)
                            : 0;
  if (ss_stages == 0) {
    DD_TRY(score_impl(c, a->q, a->lm, scores, a->lm_kind == DD_LM_MINMAX, trace, stream));
    DD_TRY(mark(1));
  }
  if (fused) {
    dd::SelectOut o{};
    o.scores = scores;
    o.sel = a->sel;
    o.attn_slot = a->attn_slot;
    o.resident_slot = a->resident_slot;
    o.union_idx = union_idx;
    o.union_slot = union_slot;
    o.union_qmask = union_qmask;
    o.union_cnt = union_cnt;
    o.unit_miss = c->unit_miss;
    o.miss_list = miss_list;
    o.miss_count = miss_count;
    o.chunk_off = c->chunk_off;
    o.flat = c->flat;
    o.lb_word = c->lb_word;
    o.lb_pref = c->lb_pref;   // the launch drops it when the units cannot all be resident
    o.ticket = c->ticket;
    o.units = c->units;
    o.Hq = d.Hq;
    o.Hkv = d.Hkv;
    o.C = c->C;
    o.k = d.k;
    o.umax = c->umax;
    o.cs = d.cs;
    o.hot_slots = c->hot_slots;
    o.max_misses = c->max_misses;
    o.status = c->status;
    o.trace = trace ? trace + 2 * dd::kTraceSlots : nullptr;
    o.sm_count = c->sm_count;
    o.after_tc_score = a->lm_kind == DD_LM_MEAN;
    if (ss_stages > 0) {
      if (!dd::make_pool_map(&o.tm_lm, a->lm, (int64_t)c->units * c->C, 128)) return DD_ERR_CUDA;
      o.q16 = static_cast<const uint16_t *>(a->q);
      o.scores_out = a->scores;
      o.trace_score = trace;
      DD_CUDA(dd::launch_score_select(o, d.n_q, ss_stages, s));
      DD_TRY(mark(1));
    } else {
      DD_CUDA(dd::launch_select_fused(o, d.n_q, s));
    }
    DD_TRY(mark(2));
    c->launches += 1;
  } else {
    if (a->mass_gamma > 0.f) {
      DD_TRY(dd_select_topk_mass(c, scores, sel, a->sel_cnt, a->mass_gamma, a->mass_k_min, a->softmax_scale,
                                 stream));
    } else {
      DD_TRY(dd_select_topk(c, scores, sel, stream));
    }
    DD_TRY(mark(2));
    DD_TRY(resolve_impl(c, sel, a->resident_slot, union_idx, union_slot, union_qmask, union_cnt, miss_list,
                        miss_count, attn_slot, true, stream));
  }
  DD_TRY(mark(3));
  // staging buffer p may still be read by the attention of layer - 2; on the
  // same stream the stream order already guarantees it, and leaving out the
  // wait lets the attention kernel launch early behind the resolver
  // While the stream is being captured into a CUDA graph the step leaves the
  // release events alone: the captured steps are ordered by the graph itself,
  // and an event recorded during a capture cannot be waited on outside it.
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  DD_CUDA(cudaStreamIsCapturing(s, &capturing));
  const bool captured = capturing != cudaStreamCaptureStatusNone;
  if (!captured && c->used[p] && c->released_on[p] != s) DD_CUDA(cudaStreamWaitEvent(s, c->released[p], 0));
  const void *kh_dev = nullptr, *vh_dev = nullptr;
  const dd_gather_mode gmode =
      a->mode == DD_GATHER_AUTO ? (c->hot_slots > 0 ? DD_GATHER_KERNEL : DD_GATHER_ZEROCOPY) : a->mode;
  if (gmode == DD_GATHER_ZEROCOPY) {
    // the attention kernel itself copies the missing chunks from host memory
    // into its tiles and into staging buffer p (one pass over the host link)
    if (c->max_misses > 0) DD_TRY(host_kv_views(c, a->Kh, a->Vh, &kh_dev, &vh_dev));
  } else {
    DD_TRY(dd_gather_kv(c, a->Kh, a->Vh, miss_list, miss_count, a->Kst[p], a->Vst[p], gmode, stream));
  }
  // memcpy mode: dd_gather_kv made this stream wait for the copy stream
  DD_TRY(mark(4));
  DD_TRY(attn_impl(c, a->q, a->Khot, a->Vhot, a->Kst[p], a->Vst[p], union_slot, union_qmask, union_cnt, miss_count,
                   a->softmax_scale, a->out, true, kh_dev, vh_dev, a->K_tail, a->V_tail, stream,
                   trace ? trace + 4 * dd::kTraceSlots : nullptr));
  DD_TRY(mark(5));
  if (!captured) {
    DD_CUDA(cudaEventRecord(c->released[p], s));
    c->released_on[p] = s;
    c->used[p] = true;
  }
  return DD_OK;
}

}  // extern "C"
