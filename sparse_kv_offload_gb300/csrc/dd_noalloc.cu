// Attention entry point for callers that cannot allocate device memory.
//
// dd_sparse_attn_decode keeps its split-K partials in the workspace that
// dd_create allocates.  Some callers cannot make that allocation: a serving
// loop whose device memory is already carved up by its own pool, or a host
// engine that forbids cudaMalloc between decode steps because the call can
// synchronise the device.  dd_sparse_attn_decode_noalloc runs the same
// attention kernel (and its plan kernel), with the partials in a fixed device array
// that is part of the library image.  That array (kNoAllocScratchBytes) is
// held by every GPU that loads the library until the process exits.
#include <mutex>

#include "dd_common.cuh"

namespace {

// Largest scratch the allocation-free attention may use: 16 MiB.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr size_t kDummyPoolBytes = 64 * 128 * 2;   // a valid base address for unused TMA maps

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices] = {};

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

// Device address of the scratch array on the current device, looked up once
// per device (the array's name is only a host-side stand-in in host code).
dd_status scratch_on_current_device(unsigned char **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return DD_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<unsigned char *>(g_scratch_addr[dev]);
  return DD_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" dd_status dd_sparse_attn_decode_noalloc(const dd_dims *dims, int64_t hot_slots, int64_t max_misses,
                                                   const void *q, const void *Khot, const void *Vhot,
                                                   const void *Kst, const void *Vst, const int32_t *union_slot,
                                                   const uint8_t *union_qmask, const int32_t *union_cnt,
                                                   const int32_t *miss_count, float softmax_scale, float *out,
                                                   int32_t *device_status, dd_stream_t stream) {
  if (!dims) return DD_ERR_INVALID_ARG;
  const dd_dims &d = *dims;
  if (d.B < 0 || d.Hq <= 0 || d.Hkv <= 0 || d.Hq % d.Hkv || d.d != dd::kD) return DD_ERR_INVALID_ARG;
  if ((d.cs != 16 && d.cs != 32 && d.cs != 64) || d.L <= 0 || d.L % d.cs) return DD_ERR_INVALID_ARG;
  const int C = d.L / d.cs;
  if (C > dd::kMaxC || d.k < 1 || d.k > C || d.n_q < 1 || d.n_q > dd::kMaxNq) return DD_ERR_INVALID_ARG;
  const int G = d.Hq / d.Hkv, NQ = d.n_q * G;
  if (NQ > dd::kMaxNQV || (int64_t)d.B * d.Hkv * C >= (int64_t(1) << 31)) return DD_ERR_INVALID_ARG;
  if (hot_slots < 0 || max_misses < 0 || hot_slots * d.cs >= (int64_t(1) << 31) ||
      max_misses * d.cs >= (int64_t(1) << 31))
    return DD_ERR_INVALID_ARG;
  const int units = d.B * d.Hkv;
  if (units == 0) return DD_OK;
  // the split-K partials and the chunk offsets of this shape must fit the fixed scratch array
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DD_ERR_CUDA;
  const int umax = d.n_q * d.k < C ? d.n_q * d.k : C;
  const dd::AttnPlan plan = dd::attn_plan(units, umax, NQ, sms);
  const size_t o_bytes = round256((size_t)plan.part_o_floats * sizeof(float));
  const size_t ml_bytes = round256((size_t)plan.part_ml_floats * sizeof(float));
  const size_t off_bytes = round256((size_t)(2 * units + 1) * sizeof(int32_t));   // + fix-up counters
  const size_t flat_bytes = round256((size_t)plan.flat_entries * 16);
  if (o_bytes + ml_bytes + off_bytes + flat_bytes + kDummyPoolBytes > kNoAllocScratchBytes)
    return DD_ERR_CAPACITY;
  if (!q || !union_slot || !union_qmask || !union_cnt || !miss_count || !out || !device_status || !aligned16(q))
    return DD_ERR_INVALID_ARG;
  if (hot_slots > 0 && (!Khot || !Vhot || !aligned16(Khot) || !aligned16(Vhot))) return DD_ERR_INVALID_ARG;
  if (max_misses > 0 && (!Kst || !Vst || !aligned16(Kst) || !aligned16(Vst))) return DD_ERR_INVALID_ARG;

  unsigned char *base = nullptr;
  const dd_status s = scratch_on_current_device(&base);
  if (s != DD_OK) return s;
  unsigned char *cur = base;
  float *part_o = reinterpret_cast<float *>(cur);
  cur += o_bytes;
  float *part_ml = reinterpret_cast<float *>(cur);
  cur += ml_bytes;
  int32_t *chunk_off = reinterpret_cast<int32_t *>(cur);
  cur += off_bytes;
  int4 *flat = reinterpret_cast<int4 *>(cur);
  cur += flat_bytes;
  const dd::AttnScratch scr = {part_o, part_ml, chunk_off, flat, cur};
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)dd::kD);
  const cudaError_t e = dd::launch_attn(q, Khot, Vhot, Kst, Vst, union_slot, union_qmask, union_cnt, miss_count,
                                        scale, out, plan, scr, false, nullptr, nullptr, device_status, d.B, d.n_q,
                                        d.Hq, d.Hkv, d.cs, umax, hot_slots, max_misses, (cudaStream_t)stream);
  return e == cudaSuccess ? DD_OK : DD_ERR_CUDA;
}
