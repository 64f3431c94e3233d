// Host side of the TMA tensor maps the attention and scoring kernels read.
#include <mutex>

#include "dd_tc.cuh"

namespace dd {

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

// A [rows, 128] bf16 pool viewed as 2-D, boxes of cs rows x 64 columns (cs:
// the chunk rows of a K/V pool, or the 128 landmark rows of a scoring tile).
// A descriptor depends on nothing but (base, rows, cs), so the last few are
// kept: a decode loop cycles through the same pools step after step.
bool make_pool_map(CUtensorMap *map, const void *base, int64_t rows, int cs) {
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

// The queries [B, n_q, Hq, 128] bf16 viewed as 4-D, boxes of 64 columns x G
// heads x n_q queries x 1 request: one box is half of the query vectors of a
// (request, KV head) unit, rows j * G + h, in the 128B-swizzled layout the
// tcgen05 attention's A operand takes.  Cached like the pool maps.
bool make_q_map(CUtensorMap *map, const void *q, int B, int n_q, int Hq, int G) {
  struct Entry {
    const void *q;
    int B, n_q, Hq, G;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[16];
  static int n = 0, next = 0;
  if (q == nullptr) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
      if (cache[i].q == q && cache[i].B == B && cache[i].n_q == n_q && cache[i].Hq == Hq && cache[i].G == G) {
        *map = cache[i].map;
        return true;
      }
  }
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {128, (cuuint64_t)Hq, (cuuint64_t)n_q, (cuuint64_t)B};
  cuuint64_t strides[3] = {256, (cuuint64_t)Hq * 256, (cuuint64_t)n_q * Hq * 256};
  cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)n_q, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(mu);
  cache[next] = {q, B, n_q, Hq, G, *map};
  next = (next + 1) % 16;
  if (n < 16) ++n;
  return true;
}

}  // namespace dd
