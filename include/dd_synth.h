/*
 * dd_synth.h -- device implementation of the seeded synthetic-input generator
 * used by the benchmark and the tests (part of libdd, not of the decode step).
 *
 * The pages measure on long-context benchmarks with real models; these
 * counter-based tensors stand in for them.  The generator is defined
 * elementwise, so the host copy of the same definition (the Python module
 * sparse_kv_offload_gb300.synth) can rebuild any element on its own:
 *
 *   word(seed, tid, n)   = SplitMix64 output n of the stream whose state is
 *                          mix((seed << 32) + tid + GAMMA)
 *                          (Steele, Lea and Flood, OOPSLA 2014)
 *   N(seed, tid, idx)    = (sum of the twelve 16-bit fields of words 3*idx,
 *                          3*idx+1, 3*idx+2  -  393210) * 2^-16, an exact fp32
 *                          (Irwin-Hall sum of twelve uniforms)
 *   K[b,g,t,i] = bf16(N(seed,tid,idx) + bias[b,g,t/cs] * u_hat[b,g,i])
 *   V[b,g,t,i] = bf16(N(seed,tid,idx))
 *   q[b,0,h,i] = bf16(N(seed, 3+64*layer, (b*Hq+h)*d+i))
 *   q[b,j,h,i] = bf16(f32(q[b,0,h,i]) + spec_scale[j] * N(seed, 8+j+64*layer, same idx))
 *
 * fp32 products and sums are rounded separately (no fused multiply-add);
 * bf16 rounding is to nearest even.  Arguments follow dd.h's conventions.
 */
#ifndef DD_SYNTH_H_
#define DD_SYNTH_H_

#include <stdint.h>

#include "dd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Fill a key (bias given) or value tensor.  With chunk_map == NULL, dst is
 * the whole bf16 [B,Hkv,L,d] tensor (device or pinned host).  Otherwise dst
 * is bf16 [n_slots,cs,d] and slot s receives chunk chunk_map[s] (packed
 * (b*Hkv+g)*C + c), i.e. a hot pool holding copies of those chunks.
 * chunk_bias fp32 [B,Hkv,C] and u_hat fp32 [B,Hkv,d] are device arrays, both
 * NULL or both given.  tensor_id carries the layer (kind + 64*layer). */
dd_status dd_synth_kv(const dd_dims *dims, uint64_t seed, int32_t tensor_id,
                      const float *chunk_bias, const float *u_hat,
                      const int32_t *chunk_map, int64_t n_slots, void *dst, dd_stream_t stream);

/* Fill q bf16 [B,n_q,Hq,d] (device) for one layer; spec_scale is a host array
 * of n_q floats (index 0 unused). */
dd_status dd_synth_queries(const dd_dims *dims, uint64_t seed, int32_t layer,
                           const float *spec_scale, void *dst, dd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DD_SYNTH_H_ */
