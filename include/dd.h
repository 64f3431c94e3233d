/*
 * dd.h -- C ABI of libdd: one layer of a predictive sparse-KV decode step on
 * one NVIDIA GB300 GPU (sm_103a).
 *
 * The step (DualDecoder: Accelerate Long Context LLM Inference by Predictive
 * Prefetch, §4.1, §5.1-§5.4 and Figs. 8 and 11):
 *   1. score the real query and the speculative query(ies) of every request
 *      together against per-chunk mean-key landmarks,
 *   2. keep the top-k chunks per (request, query, KV head),
 *   3. take the union of the queries' selections per (request, KV head) and
 *      resolve which chunks already sit in the HBM hot pool and which must
 *      come from host memory (Adaptive DHiSparse, Figs. 2 and 3),
 *   4. copy each distinct missing chunk once from pinned host memory into a
 *      layer-scoped ping-pong HBM staging buffer,
 *   5. run GQA attention of every query over the rows of its own selection.
 *
 * Extensions of the same step: Quest-style min/max landmarks and coverage
 * budgets for the selection, the step's own tokens as causal tail rows of
 * the attention, a capped LRU residency update of per-(request, KV head) hot
 * pools after a step, and a predictive prefetch of a layer's predicted
 * chunks ahead of its step (each documented at its entry point below).
 *
 * Notation: B requests, Hq query heads, Hkv KV heads, G = Hq/Hkv (query head h
 * reads KV head floor(h/G)), d head dimension, L context tokens, cs tokens per
 * chunk, C = L/cs chunks, k chunks per selection, n_q queries per request
 * (j = 0 real, j >= 1 speculative), NQ = n_q*G query vectors per KV head,
 * Umax = min(C, n_q*k) the largest possible union.
 *
 * Conventions
 *   - bf16 is IEEE bfloat16 (uint16 storage).  All tensors are dense,
 *     row-major in the layouts given per argument, and owned by the caller;
 *     the library allocates only in dd_create (workspace, one status word,
 *     two events, one copy stream, one pinned host list) and frees it in
 *     dd_destroy.
 *   - Device pointers must be 16-byte aligned.  "Host" K/V pointers must be
 *     page-locked (cudaHostAlloc, cudaMallocHost or cudaHostRegister); the
 *     kernels read them in place over the host link.  A context remembers the
 *     device-side address of the last few host K/V pointers it was given, keyed
 *     by the host address, so a host K/V buffer must stay allocated and pinned
 *     while the context lives: a buffer freed or unregistered and another
 *     placed at the same address needs a new context.
 *   - Every call is asynchronous on the stream it is given (NULL = the legacy
 *     default stream) and returns DD_ERR_INVALID_ARG / DD_ERR_CUDA at once for
 *     errors the host can see.  Errors found on the device (an index out of
 *     range, more misses than the staging capacity, a wait that ran out) are
 *     written to the context's status word, first error wins; kernels never
 *     trap.  While the word is non-zero the gather and attention kernels do no
 *     work.  dd_get_status reads and clears it.
 *   - A context serves one stream at a time; calls on one context must not
 *     overlap on the GPU.
 *   - Supported shapes: d = 128; cs in {16, 32, 64}; L a multiple of cs;
 *     1 <= k <= C <= 16384; 1 <= n_q <= 8; Hq a multiple of Hkv; NQ <= 64;
 *     B*Hkv*C < 2^31; B = 0 is accepted and every call is then a no-op.
 */
#ifndef DD_H_
#define DD_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *dd_stream_t;

typedef enum {
  DD_OK = 0,
  DD_ERR_INVALID_ARG = 1,   /* bad shape, pointer, alignment or enum (host-side check) */
  DD_ERR_CUDA = 2,          /* a CUDA runtime call failed */
  DD_ERR_CAPACITY = 3,      /* device: more missing chunks than the staging buffer holds */
  DD_ERR_TIMEOUT = 4,       /* device: a bounded wait inside a kernel ran out */
  DD_ERR_DEVICE_CHECK = 5   /* device: an index or slot read from memory was out of range */
} dd_status;

typedef struct {
  int32_t B, Hq, Hkv, d, L, cs, k, n_q;
} dd_dims;

typedef enum {
  DD_GATHER_ZEROCOPY = 0,   /* a kernel loads the host chunks over the host link (no host sync); in
                               dd_step that kernel is the attention itself: one warp per CTA copies
                               the missing chunks of the CTA's slice into staging, in slice order and
                               as far ahead as the link allows, while another streams every tile
                               (hot pool or staging) by TMA */
  DD_GATHER_MEMCPY = 1,     /* miss list read back to the host, one cudaMemcpyAsync per run of
                               consecutive chunks on the context's copy stream (host sync) */
  DD_GATHER_KERNEL = 2,     /* a separate zero-copy gather kernel copies every missing chunk into
                               the staging buffer with all SMs' loads in flight, then the attention
                               reads staging like the hot pool; for steps where most chunks are
                               resident and the misses are few and scattered */
  DD_GATHER_AUTO = 3        /* dd_step only: DD_GATHER_KERNEL when the context has a hot pool
                               (hot_slots > 0), else DD_GATHER_ZEROCOPY.  Measured on one GB300:
                               with 10-50% of the union missing the separate gather kernel keeps the
                               host link at 84-93% of its peak where the fused one reaches 51-69%
                               (the misses fall unevenly on the attention's slices); with every
                               chunk missing the fused gather is 3% faster */
} dd_gather_mode;

typedef struct dd_ctx dd_ctx;

#define DD_TRACE_SLOTS 256   /* per-SM slots of dd_step_args.trace */

/* Create a context for one shape.  max_misses: capacity of each staging
 * buffer in chunks (M_cap); B*Hkv*Umax guarantees DD_ERR_CAPACITY never
 * occurs.  hot_slots: number of chunk slots of the caller's hot pool (0 when
 * there is none); resident slots are checked against it.  The current CUDA
 * device at creation is the context's device. */
dd_status dd_create(const dd_dims *dims, int64_t max_misses, int64_t hot_slots, dd_ctx **out);
dd_status dd_destroy(dd_ctx *ctx);

/* Chunk-mean key landmarks (DualDecoder §2.2 and §4.1; built once, before
 * decoding).  K: bf16 [B,Hkv,L,d], device or pinned host.  lm: bf16
 * [B,Hkv,C,d] device.  lm[b,g,c,i] = bf16_rne(fp32 sum over t = 0..cs-1 in
 * order of K[b,g,c*cs+t,i], divided by cs). */
dd_status dd_build_landmarks(dd_ctx *ctx, const void *K, void *lm, dd_stream_t stream);

/* Landmark scores of all n_q queries in one pass over lm (DualDecoder §4.1,
 * §5.2).  q: bf16 [B,n_q,Hq,d]; lm: bf16 [B,Hkv,C,d]; scores: fp32
 * [B,n_q,Hkv,C] = sum over the G q-heads h of KV head g of q[b,j,h,:].lm[b,g,c,:]
 * (unscaled; fp32 accumulation).  Ordering: the kernel starts reading lm
 * while the kernel before it on the stream may still be finishing (it waits
 * for that kernel only before reading q and writing scores), so lm must not
 * be written by that kernel.  libdd's landmark builders and any kernel
 * launched without programmatic dependent launch are safe predecessors; so
 * is a copy.  The same holds for the lm of dd_step. */
dd_status dd_score_landmarks(dd_ctx *ctx, const void *q, const void *lm, float *scores, dd_stream_t stream);

/* Top-k with a coverage budget (MOIRA: per request, layer, KV head and step,
 * the smallest set of chunks whose estimated attention mass reaches gamma;
 * the budget varies per row).  scores: fp32 [B,n_q,Hkv,C].  The estimated
 * mass of chunk c in a row is w_c = exp(tau*(s_c - max s)) / sum exp(...),
 * tau = softmax_scale/G (one query head's logit scale; softmax_scale <= 0
 * selects 1/sqrt(d)); k_row = the least count of chunks, taken in (score
 * desc, chunk asc) order, whose mass reaches gamma, clamped to
 * [k_min, k] (k = the context's k, at most 4096).  sel: int32 [B,n_q,Hkv,k],
 * each row's k_row chunks ascending then -1 (which the resolver skips);
 * sel_cnt: int32 [B,n_q,Hkv] or NULL, k_row per row.  The masses are fp32
 * sums in a fixed order, so the result repeats exactly from run to run. */
dd_status dd_select_topk_mass(dd_ctx *ctx, const float *scores, int32_t *sel, int32_t *sel_cnt, float gamma,
                              int32_t k_min, float softmax_scale, dd_stream_t stream);

/* Landmark kinds (dd_step_args.lm_kind). */
typedef enum { DD_LM_MEAN = 0, DD_LM_MINMAX = 1 } dd_landmark_kind;

/* Quest-style min/max landmarks (OasisKV summary, Methodology: two summary
 * vectors per block, its coordinate-wise minimum and maximum key).  K: bf16
 * [B,Hkv,L,d], device or pinned host.  lm2: bf16 [B,Hkv,C,2,d] device, twice
 * the size of mean landmarks; lm2[b,g,c,0,i] and lm2[b,g,c,1,i] are the
 * smallest and the largest of K[b,g,c*cs+t,i] over t < cs, -0 counting as
 * below +0.  Exact (no rounding). */
dd_status dd_build_landmarks_minmax(dd_ctx *ctx, const void *K, void *lm2, dd_stream_t stream);

/* Upper-bound scores on min/max landmarks, all n_q queries in one pass.
 * q: bf16 [B,n_q,Hq,d]; lm2: bf16 [B,Hkv,C,2,d]; scores: fp32 [B,n_q,Hkv,C] =
 * sum_i max(Q_i * lm2[b,g,c,0,i], Q_i * lm2[b,g,c,1,i]) with Q the fp32 sum
 * of the G q-heads of KV head g: the largest value Q.k takes over any key k
 * inside the chunk's min/max box, hence never below Q.k_t for a token t of
 * the chunk (fp32 accumulation). */
dd_status dd_score_landmarks_minmax(dd_ctx *ctx, const void *q, const void *lm2, float *scores,
                                    dd_stream_t stream);

/* Top-k chunks per row (OasisKV summary, Methodology: top-K per KV head).
 * scores: fp32 [B,n_q,Hkv,C]; sel: int32 [B,n_q,Hkv,k], the k chunks with the
 * largest scores ordered by (score desc, chunk asc), written in ascending
 * chunk order.  -0.0 equals +0.0; NaN ranks below every number. */
dd_status dd_select_topk(dd_ctx *ctx, const float *scores, int32_t *sel, dd_stream_t stream);

/* Union of the queries' selections and residency resolution (Adaptive
 * DHiSparse, Figs. 2 and 3).  sel: int32 [B,n_q,Hkv,k] ascending;
 * resident_slot: int32 [B,Hkv,C], hot-pool slot or -1.  Outputs (device):
 *   union_idx   int32 [B,Hkv,Umax]  union chunks, ascending (entries past union_cnt untouched)
 *   union_slot  int32 [B,Hkv,Umax]  resident slot (>= 0) or -(m+1) for staging slot m
 *   union_qmask uint8 [B,Hkv,Umax]  bit j set when query j selected the chunk
 *   union_cnt   int32 [B,Hkv]
 *   miss_list   int32 [max_misses]  miss m -> (b*Hkv+g)*C + c, m dense in (b,g,c) order
 *   miss_count  int32 [1]           total misses M (may exceed max_misses: DD_ERR_CAPACITY)
 *   attn_slot   int32 [B,n_q,Hkv,k] encoded slot of sel[b,j,g,r] (may be NULL: not written) */
dd_status dd_resolve_union(dd_ctx *ctx, const int32_t *sel, const int32_t *resident_slot,
                           int32_t *union_idx, int32_t *union_slot, uint8_t *union_qmask,
                           int32_t *union_cnt, int32_t *miss_list, int32_t *miss_count,
                           int32_t *attn_slot, dd_stream_t stream);

/* Copy missing chunk m from the pinned host K/V (bf16 [B,Hkv,L,d]) into
 * staging slot m of Kst/Vst (bf16 [max_misses,cs,d], device), byte-exact
 * (DualDecoder §5.4, GPU-side sparse KV assembly).  miss_list/miss_count are
 * device arrays as written by dd_resolve_union.  DD_GATHER_MEMCPY blocks the
 * calling thread until the miss list is on the host. */
dd_status dd_gather_kv(dd_ctx *ctx, const void *Kh, const void *Vh, const int32_t *miss_list,
                       const int32_t *miss_count, void *Kst, void *Vst, dd_gather_mode mode,
                       dd_stream_t stream);

/* Split-K GQA decode attention of every query over its own selected rows,
 * each union row read once for all queries that selected it (DualDecoder
 * §5.2 co-batched dual-token attention; Adaptive DHiSparse Fig. 3).
 * q: bf16 [B,n_q,Hq,d]; Khot/Vhot: bf16 [hot_slots,cs,d] (may be NULL when
 * hot_slots = 0); Kst/Vst: bf16 [max_misses,cs,d]; union_slot, union_qmask,
 * union_cnt, miss_count as written by dd_resolve_union.
 * out: fp32 [B,n_q,Hq,d], out[b,j,h] = sum_t softmax_t(scale*q.K_t) V_t over
 * the rows of the chunks whose qmask has bit j.  softmax_scale <= 0 selects
 * 1/sqrt(d).  K_tail/V_tail (both NULL, or both given): bf16 [B,n_q,Hkv,d]
 * device, the keys and values of the step's own n_q new tokens; query j then
 * also attends to tail rows 0..j of its KV head (DualDecoder §5.2: the
 * tokens of a step lie one after the other along the sequence under a
 * causal mask; Adaptive DHiSparse Fig. 3 (4)). */
dd_status dd_sparse_attn_decode(dd_ctx *ctx, const void *q, const void *Khot, const void *Vhot,
                                const void *Kst, const void *Vst, const void *K_tail, const void *V_tail,
                                const int32_t *union_slot, const uint8_t *union_qmask,
                                const int32_t *union_cnt, const int32_t *miss_count, float softmax_scale,
                                float *out, dd_stream_t stream);

/* Allocation-free variant of dd_sparse_attn_decode.  The pages have no
 * counterpart: it exists for callers that cannot allocate device memory --
 * a serving loop whose memory is already carved up by its own pool, or a
 * host engine that forbids cudaMalloc between decode steps because the call
 * can synchronise the device -- and therefore cannot create a dd_ctx.
 * It takes no context: dims, hot_slots and max_misses describe the tensors as
 * for dd_create, and the other arguments are those of dd_sparse_attn_decode.
 * device_status: caller-owned device int32, zero before the call; a kernel
 * that finds an error writes its dd_status code there (first error wins).
 * The split-K partials live in one fixed 16 MiB device array inside the
 * library, which every GPU that loads the library holds until the process
 * exits.  A shape whose partials ((CTAs + B*Hkv) slots * NQ * 130 floats,
 * with NQ = n_q*Hq/Hkv and CTAs = 2 * SM count for NQ <= 16, else the SM
 * count), chunk table (16 bytes per union chunk, B*Hkv*min(C, n_q*k)) and
 * chunk offsets do not fit is refused at once with DD_ERR_CAPACITY.  The first call on a device
 * looks up that array's device address (once per device); make that first
 * call before any stream capture.  Nothing in the array needs to start at
 * zero, but every call shares it: calls that overlap on the GPU (on any
 * streams, from any thread) race on it and must be serialised by the
 * caller. */
dd_status dd_sparse_attn_decode_noalloc(const dd_dims *dims, int64_t hot_slots, int64_t max_misses,
                                        const void *q, const void *Khot, const void *Vhot,
                                        const void *Kst, const void *Vst, const int32_t *union_slot,
                                        const uint8_t *union_qmask, const int32_t *union_cnt,
                                        const int32_t *miss_count, float softmax_scale, float *out,
                                        int32_t *device_status, dd_stream_t stream);

/* One layer: score -> top-k -> resolve -> gather into staging buffer
 * p = layer & 1 -> attention (DualDecoder §5.4, Fig. 11, two-layer ping-pong).
 * The gather into buffer p waits on the event recorded when the attention of
 * the previous use of p (layer - 2) finished; attention waits for the gather.
 * Intermediate outputs are written to the caller's arrays when given, else to
 * the context's workspace. */
typedef struct {
  int32_t layer;
  const void *q;                 /* bf16 [B,n_q,Hq,d] device */
  const void *lm;                /* bf16 [B,Hkv,C,d] device (mean) or [B,Hkv,C,2,d] (min/max, see lm_kind) */
  const void *Kh, *Vh;           /* bf16 [B,Hkv,L,d] pinned host */
  const int32_t *resident_slot;  /* int32 [B,Hkv,C] device */
  const void *Khot, *Vhot;       /* bf16 [hot_slots,cs,d] device or NULL */
  void *Kst[2], *Vst[2];         /* bf16 [max_misses,cs,d] device: the ping-pong pair */
  dd_gather_mode mode;
  float softmax_scale;           /* <= 0: 1/sqrt(d) */
  float *out;                    /* fp32 [B,n_q,Hq,d] device */
  /* optional intermediates (NULL: context workspace) */
  float *scores;
  int32_t *sel, *union_idx, *union_slot, *union_cnt, *miss_list, *miss_count, *attn_slot;
  uint8_t *union_qmask;
  /* optional instrumentation: cudaEvent_t handles (NULL entries skipped)
   * recorded on the stream before scoring and after scoring, top-k, resolve,
   * gather and attention (with the scoring folded into the selection kernel,
   * see dd_step_folds_scoring, "after scoring" follows that one kernel) */
  void *stage_events[6];
  dd_landmark_kind lm_kind;      /* DD_LM_MEAN (0) or DD_LM_MINMAX: how lm is laid out and scored */
  const void *K_tail, *V_tail;   /* bf16 [B,n_q,Hkv,d] device or NULL: the step's own tokens (causal) */
  float mass_gamma;              /* > 0: coverage budgets (dd_select_topk_mass) instead of a fixed k */
  int32_t mass_k_min;            /* with mass_gamma: the shortest row */
  int32_t *sel_cnt;              /* with mass_gamma: optional int32 [B,n_q,Hkv] row lengths */
  /* optional in-step timing, device uint64 [3][2][DD_TRACE_SLOTS] or NULL:
   * for the scoring, selection and attention kernels (i = 0, 1, 2), every
   * CTA records when its wait for the kernel before it returned (attention:
   * when it issues its first copy; the scoring kernel's first landmark
   * requests come before that wait and are not counted) with an
   * atomic min into trace[i][0][s] and when it finished with an atomic max
   * into trace[i][1][s], s = the SM it ran on (%smid mod DD_TRACE_SLOTS; ns of
   * %globaltimer).  The kernel's window is the minimum of row 0 and the
   * maximum of row 1.  The caller sets every trace[i][0][s] to UINT64_MAX and
   * every trace[i][1][s] to 0 before the step.  Unlike events between the
   * kernels it leaves their overlap in place, and one pair of words per SM
   * keeps the atomics from contending.  Fused selection and attention only
   * (the stage kernels of the other paths record nothing).  With the scoring
   * folded into the selection kernel, i = 0 is that kernel's scoring phase
   * (from its dependency wait to its last CTA's last key row) and i = 1 its
   * selection phase (from the first CTA done scoring to the last CTA's end). */
  uint64_t *trace;
} dd_step_args;

/* dd_step may be captured into a CUDA graph (zero-copy, kernel and auto
 * gather modes; the memcpy mode reads the miss list on the host): it keeps no per-call state on the
 * host that a replay would repeat wrongly.  While the stream is capturing, the
 * release events of the staging buffers are left alone -- the graph orders
 * its own steps -- so a caller that replays such a graph and also runs steps
 * on another stream orders the two itself.
 *
 * When all of the step's selection CTAs (one per (request, KV head) unit)
 * fit on the device at once, the last to finish its counts hands every unit
 * its union and miss offsets and the others wait for it, so all of them must
 * be able to start: under MPS with an SM limit below the device's SM count,
 * or beside a kernel on another stream that holds SMs and waits for this
 * step, some may not, and the bounded wait then ends the step with
 * DD_ERR_TIMEOUT in the status word instead of hanging. */
dd_status dd_step(dd_ctx *ctx, const dd_step_args *args, dd_stream_t stream);

/* Whether dd_step scores the landmarks inside its selection kernel, for a
 * context of these dimensions on a device of sm_count SMs: with mean
 * landmarks, a fixed k and (request, KV head) units filling 3/4 of the SMs or
 * more in one wave, each selection CTA streams its own unit's landmarks and
 * scores them on the tensor cores (one kernel fewer per step, the score rows
 * never leave the SM).  Returns the depth of its landmark ring (3-5), or 0
 * when the step runs the scoring kernel first (then also for invalid
 * dimensions).  Host only: no device call. */
int32_t dd_step_folds_scoring(const dd_dims *dims, int32_t sm_count, dd_landmark_kind lm_kind, float mass_gamma);

/* Predictive prefetch of a layer's predicted selection into its transfer
 * buffer (DualDecoder §4.1-§4.2: the selection computed from the speculative
 * token of step i predicts the one the real token needs at step i+1; §5.3:
 * the layer's prefetch runs ahead of its attention on a low-priority stream
 * and the chunks the prediction missed are fetched urgently by the step;
 * §5.4: prefetched entries wait in temporary slots of the layer's buffer).
 * sel: int32 [B,sel_rows,Hkv,k] device, ascending rows; rows first_row ..
 * first_row+n_pred-1 of each request are the prediction, 1 <= n_pred <= n_q
 * (e.g. the speculative rows j = 1..n_q-1 of the previous step's sel:
 * sel_rows = n_q, first_row = 1).
 * The union of the predicted rows of each (b,g) takes dense slots m in
 * (b,g,c) order; chunk c of unit (b,g) is copied from the pinned host K/V
 * (bf16 [B,Hkv,L,d]) into Kpf/Vpf[m] (bf16 [max_misses,cs,d] device) and
 * pf_map[b,g,c] (int32 [B,Hkv,C] device) = m, -1 for chunks not predicted.
 * pf_count (int32[1] device or NULL) = the number of predicted chunks; more
 * than max_misses raises DD_ERR_CAPACITY and nothing is copied.
 * ctas_per_sm (1..8, other values 8) caps the copy kernel's residency so it
 * leaves room on the SMs for a step running concurrently.  The consuming
 * dd_step passes pf_map as resident_slot and Kpf/Vpf as its hot pool
 * (hot_slots = this context's max_misses).  The prefetch uses the
 * context's resolver workspace: run it on its own context when it overlaps
 * a step on another stream. */
dd_status dd_prefetch_kv(dd_ctx *ctx, const int32_t *sel, int32_t sel_rows, int32_t first_row, int32_t n_pred,
                         const void *Kh, const void *Vh, void *Kpf, void *Vpf, int32_t *pf_map, int32_t *pf_count,
                         int32_t ctas_per_sm, dd_stream_t stream);

/* Residency update after a step: delta selection with capped LRU eviction
 * (OasisKV summary, Methodology; Adaptive DHiSparse Fig. 3 (3): promoted rows
 * are copied from the staging arena into the hot cache).  The hot pool of the
 * context (hot_slots = B*Hkv*slots_per_unit, 1 <= slots_per_unit <= 4096) is
 * split per (b,g) unit u: slots u*S .. u*S+S-1, S = slots_per_unit.  State
 * (device, updated in place): resident_slot int32 [B,Hkv,C] (global slot or
 * -1), slot_chunk int32 [B,Hkv,S] (chunk in the slot or -1 = free),
 * last_used int32 [B,Hkv,S] (step the slot's chunk was last selected; -1 or
 * a step >= 0), Khot/Vhot bf16 [hot_slots,cs,d].  Per unit, in order:
 *   1. every resident chunk of the union gets last_used = step and is kept;
 *   2. targets: free slots by ascending slot, then the other resident slots
 *      by (last_used, slot) ascending;
 *   3. the union's missing chunks in ascending chunk order take the first
 *      A = min(cap, #misses, #targets) targets: the target's old chunk leaves
 *      resident_slot, the new chunk enters it, and its rows are copied from
 *      staging slot m (union_slot = -(m+1)) of Kst/Vst.
 * union_idx / union_slot / union_cnt / miss_count are the step's resolver
 * outputs (NULL: the context's workspace, i.e. the last dd_step or
 * dd_resolve_union that used it); Kst/Vst the staging buffer that step
 * gathered into.  admitted: int32 [B,Hkv] or NULL, A per unit.  At most
 * cap*B*Hkv chunks are copied per call. */
dd_status dd_update_residency(dd_ctx *ctx, int32_t step, int32_t cap, int32_t slots_per_unit,
                              const int32_t *union_idx, const int32_t *union_slot, const int32_t *union_cnt,
                              const int32_t *miss_count, const void *Kst, const void *Vst,
                              int32_t *resident_slot, int32_t *slot_chunk, int32_t *last_used, void *Khot,
                              void *Vhot, int32_t *admitted, dd_stream_t stream);

/* Diagnostics for failure detection: runs one of the library's bounded
 * device waits on something that nothing will ever signal -- kind 0: an
 * mbarrier no thread arrives on and no copy completes (the waits of the
 * attention pipeline and of the selection's landmark ring); kind 1: a
 * look-back word no unit publishes (the selection's sum over earlier
 * units).  The wait gives up by itself after about 2 s and records
 * DD_ERR_TIMEOUT in the status word; the context stays usable once
 * dd_get_status has read and cleared it.  No fault or trap is involved. */
dd_status dd_selftest_bounded_wait(dd_ctx *ctx, int32_t kind, dd_stream_t stream);

/* Wait for the device, read the status word into *device_status (a dd_status
 * value) and clear it. */
dd_status dd_get_status(dd_ctx *ctx, int32_t *device_status);

/* Number of kernel launches issued by the context since creation (all calls). */
int64_t dd_launch_count(const dd_ctx *ctx);

const char *dd_status_str(dd_status status);

/* Text of the CUDA runtime error behind the calling thread's most recent
 * DD_ERR_CUDA ("" when there was none). */
const char *dd_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DD_H_ */
