"""Plain CPU restatement of one sparse-KV decode layer -- TEST INFRASTRUCTURE ONLY.

Arrays of bf16 values are passed as their uint16 bit patterns.  Floating-point
stages compute in fp64 unless a stage produces a quantised value (the bf16
landmark), where the decision is taken in the precision the stage defines
(fp32 accumulation, then round-to-nearest-even to bf16).

Notation (from the pages, with the readings where they are silent):
  B requests, Hq query heads, Hkv KV heads, G = Hq/Hkv (query head h reads KV
  head floor(h/G)), d head dimension, L context tokens, cs tokens per chunk,
  C = L/cs chunks, k chunks selected per (request, query, KV head), n_q
  queries per request (j = 0 the real query, j >= 1 speculative ones).

Parity pins: every function below is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_decode", "bf16_encode", "build_landmarks", "score_landmarks", "select_topk",
    "resolve_union", "gather_kv", "sparse_attn_decode", "step", "kv_footprint_bytes",
    "max_batch", "per_step_budget_bytes", "union_of_query_selections",
    "build_minmax_landmarks", "score_minmax_landmarks", "bf16_total_order_key", "update_residency",
    "prefetch_kv", "select_by_mass", "NO_SLOT",
]


# ---------------------------------------------------------------------------
# bf16 encoding (IEEE bfloat16: the top 16 bits of an fp32)
# ---------------------------------------------------------------------------

def _bf16_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_decode(u: np.ndarray) -> np.ndarray:
    """bf16 bits -> fp64 values (exact)."""
    return _bf16_to_f32(u).astype(np.float64)


def bf16_encode(x: np.ndarray) -> np.ndarray:
    """fp32 values -> bf16 bits, rounding to nearest, ties to even (finite inputs)."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    return ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


# ---------------------------------------------------------------------------
# a0: chunk landmarks
# ---------------------------------------------------------------------------

def build_landmarks(K: np.ndarray, cs: int) -> np.ndarray:
    """Chunk-mean key landmarks, bf16 bits [B, Hkv, C, d].

    DualDecoder §2.2: adjacent KV entries are grouped into chunks and each
    chunk keeps one compact landmark used to rank chunks for a query; §4.1:
    the landmarks are made once, ahead of the decode loop.  The landmark
    is the mean key of the chunk.  Reading: the sum runs in fp32 over the
    chunk's tokens in order t = 0..cs-1, is divided by cs in fp32 and rounded
    to bf16 (the KV dtype, as the "1/16 of the KV cache" summary size in the
    OasisKV Methodology implies).
    """
    B, H, L, d = K.shape
    if L % cs:
        raise ValueError("L must be a multiple of the chunk size")
    C = L // cs
    k32 = _bf16_to_f32(K).reshape(B, H, C, cs, d)
    acc = np.zeros((B, H, C, d), dtype=np.float32)
    for t in range(cs):
        acc = acc + k32[:, :, :, t, :]
    return bf16_encode(acc / np.float32(cs))


# ---------------------------------------------------------------------------
# a1: landmark scores for all queries of a request
# ---------------------------------------------------------------------------

def score_landmarks(q: np.ndarray, lm: np.ndarray) -> np.ndarray:
    """s[b, j, g, c] = sum over the q-heads h of KV head g of q[b,j,h,:] . lm[b,g,c,:] (fp64).

    DualDecoder §4.1: the retrieval index is computed from the token being
    decoded and the landmarks; the speculative token is scored against the
    same landmarks (§5.2 runs both tokens in one pass).  OasisKV Methodology:
    blocks are ranked independently for every KV head.  Reading: the per-KV-
    head score sums the group's query-head dot products; the 1/sqrt(d) scale
    is left out because it does not change the ranking.
    """
    B, n_q, Hq, d = q.shape
    _, Hkv, C, _ = lm.shape
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    qf = bf16_decode(q)
    lf = bf16_decode(lm)
    s = np.zeros((B, n_q, Hkv, C), dtype=np.float64)
    for g in range(Hkv):
        for h in range(g * G, (g + 1) * G):
            s[:, :, g, :] += np.einsum("bji,bci->bjc", qf[:, :, h, :], lf[:, g, :, :])
    return s


# ---------------------------------------------------------------------------
# a0 / a1, second landmark kind: coordinate-wise min / max key per chunk
# ---------------------------------------------------------------------------

def bf16_total_order_key(u: np.ndarray) -> np.ndarray:
    """uint16 bf16 bits -> uint32 keys that order the values (finite inputs),
    with -0 below +0 (the IEEE 754 totalOrder predicate on non-NaN values)."""
    u = np.asarray(u, dtype=np.uint16).astype(np.uint32)
    return np.where(u & 0x8000, (~u) & 0xFFFF, u | 0x8000)


def build_minmax_landmarks(K: np.ndarray, cs: int) -> np.ndarray:
    """Per-chunk coordinate-wise minimum and maximum key, bf16 bits [B, Hkv, C, 2, d]
    (index 0 of the fourth axis the minimum, 1 the maximum).

    OasisKV Methodology: the draft query ranks blocks on compressed key
    summaries made by Quest-style min/max pooling, two vectors per block
    (coordinate-wise minimum and maximum).  The extremes of bf16 values are
    bf16 values, so nothing is rounded.  Reading: -0 counts as below +0,
    which makes the result a single well-defined bit pattern.
    """
    B, H, L, d = K.shape
    if L % cs:
        raise ValueError("L must be a multiple of the chunk size")
    C = L // cs
    bits = np.asarray(K, dtype=np.uint16).reshape(B, H, C, cs, d)
    key = bf16_total_order_key(bits)
    lo = np.take_along_axis(bits, np.argmin(key, axis=3)[:, :, :, None, :], axis=3)[:, :, :, 0, :]
    hi = np.take_along_axis(bits, np.argmax(key, axis=3)[:, :, :, None, :], axis=3)[:, :, :, 0, :]
    return np.stack([lo, hi], axis=3)


def score_minmax_landmarks(q: np.ndarray, lm2: np.ndarray) -> np.ndarray:
    """s[b, j, g, c] = sum_i max(Q_i * min_i, Q_i * max_i) with Q the sum of the
    group's query heads q[b, j, h, :] (fp64).

    OasisKV Methodology (Quest-style min/max summaries): the score of a block
    is the largest value the query's dot product can take over any key whose
    coordinates lie between the block's minimum and maximum, which bounds
    every token of the block from above.  Reading: as for the mean
    landmarks, the per-KV-head score is that of the group-summed query, so
    it bounds the group's summed dot product sum_h q_h . k_t for every token
    t of the chunk.
    """
    B, n_q, Hq, d = q.shape
    _, Hkv, C, two, _ = lm2.shape
    if Hq % Hkv or two != 2:
        raise ValueError("need Hq a multiple of Hkv and lm2 of shape [B, Hkv, C, 2, d]")
    G = Hq // Hkv
    Q = bf16_decode(q).reshape(B, n_q, Hkv, G, d).sum(axis=3)   # [B, n_q, Hkv, d]
    lo = bf16_decode(lm2[:, :, :, 0, :])                         # [B, Hkv, C, d]
    hi = bf16_decode(lm2[:, :, :, 1, :])
    s = np.zeros((B, n_q, Hkv, C), dtype=np.float64)
    for j in range(n_q):
        Qj = Q[:, j, :, None, :]                                  # [B, Hkv, 1, d]
        s[:, j] = np.maximum(Qj * lo, Qj * hi).sum(axis=-1)
    return s


# ---------------------------------------------------------------------------
# a2: top-k chunks per (request, query, KV head)
# ---------------------------------------------------------------------------

def select_topk(s: np.ndarray, k: int) -> np.ndarray:
    """The k chunks with the largest scores per row, returned in ascending chunk order.

    OasisKV Methodology: top-K blocks per KV head.  Reading: rows are ordered
    by (score descending, chunk index ascending), so among exactly equal
    scores the lower chunk index is selected first; the chosen set is then
    listed in ascending chunk index.
    """
    *lead, C = s.shape
    if not 1 <= k <= C:
        raise ValueError("need 1 <= k <= C")
    rows = np.asarray(s, dtype=np.float64).reshape(-1, C)
    out = np.empty((rows.shape[0], k), dtype=np.int32)
    chunk = np.arange(C)
    for r in range(rows.shape[0]):
        order = np.lexsort((chunk, -rows[r]))   # last key is primary
        out[r] = np.sort(order[:k])
    return out.reshape(*lead, k)


def select_by_mass(s: np.ndarray, k_max: int, gamma: float, tau: float, k_min: int = 1):
    """Per row, the smallest set of chunks whose estimated attention mass reaches gamma.

    MOIRA (abstract): for every request, layer, KV head and step, a coverage
    rule keeps the smallest set of pages whose estimated attention mass
    reaches a fraction gamma, so the budget varies per head and layer.
    Readings: the estimated mass of chunk c in a row is
    w_c = exp(tau * (s_c - max s)) / sum_c' exp(tau * (s_c' - max s)) (fp64),
    tau being the logit scale of one query head (the attention scale over G,
    since s sums the group's G dot products); the smallest set is the
    first k_row chunks in (score descending, chunk ascending) order, k_row
    the least count whose mass sum reaches gamma, then clamped to
    [k_min, k_max].  Returns sel [..., k_max] (the chosen chunks ascending,
    then -1) and the per-row counts [...].
    """
    *lead, C = s.shape
    if not 1 <= k_min <= k_max <= C:
        raise ValueError("need 1 <= k_min <= k_max <= C")
    rows = np.asarray(s, dtype=np.float64).reshape(-1, C)
    sel = np.full((rows.shape[0], k_max), -1, dtype=np.int32)
    cnt = np.empty(rows.shape[0], dtype=np.int32)
    chunk = np.arange(C)
    for r in range(rows.shape[0]):
        row = rows[r]
        w = np.exp(tau * (row - row.max()))
        w /= w.sum()
        order = np.lexsort((chunk, -row))
        csum = np.cumsum(w[order])
        k_row = int(np.searchsorted(csum, gamma, side="left")) + 1   # first prefix reaching gamma
        k_row = min(max(k_row, k_min), k_max)
        cnt[r] = k_row
        sel[r, :k_row] = np.sort(order[:k_row])
    return sel.reshape(*lead, k_max), cnt.reshape(*lead)


# ---------------------------------------------------------------------------
# a3: union across queries, residency, miss ordinals
# ---------------------------------------------------------------------------

def union_of_query_selections(sel: np.ndarray, b: int, g: int) -> list:
    """Ascending union of the selections of all queries of request b, KV head g."""
    n_q = sel.shape[1]
    u = set()
    for j in range(n_q):
        u |= set(int(c) for c in sel[b, j, g] if c >= 0)   # -1: padding of a shorter row
    return sorted(u)


NO_SLOT = -(2 ** 31)   # attn_slot of a padding entry (-1) of a shorter selection row


def resolve_union(sel: np.ndarray, resident_slot: np.ndarray) -> dict:
    """Resolve the union of the queries' selections against the HBM pool.

    Adaptive DHiSparse Fig. 3: the selections of the several queries of a
    request and KV source are resolved in one pass, so a chunk picked by
    several queries is fetched from the host a single time; attention still
    uses every query's own top-k.  Fig. 2: a selected row is looked up in the HBM tiers first
    and copied from host DRAM only when it is found in none of them.

    Readings: per (b, g) the union U lists chunks in ascending order; a chunk
    is resident when ``resident_slot[b,g,c] >= 0`` (its slot in the hot pool)
    and missing otherwise; missing chunks take dense ordinals m = 0..M-1 in
    (b, g, c) lexicographic order and are addressed as staging slot m,
    encoded -(m+1).  ``miss_list[m] = (b*Hkv + g)*C + c``.  ``union_qmask``
    has bit j set when query j selected the chunk.  ``attn_slot[b,j,g,r]`` is
    the encoded slot of the r-th chunk of query j's selection (NO_SLOT for a
    padding entry -1 of a row shorter than k).
    Entries of the union arrays past ``union_cnt`` are padding (-1 / 0).
    """
    B, n_q, Hkv, k = sel.shape
    C = resident_slot.shape[2]
    umax = min(C, n_q * k)
    union_idx = np.full((B, Hkv, umax), -1, dtype=np.int32)
    union_slot = np.full((B, Hkv, umax), -1, dtype=np.int32)
    union_qmask = np.zeros((B, Hkv, umax), dtype=np.uint8)
    union_cnt = np.zeros((B, Hkv), dtype=np.int32)
    attn_slot = np.empty((B, n_q, Hkv, k), dtype=np.int32)
    miss_list = []
    for b in range(B):
        for g in range(Hkv):
            per_query = [set(int(c) for c in sel[b, j, g] if c >= 0) for j in range(n_q)]
            U = union_of_query_selections(sel, b, g)
            union_cnt[b, g] = len(U)
            slot_of = {}
            for u, c in enumerate(U):
                rs = int(resident_slot[b, g, c])
                if rs >= 0:
                    slot_of[c] = rs
                else:
                    m = len(miss_list)
                    miss_list.append((b * Hkv + g) * C + c)
                    slot_of[c] = -(m + 1)
                union_idx[b, g, u] = c
                union_slot[b, g, u] = slot_of[c]
                union_qmask[b, g, u] = sum(1 << j for j in range(n_q) if c in per_query[j])
            for j in range(n_q):
                for r in range(k):
                    c = int(sel[b, j, g, r])
                    attn_slot[b, j, g, r] = slot_of[c] if c >= 0 else NO_SLOT
    return {
        "union_idx": union_idx, "union_cnt": union_cnt, "union_slot": union_slot,
        "union_qmask": union_qmask, "miss_list": np.asarray(miss_list, dtype=np.int32),
        "miss_count": len(miss_list), "attn_slot": attn_slot,
    }


# ---------------------------------------------------------------------------
# a4: gather of missing chunks into the staging buffer
# ---------------------------------------------------------------------------

def gather_kv(Kh: np.ndarray, Vh: np.ndarray, miss_list: np.ndarray, cs: int):
    """Copy chunk ``miss_list[m]`` of the host K and V into staging slot m.

    DualDecoder §5.4 (GPU-side sparse KV assembly): selected KV blocks are
    moved from host memory into a GPU staging region and placed in the
    attention layout there.  Reading: staging slot m holds the cs rows of
    the m-th missing chunk, K and V in separate arrays [M, cs, d].
    """
    B, H, L, d = Kh.shape
    C = L // cs
    M = len(miss_list)
    Kst = np.empty((M, cs, d), dtype=Kh.dtype)
    Vst = np.empty((M, cs, d), dtype=Vh.dtype)
    for m, packed in enumerate(np.asarray(miss_list).tolist()):
        unit, c = divmod(int(packed), C)
        b, g = divmod(unit, H)
        Kst[m] = Kh[b, g, c * cs:(c + 1) * cs]
        Vst[m] = Vh[b, g, c * cs:(c + 1) * cs]
    return Kst, Vst


# ---------------------------------------------------------------------------
# a5: attention of every query over its own selected rows
# ---------------------------------------------------------------------------

def _rows(pool_hot, pool_stage, slot: int):
    return pool_hot[slot] if slot >= 0 else pool_stage[-slot - 1]


def sparse_attn_decode(q, Khot, Vhot, Kst, Vst, attn_slot, cs: int, scale: float | None = None,
                       K_tail=None, V_tail=None):
    """o[b,j,h,:] = sum over the selected rows t of softmax_t(scale * q . K_t) * V_t (fp64).

    DualDecoder §5.2: the output and speculative tokens attend in one pass;
    OasisKV Methodology: normal and draft queries attend together over one
    resident working set; Adaptive DHiSparse Fig. 3: each query attends over
    the chunks it picked itself.  Readings: scale = 1/sqrt(d); query head h uses KV
    head floor(h/G); the rows of query j are those of the k chunks in
    ``attn_slot[b,j,g,:]``.

    A query with no selected chunk attends to its tail rows alone; with no
    rows at all its output is zero (the softmax over an empty set is
    undefined; zero is the library's convention).

    Tail rows (optional): ``K_tail, V_tail`` bf16 [B, n_q, Hkv, d] are the
    keys and values of the step's own new tokens, token j being query j's.
    DualDecoder §5.2 places the tokens of a step one after the other along
    the sequence with a causal mask, so query j also attends to tail rows
    0..j and never to a later token's row (Adaptive DHiSparse Fig. 3 (4):
    every query's row is written to the tail, which the resolver reads
    first).
    """
    B, n_q, Hq, d = q.shape
    Hkv = attn_slot.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qf = bf16_decode(q)
    out = np.zeros((B, n_q, Hq, d), dtype=np.float64)
    for b in range(B):
        for j in range(n_q):
            for g in range(Hkv):
                slots = [int(s) for s in attn_slot[b, j, g] if s != NO_SLOT]
                Kr = np.zeros((0, d)) if not slots else bf16_decode(
                    np.concatenate([_rows(Khot, Kst, s) for s in slots], axis=0))
                Vr = np.zeros((0, d)) if not slots else bf16_decode(
                    np.concatenate([_rows(Vhot, Vst, s) for s in slots], axis=0))
                if K_tail is not None:
                    Kr = np.concatenate([Kr, bf16_decode(K_tail[b, :j + 1, g])], axis=0)
                    Vr = np.concatenate([Vr, bf16_decode(V_tail[b, :j + 1, g])], axis=0)
                if Kr.shape[0] == 0:
                    continue        # nothing to attend to: the output stays zero (library convention)
                for h in range(g * G, (g + 1) * G):
                    z = (Kr @ qf[b, j, h]) * scale
                    p = np.exp(z - z.max())
                    p /= p.sum()
                    out[b, j, h] = p @ Vr
    return out


# ---------------------------------------------------------------------------
# ahead of a step: predictive prefetch into the layer's transfer buffer
# ---------------------------------------------------------------------------

def prefetch_kv(sel_pred: np.ndarray, Kh: np.ndarray, Vh: np.ndarray, cs: int) -> dict:
    """Fetch the chunks of a predicted selection ahead of the step that needs them.

    DualDecoder §4.1-§4.2: the selection computed from the speculative token
    of step i predicts the one the real token needs at step i+1, so its
    chunks can be fetched before they are consumed; §5.3: for a layer the
    prefetch runs ahead of its attention, and chunks the true selection needs
    but the prediction missed are fetched urgently; §5.4: prefetched entries
    sit in temporary slots of the layer's transfer buffer until the true
    index is resolved.  The attention result does not depend on the
    prediction.

    Readings: per (b, g) unit the predicted chunks are the union of the
    predicted rows ``sel_pred`` [B, n_pred, Hkv, k]; they take dense slots
    m in (b, g, c) order, the same layout as the step's misses (so the
    prefetch is the resolver and the gather run on the predicted selection
    with nothing resident).  Returns ``pf_map`` [B, Hkv, C] (slot of each
    prefetched chunk, -1 elsewhere), the rows ``K``, ``V`` [P, cs, d] and
    ``count`` P.  The step that consumes the prefetch resolves its true
    selection against ``pf_map`` as if it were the resident map, with the
    prefetched rows as the pool.
    """
    B, Hkv, L, d = Kh.shape
    C = L // cs
    res = resolve_union(sel_pred, np.full((B, Hkv, C), -1, np.int32))
    K, V = gather_kv(Kh, Vh, res["miss_list"], cs)
    pf_map = np.full(B * Hkv * C, -1, np.int32)
    for m, packed in enumerate(res["miss_list"].tolist()):
        pf_map[packed] = m
    return {"pf_map": pf_map.reshape(B, Hkv, C), "K": K, "V": V, "count": res["miss_count"]}


# ---------------------------------------------------------------------------
# after a step: residency update of the per-(request, KV head) hot pools
# ---------------------------------------------------------------------------

def update_residency(step_id: int, cap: int, union_idx, union_slot, union_cnt, Kst, Vst,
                     resident_slot, slot_chunk, last_used, Khot, Vhot):
    """Delta selection with capped LRU eviction; returns the updated copies
    (resident_slot, slot_chunk, last_used, Khot, Vhot) and the admitted count per unit.

    OasisKV summary, Methodology (delta selection and capped eviction), per
    KV head and decoding step: chunks of the selection that are resident
    cost no traffic; resident chunks outside the selection are ranked by the
    step they were last selected in; each admitted non-resident chunk is
    paired with one eviction target, least recently used first; at most
    ``cap`` pairs are admitted, which bounds the traffic to cap * H entries.
    Adaptive DHiSparse Fig. 3 (3): promoted rows are copied from the staging
    arena into the hot cache.

    Readings: every (b, g) unit owns the S = slot_chunk.shape[-1] pool slots
    u*S .. u*S+S-1 (resident_slot holds these global slot numbers, -1 when
    absent); a slot whose slot_chunk is -1 is free and is used before any
    eviction, lowest slot first; eviction order is (last_used ascending, slot
    ascending); resident chunks of the current union get last_used = step_id
    and are never evicted; the missing chunks of the union are admitted in
    ascending chunk order, the i-th admitted one going into the i-th target;
    its K and V come from staging slot m of union_slot = -(m+1).
    """
    resident_slot = np.array(resident_slot, dtype=np.int32, copy=True)
    slot_chunk = np.array(slot_chunk, dtype=np.int32, copy=True)
    last_used = np.array(last_used, dtype=np.int32, copy=True)
    Khot = np.array(Khot, copy=True)
    Vhot = np.array(Vhot, copy=True)
    B, Hkv, C = resident_slot.shape
    S = slot_chunk.shape[-1]
    sc = slot_chunk.reshape(B * Hkv, S)
    lu = last_used.reshape(B * Hkv, S)
    rs = resident_slot.reshape(B * Hkv, C)
    admitted = np.zeros(B * Hkv, dtype=np.int32)
    umax = union_idx.shape[-1]
    ui = np.asarray(union_idx).reshape(B * Hkv, umax)
    us = np.asarray(union_slot).reshape(B * Hkv, umax)
    for u in range(B * Hkv):
        base = u * S
        n = int(np.asarray(union_cnt).reshape(-1)[u])
        entries = [(int(ui[u, i]), int(us[u, i])) for i in range(n)]
        in_union = set()
        for c, sl in entries:
            if sl >= 0:
                in_union.add(sl - base)
                lu[u, sl - base] = step_id
        misses = [(c, -sl - 1) for c, sl in entries if sl < 0]
        free = [t for t in range(S) if sc[u, t] < 0]
        evictable = sorted((t for t in range(S) if sc[u, t] >= 0 and t not in in_union),
                           key=lambda t: (int(lu[u, t]), t))
        targets = free + evictable
        A = min(cap, len(misses), len(targets))
        for i in range(A):
            c, m = misses[i]
            t = targets[i]
            old = int(sc[u, t])
            if old >= 0:
                rs[u, old] = -1
            rs[u, c] = base + t
            sc[u, t] = c
            lu[u, t] = step_id
            Khot[base + t] = Kst[m]
            Vhot[base + t] = Vst[m]
        admitted[u] = A
    return {"resident_slot": resident_slot, "slot_chunk": slot_chunk, "last_used": last_used,
            "Khot": Khot, "Vhot": Vhot, "admitted": admitted.reshape(B, Hkv)}


# ---------------------------------------------------------------------------
# a6: one layer's step
# ---------------------------------------------------------------------------

def step(q, lm, Kh, Vh, resident_slot, Khot, Vhot, k: int, cs: int, scale=None, K_tail=None, V_tail=None,
         gamma=None, k_min: int = 1) -> dict:
    """Score -> top-k -> union/resolve -> gather -> attention for one layer.

    DualDecoder Fig. 8 / §5.1-§5.4: retrieval index from the query and the
    landmarks, missing entries fetched from host into the layer's staging
    buffer, then sparse attention over the selected entries.  ``lm`` holds
    mean landmarks [B, Hkv, C, d] or min/max landmarks [B, Hkv, C, 2, d];
    the score follows the kind.  With ``gamma`` the rows are chosen by the
    coverage rule of ``select_by_mass`` (k is then the longest row allowed).
    """
    s = score_minmax_landmarks(q, lm) if lm.ndim == 5 else score_landmarks(q, lm)
    sel_cnt = None
    if gamma is None:
        sel = select_topk(s, k)
    else:   # coverage budget: k is the largest row length
        G = q.shape[2] // lm.shape[1]
        tau = (1.0 / math.sqrt(q.shape[-1]) if scale is None else scale) / G
        sel, sel_cnt = select_by_mass(s, k, gamma, tau, k_min)
    res = resolve_union(sel, resident_slot)
    Kst, Vst = gather_kv(Kh, Vh, res["miss_list"], cs)
    out = sparse_attn_decode(q, Khot, Vhot, Kst, Vst, res["attn_slot"], cs, scale, K_tail, V_tail)
    res.update(scores=s, sel=sel, sel_cnt=sel_cnt, Kst=Kst, Vst=Vst, out=out)
    return res


# ---------------------------------------------------------------------------
# OasisKV eqs. (1)-(3)
# ---------------------------------------------------------------------------

def kv_footprint_bytes(B: int, L: int, n_layer: int, n_kv: int, d_h: int, s: int) -> int:
    """OasisKV eq. (1): M_KV = B * L * N_layer * 2 * N_kv * d_h * s."""
    return B * L * n_layer * 2 * n_kv * d_h * s


def max_batch(m_hbm: int, L: int, n_layer: int, n_kv: int, d_h: int, s: int) -> int:
    """OasisKV eq. (2): B_max = floor(M_HBM / (L * N_layer * 2 * N_kv * d_h * s))."""
    return m_hbm // (L * n_layer * 2 * n_kv * d_h * s)


def per_step_budget_bytes(b_link: float, t_decode: float) -> float:
    """OasisKV eq. (3): C_token = B_link * T_decode (bytes the link can move in one step)."""
    return b_link * t_decode
