"""Seeded, counter-based synthetic inputs for the sparse-KV decode step.

This module is the one piece that both the CUDA path (through its own device
implementation of the same generator, ``dd_synth_*`` in the C ABI) and the CPU
oracle's tests draw inputs from.  It holds none of the decode step's
arithmetic: it only makes keys, values, queries, chunk-bias tables and
residency tables.

Generator (published definitions, restated here):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): the sequence ``mix(state + (i+1)*GAMMA)`` with
  ``GAMMA = 0x9E3779B97F4A7C15`` and the finaliser
  ``z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27; z *= 0x94D049BB133111EB;
  z ^= z>>31``.  Being counter-based, element ``idx`` of any tensor can be
  drawn on its own, which is what lets a test rebuild a sampled slice of a
  tensor the GPU generated in full.
* Normal variates by the Irwin-Hall sum of twelve uniforms: the twelve 16-bit
  fields of three consecutive SplitMix64 words (``3*idx``, ``3*idx+1``,
  ``3*idx+2``) are summed as integers, centred on their mean 393210 and scaled
  by 2^-16.  The result has mean 0, variance 1 - 2^-32 and lies in (-6, 6); it
  is an exact fp32 number, so the host and the device produce the same bits
  with no transcendental function involved.

Derived tensors (the recipe for the synthetic workloads):

* ``q_real[b,h,i] = bf16(N(seed, Q_REAL, idx))``
* ``q[b,j,h,i] = bf16(f32(q_real) + spec_scale[j] * N(seed, Q_NOISE+j, idx))``
  for the speculative queries ``j >= 1`` (fp32 multiply, then fp32 add).
* ``K[b,g,t,i] = bf16(N(seed, K, idx) + bias[b,g,t//cs] * u_hat[b,g,i])`` --
  a key bias along the direction of the group's summed real query, used for
  the "hot chunk" and Zipf-weighted workloads (fp32 multiply, then fp32 add).
* ``V[b,g,t,i] = bf16(N(seed, V, idx))``.

All bf16 conversions round to nearest even.  Tensor ids are offset by
``64 * layer`` so that every layer of a multi-layer run has its own data.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
IH_MEAN = 393210  # 12 * 32767.5, the mean of twelve 16-bit uniforms

# tensor ids (the low 6 bits); a layer adds 64 * layer
TID_K = 1
TID_V = 2
TID_Q_REAL = 3
TID_HOT_PICK = 4
TID_ZIPF_PERM = 5
TID_RESIDENT_PICK = 6
TID_CARRY_PICK = 7
TID_Q_NOISE = 8  # + j for speculative query j (1..7)
TID_SCORE = 16   # seeded stand-alone score rows for select tests
TID_SEL = 17     # seeded stand-alone selections for resolve tests
TID_DRIFT = 32   # + t: drift of the real query at decode step t (t < 16)
TID_DRIFT_SPEC = 48   # + t: error of the speculative queries of decode step t (t < 16)

_BLOCK = 1 << 21


def tensor_id(kind: int, layer: int = 0) -> int:
    return int(kind) + 64 * int(layer)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tid: int) -> np.uint64:
    """State of the SplitMix64 stream for (seed, tensor id)."""
    with np.errstate(over="ignore"):
        s = np.array([((int(seed) << 32) + int(tid)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix(s + GAMMA)[0]


def words(seed: int, tid: int, counter: np.ndarray) -> np.ndarray:
    """SplitMix64 outputs number ``counter`` (0-based) of the (seed, tid) stream."""
    key = stream_key(seed, tid)
    c = np.asarray(counter, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + (c + np.uint64(1)) * GAMMA)


def normal_f32(seed: int, tid: int, idx: np.ndarray) -> np.ndarray:
    """Irwin-Hall(12) normal variates for element indices ``idx`` (fp32, exact)."""
    idx = np.asarray(idx, dtype=np.uint64)
    flat = idx.reshape(-1)
    out = np.empty(flat.shape, dtype=np.float32)
    mask = np.uint64(0xFFFF)
    for s in range(0, flat.size, _BLOCK):
        i = flat[s:s + _BLOCK]
        acc = np.zeros(i.shape, dtype=np.uint64)
        with np.errstate(over="ignore"):
            for r in range(3):
                w = words(seed, tid, np.uint64(3) * i + np.uint64(r))
                for f in range(4):
                    acc += (w >> np.uint64(16 * f)) & mask
        out[s:s + _BLOCK] = (acc.astype(np.int64) - IH_MEAN).astype(np.float32) * np.float32(2.0 ** -16)
    return out.reshape(idx.shape)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 bits, nearest-even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = b.astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# derived tensors
# ---------------------------------------------------------------------------

def drift_queries(seed: int, B: int, n_q: int, Hq: int, d: int, T: int, sigma_drift: float, sigma_spec: float,
                  layer: int = 0) -> np.ndarray:
    """bf16 bits [T, B, n_q, Hq, d]: T decode steps of one layer, cyclic.

    The real query of step t is base + sigma_drift * xi_t, base being the
    layer's real query of ``queries``; every speculative query of step t is
    the real query of step t+1 (mod T) + sigma_spec * eta_t,j: a draft of
    the next step's query."""
    if not 1 <= T <= 16:
        raise ValueError("1 <= T <= 16")
    n = B * Hq * d
    idx = np.arange(n, dtype=np.uint64)
    base = bf16_to_f32(f32_to_bf16(normal_f32(seed, tensor_id(TID_Q_REAL, layer), idx)))
    real = [bf16_to_f32(f32_to_bf16(base + np.float32(sigma_drift)
                                    * normal_f32(seed, tensor_id(TID_DRIFT + t, layer), idx))) for t in range(T)]
    out = np.empty((T, B, n_q, Hq, d), dtype=np.uint16)
    for t in range(T):
        out[t, :, 0] = f32_to_bf16(real[t]).reshape(B, Hq, d)
        for j in range(1, n_q):
            eta = normal_f32(seed, tensor_id(TID_DRIFT_SPEC + t, layer), idx + np.uint64(j * n))
            out[t, :, j] = f32_to_bf16(real[(t + 1) % T] + np.float32(sigma_spec) * eta).reshape(B, Hq, d)
    return out


def queries(seed: int, B: int, n_q: int, Hq: int, d: int, spec_scale, layer: int = 0) -> np.ndarray:
    """bf16 bits [B, n_q, Hq, d]: query j=0 is the real query, j>=1 speculative."""
    n = B * Hq * d
    idx = np.arange(n, dtype=np.uint64)
    real32 = bf16_to_f32(f32_to_bf16(normal_f32(seed, tensor_id(TID_Q_REAL, layer), idx)))
    q = np.empty((B, n_q, Hq, d), dtype=np.uint16)
    q[:, 0] = f32_to_bf16(real32).reshape(B, Hq, d)
    for j in range(1, n_q):
        noise = normal_f32(seed, tensor_id(TID_Q_NOISE + j, layer), idx)
        v = real32 + np.float32(spec_scale[j]) * noise
        q[:, j] = f32_to_bf16(v).reshape(B, Hq, d)
    return q


def query_direction(q: np.ndarray, Hkv: int) -> np.ndarray:
    """u_hat [B, Hkv, d] fp32: unit vector of the group's summed real query."""
    B, _, Hq, d = q.shape
    G = Hq // Hkv
    real = bf16_to_f32(q[:, 0]).reshape(B, Hkv, G, d)
    s = np.zeros((B, Hkv, d), dtype=np.float32)
    for h in range(G):
        s = s + real[:, :, h, :]
    norm = np.sqrt((s.astype(np.float64) ** 2).sum(-1, keepdims=True)).astype(np.float32)
    return (s / norm).astype(np.float32)


def random_order(seed: int, tid: int, n_units: int, C: int) -> np.ndarray:
    """Per unit, a seeded permutation of 0..C-1 (argsort of SplitMix64 words)."""
    w = words(seed, tid, np.arange(n_units * C, dtype=np.uint64)).reshape(n_units, C)
    return np.argsort(w, axis=1, kind="stable")


def hot_chunk_bias(seed: int, B: int, Hkv: int, C: int, frac: float, sigma: float, layer: int = 0) -> np.ndarray:
    """bias [B,Hkv,C] fp32: round(frac*C) seeded chunks per unit get ``sigma``."""
    n_hot = int(round(frac * C))
    order = random_order(seed, tensor_id(TID_HOT_PICK, layer), B * Hkv, C)
    bias = np.zeros((B * Hkv, C), dtype=np.float32)
    rows = np.arange(B * Hkv)[:, None]
    bias[rows, order[:, :n_hot]] = np.float32(sigma)
    return bias.reshape(B, Hkv, C)


def zipf_chunk_bias(seed: int, B: int, Hkv: int, C: int, alpha: float, sigma: float, layer: int = 0) -> np.ndarray:
    """bias [B,Hkv,C] fp32 = sigma * rank^-alpha, ranks a seeded permutation."""
    order = random_order(seed, tensor_id(TID_ZIPF_PERM, layer), B * Hkv, C)
    rank = np.empty_like(order)
    rows = np.arange(B * Hkv)[:, None]
    rank[rows, order] = np.arange(1, C + 1)[None, :]
    bias = (sigma * rank.astype(np.float64) ** (-alpha)).astype(np.float32)
    return bias.reshape(B, Hkv, C)


def kv_rows(seed: int, tid: int, B: int, Hkv: int, L: int, d: int, cs: int,
            units: np.ndarray, t0: np.ndarray, nrows: int,
            bias: np.ndarray | None = None, u_hat: np.ndarray | None = None) -> np.ndarray:
    """bf16 bits of ``nrows`` consecutive rows starting at token t0[n] of unit units[n].

    Returns [len(units), nrows, d].  ``bias``/``u_hat`` apply the key bias.
    """
    units = np.asarray(units, dtype=np.int64).reshape(-1)
    t0 = np.asarray(t0, dtype=np.int64).reshape(-1)
    t = t0[:, None] + np.arange(nrows)[None, :]                      # [n, nrows]
    base = (units[:, None] * L + t) * d                               # [n, nrows]
    idx = (base[:, :, None] + np.arange(d)[None, None, :]).astype(np.uint64)
    x = normal_f32(seed, tid, idx)
    if bias is not None:
        bb = bias.reshape(B * Hkv, -1)[units[:, None], t // cs]       # [n, nrows]
        uu = u_hat.reshape(B * Hkv, d)[units]                         # [n, d]
        x = x + bb[:, :, None].astype(np.float32) * uu[:, None, :]
    return f32_to_bf16(x)


def kv_tensor(seed: int, kind: int, B: int, Hkv: int, L: int, d: int, cs: int,
              bias: np.ndarray | None = None, u_hat: np.ndarray | None = None,
              layer: int = 0) -> np.ndarray:
    """Full K (kind=TID_K, with optional bias) or V tensor, bf16 bits [B,Hkv,L,d]."""
    units = np.arange(B * Hkv)
    out = kv_rows(seed, tensor_id(kind, layer), B, Hkv, L, d, cs, units, np.zeros_like(units), L,
                  bias if kind == TID_K else None, u_hat if kind == TID_K else None)
    return out.reshape(B, Hkv, L, d)


def dense_slots(resident: np.ndarray) -> np.ndarray:
    """resident bool [B,Hkv,C] -> slot int32 [B,Hkv,C], dense in (b,g,c) order, -1 absent."""
    flat = resident.reshape(-1)
    slot = np.full(flat.shape, -1, dtype=np.int32)
    slot[flat] = np.arange(int(flat.sum()), dtype=np.int32)
    return slot.reshape(resident.shape)


def uniform_residency(seed: int, B: int, Hkv: int, C: int, frac: float, layer: int = 0) -> np.ndarray:
    """A seeded uniform subset of round(frac*C) chunks per unit is resident."""
    n_res = int(round(frac * C))
    order = random_order(seed, tensor_id(TID_RESIDENT_PICK, layer), B * Hkv, C)
    res = np.zeros((B * Hkv, C), dtype=bool)
    res[np.arange(B * Hkv)[:, None], order[:, :n_res]] = True
    return dense_slots(res.reshape(B, Hkv, C))


def carried_residency(seed: int, union_sets, B: int, Hkv: int, C: int, frac: float, layer: int = 0) -> np.ndarray:
    """Temporal-locality residency: per unit, round(frac*|U|) members of the
    given union U (the previous step's selection) are resident, plus as many
    seeded non-members (chunks the previous step dropped), so the resident
    set has |U| chunks."""
    order = random_order(seed, tensor_id(TID_CARRY_PICK, layer), B * Hkv, C)
    res = np.zeros((B * Hkv, C), dtype=bool)
    for u in range(B * Hkv):
        U = np.asarray(sorted(union_sets[u]), dtype=np.int64)
        in_u = np.zeros(C, dtype=bool)
        in_u[U] = True
        keep = int(round(frac * U.size))
        ranked = order[u]
        members = ranked[in_u[ranked]][:keep]
        others = ranked[~in_u[ranked]][:U.size - keep]
        res[u, members] = True
        res[u, others] = True
    return dense_slots(res.reshape(B, Hkv, C))


def hot_pool(seed: int, slot: np.ndarray, kind: int, B: int, Hkv: int, L: int, d: int, cs: int,
             bias=None, u_hat=None, layer: int = 0) -> np.ndarray:
    """The HBM hot pool [S_hot, cs, d] for resident chunks: a copy of host rows."""
    flat = slot.reshape(-1)
    C = L // cs
    chunks = np.nonzero(flat >= 0)[0]
    order = np.argsort(flat[chunks])
    chunks = chunks[order]
    if chunks.size == 0:
        return np.zeros((0, cs, d), dtype=np.uint16)
    units = chunks // C
    t0 = (chunks % C) * cs
    return kv_rows(seed, tensor_id(kind, layer), B, Hkv, L, d, cs, units, t0, cs,
                   bias if kind == TID_K else None, u_hat if kind == TID_K else None)


def random_scores(seed: int, rows: int, C: int, tie_every: int = 0) -> np.ndarray:
    """fp32 score rows for stand-alone selection tests; optional forced ties."""
    x = normal_f32(seed, TID_SCORE, np.arange(rows * C, dtype=np.uint64)).reshape(rows, C)
    if tie_every:
        # quantise so that many exact ties occur
        x = (np.round(x * tie_every) / tie_every).astype(np.float32)
    return x


def random_selection(seed: int, B: int, n_q: int, Hkv: int, C: int, k: int, overlap: float) -> np.ndarray:
    """Seeded sorted selections [B,n_q,Hkv,k] whose queries share about
    ``overlap`` of their chunks with query 0."""
    order = random_order(seed, TID_SEL, B * Hkv * n_q, C).reshape(B, Hkv, n_q, C)
    sel = np.empty((B, n_q, Hkv, k), dtype=np.int32)
    n_shared = int(round(overlap * k))
    for b in range(B):
        for g in range(Hkv):
            base = order[b, g, 0, :k]
            sel[b, 0, g] = np.sort(base)
            for j in range(1, n_q):
                own = [c for c in order[b, g, j] if c not in set(base[:n_shared])][:k - n_shared]
                sel[b, j, g] = np.sort(np.concatenate([base[:n_shared], np.asarray(own, dtype=np.int64)]))
    return sel


def hot_pool_from(X: np.ndarray, slot: np.ndarray, cs: int) -> np.ndarray:
    """Hot pool [S_hot, cs, d] copied from a full host tensor X [B,Hkv,L,d]."""
    B, H, L, d = X.shape
    C = L // cs
    flat = slot.reshape(-1)
    chunks = np.nonzero(flat >= 0)[0]
    chunks = chunks[np.argsort(flat[chunks])]
    return np.ascontiguousarray(X.reshape(B * H, C, cs, d)[chunks // C, chunks % C])
