"""Shared helpers of the test-suite: seeded inputs of a workload, host <-> torch
conversion, and the parity checks (bit-exact indices modulo the score tie
band, attention within max-abs 2e-2 and relative-L2 1e-3)."""
from __future__ import annotations

import numpy as np

import oracle
from sparse_kv_offload_gb300 import synth
from sparse_kv_offload_gb300.workloads import Workload

ATOL_MAX = 2e-2       # attention: max |gpu - oracle|
REL_L2 = 1e-3         # attention: ||gpu - oracle||_2 / ||oracle||_2
TIE_REL = 1e-5        # top-k: a selection may differ only where the k-th and (k+1)-th scores are this close


# --------------------------------------------------------------------- inputs

def key_bias(w: Workload, q, layer=0):
    if w.key_bias == "hot":
        return synth.hot_chunk_bias(w.seed, w.B, w.Hkv, w.C, w.hot_frac, w.bias_sigma, layer), \
            synth.query_direction(q, w.Hkv)
    if w.key_bias == "zipf":
        return synth.zipf_chunk_bias(w.seed, w.B, w.Hkv, w.C, w.zipf_alpha, w.bias_sigma, layer), \
            synth.query_direction(q, w.Hkv)
    return None, None


def host_inputs(w: Workload, layer: int = 0) -> dict:
    """Every input of one layer step as numpy arrays (bf16 as uint16 bits)."""
    q = synth.queries(w.seed, w.B, w.n_q, w.Hq, w.d, w.spec_scale, layer)
    bias, u_hat = key_bias(w, q, layer)
    K = synth.kv_tensor(w.seed, synth.TID_K, w.B, w.Hkv, w.L, w.d, w.cs, bias, u_hat, layer)
    V = synth.kv_tensor(w.seed, synth.TID_V, w.B, w.Hkv, w.L, w.d, w.cs, layer=layer)
    lm = oracle.build_landmarks(K, w.cs)
    if w.residency == "uniform":
        slot = synth.uniform_residency(w.seed, w.B, w.Hkv, w.C, w.resident_frac, layer)
    elif w.residency == "carry":
        # the previous step's selection: the oracle's selection for this step's
        # queries stands in for it (temporal locality), then a seeded share of
        # it is resident
        sel = oracle.select_topk(oracle.score_landmarks(q, lm), w.k)
        U = [set(oracle.union_of_query_selections(sel, b, g)) for b in range(w.B) for g in range(w.Hkv)]
        slot = synth.carried_residency(w.seed, U, w.B, w.Hkv, w.C, w.resident_frac, layer)
    else:
        slot = np.full((w.B, w.Hkv, w.C), -1, np.int32)
    Khot = synth.hot_pool_from(K, slot, w.cs)
    Vhot = synth.hot_pool_from(V, slot, w.cs)
    return dict(q=q, K=K, V=V, lm=lm, slot=slot, Khot=Khot, Vhot=Vhot, bias=bias, u_hat=u_hat)


# --------------------------------------------------------------------- torch

def to_bf16(a: np.ndarray, device="cuda", pin=False):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    if device == "cpu":
        return t.pin_memory() if pin else t.clone()
    return t.to(device)


def from_bf16(t) -> np.ndarray:
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_i32(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


# --------------------------------------------------------------------- checks

def check_attention(got: np.ndarray, want: np.ndarray, mask=None):
    """max-abs and relative-L2 over the selected outputs (mask over leading dims)."""
    g = np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    if mask is not None:
        g, w = g[mask], w[mask]
    if w.size == 0:
        return 0.0, 0.0
    err = np.abs(g - w).max()
    rel = np.linalg.norm(g - w) / max(np.linalg.norm(w), 1e-300)
    assert err <= ATOL_MAX, f"max-abs error {err:.3e} > {ATOL_MAX}"
    assert rel <= REL_L2, f"relative-L2 error {rel:.3e} > {REL_L2}"
    return err, rel


def selection_rows_match(gpu_sel: np.ndarray, scores64: np.ndarray, oracle_sel: np.ndarray, k: int):
    """Per row: True when the GPU selection equals the oracle's; rows that
    differ must differ only inside the tie band.  Returns the bool row mask."""
    C = scores64.shape[-1]
    g = gpu_sel.reshape(-1, k)
    o = oracle_sel.reshape(-1, k)
    s = scores64.reshape(-1, C)
    same = np.all(g == o, axis=1)
    for r in np.nonzero(~same)[0]:
        row = s[r]
        order = np.lexsort((np.arange(C), -row))
        sk = row[order[k - 1]]
        sk1 = row[order[k]] if k < C else -np.inf
        tau = TIE_REL * max(abs(sk), abs(sk1))
        gset = set(g[r].tolist())
        assert len(gset) == k and list(g[r]) == sorted(gset), f"row {r}: not k distinct ascending chunks"
        must = set(np.nonzero(row > sk + tau)[0].tolist())
        never = set(np.nonzero(row < sk1 - tau)[0].tolist())
        assert must <= gset, f"row {r}: GPU dropped a chunk clearly above the k-th score"
        assert not (gset & never), f"row {r}: GPU kept a chunk clearly below the (k+1)-th score"
    return same.reshape(gpu_sel.shape[:-1])


# ------------------------------------------------ a3-a5 on the GPU's selection

# How often the step-level checks took the tie path: units whose GPU selection
# differs from the oracle's inside the tie band, so that the oracle's union,
# gather and attention were re-run on the GPU's own selection.  Printed in the
# terminal summary of every run (tests/conftest.py).
TIE_TALLY = {"checks": 0, "units": 0, "tie_units": 0, "tie_rows": 0}


def follow_gpu_selection(gpu_sel, want, q, K, V, slot, Khot, Vhot, cs, scale=None, K_tail=None, V_tail=None):
    """The oracle's a3-a5 driven by the GPU's own selection.

    A selection may differ from the oracle's only inside the tie band (the
    k-th and (k+1)-th scores within TIE_REL), and the caller has checked that
    with ``selection_rows_match`` (or the coverage rule's own check).  The
    union, the residency lookup, the miss ordinals, the staging layout and
    the attention are exact functions of the selection, so they are compared
    bit-exact (attention within the tolerances) against the oracle run on the
    GPU's rows.  Where every row agrees this is the oracle's own step.
    Returns (reference dict, tie-unit mask [B, Hkv])."""
    gpu_sel = np.asarray(gpu_sel).reshape(want["sel"].shape)
    diff_rows = np.any(gpu_sel != want["sel"], axis=-1)          # [B, n_q, Hkv]
    tie_units = diff_rows.any(axis=1)                            # [B, Hkv]
    TIE_TALLY["checks"] += 1
    TIE_TALLY["units"] += int(tie_units.size)
    TIE_TALLY["tie_units"] += int(tie_units.sum())
    TIE_TALLY["tie_rows"] += int(diff_rows.sum())
    if not tie_units.any():
        return want, tie_units
    ref = oracle.resolve_union(gpu_sel, slot)
    Kst, Vst = oracle.gather_kv(K, V, ref["miss_list"], cs)
    ref["out"] = oracle.sparse_attn_decode(q, Khot, Vhot, Kst, Vst, ref["attn_slot"], cs, scale, K_tail, V_tail)
    ref.update(Kst=Kst, Vst=Vst, sel=gpu_sel, scores=want["scores"])
    return ref, tie_units


def check_layout(g: dict, ref: dict, B: int, Hkv: int, umax: int, Kst=None, Vst=None):
    """Every unit's union, query mask, slots, the miss list, the per-entry slots
    and (when the staging buffer is given) the staged bytes, bit-exact.
    ``g`` holds the step's intermediates as numpy arrays; absent keys are skipped."""
    M = int(g["miss_count"][0]) if "miss_count" in g else None
    if M is not None:
        assert M == ref["miss_count"], f"miss count {M} != {ref['miss_count']}"
    if "union_cnt" in g:
        cnt = g["union_cnt"].reshape(B, Hkv)
        assert np.array_equal(cnt, ref["union_cnt"]), "union sizes differ"
        for name in ("union_idx", "union_slot", "union_qmask"):
            if name not in g:
                continue
            a = g[name].reshape(B, Hkv, umax)
            for b in range(B):
                for h in range(Hkv):
                    n = cnt[b, h]
                    assert np.array_equal(a[b, h, :n], ref[name][b, h, :n]), f"{name} of unit ({b},{h}) differs"
    if "miss_list" in g and M is not None:
        assert np.array_equal(g["miss_list"][:M], ref["miss_list"]), "miss lists differ"
    if "attn_slot" in g:
        assert np.array_equal(g["attn_slot"].reshape(ref["attn_slot"].shape), ref["attn_slot"]), "attn_slot differs"
    if Kst is not None and M is not None:
        gk = from_bf16(Kst).reshape(-1, ref["Kst"].shape[1], ref["Kst"].shape[2])[:M]
        gv = from_bf16(Vst).reshape(-1, ref["Vst"].shape[1], ref["Vst"].shape[2])[:M]
        assert np.array_equal(gk, ref["Kst"]) and np.array_equal(gv, ref["Vst"]), "staged bytes differ"


def _bf16_bits(v: float) -> int:
    return int(synth.f32_to_bf16(np.array([v], np.float32))[0])


def tie_band_inputs():
    """A small step whose selections tie in fp32 but not in fp64.

    Per (request, KV head): k-1 chunks score far above the rest, and two
    chunks B < A (by index) come next.  The real query is 1 in coordinates 0
    and 1 (every head), so its score is G*2^16 + G*2^-9 for A and G*2^16 for
    B; 2^-7 is below half an fp32 ulp at 2^18, so fp32 sums see a tie (the
    lower index, B, wins) where fp64 keeps A.  The speculative query is 1 in
    coordinates 0 and 2, so it scores A and B exactly equal (both keep B).
    Returns (workload, host inputs, q, lm)."""
    w = Workload("tie_band", B=2, Hq=8, Hkv=2, d=128, L=1024, cs=16, k=8, n_q=2, spec_scale=(0.0, 0.3), seed=91,
                 residency="uniform", resident_frac=0.3)
    x = host_inputs(w)
    one = _bf16_bits(1.0)
    q = np.zeros((w.B, w.n_q, w.Hq, w.d), np.uint16)
    q[:, 0, :, 0] = q[:, 0, :, 1] = one                      # real query: coordinates 0 and 1
    q[:, 1, :, 0] = q[:, 1, :, 2] = one                      # speculative query: coordinates 0 and 2
    rng = np.random.default_rng(5)
    lm = synth.f32_to_bf16(rng.uniform(-1, 1, (w.B, w.Hkv, w.C, w.d)).astype(np.float32) * np.float32(0.01))
    lm[..., 0] = _bf16_bits(0.5)
    for b in range(w.B):
        for g in range(w.Hkv):
            perm = rng.permutation(w.C)
            big = perm[:w.k - 1]
            lo, hi = sorted(int(c) for c in perm[w.k - 1:w.k + 1])   # B = lo, A = hi
            lm[b, g, big, 0] = _bf16_bits(2.0 ** 17)
            lm[b, g, [lo, hi], :] = 0
            lm[b, g, [lo, hi], 0] = _bf16_bits(2.0 ** 16)
            lm[b, g, hi, 1] = _bf16_bits(2.0 ** -9)
    x["q"], x["lm"] = q, lm
    return w, x, q, lm
