"""Pins of the CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to a closed form, a library routine on a
special case, brute force on a tiny input, an invariant, or a number printed
on the pages, so that a dropped term, a wrong index or sign, or a transposed
operand in the oracle fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_kv_offload_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def enc(x):
    """fp32 -> bf16 bits through the generator module's encoder (not the oracle's)."""
    return synth.f32_to_bf16(np.asarray(x, dtype=np.float32))


# ---------------------------------------------------------------- eqs. (1)-(3)

def test_eq1_eq2_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "oasiskv_footprint.json")))
    per_token = oracle.kv_footprint_bytes(1, 1, g["n_layer"], g["n_kv"], g["d_h"], g["s_bytes"])
    assert per_token == g["bytes_per_token"] == 256 * 1024
    one_request = oracle.kv_footprint_bytes(1, g["context_tokens"], g["n_layer"], g["n_kv"], g["d_h"], g["s_bytes"])
    assert round(one_request / 1e9, 1) == g["request_gb_approx"]
    assert oracle.max_batch(g["hbm_gb"] * 10**9, g["context_tokens"], g["n_layer"], g["n_kv"], g["d_h"],
                            g["s_bytes"]) == g["max_batch"]
    # linear in B and L
    assert oracle.kv_footprint_bytes(3, 10, 2, 8, 128, 2) == 3 * 10 * oracle.kv_footprint_bytes(1, 1, 2, 8, 128, 2)


def test_eq3_step_budget():
    g = json.load(open(os.path.join(GOLDEN, "oasiskv_step_budget.json")))
    c = oracle.per_step_budget_bytes(g["b_link_bytes_per_s"], g["t_decode_s"])
    assert c == pytest.approx(1.088e9)
    m = g["qwen3_8b"]
    per_tok = oracle.kv_footprint_bytes(1, 1, m["n_layer"], m["n_kv"], m["d_h"], m["s_bytes"])
    implied_batch = c / per_tok / g["tokens_per_request"]
    assert 55 < implied_batch < 70


# ---------------------------------------------------------------- landmarks

def test_landmark_of_constant_chunk_is_the_key():
    rng = np.random.default_rng(0)
    B, H, cs, C, d = 2, 3, 16, 5, 128
    v = enc(rng.standard_normal((B, H, C, 1, d)))
    K = np.broadcast_to(v, (B, H, C, cs, d)).reshape(B, H, C * cs, d).copy()
    lm = oracle.build_landmarks(K, cs)
    assert np.array_equal(lm, v[:, :, :, 0, :])


def test_landmark_chunk_boundaries_and_heads():
    # K[b,g,t,i] = sign(b,g,i) * t: chunk c's mean is sign * (c*cs + (cs-1)/2), exact in bf16
    # (the largest mean, 119.5, still fits bf16's 8 significant bits)
    B, H, L, d, cs = 2, 4, 128, 128, 16
    t = np.arange(L, dtype=np.float32)
    sign = np.where((np.arange(B)[:, None, None] + np.arange(H)[None, :, None] + np.arange(d)[None, None, :]) % 2,
                    -1.0, 1.0).astype(np.float32)
    K = enc(sign[:, :, None, :] * t[None, None, :, None])
    lm = oracle.build_landmarks(K, cs)
    C = L // cs
    want = sign[:, :, None, :] * (np.arange(C, dtype=np.float32) * cs + (cs - 1) / 2)[None, None, :, None]
    assert np.array_equal(oracle.bf16_decode(lm), want.astype(np.float64))


@pytest.mark.parametrize("cs", [1, 4, 16, 64])
def test_landmark_equals_exact_mean_when_sums_are_exact(cs):
    # values on a 2^-7 grid within +-4: every fp32 partial sum is exact, so the
    # landmark is the bf16 rounding of the exact mean (numpy fp64 mean)
    rng = np.random.default_rng(cs)
    B, H, C, d = 1, 2, 7, 128
    x = np.clip(np.round(rng.standard_normal((B, H, C * cs, d)) * 128) / 128, -3.99, 3.99)
    K = enc(x)
    xf = synth.bf16_to_f32(K).astype(np.float64)
    mean = xf.reshape(B, H, C, cs, d).mean(axis=3)
    assert np.array_equal(oracle.build_landmarks(K, cs), enc(mean.astype(np.float32)))


# ---------------------------------------------------------------- scores

def test_score_one_hot_picks_the_right_head_and_coordinate():
    B, n_q, Hq, Hkv, C, d = 2, 2, 8, 2, 6, 128
    G = Hq // Hkv
    q = np.zeros((B, n_q, Hq, d), np.float32)
    lm = np.zeros((B, Hkv, C, d), np.float32)
    b, j, h, i = 1, 1, 6, 37          # head 6 belongs to KV head 1
    q[b, j, h, i] = 2.0
    lm[b, h // G, :, i] = np.arange(1, C + 1)
    lm[b, 0, :, i] = 100.0            # must not leak into KV head 1
    lm[b, h // G, :, i + 1] = 50.0    # other coordinate must not leak
    s = oracle.score_landmarks(enc(q), enc(lm))
    want = np.zeros((B, n_q, Hkv, C))
    want[b, j, h // G] = 2.0 * np.arange(1, C + 1)
    assert np.array_equal(s, want)


def test_score_with_constant_landmark_is_group_sum_of_query():
    rng = np.random.default_rng(3)
    B, n_q, Hq, Hkv, C, d = 2, 3, 12, 3, 5, 128
    G = Hq // Hkv
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    beta = np.array([1.0, -2.0, 0.5, 4.0, 0.0], np.float32)
    lm = enc(np.broadcast_to(beta[None, None, :, None], (B, Hkv, C, d)))
    s = oracle.score_landmarks(q, lm)
    qf = synth.bf16_to_f32(q).astype(np.float64)
    gsum = qf.reshape(B, n_q, Hkv, G, d).sum(axis=(3, 4))
    np.testing.assert_allclose(s, gsum[..., None] * beta[None, None, None, :], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- top-k

def _brute_topk(row, k):
    C = len(row)
    hits = []
    for S in itertools.combinations(range(C), k):
        inside = set(S)
        ok = all((row[a] > row[o]) or (row[a] == row[o] and a < o)
                 for a in inside for o in range(C) if o not in inside)
        if ok:
            hits.append(list(S))
    assert len(hits) == 1
    return hits[0]


@pytest.mark.parametrize("C,k", [(5, 1), (7, 3), (8, 4), (9, 8), (6, 6)])
def test_topk_brute_force(C, k):
    rng = np.random.default_rng(C * 10 + k)
    for trial in range(20):
        row = np.round(rng.standard_normal(C) * 2) / 2   # frequent exact ties
        got = oracle.select_topk(row[None, :], k)[0]
        assert list(got) == _brute_topk(row, k)


def test_topk_ties_take_lowest_index_and_output_is_ascending():
    s = np.array([[1.0, 2.0, 2.0, 2.0, 0.0, 2.0]])
    assert oracle.select_topk(s, 2).tolist() == [[1, 2]]
    assert oracle.select_topk(np.zeros((1, 9)), 4).tolist() == [[0, 1, 2, 3]]
    assert oracle.select_topk(np.array([[0.0, -0.0, 0.0]]), 1).tolist() == [[0]]
    s = np.array([[3.0, 9.0, 1.0, 7.0]])
    assert oracle.select_topk(s, 2).tolist() == [[1, 3]]
    assert oracle.select_topk(s, 4).tolist() == [[0, 1, 2, 3]]


# ---------------------------------------------------------------- union / residency

def test_union_worked_example_dedups_shared_rows():
    # Adaptive DHiSparse Fig. 3: K=4 queries, k=3; row a selected by three
    # queries, row b by two -- both must be fetched a single time.
    a, b_, C = 5, 9, 16
    sel = np.array([[[[a, b_, 1]], [[a, 2, 3]], [[a, b_, 4]], [[6, 7, 8]]]], dtype=np.int32)
    sel = np.sort(sel, axis=-1)
    res = oracle.resolve_union(sel, np.full((1, 1, C), -1, np.int32))
    U = [1, 2, 3, 4, a, 6, 7, 8, b_]
    assert res["union_cnt"][0, 0] == len(U) == res["miss_count"]
    assert res["union_idx"][0, 0, :len(U)].tolist() == sorted(U)
    assert sorted(res["miss_list"].tolist()) == sorted(U)
    qm = dict(zip(res["union_idx"][0, 0, :len(U)].tolist(), res["union_qmask"][0, 0, :len(U)].tolist()))
    assert bin(qm[a]).count("1") == 3 and bin(qm[b_]).count("1") == 2


def _check_union_invariants(sel, slot, res):
    B, n_q, Hkv, k = sel.shape
    C = slot.shape[2]
    expect_m = 0
    for b in range(B):
        for g in range(Hkv):
            sets = [set(sel[b, j, g].tolist()) for j in range(n_q)]
            U = sorted(set.union(*sets))
            n = res["union_cnt"][b, g]
            assert n == len(U) and k <= n <= min(C, n_q * k)
            assert res["union_idx"][b, g, :n].tolist() == U
            n_res = 0
            for u, c in enumerate(U):
                assert res["union_qmask"][b, g, u] == sum(1 << j for j in range(n_q) if c in sets[j])
                sl = res["union_slot"][b, g, u]
                if slot[b, g, c] >= 0:
                    assert sl == slot[b, g, c]
                    n_res += 1
                else:
                    assert sl == -(expect_m + 1)                      # dense, (b,g,c) order
                    assert res["miss_list"][expect_m] == (b * Hkv + g) * C + c
                    expect_m += 1
            for j in range(n_q):
                for r in range(k):
                    c = sel[b, j, g, r]
                    assert res["attn_slot"][b, j, g, r] == res["union_slot"][b, g, U.index(c)]
    assert res["miss_count"] == expect_m == len(res["miss_list"])


@pytest.mark.parametrize("n_q,overlap,res_frac", [(2, 0.7, 0.0), (2, 0.3, 0.5), (5, 0.5, 0.2), (1, 1.0, 0.9)])
def test_union_invariants(n_q, overlap, res_frac):
    B, Hkv, C, k = 3, 2, 40, 6
    sel = synth.random_selection(77 + n_q, B, n_q, Hkv, C, k, overlap)
    slot = synth.uniform_residency(5, B, Hkv, C, res_frac)
    res = oracle.resolve_union(sel, slot)
    _check_union_invariants(sel, slot, res)


# ---------------------------------------------------------------- gather

def test_gather_copies_exact_bytes():
    rng = np.random.default_rng(9)
    B, H, L, d, cs = 2, 3, 64, 128, 16
    C = L // cs
    Kh = rng.integers(0, 65535, (B, H, L, d), dtype=np.uint16)
    Vh = rng.integers(0, 65535, (B, H, L, d), dtype=np.uint16)
    miss = np.array([(1 * H + 2) * C + 3, 0, (0 * H + 1) * C + 2], np.int32)
    Kst, Vst = oracle.gather_kv(Kh, Vh, miss, cs)
    assert np.array_equal(Kst[0], Kh[1, 2, 48:64]) and np.array_equal(Vst[0], Vh[1, 2, 48:64])
    assert np.array_equal(Kst[1], Kh[0, 0, 0:16]) and np.array_equal(Vst[2], Vh[0, 1, 32:48])
    e = oracle.gather_kv(Kh, Vh, np.zeros(0, np.int32), cs)
    assert e[0].shape == (0, cs, d)


# ---------------------------------------------------------------- attention

def _sdpa(qf, Kf, Vf, scale):
    t = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qf)[None, None, None, :], torch.from_numpy(Kf)[None, None],
        torch.from_numpy(Vf)[None, None], scale=scale)
    return t[0, 0, 0].numpy()


def test_attention_all_chunks_equals_dense_sdpa():
    rng = np.random.default_rng(11)
    B, n_q, Hq, Hkv, L, d, cs = 2, 2, 4, 2, 64, 128, 16
    C = L // cs
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    Kh = enc(rng.standard_normal((B, Hkv, L, d)))
    Vh = enc(rng.standard_normal((B, Hkv, L, d)))
    sel = np.broadcast_to(np.arange(C, dtype=np.int32), (B, n_q, Hkv, C)).copy()
    res = oracle.resolve_union(sel, np.full((B, Hkv, C), -1, np.int32))
    Kst, Vst = oracle.gather_kv(Kh, Vh, res["miss_list"], cs)
    empty = np.zeros((0, cs, d), np.uint16)
    out = oracle.sparse_attn_decode(q, empty, empty, Kst, Vst, res["attn_slot"], cs)
    qf, Kf, Vf = (synth.bf16_to_f32(x).astype(np.float64) for x in (q, Kh, Vh))
    G = Hq // Hkv
    for b in range(B):
        for j in range(n_q):
            for h in range(Hq):
                want = _sdpa(qf[b, j, h], Kf[b, h // G], Vf[b, h // G], 1 / math.sqrt(d))
                np.testing.assert_allclose(out[b, j, h], want, rtol=1e-10, atol=1e-12)


def test_attention_single_row_and_uniform_weights():
    rng = np.random.default_rng(12)
    d = 128
    Vh = enc(rng.standard_normal((1, 1, 8, d)))
    Kh = enc(rng.standard_normal((1, 1, 8, d)))
    q = enc(rng.standard_normal((1, 1, 1, d)))
    # cs = 1, k = 1: the output is the selected V row
    sel = np.array([[[[5]]]], np.int32)
    res = oracle.resolve_union(sel, np.full((1, 1, 8), -1, np.int32))
    Kst, Vst = oracle.gather_kv(Kh, Vh, res["miss_list"], 1)
    out = oracle.sparse_attn_decode(q, Kst[:0], Vst[:0], Kst, Vst, res["attn_slot"], 1)
    assert np.array_equal(out[0, 0, 0], synth.bf16_to_f32(Vh[0, 0, 5]).astype(np.float64))
    # q = 0: equal logits, the output is the mean of the selected V rows
    sel = np.array([[[[1, 4, 6]]]], np.int32)
    res = oracle.resolve_union(sel, np.full((1, 1, 8), -1, np.int32))
    Kst, Vst = oracle.gather_kv(Kh, Vh, res["miss_list"], 1)
    out = oracle.sparse_attn_decode(np.zeros_like(q), Kst[:0], Vst[:0], Kst, Vst, res["attn_slot"], 1)
    want = synth.bf16_to_f32(Vh[0, 0, [1, 4, 6]]).astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(out[0, 0, 0], want, rtol=1e-12, atol=1e-14)


def test_attention_uses_floor_h_over_G_and_is_order_invariant():
    rng = np.random.default_rng(13)
    B, n_q, Hq, Hkv, d, cs, S = 1, 1, 6, 3, 128, 4, 10
    Khot = enc(rng.standard_normal((S, cs, d)))
    # V of the chunks of KV head g is the constant g+1, so a zero query gives g+1
    Vhot = enc(np.repeat(np.arange(S, dtype=np.float32)[:, None, None], cs, 1) * np.ones((1, 1, d), np.float32))
    slots = np.array([[[[0, 1], [3, 4], [7, 8]]]], np.int32)       # [B,n_q,Hkv,k]
    zero = np.zeros((B, n_q, Hq, d), np.uint16)
    out = oracle.sparse_attn_decode(zero, Khot, Vhot, Khot[:0], Vhot[:0], slots, cs)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        assert np.all(out[0, 0, h] == slots[0, 0, g].mean())
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    Vhot = enc(rng.standard_normal((S, cs, d)))
    a = oracle.sparse_attn_decode(q, Khot, Vhot, Khot[:0], Vhot[:0], slots, cs)
    b = oracle.sparse_attn_decode(q, Khot, Vhot, Khot[:0], Vhot[:0], slots[..., ::-1].copy(), cs)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- whole step

@pytest.mark.parametrize("resident_frac", [0.0, 0.5])
def test_step_with_all_chunks_equals_dense_attention(resident_frac):
    w = dict(B=1, n_q=2, Hq=4, Hkv=2, L=128, d=128, cs=16)
    C = w["L"] // w["cs"]
    rng = np.random.default_rng(21)
    q = enc(rng.standard_normal((w["B"], w["n_q"], w["Hq"], w["d"])))
    Kh = enc(rng.standard_normal((w["B"], w["Hkv"], w["L"], w["d"])))
    Vh = enc(rng.standard_normal((w["B"], w["Hkv"], w["L"], w["d"])))
    lm = oracle.build_landmarks(Kh, w["cs"])
    slot = synth.uniform_residency(3, w["B"], w["Hkv"], C, resident_frac)
    Khot = synth.hot_pool_from(Kh, slot, w["cs"]) if resident_frac else np.zeros((0, w["cs"], w["d"]), np.uint16)
    Vhot = synth.hot_pool_from(Vh, slot, w["cs"]) if resident_frac else np.zeros((0, w["cs"], w["d"]), np.uint16)
    r = oracle.step(q, lm, Kh, Vh, slot, Khot, Vhot, C, w["cs"])
    assert r["miss_count"] == int((slot < 0).sum())
    qf, Kf, Vf = (synth.bf16_to_f32(x).astype(np.float64) for x in (q, Kh, Vh))
    G = w["Hq"] // w["Hkv"]
    for j in range(w["n_q"]):
        for h in range(w["Hq"]):
            want = _sdpa(qf[0, j, h], Kf[0, h // G], Vf[0, h // G], 1 / math.sqrt(w["d"]))
            np.testing.assert_allclose(r["out"][0, j, h], want, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- min/max landmarks (Quest-style)

def _total_key(x):
    """Python ordering of a float with -0 below +0."""
    return (x, math.copysign(1.0, x))


def test_minmax_landmarks_brute_force_with_signed_zeros():
    rng = np.random.default_rng(11)
    B, H, cs, C, d = 2, 2, 4, 3, 5
    K = enc(rng.standard_normal((B, H, C * cs, d)))
    # one chunk holds both zeros in one coordinate, another only -0 and +0 mixed with negatives
    K[0, 1, 0:4, 2] = [0x8000, 0x0000, 0x8000, 0x0000]
    K[1, 0, 4:8, 0] = [0x0000, 0xBF80, 0x8000, 0x0000]   # +0, -1, -0, +0
    lm2 = oracle.build_minmax_landmarks(K, cs)
    assert lm2.shape == (B, H, C, 2, d) and lm2.dtype == np.uint16
    vals = synth.bf16_to_f32(K).astype(np.float64)
    for b, h, c, i in itertools.product(range(B), range(H), range(C), range(d)):
        col = [(vals[b, h, c * cs + t, i], K[b, h, c * cs + t, i]) for t in range(cs)]
        lo = min(col, key=lambda e: _total_key(e[0]))[1]
        hi = max(col, key=lambda e: _total_key(e[0]))[1]
        assert lm2[b, h, c, 0, i] == lo and lm2[b, h, c, 1, i] == hi, (b, h, c, i)
    assert lm2[0, 1, 0, 0, 2] == 0x8000 and lm2[0, 1, 0, 1, 2] == 0x0000
    assert lm2[1, 0, 1, 0, 0] == 0xBF80 and lm2[1, 0, 1, 1, 0] == 0x0000


def test_minmax_landmarks_of_one_token_chunks_are_the_keys():
    rng = np.random.default_rng(12)
    K = enc(rng.standard_normal((1, 3, 7, 128)))
    lm2 = oracle.build_minmax_landmarks(K, 1)
    assert np.array_equal(lm2[:, :, :, 0, :], K) and np.array_equal(lm2[:, :, :, 1, :], K)


def test_minmax_score_is_best_corner_of_the_box():
    # brute force over all 2^d corners of each chunk's box, group sum done by hand
    rng = np.random.default_rng(13)
    B, n_q, Hq, Hkv, C, cs, d = 2, 2, 4, 2, 3, 4, 5
    G = Hq // Hkv
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    K = enc(rng.standard_normal((B, Hkv, C * cs, d)))
    lm2 = oracle.build_minmax_landmarks(K, cs)
    s = oracle.score_minmax_landmarks(q, lm2)
    qf = synth.bf16_to_f32(q).astype(np.float64)
    lf = synth.bf16_to_f32(lm2).astype(np.float64)
    for b, j, g, c in itertools.product(range(B), range(n_q), range(Hkv), range(C)):
        Q = sum(qf[b, j, h] for h in range(g * G, (g + 1) * G))
        best = max(sum(Q[i] * lf[b, g, c, pick[i], i] for i in range(d))
                   for pick in itertools.product((0, 1), repeat=d))
        assert math.isclose(s[b, j, g, c], best, rel_tol=1e-12, abs_tol=1e-12), (b, j, g, c)


def test_minmax_score_bounds_every_token_and_is_attained_at_the_corner():
    rng = np.random.default_rng(14)
    B, n_q, Hq, Hkv, C, cs, d = 2, 3, 8, 2, 6, 8, 128
    G = Hq // Hkv
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    K = enc(rng.standard_normal((B, Hkv, C * cs, d)))
    qf = synth.bf16_to_f32(q).astype(np.float64)
    Q = qf.reshape(B, n_q, Hkv, G, d).sum(axis=3)
    # chunk 2 of (b=1, g=0) gets, as token 5, the corner that query j=1 prefers
    kf = synth.bf16_to_f32(K).astype(np.float64)
    blk = kf[1, 0, 2 * cs:3 * cs]
    corner = np.where(Q[1, 1, 0] >= 0, blk.max(axis=0), blk.min(axis=0))
    K[1, 0, 2 * cs + 5] = enc(corner)
    kf = synth.bf16_to_f32(K).astype(np.float64)
    s = oracle.score_minmax_landmarks(q, oracle.build_minmax_landmarks(K, cs))
    dots = np.einsum("bjgi,bgti->bjgt", Q, kf).reshape(B, n_q, Hkv, C, cs)
    assert np.all(s >= dots.max(axis=-1) - 1e-9 * np.abs(s))
    assert math.isclose(s[1, 1, 0, 2], dots[1, 1, 0, 2, 5], rel_tol=1e-12)


def test_minmax_score_with_one_token_chunks_equals_mean_score():
    rng = np.random.default_rng(15)
    B, n_q, Hq, Hkv, L, d = 2, 2, 8, 2, 9, 128
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    K = enc(rng.standard_normal((B, Hkv, L, d)))
    s_mm = oracle.score_minmax_landmarks(q, oracle.build_minmax_landmarks(K, 1))
    s_mean = oracle.score_landmarks(q, oracle.build_landmarks(K, 1))
    np.testing.assert_allclose(s_mm, s_mean, rtol=1e-12, atol=1e-12)


def test_minmax_score_with_same_sign_query_uses_one_bound():
    rng = np.random.default_rng(16)
    B, n_q, Hq, Hkv, C, cs, d = 1, 2, 4, 1, 5, 4, 128
    q = np.abs(rng.standard_normal((B, n_q, Hq, d))).astype(np.float32)
    q[:, 1] = -q[:, 1]                              # query 0 all positive, query 1 all negative
    q = enc(q)
    K = enc(rng.standard_normal((B, Hkv, C * cs, d)))
    lm2 = oracle.build_minmax_landmarks(K, cs)
    s = oracle.score_minmax_landmarks(q, lm2)
    Q = synth.bf16_to_f32(q).astype(np.float64).sum(axis=2)       # G = Hq, one KV head
    lf = synth.bf16_to_f32(lm2).astype(np.float64)
    np.testing.assert_allclose(s[0, 0, 0], lf[0, 0, :, 1, :] @ Q[0, 0], rtol=1e-12)
    np.testing.assert_allclose(s[0, 1, 0], lf[0, 0, :, 0, :] @ Q[0, 1], rtol=1e-12)


def test_step_with_minmax_landmarks_selects_by_the_bound():
    rng = np.random.default_rng(17)
    B, n_q, Hq, Hkv, C, cs, d, k = 1, 2, 4, 2, 6, 4, 128, 2
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    Kh = enc(rng.standard_normal((B, Hkv, C * cs, d)))
    Vh = enc(rng.standard_normal((B, Hkv, C * cs, d)))
    lm2 = oracle.build_minmax_landmarks(Kh, cs)
    slot = np.full((B, Hkv, C), -1, np.int32)
    r = oracle.step(q, lm2, Kh, Vh, slot, None, None, k, cs)
    assert np.array_equal(r["scores"], oracle.score_minmax_landmarks(q, lm2))
    assert np.array_equal(r["sel"], oracle.select_topk(r["scores"], k))


# ---------------------------------------------------------------- tail rows (the step's own tokens)

def test_attention_tail_rows_equal_dense_causal_sdpa():
    # every chunk selected + the n_q new tokens appended with a causal mask among them
    rng = np.random.default_rng(21)
    B, n_q, Hq, Hkv, L, d, cs = 2, 3, 4, 2, 64, 128, 16
    C = L // cs
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    Kh = enc(rng.standard_normal((B, Hkv, L, d)))
    Vh = enc(rng.standard_normal((B, Hkv, L, d)))
    Kt = enc(rng.standard_normal((B, n_q, Hkv, d)))
    Vt = enc(rng.standard_normal((B, n_q, Hkv, d)))
    sel = np.broadcast_to(np.arange(C, dtype=np.int32), (B, n_q, Hkv, C)).copy()
    res = oracle.resolve_union(sel, np.full((B, Hkv, C), -1, np.int32))
    Kst, Vst = oracle.gather_kv(Kh, Vh, res["miss_list"], cs)
    empty = np.zeros((0, cs, d), np.uint16)
    out = oracle.sparse_attn_decode(q, empty, empty, Kst, Vst, res["attn_slot"], cs, K_tail=Kt, V_tail=Vt)
    G = Hq // Hkv
    qf, Kf, Vf, Ktf, Vtf = (torch.from_numpy(synth.bf16_to_f32(x).astype(np.float64)) for x in (q, Kh, Vh, Kt, Vt))
    # sequence = L context rows then the n_q new tokens; query j sits at position L + j
    Kseq = torch.cat([Kf, Ktf.permute(0, 2, 1, 3)], dim=2)             # [B, Hkv, L + n_q, d]
    Vseq = torch.cat([Vf, Vtf.permute(0, 2, 1, 3)], dim=2)
    Kseq = Kseq.repeat_interleave(G, dim=1)                              # query head h -> KV head h // G
    Vseq = Vseq.repeat_interleave(G, dim=1)
    Q = qf.permute(0, 2, 1, 3)                                           # [B, Hq, n_q, d]
    pos_q = L + torch.arange(n_q)[:, None]
    mask = torch.arange(L + n_q)[None, :] <= pos_q                       # causal
    want = torch.nn.functional.scaled_dot_product_attention(Q, Kseq, Vseq, attn_mask=mask, scale=1 / math.sqrt(d))
    np.testing.assert_allclose(out, want.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12)


def test_attention_tail_row_of_a_later_token_is_masked():
    # a later token's tail row with an enormous logit must not reach an earlier query
    rng = np.random.default_rng(22)
    B, n_q, Hq, Hkv, d, cs, S = 1, 2, 2, 1, 128, 4, 3
    Khot = enc(rng.standard_normal((S, cs, d)) * 0.1)
    Vhot = enc(rng.standard_normal((S, cs, d)))
    q = enc(np.ones((B, n_q, Hq, d), np.float32))
    Kt = enc(np.stack([np.zeros((1, d)), np.full((1, d), 8.0)], axis=0)[None].astype(np.float32))  # [1,2,1,d]
    Vt = enc(np.stack([np.zeros((1, d)), np.full((1, d), 5.0)], axis=0)[None].astype(np.float32))
    slots = np.array([[[[0, 2]], [[0, 2]]]], np.int32)
    out = oracle.sparse_attn_decode(q, Khot, Vhot, Khot[:0], Vhot[:0], slots, cs, K_tail=Kt, V_tail=Vt)
    base = oracle.sparse_attn_decode(q, Khot, Vhot, Khot[:0], Vhot[:0], slots, cs)
    # query 0 sees only its own tail row (K = V = 0): the context output diluted by that one zero row
    z = (synth.bf16_to_f32(Khot[[0, 2]]).astype(np.float64).reshape(-1, d) @ np.ones(d)) / math.sqrt(d)
    w0 = np.exp(z - z.max()).sum() / (np.exp(z - z.max()).sum() + np.exp(-z.max()))
    np.testing.assert_allclose(out[0, 0], w0 * base[0, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out[0, 1], 5.0, rtol=0, atol=1e-9)   # its own row dominates (logit 8*128/sqrt(128))


def test_attention_with_no_selected_chunk_is_causal_sdpa_over_the_tail_rows():
    # a query with no selected chunk attends to tail rows 0..j alone; with no tail either, zero
    rng = np.random.default_rng(23)
    B, n_q, Hq, Hkv, d, cs = 1, 3, 4, 2, 128, 16
    G = Hq // Hkv
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    Kt = enc(rng.standard_normal((B, n_q, Hkv, d)))
    Vt = enc(rng.standard_normal((B, n_q, Hkv, d)))
    none = np.full((B, n_q, Hkv, 2), oracle.NO_SLOT, np.int32)
    empty = np.zeros((0, cs, d), np.uint16)
    out = oracle.sparse_attn_decode(q, empty, empty, empty, empty, none, cs, K_tail=Kt, V_tail=Vt)
    qf, Ktf, Vtf = (torch.from_numpy(synth.bf16_to_f32(x).astype(np.float64)) for x in (q, Kt, Vt))
    Kseq = Ktf.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)           # [B, Hq, n_q, d]
    Vseq = Vtf.permute(0, 2, 1, 3).repeat_interleave(G, dim=1)
    mask = torch.arange(n_q)[None, :] <= torch.arange(n_q)[:, None]      # query j sees tokens 0..j
    want = torch.nn.functional.scaled_dot_product_attention(qf.permute(0, 2, 1, 3), Kseq, Vseq, attn_mask=mask,
                                                            scale=1 / math.sqrt(d))
    np.testing.assert_allclose(out, want.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12)
    assert np.all(oracle.sparse_attn_decode(q, empty, empty, empty, empty, none, cs) == 0)


# ---------------------------------------------------------------- residency update (delta selection, capped LRU)

def _res_step(state, union, step_id, cap, cs=1, d=2):
    """Resolve `union` (one request, one KV head, one query) against the state and
    update; staging rows of ordinal m hold the value 16*step + m (exact in bf16)."""
    C = state["resident_slot"].shape[-1]
    sel = np.array(sorted(union), np.int32)[None, None, None, :]
    res = oracle.resolve_union(sel, state["resident_slot"])
    M = res["miss_count"]
    Kst = enc(np.repeat((16.0 * step_id + np.arange(M, dtype=np.float32))[:, None, None], cs, 1)
              * np.ones((1, 1, d), np.float32))
    new = oracle.update_residency(step_id, cap, res["union_idx"], res["union_slot"], res["union_cnt"], Kst, Kst,
                                  state["resident_slot"], state["slot_chunk"], state["last_used"],
                                  state["Khot"], state["Vhot"])
    return new, res


def test_residency_worked_example():
    S, C, cs, d = 3, 10, 1, 2
    st = {"resident_slot": np.full((1, 1, C), -1, np.int32), "slot_chunk": np.full((1, 1, S), -1, np.int32),
          "last_used": np.full((1, 1, S), -1, np.int32), "Khot": np.zeros((S, cs, d), np.uint16),
          "Vhot": np.zeros((S, cs, d), np.uint16)}
    # step 0: four misses, cap 2 -> chunks 2 and 5 into the free slots 0 and 1
    st, res = _res_step(st, [2, 5, 7, 9], 0, cap=2)
    assert res["miss_count"] == 4 and st["admitted"][0, 0] == 2
    assert st["slot_chunk"][0, 0].tolist() == [2, 5, -1] and st["last_used"][0, 0].tolist() == [0, 0, -1]
    assert st["resident_slot"][0, 0, [2, 5, 7, 9]].tolist() == [0, 1, -1, -1]
    assert synth.bf16_to_f32(st["Khot"][:2, 0, 0]).tolist() == [0.0, 1.0]       # staging ordinals 0, 1
    # step 1: 2 is resident (refreshed), 7 goes to the last free slot
    st, res = _res_step(st, [2, 7], 1, cap=2)
    assert res["miss_count"] == 1
    assert st["slot_chunk"][0, 0].tolist() == [2, 5, 7] and st["last_used"][0, 0].tolist() == [1, 0, 1]
    assert synth.bf16_to_f32(st["Khot"][2, 0, 0]) == 16.0
    # step 2: 7 resident; misses 1, 3; evict LRU first: slot 1 (chunk 5, step 0), then slot 0 (chunk 2, step 1)
    st, res = _res_step(st, [1, 3, 7], 2, cap=2)
    assert st["slot_chunk"][0, 0].tolist() == [3, 1, 7] and st["last_used"][0, 0].tolist() == [2, 2, 2]
    assert st["resident_slot"][0, 0, [1, 2, 3, 5, 7]].tolist() == [1, -1, 0, -1, 2]
    assert synth.bf16_to_f32(st["Khot"][:, 0, 0]).tolist() == [33.0, 32.0, 16.0]
    # step 3: every slot holds a chunk of the union -> nothing can be evicted
    st, res = _res_step(st, [0, 1, 3, 7, 8], 3, cap=1)
    assert res["miss_count"] == 2 and st["admitted"][0, 0] == 0
    assert st["slot_chunk"][0, 0].tolist() == [3, 1, 7] and st["last_used"][0, 0].tolist() == [3, 3, 3]


@pytest.mark.parametrize("S,cap", [(4, 2), (16, 3), (40, 100)])
def test_residency_invariants_over_random_steps(S, cap):
    rng = np.random.default_rng(23 + S)
    B, Hkv, n_q, C, k, cs, d = 2, 2, 2, 48, 6, 2, 4
    units = B * Hkv
    Kh = enc(rng.standard_normal((B, Hkv, C * cs, d)))
    Vh = enc(rng.standard_normal((B, Hkv, C * cs, d)))
    rs = np.full((B, Hkv, C), -1, np.int32)
    sc = np.full((B, Hkv, S), -1, np.int32)
    lu = np.full((B, Hkv, S), -1, np.int32)
    Khot = np.zeros((units * S, cs, d), np.uint16)
    Vhot = np.zeros((units * S, cs, d), np.uint16)
    hot_pref = rng.permutation(C)[:10]                       # temporal locality: a hot set picked often
    for step_id in range(12):
        sel = np.empty((B, n_q, Hkv, k), np.int32)
        for idx in np.ndindex(B, n_q, Hkv):
            pool = np.concatenate([hot_pref, rng.permutation(C)[:k]])
            sel[idx] = np.sort(rng.choice(np.unique(pool), size=k, replace=False))
        res = oracle.resolve_union(sel, rs)
        Kst, Vst = oracle.gather_kv(Kh, Vh, res["miss_list"], cs)
        new = oracle.update_residency(step_id, cap, res["union_idx"], res["union_slot"], res["union_cnt"], Kst, Vst,
                                      rs, sc, lu, Khot, Vhot)
        for u in range(units):
            b, g = divmod(u, Hkv)
            n = int(res["union_cnt"][b, g])
            U = res["union_idx"][b, g, :n]
            slots = res["union_slot"][b, g, :n]
            n_miss = int((slots < 0).sum())
            old_sc, new_sc = sc[b, g], new["slot_chunk"][b, g]
            union_res = {int(s) - u * S for s in slots if s >= 0}
            n_free = int((old_sc < 0).sum())
            n_evictable = int(((old_sc >= 0) & ~np.isin(np.arange(S), list(union_res))).sum())
            A = int(new["admitted"][b, g])
            assert A == min(cap, n_miss, n_free + n_evictable)          # the cap bounds the traffic
            for t in union_res:                                          # union residents stay, refreshed
                assert new_sc[t] == old_sc[t] and new["last_used"][b, g, t] == step_id
            admitted = set(U[slots < 0][:A].tolist())                    # lowest missing chunks first
            assert admitted == {int(c) for c in new_sc if c >= 0} - {int(c) for c in old_sc if c >= 0}
            evicted = [t for t in range(S) if old_sc[t] >= 0 and new_sc[t] != old_sc[t]]
            kept = [t for t in range(S) if old_sc[t] >= 0 and new_sc[t] == old_sc[t] and t not in union_res]
            assert len(evicted) == max(0, A - n_free)                    # free slots go first
            for e in evicted:                                            # least recently used go first
                for kk in kept:
                    assert (lu[b, g, e], e) < (lu[b, g, kk], kk)
            # maps stay inverse and every resident chunk's hot rows are its host rows
            for t in range(S):
                c = int(new_sc[t])
                if c >= 0:
                    assert new["resident_slot"][b, g, c] == u * S + t
                    assert np.array_equal(new["Khot"][u * S + t], Kh[b, g, c * cs:(c + 1) * cs])
                    assert np.array_equal(new["Vhot"][u * S + t], Vh[b, g, c * cs:(c + 1) * cs])
            assert int((new["resident_slot"][b, g] >= 0).sum()) == int((new_sc >= 0).sum())
        rs, sc, lu, Khot, Vhot = (new[x] for x in ("resident_slot", "slot_chunk", "last_used", "Khot", "Vhot"))


def test_residency_repeated_selection_needs_no_transfer():
    # delta selection: once admitted, a repeated selection resolves entirely in HBM
    rng = np.random.default_rng(24)
    B, Hkv, n_q, C, k, cs, d, S = 1, 2, 2, 32, 5, 2, 4, 12
    Kh = enc(rng.standard_normal((B, Hkv, C * cs, d)))
    sel = np.sort(rng.permuted(np.tile(np.arange(C, dtype=np.int32), (B, n_q, Hkv, 1)), axis=-1)[..., :k], axis=-1)
    rs = np.full((B, Hkv, C), -1, np.int32)
    state = (rs, np.full((B, Hkv, S), -1, np.int32), np.full((B, Hkv, S), -1, np.int32),
             np.zeros((B * Hkv * S, cs, d), np.uint16), np.zeros((B * Hkv * S, cs, d), np.uint16))
    res = oracle.resolve_union(sel, rs)
    Kst, Vst = oracle.gather_kv(Kh, Kh, res["miss_list"], cs)
    new = oracle.update_residency(0, S, res["union_idx"], res["union_slot"], res["union_cnt"], Kst, Vst, *state)
    again = oracle.resolve_union(sel, new["resident_slot"])
    assert res["miss_count"] == int(res["union_cnt"].sum()) and again["miss_count"] == 0


# ---------------------------------------------------------------- predictive prefetch

@pytest.mark.parametrize("overlap", [1.0, 0.6, 0.0])
def test_prefetch_changes_no_output_and_leaves_only_unpredicted_misses(overlap):
    # the prediction only moves transfers ahead of time: the step's output is the
    # output without prefetch, and the urgent misses are the true union minus the predicted one
    rng = np.random.default_rng(31)
    B, n_q, Hq, Hkv, L, d, cs, k = 2, 2, 4, 2, 256, 128, 16, 5
    C = L // cs
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    Kh = enc(rng.standard_normal((B, Hkv, L, d)))
    Vh = enc(rng.standard_normal((B, Hkv, L, d)))
    lm = oracle.build_landmarks(Kh, cs)
    true_sel = oracle.select_topk(oracle.score_landmarks(q, lm), k)
    pred = np.empty((B, 1, Hkv, k), np.int32)
    for b, g in np.ndindex(B, Hkv):
        keep = int(round(overlap * k))
        own = list(true_sel[b, 0, g][:keep])
        rest = [c for c in rng.permutation(C) if c not in set(true_sel[b, 0, g])][:k - keep]
        pred[b, 0, g] = np.sort(np.array(own + rest, np.int32))
    pf = oracle.prefetch_kv(pred, Kh, Vh, cs)
    assert pf["count"] == sum(len(set(pred[b, 0, g])) for b, g in np.ndindex(B, Hkv))
    for b, g, c in np.ndindex(B, Hkv, C):              # the map points at the chunk's host rows
        m = pf["pf_map"][b, g, c]
        assert (m >= 0) == (c in set(pred[b, 0, g]))
        if m >= 0:
            assert np.array_equal(pf["K"][m], Kh[b, g, c * cs:(c + 1) * cs])
            assert np.array_equal(pf["V"][m], Vh[b, g, c * cs:(c + 1) * cs])
    plain = oracle.step(q, lm, Kh, Vh, np.full((B, Hkv, C), -1, np.int32), None, None, k, cs)
    with_pf = oracle.step(q, lm, Kh, Vh, pf["pf_map"], pf["K"], pf["V"], k, cs)
    np.testing.assert_allclose(with_pf["out"], plain["out"], rtol=1e-12, atol=1e-14)
    urgent = sum(len(set(oracle.union_of_query_selections(true_sel, b, g)) - set(pred[b, 0, g]))
                 for b, g in np.ndindex(B, Hkv))
    assert with_pf["miss_count"] == urgent


# ---------------------------------------------------------------- coverage budgets (MOIRA reading)

def _mass(row, tau):
    w = np.exp(tau * (row - row.max()))
    return w / w.sum()


@pytest.mark.parametrize("gamma", [0.3, 0.6, 0.9, 0.99])
def test_mass_selection_is_the_smallest_set_by_brute_force(gamma):
    rng = np.random.default_rng(41)
    C, tau = 8, 0.7
    s = rng.standard_normal((5, C)) * 2.0
    s[4, 3] = s[4, 5]                                     # a tie: the lower index ranks first
    sel, cnt = oracle.select_by_mass(s, C, gamma, tau)
    for r in range(s.shape[0]):
        w = _mass(s[r], tau)
        best = None
        for size in range(1, C + 1):                      # the least size some subset reaching gamma has
            if any(w[list(sub)].sum() >= gamma for sub in itertools.combinations(range(C), size)):
                best = size
                break
        assert cnt[r] == best
        chosen = sel[r, :cnt[r]]
        assert list(chosen) == sorted(chosen) and np.all(sel[r, cnt[r]:] == -1)
        assert w[chosen].sum() >= gamma
        # the chosen set is the top cnt[r] by (score desc, index asc)
        order = sorted(range(C), key=lambda c: (-s[r, c], c))
        assert set(chosen.tolist()) == set(order[:cnt[r]])


def test_mass_selection_uniform_peaked_and_clamped():
    C = 16
    flat = np.zeros((1, C))
    for gamma, want in ((0.5, 8), (0.25, 4), (0.26, 5), (1.0, 16)):
        assert oracle.select_by_mass(flat, C, gamma, 1.0)[1][0] == want      # ceil(gamma * C)
    peaked = np.zeros((1, C))
    peaked[0, 9] = 100.0
    sel, cnt = oracle.select_by_mass(peaked, C, 0.99, 1.0)
    assert cnt[0] == 1 and sel[0, 0] == 9
    assert oracle.select_by_mass(peaked, C, 0.99, 1.0, k_min=3)[1][0] == 3   # clamped below
    assert oracle.select_by_mass(flat, 6, 0.9, 1.0)[1][0] == 6               # clamped above (k_max)


def test_padded_rows_resolve_and_attend_like_shorter_rows():
    rng = np.random.default_rng(42)
    B, n_q, Hq, Hkv, C, cs, d = 1, 2, 4, 2, 12, 4, 128
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    Kh = enc(rng.standard_normal((B, Hkv, C * cs, d)))
    Vh = enc(rng.standard_normal((B, Hkv, C * cs, d)))
    rows = {(0, 0): [1, 4, 7], (0, 1): [0, 2, 4, 6, 8], (1, 0): [3], (1, 1): [4, 5, 10]}
    sel = np.full((B, n_q, Hkv, 5), -1, np.int32)
    for (j, g), cs_ in rows.items():
        sel[0, j, g, :len(cs_)] = cs_
    res = oracle.resolve_union(sel, np.full((B, Hkv, C), -1, np.int32))
    assert res["union_cnt"].tolist() == [[4, 7]]                              # {1,3,4,7}, {0,2,4,5,6,8,10}
    assert np.all(res["attn_slot"][sel < 0] == oracle.NO_SLOT) and np.all(res["attn_slot"][sel >= 0] < 0)
    Kst, Vst = oracle.gather_kv(Kh, Vh, res["miss_list"], cs)
    out = oracle.sparse_attn_decode(q, Kst[:0], Vst[:0], Kst, Vst, res["attn_slot"], cs)
    G = Hq // Hkv
    qf, Kf, Vf = (synth.bf16_to_f32(x).astype(np.float64) for x in (q, Kh, Vh))
    for (j, g), chunks in rows.items():
        idx = np.concatenate([np.arange(c * cs, (c + 1) * cs) for c in chunks])
        for h in range(g * G, (g + 1) * G):
            want = _sdpa(qf[0, j, h], Kf[0, g, idx], Vf[0, g, idx], 1 / math.sqrt(d))
            np.testing.assert_allclose(out[0, j, h], want, rtol=1e-10, atol=1e-12)


def test_step_with_coverage_budget_uses_the_head_logit_scale():
    rng = np.random.default_rng(43)
    B, n_q, Hq, Hkv, L, d, cs, k = 1, 2, 8, 2, 256, 128, 16, 12
    q = enc(rng.standard_normal((B, n_q, Hq, d)))
    Kh = enc(rng.standard_normal((B, Hkv, L, d)))
    lm = oracle.build_landmarks(Kh, cs)
    r = oracle.step(q, lm, Kh, Kh, np.full((B, Hkv, L // cs), -1, np.int32), None, None, k, cs, gamma=0.8)
    sel, cnt = oracle.select_by_mass(oracle.score_landmarks(q, lm), k, 0.8, 1 / math.sqrt(d) / (Hq // Hkv))
    assert np.array_equal(r["sel"], sel) and np.array_equal(r["sel_cnt"], cnt)
