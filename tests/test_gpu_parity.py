"""GPU parity of every stage of the decode step against the CPU oracle.

Each test feeds the same seeded inputs to the CUDA library (through the C ABI
binding) and to the oracle and compares: bit-exact for landmarks, indices,
union/miss layouts and gathered bytes; within the stated tolerances for
scores and attention.
"""
import math

import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300 import synth
from sparse_kv_offload_gb300.workloads import GQA32B_5Q, LLAMA8B_32K, QWEN8B_128K, STRESS_512K, TINY, Workload

import dd_testlib as tl

pytestmark = pytest.mark.gpu

# reduced-size versions of the five workloads (several tiles and ragged tails,
# small enough for the oracle), plus degenerate shapes
V_HOT = LLAMA8B_32K.scaled(name="llama_hot_small", B=2, L=8192, k=48)
V_CARRY = QWEN8B_128K.scaled(name="qwen_carry_small", B=2, L=8192, k=24)
V_5Q = GQA32B_5Q.scaled(name="gqa32b_5q_small", B=2, L=4096, k=40)
V_ZIPF = STRESS_512K.scaled(name="stress_zipf_small", B=1, L=16384, k=16)
V_NQ64 = Workload("nq64", B=1, Hq=64, Hkv=8, d=128, L=4096, cs=16, k=16, n_q=8,
                  spec_scale=(0.0,) + (0.1,) * 7, seed=77)
V_ALL = Workload("k_equals_C", B=1, Hq=8, Hkv=2, d=128, L=1024, cs=16, k=64, n_q=2,
                 spec_scale=(0.0, 0.3), seed=78)
V_ONEQ = Workload("one_query", B=3, Hq=16, Hkv=4, d=128, L=2048, cs=32, k=7, n_q=1, seed=79,
                  residency="uniform", resident_frac=0.25)
# C = 1000: a ragged last landmark stage, union words not a multiple of 32, three queries
V_ODD = Workload("odd_c", B=3, Hq=12, Hkv=3, d=128, L=16000, cs=16, k=37, n_q=3, spec_scale=(0.0, 0.2, 0.4),
                 seed=83, residency="uniform", resident_frac=0.3)
# 128 (request, KV head) units fill most of the 152 SMs in one wave: the step
# then scores inside the selection kernel on the tensor cores (C = 200: a
# ragged second landmark tile; 2, 5 and 8 queries, N = 16 and 32)
V_FOLD2 = Workload("fold_nq2", B=16, Hq=32, Hkv=8, d=128, L=3200, cs=16, k=16, n_q=2, spec_scale=(0.0, 0.3),
                   seed=91, residency="uniform", resident_frac=0.4)
V_FOLD5 = Workload("fold_nq5", B=16, Hq=64, Hkv=8, d=128, L=4096, cs=16, k=24, n_q=5,
                   spec_scale=(0.0, 0.2, 0.4, 0.6, 0.8), seed=92)
V_FOLD8 = Workload("fold_nq8", B=16, Hq=32, Hkv=8, d=128, L=2048, cs=16, k=8, n_q=8,
                   spec_scale=(0.0,) + (0.1,) * 7, seed=93, residency="uniform", resident_frac=0.5)
# 384 units: more selection CTAs than fit on the device at once (two per SM),
# so the selection sums the earlier units' counts by its look-back instead of
# leaving them to the last CTA to arrive
V_WAVES = Workload("two_waves", B=48, Hq=16, Hkv=8, d=128, L=512, cs=16, k=4, n_q=2, spec_scale=(0.0, 0.3),
                   seed=94, residency="uniform", resident_frac=0.5)
STEP_CASES = [TINY, V_HOT, V_CARRY, V_5Q, V_ZIPF, V_NQ64, V_ALL, V_ONEQ, V_ODD, V_FOLD2, V_FOLD5, V_FOLD8, V_WAVES]


@pytest.fixture(scope="module")
def dd():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from sparse_kv_offload_gb300 import build
    build.build()
    from sparse_kv_offload_gb300 import dd as mod
    return mod


def shape_of(w):
    from sparse_kv_offload_gb300.dd import Shape
    return Shape(w.B, w.Hq, w.Hkv, w.d, w.L, w.cs, w.k, w.n_q)


# ------------------------------------------------------------------ generator

def test_device_generator_matches_host_generator(dd):
    import torch
    w = Workload("gen", B=2, Hq=8, Hkv=2, d=128, L=512, cs=16, k=4, n_q=3, spec_scale=(0.0, 0.2, 0.4), seed=5)
    sh = shape_of(w)
    q = torch.empty(w.B * w.n_q * w.Hq * w.d, dtype=torch.bfloat16, device="cuda")
    dd.synth_queries(sh, w.seed, 2, w.spec_scale, q)
    q_host = synth.queries(w.seed, w.B, w.n_q, w.Hq, w.d, w.spec_scale, layer=2)
    assert np.array_equal(tl.from_bf16(q).reshape(q_host.shape), q_host)

    bias = synth.hot_chunk_bias(w.seed, w.B, w.Hkv, w.C, 0.1, 3.0)
    u_hat = synth.query_direction(q_host, w.Hkv)
    K = torch.empty(w.B * w.Hkv * w.L * w.d, dtype=torch.bfloat16, device="cuda")
    dd.synth_kv(sh, w.seed, synth.tensor_id(synth.TID_K, 2), K, torch.from_numpy(bias).cuda(),
                torch.from_numpy(u_hat).cuda())
    K_host = synth.kv_tensor(w.seed, synth.TID_K, w.B, w.Hkv, w.L, w.d, w.cs, bias, u_hat, layer=2)
    assert np.array_equal(tl.from_bf16(K).reshape(K_host.shape), K_host)

    V = torch.empty(w.B * w.Hkv * w.L * w.d, dtype=torch.bfloat16).pin_memory()
    dd.synth_kv(sh, w.seed, synth.tensor_id(synth.TID_V, 2), V)
    torch.cuda.synchronize()
    V_host = synth.kv_tensor(w.seed, synth.TID_V, w.B, w.Hkv, w.L, w.d, w.cs, layer=2)
    assert np.array_equal(tl.from_bf16(V).reshape(V_host.shape), V_host)

    slot = synth.uniform_residency(w.seed, w.B, w.Hkv, w.C, 0.5)
    flat = slot.reshape(-1)
    chunk_map = np.empty(int((flat >= 0).sum()), np.int32)
    chunk_map[flat[flat >= 0]] = np.nonzero(flat >= 0)[0]
    pool = torch.empty(chunk_map.size * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
    dd.synth_kv(sh, w.seed, synth.tensor_id(synth.TID_K, 2), pool, torch.from_numpy(bias).cuda(),
                torch.from_numpy(u_hat).cuda(), chunk_map=tl.to_i32(chunk_map))
    assert np.array_equal(tl.from_bf16(pool).reshape(-1, w.cs, w.d), synth.hot_pool_from(K_host, slot, w.cs))


# ------------------------------------------------------------------ a0 landmarks

@pytest.mark.parametrize("w", [TINY, V_CARRY, V_ZIPF], ids=lambda w: w.name)
@pytest.mark.parametrize("where", ["device", "pinned_host"])
def test_landmarks_bit_exact(dd, w, where):
    import torch
    K = synth.kv_tensor(w.seed, synth.TID_K, w.B, w.Hkv, w.L, w.d, w.cs)
    Kt = tl.to_bf16(K) if where == "device" else tl.to_bf16(K, device="cpu", pin=True)
    lm = torch.empty(w.B * w.Hkv * w.C * w.d, dtype=torch.bfloat16, device="cuda")
    with dd.Context(shape_of(w), max_misses=1) as ctx:
        ctx.build_landmarks(Kt, lm)
        assert ctx.status() == 0
    assert np.array_equal(tl.from_bf16(lm).reshape(w.B, w.Hkv, w.C, w.d), oracle.build_landmarks(K, w.cs))


# ------------------------------------------------------------------ a1 scores

# the tensor-core scoring's instantiations: N = NQ rounded up to 16 (16, 32,
# 48, 64) with the group size unrolled (G = 4, 8) or generic (G = 1, 2, 6,
# 16); C = 1000 leaves a ragged last tile of 104 landmark rows, and several
# units share a CTA's span of tiles
def _sc(name, Hq, Hkv, n_q, B=3, L=16000, seed=0):
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, d=128, L=L, cs=16, k=8, n_q=n_q,
                    spec_scale=(0.0,) + (0.2,) * (n_q - 1), seed=300 + seed)


SCORE_TC_CASES = [_sc("g1_nq3", 8, 8, 3, seed=1), _sc("g2_nq16", 8, 4, 8, seed=2), _sc("g16_nq64", 32, 2, 4, seed=3),
                  _sc("g16_nq32", 32, 2, 2, seed=4), _sc("g6_nq48", 12, 2, 8, seed=5),
                  _sc("g8_nq16", 64, 8, 2, seed=6), _sc("g8_nq24", 64, 8, 3, seed=7),
                  _sc("g4_nq32", 32, 8, 8, seed=8), _sc("g4_nq20", 32, 8, 5, seed=9)]


@pytest.mark.parametrize("w", [TINY, V_5Q, V_NQ64, V_ZIPF] + SCORE_TC_CASES, ids=lambda w: w.name)
def test_scores_within_fp32_bound(dd, w):
    import torch
    q = synth.queries(w.seed, w.B, w.n_q, w.Hq, w.d, w.spec_scale)
    lm = synth.f32_to_bf16(synth.normal_f32(w.seed, 40, np.arange(w.B * w.Hkv * w.C * w.d, dtype=np.uint64))
                           * np.float32(0.25)).reshape(w.B, w.Hkv, w.C, w.d)
    scores = torch.empty(w.B * w.n_q * w.Hkv * w.C, dtype=torch.float32, device="cuda")
    with dd.Context(shape_of(w), max_misses=1) as ctx:
        ctx.score_landmarks(tl.to_bf16(q), tl.to_bf16(lm), scores)
        assert ctx.status() == 0
    got = scores.cpu().numpy().reshape(w.B, w.n_q, w.Hkv, w.C).astype(np.float64)
    want = oracle.score_landmarks(q, lm)
    # fp32 accumulation bound: |err| <= 2e-5 * sum |q_h,i * lm_i| (n <= 1024 terms)
    qa = np.abs(synth.bf16_to_f32(q).astype(np.float64)).reshape(w.B, w.n_q, w.Hkv, w.G, w.d).sum(3)
    bound = 2e-5 * np.einsum("bjgi,bgci->bjgc", qa, np.abs(synth.bf16_to_f32(lm).astype(np.float64)))
    assert np.all(np.abs(got - want) <= bound + 1e-30)


# ------------------------------------------------------------------ a2 top-k

@pytest.mark.parametrize("C,k,ties", [(256, 16, 0), (256, 1, 0), (1000, 37, 4), (2048, 64, 0), (4096, 4095, 2),
                                      (8192, 32, 0), (16384, 128, 1), (64, 64, 0)])
def test_topk_bit_exact(dd, C, k, ties):
    import torch
    from sparse_kv_offload_gb300.dd import Shape
    B, n_q, Hkv = 3, 2, 2
    sh = Shape(B, 2 * Hkv, Hkv, 128, C * 16, 16, k, n_q)
    s = synth.random_scores(C + k, B * n_q * Hkv, C, tie_every=ties)
    s[0, :8] = -0.0                         # -0 ties with +0
    s[1, ::3] = 0.0
    sel = torch.empty(B * n_q * Hkv * k, dtype=torch.int32, device="cuda")
    with dd.Context(sh, max_misses=1) as ctx:
        ctx.select_topk(torch.from_numpy(s).cuda(), sel)
        assert ctx.status() == 0
    want = oracle.select_topk(s.astype(np.float64), k)
    assert np.array_equal(sel.cpu().numpy().reshape(want.shape), want)


# ------------------------------------------------------------------ a3 resolve

def _resolve_on_gpu(dd, ctx, w, sel, slot, max_misses, attn=True):
    import torch
    nu = w.B * w.Hkv * w.max_union
    out = dict(
        union_idx=torch.full((nu,), -7, dtype=torch.int32, device="cuda"),
        union_slot=torch.full((nu,), -7, dtype=torch.int32, device="cuda"),
        union_qmask=torch.zeros(nu, dtype=torch.uint8, device="cuda"),
        union_cnt=torch.zeros(w.B * w.Hkv, dtype=torch.int32, device="cuda"),
        miss_list=torch.full((max(1, max_misses),), -7, dtype=torch.int32, device="cuda"),
        miss_count=torch.zeros(1, dtype=torch.int32, device="cuda"),
        attn_slot=torch.zeros(sel.size, dtype=torch.int32, device="cuda") if attn else None,
    )
    ctx.resolve_union(tl.to_i32(sel), tl.to_i32(slot), out["union_idx"], out["union_slot"], out["union_qmask"],
                      out["union_cnt"], out["miss_list"], out["miss_count"], out["attn_slot"])
    return out


def _compare_resolve(w, got, want, max_misses):
    cnt = got["union_cnt"].cpu().numpy().reshape(w.B, w.Hkv)
    assert np.array_equal(cnt, want["union_cnt"])
    for name in ("union_idx", "union_slot", "union_qmask"):
        g = got[name].cpu().numpy().reshape(w.B, w.Hkv, w.max_union)
        for b in range(w.B):
            for h in range(w.Hkv):
                n = cnt[b, h]
                assert np.array_equal(g[b, h, :n], want[name][b, h, :n]), name
    M = int(got["miss_count"].item())
    assert M == want["miss_count"]
    m = min(M, max_misses)
    assert np.array_equal(got["miss_list"].cpu().numpy()[:m], want["miss_list"][:m])
    if got["attn_slot"] is not None:
        assert np.array_equal(got["attn_slot"].cpu().numpy().reshape(want["attn_slot"].shape), want["attn_slot"])


@pytest.mark.parametrize("n_q,overlap,res_frac,C,k", [(2, 0.7, 0.0, 2048, 64), (2, 0.5, 0.5, 8192, 32),
                                                       (5, 0.4, 0.1, 2048, 128), (8, 0.9, 0.3, 300, 20),
                                                       (1, 1.0, 0.9, 16384, 100), (3, 0.0, 0.0, 64, 64)])
def test_resolve_bit_exact(dd, n_q, overlap, res_frac, C, k):
    w = Workload("resolve", B=4, Hq=8, Hkv=4, d=128, L=C * 16, cs=16, k=k, n_q=n_q, seed=3)
    sel = synth.random_selection(11 + n_q, w.B, w.n_q, w.Hkv, w.C, w.k, overlap)
    slot = synth.uniform_residency(13, w.B, w.Hkv, w.C, res_frac)
    want = oracle.resolve_union(sel, slot)
    cap = w.max_misses
    with dd.Context(shape_of(w), max_misses=cap, hot_slots=int((slot >= 0).sum())) as ctx:
        got = _resolve_on_gpu(dd, ctx, w, sel, slot, cap)
        assert ctx.status() == 0
    _compare_resolve(w, got, want, cap)


def test_resolve_capacity_and_range_errors(dd):
    w = Workload("cap", B=2, Hq=8, Hkv=2, d=128, L=4096, cs=16, k=16, n_q=2, seed=4)
    sel = synth.random_selection(5, w.B, w.n_q, w.Hkv, w.C, w.k, 0.5)
    slot = np.full((w.B, w.Hkv, w.C), -1, np.int32)
    want = oracle.resolve_union(sel, slot)
    cap = want["miss_count"] // 2
    with dd.Context(shape_of(w), max_misses=cap) as ctx:
        got = _resolve_on_gpu(dd, ctx, w, sel, slot, cap)
        assert ctx.status() == dd.DD_ERR_CAPACITY
        assert ctx.status() == 0                          # read clears it
        _compare_resolve(w, got, want, cap)               # everything below the capacity is still right
        bad = sel.copy()
        bad[1, 1, 1, 3] = w.C + 5                         # out-of-range chunk index
        _resolve_on_gpu(dd, ctx, w, bad, slot, cap)
        assert ctx.status() == dd.DD_ERR_DEVICE_CHECK
    with dd.Context(shape_of(w), max_misses=w.max_misses, hot_slots=4) as ctx:
        bad_slot = slot.copy()
        bad_slot[0, 0, sel[0, 0, 0, 0]] = 99              # slot beyond the hot pool
        _resolve_on_gpu(dd, ctx, w, sel, bad_slot, w.max_misses)
        assert ctx.status() == dd.DD_ERR_DEVICE_CHECK


# ------------------------------------------------------------------ a4 gather

@pytest.mark.parametrize("mode", ["zerocopy", "memcpy", "kernel"])
@pytest.mark.parametrize("cs", [16, 64])
def test_gather_bytes_exact(dd, mode, cs):
    import torch
    w = Workload("gather", B=2, Hq=8, Hkv=4, d=128, L=256 * cs, cs=cs, k=32, n_q=2, seed=6)
    rng = np.random.default_rng(cs)
    Kh = rng.integers(0, 1 << 16, (w.B, w.Hkv, w.L, w.d), dtype=np.uint16)
    Vh = rng.integers(0, 1 << 16, (w.B, w.Hkv, w.L, w.d), dtype=np.uint16)
    n_total = w.B * w.Hkv * w.C
    M = 301
    miss = np.sort(rng.choice(n_total, M, replace=False)).astype(np.int32)
    miss[100:110] = np.arange(miss[99] + 1, miss[99] + 11)           # a run of consecutive chunks
    miss = np.unique(miss).astype(np.int32)
    M = miss.size
    cap = M + 3
    Kst = torch.full((cap * cs * w.d,), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    Vst = torch.full((cap * cs * w.d,), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    with dd.Context(shape_of(w), max_misses=cap) as ctx:
        ctx.gather_kv(tl.to_bf16(Kh, "cpu", pin=True), tl.to_bf16(Vh, "cpu", pin=True), tl.to_i32(miss),
                      tl.to_i32(np.array([M])), Kst, Vst,
                      {"zerocopy": dd.GATHER_ZEROCOPY, "kernel": dd.GATHER_KERNEL, "memcpy": dd.GATHER_MEMCPY}[mode])
        assert ctx.status() == 0
    wk, wv = oracle.gather_kv(Kh, Vh, miss, cs)
    gk = tl.from_bf16(Kst).reshape(cap, cs, w.d)
    gv = tl.from_bf16(Vst).reshape(cap, cs, w.d)
    assert np.array_equal(gk[:M], wk) and np.array_equal(gv[:M], wv)
    assert np.all(gk[M:] == 7) and np.all(gv[M:] == 7)                # nothing written past M


def test_gather_rejects_bad_index(dd):
    import torch
    w = Workload("gather_bad", B=1, Hq=8, Hkv=2, d=128, L=1024, cs=16, k=8, n_q=2, seed=6)
    Kh = np.zeros((w.B, w.Hkv, w.L, w.d), np.uint16)
    Kst = torch.zeros(4 * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
    with dd.Context(shape_of(w), max_misses=4) as ctx:
        ctx.gather_kv(tl.to_bf16(Kh, "cpu", pin=True), tl.to_bf16(Kh, "cpu", pin=True),
                      tl.to_i32(np.array([3, w.B * w.Hkv * w.C + 1])), tl.to_i32(np.array([2])), Kst, Kst.clone())
        assert ctx.status() == dd.DD_ERR_DEVICE_CHECK


# ------------------------------------------------------------------ a5 attention (after resolve)

@pytest.mark.parametrize("w", [TINY, V_HOT, V_CARRY, V_5Q, V_ZIPF, V_NQ64, V_ALL], ids=lambda w: w.name)
def test_attention_matches_oracle(dd, w):
    import torch
    x = tl.host_inputs(w)
    sel = oracle.select_topk(oracle.score_landmarks(x["q"], x["lm"]), w.k)
    want_res = oracle.resolve_union(sel, x["slot"])
    Kst_o, Vst_o = oracle.gather_kv(x["K"], x["V"], want_res["miss_list"], w.cs)
    want = oracle.sparse_attn_decode(x["q"], x["Khot"], x["Vhot"], Kst_o, Vst_o, want_res["attn_slot"], w.cs)
    cap = w.max_misses
    hot = x["Khot"].shape[0]
    with dd.Context(shape_of(w), max_misses=cap, hot_slots=hot) as ctx:
        got = _resolve_on_gpu(dd, ctx, w, sel, x["slot"], cap)
        Kst = torch.empty(cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
        Vst = torch.empty_like(Kst)
        ctx.gather_kv(tl.to_bf16(x["K"], "cpu", pin=True), tl.to_bf16(x["V"], "cpu", pin=True), got["miss_list"],
                      got["miss_count"], Kst, Vst)
        out = torch.full((w.B * w.n_q * w.Hq * w.d,), float("nan"), device="cuda")
        ctx.sparse_attn_decode(tl.to_bf16(x["q"]), tl.to_bf16(x["Khot"]) if hot else None,
                               tl.to_bf16(x["Vhot"]) if hot else None, Kst, Vst, got["union_slot"],
                               got["union_qmask"], got["union_cnt"], got["miss_count"], out)
        assert ctx.status() == 0
    _compare_resolve(w, got, want_res, cap)
    tl.check_attention(out.cpu().numpy().reshape(want.shape), want)


def test_attention_custom_scale(dd):
    import torch
    w = TINY
    x = tl.host_inputs(w)
    sel = oracle.select_topk(oracle.score_landmarks(x["q"], x["lm"]), w.k)
    res = oracle.resolve_union(sel, x["slot"])
    Kst_o, Vst_o = oracle.gather_kv(x["K"], x["V"], res["miss_list"], w.cs)
    want = oracle.sparse_attn_decode(x["q"], x["Khot"], x["Vhot"], Kst_o, Vst_o, res["attn_slot"], w.cs, scale=0.25)
    with dd.Context(shape_of(w), max_misses=w.max_misses) as ctx:
        got = _resolve_on_gpu(dd, ctx, w, sel, x["slot"], w.max_misses)
        Kst = torch.empty(w.max_misses * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
        Vst = torch.empty_like(Kst)
        ctx.gather_kv(tl.to_bf16(x["K"], "cpu", pin=True), tl.to_bf16(x["V"], "cpu", pin=True), got["miss_list"],
                      got["miss_count"], Kst, Vst)
        out = torch.empty(w.B * w.n_q * w.Hq * w.d, device="cuda")
        ctx.sparse_attn_decode(tl.to_bf16(x["q"]), None, None, Kst, Vst, got["union_slot"], got["union_qmask"],
                               got["union_cnt"], got["miss_count"], out, softmax_scale=0.25)
        assert ctx.status() == 0
    tl.check_attention(out.cpu().numpy().reshape(want.shape), want)
