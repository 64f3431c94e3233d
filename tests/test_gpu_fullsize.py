"""Parity at the workloads' full sizes, in the launch configuration the bench
times (dd_step, zero-copy gather fused into the attention, one stream).

The oracle cannot run a whole full-size step, so (b, g) units are sampled:
their keys and values are regenerated on the host from the counter-based
generator and each sampled unit goes through the oracle stage by stage
(landmarks bit-exact, scores within the fp32 bound, selections modulo the
tie band, union / query masks / staging bytes bit-exact, attention within
the tolerances).  Over all units the GPU outputs must also satisfy the
properties that hold at any size: union sizes in [k, min(C, n_q k)],
ascending unions, resident slots equal to the residency map, misses
numbered densely in (b, g, c) order with the miss list pointing back at
them."""
import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300 import synth
from sparse_kv_offload_gb300.workloads import ALL

import dd_testlib as tl
from test_gpu_parity import shape_of

pytestmark = pytest.mark.gpu

N_SAMPLE = 3


@pytest.fixture(scope="module")
def dd():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from sparse_kv_offload_gb300 import build
    build.build()
    from sparse_kv_offload_gb300 import dd as mod
    return mod


def _sampled_units(w):
    units = w.B * w.Hkv
    rng = np.random.default_rng(w.seed)
    extra = rng.choice(np.arange(1, units - 1), size=max(0, N_SAMPLE - 2), replace=False) if units > 2 else []
    return sorted({0, units - 1, *[int(u) for u in extra]})


def _unit_rows(w, tid, u, bias, u_hat):
    x = synth.kv_rows(w.seed, tid, w.B, w.Hkv, w.L, w.d, w.cs, np.array([u]), np.array([0]), w.L, bias, u_hat)
    return x.reshape(1, 1, w.L, w.d)


def _residency(w, q_host, bias, u_hat, sample):
    """The workload's residency map [B, Hkv, C]; the carried kind uses the oracle's
    union for the sampled units and a seeded stand-in set of k chunks elsewhere."""
    if w.residency == "uniform":
        return synth.uniform_residency(w.seed, w.B, w.Hkv, w.C, w.resident_frac)
    if w.residency == "carry":
        order = synth.random_order(w.seed, 31, w.B * w.Hkv, w.C)   # an id no workload tensor uses
        sets = [set(order[u, :w.k].tolist()) for u in range(w.B * w.Hkv)]
        G = w.Hq // w.Hkv
        for u in sample:
            b, g = divmod(u, w.Hkv)
            K_u = _unit_rows(w, synth.TID_K, u, bias, u_hat)
            s_u = oracle.score_landmarks(q_host[b:b + 1, :, g * G:(g + 1) * G], oracle.build_landmarks(K_u, w.cs))
            sets[u] = set(oracle.union_of_query_selections(oracle.select_topk(s_u, w.k), 0, 0))
        return synth.carried_residency(w.seed, sets, w.B, w.Hkv, w.C, w.resident_frac)
    return np.full((w.B, w.Hkv, w.C), -1, np.int32)


@pytest.mark.parametrize("w", ALL, ids=lambda w: w.name)
def test_full_size_step_on_sampled_units(dd, w):
    import torch
    sh = shape_of(w)
    G = w.Hq // w.Hkv
    units = w.B * w.Hkv
    sample = _sampled_units(w)
    # device inputs, from the same generator definition as the host regeneration below
    q = torch.empty(w.B * w.n_q * w.Hq * w.d, dtype=torch.bfloat16, device="cuda")
    dd.synth_queries(sh, w.seed, 0, w.spec_scale, q)
    q_host = synth.queries(w.seed, w.B, w.n_q, w.Hq, w.d, w.spec_scale)
    bias, u_hat = tl.key_bias(w, q_host)
    bias_d = None if bias is None else torch.from_numpy(bias).cuda()
    uhat_d = None if u_hat is None else torch.from_numpy(u_hat).cuda()
    n = w.B * w.Hkv * w.L * w.d
    Kh = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    Vh = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    dd.synth_kv(sh, w.seed, synth.tensor_id(synth.TID_K, 0), Kh, bias_d, uhat_d)
    dd.synth_kv(sh, w.seed, synth.tensor_id(synth.TID_V, 0), Vh)
    slot = _residency(w, q_host, bias, u_hat, sample)
    flat = slot.reshape(-1)
    n_hot = int((flat >= 0).sum())
    Khot = Vhot = None
    if n_hot:
        chunk_map = np.empty(n_hot, np.int32)
        chunk_map[flat[flat >= 0]] = np.nonzero(flat >= 0)[0]
        cm = tl.to_i32(chunk_map)
        Khot = torch.empty(n_hot * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
        Vhot = torch.empty(n_hot * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
        dd.synth_kv(sh, w.seed, synth.tensor_id(synth.TID_K, 0), Khot, bias_d, uhat_d, chunk_map=cm)
        dd.synth_kv(sh, w.seed, synth.tensor_id(synth.TID_V, 0), Vhot, chunk_map=cm)
    cap = w.max_misses
    lm = torch.empty(units * w.C * w.d, dtype=torch.bfloat16, device="cuda")
    Kst = [torch.empty(cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    Vst = [torch.empty(cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    out = torch.empty(w.B * w.n_q * w.Hq * w.d, dtype=torch.float32, device="cuda")
    nu = units * w.max_union
    inter = dict(
        scores=torch.empty(w.B * w.n_q * w.Hkv * w.C, dtype=torch.float32, device="cuda"),
        sel=torch.empty(w.B * w.n_q * w.Hkv * w.k, dtype=torch.int32, device="cuda"),
        union_idx=torch.empty(nu, dtype=torch.int32, device="cuda"),
        union_slot=torch.empty(nu, dtype=torch.int32, device="cuda"),
        union_qmask=torch.empty(nu, dtype=torch.uint8, device="cuda"),
        union_cnt=torch.empty(units, dtype=torch.int32, device="cuda"),
        miss_list=torch.empty(cap, dtype=torch.int32, device="cuda"),
        miss_count=torch.empty(1, dtype=torch.int32, device="cuda"),
        attn_slot=torch.empty(w.B * w.n_q * w.Hkv * w.k, dtype=torch.int32, device="cuda"),
    )
    with dd.Context(sh, max_misses=cap, hot_slots=n_hot) as ctx:
        ctx.build_landmarks(Kh, lm)
        ctx.step(0, q, lm, Kh, Vh, tl.to_i32(slot), Khot, Vhot, Kst, Vst, out, intermediates=inter)
        assert ctx.status() == 0
    g_ = {k: v.cpu().numpy() for k, v in inter.items()}
    umax = w.max_union
    cnt = g_["union_cnt"]
    uidx = g_["union_idx"].reshape(units, umax)
    uslot = g_["union_slot"].reshape(units, umax)
    M = int(g_["miss_count"][0])
    mlist = g_["miss_list"][:M]
    rs = slot.reshape(units, w.C)

    # ---- properties over every unit
    assert np.all((cnt >= w.k) & (cnt <= min(w.C, w.n_q * w.k)))
    seen = 0
    for u in range(units):
        c_u, s_u = uidx[u, :cnt[u]], uslot[u, :cnt[u]]
        assert np.all(np.diff(c_u) > 0)
        res = s_u >= 0
        assert np.array_equal(s_u[res], rs[u, c_u[res]])
        assert np.all(rs[u, c_u[~res]] < 0)
        m = -s_u[~res] - 1
        assert np.array_equal(m, np.arange(seen, seen + m.size))          # dense, in (b, g, c) order
        assert np.array_equal(mlist[m], u * w.C + c_u[~res])
        seen += m.size
    assert seen == M

    # ---- sampled units against the oracle
    lm_h = tl.from_bf16(lm).reshape(units, w.C, w.d)
    scores = g_["scores"].reshape(w.B, w.n_q, w.Hkv, w.C)
    sel = g_["sel"].reshape(w.B, w.n_q, w.Hkv, w.k)
    qmask = g_["union_qmask"].reshape(units, umax)
    out_h = out.cpu().numpy().reshape(w.B, w.n_q, w.Hq, w.d)
    kst = tl.from_bf16(Kst[0]).reshape(-1, w.cs, w.d)
    vst = tl.from_bf16(Vst[0]).reshape(-1, w.cs, w.d)
    for u in sample:
        b, g = divmod(u, w.Hkv)
        K_u = _unit_rows(w, synth.TID_K, u, bias, u_hat)
        V_u = _unit_rows(w, synth.TID_V, u, None, None)
        lm_u = oracle.build_landmarks(K_u, w.cs)
        assert np.array_equal(lm_h[u], lm_u[0, 0])
        q_u = np.ascontiguousarray(q_host[b:b + 1, :, g * G:(g + 1) * G])
        s_u = oracle.score_landmarks(q_u, lm_u)                             # [1, n_q, 1, C]
        got_s = scores[b, :, g].astype(np.float64)
        assert np.abs(got_s - s_u[0, :, 0]).max() <= 1e-4 * max(1.0, np.abs(s_u).max())
        sel_u = oracle.select_topk(s_u, w.k)
        gsel_u = sel[b:b + 1, :, g:g + 1]
        tl.selection_rows_match(gsel_u, s_u, sel_u, w.k)
        # the rest of the unit follows the GPU's own selection (the oracle's where they agree)
        tie = not np.array_equal(gsel_u, sel_u)
        tl.TIE_TALLY["checks"] += 1
        tl.TIE_TALLY["units"] += 1
        tl.TIE_TALLY["tie_units"] += int(tie)
        tl.TIE_TALLY["tie_rows"] += int(np.any(gsel_u != sel_u, axis=-1).sum())
        sel_u = np.ascontiguousarray(gsel_u)
        U = oracle.union_of_query_selections(sel_u, 0, 0)
        assert cnt[u] == len(U) and np.array_equal(uidx[u, :cnt[u]], U)
        want_qm = [sum(1 << j for j in range(w.n_q) if c in set(sel_u[0, j, 0].tolist())) for c in U]
        assert np.array_equal(qmask[u, :cnt[u]], want_qm)
        for i, c in enumerate(U):                                           # staging bytes of the misses
            if uslot[u, i] < 0:
                m = -uslot[u, i] - 1
                assert np.array_equal(kst[m], K_u[0, 0, c * w.cs:(c + 1) * w.cs])
                assert np.array_equal(vst[m], V_u[0, 0, c * w.cs:(c + 1) * w.cs])
        res_u = oracle.resolve_union(sel_u, np.full((1, 1, w.C), -1, np.int32))
        Ks, Vs = oracle.gather_kv(K_u, V_u, res_u["miss_list"], w.cs)
        empty = np.zeros((0, w.cs, w.d), np.uint16)
        want = oracle.sparse_attn_decode(q_u, empty, empty, Ks, Vs, res_u["attn_slot"], w.cs)
        tl.check_attention(out_h[b:b + 1, :, g * G:(g + 1) * G], want)
