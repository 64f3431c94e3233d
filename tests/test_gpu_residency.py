"""GPU parity of the step's tail rows (the new tokens under the causal mask)
and of the capped LRU residency update, over sequences of steps."""
import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300 import synth
from sparse_kv_offload_gb300.workloads import TINY, Workload

import dd_testlib as tl
from test_gpu_parity import V_5Q, V_HOT, V_NQ64, V_ONEQ, shape_of
from test_gpu_step import StepBuffers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dd():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from sparse_kv_offload_gb300 import build
    build.build()
    from sparse_kv_offload_gb300 import dd as mod
    return mod


def _tails(w, seed):
    n = w.B * w.n_q * w.Hkv * w.d
    kt = synth.f32_to_bf16(synth.normal_f32(seed, 50, np.arange(n, dtype=np.uint64))).reshape(w.B, w.n_q, w.Hkv, w.d)
    vt = synth.f32_to_bf16(synth.normal_f32(seed, 51, np.arange(n, dtype=np.uint64))).reshape(w.B, w.n_q, w.Hkv, w.d)
    return kt, vt


@pytest.mark.parametrize("w", [TINY, V_HOT, V_5Q, V_NQ64, V_ONEQ], ids=lambda w: w.name)
@pytest.mark.parametrize("mode", [0, 1, 2], ids=["zerocopy", "memcpy", "kernel"])
def test_step_with_tail_rows_matches_oracle(dd, w, mode):
    x = tl.host_inputs(w)
    kt, vt = _tails(w, w.seed)
    want = oracle.step(x["q"], x["lm"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.k, w.cs,
                       K_tail=kt, V_tail=vt)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=buf.hot) as ctx:
        ctx.step(0, buf.q, buf.lm, buf.Kh, buf.Vh, buf.slot, buf.Khot, buf.Vhot, buf.Kst, buf.Vst, buf.out,
                 mode=mode, intermediates=buf.inter, K_tail=tl.to_bf16(kt), V_tail=tl.to_bf16(vt))
        assert ctx.status() == 0
    g = {k: v.cpu().numpy() for k, v in buf.inter.items()}
    sel = g["sel"].reshape(want["sel"].shape)
    tl.selection_rows_match(sel, want["scores"], want["sel"], w.k)
    ref, _ = tl.follow_gpu_selection(sel, want, x["q"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.cs,
                                     K_tail=kt, V_tail=vt)
    tl.check_layout(g, ref, w.B, w.Hkv, w.max_union, buf.Kst[0], buf.Vst[0])
    tl.check_attention(buf.out.cpu().numpy().reshape(ref["out"].shape), ref["out"])


def test_attention_with_tail_rows_only_masks_later_tokens(dd):
    # stand-alone attention: a later token's tail row with a huge logit must not reach query 0
    import torch
    w = Workload("tail_mask", B=1, Hq=4, Hkv=2, d=128, L=256, cs=16, k=4, n_q=2, spec_scale=(0.0, 0.3), seed=81)
    x = tl.host_inputs(w)
    res = oracle.resolve_union(oracle.select_topk(oracle.score_landmarks(x["q"], x["lm"]), w.k), x["slot"])
    Kst, Vst = oracle.gather_kv(x["K"], x["V"], res["miss_list"], w.cs)
    kt, vt = _tails(w, 82)
    kt[:, 1] = synth.f32_to_bf16(np.float32(30.0) * synth.bf16_to_f32(x["q"][:, 1, ::2]))   # token 1's key ~ q_1
    want = oracle.sparse_attn_decode(x["q"], x["Khot"], x["Vhot"], Kst, Vst, res["attn_slot"], w.cs,
                                     K_tail=kt, V_tail=vt)
    sh = shape_of(w)
    out = torch.empty(w.B * w.n_q * w.Hq * w.d, device="cuda")
    with dd.Context(sh, max_misses=max(1, res["miss_count"])) as ctx:
        ctx.sparse_attn_decode(tl.to_bf16(x["q"]), None, None, tl.to_bf16(Kst), tl.to_bf16(Vst),
                               tl.to_i32(res["union_slot"]), torch.from_numpy(res["union_qmask"]).cuda(),
                               tl.to_i32(res["union_cnt"]), tl.to_i32(np.array([res["miss_count"]])), out,
                               K_tail=tl.to_bf16(kt), V_tail=tl.to_bf16(vt))
        assert ctx.status() == 0
    tl.check_attention(out.cpu().numpy().reshape(want.shape), want)


@pytest.mark.parametrize("with_tail", [False, True], ids=["no_tail", "tail"])
def test_attention_units_with_empty_unions(dd, with_tail):
    # units whose union is empty: no attention CTA visits them, so the plan
    # kernel writes their output (the tail rows alone, or zero)
    import torch
    w = Workload("empty_units", B=2, Hq=8, Hkv=2, d=128, L=1024, cs=16, k=8, n_q=2, spec_scale=(0.0, 0.3), seed=83)
    x = tl.host_inputs(w)
    res = oracle.resolve_union(oracle.select_topk(oracle.score_landmarks(x["q"], x["lm"]), w.k), x["slot"])
    Kst, Vst = oracle.gather_kv(x["K"], x["V"], res["miss_list"], w.cs)
    cnt = res["union_cnt"].copy()
    attn_slot = res["attn_slot"].copy()
    for b, g in ((0, 1), (1, 0)):                                      # two of the four units emptied
        cnt[b, g] = 0
        attn_slot[b, :, g] = oracle.NO_SLOT
    kt, vt = _tails(w, 84) if with_tail else (None, None)
    want = oracle.sparse_attn_decode(x["q"], x["Khot"], x["Vhot"], Kst, Vst, attn_slot, w.cs, K_tail=kt, V_tail=vt)
    out = torch.full((w.B * w.n_q * w.Hq * w.d,), float("nan"), device="cuda")
    tails = dict(K_tail=tl.to_bf16(kt), V_tail=tl.to_bf16(vt)) if with_tail else {}
    with dd.Context(shape_of(w), max_misses=max(1, res["miss_count"])) as ctx:
        ctx.sparse_attn_decode(tl.to_bf16(x["q"]), None, None, tl.to_bf16(Kst), tl.to_bf16(Vst),
                               tl.to_i32(res["union_slot"]), torch.from_numpy(res["union_qmask"]).cuda(),
                               tl.to_i32(cnt), tl.to_i32(np.array([res["miss_count"]])), out, **tails)
        assert ctx.status() == 0
    got = out.cpu().numpy().reshape(want.shape)
    if not with_tail:
        assert np.all(got[0, :, 4:] == 0) and np.all(got[1, :, :4] == 0)   # query heads of the emptied units
    tl.check_attention(got, want)


def test_tail_rows_need_both_tensors(dd):
    w = TINY
    x = tl.host_inputs(w)
    kt, _ = _tails(w, 5)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap) as ctx:
        with pytest.raises(dd.DDError):
            ctx.step(0, buf.q, buf.lm, buf.Kh, buf.Vh, buf.slot, None, None, buf.Kst, buf.Vst, buf.out,
                     K_tail=tl.to_bf16(kt))


class Pool:
    """Device residency state of one layer and its oracle twin."""

    def __init__(self, w, S):
        import torch
        units = w.B * w.Hkv
        self.S = S
        self.rs = np.full((w.B, w.Hkv, w.C), -1, np.int32)
        self.sc = np.full((w.B, w.Hkv, S), -1, np.int32)
        self.lu = np.full((w.B, w.Hkv, S), -1, np.int32)
        self.Khot = np.zeros((units * S, w.cs, w.d), np.uint16)
        self.Vhot = np.zeros((units * S, w.cs, w.d), np.uint16)
        self.d_rs, self.d_sc, self.d_lu = tl.to_i32(self.rs), tl.to_i32(self.sc), tl.to_i32(self.lu)
        self.d_Khot, self.d_Vhot = tl.to_bf16(self.Khot), tl.to_bf16(self.Vhot)
        self.d_adm = torch.empty(units, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("S,cap", [(24, 10), (40, 64), (8, 3)])
def test_residency_over_steps_matches_oracle(dd, S, cap):
    import torch
    w = TINY
    x = tl.host_inputs(w)
    pool = Pool(w, S)
    queries = [synth.queries(w.seed, w.B, w.n_q, w.Hq, w.d, w.spec_scale, layer=l) for l in (0, 1, 0, 2, 0)]
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=w.B * w.Hkv * S) as ctx:
        for step_id, q in enumerate(queries):
            buf.q = tl.to_bf16(q)
            ctx.step(step_id, buf.q, buf.lm, buf.Kh, buf.Vh, pool.d_rs, pool.d_Khot, pool.d_Vhot, buf.Kst, buf.Vst,
                     buf.out, intermediates=buf.inter)
            p = step_id & 1
            ctx.update_residency(step_id, cap, S, buf.Kst[p], buf.Vst[p], pool.d_rs, pool.d_sc, pool.d_lu,
                                 pool.d_Khot, pool.d_Vhot, admitted=pool.d_adm, union_idx=buf.inter["union_idx"],
                                 union_slot=buf.inter["union_slot"], union_cnt=buf.inter["union_cnt"],
                                 miss_count=buf.inter["miss_count"])
            assert ctx.status() == 0
            # oracle on the same selection (the GPU's, once it is checked against the oracle's)
            scores = oracle.score_landmarks(q, x["lm"])
            sel = buf.inter["sel"].cpu().numpy().reshape(w.B, w.n_q, w.Hkv, w.k)
            tl.selection_rows_match(sel, scores, oracle.select_topk(scores, w.k), w.k)
            res = oracle.resolve_union(sel, pool.rs)
            assert int(buf.inter["miss_count"].item()) == res["miss_count"]
            Kst, Vst = oracle.gather_kv(x["K"], x["V"], res["miss_list"], w.cs)
            out = oracle.sparse_attn_decode(q, pool.Khot, pool.Vhot, Kst, Vst, res["attn_slot"], w.cs)
            tl.check_attention(buf.out.cpu().numpy().reshape(out.shape), out)
            new = oracle.update_residency(step_id, cap, res["union_idx"], res["union_slot"], res["union_cnt"], Kst,
                                          Vst, pool.rs, pool.sc, pool.lu, pool.Khot, pool.Vhot)
            pool.rs, pool.sc, pool.lu = new["resident_slot"], new["slot_chunk"], new["last_used"]
            pool.Khot, pool.Vhot = new["Khot"], new["Vhot"]
            assert np.array_equal(pool.d_adm.cpu().numpy().reshape(w.B, w.Hkv), new["admitted"])
            assert np.array_equal(pool.d_rs.cpu().numpy().reshape(pool.rs.shape), pool.rs)
            assert np.array_equal(pool.d_sc.cpu().numpy().reshape(pool.sc.shape), pool.sc)
            assert np.array_equal(pool.d_lu.cpu().numpy().reshape(pool.lu.shape), pool.lu)
            assert np.array_equal(tl.from_bf16(pool.d_Khot).reshape(pool.Khot.shape), pool.Khot)
            assert np.array_equal(tl.from_bf16(pool.d_Vhot).reshape(pool.Vhot.shape), pool.Vhot)
        # the repeated query of steps 0, 2, 4 finds its chunks resident: fewer misses each time
    assert pool.sc.max() >= 0


def test_residency_rejects_a_pool_that_does_not_split_per_unit(dd):
    w = TINY
    x = tl.host_inputs(w)
    pool = Pool(w, 8)
    buf = StepBuffers(w, x)
    import torch
    hot = w.B * w.Hkv * 8 + 1
    Khot = torch.zeros(hot * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=hot) as ctx:
        with pytest.raises(dd.DDError):
            ctx.update_residency(0, 4, 8, buf.Kst[0], buf.Vst[0], pool.d_rs, pool.d_sc, pool.d_lu, Khot, Khot)
