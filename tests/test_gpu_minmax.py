"""GPU parity of the second landmark kind: Quest-style coordinate-wise min/max
key summaries (OasisKV summary, Methodology) and their upper-bound score,
stage by stage and through the whole step."""
import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300 import synth
from sparse_kv_offload_gb300.workloads import TINY, Workload

import dd_testlib as tl
from test_gpu_parity import V_5Q, V_CARRY, V_HOT, V_NQ64, V_ONEQ, V_ZIPF, shape_of
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


def _keys_with_signed_zeros(w):
    K = synth.kv_tensor(w.seed, synth.TID_K, w.B, w.Hkv, w.L, w.d, w.cs).copy()
    # plant zeros of both signs (and a chunk of only zeros) in a few places
    K[0, 0, 0:w.cs, 3] = np.where(np.arange(w.cs) % 2 == 0, 0x8000, 0x0000)
    K[0, 0, w.cs:2 * w.cs, 5] = 0x8000
    K[-1, -1, -w.cs:, 7] = 0x0000
    K[-1, -1, -w.cs, 7] = 0x8000
    return K


@pytest.mark.parametrize("w", [TINY, V_CARRY, V_ZIPF], ids=lambda w: w.name)
@pytest.mark.parametrize("where", ["device", "pinned_host"])
def test_minmax_landmarks_bit_exact(dd, w, where):
    import torch
    K = _keys_with_signed_zeros(w)
    Kt = tl.to_bf16(K) if where == "device" else tl.to_bf16(K, device="cpu", pin=True)
    lm2 = torch.empty(w.B * w.Hkv * w.C * 2 * w.d, dtype=torch.bfloat16, device="cuda")
    with dd.Context(shape_of(w), max_misses=1) as ctx:
        ctx.build_landmarks_minmax(Kt, lm2)
        assert ctx.status() == 0
    want = oracle.build_minmax_landmarks(K, w.cs)
    assert np.array_equal(tl.from_bf16(lm2).reshape(want.shape), want)


@pytest.mark.parametrize("w", [TINY, V_5Q, V_NQ64, V_ZIPF, V_ONEQ], ids=lambda w: w.name)
def test_minmax_scores_within_fp32_bound(dd, w):
    import torch
    q = synth.queries(w.seed, w.B, w.n_q, w.Hq, w.d, w.spec_scale)
    K = synth.kv_tensor(w.seed, synth.TID_K, w.B, w.Hkv, w.L, w.d, w.cs)
    lm2 = oracle.build_minmax_landmarks(K, w.cs)
    scores = torch.empty(w.B * w.n_q * w.Hkv * w.C, dtype=torch.float32, device="cuda")
    with dd.Context(shape_of(w), max_misses=1) as ctx:
        ctx.score_landmarks_minmax(tl.to_bf16(q), tl.to_bf16(lm2), scores)
        assert ctx.status() == 0
    got = scores.cpu().numpy().reshape(w.B, w.n_q, w.Hkv, w.C).astype(np.float64)
    want = oracle.score_minmax_landmarks(q, lm2)
    # fp32 group sum and accumulation: |err| <= 2e-5 * sum_i (sum_h |q_h,i|) * max(|min_i|, |max_i|)
    qa = np.abs(synth.bf16_to_f32(q).astype(np.float64)).reshape(w.B, w.n_q, w.Hkv, w.G, w.d).sum(3)
    ext = np.abs(synth.bf16_to_f32(lm2).astype(np.float64)).max(axis=3)
    bound = 2e-5 * np.einsum("bjgi,bgci->bjgc", qa, ext)
    assert np.all(np.abs(got - want) <= bound + 1e-30)
    # and the bound property itself holds on the GPU scores up to that error
    kf = synth.bf16_to_f32(K).astype(np.float64).reshape(w.B, w.Hkv, w.C, w.cs, w.d)
    Q = synth.bf16_to_f32(q).astype(np.float64).reshape(w.B, w.n_q, w.Hkv, w.G, w.d).sum(3)
    best = np.einsum("bjgi,bgcti->bjgct", Q, kf).max(axis=-1)
    assert np.all(got >= best - bound - 1e-9)


@pytest.mark.parametrize("w", [TINY, V_HOT, V_CARRY, V_5Q, V_ZIPF], ids=lambda w: w.name)
@pytest.mark.parametrize("mode", [0, 1, 2], ids=["zerocopy", "memcpy", "kernel"])
def test_step_with_minmax_landmarks_matches_oracle(dd, w, mode):
    x = tl.host_inputs(w)
    lm2 = oracle.build_minmax_landmarks(x["K"], w.cs)
    want = oracle.step(x["q"], lm2, x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.k, w.cs)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=buf.hot) as ctx:
        buf.run(ctx, layer=1, mode=mode, lm=tl.to_bf16(lm2), lm_kind=dd.LM_MINMAX)
        assert ctx.status() == 0
    g = {k: v.cpu().numpy() for k, v in buf.inter.items()}
    s = g["scores"].reshape(want["scores"].shape).astype(np.float64)
    assert np.abs(s - want["scores"]).max() <= 1e-4 * max(1.0, np.abs(want["scores"]).max())
    sel = g["sel"].reshape(want["sel"].shape)
    tl.selection_rows_match(sel, want["scores"], want["sel"], w.k)
    ref, _ = tl.follow_gpu_selection(sel, want, x["q"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.cs)
    tl.check_layout(g, ref, w.B, w.Hkv, w.max_union, buf.Kst[1], buf.Vst[1])
    tl.check_attention(buf.out.cpu().numpy().reshape(ref["out"].shape), ref["out"])


def test_step_rejects_unknown_landmark_kind(dd):
    w = TINY
    x = tl.host_inputs(w)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap) as ctx:
        with pytest.raises(dd.DDError):
            buf.run(ctx, lm_kind=7)
