"""GPU parity of the predictive prefetch (DualDecoder §4.2, §5.3-§5.4): the
prefetch map and the prefetched bytes against the oracle, the step that
consumes a prefetch against the plain step, and a prefetch running on a
low-priority stream beside a step on a high-priority one."""
import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300 import synth
from sparse_kv_offload_gb300.workloads import TINY

import dd_testlib as tl
from test_gpu_parity import V_5Q, V_HOT, V_ZIPF, shape_of
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


def _selection(w, x):
    """A step's selection; its speculative rows j >= 1 predict the next step."""
    return oracle.select_topk(oracle.score_landmarks(x["q"], x["lm"]), w.k)   # [B, n_q, Hkv, k]


@pytest.mark.parametrize("w", [TINY, V_HOT, V_5Q, V_ZIPF], ids=lambda w: w.name)
def test_prefetch_map_and_bytes_match_oracle(dd, w):
    import torch
    x = tl.host_inputs(w)
    sel = _selection(w, x)
    n_pred = w.n_q - 1
    want = oracle.prefetch_kv(np.ascontiguousarray(sel[:, 1:]), x["K"], x["V"], w.cs)
    cap = w.max_misses
    Kpf = torch.full((cap * w.cs * w.d,), 3, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    Vpf = torch.full((cap * w.cs * w.d,), 3, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    pf_map = torch.zeros(w.B * w.Hkv * w.C, dtype=torch.int32, device="cuda")
    pf_count = torch.zeros(1, dtype=torch.int32, device="cuda")
    with dd.Context(shape_of(w), max_misses=cap) as ctx:
        # rows 1 .. n_q-1 of the step's selection, read in place
        ctx.prefetch_kv(tl.to_i32(sel), n_pred, tl.to_bf16(x["K"], "cpu", pin=True),
                        tl.to_bf16(x["V"], "cpu", pin=True), Kpf, Vpf, pf_map, pf_count, ctas_per_sm=2,
                        sel_rows=w.n_q, first_row=1)
        assert ctx.status() == 0
    P = want["count"]
    assert int(pf_count.item()) == P
    assert np.array_equal(pf_map.cpu().numpy().reshape(want["pf_map"].shape), want["pf_map"])
    assert np.array_equal(tl.from_bf16(Kpf).reshape(-1, w.cs, w.d)[:P], want["K"])
    assert np.array_equal(tl.from_bf16(Vpf).reshape(-1, w.cs, w.d)[:P], want["V"])
    assert np.all(tl.from_bf16(Kpf).view(np.int16).reshape(-1, w.cs, w.d)[P:] == 3)   # nothing past P


@pytest.mark.parametrize("w", [TINY, V_HOT, V_5Q], ids=lambda w: w.name)
def test_step_on_a_prefetch_equals_the_plain_step(dd, w):
    import torch
    x = tl.host_inputs(w)                               # this step's inputs
    prev = tl.host_inputs(w, layer=1)                   # another step's queries predict this one loosely
    pred = np.ascontiguousarray(oracle.select_topk(oracle.score_landmarks(prev["q"], x["lm"]), w.k)[:, 1:])
    n_pred = pred.shape[1]
    pf = oracle.prefetch_kv(pred, x["K"], x["V"], w.cs)
    want = oracle.step(x["q"], x["lm"], x["K"], x["V"], pf["pf_map"], pf["K"], pf["V"], w.k, w.cs)
    plain = oracle.step(x["q"], x["lm"], x["K"], x["V"], np.full((w.B, w.Hkv, w.C), -1, np.int32), None, None,
                        w.k, w.cs)
    np.testing.assert_allclose(want["out"], plain["out"], rtol=1e-12, atol=1e-14)

    P_cap = w.max_misses
    Kpf = torch.zeros(P_cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
    Vpf = torch.zeros(P_cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
    pf_map = torch.empty(w.B * w.Hkv * w.C, dtype=torch.int32, device="cuda")
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=P_cap) as ctx_pf, \
            dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=P_cap) as ctx:
        ctx_pf.prefetch_kv(tl.to_i32(pred), n_pred, buf.Kh, buf.Vh, Kpf, Vpf, pf_map)
        ctx.step(0, buf.q, buf.lm, buf.Kh, buf.Vh, pf_map, Kpf, Vpf, buf.Kst, buf.Vst, buf.out,
                 intermediates=buf.inter)
        assert ctx_pf.status() == 0 and ctx.status() == 0
    g = {k: v.cpu().numpy() for k, v in buf.inter.items()}
    sel = g["sel"].reshape(want["sel"].shape)
    tl.selection_rows_match(sel, want["scores"], want["sel"], w.k)
    # only the unpredicted chunks are missing; every unit's layout on the GPU's own selection
    ref, _ = tl.follow_gpu_selection(sel, want, x["q"], x["K"], x["V"], pf["pf_map"], pf["K"], pf["V"], w.cs)
    tl.check_layout(g, ref, w.B, w.Hkv, w.max_union, buf.Kst[0], buf.Vst[0])
    tl.check_attention(buf.out.cpu().numpy().reshape(ref["out"].shape), ref["out"])
    if not np.array_equal(sel, want["sel"]):
        return
    tl.check_attention(buf.out.cpu().numpy().reshape(plain["out"].shape), plain["out"])


def test_prefetch_on_a_low_priority_stream_beside_a_step(dd):
    # layer A's prefetch runs on a low-priority stream while layer B's step runs on a
    # high-priority one; layer A's step then waits for the prefetch's event
    import torch
    w = V_HOT
    xa, xb = tl.host_inputs(w, layer=0), tl.host_inputs(w, layer=1)
    pred = np.ascontiguousarray(oracle.select_topk(oracle.score_landmarks(xa["q"], xa["lm"]), w.k)[:, 1:])
    want_a = oracle.step(xa["q"], xa["lm"], xa["K"], xa["V"], np.full((w.B, w.Hkv, w.C), -1, np.int32), None, None,
                         w.k, w.cs)
    want_b = oracle.step(xb["q"], xb["lm"], xb["K"], xb["V"], np.full((w.B, w.Hkv, w.C), -1, np.int32), None, None,
                         w.k, w.cs)
    lo = torch.cuda.Stream(priority=0)
    hi = torch.cuda.Stream(priority=-1)
    P_cap = w.max_misses
    Kpf = torch.zeros(P_cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
    Vpf = torch.zeros(P_cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
    pf_map = torch.empty(w.B * w.Hkv * w.C, dtype=torch.int32, device="cuda")
    none_resident = tl.to_i32(np.full((w.B, w.Hkv, w.C), -1, np.int32))
    spare = torch.zeros(P_cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda")   # layer B's (unused) pool
    ba, bb = StepBuffers(w, xa), StepBuffers(w, xb)
    sel_pred = tl.to_i32(pred)
    torch.cuda.synchronize()
    done = torch.cuda.Event()
    with dd.Context(shape_of(w), max_misses=P_cap) as ctx_pf, \
            dd.Context(shape_of(w), max_misses=ba.cap, hot_slots=P_cap) as ctx:
        ctx_pf.prefetch_kv(sel_pred, w.n_q - 1, ba.Kh, ba.Vh, Kpf, Vpf, pf_map, ctas_per_sm=2, stream=lo)
        done.record(lo)
        ctx.step(1, bb.q, bb.lm, bb.Kh, bb.Vh, none_resident, spare, spare, bb.Kst, bb.Vst, bb.out, stream=hi)
        hi.wait_event(done)
        ctx.step(2, ba.q, ba.lm, ba.Kh, ba.Vh, pf_map, Kpf, Vpf, ba.Kst, ba.Vst, ba.out, stream=hi)
        torch.cuda.synchronize()
        assert ctx_pf.status() == 0 and ctx.status() == 0
    tl.check_attention(bb.out.cpu().numpy().reshape(want_b["out"].shape), want_b["out"])
    tl.check_attention(ba.out.cpu().numpy().reshape(want_a["out"].shape), want_a["out"])


def test_prefetch_rejects_bad_row_counts(dd):
    import torch
    w = TINY
    x = tl.host_inputs(w)
    sel = torch.zeros(w.B * (w.n_q + 1) * w.Hkv * w.k, dtype=torch.int32, device="cuda")
    pf_map = torch.empty(w.B * w.Hkv * w.C, dtype=torch.int32, device="cuda")
    K = tl.to_bf16(x["K"], "cpu", pin=True)
    with dd.Context(shape_of(w), max_misses=w.max_misses) as ctx:
        for n_pred in (0, w.n_q + 1):
            with pytest.raises(dd.DDError):
                ctx.prefetch_kv(sel, n_pred, K, K, None, None, pf_map)
