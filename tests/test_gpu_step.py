"""GPU parity of the whole one-layer step (dd_step) against oracle.step, plus
the ping-pong buffer, determinism, empty batches and the device error word."""
import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300 import synth
from sparse_kv_offload_gb300.workloads import TINY, Workload

import dd_testlib as tl
from test_gpu_parity import STEP_CASES, V_HOT, shape_of

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


class StepBuffers:
    """Device / pinned buffers of one workload's step."""

    def __init__(self, w, x, cap=None):
        import torch
        self.w = w
        self.cap = w.max_misses if cap is None else cap
        self.q = tl.to_bf16(x["q"])
        self.lm = tl.to_bf16(x["lm"])
        self.Kh = tl.to_bf16(x["K"], "cpu", pin=True)
        self.Vh = tl.to_bf16(x["V"], "cpu", pin=True)
        self.slot = tl.to_i32(x["slot"])
        self.hot = x["Khot"].shape[0]
        self.Khot = tl.to_bf16(x["Khot"]) if self.hot else None
        self.Vhot = tl.to_bf16(x["Vhot"]) if self.hot else None
        n = max(1, self.cap) * w.cs * w.d
        self.Kst = [torch.full((n,), 3, dtype=torch.int16, device="cuda").view(torch.bfloat16) for _ in range(2)]
        self.Vst = [torch.full((n,), 3, dtype=torch.int16, device="cuda").view(torch.bfloat16) for _ in range(2)]
        self.out = torch.full((w.B * w.n_q * w.Hq * w.d,), float("nan"), device="cuda")
        nu = w.B * w.Hkv * w.max_union
        self.inter = dict(
            scores=torch.empty(w.B * w.n_q * w.Hkv * w.C, dtype=torch.float32, device="cuda"),
            sel=torch.empty(w.B * w.n_q * w.Hkv * w.k, dtype=torch.int32, device="cuda"),
            union_idx=torch.empty(nu, dtype=torch.int32, device="cuda"),
            union_slot=torch.empty(nu, dtype=torch.int32, device="cuda"),
            union_qmask=torch.empty(nu, dtype=torch.uint8, device="cuda"),
            union_cnt=torch.empty(w.B * w.Hkv, dtype=torch.int32, device="cuda"),
            miss_list=torch.empty(max(1, self.cap), dtype=torch.int32, device="cuda"),
            miss_count=torch.empty(1, dtype=torch.int32, device="cuda"),
            attn_slot=torch.empty(w.B * w.n_q * w.Hkv * w.k, dtype=torch.int32, device="cuda"),
        )

    def run(self, ctx, layer=0, mode=0, lm=None, lm_kind=0):
        ctx.step(layer, self.q, self.lm if lm is None else lm, self.Kh, self.Vh, self.slot, self.Khot, self.Vhot,
                 self.Kst, self.Vst, self.out, mode=mode, intermediates=self.inter, lm_kind=lm_kind)


@pytest.mark.parametrize("w", STEP_CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("mode", [0, 1, 2, 3], ids=["zerocopy", "memcpy", "kernel", "auto"])
def test_step_matches_oracle(dd, w, mode):
    x = tl.host_inputs(w)
    want = oracle.step(x["q"], x["lm"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.k, w.cs)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=buf.hot) as ctx:
        buf.run(ctx, layer=0, mode=mode)
        assert ctx.status() == 0
    g = {k: v.cpu().numpy() for k, v in buf.inter.items()}
    # a1: scores within the fp32 bound relative to the score scale
    s = g["scores"].reshape(want["scores"].shape).astype(np.float64)
    assert np.abs(s - want["scores"]).max() <= 1e-4 * max(1.0, np.abs(want["scores"]).max())
    # a2: selections bit-exact except inside the tie band
    sel = g["sel"].reshape(want["sel"].shape)
    tl.selection_rows_match(sel, want["scores"], want["sel"], w.k)
    # a3/a4/a5 for every unit, on the GPU's own selection where a row took the tie band
    ref, _ = tl.follow_gpu_selection(sel, want, x["q"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.cs)
    tl.check_layout(g, ref, w.B, w.Hkv, w.max_union, buf.Kst[0], buf.Vst[0])
    tl.check_attention(buf.out.cpu().numpy().reshape(ref["out"].shape), ref["out"])


def test_step_ping_pong_uses_buffer_of_layer_parity(dd):
    w = TINY
    x = tl.host_inputs(w)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap) as ctx:
        buf.run(ctx, layer=5)                       # odd layer -> buffer 1
        assert ctx.status() == 0
        M = int(buf.inter["miss_count"].item())
        assert M > 0
        assert np.all(tl.from_bf16(buf.Kst[0]).view(np.int16) == 3)     # buffer 0 untouched
        k1 = tl.from_bf16(buf.Kst[1]).reshape(-1, w.cs, w.d)[:M].copy()
        out1 = buf.out.clone()
        buf.run(ctx, layer=6)                       # even layer -> buffer 0, same data
        assert ctx.status() == 0
        assert np.array_equal(tl.from_bf16(buf.Kst[0]).reshape(-1, w.cs, w.d)[:M], k1)
        assert (buf.out == out1).all()              # bitwise deterministic


def test_step_capacity_error_skips_gather_and_attention(dd):
    w = TINY
    x = tl.host_inputs(w)
    buf = StepBuffers(w, x, cap=5)
    with dd.Context(shape_of(w), max_misses=5) as ctx:
        buf.run(ctx)
        assert ctx.status() == dd.DD_ERR_CAPACITY
        assert bool(buf.out.isnan().all())                   # attention did not run
        assert np.all(tl.from_bf16(buf.Kst[0]).view(np.int16) == 3)
    buf2 = StepBuffers(w, x)                                 # a context of the right size works
    with dd.Context(shape_of(w), max_misses=buf2.cap) as ctx:
        buf2.run(ctx)
        assert ctx.status() == 0
        assert not bool(buf2.out.isnan().any())


def test_empty_batch_is_a_no_op(dd):
    import torch
    w = Workload("empty", B=0, Hq=8, Hkv=2, d=128, L=1024, cs=16, k=8, n_q=2)
    with dd.Context(shape_of(w), max_misses=0) as ctx:
        e = torch.empty(0, device="cuda")
        z16 = torch.empty(0, dtype=torch.bfloat16, device="cuda")
        zi = torch.zeros(1, dtype=torch.int32, device="cuda")
        zu = torch.empty(0, dtype=torch.uint8, device="cuda")
        ctx.score_landmarks(z16, z16, e)
        zi.fill_(9)
        ctx.resolve_union(zi[:0], zi[:0], zi[:0], zi[:0], zu, zi[:0], zi, zi)
        assert int(zi.item()) == 0                           # miss_count written as 0
        assert ctx.status() == 0


def test_invalid_arguments_are_rejected_on_the_host(dd):
    from sparse_kv_offload_gb300.dd import Shape
    for bad in (Shape(1, 8, 2, 64, 1024, 16, 8, 2), Shape(1, 8, 3, 128, 1024, 16, 8, 2),
                Shape(1, 8, 2, 128, 1024, 24, 8, 2), Shape(1, 8, 2, 128, 1024, 16, 65, 2),
                Shape(1, 8, 2, 128, 1024, 16, 0, 2), Shape(1, 8, 2, 128, 1024, 16, 8, 9),
                Shape(1, 128, 2, 128, 1024, 16, 8, 2)):
        with pytest.raises(dd.DDError) as e:
            dd.Context(bad, max_misses=4)
        assert e.value.status == dd.DD_ERR_INVALID_ARG
    w = TINY
    import torch
    with dd.Context(shape_of(w), max_misses=4) as ctx:
        pageable = torch.zeros(w.B * w.Hkv * w.L * w.d, dtype=torch.bfloat16)
        with pytest.raises(ValueError):
            ctx.gather_kv(pageable, pageable, torch.zeros(1, dtype=torch.int32, device="cuda"),
                          torch.zeros(1, dtype=torch.int32, device="cuda"),
                          torch.empty(4 * w.cs * w.d, dtype=torch.bfloat16, device="cuda"),
                          torch.empty(4 * w.cs * w.d, dtype=torch.bfloat16, device="cuda"))


@pytest.mark.parametrize("w", STEP_CASES[:3], ids=lambda w: w.name)
def test_step_without_intermediates_gives_the_same_output(dd, w):
    # the step produces scores, selections and per-entry slots only when asked;
    # the attention output must not depend on that
    import torch
    x = tl.host_inputs(w)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=buf.hot) as ctx:
        buf.run(ctx, layer=0)
        full = buf.out.clone()
        mc = torch.empty(1, dtype=torch.int32, device="cuda")
        ctx.step(2, buf.q, buf.lm, buf.Kh, buf.Vh, buf.slot, buf.Khot, buf.Vhot, buf.Kst, buf.Vst, buf.out,
                 intermediates={"miss_count": mc})
        assert ctx.status() == 0
    assert torch.equal(full, buf.out)
    assert int(mc.item()) == int(buf.inter["miss_count"].item())


@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier", "lookback_word"])
def test_bounded_wait_runs_out_and_the_context_stays_usable(dd, kind):
    # a wait on something nothing signals gives up by itself (~2 s), reports a
    # timeout through the status word, and the next step on the context works
    import time
    w = TINY
    x = tl.host_inputs(w)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap) as ctx:
        t0 = time.perf_counter()
        ctx.selftest_bounded_wait(kind)
        assert ctx.status() == dd.DD_ERR_TIMEOUT
        assert 1.0 < time.perf_counter() - t0 < 30.0
        assert ctx.status() == 0                       # read and cleared
        buf.run(ctx)
        assert ctx.status() == 0
        assert not bool(buf.out.isnan().any())


def test_step_replays_in_a_cuda_graph(dd):
    # the step keeps no per-call state on the host that a replay would repeat
    # wrongly (the look-back epoch lives on the device), so a captured step
    # replays correctly, also after its inputs change in place
    import torch

    w = V_HOT
    x = tl.host_inputs(w)
    buf = StepBuffers(w, x)
    q2 = synth.queries(w.seed + 1, w.B, w.n_q, w.Hq, w.d, w.spec_scale)
    want = oracle.step(x["q"], x["lm"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.k, w.cs)
    want2 = oracle.step(q2, x["lm"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.k, w.cs)
    s = torch.cuda.Stream()
    mc = torch.zeros(1, dtype=torch.int32, device="cuda")
    sel = torch.zeros(w.B * w.n_q * w.Hkv * w.k, dtype=torch.int32, device="cuda")

    def step():
        ctx.step(0, buf.q, buf.lm, buf.Kh, buf.Vh, buf.slot, buf.Khot, buf.Vhot, buf.Kst, buf.Vst, buf.out,
                 intermediates={"miss_count": mc, "sel": sel}, stream=s)

    def check(want_):
        got_sel = sel.cpu().numpy().reshape(want_["sel"].shape)
        tl.selection_rows_match(got_sel, want_["scores"], want_["sel"], w.k)
        q_ = tl.from_bf16(buf.q).reshape(x["q"].shape)
        ref, _ = tl.follow_gpu_selection(got_sel, want_, q_, x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.cs)
        assert int(mc.item()) == ref["miss_count"]
        tl.check_attention(buf.out.cpu().numpy().reshape(ref["out"].shape), ref["out"])

    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=buf.hot) as ctx:
        with torch.cuda.stream(s):
            step()                                  # warm-up: host views, kernel attributes
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            step()
        for _ in range(3):
            buf.out.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert ctx.status() == 0
            check(want)
        buf.q.copy_(tl.to_bf16(q2))
        g.replay()
        torch.cuda.synchronize()
        assert ctx.status() == 0
        check(want2)


def test_step_trace_orders_the_kernels(dd):
    # the kernels' own timing words: a non-empty window per kernel, each kernel
    # starting after the one before it has finished (each waits for it before
    # its work), and the step's results unchanged
    import torch
    w = V_HOT
    x = tl.host_inputs(w)
    want = oracle.step(x["q"], x["lm"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.k, w.cs)
    buf = StepBuffers(w, x)
    trace = torch.zeros((3, 2, dd.TRACE_SLOTS), dtype=torch.int64, device="cuda")
    trace[:, 0] = -1
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=buf.hot) as ctx:
        ctx.step(0, buf.q, buf.lm, buf.Kh, buf.Vh, buf.slot, buf.Khot, buf.Vhot, buf.Kst, buf.Vst, buf.out,
                 trace=trace)
        torch.cuda.synchronize()
        assert ctx.status() == 0
    raw = trace.cpu().numpy().view(np.uint64)
    start, end = raw[:, 0].min(axis=1), raw[:, 1].max(axis=1)
    for j in range(3):
        assert 0 < start[j] < end[j] < np.uint64(2 ** 63), f"kernel {j}: window {start[j]}..{end[j]}"
    assert end[0] <= start[1] and end[1] <= start[2]
    assert np.all((raw[:, 0] == np.uint64(2 ** 64 - 1)) == (raw[:, 1] == 0))   # an SM either ran CTAs or not
    tl.check_attention(buf.out.cpu().numpy().reshape(want["out"].shape), want["out"])


@pytest.mark.parametrize("mode", [0, 2], ids=["zerocopy", "kernel"])
def test_step_follows_the_gpu_selection_in_the_tie_band(dd, mode):
    # Landmarks built so that two chunks A > B tie in fp32 but not in fp64:
    # the real query's scores are G*2^16 + G*2^-9 for A and G*2^16 for B, and
    # 2^-7 is below half an fp32 ulp at 2^18, so the GPU sees equal scores and
    # keeps the lower index B where the oracle keeps A.  The speculative query
    # scores A and B exactly equal (both keep B), so the oracle's union has one
    # chunk more than the GPU's.  The step must then match the oracle's union,
    # miss list, staging bytes and attention on the GPU's own selection.
    w, x, q, lm = tl.tie_band_inputs()
    want = oracle.step(q, lm, x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.k, w.cs)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=buf.hot) as ctx:
        buf.run(ctx, layer=0, mode=mode)
        assert ctx.status() == 0
    g = {k: v.cpu().numpy() for k, v in buf.inter.items()}
    sel = g["sel"].reshape(want["sel"].shape)
    tl.selection_rows_match(sel, want["scores"], want["sel"], w.k)
    ref, tie_units = tl.follow_gpu_selection(sel, want, q, x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.cs)
    assert tie_units.all()                                   # every unit took the tie path on purpose
    assert np.all(ref["union_cnt"] == want["union_cnt"] - 1)
    tl.check_layout(g, ref, w.B, w.Hkv, w.max_union, buf.Kst[0], buf.Vst[0])
    tl.check_attention(buf.out.cpu().numpy().reshape(ref["out"].shape), ref["out"])
