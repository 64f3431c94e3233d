"""A seeded sweep of small random shapes through the whole step against the
oracle: queries per request, group size, chunk size, context (ragged chunk
counts), k up to C, residency, single-unit batches.  Each case checks the
selections (modulo the tie band), the union and miss layout, the staging
bytes and the attention output, in both gather modes."""
import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300.workloads import Workload

import dd_testlib as tl
from test_gpu_parity import shape_of
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


def _cases(n=16, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        n_q = int(rng.integers(1, 9))
        Hkv = int(rng.choice([1, 2, 3, 4]))
        G = int(rng.choice([1, 2, 4, 8]))
        while n_q * G > 64:
            G //= 2
        cs = int(rng.choice([16, 32, 64]))
        C = int(rng.integers(3, 700))
        k = int(rng.integers(1, min(C, 96) + 1)) if i % 5 else C      # every fifth case: k = C
        B = int(rng.integers(1, 4))
        spec = (0.0,) + tuple(float(x) for x in rng.uniform(0.05, 0.5, n_q - 1))
        res = ["none", "uniform"][int(rng.integers(0, 2))]
        out.append(Workload(f"rand{i}", B=B, Hq=Hkv * G, Hkv=Hkv, d=128, L=C * cs, cs=cs, k=k, n_q=n_q,
                            spec_scale=spec, seed=3000 + i, residency=res, resident_frac=float(rng.uniform(0.1, 0.6))))
    return out


CASES = _cases()
_INPUTS = {}


def _inputs(w):
    """Host inputs and the oracle's step, shared by both gather modes."""
    if w.name not in _INPUTS:
        x = tl.host_inputs(w)
        _INPUTS[w.name] = (x, oracle.step(x["q"], x["lm"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"],
                                          w.k, w.cs))
    return _INPUTS[w.name]


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["zerocopy", "memcpy", "kernel"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: f"{w.name}_B{w.B}_G{w.G}_nq{w.n_q}_C{w.C}_k{w.k}_cs{w.cs}")
def test_random_shape_step_matches_oracle(dd, w, mode):
    x, want = _inputs(w)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=buf.hot) as ctx:
        buf.run(ctx, layer=3, mode=mode)
        assert ctx.status() == 0
    g = {k: v.cpu().numpy() for k, v in buf.inter.items()}
    sel = g["sel"].reshape(want["sel"].shape)
    tl.selection_rows_match(sel, want["scores"], want["sel"], w.k)
    # union, query masks, slots, miss list and staging bytes of every unit, on the
    # GPU's own selection where a row took the tie band
    ref, _ = tl.follow_gpu_selection(sel, want, x["q"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.cs)
    tl.check_layout(g, ref, w.B, w.Hkv, w.max_union, buf.Kst[1], buf.Vst[1])
    tl.check_attention(buf.out.cpu().numpy().reshape(ref["out"].shape), ref["out"])
