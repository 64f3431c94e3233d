"""The allocation-free attention entry point, for callers that cannot
allocate device memory (their device memory is owned by their own pool, or
they may not call cudaMalloc between decode steps because it can synchronise
the device): its output must equal the context-based dd_sparse_attn_decode's
and the oracle's, within the attention tolerance of the other tests, on two
calls in a row that share the library's fixed scratch array.

Collected last on purpose, so that a run stopping at the first failure has
already run every other test; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300.workloads import STRESS_512K, Workload

import dd_testlib as tl

pytestmark = pytest.mark.gpu

CASES = [
    STRESS_512K.scaled(name="noalloc_hot_and_staging", B=1, L=16384, k=16),        # cs=64, half resident
    Workload("noalloc_five_queries", B=2, Hq=64, Hkv=8, d=128, L=4096, cs=16, k=40, n_q=5,
             spec_scale=(0.0, 0.2, 0.4, 0.6, 0.8), seed=1104),
]


@pytest.fixture(scope="module")
def dd():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from sparse_kv_offload_gb300 import build
    build.build()
    from sparse_kv_offload_gb300 import dd as mod
    return mod


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_attention_equals_context_attention_twice(dd, w):
    import torch
    x = tl.host_inputs(w)
    sel = oracle.select_topk(oracle.score_landmarks(x["q"], x["lm"]), w.k)
    # the oracle's attention on this selection, from its own union and gather
    res = oracle.resolve_union(sel, x["slot"])
    Ks, Vs = oracle.gather_kv(x["K"], x["V"], res["miss_list"], w.cs)
    want_oracle = oracle.sparse_attn_decode(x["q"], x["Khot"], x["Vhot"], Ks, Vs, res["attn_slot"], w.cs)
    shape = dd.Shape(w.B, w.Hq, w.Hkv, w.d, w.L, w.cs, w.k, w.n_q)
    cap, hot = w.max_misses, x["Khot"].shape[0]
    nu = w.B * w.Hkv * w.max_union
    with dd.Context(shape, max_misses=cap, hot_slots=hot) as ctx:
        union_idx = torch.empty(nu, dtype=torch.int32, device="cuda")
        union_slot = torch.empty(nu, dtype=torch.int32, device="cuda")
        union_qmask = torch.empty(nu, dtype=torch.uint8, device="cuda")
        union_cnt = torch.empty(w.B * w.Hkv, dtype=torch.int32, device="cuda")
        miss_list = torch.empty(cap, dtype=torch.int32, device="cuda")
        miss_count = torch.empty(1, dtype=torch.int32, device="cuda")
        ctx.resolve_union(tl.to_i32(sel), tl.to_i32(x["slot"]), union_idx, union_slot, union_qmask, union_cnt,
                          miss_list, miss_count)
        Kst = torch.empty(cap * w.cs * w.d, dtype=torch.bfloat16, device="cuda")
        Vst = torch.empty_like(Kst)
        ctx.gather_kv(tl.to_bf16(x["K"], "cpu", pin=True), tl.to_bf16(x["V"], "cpu", pin=True), miss_list,
                      miss_count, Kst, Vst)
        q = tl.to_bf16(x["q"])
        Khot = tl.to_bf16(x["Khot"]) if hot else None
        Vhot = tl.to_bf16(x["Vhot"]) if hot else None
        ref = torch.empty(w.B * w.n_q * w.Hq * w.d, device="cuda")
        ctx.sparse_attn_decode(q, Khot, Vhot, Kst, Vst, union_slot, union_qmask, union_cnt, miss_count, ref)
        assert ctx.status() == 0
        want = ref.cpu().numpy().reshape(w.B, w.n_q, w.Hq, w.d)
        tl.check_attention(want, want_oracle)
        for call in range(2):
            out = torch.full_like(ref, float("nan"))
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            dd.sparse_attn_decode_noalloc(shape, hot, cap, q, Khot, Vhot, Kst, Vst, union_slot, union_qmask,
                                          union_cnt, miss_count, out, status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
            got = out.cpu().numpy().reshape(want.shape)
            tl.check_attention(got, want)
            tl.check_attention(got, want_oracle)


def test_noalloc_refuses_shapes_beyond_its_scratch(dd):
    # the 32B-class, five-query layer at 128 requests: its per-unit partials
    # alone (units x 40 query vectors x 128 fp32) exceed the 16 MiB array,
    # whatever the GPU's SM count adds for the per-CTA partials
    B, Hq, Hkv, L, cs, k, n_q = 128, 64, 8, 32768, 16, 128, 5
    per_unit_partials = B * Hkv * (n_q * Hq // Hkv) * 128 * 4
    assert per_unit_partials > 16 << 20
    big = dd.Dims(B, Hq, Hkv, 128, L, cs, k, n_q)
    lib = ctypes.CDLL(dd.LIB_PATH)
    fn = lib.dd_sparse_attn_decode_noalloc
    fn.restype = ctypes.c_int32
    fn.argtypes = dd._lib.dd_sparse_attn_decode_noalloc.argtypes
    r = fn(ctypes.byref(big), 0, 1000, *([None] * 9), 0.0, None, None, None)
    assert r == dd.DD_ERR_CAPACITY
