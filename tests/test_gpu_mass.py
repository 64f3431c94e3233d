"""GPU parity of the coverage-budget selection (MOIRA reading: per row, the
smallest chunk set whose estimated attention mass reaches gamma) and of a
step that uses it.  The GPU sums the masses in fp32 and the oracle in fp64,
so where a row's count sits on the gamma boundary either count is correct:
the test takes the GPU's count when the fp64 masses put it within 1e-5 of
gamma, and requires exactly the oracle's chunks otherwise."""
import math

import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300 import synth
from sparse_kv_offload_gb300.workloads import TINY

import dd_testlib as tl
from test_gpu_parity import V_5Q, V_HOT, shape_of
from test_gpu_step import StepBuffers

pytestmark = pytest.mark.gpu

MASS_EPS = 1e-5


@pytest.fixture(scope="module")
def dd():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from sparse_kv_offload_gb300 import build
    build.build()
    from sparse_kv_offload_gb300 import dd as mod
    return mod


def check_mass_rows(gpu_sel, gpu_cnt, scores, k_max, gamma, tau, k_min=1):
    """Every GPU row is a valid coverage selection of the fp64 scores; returns the
    mask of rows equal to the oracle's."""
    want_sel, want_cnt = oracle.select_by_mass(scores, k_max, gamma, tau, k_min)
    C = scores.shape[-1]
    g_sel, g_cnt = gpu_sel.reshape(-1, k_max), gpu_cnt.reshape(-1)
    w_sel, w_cnt = want_sel.reshape(-1, k_max), want_cnt.reshape(-1)
    s = scores.reshape(-1, C)
    same = np.all(g_sel == w_sel, axis=1) & (g_cnt == w_cnt)
    for r in np.nonzero(~same)[0]:
        n = int(g_cnt[r])
        assert k_min <= n <= k_max
        assert np.all(g_sel[r, n:] == -1)
        chosen = g_sel[r, :n]
        assert list(chosen) == sorted(set(chosen.tolist())), f"row {r}: not ascending distinct"
        row = s[r]
        w = np.exp(tau * (row - row.max()))
        w /= w.sum()
        order = np.lexsort((np.arange(C), -row))
        csum = np.cumsum(w[order])
        # the count: gamma reached at n (unless clamped at k_max), not yet at n - 1 (unless clamped at k_min)
        assert n == k_max or csum[n - 1] >= gamma - MASS_EPS, f"row {r}: mass {csum[n - 1]} < gamma"
        assert n == k_min or csum[n - 2] < gamma + MASS_EPS, f"row {r}: a smaller set already reaches gamma"
        # the chunks: the top n, ties inside the top-k band
        tl.selection_rows_match(chosen[None], row[None], np.sort(order[:n])[None], n)
    return same.reshape(gpu_cnt.shape)


@pytest.mark.parametrize("C,k_max,gamma,tau", [(256, 64, 0.9, 0.3), (2048, 256, 0.5, 0.05), (2048, 64, 0.99, 2.0),
                                               (4096, 1024, 0.8, 0.02), (1000, 37, 0.7, 0.5), (64, 64, 1.0, 0.05),
                                               (64, 64, 0.999, 0.3)])
def test_topk_mass_matches_oracle_and_repeats(dd, C, k_max, gamma, tau):
    import torch
    from sparse_kv_offload_gb300.dd import Shape
    B, n_q, Hkv, G = 2, 2, 3, 4
    sh = Shape(B, G * Hkv, Hkv, 128, C * 16, 16, k_max, n_q)
    rows = B * n_q * Hkv
    s = synth.normal_f32(C + k_max, synth.TID_SCORE, np.arange(rows * C, dtype=np.uint64)) * np.float32(8.0)
    s = s.reshape(B, n_q, Hkv, C)
    s[0, 0, 0, 5:9] = s[0, 0, 0, 5]                          # exact ties
    scores = torch.from_numpy(s.reshape(-1)).cuda()
    scale = tau * G                                            # tau = scale / G
    sel = torch.empty(rows * k_max, dtype=torch.int32, device="cuda")
    cnt = torch.empty(rows, dtype=torch.int32, device="cuda")
    with dd.Context(sh, max_misses=1) as ctx:
        ctx.select_topk_mass(scores, sel, gamma, k_min=1, sel_cnt=cnt, softmax_scale=scale)
        first = (sel.clone(), cnt.clone())
        ctx.select_topk_mass(scores, sel, gamma, k_min=1, sel_cnt=cnt, softmax_scale=scale)
        assert ctx.status() == 0
    assert torch.equal(first[0], sel) and torch.equal(first[1], cnt)
    same = check_mass_rows(sel.cpu().numpy(), cnt.cpu().numpy(), s.astype(np.float64), k_max, gamma,
                           float(np.float32(scale)) / G)
    assert same.mean() > 0.8


def test_topk_mass_clamps_to_k_min(dd):
    import torch
    from sparse_kv_offload_gb300.dd import Shape
    C, k_max = 512, 32
    sh = Shape(1, 8, 2, 128, C * 16, 16, k_max, 2)
    s = np.zeros((1, 2, 2, C), np.float32)
    s[..., 17] = 1000.0                                        # one chunk holds all the mass
    sel = torch.empty(4 * k_max, dtype=torch.int32, device="cuda")
    cnt = torch.empty(4, dtype=torch.int32, device="cuda")
    with dd.Context(sh, max_misses=1) as ctx:
        ctx.select_topk_mass(torch.from_numpy(s.reshape(-1)).cuda(), sel, 0.9, k_min=3, sel_cnt=cnt,
                             softmax_scale=1.0)
        assert ctx.status() == 0
    assert cnt.cpu().tolist() == [3, 3, 3, 3]
    rows = sel.cpu().numpy().reshape(4, k_max)
    assert np.all(rows[:, :3] == [0, 1, 17]) and np.all(rows[:, 3:] == -1)


# scales sharper than 1/sqrt(d) so that the budgets vary across rows of these random inputs
@pytest.mark.parametrize("w,scale,gamma", [(TINY, 4.0, 0.9), (TINY, 2.0, 0.5), (V_HOT, 1.0, 0.9),
                                           (V_5Q, 2.0, 0.9), (V_5Q, 1.0, 0.5)],
                         ids=["tiny_s4_g.9", "tiny_s2_g.5", "hot_s1_g.9", "5q_s2_g.9", "5q_s1_g.5"])
def test_step_with_coverage_budget_matches_oracle(dd, w, scale, gamma):
    import torch
    x = tl.host_inputs(w)
    want = oracle.step(x["q"], x["lm"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.k, w.cs, scale=scale,
                       gamma=gamma)
    buf = StepBuffers(w, x)
    cnt = torch.empty(w.B * w.n_q * w.Hkv, dtype=torch.int32, device="cuda")
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=buf.hot) as ctx:
        ctx.step(0, buf.q, buf.lm, buf.Kh, buf.Vh, buf.slot, buf.Khot, buf.Vhot, buf.Kst, buf.Vst, buf.out,
                 softmax_scale=scale, intermediates=buf.inter, mass_gamma=gamma, sel_cnt=cnt)
        assert ctx.status() == 0
    G = w.Hq // w.Hkv
    sel = buf.inter["sel"].cpu().numpy().reshape(want["sel"].shape)
    same = check_mass_rows(sel, cnt.cpu().numpy().reshape(want["sel_cnt"].shape), want["scores"], w.k, gamma,
                           scale / G)
    assert len(set(want["sel_cnt"].reshape(-1).tolist())) > 1          # the budgets do vary
    # union, miss list, slots, staging bytes and attention of every unit, on the GPU's own
    # rows where a row's count or chunks took the gamma boundary or the tie band
    g = {k: v.cpu().numpy() for k, v in buf.inter.items()}
    ref, _ = tl.follow_gpu_selection(sel, want, x["q"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.cs,
                                     scale=scale)
    tl.check_layout(g, ref, w.B, w.Hkv, w.max_union, buf.Kst[0], buf.Vst[0])
    tl.check_attention(buf.out.cpu().numpy().reshape(ref["out"].shape), ref["out"])


def test_coverage_budget_rejects_bad_arguments(dd):
    import torch
    w = TINY
    x = tl.host_inputs(w)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap) as ctx:
        for k_min in (0, w.k + 1):
            with pytest.raises(dd.DDError):
                ctx.step(0, buf.q, buf.lm, buf.Kh, buf.Vh, buf.slot, None, None, buf.Kst, buf.Vst, buf.out,
                         mass_gamma=0.9, mass_k_min=k_min)
