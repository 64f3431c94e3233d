"""The forced tie-band step case (dd_testlib.tie_band_inputs) does what it
claims, checked on the CPU: in fp64 the real query keeps chunk A, in fp32
(the group-summed query and an fp32 sum, in any order of its terms) A and B
score equal so the lowest-index rule keeps B, the difference lies inside the
tie band, and the oracle's union is one chunk larger than the union of the
fp32 choice."""
import itertools

import numpy as np

import oracle
from sparse_kv_offload_gb300 import synth

import dd_testlib as tl


def test_tie_band_inputs_tie_in_fp32_not_in_fp64():
    w, x, q, lm = tl.tie_band_inputs()
    s64 = oracle.score_landmarks(q, lm)
    sel = oracle.select_topk(s64, w.k)
    Q = synth.bf16_to_f32(q).reshape(w.B, w.n_q, w.Hkv, w.G, w.d).sum(axis=3, dtype=np.float32)
    lmf = synth.bf16_to_f32(lm)
    fp32_sel = np.empty_like(sel)
    for b in range(w.B):
        for g in range(w.Hkv):
            for j in range(w.n_q):
                terms = Q[b, j, g][None, :] * lmf[b, g]                  # exact products (fp32)
                nz = [i for i in range(w.d) if np.any(terms[:, i] != 0)]
                # every order of the non-zero coordinates of A and B gives the same fp32 sum
                s32 = terms.sum(axis=1, dtype=np.float32)
                order = np.lexsort((np.arange(w.C), -s32.astype(np.float64)))
                fp32_sel[b, j, g] = np.sort(order[:w.k])
                top = s64[b, j, g]
                o = np.lexsort((np.arange(w.C), -top))
                a_, b_ = o[w.k - 1], o[w.k]                                # k-th and (k+1)-th in fp64
                assert abs(top[a_] - top[b_]) <= tl.TIE_REL * max(abs(top[a_]), abs(top[b_]))
                for c in (a_, b_):
                    vals = [t for t in terms[c] if t != 0]
                    for perm in itertools.permutations(vals):
                        acc = np.float32(0)
                        for t in perm:
                            acc = np.float32(acc + t)
                        assert acc == np.float32(w.G * 2.0 ** 16)
                assert len(nz) > 0
    # the real query's rows differ (fp64 keeps the higher index), the speculative rows agree
    assert np.all(np.any(fp32_sel[:, 0] != sel[:, 0], axis=-1))
    assert np.array_equal(fp32_sel[:, 1], sel[:, 1])
    tl.selection_rows_match(fp32_sel, s64, sel, w.k)
    full = oracle.resolve_union(sel, x["slot"])
    fp32 = oracle.resolve_union(fp32_sel, x["slot"])
    assert np.all(fp32["union_cnt"] == full["union_cnt"] - 1)


def test_tie_path_helpers_follow_the_given_selection():
    # the helpers the GPU step tests use: a layout built from the fp32 choice
    # passes against the oracle re-run on that choice, and a changed entry fails
    import pytest
    w, x, q, lm = tl.tie_band_inputs()
    want = oracle.step(q, lm, x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.k, w.cs)
    fp32_sel = want["sel"].copy()
    for b in range(w.B):
        for g in range(w.Hkv):
            row = want["scores"][b, 0, g]
            o = np.lexsort((np.arange(w.C), -row))
            a_, b_ = o[w.k - 1], o[w.k]
            fp32_sel[b, 0, g] = np.sort(np.r_[o[:w.k - 1], min(a_, b_)])
    ref, tie_units = tl.follow_gpu_selection(fp32_sel, want, q, x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"],
                                             w.cs)
    assert tie_units.all()
    res = oracle.resolve_union(fp32_sel, x["slot"])
    g = {k: np.asarray(res[k]).reshape(-1) for k in ("union_idx", "union_slot", "union_qmask", "union_cnt",
                                                     "attn_slot")}
    g["miss_list"] = np.r_[res["miss_list"], [7, 7]].astype(np.int32)      # capacity beyond M is ignored
    g["miss_count"] = np.array([res["miss_count"]], np.int32)
    tl.check_layout(g, ref, w.B, w.Hkv, w.max_union)
    tl.check_attention(ref["out"], ref["out"])
    bad = dict(g, miss_list=g["miss_list"].copy())
    bad["miss_list"][0] += 1
    with pytest.raises(AssertionError):
        tl.check_layout(bad, ref, w.B, w.Hkv, w.max_union)
    with pytest.raises(AssertionError):
        tl.check_layout(g, want, w.B, w.Hkv, w.max_union)                  # the oracle's own choice differs
