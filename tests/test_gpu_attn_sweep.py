"""A seeded sweep of the stand-alone attention call against the oracle, built
from random per-query selections rather than from a scoring pass, so that the
split-K merge sees what real selections rarely produce together: units whose
union spans one CTA's slice or many, empty unions next to full ones, queries
that selected nothing, two to four m-tiles of query vectors, chunks from the
hot pool and from staging in any mix, and the step's tail rows on or off."""
import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300 import synth

import dd_testlib as tl

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def dd():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from sparse_kv_offload_gb300 import build
    build.build()
    from sparse_kv_offload_gb300 import dd as mod
    return mod


def _bf16(rng, shape, scale=1.0):
    return synth.f32_to_bf16((rng.standard_normal(shape) * scale).astype(np.float32))


def make_case(seed):
    """Random selections of one attention call and everything the call and the oracle need."""
    rng = np.random.default_rng(seed)
    n_q = int(rng.integers(1, 9))
    G = int(rng.choice([1, 2, 4, 8]))
    while n_q * G > 64:
        G //= 2
    B, Hkv = int(rng.integers(1, 4)), int(rng.choice([1, 2, 4]))
    cs = int(rng.choice([16, 32, 64]))
    C = int(rng.integers(4, 600))
    k = int(rng.integers(1, min(C, 48) + 1))
    p_hot = float(rng.choice([0.0, 0.5, 1.0]))
    umax = min(C, n_q * k)
    NO = oracle.NO_SLOT
    attn_slot = np.full((B, n_q, Hkv, k), NO, np.int32)
    union_slot = np.zeros((B, Hkv, umax), np.int32)
    union_qmask = np.zeros((B, Hkv, umax), np.uint8)
    union_cnt = np.zeros((B, Hkv), np.int32)
    n_hot = n_miss = 0
    for b in range(B):
        for g in range(Hkv):
            empty_unit = rng.random() < 0.15
            picks = []
            for j in range(n_q):
                kj = 0 if empty_unit or rng.random() < 0.1 else int(rng.integers(1, k + 1))
                picks.append(set(rng.choice(C, size=kj, replace=False).tolist()))
            union = sorted(set().union(*picks))
            union_cnt[b, g] = len(union)
            for i, c in enumerate(union):
                if rng.random() < p_hot:
                    union_slot[b, g, i] = n_hot
                    n_hot += 1
                else:
                    union_slot[b, g, i] = -(n_miss + 1)          # dense ordinals in (b, g, c) order
                    n_miss += 1
                union_qmask[b, g, i] = sum(1 << j for j in range(n_q) if c in picks[j])
            for j in range(n_q):
                codes = [union_slot[b, g, union.index(c)] for c in sorted(picks[j])]
                attn_slot[b, j, g, :len(codes)] = codes
    # hot-pool slots in a shuffled order, with spare slots nothing points to
    pool = n_hot + int(rng.integers(0, 4))
    if pool:
        perm = rng.permutation(pool)
        union_slot = np.where(union_slot >= 0, perm[np.maximum(union_slot, 0)], union_slot).astype(np.int32)
        attn_slot = np.where(attn_slot >= 0, perm[np.maximum(attn_slot, 0)], attn_slot).astype(np.int32)
    return dict(B=B, Hkv=Hkv, G=G, n_q=n_q, cs=cs, C=C, k=k, umax=umax,
                q=_bf16(rng, (B, n_q, Hkv * G, D)),
                Khot=_bf16(rng, (pool, cs, D)), Vhot=_bf16(rng, (pool, cs, D)),
                Kst=_bf16(rng, (max(1, n_miss), cs, D)), Vst=_bf16(rng, (max(1, n_miss), cs, D)),
                Kt=_bf16(rng, (B, n_q, Hkv, D)), Vt=_bf16(rng, (B, n_q, Hkv, D)),
                attn_slot=attn_slot, union_slot=union_slot, union_qmask=union_qmask, union_cnt=union_cnt,
                n_hot_pool=pool, n_miss=n_miss)


CASES = list(range(5100, 5116))


@pytest.mark.parametrize("tails", [False, True], ids=["no_tail", "tail"])
@pytest.mark.parametrize("seed", CASES)
def test_attention_sweep_matches_oracle(dd, seed, tails):
    import torch
    x = make_case(seed)
    kt, vt = (x["Kt"], x["Vt"]) if tails else (None, None)
    want = oracle.sparse_attn_decode(x["q"], x["Khot"], x["Vhot"], x["Kst"], x["Vst"], x["attn_slot"], x["cs"],
                                     K_tail=kt, V_tail=vt)
    B, n_q, Hkv, G = x["B"], x["n_q"], x["Hkv"], x["G"]
    sh = dd.Shape(B, Hkv * G, Hkv, D, x["C"] * x["cs"], x["cs"], x["k"], n_q)
    out = torch.full((B * n_q * Hkv * G * D,), float("nan"), device="cuda")
    extra = dict(K_tail=tl.to_bf16(kt), V_tail=tl.to_bf16(vt)) if tails else {}
    with dd.Context(sh, max_misses=max(1, x["n_miss"]), hot_slots=x["n_hot_pool"]) as ctx:
        ctx.sparse_attn_decode(tl.to_bf16(x["q"]), tl.to_bf16(x["Khot"]), tl.to_bf16(x["Vhot"]),
                               tl.to_bf16(x["Kst"]), tl.to_bf16(x["Vst"]), tl.to_i32(x["union_slot"]),
                               torch.from_numpy(x["union_qmask"].reshape(-1)).cuda(), tl.to_i32(x["union_cnt"]),
                               tl.to_i32(np.array([x["n_miss"]])), out, **extra)
        assert ctx.status() == 0
    tl.check_attention(out.cpu().numpy().reshape(want.shape), want)
