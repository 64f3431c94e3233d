"""Rows the fused selection cannot settle by its threshold filter alone: when
many chunks share the top score, more chunks than the candidate capacity pass
the filter and the row is selected by a radix select over the whole row.
Equal scores are broken by the lower chunk index, as in the oracle (OasisKV
summary, Methodology: top-K blocks per KV head)."""
import numpy as np
import pytest

import oracle
from sparse_kv_offload_gb300.workloads import Workload

import dd_testlib as tl
from test_gpu_parity import shape_of
from test_gpu_step import StepBuffers

pytestmark = pytest.mark.gpu

# 2,048 chunks, top-16: the filter keeps at most 256 candidates per row
W_TIES = Workload("ties_b2_ctx32k", B=2, Hq=8, Hkv=2, d=128, L=32768, cs=16, k=16, n_q=2,
                  spec_scale=(0.0, 0.3), seed=4100)


@pytest.fixture(scope="module")
def dd():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from sparse_kv_offload_gb300 import build
    build.build()
    from sparse_kv_offload_gb300 import dd as mod
    return mod


def _with_landmarks(w, make):
    x = dict(tl.host_inputs(w))
    lm = x["lm"].copy()                       # [B, Hkv, C, d] bf16 bits
    make(lm)
    x["lm"] = lm
    return x


def _zero(lm):
    lm[:] = 0                                 # every score 0: the first k chunks win


def _tied_block(lm):
    # 600 chunks of every unit share one landmark (a copy of chunk 7's), the
    # rest keep their own: most query rows rank the tied block first or near it
    idx = np.random.default_rng(5).choice(lm.shape[2], 600, replace=False)
    lm[:, :, idx] = lm[:, :, 7:8]


@pytest.mark.parametrize("make", [_zero, _tied_block], ids=["all_zero", "tied_block"])
def test_tied_rows_fall_back_and_match_oracle(dd, make):
    w = W_TIES
    x = _with_landmarks(w, make)
    want = oracle.step(x["q"], x["lm"], x["K"], x["V"], x["slot"], x["Khot"], x["Vhot"], w.k, w.cs)
    buf = StepBuffers(w, x)
    with dd.Context(shape_of(w), max_misses=buf.cap, hot_slots=buf.hot) as ctx:
        buf.run(ctx, layer=0)
        assert ctx.status() == 0
    sel = buf.inter["sel"].cpu().numpy().reshape(want["sel"].shape)
    if make is _zero:
        assert np.all(sel == np.arange(w.k))                              # lowest chunks among equal scores
    ok = tl.selection_rows_match(sel, want["scores"], want["sel"], w.k)
    assert ok.all()
    M = int(buf.inter["miss_count"].item())
    assert M == want["miss_count"]
    assert np.array_equal(buf.inter["miss_list"].cpu().numpy()[:M], want["miss_list"])
    assert np.array_equal(buf.inter["attn_slot"].cpu().numpy().reshape(want["attn_slot"].shape), want["attn_slot"])
    tl.check_attention(buf.out.cpu().numpy().reshape(want["out"].shape), want["out"])
