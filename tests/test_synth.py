"""The seeded input generator (CPU): published test vector, distribution, structure."""
import numpy as np

from sparse_kv_offload_gb300 import synth
from sparse_kv_offload_gb300.workloads import LLAMA8B_32K, STRESS_512K


def test_splitmix64_reference_vector():
    # SplitMix64 seeded with 1234567: the first five outputs of the reference generator
    state = np.uint64(1234567)
    with np.errstate(over="ignore"):
        out = synth._mix(state + (np.arange(5, dtype=np.uint64) + np.uint64(1)) * synth.GAMMA)
    assert [int(x) for x in out] == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                                     4593380528125082431, 16408922859458223821]


def test_irwin_hall_normal_is_exact_and_standard():
    x = synth.normal_f32(7, 1, np.arange(1 << 20, dtype=np.uint64))
    assert abs(float(x.mean())) < 5e-3 and abs(float(x.var()) - 1) < 5e-3
    assert x.min() > -6 and x.max() < 6
    assert np.all(x * 65536 == np.round(x * 65536))           # multiples of 2^-16
    # counter-based: any element can be drawn on its own
    idx = np.array([5, 1 << 33, 123456789], np.uint64)
    full = synth.normal_f32(7, 1, idx)
    assert np.array_equal(full, np.array([synth.normal_f32(7, 1, np.array([i], np.uint64))[0] for i in idx]))


def test_bf16_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 0.0, 1.0 + 2**-7 + 2**-9], np.float32)
    got = synth.bf16_to_f32(synth.f32_to_bf16(vals))
    assert got.tolist() == [1.0, 1.0, 1.0 + 2**-6, -2.5, 0.0, 1.0 + 2**-7]


def test_hot_bias_and_zipf_structure():
    w = LLAMA8B_32K
    bias = synth.hot_chunk_bias(w.seed, 2, w.Hkv, w.C, w.hot_frac, w.bias_sigma)
    assert np.all((bias == 0) | (bias == 3.0))
    assert np.all((bias > 0).sum(-1) == round(0.01 * w.C))
    z = synth.zipf_chunk_bias(STRESS_512K.seed, 1, 2, 64, 1.1, 3.0)
    assert np.isclose(z.max(), 3.0) and np.all(np.sort(z[0, 0])[::-1] == np.sort(z[0, 1])[::-1])


def test_residency_tables():
    slot = synth.uniform_residency(3, 2, 3, 10, 0.5)
    assert np.all((slot >= 0).sum(-1) == 5)
    assert sorted(slot[slot >= 0].tolist()) == list(range(30))
    U = [set(range(0, 10, 2)) for _ in range(6)]
    carry = synth.carried_residency(4, U, 2, 3, 20, 0.8)
    for u in range(6):
        row = carry.reshape(6, 20)[u]
        assert (row >= 0).sum() == 5 and sum(1 for c in U[u] if row[c] >= 0) == 4


def test_queries_spec_is_real_plus_scaled_noise():
    q = synth.queries(9, 2, 3, 4, 128, (0.0, 0.2, 0.4))
    real = synth.bf16_to_f32(q[:, 0]).astype(np.float64)
    for j, s in ((1, 0.2), (2, 0.4)):
        diff = synth.bf16_to_f32(q[:, j]).astype(np.float64) - real
        assert 0.8 * s < diff.std() < 1.2 * s


def test_drift_queries_follow_their_definition():
    seed, B, n_q, Hq, d, T = 7, 2, 3, 4, 128, 5
    q = synth.drift_queries(seed, B, n_q, Hq, d, T, 0.3, 0.1, layer=2)
    assert q.shape == (T, B, n_q, Hq, d) and q.dtype == np.uint16
    n = B * Hq * d
    idx = np.arange(n, dtype=np.uint64)
    base = synth.bf16_to_f32(synth.f32_to_bf16(synth.normal_f32(seed, synth.tensor_id(synth.TID_Q_REAL, 2), idx)))
    # the base is the layer's real query of the plain generator
    assert np.array_equal(synth.f32_to_bf16(base).reshape(B, Hq, d), synth.queries(seed, B, 1, Hq, d, (0.0,), 2)[:, 0])
    real = [synth.bf16_to_f32(q[t, :, 0]).reshape(-1) for t in range(T)]
    for t in range(T):
        drift = synth.normal_f32(seed, synth.tensor_id(synth.TID_DRIFT + t, 2), idx)
        assert np.array_equal(q[t, :, 0].reshape(-1), synth.f32_to_bf16(base + np.float32(0.3) * drift))
        for j in range(1, n_q):
            eta = synth.normal_f32(seed, synth.tensor_id(synth.TID_DRIFT_SPEC + t, 2), idx + np.uint64(j * n))
            want = synth.f32_to_bf16(real[(t + 1) % T] + np.float32(0.1) * eta)
            assert np.array_equal(q[t, :, j].reshape(-1), want)
    assert np.array_equal(q, synth.drift_queries(seed, B, n_q, Hq, d, T, 0.3, 0.1, layer=2))
