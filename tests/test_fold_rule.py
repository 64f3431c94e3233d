"""When dd_step folds the landmark scoring into its selection kernel (host
rule, no device call): mean landmarks, a fixed k, units filling 3/4 of the
SMs or more in one wave, and the unit's key rows and landmark ring fitting
one CTA's shared memory."""
import pytest

from sparse_kv_offload_gb300 import dd


def shape(B, Hkv=8, Hq=32, L=32768, cs=16, k=64, n_q=2):
    return dd.Shape(B, Hq, Hkv, 128, L, cs, k, n_q)


def test_folds_when_the_units_fill_one_wave():
    assert dd.step_folds_scoring(shape(16), 152) == 5           # 128 units on 152 SMs
    assert dd.step_folds_scoring(shape(19), 152) == 5           # 152 units: one per SM
    assert dd.step_folds_scoring(shape(15), 152) == 5           # 120 units >= 114


@pytest.mark.parametrize("B", [8, 14, 20, 32])
def test_keeps_the_scoring_kernel_outside_one_wave(B):
    # 64 and 112 units leave SMs idle, 160 and 256 need a second wave
    assert dd.step_folds_scoring(shape(B), 152) == 0


def test_keeps_the_scoring_kernel_for_min_max_landmarks_and_coverage_budgets():
    assert dd.step_folds_scoring(shape(16), 152, lm_kind=dd.LM_MINMAX) == 0
    assert dd.step_folds_scoring(shape(16), 152, mass_gamma=0.9) == 0


def test_ring_depth_follows_the_key_rows():
    # 8 queries x 16,384 chunks of keys leave no room for a ring beside them
    assert dd.step_folds_scoring(shape(16, L=16384 * 16, n_q=8, k=16), 152) == 0
    assert 3 <= dd.step_folds_scoring(shape(16, L=8192 * 16, n_q=2, k=16), 152) <= 5


def test_invalid_dimensions_do_not_fold():
    assert dd.step_folds_scoring(dd.Shape(16, 30, 8, 128, 32768, 16, 64, 2), 152) == 0   # Hq % Hkv != 0
    assert dd.step_folds_scoring(shape(16), 0) == 0
