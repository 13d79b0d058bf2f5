"""Checks of the seeded input generators (synth): the C pool generator and the
numpy one agree bit for bit, the weights have the stated moments, the AR(1)
routing trace has its closed-form stationary statistics, and the bf16/FP4
encoders round to nearest even."""
import numpy as np
import pytest

import synth


@pytest.fixture(scope="module", autouse=True)
def _need_lib():
    try:
        synth._lib()
    except RuntimeError as e:  # built by __graft_entry__.build()
        pytest.skip(str(e))


@pytest.mark.parametrize("wd,H,I", [(0, 64, 32), (1, 256, 128), (2, 256, 128), (2, 512, 256), (1, 2048, 512)])
def test_c_generator_matches_numpy(wd, H, I):
    for key in (0, 17, 10239, 2 ** 31 + 5):
        a = synth.expert_record(4, key, H, I, wd)
        b = synth.records_array(4, key, 1, H, I, wd)[0]
        assert a.shape == b.shape and (a == b).all()


def test_c_generator_multi_key_layout():
    recs = synth.records_array(9, 100, 3, 64, 32, synth.WD_FP4)
    for i in range(3):
        assert (recs[i] == synth.expert_record(9, 100 + i, 64, 32, synth.WD_FP4)).all()


def test_weight_moments():
    v = synth.element_values(1, 3, 0, 1 << 21, 0.02).astype(np.float64)
    assert abs(v.mean()) < 1e-4
    assert abs(v.std() / 0.02 - 1) < 0.01


def test_ar1_stationary_statistics():
    # logit_t = 0.8 logit_{t-1} + 0.6 eps: stationary variance 0.36 / (1 - 0.64) = 1, lag-1 correlation 0.8
    z = synth.ar1_logits(2, 256, 4, 2, 256).astype(np.float64)
    assert abs(z.var() - 1.0) < 0.05
    a, b = z[1:].reshape(-1), z[:-1].reshape(-1)
    assert abs(np.corrcoef(a, b)[0, 1] - 0.8) < 0.02


def test_bf16_round_to_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -8 + 2 ** -20], dtype=np.float32)
    assert list(synth.to_bf16_bits(f)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81]


def test_encoders_ties_to_even():
    assert list(synth._rne_encode(np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 9.0]), synth.E2M1_ENC)) == \
        [0, 2, 2, 4, 4, 6, 6, 7]
    # e4m3: 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39) -> even code 0x38
    assert synth._rne_encode(np.float32([1.0625, 1.1875, 500.0, 0.0]), synth.E4M3_ENC).tolist() == [0x38, 0x3A, 0x7E, 0]
