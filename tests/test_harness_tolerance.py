"""The output tolerance helper: bf16 rounding of the reference itself passes,
a real error of 3% of RMS on one element does not."""
import numpy as np
import pytest
import torch

from tests._harness import assert_delta_close, bf16_half_ulp


def _bf16(a):
    return torch.from_numpy(a).to(torch.bfloat16).double().numpy()


def test_half_ulp_matches_bf16_rounding():
    rng = np.random.default_rng(0)
    v = rng.standard_normal(100000) * 10.0 ** rng.uniform(-3, 2, 100000)
    assert np.all(np.abs(_bf16(v) - v) <= bf16_half_ulp(v) * (1 + 1e-12))
    assert bf16_half_ulp(np.array([8.0, 9.5, 15.9]))[0] == 2.0 ** -5


def test_rounded_reference_passes_real_error_fails():
    rng = np.random.default_rng(1)
    ref = rng.standard_normal((64, 256))
    ref[3, 7] = 11.0                                  # an outlier whose bf16 spacing is 0.0625
    assert_delta_close(_bf16(ref), ref)
    bad = _bf16(ref)
    bad[5, 9] += 0.03 * np.sqrt((ref ** 2).mean()) + 0.01
    with pytest.raises(AssertionError):
        assert_delta_close(bad, ref)
