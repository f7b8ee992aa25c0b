"""The attention tolerance helpers themselves (CPU)."""
import numpy as np
import pytest
import torch

from helpers import assert_attention_close, ulp


def test_ulp_matches_numpy_for_fp16():
    x = np.array([1e-7, 3e-5, 0.01, 0.3, 1.0, 1.5, 3.9, 100.0])
    ref = np.spacing(np.abs(x).astype(np.float16)).astype(np.float64)
    assert np.array_equal(ulp(x, torch.float16), ref)


def test_rounding_to_output_type_passes_and_a_real_error_fails():
    rng = np.random.default_rng(0)
    exact = rng.normal(size=(4, 8, 64)) * np.array([1e-4, 1e-2, 1.0, 4.0])[:, None, None]
    for dt in (torch.float16, torch.bfloat16):
        rounded = torch.from_numpy(exact).to(dt)
        assert_attention_close(rounded, exact, "rounded")
        wrong = rounded.clone()
        wrong[1, 2, 3] += 0.01
        with pytest.raises(AssertionError):
            assert_attention_close(wrong, exact, "perturbed")
