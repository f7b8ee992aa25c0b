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
    # attention outputs are convex combinations of N(0,1) values: below 8 in magnitude
    exact = rng.normal(size=(4, 8, 64)) * np.array([1e-4, 1e-2, 1.0, 2.0])[:, None, None]
    exact = np.clip(exact, -7.9, 7.9)
    for dt in (torch.float16, torch.bfloat16):
        rounded = torch.from_numpy(exact).to(dt)
        assert_attention_close(rounded, exact, "rounded")
        wrong = rounded.clone()
        wrong[1, 2, 3] += 0.01
        with pytest.raises(AssertionError):
            assert_attention_close(wrong, exact, "perturbed")


def test_fp16_outputs_also_meet_both_stated_bounds():
    # near 5 an fp16 ulp (2^-8) is within the ulp check but above 2e-3 absolute
    exact = np.full((1, 1, 8), 5.0)
    off = torch.from_numpy(exact + 0.0025).to(torch.float16)
    assert float(off.double()[0, 0, 0]) - 5.0 > 2e-3
    with pytest.raises(AssertionError, match="abs err"):
        assert_attention_close(off, exact, "one ulp off at 5")
    # bf16 takes the allclose gate only (its half ulp exceeds 2e-3 above 1)
    assert_attention_close(torch.from_numpy(exact).to(torch.bfloat16), exact, "bf16 at 5")
    # near zero the relative bound (floor 1e-3) is the tighter one
    small = np.full((1, 1, 8), 5e-4)
    got = torch.from_numpy(small + 1.5e-5).to(torch.float16)
    with pytest.raises(AssertionError, match="rel err"):
        assert_attention_close(got, small, "1.5e-5 off near zero")
