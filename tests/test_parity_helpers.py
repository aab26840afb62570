"""CPU checks of the comparison used by every parity test: it must reject planted errors."""
import math

import numpy as np
import pytest
import torch

import _parity


def _bf16(x):
    return torch.from_numpy(x).to(torch.bfloat16)


def test_faithful_rounding_accepts_both_neighbours_and_rejects_two_ulps():
    rng = np.random.default_rng(1)
    ref = rng.standard_normal((4, 3, 128)) * 0.05
    _parity.compare(_bf16(ref), ref, "bf16")                     # round to nearest
    down = np.nextafter(ref.astype(np.float32), -np.inf).astype(np.float64)
    _parity.compare(torch.from_numpy(down).to(torch.bfloat16), ref, "bf16")
    ulp = _parity.ulp(ref, "bf16")
    bad = ref.copy()
    bad[1, 2, 7] += 2.5 * ulp[1, 2, 7]
    with pytest.raises(AssertionError, match="faithful"):
        _parity.compare(_bf16(bad), ref, "bf16")


def test_fp32_bar_rejects_relative_error_above_1e_3():
    rng = np.random.default_rng(2)
    ref = rng.standard_normal((2, 4, 64)) * 0.02
    _parity.compare(torch.from_numpy(ref * (1 + 5e-4)).float(), ref, "f32")
    with pytest.raises(AssertionError, match="rel-L2"):
        _parity.compare(torch.from_numpy(ref * (1 + 2e-3)).float(), ref, "f32")
    worse = ref.copy()
    worse[0, 0, 0] += 3e-3
    with pytest.raises(AssertionError):
        _parity.compare(torch.from_numpy(worse).float(), ref, "f32")


def test_f16_ulp_matches_numpy_spacing():
    x = np.array([1.0, 0.75, 3.0, 1e-3, 60000.0])
    want = np.spacing(x.astype(np.float16)).astype(np.float64)
    assert np.array_equal(_parity.ulp(x, "f16"), want)


def _rz_bf16(x):
    """x rounded toward zero to bf16 (a truncating cast), as a bf16 tensor."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return torch.from_numpy(b.view(np.float32).astype(np.float32)).to(torch.bfloat16)


def test_round_nearest_even_matches_numpy_half_and_ties_to_even():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(4096) * 0.03
    r, _ = _parity.round_nearest_even(x, "f16")
    assert np.array_equal(r, x.astype(np.float16).astype(np.float64))
    # bf16 ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 and rounds to the even 1.0;
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6 and rounds up to the even one
    r, mid = _parity.round_nearest_even(np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]), "bf16")
    assert r.tolist() == [1.0, 1 + 2.0 ** -6] and mid.tolist() == [0.0, 0.0]


def test_truncating_cast_fails_the_rounding_mode_check():
    rng = np.random.default_rng(4)
    ref = rng.standard_normal((4, 3, 128)) * 0.05
    rne, _ = _parity.round_nearest_even(ref, "bf16")
    _parity.compare(torch.from_numpy(rne).to(torch.bfloat16), ref, "bf16")   # exact RNE passes
    got = _rz_bf16(ref)
    assert (got.double().numpy() != rne).any()
    with pytest.raises(AssertionError, match="nearest even"):
        _parity.compare(got, ref, "bf16")


def test_rounding_mode_check_allows_either_side_near_a_midpoint():
    # values within the FP32 error band of a midpoint may round either way; the rest must not
    rng = np.random.default_rng(5)
    ref = rng.standard_normal((1, 1, 128)) * 0.05
    sp = 2.0 ** -7 * 2.0 ** -4            # bf16 spacing in [2^-4, 2^-3)
    mid = 2.0 ** -4 + 37.5 * sp           # exactly a midpoint
    ref[0, 0, :4] = mid + np.array([-1e-9, 0.0, 1e-9, 2e-9])
    rne, _ = _parity.round_nearest_even(ref, "bf16")
    for side in (37, 38):
        got = rne.copy()
        got[0, 0, :4] = 2.0 ** -4 + side * sp
        _parity.compare(torch.from_numpy(got).to(torch.bfloat16), ref, "bf16")
    got = rne.copy()
    got[0, 0, 10] = rne[0, 0, 10] + _parity.ulp(rne[0, 0, 10], "bf16")   # far from a midpoint
    with pytest.raises(AssertionError, match="nearest even"):
        _parity.compare(torch.from_numpy(got).to(torch.bfloat16), ref, "bf16")


def test_lse_bound_rejects_a_lost_split():
    # 128 equal splits of a 32K row: losing one changes the LSE by ln(1 - 1/128)
    lse = np.full((1, 32), math.log(32768.0) + 0.5)
    _parity.compare_lse(torch.from_numpy(lse + 1e-6).float(), lse)
    lost = lse + math.log(1 - 1 / 128)
    with pytest.raises(AssertionError, match="lse error"):
        _parity.compare_lse(torch.from_numpy(lost).float(), lse)
    # one 16-token piece of a 131072-token row
    lost = lse + math.log(1 - 16 / 131072)
    with pytest.raises(AssertionError, match="lse error"):
        _parity.compare_lse(torch.from_numpy(lost).float(), lse)
