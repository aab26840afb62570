"""CPU checks of the comparison used by every parity test: it must reject planted errors."""
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
