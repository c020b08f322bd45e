"""The comparison helpers of the GPU parity tests, checked on the CPU.

cell_err must be an exact lower bound on the error of a value before its
one rounding to bf16: zero when the stored value is the correctly rounded
oracle value, never above the true pre-rounding error, and close to it once
the error spans several ulps.  torch's float -> bf16 conversion (round to
nearest even) does the rounding.
"""
import numpy as np
import pytest
import torch

from _parity import bf16_cell_halfwidth, cell_err


def _bf16(x):
    return torch.tensor(np.asarray(x, np.float64), dtype=torch.float64).to(torch.bfloat16).double().numpy()


def _case(seed, rel_err):
    rng = np.random.default_rng(seed)
    w = 0.02 * rng.standard_normal((96, 80))
    d = 5e-4 * rng.standard_normal((96, 80))
    ref = w + d
    v = ref + rel_err * np.linalg.norm(d) / np.sqrt(d.size) * rng.standard_normal(d.shape)
    return w, ref, v


def test_correct_rounding_has_zero_cell_error():
    w, ref, _ = _case(0, 0.0)
    assert cell_err(_bf16(ref), ref, w) == 0.0


@pytest.mark.parametrize("rel_err", [1e-3, 1e-2, 1e-1, 1.0, 3.0])
def test_cell_error_is_a_lower_bound_that_tightens(rel_err):
    w, ref, v = _case(1, rel_err)
    true = np.linalg.norm(v - ref) / np.linalg.norm(ref - w)
    bound = cell_err(_bf16(v), ref, w)
    assert bound <= true * (1 + 1e-12)
    if rel_err >= 1.0:            # errors of many ulps: the bound is nearly the error
        assert bound > 0.8 * true


def test_cells_of_powers_of_two_are_asymmetric():
    up, down = bf16_cell_halfwidth(np.array([1.0, -0.25, 1.5]))
    assert up.tolist() == [2.0 ** -8, 2.0 ** -10, 2.0 ** -8]
    assert down.tolist() == [2.0 ** -9, 2.0 ** -11, 2.0 ** -8]
    # every value inside the cell rounds to the stored value, and just outside does not
    for w, u, dn in zip([1.0, -0.25, 1.5], up, down):
        s = np.sign(w)
        assert _bf16(w + s * 0.99 * u) == w and _bf16(w - s * 0.99 * dn) == w
        assert _bf16(w + s * 1.01 * u) != w and _bf16(w - s * 1.01 * dn) != w
