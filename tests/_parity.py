"""Comparison helpers shared by the GPU parity tests (numpy only).

A bf16 parameter is rounded once to bf16 after its update, and the update is
only a few bf16 ulps of the parameter, so the stored value cannot show the
update's error directly.  What it fixes exactly: every real that rounds to
nearest to the stored bf16 value w lies in the cell [w - ulp/2, w + ulp/2]
(the lower half of the cell of a power of two is half as wide), so the GPU's
value before rounding is at least dist(oracle value, cell) from the
oracle's, element by element.  ``cell_err`` is that exact lower bound over
the norm of the oracle's update.
"""
import numpy as np


def bf16_cell_halfwidth(w_stored):
    """Half the width of the interval of reals that round to nearest to each
    stored bf16 value: half an ulp, where the ulp below a power of two (the
    lower half of the cell of an exact power of two) is half as wide."""
    w = np.abs(np.asarray(w_stored, np.float64))
    e = np.floor(np.log2(np.maximum(w, 1e-38)))
    up = np.exp2(e - 7)                                  # ulp above |w|
    down = np.where(w == np.exp2(e), np.exp2(e - 8), up)  # ulp below |w|
    return 0.5 * up, 0.5 * down


def cell_err(w_gpu, w_ref, base):
    """Exact lower bound on the relative error of the GPU's update before its
    one rounding to bf16: the distance from the oracle's value to the cell of
    values that round to the stored w_gpu, over the update's norm."""
    w_gpu = np.asarray(w_gpu, np.float64)
    w_ref = np.asarray(w_ref, np.float64)
    up, down = bf16_cell_halfwidth(w_gpu)
    # the cell extends `up` away from zero and `down` towards zero
    away = np.sign(w_gpu) * (w_ref - w_gpu)              # > 0: w_ref lies further from zero
    d = np.where(away > 0, np.maximum(away - up, 0.0), np.maximum(-away - down, 0.0))
    d = np.where(w_gpu == 0, np.maximum(np.abs(w_ref) - 2.0 ** -134, 0.0), d)
    return float(np.linalg.norm(d) / np.linalg.norm(w_ref - base))
