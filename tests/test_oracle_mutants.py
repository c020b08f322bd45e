"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
used in test_oracle_pins.py catch every one: a dropped term, a wrong sign, a
transposed operand, a wrong scale, a missing Nesterov or decay term."""
import math

import numpy as np
import pytest

import oracle
from oracle import muon_oracle as mo
from tests.test_oracle_pins import svd_closed_form, rel, QUINTIC, msign_svd, GOLD


def _ns_mutant(kind):
    def ns(X, steps=5, coeffs=QUINTIC, eps=0.0):
        a, b, c = coeffs
        X = np.asarray(X, np.float64)
        t = X.shape[0] > X.shape[1]
        if t and kind != "no_transpose":
            X = X.T
        X = X / (np.linalg.norm(X) + eps)
        for _ in range(steps):
            A = X @ X.T
            if kind == "drop_c":
                B = b * A
            elif kind == "sign_b":
                B = -b * A + c * (A @ A)
            else:
                B = b * A + c * (A @ A)
            X = a * X + (X @ B if kind == "xb_order" else B @ X)
            if kind == "no_a":
                X = X - a * X + X
        if kind == "forget_back":
            return X
        return X.T if t and kind != "no_transpose" else X
    return ns


@pytest.mark.parametrize("kind", ["drop_c", "sign_b", "no_a"])
def test_ns_mutants_fail_closed_form(kind):
    X = np.random.default_rng(1).standard_normal((16, 40))
    assert rel(_ns_mutant(kind)(X), svd_closed_form(X, 5, QUINTIC)) > 1e-3


def test_operand_order_mutant_fails_closed_form():
    X = np.random.default_rng(3).standard_normal((24, 24))
    assert rel(_ns_mutant("xb_order")(X), svd_closed_form(X, 5, QUINTIC)) > 1e-3


def test_forgetting_transpose_back_fails_shape_or_closed_form():
    X = np.random.default_rng(2).standard_normal((40, 16))
    out = _ns_mutant("forget_back")(X)
    assert out.shape != X.shape


def test_update_scale_mutants_fail_rms_pin(monkeypatch):
    shape = (64, 256)
    W = np.zeros(shape)
    G = np.random.default_rng(2).standard_normal(shape) + 4 * np.eye(*shape)
    newton = tuple(GOLD["newton_cubic"]["value"])
    for bad in (lambda s, r=0.2, *_: r * math.sqrt(min(s[0], s[1])),
                lambda s, r=0.2, *_: math.sqrt(max(s[0], s[1])),
                lambda s, r=0.2, *_: r * max(s[0], s[1])):
        monkeypatch.setattr(mo, "update_scale", bad)
        Wn, _ = mo.muon_step(W, G, np.zeros(shape), lr=0.02, wd=0.0, steps=80, coeffs=newton)
        rms = math.sqrt(np.mean((Wn - W) ** 2)) / 0.02
        assert abs(rms - 0.2) > 1e-3


def test_mup_scale_mutants_fail_rms_to_rms_pin(monkeypatch):
    # inverted ratio, RMS-mode factor, or no square root: the update's
    # RMS -> RMS operator norm is no longer 1 on a non-square parameter
    newton = tuple(GOLD["newton_cubic"]["value"])
    real = mo.update_scale
    for bad_base in (lambda A, B: math.sqrt(B / A), lambda A, B: 0.2 * math.sqrt(max(A, B)), lambda A, B: A / B):
        def bad(shape, update_rms=0.2, mode="rms", extra=1.0, f=bad_base):
            if mode == "mup":
                return extra * f(int(shape[0]), int(shape[1]))
            return real(shape, update_rms, mode, extra)
        monkeypatch.setattr(mo, "update_scale", bad)
        for shape in ((24, 96), (96, 24)):
            G = np.random.default_rng(4).standard_normal(shape)
            Wn, _ = mo.muon_step(np.zeros(shape), G, np.zeros(shape), lr=0.02, wd=0.0, steps=80, coeffs=newton,
                                 scale_mode="mup")
            D = (Wn / -0.02)
            norm = math.sqrt(shape[1] / shape[0]) * np.linalg.svd(D, compute_uv=False)[0]
            if abs(norm - 1.0) > 1e-3:
                break
        else:
            raise AssertionError("mutant passed the RMS->RMS pin")
    monkeypatch.undo()


def test_nesterov_and_decay_mutants_fail_pins(monkeypatch):
    G = np.random.default_rng(31).standard_normal((5, 7))
    mu = 0.95

    def no_nesterov(M, G, mu, nesterov):
        M_new = mu * M + G
        return M_new, M_new
    monkeypatch.setattr(mo, "momentum_update", no_nesterov)
    M = np.zeros_like(G)
    M, U = mo.momentum_update(M, G, mu, True)
    M, U = mo.momentum_update(M, G, mu, True)
    assert rel(U, G * (1 - mu ** 3) / (1 - mu)) > 1e-3
    monkeypatch.undo()

    def no_decay(W, O, lr, wd, shape, update_rms=0.2, *_):
        return np.asarray(W, np.float64) - lr * mo.update_scale(shape, update_rms) * O
    monkeypatch.setattr(mo, "apply_update", no_decay)
    W = np.random.default_rng(3).standard_normal((8, 12))
    Wn, _ = mo.muon_step(W, np.zeros((8, 12)), np.zeros((8, 12)), lr=0.02, wd=0.1)
    assert not np.array_equal(Wn, W * (1 - 0.02 * 0.1))


def test_adamw_mutant_without_bias_correction_fails_closed_form():
    g = np.array([1e-3, -2.0, 0.3])
    b1, b2, eps, lr = 0.9, 0.95, 1e-8, 1e-3
    p, m, v = np.zeros(3), np.zeros(3), np.zeros(3)
    m = m + (1 - b1) * (g - m)
    v = v + (1 - b2) * (g * g - v)
    p_bad = p - lr * m / (eps + np.sqrt(v))          # bias correction dropped
    bc2 = 1 - b2
    expect = -lr * g * math.sqrt(bc2) / (eps + math.sqrt(bc2) * np.abs(g))
    assert rel(p_bad, expect) > 1e-2
    p_ok, _, _ = oracle.adamw_step(np.zeros(3), g, np.zeros(3), np.zeros(3), 1,
                                   lr=lr, beta1=b1, beta2=b2, eps=eps, wd=0.0)
    assert rel(p_ok, expect) < 1e-12


def test_gram_mutant_q_order_still_commutes_but_missing_p_fails():
    # R <- P R (one-sided) instead of P R P breaks gram == standard
    X = np.random.default_rng(4).standard_normal((12, 30))
    a, b, c = QUINTIC
    X0 = X / np.linalg.norm(X)
    R, Q, I = X0 @ X0.T, np.eye(12), np.eye(12)
    for _ in range(5):
        P = a * I + b * R + c * R @ R
        Q = P @ Q
        R = P @ R
    assert rel(Q @ X0, svd_closed_form(X, 5, QUINTIC)) > 1e-3


def test_schedule_mutant_using_the_first_triple_fails_the_closed_form(monkeypatch):
    # an oracle that ignored the schedule (every step with the first triple)
    newton = tuple(GOLD["newton_cubic"]["value"])
    sched = [mo.QUINTIC] * 8 + [newton] * 2
    X = np.random.default_rng(13).standard_normal((16, 40))
    monkeypatch.setattr(mo, "step_coeffs", lambda coeffs, steps: [tuple(coeffs[0])] * steps)
    bad = mo.newton_schulz(X, steps=10, coeffs=sched)
    monkeypatch.undo()
    U, s, Vt = np.linalg.svd(X, full_matrices=False)
    x = s / np.linalg.norm(X)
    for a, b, c in sched:
        x = a * x + b * x ** 3 + c * x ** 5
    assert rel(bad, (U * x) @ Vt) > 1e-3
