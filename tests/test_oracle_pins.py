"""Pins for the fp64 oracle: closed forms, library routines and invariants that
fix what the method computes independently of the oracle's own code.

Each test names the fact it checks and where the pages state it; the numbers
the pages print are read from tests/golden/page_constants.json.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from newton_schulz_orthogonalized_muon_gb300 import workloads as wl

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))
QUINTIC = tuple(GOLD["quintic_coefficients"]["value"])


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(b), 1e-300))


def svd_closed_form(X, steps, coeffs):
    """U diag(g^steps(sigma_i/||X||_F)) V^T with g(x) = ax + bx^3 + cx^5, from
    the LAPACK SVD: the quintic only moves singular values
    (Muon Optimizer and the Distributed Implementation, §Newton-Schulz
    Iteration)."""
    a, b, c = coeffs
    X = np.asarray(X, np.float64)
    U, s, Vt = np.linalg.svd(X, full_matrices=False)
    x = s / np.linalg.norm(X)
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return (U * x) @ Vt


def msign_svd(G):
    U, _, Vt = np.linalg.svd(np.asarray(G, np.float64), full_matrices=False)
    return U @ Vt


def rand(seed, shape):
    return np.random.default_rng(seed).standard_normal(shape)


SHAPES = [(8, 8), (16, 40), (40, 16), (1, 7), (7, 1), (33, 65), (65, 33)]


def test_quintic_scalar_facts():
    a, b, c = QUINTIC
    g = lambda x: a * x + b * x ** 3 + c * x ** 5
    h = 1e-7
    assert abs((g(h) - g(-h)) / (2 * h) - 3.4445) < 1e-6      # g'(0) = a
    assert abs(g(1.0) - 0.701) < 1e-12                        # a + b + c
    assert QUINTIC == (3.4445, -4.7750, 2.0315)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("method", ["standard", "gram"])
def test_ns_matches_svd_closed_form(shape, method):
    X = rand(sum(shape), shape)
    got = oracle.orthogonalize(X, 5, QUINTIC, method, eps=0.0)
    assert rel(got, svd_closed_form(X, 5, QUINTIC)) < 1e-11


def test_ns_closed_form_on_lowrank_grad():
    G = wl.lowrank_grad(0, 256, 512, 256)
    got = oracle.newton_schulz(G, 5, QUINTIC, eps=0.0)
    assert rel(got, svd_closed_form(G, 5, QUINTIC)) < 1e-11


@pytest.mark.parametrize("steps", [0, 1, 2, 7])
def test_ns_step_count(steps):
    X = rand(3, (12, 20))
    assert rel(oracle.newton_schulz(X, steps, QUINTIC, eps=0.0), svd_closed_form(X, steps, QUINTIC)) < 1e-11


@pytest.mark.parametrize("shape", [(6, 6), (5, 9), (9, 5)])
def test_newton_cubic_converges_to_msign(shape):
    # Sign of a Matrix: Newton on x^-2 - 1 gives 1.5x - 0.5x^3 -> msign(G) = UV^T
    coeffs = tuple(GOLD["newton_cubic"]["value"])
    G = rand(11, shape) + 3 * np.eye(*shape)       # well conditioned
    got = oracle.newton_schulz(G, 80, coeffs, eps=0.0)
    assert rel(got, msign_svd(G)) < 1e-10


def test_taylor_coefficients_corrected_vs_printed():
    G = rand(5, (6, 10)) + 2 * np.eye(6, 10)
    fixed = tuple(GOLD["taylor_quadratic_corrected"]["value"])
    assert rel(oracle.newton_schulz(G, 60, fixed, eps=0.0), msign_svd(G)) < 1e-10
    # the printed -7/8 makes f(1) = 1.375: the fixed point is not 1
    a, b, c = GOLD["taylor_quadratic_as_printed"]["value"]
    assert abs(a + b + c - 1.375) < 1e-12
    a, b, c = fixed
    assert abs(a + b + c - 1.0) < 1e-12


@pytest.mark.parametrize("shape", [(3, 5), (4, 4), (5, 3)])
def test_msign_two_forms(shape):
    # Sign of a Matrix: msign(G) = UV^T = (GG^T)^(-1/2) G = G (G^T G)^(-1/2)
    G = rand(7, shape)
    if shape[0] <= shape[1]:
        w, Q = np.linalg.eigh(G @ G.T)
        polar = (Q / np.sqrt(w)) @ Q.T @ G
    else:
        w, Q = np.linalg.eigh(G.T @ G)
        polar = G @ ((Q / np.sqrt(w)) @ Q.T)
    assert rel(msign_svd(G), polar) < 1e-12
    # and the semi-orthogonal corollary: ||O||_F^2 = min(m, n)
    assert abs(np.sum(msign_svd(G) ** 2) - min(shape)) < 1e-12


@pytest.mark.parametrize("shape", [(16, 48), (48, 16), (64, 64), (1, 9)])
def test_gram_equals_standard(shape):
    X = wl.lowrank_grad(1, shape[0], shape[1], 8)
    assert rel(oracle.gram_newton_schulz(X), oracle.newton_schulz(X)) < 1e-10


def test_invariants():
    X = rand(21, (24, 40))
    O = oracle.newton_schulz(X, eps=0.0)
    assert rel(oracle.newton_schulz(X.T, eps=0.0), O.T) < 1e-12
    assert rel(oracle.newton_schulz(7.5 * X, eps=0.0), O) < 1e-12
    P, _ = np.linalg.qr(rand(22, (24, 24)))
    Q, _ = np.linalg.qr(rand(23, (40, 40)))
    assert rel(oracle.newton_schulz(P @ X @ Q, eps=0.0), P @ O @ Q) < 1e-11


def test_singular_value_band_and_frobenius():
    # output singular values = g^5 of the normalised inputs; for every input
    # singular value >= 3e-3 of the norm they sit in about 0.7-1.3 (the band
    # the Newton-Schulz section accepts), measured bounds [0.68, 1.21].
    G = wl.lowrank_grad(0, 256, 512, 256)
    O = oracle.newton_schulz(G)
    s = np.linalg.svd(O, compute_uv=False)
    lo, hi = GOLD["acceptable_singular_value_band"]["value"]
    assert s.min() > lo - 0.02 and s.max() < hi - 0.09
    assert 0.46 * 256 < np.sum(O ** 2) < 1.46 * 256


def test_zero_matrix_gives_zero():
    assert np.all(oracle.newton_schulz(np.zeros((4, 6))) == 0)
    assert np.all(oracle.gram_newton_schulz(np.zeros((4, 6))) == 0)


def test_momentum_closed_form_constant_grad():
    G = rand(31, (5, 7))
    mu = 0.95
    M = np.zeros_like(G)
    for k in range(1, 9):
        M, U = oracle.momentum_update(M, G, mu, nesterov=True)
        geo = lambda j: (1 - mu ** j) / (1 - mu)
        assert rel(M, G * geo(k)) < 1e-14
        assert rel(U, G * geo(k + 1)) < 1e-14      # Nesterov look-ahead = next M
        _, U_plain = oracle.momentum_update(M / mu - G / mu, G, mu, nesterov=False)
        assert rel(U_plain, M) < 1e-12


def test_momentum_unrolled_sum():
    mu = 0.9
    Gs = [rand(40 + k, (3, 4)) for k in range(6)]
    M = np.zeros((3, 4))
    for k, G in enumerate(Gs):
        M, _ = oracle.momentum_update(M, G, mu, nesterov=False)
        expect = sum(mu ** (k - j) * Gs[j] for j in range(k + 1))
        assert rel(M, expect) < 1e-13


@pytest.mark.parametrize("shape", [(64, 256), (256, 64), (100, 100)])
def test_update_rms_is_0p2_for_exact_msign(shape):
    # Moonlight §2: 0.2*sqrt(max(A,B)) makes the update RMS 0.2 for an
    # orthogonal O; run the Newton cubic to convergence to get O = msign.
    W = wl.weight(1, shape).astype(np.float64)
    G = rand(2, shape) + 4 * np.eye(*shape)
    M = np.zeros(shape)
    lr = 0.02
    Wn, _ = oracle.muon_step(W, G, M, lr=lr, wd=0.0, steps=80,
                             coeffs=tuple(GOLD["newton_cubic"]["value"]))
    rms = math.sqrt(np.mean((Wn - W) ** 2)) / lr
    assert abs(rms - GOLD["update_rms"]["value"]) < 1e-10
    assert np.sum((Wn - W) * msign_svd(G)) < 0     # a descent step along -msign


@pytest.mark.parametrize("shape", [(48, 192), (192, 48), (80, 80)])
def test_mup_update_has_unit_rms_to_rms_norm(shape):
    # Chensy §Variation of Muon Optimizer: the dual of G under the RMS->RMS
    # operator norm, ||A||_{RMS->RMS} = sqrt(d_in / d_out) ||A||_2, is the
    # update of RMS->RMS norm 1, sqrt(d_out / d_in) msign(G).  With the weight
    # stored (d_out, d_in) and O = msign (Newton cubic run to convergence),
    # the muP step's direction must have that norm exactly, and be a descent
    # direction along -msign(G).
    d_out, d_in = shape
    W = wl.weight(6, shape).astype(np.float64)
    G = rand(7, shape)
    lr = 0.02
    Wn, _ = oracle.muon_step(W, G, np.zeros(shape), lr=lr, wd=0.0, steps=80,
                             coeffs=tuple(GOLD["newton_cubic"]["value"]), scale_mode="mup")
    D = (W - Wn) / lr
    sig = np.linalg.svd(D, compute_uv=False)
    assert abs(math.sqrt(d_in / d_out) * sig[0] - 1.0) < 1e-10
    assert abs(sig[-1] - sig[0]) < 1e-10 * sig[0]          # every direction equally scaled
    assert np.sum(D * msign_svd(G)) > 0


@pytest.mark.parametrize("gamma", [0.18, 0.25])
def test_deepseek_gamma_sets_the_update_rms(gamma):
    # Chensy §Variation (DeepSeek-V4): O' sqrt(max(n, m)) gamma makes the
    # update RMS gamma for an orthogonal O'; here gamma is update_rms, and
    # the extra scale factor multiplies the step on top of it.
    shape = (64, 160)
    W = wl.weight(8, shape).astype(np.float64)
    G = rand(9, shape)
    lr = 0.02
    for extra in (1.0, 1.5):
        Wn, _ = oracle.muon_step(W, G, np.zeros(shape), lr=lr, wd=0.0, steps=80,
                                 coeffs=tuple(GOLD["newton_cubic"]["value"]), update_rms=gamma,
                                 extra_scale=extra)
        rms = math.sqrt(np.mean((Wn - W) ** 2)) / lr
        assert abs(rms - gamma * extra) < 1e-10


def test_weight_decay_only_when_grad_zero():
    W = wl.weight(3, (8, 12)).astype(np.float64)
    Wn, Mn = oracle.muon_step(W, np.zeros((8, 12)), np.zeros((8, 12)), lr=0.02, wd=0.1)
    assert np.array_equal(Wn, W * (1 - 0.02 * 0.1))
    assert np.all(Mn == 0)


def test_split_heads_row_blocks():
    # row blocks with mutually orthogonal row spaces: msign of the whole equals
    # the stack of per-block msigns, so split == unsplit for the converged
    # iteration; a column split would not match the per-block closed form.
    rng = np.random.default_rng(5)
    Vfull, _ = np.linalg.qr(rng.standard_normal((32, 32)))
    blocks = [rng.standard_normal((4, 4)) + 3 * np.eye(4) for _ in range(4)]
    U = np.concatenate([blocks[i] @ Vfull[:, 8 * i:8 * i + 4].T for i in range(4)], axis=0)
    newton = tuple(GOLD["newton_cubic"]["value"])
    split = oracle.orthogonalize_split(U, 4, 80, newton)
    assert rel(split, msign_svd(U)) < 1e-10
    # quintic, 5 steps: every block follows its own closed form
    split5 = oracle.orthogonalize_split(U, 4)
    for i in range(4):
        blk = U[4 * i:4 * i + 4]
        assert rel(split5[4 * i:4 * i + 4], svd_closed_form(blk, 5, QUINTIC)) < 1e-6
    with pytest.raises(ValueError):
        oracle.orthogonalize_split(U, 3)


def test_adamw_matches_torch_when_eps_zero():
    torch = pytest.importorskip("torch")
    # With eps = 0 the printed AdamW backup (eps on the raw v, bias correction
    # folded into the step size) equals torch.optim.AdamW exactly.
    rng = np.random.default_rng(9)
    p0 = rng.standard_normal(50)
    tp = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([tp], lr=3e-3, betas=(0.9, 0.95), eps=0.0, weight_decay=0.1)
    p, m, v = p0.copy(), np.zeros(50), np.zeros(50)
    for t in range(1, 6):
        g = rng.standard_normal(50)
        tp.grad = torch.tensor(g)
        opt.step()
        p, m, v = oracle.adamw_step(p, g, m, v, t, lr=3e-3, beta1=0.9, beta2=0.95, eps=0.0, wd=0.1)
        assert rel(p, tp.detach().numpy()) < 1e-13


def test_adamw_constant_grad_closed_form():
    # constant g: m_t = (1-b1^t) g, v_t = (1-b2^t) g^2, so the step is
    # -lr * g*sqrt(bc2) / (eps + sqrt(bc2)|g|) for every t.
    g = np.array([1e-3, -2.0, 5e-9, 0.3])
    b1, b2, eps, lr = 0.9, 0.95, 1e-8, 1e-3
    p, m, v = np.zeros(4), np.zeros(4), np.zeros(4)
    for t in range(1, 7):
        p_prev = p
        p, m, v = oracle.adamw_step(p, g, m, v, t, lr=lr, beta1=b1, beta2=b2, eps=eps, wd=0.0)
        bc2 = 1 - b2 ** t
        expect = -lr * g * math.sqrt(bc2) / (eps + math.sqrt(bc2) * np.abs(g))
        assert rel(p - p_prev, expect) < 1e-12


def test_full_step_against_torch_muon():
    torch = pytest.importorskip("torch")
    if not hasattr(torch.optim, "Muon"):
        pytest.skip("torch.optim.Muon not available")
    # torch.optim.Muon keeps an EMA buffer ((1-mu) times the pages' buffer,
    # same direction after normalisation) and runs NS in bf16; with
    # adjust_lr_fn="match_rms_adamw" it is the Moonlight step.  Agreement to
    # bf16 accuracy pins momentum, Nesterov, transpose, scale and decay.  A
    # dropped Nesterov term alone moves the update by ~30% on these inputs.
    for shape in [(48, 96), (96, 48)]:
        W0 = wl.weight(7, shape).astype(np.float64)
        tp = torch.nn.Parameter(torch.tensor(W0, dtype=torch.float32))
        opt = torch.optim.Muon([tp], lr=0.02, weight_decay=0.1, momentum=0.95, nesterov=True,
                               adjust_lr_fn="match_rms_adamw")
        W, M = W0.copy(), np.zeros(shape)
        for k in range(3):
            G = rand(100 + k, shape)       # well conditioned: bf16 NS is accurate here
            tp.grad = torch.tensor(G, dtype=torch.float32)
            opt.step()
            W_prev = W
            G = G.astype(np.float32).astype(np.float64)
            W, M = oracle.muon_step(W, G, M, lr=0.02, wd=0.1, mu=0.95, nesterov=True)
            d_ref = W - W_prev * (1 - 0.02 * 0.1)
            d_t = tp.detach().double().numpy() - W_prev * (1 - 0.02 * 0.1)
            assert rel(d_t, d_ref) < 3e-2


def test_classification():
    assert oracle.is_muon_param("layers.0.attn.q_proj.weight", 2)
    assert not oracle.is_muon_param("model.embed_tokens.weight", 2)
    assert not oracle.is_muon_param("lm_head.weight", 2)
    assert not oracle.is_muon_param("layers.0.ln.weight", 1)
    assert not oracle.is_muon_param("conv.weight", 4)


def test_flattened_grad_and_shape_scale():
    # a >2-D grad is viewed as (size0, -1); the scale uses the first two dims
    W = wl.weight(2, (6, 4, 5)).astype(np.float64)
    G = rand(3, (6, 4, 5))
    Wn, Mn = oracle.muon_step(W, G, np.zeros_like(G), lr=0.01, wd=0.0)
    O = oracle.newton_schulz(1.95 * G.reshape(6, 20))    # Nesterov, zero buffer: U = (1+mu) G
    assert rel((W - Wn).reshape(6, 20), 0.01 * 0.2 * math.sqrt(6) * O) < 1e-13


# ------------------------------------------------ per-step coefficient schedules

def svd_closed_form_schedule(X, schedule):
    """As svd_closed_form, with step k moving each normalised singular value by
    its own odd quintic g_k(x) = a_k x + b_k x^3 + c_k x^5 (applied in order)."""
    X = np.asarray(X, np.float64)
    U, s, Vt = np.linalg.svd(X, full_matrices=False)
    x = s / np.linalg.norm(X)
    for a, b, c in schedule:
        x = a * x + b * x ** 3 + c * x ** 5
    return (U * x) @ Vt


HYBRID = [QUINTIC] * 8 + [tuple(GOLD["newton_cubic"]["value"])] * 2


@pytest.mark.parametrize("shape", [(16, 40), (40, 16), (24, 24)])
@pytest.mark.parametrize("method", ["standard", "gram"])
def test_hybrid_schedule_matches_composed_closed_form(shape, method):
    # Chensy §Variation of Muon Optimizer (DeepSeek-V4): 8 steps with the
    # quintic's magic numbers, then steps with other coefficients; here the
    # last two are the Newton cubic of §Sign of a Matrix.  The singular
    # values follow the composition of the per-step scalar maps.
    X = rand(11, shape)
    got = oracle.orthogonalize(X, steps=10, coeffs=HYBRID, method=method, eps=0.0)
    assert rel(got, svd_closed_form_schedule(X, HYBRID)) < 1e-11
    # the polynomials do not commute: reversing the schedule changes the result
    assert rel(got, svd_closed_form_schedule(X, HYBRID[::-1])) > 1e-3


def test_hybrid_newton_tail_tightens_the_singular_values():
    # the Newton tail pulls every singular value of the quintic's output
    # toward 1 (g_N(x) = 1.5x - 0.5x^3 has g_N(1) = 1 and g_N'(1) = 0)
    X = rand(12, (32, 96))
    plain = np.linalg.svd(oracle.newton_schulz(X, steps=8), compute_uv=False)
    hybrid = np.linalg.svd(oracle.newton_schulz(X, steps=10, coeffs=HYBRID), compute_uv=False)
    assert np.max(np.abs(hybrid - 1)) < 0.5 * np.max(np.abs(plain - 1))
