"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.

Tolerances (relative Frobenius error): fp32 path 1e-4, bf16 path 2e-2,
momentum and the update arithmetic 1e-6.  bf16 inputs are compared against
the oracle run on the same bf16 values widened exactly to fp64.

The update is compared as dW = W_new - W_old*(1 - lr*wd), each step on its
own: the oracle takes the step from the parameter the GPU holds before it.
A bf16 parameter is rounded once to bf16 after the update, and dW is a few
bf16 ulps of W, so the stored value cannot show the update's error directly.
What it does fix exactly: every value that rounds (to nearest) to the stored
bf16 w lies in the cell [w - ulp/2, w + ulp/2], so the GPU's update before
rounding is at least dist(oracle value, cell) away from the oracle's, per
element.  bf16 parameters are held to that lower bound (``cell_err``); the
same NS path with fp32 parameters (``ns_dtype`` bf16, fp32 destination)
shows dW itself and is held to the bar directly.  Every achieved error is
recorded and printed at the end of the run (tests/_margins.py).
"""
import numpy as np
import pytest
import torch

import oracle
from _margins import record
from _parity import cell_err
from newton_schulz_orthogonalized_muon_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_F32, TOL_BF16, TOL_EXACT = 1e-4, 2e-2, 1e-6


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as p
    p.load_library()
    torch.cuda.set_device(0)
    return p


def to_dev(x, dtype):
    return torch.tensor(np.asarray(x, np.float32)).to(dtype).cuda()


def host64(t):
    return t.detach().double().cpu().numpy()


def bf16_budget(w_new):
    """Frobenius norm of the worst-case bf16 rounding of w_new (half ulp)."""
    w = np.abs(np.asarray(w_new, np.float64))
    ulp = np.exp2(np.floor(np.log2(np.maximum(w, 1e-30))) - 7)
    return float(np.linalg.norm(0.5 * ulp))


def f32_budget(w_new):
    """Frobenius norm of one fp32 rounding of w_new (half ulp); the decay
    factor 1 - lr*wd held in fp32 adds at most one more."""
    w = np.abs(np.asarray(w_new, np.float64))
    ulp = np.exp2(np.floor(np.log2(np.maximum(w, 1e-30))) - 23)
    return float(np.linalg.norm(0.5 * ulp))


# ------------------------------------------------------------ self-test

def test_bounded_wait_times_out_and_context_survives(pkg):
    h = pkg.default_handle()
    assert h.check() == 0
    st = pkg.selftest_timeout(2_000_000)
    assert st == 6                       # MUON_ERR_TIMEOUT
    assert h.check() == 0                # word cleared, context usable
    x = torch.ones(4, 4, device="cuda")
    assert float(x.sum()) == 16.0


# ------------------------------------------------------- orthogonalize

ORTHO_SHAPES = [(256, 512), (100, 300), (300, 100), (1, 50), (50, 1), (64, 64), (129, 257)]


@pytest.mark.parametrize("shape", ORTHO_SHAPES)
def test_orthogonalize_fp32(pkg, shape):
    X = wl.lowrank_grad(7, shape[0], shape[1], 32)
    t = to_dev(X, torch.float32)
    pkg.muon_orthogonalize(t)
    ref = oracle.newton_schulz(X.astype(np.float64))
    assert record(f"orthogonalize fp32 {shape}", rel(host64(t), ref), TOL_F32) < TOL_F32


BF16_SHAPES = [(128, 512), (256, 1024), (200, 700), (700, 200), (1, 300), (300, 1), (384, 1536), (768, 768),
               (130, 4100)]


@pytest.mark.parametrize("shape", BF16_SHAPES)
def test_orthogonalize_bf16(pkg, shape):
    X = wl.lowrank_grad(8, shape[0], shape[1], 64)
    t = to_dev(X, torch.bfloat16)
    ref = oracle.newton_schulz(host64(t))
    pkg.muon_orthogonalize(t)
    assert record(f"orthogonalize bf16 {shape}", rel(host64(t), ref), TOL_BF16) < TOL_BF16


def test_orthogonalize_batched_bf16(pkg):
    B, m, n = 5, 192, 320
    X = np.stack([wl.lowrank_grad(50 + i, m, n, 32) for i in range(B)])
    t = to_dev(X, torch.bfloat16)
    inp = host64(t)
    pkg.muon_orthogonalize(t)
    out = host64(t)
    for i in range(B):
        assert rel(out[i], oracle.newton_schulz(inp[i])) < TOL_BF16


@pytest.mark.parametrize("steps", [0, 1, 2])
def test_orthogonalize_step_counts(pkg, steps):
    X = wl.lowrank_grad(9, 96, 200, 16)
    t32 = to_dev(X, torch.float32)
    pkg.muon_orthogonalize(t32, steps=steps)
    assert rel(host64(t32), oracle.newton_schulz(X.astype(np.float64), steps)) < TOL_F32
    tb = to_dev(X, torch.bfloat16)
    ref = oracle.newton_schulz(host64(tb), steps)
    pkg.muon_orthogonalize(tb, steps=steps)
    assert rel(host64(tb), ref) < TOL_BF16


def test_orthogonalize_zero_and_empty(pkg):
    z = torch.zeros(64, 128, device="cuda", dtype=torch.bfloat16)
    pkg.muon_orthogonalize(z)
    assert torch.count_nonzero(z).item() == 0
    e = torch.zeros(0, 64, 128, device="cuda", dtype=torch.bfloat16)
    pkg.muon_orthogonalize(e)


# ----------------------------------------------------------- muon_step

def run_step_per_step(pkg, specs, dtype, steps=1, ns_steps=5, lr=0.02, wd=0.1, mu=0.95, nesterov=True, seed=0,
                      grad_dtype=None, ns_dtype=None, **scale):
    """Run `steps` Muon steps on the GPU; the oracle takes each step from the
    parameter the GPU held before it (its momentum chain is its own).
    Returns, per step, per param, (W_gpu, W_ref, W_prev * (1 - lr*wd)), and
    the final (M_gpu, M_ref) per param."""
    W = [wl.weight(seed + 100 + i, s.shape) for i, s in enumerate(specs)]
    Wd = [to_dev(w, dtype) for w in W]
    Md = [torch.zeros(s.shape, dtype=torch.float32, device="cuda") for s in specs]
    M_ref = [np.zeros(s.shape) for s in specs]
    out = []
    for k in range(steps):
        W_prev = [host64(w) for w in Wd]
        G = [wl.lowrank_grad(seed + 1000 * k + i, s.shape[0], s.shape[1], 16, scale=1.0) for i, s in enumerate(specs)]
        Gd = [to_dev(g, grad_dtype or dtype) for g in G]
        pkg.muon_step(Wd, Gd, Md, lr=lr, wd=wd, mu=mu, nesterov=nesterov, ns_steps=ns_steps,
                      split_heads=[s.split_heads for s in specs], ns_dtype=ns_dtype, **scale)
        row = []
        for i, s in enumerate(specs):
            w_ref, M_ref[i] = oracle.muon_step(W_prev[i], host64(Gd[i]), M_ref[i], lr=lr, wd=wd, mu=mu,
                                               nesterov=nesterov, steps=ns_steps, split_heads=s.split_heads,
                                               **scale)
            row.append((host64(Wd[i]), w_ref, W_prev[i] * (1 - lr * wd)))
        out.append(row)
    torch.cuda.synchronize()
    assert pkg.default_handle().check() == 0
    return out, [(host64(Md[i]), M_ref[i]) for i in range(len(specs))]


def run_step(pkg, specs, dtype, steps=1, **kw):
    """run_step_per_step, flattened to the last step: per param
    (W_gpu, W_ref, W_prev * (1 - lr*wd), M_gpu, M_ref)."""
    per_step, moms = run_step_per_step(pkg, specs, dtype, steps, **kw)
    return [w + m for w, m in zip(per_step[-1], moms)]


def delta_err(w_gpu, w_ref, base):
    """Relative error of the update W - base."""
    return rel(w_gpu - base, w_ref - base)


def check_bf16_steps(per_step, tol, name):
    """cell_err of every step of every parameter below tol (recorded)."""
    for k, row in enumerate(per_step):
        for i, (w_gpu, w_ref, base) in enumerate(row):
            err = record(f"{name} step {k} param {i} (bf16 cell bound)", cell_err(w_gpu, w_ref, base), tol)
            assert err < tol, (name, k, i, err)


def test_step_single_fp32_matrix(pkg):
    # the single fp32 256x512 case: full-rank geometric spectrum, one step
    ws = wl.single_matrix_256x512()
    W0 = wl.weight(0, (256, 512))
    G = wl.lowrank_grad(0, 256, 512, 256)
    Wd, Gd = to_dev(W0, torch.float32), to_dev(G, torch.float32)
    Md = torch.zeros(256, 512, dtype=torch.float32, device="cuda")
    pkg.muon_step([Wd], [Gd], [Md], lr=0.02, wd=0.1, mu=0.95, nesterov=True)
    W_ref, M_ref = oracle.muon_step(W0.astype(np.float64), G.astype(np.float64), np.zeros((256, 512)), lr=0.02,
                                    wd=0.1, mu=0.95)
    assert ws.muon[0].shape == (256, 512)
    err = record("single fp32 256x512 step dW", delta_err(host64(Wd), W_ref, W0.astype(np.float64) * (1 - 0.02 * 0.1)),
                 TOL_F32)
    assert err < TOL_F32
    assert record("single fp32 256x512 momentum", rel(host64(Md), M_ref), TOL_EXACT) < TOL_EXACT


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_step_without_ns_checks_momentum_and_update_arithmetic(pkg, dtype):
    # ns_steps = 0: O = U/||U||_F, so W_new and M are fixed by plain arithmetic
    specs = [wl.ParamSpec("a", (100, 300)), wl.ParamSpec("b", (300, 100)), wl.ParamSpec("c", (1, 77)),
             wl.ParamSpec("d", (77, 1)), wl.ParamSpec("e", (64, 64))]
    per_step, moms = run_step_per_step(pkg, specs, dtype, steps=2, ns_steps=0)
    for m_gpu, m_ref in moms:
        assert rel(m_gpu, m_ref) < TOL_EXACT
    if dtype == torch.float32:
        for row in per_step:
            for w_gpu, w_ref, base in row:
                # one step: one rounding of W and one of the fp32 decay factor
                err = (np.linalg.norm(w_gpu - w_ref) - 2 * f32_budget(w_ref)) / np.linalg.norm(w_ref - base)
                assert record("ns_steps=0 fp32 dW beyond two roundings", max(err, 0.0), TOL_EXACT) < TOL_EXACT
    else:
        check_bf16_steps(per_step, TOL_EXACT, "ns_steps=0 bf16")


def test_step_fp32_path_mixed_shapes(pkg):
    specs = [wl.ParamSpec("a", (96, 160)), wl.ParamSpec("b", (160, 96)), wl.ParamSpec("c", (96, 160))]
    per_step, moms = run_step_per_step(pkg, specs, torch.float32, steps=2)
    for k, row in enumerate(per_step):
        for i, (w_gpu, w_ref, base) in enumerate(row):
            assert record(f"fp32 path mixed shapes step {k} param {i} dW", delta_err(w_gpu, w_ref, base),
                          TOL_F32) < TOL_F32
    for m_gpu, m_ref in moms:
        assert rel(m_gpu, m_ref) < TOL_EXACT


def test_step_bf16_gpt2_like(pkg):
    # two layers of the GPT-2-small shapes, three consecutive steps
    specs = wl.gpt2_small(layers=2).muon
    per_step, moms = run_step_per_step(pkg, specs, torch.bfloat16, steps=3)
    check_bf16_steps(per_step, TOL_BF16, "gpt2-like bf16")
    for m_gpu, m_ref in moms:
        assert rel(m_gpu, m_ref) < TOL_EXACT


def test_step_bf16_ns_into_fp32_params_shows_dw(pkg):
    # the bf16 tensor-core path writing fp32 parameters (bf16 gradients): the
    # stored update is the computed one up to one fp32 rounding, so dW is
    # held to the bf16 path's bar directly; three steps, wide, tall, split
    specs = wl.gpt2_small(layers=1).muon + [wl.ParamSpec("q", (512, 256), split_heads=4),
                                            wl.ParamSpec("big", (1024, 2560))]
    per_step, moms = run_step_per_step(pkg, specs, torch.float32, steps=3, grad_dtype=torch.bfloat16,
                                       ns_dtype=torch.bfloat16)
    for k, row in enumerate(per_step):
        for i, (w_gpu, w_ref, base) in enumerate(row):
            err = record(f"bf16 NS -> fp32 params step {k} {specs[i].name} dW", delta_err(w_gpu, w_ref, base),
                         TOL_BF16)
            assert err < TOL_BF16, (k, specs[i].name, err)
    for m_gpu, m_ref in moms:
        assert rel(m_gpu, m_ref) < TOL_EXACT


def test_step_bf16_split_heads(pkg):
    specs = [wl.ParamSpec("q", (512, 256), split_heads=4), wl.ParamSpec("k", (256, 512), split_heads=2)]
    per_step, _ = run_step_per_step(pkg, specs, torch.bfloat16, steps=1)
    check_bf16_steps(per_step, TOL_BF16, "split heads bf16")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("scale", [dict(scale_mode="mup"), dict(scale_mode="mup", extra_scale=1.5),
                                   dict(update_rms=0.18, extra_scale=0.5)])
def test_step_scale_modes(pkg, dtype, scale):
    # muP sqrt(d_out / d_in), DeepSeek-V4 gamma as update_rms, and the extra
    # scale factor, on wide, tall and square parameters
    specs = [wl.ParamSpec("a", (128, 384)), wl.ParamSpec("b", (384, 128)), wl.ParamSpec("c", (192, 192))]
    per_step, moms = run_step_per_step(pkg, specs, dtype, steps=1, **scale)
    if dtype == torch.float32:
        for w_gpu, w_ref, base in per_step[0]:
            assert record(f"scale mode {scale} fp32 dW", delta_err(w_gpu, w_ref, base), TOL_F32) < TOL_F32
    else:
        check_bf16_steps(per_step, TOL_BF16, f"scale mode {scale} bf16")
    for m_gpu, m_ref in moms:
        assert rel(m_gpu, m_ref) < TOL_EXACT


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("method", ["standard", "gram"])
def test_step_coefficient_schedule(pkg, dtype, method):
    # a hybrid 10-step iteration: 8 quintic steps, then 2 Newton cubic steps
    sched = [oracle.QUINTIC] * 8 + [(1.5, -0.5, 0.0)] * 2
    specs = [wl.ParamSpec("a", (128, 384)), wl.ParamSpec("b", (384, 128))]
    W = [wl.weight(300 + i, s.shape) for i, s in enumerate(specs)]
    G = [wl.lowrank_grad(310 + i, s.shape[0], s.shape[1], 16, scale=1.0) for i, s in enumerate(specs)]
    Wd, Gd = [to_dev(w, dtype) for w in W], [to_dev(g, dtype) for g in G]
    Md = [torch.zeros(s.shape, device="cuda") for s in specs]
    W0 = [host64(w) for w in Wd]
    pkg.muon_step(Wd, Gd, Md, lr=0.02, wd=0.1, ns_steps=10, coeffs=sched, ns_method=method)
    torch.cuda.synchronize()
    assert pkg.default_handle().check() == 0
    for i, s_ in enumerate(specs):
        w_ref, _ = oracle.muon_step(W0[i], host64(Gd[i]), np.zeros(s_.shape), lr=0.02, wd=0.1, steps=10,
                                    coeffs=sched, method=method)
        base = W0[i] * (1 - 0.02 * 0.1)
        if dtype == torch.float32:
            err = record(f"schedule {method} fp32 dW", delta_err(host64(Wd[i]), w_ref, base), TOL_F32)
            assert err < TOL_F32
        else:
            err = record(f"schedule {method} bf16 (cell bound)", cell_err(host64(Wd[i]), w_ref, base), TOL_BF16)
            assert err < TOL_BF16
    with pytest.raises(ValueError):
        pkg.muon_step(Wd, Gd, Md, lr=0.02, wd=0.1, ns_steps=5, coeffs=sched)


def test_step_is_deterministic(pkg):
    specs = [wl.ParamSpec("a", (200, 640)), wl.ParamSpec("b", (640, 200))]
    outs = []
    for _ in range(2):
        outs.append([r[0] for r in run_step(pkg, specs, torch.bfloat16, steps=2)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_step_nonfinite_gradient_is_reported(pkg):
    W = to_dev(wl.weight(1, (64, 128)), torch.bfloat16)
    G = to_dev(wl.gaussian(2, (64, 128)), torch.bfloat16)
    G[3, 5] = float("nan")
    M = torch.zeros(64, 128, device="cuda")
    pkg.muon_step([W], [G], [M], lr=0.02, wd=0.1)
    assert pkg.default_handle().check() == 5      # MUON_ERR_NONFINITE
    assert pkg.default_handle().check() == 0


def test_step_rejects_bad_arguments(pkg):
    W = torch.zeros(64, 128, device="cuda", dtype=torch.bfloat16)
    M = torch.zeros(64, 128, device="cuda")
    with pytest.raises(pkg.MuonError) as e:
        pkg.muon_step([W], [W], [M], lr=0.02, wd=0.1, split_heads=[3])
    assert e.value.status == 1
    with pytest.raises(ValueError):
        pkg.muon_step([W], [W], [M.to(torch.bfloat16)], lr=0.02, wd=0.1)
    with pytest.raises(pkg.MuonError) as e:
        pkg.muon_step([W], [W], [M], lr=0.02, wd=0.1, extra_scale=float("inf"))
    assert e.value.status == 1
    with pytest.raises(ValueError):
        pkg.muon_step([W], [W], [M], lr=0.02, wd=0.1, scale_mode="spectral")
    pkg.muon_step([], [], [], lr=0.02, wd=0.1)     # no-op


# --------------------------------------------------------------- AdamW

@pytest.mark.parametrize("pdtype", [torch.float32, torch.bfloat16])
def test_adamw_vs_oracle(pkg, pdtype):
    sizes = [1, 17, 768, 3072, 40000]
    P = [wl.gaussian(200 + i, (s,)) for i, s in enumerate(sizes)]
    Pd = [to_dev(p, pdtype) for p in P]
    Md = [torch.zeros(s, device="cuda") for s in sizes]
    Vd = [torch.zeros(s, device="cuda") for s in sizes]
    ref = [(host64(p), np.zeros(s), np.zeros(s)) for p, s in zip(Pd, sizes)]
    kw = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, wd=0.1)
    for t in range(1, 4):
        G = [wl.gaussian(300 + 10 * t + i, (s,)) for i, s in enumerate(sizes)]
        Gd = [to_dev(g, pdtype) for g in G]
        pkg.adamw_step(Pd, Gd, Md, Vd, step=t, **kw)
        ref = [oracle.adamw_step(p, host64(g), m, v, t, **kw) for (p, m, v), g in zip(ref, Gd)]
    torch.cuda.synchronize()
    for (p, m, v), pd, md, vd in zip(ref, Pd, Md, Vd):
        assert rel(host64(md), m) < TOL_EXACT
        assert rel(host64(vd), v) < TOL_EXACT
        if pdtype == torch.float32:
            assert rel(host64(pd), p) < TOL_EXACT
        else:
            assert np.linalg.norm(host64(pd) - p) <= 3 * bf16_budget(p) + TOL_EXACT * np.linalg.norm(p)


# ---------------------------------------------------------------- Gram

GRAM_BF16 = [(256, 4096), (128, 2048), (200, 700), (700, 200), (1, 300), (130, 1000), (256, 512)]


@pytest.mark.parametrize("shape", GRAM_BF16)
def test_orthogonalize_gram_bf16(pkg, shape):
    rank = min(shape) if shape == (256, 512) else 64
    X = wl.lowrank_grad(11, shape[0], shape[1], rank)
    t = to_dev(X, torch.bfloat16)
    ref = oracle.gram_newton_schulz(host64(t))
    pkg.muon_orthogonalize(t, ns_method="gram")
    assert record(f"orthogonalize gram bf16 {shape}", rel(host64(t), ref), TOL_BF16) < TOL_BF16


@pytest.mark.parametrize("shape", [(100, 300), (300, 100), (64, 512), (1, 40)])
def test_orthogonalize_gram_fp32(pkg, shape):
    X = wl.lowrank_grad(12, shape[0], shape[1], 32)
    t = to_dev(X, torch.float32)
    pkg.muon_orthogonalize(t, ns_method="gram")
    err = rel(host64(t), oracle.gram_newton_schulz(X.astype(np.float64)))
    assert record(f"orthogonalize gram fp32 {shape}", err, TOL_F32) < TOL_F32


@pytest.mark.parametrize("steps", [0, 1, 3])
def test_orthogonalize_gram_step_counts(pkg, steps):
    X = wl.lowrank_grad(13, 96, 640, 16)
    tb = to_dev(X, torch.bfloat16)
    ref = oracle.gram_newton_schulz(host64(tb), steps)
    pkg.muon_orthogonalize(tb, steps=steps, ns_method="gram")
    assert rel(host64(tb), ref) < TOL_BF16


def test_step_gram_bf16(pkg):
    specs = [wl.ParamSpec("a", (128, 1024)), wl.ParamSpec("b", (1024, 128)), wl.ParamSpec("c", (256, 768))]
    W = [wl.weight(400 + i, s.shape) for i, s in enumerate(specs)]
    Wd = [to_dev(w, torch.bfloat16) for w in W]
    Md = [torch.zeros(s.shape, device="cuda") for s in specs]
    W0 = [host64(w) for w in Wd]
    G = [to_dev(wl.lowrank_grad(500 + i, s.shape[0], s.shape[1], 32), torch.bfloat16) for i, s in enumerate(specs)]
    pkg.muon_step(Wd, G, Md, lr=0.02, wd=0.1, ns_method="gram")
    assert pkg.default_handle().check() == 0
    for i in range(len(specs)):
        w_ref, m_ref = oracle.muon_step(W0[i], host64(G[i]), np.zeros(specs[i].shape), lr=0.02, wd=0.1,
                                        method="gram")
        base = W0[i] * (1 - 0.02 * 0.1)
        err = record(f"gram step bf16 {specs[i].shape} (cell bound)", cell_err(host64(Wd[i]), w_ref, base), TOL_BF16)
        assert err < TOL_BF16
        assert rel(host64(Md[i]), m_ref) < TOL_EXACT


# ------------------------------------------------ rank-1 and >2-D params

RANK1_SHAPES = [(1024, 4096), (4096, 1024), (1408, 2048), (768, 3072), (96, 200)]


def rank1(seed, rows, cols):
    """A rank-1 matrix s u v^T (unit u, v) with no noise: every iterate stays
    rank-1, and the update's b*A + c*A^2 part cancels most of a*X on the
    diagonal of P."""
    rng = np.random.default_rng(seed)
    u = rng.standard_normal(rows)
    v = rng.standard_normal(cols)
    return (0.7 * np.outer(u / np.linalg.norm(u), v / np.linalg.norm(v))).astype(np.float32)


@pytest.mark.parametrize("shape", RANK1_SHAPES)
@pytest.mark.parametrize("method", ["standard", "gram"])
def test_orthogonalize_rank1_bf16(pkg, shape, method):
    t = to_dev(rank1(21, *shape), torch.bfloat16)
    ref = oracle.orthogonalize(host64(t), method=method)
    pkg.muon_orthogonalize(t, ns_method=method)
    err = record(f"orthogonalize rank-1 {method} bf16 {shape}", rel(host64(t), ref), TOL_BF16)
    assert err < TOL_BF16


@pytest.mark.parametrize("shape", [(1024, 4096), (4096, 1024)])
def test_step_rank1_gradient(pkg, shape):
    # a rank-1 gradient through the whole step, both into bf16 parameters
    # (cell bound) and into fp32 parameters (dW itself)
    for pdt in (torch.bfloat16, torch.float32):
        W = to_dev(wl.weight(31, shape), pdt)
        G = to_dev(rank1(32, *shape), torch.bfloat16)
        M = torch.zeros(shape, device="cuda")
        W0 = host64(W)
        pkg.muon_step([W], [G], [M], lr=0.02, wd=0.1, ns_dtype=torch.bfloat16)
        assert pkg.default_handle().check() == 0
        w_ref, m_ref = oracle.muon_step(W0, host64(G), np.zeros(shape), lr=0.02, wd=0.1)
        base = W0 * (1 - 0.02 * 0.1)
        if pdt == torch.bfloat16:
            err = record(f"rank-1 step bf16 params {shape} (cell bound)", cell_err(host64(W), w_ref, base), TOL_BF16)
        else:
            err = record(f"rank-1 step fp32 params {shape} dW", delta_err(host64(W), w_ref, base), TOL_BF16)
        assert err < TOL_BF16
        assert rel(host64(M), m_ref) < TOL_EXACT


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_step_higher_rank_params_with_scale_dim(pkg, dtype):
    # parameters with more than two dimensions: the gradient is viewed as
    # (size(0), -1) and the update scale uses the parameter's first two
    # dimensions ("迎接DeepSeek开源周…Muon优化器", §代码: g.view(g.size(0), -1)
    # and p.shape[:2]).  Through the C ABI: the flattened 2-D view and
    # scale_dim = max of the first two dimensions.
    shapes = [(64, 16, 3, 3), (32, 128, 4), (96, 8, 40)]
    tol = TOL_F32 if dtype == torch.float32 else TOL_BF16
    Wf = [wl.weight(40 + i, s) for i, s in enumerate(shapes)]
    Gf = [wl.gaussian(50 + i, s, 0.01) for i, s in enumerate(shapes)]
    Wd = [to_dev(w, dtype) for w in Wf]
    Gd = [to_dev(g, dtype) for g in Gf]
    Md = [torch.zeros(s, device="cuda") for s in shapes]
    W0 = [host64(w) for w in Wd]
    flat = lambda t: t.view(t.shape[0], -1)
    pkg.muon_step([flat(w) for w in Wd], [flat(g) for g in Gd], [flat(m) for m in Md], lr=0.02, wd=0.1,
                  scale_dims=[max(s[0], s[1]) for s in shapes])
    assert pkg.default_handle().check() == 0
    for i, s in enumerate(shapes):
        w_ref, m_ref = oracle.muon_step(W0[i], host64(Gd[i]), np.zeros(s), lr=0.02, wd=0.1)
        assert w_ref.shape == s and m_ref.shape == s
        base = W0[i] * (1 - 0.02 * 0.1)
        got = host64(Wd[i])
        err = delta_err(got, w_ref, base) if dtype == torch.float32 else cell_err(got, w_ref, base)
        assert record(f"scale_dim step {dtype} {s}", err, tol) < tol, (s, err)
        assert rel(host64(Md[i]), m_ref) < TOL_EXACT
    # without scale_dim the flattened shape would set the scale: a different update
    w_wrong = oracle.muon_step(W0[1].reshape(32, -1), host64(Gd[1]).reshape(32, -1), np.zeros((32, 512)),
                               lr=0.02, wd=0.1)[0]
    assert rel(w_wrong - W0[1].reshape(32, -1) * 0.998, host64(Wd[1]).reshape(32, -1) - W0[1].reshape(32, -1) * 0.998) > 0.5


# ------------------------------------------------------- workspace sizing

def test_workspace_size_matches_the_allocation_of_a_step():
    """muon_workspace_size predicts what the first step allocates (rounded to
    64 MiB), follows the handle's limit, and enqueues nothing."""
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    specs = [wl.ParamSpec("a", (1024, 4096)), wl.ParamSpec("b", (4096, 1024)), wl.ParamSpec("c", (512, 512)),
             wl.ParamSpec("q", (512, 256), split_heads=2)]
    shapes = [s.shape for s in specs]
    split = [s.split_heads for s in specs]
    h = pkg.MuonHandle(0)
    need = pkg.workspace_size(shapes, split_heads=split, handle=h)
    assert need > 0
    # a limit below one group's need shrinks the chunks, never below one matrix
    h.set_workspace_limit(need // 2)
    small = pkg.workspace_size(shapes, split_heads=split, handle=h)
    assert 0 < small < need
    h.set_workspace_limit(64 << 30)
    W = [torch.zeros(s.shape, device="cuda", dtype=torch.bfloat16) for s in specs]
    G = [torch.randn(s.shape, device="cuda").to(torch.bfloat16) for s in specs]
    M = [torch.zeros(s.shape, device="cuda") for s in specs]
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    pkg.muon_step(W, G, M, lr=0.02, wd=0.1, split_heads=split, handle=h)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert h.check() == 0
    used = free0 - free1
    rounded = -(-need // (64 << 20)) * (64 << 20)
    # the workspace plus a descriptor buffer of at most a few MiB
    assert rounded <= used <= rounded + (16 << 20), (need, rounded, used)
    assert pkg.workspace_size([], handle=h) == 0


# ------------------------------------------- fp32 path: tensor cores vs CUDA cores

@pytest.fixture(scope="module")
def cuda_core_handle(pkg):
    """A handle whose fp32 path runs on the CUDA cores (MUON_F32_TC=0)."""
    import os
    old = os.environ.get("MUON_F32_TC")
    os.environ["MUON_F32_TC"] = "0"
    try:
        return pkg.MuonHandle(0)
    finally:
        if old is None:
            del os.environ["MUON_F32_TC"]
        else:
            os.environ["MUON_F32_TC"] = old


F32_TC_SHAPES = ORTHO_SHAPES + [(768, 3072), (3072, 768), (768, 768), (130, 4100)]


@pytest.mark.parametrize("shape", F32_TC_SHAPES)
def test_fp32_tensor_core_path_matches_oracle_and_cuda_cores(pkg, cuda_core_handle, shape):
    # fp32 inputs: the default handle runs the standard method on the tensor
    # cores with three-plane bf16 operands (six MMAs per product); both it and
    # the CUDA-core path are held to the fp32 bar against the oracle
    X = wl.lowrank_grad(17, shape[0], shape[1], 32)
    ref = oracle.newton_schulz(X.astype(np.float64))
    a, b = to_dev(X, torch.float32), to_dev(X, torch.float32)
    pkg.muon_orthogonalize(a)
    pkg.muon_orthogonalize(b, handle=cuda_core_handle)
    torch.cuda.synchronize()
    assert pkg.default_handle().check() == 0 and cuda_core_handle.check() == 0
    e_tc = record(f"fp32 tensor-core path {shape}", rel(host64(a), ref), TOL_F32)
    e_cc = record(f"fp32 CUDA-core path {shape}", rel(host64(b), ref), TOL_F32)
    assert e_tc < TOL_F32 and e_cc < TOL_F32


def test_fp32_tensor_core_step_gpt2_layer_three_steps(pkg):
    # one GPT-2-small layer in fp32 parameters and gradients, three steps on
    # the tensor-core fp32 path; the oracle takes each step from the GPU's
    # parameter, dW held to the fp32 bar
    specs = wl.gpt2_small(layers=1).muon
    per_step, moms = run_step_per_step(pkg, specs, torch.float32, steps=3)
    for k, row in enumerate(per_step):
        for i, (w_gpu, w_ref, base) in enumerate(row):
            err = record(f"fp32 tensor-core step {k} {specs[i].name} dW", delta_err(w_gpu, w_ref, base), TOL_F32)
            assert err < TOL_F32
    for m_gpu, m_ref in moms:
        assert rel(m_gpu, m_ref) < TOL_EXACT


@pytest.mark.parametrize("shape", [(2048, 8192), (2048, 2048), (4096, 4096)])
def test_fp32_large_m_runs_within_the_bar(pkg, shape):
    # up to m = 2048 the fp32 path runs on the tensor cores (three-plane
    # products, two accumulators per tile); above, the products' fp32
    # accumulation error, which grows with K = m, would near the bar
    # (7.5e-5 at 4096 x 4096) and they stay on the CUDA cores
    X = wl.lowrank_grad(18, shape[0], shape[1], 64)
    t = to_dev(X, torch.float32)
    pkg.muon_orthogonalize(t)
    err = record(f"fp32 path, large m {shape}", rel(host64(t), oracle.newton_schulz(X.astype(np.float64))), TOL_F32)
    assert err < TOL_F32
