"""fp64 CPU oracle for the Muon optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: it is used by ``tests/``, by ``__graft_entry__.smoke()``
and by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  It
shares no code, header, table or constant with the CUDA library under
``newton_schulz_orthogonalized_muon_gb300/csrc``; both sides only read the
same seeded inputs.

Every function is written plainly, in float64 numpy, with ``@`` (a library
matmul) as the only building block above elementwise arithmetic.  Each one
cites the passage of the source pages that defines it.  The pages are:

* [Moonlight] "迎接DeepSeek开源周[Kimi先开为敬]发布开源最新Muon优化器可替代
  AdamW计算效率直接翻倍" (coreui.cn): §1 权重衰减机制, §2 参数更新尺度调整,
  and the Muon optimizer class printed under §代码 (Muon step and its AdamW
  backup).
* [DeepSpeed] "DeepSpeed 集成 Muon 优化器实战从正交化原理到 ZeRO 微调配置"
  (lshu.cn): §use_muon 参数打标, §核心算子牛顿-舒尔茨正交化内核.
* [MindSpeed] "Muon 优化器" (gitcode.com/Ascend/MindSpeed feature doc):
  §TP 兼容适配 item 4 (QKV split).
* [Chensy] "Muon Optimizer and the Distributed Implementation"
  (blog.chensy.moe): §Formulation of Muon Optimizer, §Orthogonalization of
  Gradients, §Sign of a Matrix, §Newton-Schulz Iteration, §Variation of Muon
  Optimizer.

Readings taken where the pages are silent or garbled (each repeated where
it is used):

* normalisation epsilon: X0 = U / (||U||_F + eps), eps = 1e-7; a zero U
  gives O = 0;
* rows > cols: iterate on the transpose and transpose back;
* the Gram variant iterates R_{k+1} = P_k R_k P_k, Q_{k+1} = P_k Q_k with
  P_k = aI + bR_k + cR_k^2, R_0 = X0 X0^T, Q_0 = I, and returns Q X0;
* split heads: steps 2-6 of the step run per row block, the update scale
  uses the full parameter's first two dimensions.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, library routines, invariants); none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

# The quintic coefficients chosen to maximise the slope at zero
# ([DeepSpeed] §核心算子; [Chensy] §Newton-Schulz Iteration).
QUINTIC = (3.4445, -4.7750, 2.0315)
NS_STEPS = 5
NORM_EPS = 1e-7
UPDATE_RMS = 0.2


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def is_muon_param(name: str, ndim: int) -> bool:
    """Parameter tagging: a parameter takes the Muon path iff it is 2-D and
    its name contains neither "embed" nor "lm_head"; everything else falls
    back to AdamW ([DeepSpeed] §use_muon 参数打标, set_optimizer_flags)."""
    lowered = name.lower()
    return ndim == 2 and not any(k in lowered for k in ("embed", "lm_head"))


def momentum_update(M, G, mu: float, nesterov: bool):
    """Momentum buffer and the matrix handed to Newton-Schulz.

    M <- mu*M + G; the update direction is G + mu*M (with the new M) when
    Nesterov is on, else M itself ([Moonlight] §代码, Muon step;
    [Chensy] §Variation of Muon Optimizer, Nesterov form mu*M_t + G_t).
    Returns (M_new, U).
    """
    M_new = mu * _f64(M) + _f64(G)
    U = _f64(G) + mu * M_new if nesterov else M_new
    return M_new, U


def frobenius_normalize(X, eps: float = NORM_EPS):
    """X / (||X||_F + eps): puts every singular value in [0, 1]
    ([Chensy] §Newton-Schulz Iteration, first condition).  The eps is a
    reading: the page divides by the bare norm."""
    X = _f64(X)
    return X / (math.sqrt(float(np.sum(X * X))) + eps)


def step_coeffs(coeffs, steps: int):
    """The (a, b, c) of every step: one triple repeated, or a schedule of
    ``steps`` triples (a hybrid iteration such as DeepSeek-V4's, whose last
    steps use other coefficients: [Chensy] §Variation of Muon Optimizer)."""
    if len(coeffs) == 3 and not hasattr(coeffs[0], "__len__"):
        return [tuple(float(v) for v in coeffs)] * steps
    sched = [tuple(float(v) for v in c) for c in coeffs]
    if len(sched) != steps or any(len(c) != 3 for c in sched):
        raise ValueError("a coefficient schedule needs one (a, b, c) per step")
    return sched


def newton_schulz(X, steps: int = NS_STEPS, coeffs=QUINTIC, eps: float = NORM_EPS):
    """Quintic Newton-Schulz orthogonalisation ("standard" method).

    phi(X) = (aI + b XX^T + c (XX^T)^2) X applied ``steps`` times to the
    Frobenius-normalised input (``coeffs``: one (a, b, c), or one per step),
    evaluated in Horner form as
    A = XX^T, B = bA + cA^2, X <- aX + BX ([Chensy] §Newton-Schulz
    Iteration; [DeepSpeed] §核心算子, zeropower_via_newtonschulz5).

    Reading: when rows > cols the iteration runs on X^T (so A is the smaller
    Gram matrix) and the result is transposed back; phi commutes with
    transposition, so this changes cost only.
    """
    sched = step_coeffs(coeffs, steps)
    X = _f64(X)
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    X = frobenius_normalize(X, eps)
    for a, b, c in sched:
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if transposed else X


def gram_newton_schulz(X, steps: int = NS_STEPS, coeffs=QUINTIC, eps: float = NORM_EPS):
    """Newton-Schulz iterated on the small square Gram matrix ("gram" method,
    [DeepSpeed] §核心算子, zeropower_via_gram_newtonschulz: iterate on
    R = XX^T to cut the flops of wide matrices).

    Reading (the page gives no steps): every iterate X_k is Q_k X0 with Q_k a
    polynomial in R0 = X0 X0^T, so with P_k = aI + bR_k + cR_k^2 one has
    X_{k+1} = P_k X_k, hence Q_{k+1} = P_k Q_k and
    R_{k+1} = X_{k+1} X_{k+1}^T = P_k R_k P_k.  The result is Q X0, equal to
    the standard method in exact arithmetic.  No restarts (the page names
    none).  Rows > cols is handled by transposition as in newton_schulz.
    """
    sched = step_coeffs(coeffs, steps)
    X = _f64(X)
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    X0 = frobenius_normalize(X, eps)
    m = X0.shape[0]
    I = np.eye(m)
    R = X0 @ X0.T
    Q = I.copy()
    for a, b, c in sched:
        P = a * I + b * R + c * (R @ R)
        Q = P @ Q
        R = P @ R @ P
    O = Q @ X0
    return O.T if transposed else O


def orthogonalize(X, steps: int = NS_STEPS, coeffs=QUINTIC, method: str = "standard",
                  eps: float = NORM_EPS):
    """Dispatch on the Newton-Schulz method name ("standard" | "gram"),
    the two members of DeepSpeed's NS_METHODS ([DeepSpeed] §核心算子)."""
    if method == "standard":
        return newton_schulz(X, steps, coeffs, eps)
    if method == "gram":
        return gram_newton_schulz(X, steps, coeffs, eps)
    raise ValueError(f"unknown Newton-Schulz method {method!r}")


def update_scale(shape, update_rms: float = UPDATE_RMS, mode: str = "rms", extra: float = 1.0) -> float:
    """The factor the orthogonalised update is multiplied by, times
    ``extra`` (MindSpeed's extra scale factor, [MindSpeed] parameter table,
    --muon-extra-scale-factor).  A, B are the parameter's first two
    dimensions.

    * "rms": update_rms * sqrt(max(A, B)), 0.2 by default: scales the update
      to the RMS of an AdamW update ([Moonlight] §2 参数更新尺度调整 and
      adjust_lr_for_muon under §代码).  DeepSeek-V4's rescaling
      sqrt(max(n, m)) * gamma is this form with update_rms = gamma ([Chensy]
      §Variation of Muon Optimizer).
    * "mup": sqrt(d_out / d_in) with the weight stored as (d_out, d_in) =
      (A, B): the dual of the gradient under the RMS -> RMS operator norm
      is sqrt(d_out / d_in) msign(G) ([Chensy] §Variation of Muon
      Optimizer, the muP form)."""
    A, B = int(shape[0]), int(shape[1])
    if mode == "rms":
        base = update_rms * math.sqrt(max(A, B))
    elif mode == "mup":
        base = math.sqrt(A / B)
    else:
        raise ValueError(f"unknown scale mode {mode!r}")
    return extra * base


def apply_update(W, O, lr: float, wd: float, shape, update_rms: float = UPDATE_RMS, mode: str = "rms",
                 extra: float = 1.0):
    """Decoupled weight decay then the scaled step:
    W <- W * (1 - lr*wd) - lr * scale * O (scale from update_scale, by
    default 0.2*sqrt(max(A,B))); the decay uses the unadjusted lr
    ([Moonlight] §1 权重衰减机制, §2 更新公式, and the Muon step under §代码)."""
    return _f64(W) * (1.0 - lr * wd) - lr * update_scale(shape, update_rms, mode, extra) * _f64(O)


def orthogonalize_split(U, split_heads: int = 1, steps: int = NS_STEPS, coeffs=QUINTIC,
                        method: str = "standard", eps: float = NORM_EPS):
    """Muon Split / QKV split: orthogonalise each of ``split_heads`` equal
    row blocks independently and concatenate them back in place
    ([DeepSpeed] TL;DR, Muon Split per attention head; [MindSpeed] §TP 兼容适配,
    QKV split)."""
    U = _f64(U)
    rows = U.shape[0]
    if split_heads < 1 or rows % split_heads:
        raise ValueError("split_heads must divide the row count")
    h = rows // split_heads
    blocks = [orthogonalize(U[i * h:(i + 1) * h], steps, coeffs, method, eps)
              for i in range(split_heads)]
    return np.concatenate(blocks, axis=0)


def muon_step(W, G, M, *, lr: float, wd: float, mu: float = 0.95, nesterov: bool = True,
              steps: int = NS_STEPS, coeffs=QUINTIC, method: str = "standard",
              split_heads: int = 1, update_rms: float = UPDATE_RMS, eps: float = NORM_EPS,
              scale_mode: str = "rms", extra_scale: float = 1.0):
    """One Muon step for one parameter ([Moonlight] §代码, Muon step):
    momentum (and Nesterov), Newton-Schulz on the (flattened) update, then
    decay and the scaled update.  A gradient with more than two dimensions is
    viewed as (size(0), -1); the update scale uses the parameter's own first
    two dimensions.  Returns (W_new, M_new) as float64 arrays of W's and M's
    shapes."""
    W = _f64(W)
    G2 = _f64(G).reshape(G.shape[0], -1)
    M2 = _f64(M).reshape(G2.shape)
    M_new, U = momentum_update(M2, G2, mu, nesterov)
    O = orthogonalize_split(U, split_heads, steps, coeffs, method, eps)
    W_new = apply_update(W.reshape(O.shape), O, lr, wd, W.shape, update_rms, scale_mode, extra_scale)
    return W_new.reshape(W.shape), M_new.reshape(np.shape(M))


def adamw_step(p, g, m, v, step: int, *, lr: float, beta1: float, beta2: float,
               eps: float, wd: float):
    """The AdamW backup of the printed Muon class ([Moonlight] §代码):

    m <- m + (1-beta1)(g - m); v <- v + (1-beta2)(g^2 - v);
    u = m / (eps + sqrt(v)); scale = (1-beta1^t) / sqrt(1-beta2^t);
    p <- p*(1 - lr*wd) - (lr/scale) * u.

    ``step`` is the count after this call's increment (t >= 1).  Note eps is
    added to sqrt of the uncorrected v, as printed.  Returns (p, m, v).
    """
    if step < 1:
        raise ValueError("step counts from 1")
    g = _f64(g)
    m = _f64(m) + (1.0 - beta1) * (g - _f64(m))
    v = _f64(v) + (1.0 - beta2) * (g * g - _f64(v))
    u = m / (eps + np.sqrt(v))
    scale = (1.0 - beta1 ** step) / math.sqrt(1.0 - beta2 ** step)
    p = _f64(p) * (1.0 - lr * wd) - (lr / scale) * u
    return p, m, v

