"""Algorithmic work counts for reporting throughput (no optimizer arithmetic).

Per m x n Newton-Schulz matrix (m <= n after the transpose rule), per
iteration of the standard method, symmetric products counted on one
triangle:  X X^T  m(m+1)n,  A A  m^2(m+1),  B X  2 m^2 n.  The dense
convention (4 m^2 n + 2 m^3 per iteration) is reported beside it.
"""
from __future__ import annotations


def ns_dims(rows: int, cols: int, split_heads: int = 1):
    r = rows // split_heads
    return (min(r, cols), max(r, cols))


def ns_flops_standard(m: int, n: int, steps: int = 5) -> float:
    return float(steps) * (m * (m + 1) * n + m * m * (m + 1) + 2.0 * m * m * n)


def ns_flops_dense(m: int, n: int, steps: int = 5) -> float:
    return float(steps) * (4.0 * m * m * n + 2.0 * m ** 3)


def ns_flops_gram(m: int, n: int, steps: int = 5) -> float:
    """Gram method, algorithmic: R0 = X0 X0^T (one triangle), O = Q X0, and
    per iteration R^2 plus, from the second iteration, P Q and the two
    products of P R P (symmetric, one triangle each).  The bf16x3 split of
    the m x m products (three MMAs each) and the two-plane final product are
    implementation overhead and not counted."""
    sym = m * m * (m + 1)
    if steps == 0:
        return 0.0
    return float(m * (m + 1) * n + 2.0 * m * m * n + (steps + 3 * (steps - 1)) * sym)


def kernel_flops_standard(m: int, n: int):
    """Algorithmic flops of one matrix in each GEMM kernel class."""
    return {"syrk": float(m * (m + 1) * n), "poly": float(m * m * (m + 1)), "update": 2.0 * m * m * n}


def set_flops(specs, steps: int = 5):
    """(algorithmic, dense) NS flops of one step over a list of ParamSpec."""
    alg = dense = 0.0
    for s in specs:
        m, n = ns_dims(s.shape[0], s.shape[1], s.split_heads)
        alg += s.split_heads * ns_flops_standard(m, n, steps)
        dense += s.split_heads * ns_flops_dense(m, n, steps)
    return alg, dense


def prepare_bytes(numel: int, grad_bytes: int = 2) -> float:
    """HBM bytes of the momentum/Nesterov/norm/cast pass of the tensor-core
    path: read G, read and write M (fp32), write the two bf16 planes of the
    master X (hi = the MMA operand copy, lo = the residual)."""
    return float(numel) * (grad_bytes + 4 + 4 + 2 + 2)


def adamw_bytes(numel: int, param_bytes: int = 2, grad_bytes: int = 2) -> float:
    """HBM bytes of AdamW: read g, p, m, v; write p, m, v."""
    return float(numel) * (grad_bytes + 2 * param_bytes + 16)
