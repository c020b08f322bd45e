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
    return {"syrk": float(m * (m + 1) * n), "poly": float(m * m * (m + 1)), "update": 2.0 * m * m * n,
            "final": 2.0 * m * m * n}


def kernel_flops_gram(m: int, n: int):
    """Gram method, algorithmic flops of one matrix in each kernel class the
    library reports: "syrk" R0 = X0 X0^T (one triangle), "poly"
    P = aI + bR + cR^2 (R^2 on one triangle), "update" one symmetric m x m
    product (P Q, P R or (P R) P, one triangle), "final" O = Q X0."""
    sym = float(m * m * (m + 1))
    return {"syrk": float(m * (m + 1) * n), "poly": sym, "update": sym, "final": 2.0 * m * m * n}


def kernel_mma_factor_gram():
    """Tensor-core work per algorithmic flop of each Gram-method class: the
    m x m products run as bf16x3 (hi*hi + hi*lo + lo*hi, three MMAs) and the
    final product applies both planes of Q (two MMAs)."""
    return {"syrk": 1.0, "poly": 3.0, "update": 3.0, "final": 2.0}


def kernel_launches(method: str, steps: int = 5):
    """Launches per same-shape chunk of each kernel class, by method."""
    if method == "gram":
        return {"syrk": 1, "poly": steps, "update": 3 * max(steps - 1, 0), "final": 1}
    return {"syrk": steps, "poly": steps, "update": max(steps - 1, 0), "final": 1}


def kernel_flops(method: str, m: int, n: int):
    return kernel_flops_gram(m, n) if method == "gram" else kernel_flops_standard(m, n)


def ns_flops(method: str, m: int, n: int, steps: int = 5) -> float:
    return ns_flops_gram(m, n, steps) if method == "gram" else ns_flops_standard(m, n, steps)


def set_flops(specs, steps: int = 5, method: str = "standard"):
    """(algorithmic, dense) NS flops of one step over a list of ParamSpec.
    Algorithmic flops are the method's own (ns_flops_standard or
    ns_flops_gram); the dense convention is the standard method's
    4 m^2 n + 2 m^3 per iteration whatever the method."""
    alg = dense = 0.0
    for s in specs:
        m, n = ns_dims(s.shape[0], s.shape[1], s.split_heads)
        alg += s.split_heads * ns_flops(method, m, n, steps)
        dense += s.split_heads * ns_flops_dense(m, n, steps)
    return alg, dense


def prepare_bytes(numel: int, grad_bytes: int = 2) -> float:
    """HBM bytes of the momentum/Nesterov/norm/cast pass of the tensor-core
    path: read G, read and write M (fp32), write the master X's two planes
    (hi = the bf16 MMA operand copy, lo = one signed byte with the next
    8 bits)."""
    return float(numel) * (grad_bytes + 4 + 4 + 2 + 1)


def adamw_bytes(numel: int, param_bytes: int = 2, grad_bytes: int = 2) -> float:
    """HBM bytes of AdamW: read g, p, m, v; write p, m, v."""
    return float(numel) * (grad_bytes + 2 * param_bytes + 16)
