"""Seeded synthetic inputs for the Muon step: weight-set shapes and generators.

This module holds only input synthesis (random numbers, orthonormal bases,
shape tables).  It contains none of the optimizer's arithmetic, so both the
CUDA path's tests/benchmark and the fp64 oracle can be fed from it.

Recipes (all seeded):

* weights ~ N(0, 0.02), stored bf16 (or fp32 for the single-matrix case);
* gradients are low-rank plus noise: U diag(sigma) V^T + noise * N(0, 1),
  U, V with orthonormal columns (QR of Gaussian matrices),
  sigma_i = 0.5 ** (i / 8), then multiplied by ``scale``;
* the wide-matrix sweep uses plain Gaussian matrices (Marchenko-Pastur
  spectrum) as momentum inputs.

Host generation uses numpy's PCG64 ``default_rng(seed)``; full-size weight
sets (billions of elements) are generated on the device with a seeded
``torch.Generator`` instead, and sampled matrices are copied back to the host
when the oracle needs them.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class ParamSpec:
    name: str
    shape: tuple            # the parameter's own shape
    split_heads: int = 1    # Muon Split: equal row blocks orthogonalised separately


@dataclass
class WeightSet:
    name: str
    muon: list = field(default_factory=list)     # list[ParamSpec], 2-D hidden matrices
    adamw: list = field(default_factory=list)    # list[ParamSpec], vectors (AdamW fallback)
    grad_rank: int = 64
    grad_scale: float = 1.0
    grad_noise: float = 1e-3

    @property
    def muon_numel(self) -> int:
        return sum(int(np.prod(p.shape)) for p in self.muon)

    @property
    def adamw_numel(self) -> int:
        return sum(int(np.prod(p.shape)) for p in self.adamw)


def single_matrix_256x512() -> WeightSet:
    """One fp32 256x512 matrix with a full-rank geometric spectrum."""
    return WeightSet("single-fp32-256x512", [ParamSpec("w", (256, 512))], [],
                     grad_rank=256, grad_scale=1.0)


def gpt2_small(layers: int = 12, d: int = 768) -> WeightSet:
    """GPT-2-small-shaped set: per layer c_attn d x 3d, c_proj d x d,
    c_fc d x 4d, mlp_proj 4d x d (Conv1D in x out layout) plus LayerNorm and
    bias vectors on the AdamW path and a final LayerNorm."""
    ws = WeightSet("gpt2-small", grad_rank=64, grad_scale=1e-3)
    for i in range(layers):
        ws.muon += [ParamSpec(f"h.{i}.attn.c_attn.weight", (d, 3 * d)),
                    ParamSpec(f"h.{i}.attn.c_proj.weight", (d, d)),
                    ParamSpec(f"h.{i}.mlp.c_fc.weight", (d, 4 * d)),
                    ParamSpec(f"h.{i}.mlp.c_proj.weight", (4 * d, d))]
        ws.adamw += [ParamSpec(f"h.{i}.ln_1.weight", (d,)), ParamSpec(f"h.{i}.ln_1.bias", (d,)),
                     ParamSpec(f"h.{i}.attn.c_attn.bias", (3 * d,)),
                     ParamSpec(f"h.{i}.attn.c_proj.bias", (d,)),
                     ParamSpec(f"h.{i}.ln_2.weight", (d,)), ParamSpec(f"h.{i}.ln_2.bias", (d,)),
                     ParamSpec(f"h.{i}.mlp.c_fc.bias", (4 * d,)),
                     ParamSpec(f"h.{i}.mlp.c_proj.bias", (d,))]
    ws.adamw += [ParamSpec("ln_f.weight", (d,)), ParamSpec("ln_f.bias", (d,))]
    return ws


def llama3_8b(layers: int = 32, vocab: int = 128256) -> WeightSet:
    """Llama-3-8B-shaped set (out x in): q, o 4096x4096; k, v 1024x4096;
    gate, up 14336x4096; down 4096x14336, per layer.  The AdamW list holds
    what the tagging rule sends to AdamW: embed_tokens and lm_head
    (vocab x 4096, 2-D but named embed / lm_head) and the RMSNorm vectors."""
    ws = WeightSet("llama3-8b", grad_rank=64, grad_scale=1.0)
    ws.adamw += [ParamSpec("model.embed_tokens.weight", (vocab, 4096)), ParamSpec("lm_head.weight", (vocab, 4096)),
                 ParamSpec("model.norm.weight", (4096,))]
    for i in range(layers):
        ws.adamw += [ParamSpec(f"layers.{i}.input_layernorm.weight", (4096,)),
                     ParamSpec(f"layers.{i}.post_attention_layernorm.weight", (4096,))]
    for i in range(layers):
        p = f"layers.{i}."
        ws.muon += [ParamSpec(p + "attn.q_proj.weight", (4096, 4096)),
                    ParamSpec(p + "attn.k_proj.weight", (1024, 4096)),
                    ParamSpec(p + "attn.v_proj.weight", (1024, 4096)),
                    ParamSpec(p + "attn.o_proj.weight", (4096, 4096)),
                    ParamSpec(p + "mlp.gate_proj.weight", (14336, 4096)),
                    ParamSpec(p + "mlp.up_proj.weight", (14336, 4096)),
                    ParamSpec(p + "mlp.down_proj.weight", (4096, 14336))]
    return ws


def moonlight_moe(layers: int = 27, experts: int = 64, hidden: int = 2048,
                  expert_ffn: int = 1408, heads: int = 16) -> WeightSet:
    """Moonlight-like MoE set: per layer 64 experts x {gate, up ffn x hidden,
    down hidden x ffn} and attention q, k, v hidden x hidden, each split into
    ``heads`` row blocks (Muon Split)."""
    ws = WeightSet("moonlight-moe", grad_rank=64, grad_scale=1.0)
    for i in range(layers):
        for e in range(experts):
            p = f"layers.{i}.experts.{e}."
            ws.muon += [ParamSpec(p + "gate_proj.weight", (expert_ffn, hidden)),
                        ParamSpec(p + "up_proj.weight", (expert_ffn, hidden)),
                        ParamSpec(p + "down_proj.weight", (hidden, expert_ffn))]
        for w in ("q", "k", "v"):
            ws.muon.append(ParamSpec(f"layers.{i}.attn.{w}_proj.weight", (hidden, hidden),
                                     split_heads=heads))
    return ws


WIDE_SWEEP = [(m, n) for m in (256, 1024, 2048) for n in (4096, 16384)]
WIDE_BATCH = 64


def matrix_seed(seed: int, index: int) -> int:
    """Independent per-matrix seed derived from a set seed and an index."""
    return (int(seed) * 1_000_003 + int(index) * 7919 + 17) % (2 ** 63)


# ----------------------------------------------------------------- host (numpy)

def orthonormal_columns(rng: np.random.Generator, rows: int, k: int) -> np.ndarray:
    q, _ = np.linalg.qr(rng.standard_normal((rows, k)))
    return q


def lowrank_grad(seed: int, rows: int, cols: int, rank: int, *, noise: float = 1e-3,
                 scale: float = 1.0) -> np.ndarray:
    """U diag(0.5**(i/8)) V^T + noise*N(0,1), times ``scale`` (float32)."""
    rng = np.random.default_rng(seed)
    r = min(rank, rows, cols)
    U = orthonormal_columns(rng, rows, r)
    V = orthonormal_columns(rng, cols, r)
    sigma = 0.5 ** (np.arange(r) / 8.0)
    g = (U * sigma) @ V.T + noise * rng.standard_normal((rows, cols))
    return (scale * g).astype(np.float32)


def gaussian(seed: int, shape, std: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (std * rng.standard_normal(shape)).astype(np.float32)


def weight(seed: int, shape) -> np.ndarray:
    """Weights ~ N(0, 0.02) (float32)."""
    return gaussian(seed, shape, 0.02)


# --------------------------------------------------------------- device (torch)

def lowrank_grad_device(gen, rows: int, cols: int, rank: int, *, noise: float = 1e-3,
                        scale: float = 1.0, device="cuda", dtype=None):
    """Device twin of ``lowrank_grad`` drawn from a seeded torch.Generator
    (different random stream from the numpy one, same recipe)."""
    import torch
    dtype = dtype or torch.bfloat16
    r = min(rank, rows, cols)
    U, _ = torch.linalg.qr(torch.randn(rows, r, generator=gen, device=device))
    V, _ = torch.linalg.qr(torch.randn(cols, r, generator=gen, device=device))
    sigma = 0.5 ** (torch.arange(r, device=device, dtype=torch.float32) / 8.0)
    g = (U * sigma) @ V.T
    g.add_(torch.randn(rows, cols, generator=gen, device=device), alpha=noise)
    if scale != 1.0:
        g.mul_(scale)
    return g.to(dtype)
