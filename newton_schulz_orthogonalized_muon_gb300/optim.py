"""Parameter classification and a torch-style optimizer over the C ABI.

Classification ("DeepSpeed 集成 Muon 优化器实战从正交化原理到 ZeRO 微调配置",
§use_muon 参数打标): a parameter takes the Muon step when it is 2-D and its
name contains neither "embed" nor "lm_head"; everything else (biases, norms,
embeddings, the output head) takes the AdamW fallback.  (The page's
comparison operator is lost in its text; it says Muon acts on 2-D weights
only, and that reading is taken.)  With ``higher_rank=True`` parameters with
more than two dimensions take the Muon step too, orthogonalised as the 2-D
view (size(0), -1), with the update scale from the first two dimensions of
their own shape (the printed Muon class of "迎接DeepSeek开源周…Muon优化器",
§代码: ``g.view(g.size(0), -1)`` and ``p.shape[:2]``), passed to the library
as ``scale_dim``.

``Muon`` keeps the fp32 momentum of every Muon parameter and the two fp32
AdamW moments of the rest on the device and calls ``muon_step`` and
``adamw_step`` once each per ``step()``; all arithmetic runs in the
library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _binding


_ADAMW_NAME_KEYS = ("embed", "lm_head")


def takes_muon(name: str, ndim: int, higher_rank: bool = False) -> bool:
    """True when a parameter of this name and rank takes the Muon step."""
    lowered = name.lower()
    rank_ok = ndim == 2 or (higher_rank and ndim > 2)
    return rank_ok and not any(k in lowered for k in _ADAMW_NAME_KEYS)


@dataclass
class MuonEntry:
    name: str
    param: torch.Tensor       # the parameter itself (any rank >= 2)
    rows: int                 # size(0)
    cols: int                 # numel / size(0)
    scale_dim: int            # max of the first two dimensions (0 for a 2-D parameter: the library's default)


def split_params(named_params, higher_rank: bool = False):
    """Split ``(name, tensor)`` pairs into Muon entries and AdamW tensors,
    keeping their order.  Parameters with ``requires_grad=False`` are left
    out."""
    muon, adamw = [], []
    for name, p in named_params:
        if not p.requires_grad:
            continue
        if takes_muon(name, p.dim(), higher_rank):
            rows = p.shape[0]
            cols = p.numel() // rows if rows else 0
            sdim = max(p.shape[0], p.shape[1]) if p.dim() > 2 else 0
            muon.append(MuonEntry(name, p, rows, cols, sdim))
        else:
            adamw.append((name, p))
    return muon, adamw


class Muon:
    """Muon with the AdamW fallback, in the form of a torch optimizer.

    ``named_params``: ``model.named_parameters()`` (or any ``(name, tensor)``
    pairs of contiguous CUDA tensors, fp32 or bf16).  Muon hyper-parameters
    follow ``muon_step``: ``lr``, ``wd`` (decoupled), ``momentum``,
    ``nesterov``, ``ns_steps``, ``ns_method`` ("standard" | "gram" | "auto"),
    ``update_rms`` (0.2: the update RMS matched to AdamW's); ``split_heads``
    maps a parameter name to its Muon-Split head count; ``higher_rank`` sends
    parameters with more than two dimensions to the Muon step (see the
    module docstring).  The AdamW fallback takes ``adamw_lr`` (default
    ``lr``), ``adamw_betas``, ``adamw_eps`` and ``adamw_wd`` (default
    ``wd``); each AdamW parameter counts its own steps for the bias
    correction, as the printed class does."""

    def __init__(self, named_params, *, lr: float, wd: float = 0.1, momentum: float = 0.95, nesterov: bool = True,
                 ns_steps: int = 5, ns_method: str = "standard", update_rms: float = 0.2, split_heads=None,
                 adamw_lr=None, adamw_betas=(0.9, 0.95), adamw_eps: float = 1e-8, adamw_wd=None, higher_rank=False,
                 ns_dtype=None, handle=None):
        self.muon, adamw = split_params(named_params, higher_rank)
        self.adamw_names = [n for n, _ in adamw]
        self.adamw_params = [p for _, p in adamw]
        for e in self.muon:
            if not e.param.is_cuda or not e.param.is_contiguous():
                raise ValueError(f"{e.name}: Muon parameters must be contiguous CUDA tensors")
        self.lr, self.wd, self.momentum, self.nesterov = float(lr), float(wd), float(momentum), bool(nesterov)
        self.ns_steps, self.ns_method, self.update_rms = int(ns_steps), ns_method, float(update_rms)
        heads = dict(split_heads or {})
        self.split = [int(heads.get(e.name, 1)) for e in self.muon]
        self.adamw_lr = float(lr if adamw_lr is None else adamw_lr)
        self.betas = (float(adamw_betas[0]), float(adamw_betas[1]))
        self.eps = float(adamw_eps)
        self.adamw_wd = float(wd if adamw_wd is None else adamw_wd)
        self.ns_dtype = ns_dtype      # None: bf16 tensor cores when every Muon parameter is bf16, else the fp32 path
        self.handle = handle
        self.momenta = [torch.zeros(e.rows, e.cols, dtype=torch.float32, device=e.param.device) for e in self.muon]
        self.exp_avg = [torch.zeros_like(p, dtype=torch.float32) for p in self.adamw_params]
        self.exp_avg_sq = [torch.zeros_like(p, dtype=torch.float32) for p in self.adamw_params]
        self.adamw_steps = [0] * len(self.adamw_params)

    def step(self, closure=None):
        """One step over every parameter whose ``.grad`` is set; ``closure``
        (optional) re-evaluates the model with gradients enabled first, and
        its loss is returned."""
        loss = None
        if closure is not None:
            with torch.enable_grad():
                loss = closure()
        with torch.no_grad():
            self._step()
        return loss

    def _step(self):
        idx = [i for i, e in enumerate(self.muon) if e.param.grad is not None]
        if idx:
            params = [self.muon[i].param.view(self.muon[i].rows, self.muon[i].cols) for i in idx]
            grads = [self.muon[i].param.grad.contiguous().view(self.muon[i].rows, self.muon[i].cols) for i in idx]
            _binding.muon_step(params, grads, [self.momenta[i] for i in idx], lr=self.lr, wd=self.wd,
                               mu=self.momentum, nesterov=self.nesterov, ns_method=self.ns_method,
                               ns_steps=self.ns_steps, update_rms=self.update_rms,
                               split_heads=[self.split[i] for i in idx],
                               scale_dims=[self.muon[i].scale_dim for i in idx], ns_dtype=self.ns_dtype,
                               handle=self.handle)
        # AdamW: one call per distinct step count (the bias correction)
        by_count = {}
        for j, p in enumerate(self.adamw_params):
            if p.grad is not None:
                self.adamw_steps[j] += 1
                by_count.setdefault(self.adamw_steps[j], []).append(j)
        for count, jdx in sorted(by_count.items()):
            _binding.adamw_step([self.adamw_params[j] for j in jdx],
                                [self.adamw_params[j].grad.contiguous() for j in jdx],
                                [self.exp_avg[j] for j in jdx], [self.exp_avg_sq[j] for j in jdx],
                                step=count, lr=self.adamw_lr, beta1=self.betas[0], beta2=self.betas[1],
                                eps=self.eps, wd=self.adamw_wd, handle=self.handle)

    def state_dict(self):
        """The optimizer state (momenta, AdamW moments and step counts, by
        parameter name, as copies on the host) and its hyper-parameters."""
        return {"muon": {e.name: self.momenta[i].detach().cpu().clone() for i, e in enumerate(self.muon)},
                "adamw": {n: {"exp_avg": self.exp_avg[j].detach().cpu().clone(),
                              "exp_avg_sq": self.exp_avg_sq[j].detach().cpu().clone(),
                              "step": self.adamw_steps[j]} for j, n in enumerate(self.adamw_names)},
                "hparams": {"lr": self.lr, "wd": self.wd, "momentum": self.momentum, "nesterov": self.nesterov,
                            "ns_steps": self.ns_steps, "ns_method": self.ns_method, "update_rms": self.update_rms,
                            "adamw_lr": self.adamw_lr, "adamw_betas": self.betas, "adamw_eps": self.eps,
                            "adamw_wd": self.adamw_wd}}

    def load_state_dict(self, state):
        """Restore a ``state_dict``: the same parameter names are required;
        the hyper-parameters are taken from it."""
        names = [e.name for e in self.muon]
        if sorted(state["muon"]) != sorted(names) or sorted(state["adamw"]) != sorted(self.adamw_names):
            raise ValueError("the state holds other parameters than this optimizer")
        for i, n in enumerate(names):
            self.momenta[i].copy_(state["muon"][n])
        for j, n in enumerate(self.adamw_names):
            st = state["adamw"][n]
            self.exp_avg[j].copy_(st["exp_avg"])
            self.exp_avg_sq[j].copy_(st["exp_avg_sq"])
            self.adamw_steps[j] = int(st["step"])
        hp = state["hparams"]
        self.lr, self.wd, self.momentum, self.nesterov = hp["lr"], hp["wd"], hp["momentum"], hp["nesterov"]
        self.ns_steps, self.ns_method, self.update_rms = hp["ns_steps"], hp["ns_method"], hp["update_rms"]
        self.adamw_lr, self.betas, self.eps, self.adamw_wd = (hp["adamw_lr"], tuple(hp["adamw_betas"]),
                                                              hp["adamw_eps"], hp["adamw_wd"])

    def zero_grad(self, set_to_none: bool = True):
        for p in [e.param for e in self.muon] + self.adamw_params:
            if p.grad is not None:
                if set_to_none:
                    p.grad = None
                else:
                    p.grad.zero_()
