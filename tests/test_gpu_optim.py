"""The optimizer wrapper on a small model: three steps of ``Muon`` over a
model with embeddings, a Muon-Split attention matrix, MLP weights, a 3-D
weight, biases and a LayerNorm, against the fp64 oracle step by step (the
oracle takes each step from the parameter the GPU held before it): Muon
parameters to the bf16 cell bound, AdamW parameters to the oracle's AdamW
within the bf16 rounding of three stores."""
import numpy as np
import pytest
import torch

import oracle
from _margins import record
from _parity import cell_err
from newton_schulz_orthogonalized_muon_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_BF16, TOL_EXACT = 2e-2, 1e-6


def _model():
    shapes = {"embed_tokens.weight": (64, 96), "attn.qkv.weight": (3 * 96, 96), "mlp.up.weight": (384, 96),
              "mlp.up.bias": (384,), "mlp.down.weight": (96, 384), "conv.weight": (48, 8, 3, 3),
              "norm.weight": (96,), "lm_head.weight": (64, 96)}
    params = {}
    for i, (n, s) in enumerate(shapes.items()):
        t = torch.tensor(wl.weight(800 + i, s)).to(torch.bfloat16).cuda()
        params[n] = t.requires_grad_(True)
    return params


def test_muon_optimizer_three_steps_against_the_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    torch.cuda.set_device(0)
    params = _model()
    opt = pkg.Muon(params.items(), lr=0.02, wd=0.1, adamw_lr=3e-4, higher_rank=True,
                   split_heads={"attn.qkv.weight": 3})
    muon_names = [e.name for e in opt.muon]
    assert muon_names == ["attn.qkv.weight", "mlp.up.weight", "mlp.down.weight", "conv.weight"]
    assert opt.adamw_names == ["embed_tokens.weight", "mlp.up.bias", "norm.weight", "lm_head.weight"]
    mom = {n: np.zeros((params[n].shape[0], params[n].numel() // params[n].shape[0])) for n in muon_names}
    adam = {n: (np.zeros(params[n].shape), np.zeros(params[n].shape)) for n in opt.adamw_names}
    for k in range(3):
        before = {n: p.detach().double().cpu().numpy() for n, p in params.items()}
        for i, (n, p) in enumerate(params.items()):
            g = wl.lowrank_grad(900 + 10 * k + i, p.shape[0], p.numel() // p.shape[0], 8) if p.dim() > 1 \
                else wl.gaussian(900 + 10 * k + i, p.shape, 1e-3)
            p.grad = torch.tensor(g).reshape(p.shape).to(torch.bfloat16).cuda()
        grads = {n: p.grad.double().cpu().numpy() for n, p in params.items()}
        opt.step()
        torch.cuda.synchronize()
        assert opt.handle is None and pkg.default_handle().check() == 0
        for n in muon_names:
            heads = 3 if n == "attn.qkv.weight" else 1
            w_ref, mom[n] = oracle.muon_step(before[n], grads[n], mom[n], lr=0.02, wd=0.1, split_heads=heads)
            got = params[n].detach().double().cpu().numpy()
            err = record(f"Muon optimizer step {k} {n} (cell bound)", cell_err(got, w_ref, before[n] * 0.998), TOL_BF16)
            assert err < TOL_BF16, (k, n, err)
        for n in opt.adamw_names:
            m, v = adam[n]
            p_ref, m, v = oracle.adamw_step(before[n], grads[n], m, v, k + 1, lr=3e-4, beta1=0.9, beta2=0.95,
                                            eps=1e-8, wd=0.1)
            adam[n] = (m, v)
            got = params[n].detach().double().cpu().numpy()
            ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(p_ref), 1e-30))) - 7)
            assert np.all(np.abs(got - p_ref) <= 0.5 * ulp + TOL_EXACT * np.abs(p_ref) + 1e-12), (k, n)
        opt.zero_grad()
    # the optimizer's momenta equal the oracle's
    for i, n in enumerate(muon_names):
        assert np.linalg.norm(opt.momenta[i].double().cpu().numpy() - mom[n]) <= TOL_EXACT * np.linalg.norm(mom[n])


def test_muon_optimizer_state_dict_resumes_bit_for_bit():
    # two steps, save, a fresh optimizer loads the state, one more step:
    # parameters equal three uninterrupted steps bit for bit
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    torch.cuda.set_device(0)

    def grads(params, k):
        for i, (n, p) in enumerate(params.items()):
            g = wl.gaussian(1000 + 10 * k + i, p.shape, 1e-2)
            p.grad = torch.tensor(g).to(torch.bfloat16).cuda()

    runs = []
    for resume in (False, True):
        params = _model()
        kw = dict(lr=0.02, wd=0.1, adamw_lr=3e-4, higher_rank=True, split_heads={"attn.qkv.weight": 3})
        opt = pkg.Muon(params.items(), **kw)
        for k in range(3):
            if resume and k == 2:
                state = opt.state_dict()
                opt = pkg.Muon(params.items(), **dict(kw, lr=1.0))   # hyper-parameters come from the state
                opt.load_state_dict(state)
            grads(params, k)
            loss = opt.step(closure=lambda: torch.zeros(()))
            assert float(loss) == 0.0
            opt.zero_grad()
        torch.cuda.synchronize()
        runs.append({n: p.detach().cpu() for n, p in params.items()})
    for n in runs[0]:
        assert torch.equal(runs[0][n], runs[1][n]), n
