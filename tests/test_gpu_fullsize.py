"""Full-size parity in the benchmark's launch configuration.

One Muon step over the whole Llama-3-8B-shaped set (32 layers, 224 matrices,
6.98e9 parameters, bf16) with the same inputs, grouping and workspace limit
that bench.py times; a few whole matrices (one per shape group, including a
transposed one) are copied back and checked against the fp64 oracle run on
their host copies.  The Moonlight-like MoE set (experts + Muon-Split heads)
is checked the same way on one expert and one split attention matrix.
"""
import numpy as np
import pytest
import torch

import bench
import oracle

pytestmark = pytest.mark.gpu

TOL_BF16, TOL_EXACT = 2e-2, 1e-6


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _budget(w):
    w = np.abs(w)
    return float(np.linalg.norm(0.5 * np.exp2(np.floor(np.log2(np.maximum(w, 1e-30))) - 7)))


def _run_and_check(name, picks, layers=None, workspace_gb=64.0):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ws = bench.weight_set(name, layers)
    specs, _ = bench.owned_specs(ws, 1, 0)
    W, G, M = bench.make_inputs(specs, dev, 0)
    idx = [next(i for i, s in enumerate(specs) if s.name.endswith(p)) for p in picks]
    host = {i: (W[i].double().cpu().numpy(), G[i].double().cpu().numpy()) for i in idx}
    h = pkg.default_handle(0)
    h.set_workspace_limit(int(workspace_gb * (1 << 30)))
    pkg.muon_step(W, G, M, lr=bench.LR, wd=bench.WD, mu=bench.MU, nesterov=True, ns_steps=bench.NS_STEPS,
                  split_heads=[s.split_heads for s in specs], handle=h)
    assert h.check() == 0
    for i in idx:
        w0, g = host[i]
        w_ref, m_ref = oracle.muon_step(w0, g, np.zeros_like(g), lr=bench.LR, wd=bench.WD, mu=bench.MU,
                                        nesterov=True, split_heads=specs[i].split_heads)
        w_gpu = W[i].double().cpu().numpy()
        base = w0 * (1 - bench.LR * bench.WD)
        err = (np.linalg.norm(w_gpu - w_ref) - _budget(w_ref)) / np.linalg.norm(w_ref - base)
        assert err < TOL_BF16, (specs[i].name, err)
        assert _rel(M[i].double().cpu().numpy(), m_ref) < TOL_EXACT
    del W, G, M
    torch.cuda.empty_cache()


def test_llama3_8b_full_set_sampled():
    _run_and_check("llama3-8b", ["layers.0.attn.k_proj.weight", "layers.17.attn.q_proj.weight",
                                 "layers.31.mlp.up_proj.weight"])


def test_moonlight_moe_full_set_sampled():
    _run_and_check("moonlight-moe", ["layers.26.experts.63.down_proj.weight", "layers.5.attn.v_proj.weight"])


def test_gpt2_small_three_steps_with_adamw():
    """The whole GPT-2-small-shaped set: 48 Muon matrices (bf16, grads
    scaled 1e-3) and 98 LayerNorm/bias vectors on AdamW, three consecutive
    steps, every tensor checked against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    from newton_schulz_orthogonalized_muon_gb300 import workloads as wl
    ws = wl.gpt2_small()
    lr, wd, lr_adam = 0.02, 0.1, 3e-4
    Wd = [torch.tensor(wl.weight(10 + i, s.shape)).to(torch.bfloat16).cuda() for i, s in enumerate(ws.muon)]
    Md = [torch.zeros(s.shape, device="cuda") for s in ws.muon]
    W_ref = [w.double().cpu().numpy() for w in Wd]
    W0 = [w.copy() for w in W_ref]
    M_ref = [np.zeros(s.shape) for s in ws.muon]
    Pd = [torch.tensor(wl.weight(900 + i, s.shape)).to(torch.bfloat16).cuda() for i, s in enumerate(ws.adamw)]
    Ad = [torch.zeros(s.shape, device="cuda") for s in ws.adamw]
    Vd = [torch.zeros(s.shape, device="cuda") for s in ws.adamw]
    P_ref = [(p.double().cpu().numpy(), np.zeros(s.shape), np.zeros(s.shape)) for p, s in zip(Pd, ws.adamw)]
    for t in range(1, 4):
        G = [torch.tensor(wl.lowrank_grad(1000 * t + i, s.shape[0], s.shape[1], 64, scale=ws.grad_scale))
             .to(torch.bfloat16).cuda() for i, s in enumerate(ws.muon)]
        Ga = [torch.tensor(wl.gaussian(5000 * t + i, s.shape, 1e-3)).to(torch.bfloat16).cuda()
              for i, s in enumerate(ws.adamw)]
        pkg.muon_step(Wd, G, Md, lr=lr, wd=wd, mu=0.95, nesterov=True)
        pkg.adamw_step(Pd, Ga, Ad, Vd, step=t, lr=lr_adam, beta1=0.9, beta2=0.95, eps=1e-8, wd=wd)
        for i in range(len(ws.muon)):
            W_ref[i], M_ref[i] = oracle.muon_step(W_ref[i], G[i].double().cpu().numpy(), M_ref[i], lr=lr, wd=wd)
        P_ref = [oracle.adamw_step(p, g.double().cpu().numpy(), m, v, t, lr=lr_adam, beta1=0.9, beta2=0.95,
                                   eps=1e-8, wd=wd) for (p, m, v), g in zip(P_ref, Ga)]
    assert pkg.default_handle().check() == 0
    for i in range(len(ws.muon)):
        base = W0[i] * (1 - lr * wd) ** 3
        w_gpu = Wd[i].double().cpu().numpy()
        err = (np.linalg.norm(w_gpu - W_ref[i]) - 3 * _budget(W_ref[i])) / np.linalg.norm(W_ref[i] - base)
        assert err < TOL_BF16, (ws.muon[i].name, err)
        assert _rel(Md[i].double().cpu().numpy(), M_ref[i]) < TOL_EXACT
    for (p, m, v), pd, md, vd in zip(P_ref, Pd, Ad, Vd):
        assert _rel(md.double().cpu().numpy(), m) < TOL_EXACT
        assert _rel(vd.double().cpu().numpy(), v) < TOL_EXACT
        assert np.linalg.norm(pd.double().cpu().numpy() - p) <= 3 * _budget(p) + TOL_EXACT * np.linalg.norm(p)
