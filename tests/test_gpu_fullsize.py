"""Full-size parity in the benchmark's launch configuration.

One Muon step over the whole Llama-3-8B-shaped set (32 layers, 224 matrices,
6.98e9 parameters, bf16) with the same inputs, grouping and workspace limit
that bench.py times; a few whole matrices (one per shape group, including a
transposed one) are copied back and checked against the fp64 oracle run on
their host copies.  The Moonlight-like MoE set (experts + Muon-Split heads)
is checked the same way on one expert and one split attention matrix.  The
Llama set is also stepped with the Gram method (its own oracle) and the
Gram method orthogonalises batches of the set's 4096 x 4096 and
4096 x 14336 shapes at full size.  A bf16 parameter is held to the exact
lower bound on the update's error before its one bf16 rounding
(tests/_parity.py).
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from _margins import record
from _parity import cell_err

pytestmark = pytest.mark.gpu

TOL_BF16, TOL_EXACT = 2e-2, 1e-6


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _budget(w):
    w = np.abs(w)
    return float(np.linalg.norm(0.5 * np.exp2(np.floor(np.log2(np.maximum(w, 1e-30))) - 7)))


def _run_and_check(name, picks, layers=None, workspace_gb=64.0, method="standard"):
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
                  split_heads=[s.split_heads for s in specs], ns_method=method, handle=h)
    assert h.check() == 0
    for i in idx:
        w0, g = host[i]
        w_ref, m_ref = oracle.muon_step(w0, g, np.zeros_like(g), lr=bench.LR, wd=bench.WD, mu=bench.MU,
                                        nesterov=True, split_heads=specs[i].split_heads, method=method)
        w_gpu = W[i].double().cpu().numpy()
        base = w0 * (1 - bench.LR * bench.WD)
        err = record(f"{name} full set {method}: {specs[i].name} (cell bound)", cell_err(w_gpu, w_ref, base),
                     TOL_BF16)
        assert err < TOL_BF16, (specs[i].name, err)
        assert _rel(M[i].double().cpu().numpy(), m_ref) < TOL_EXACT
    del W, G, M
    torch.cuda.empty_cache()


def test_llama3_8b_full_set_sampled():
    _run_and_check("llama3-8b", ["layers.0.attn.k_proj.weight", "layers.17.attn.q_proj.weight",
                                 "layers.31.mlp.up_proj.weight"])


def test_llama3_8b_full_set_gram_sampled():
    # the Gram method over the whole set in the bench's configuration
    _run_and_check("llama3-8b", ["layers.3.attn.v_proj.weight", "layers.20.attn.o_proj.weight",
                                 "layers.31.mlp.down_proj.weight"], method="gram")


@pytest.mark.parametrize("m,n,batch", [(4096, 4096, 6), (4096, 14336, 4), (14336, 4096, 2)])
def test_gram_orthogonalize_at_llama_scale(m, n, batch):
    """Gram NS on batches of the Llama set's shapes (m = 4096 after the
    transpose rule), against the oracle's Gram method and the standard one
    (equal in exact arithmetic) on the first and last matrix."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    from newton_schulz_orthogonalized_muon_gb300 import workloads as wl
    torch.cuda.set_device(0)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(wl.matrix_seed(11, m * 7 + n))
    X = torch.stack([wl.lowrank_grad_device(gen, m, n, 64) for _ in range(batch)])
    picks = [0, batch - 1]
    inputs = {k: X[k].double().cpu().numpy() for k in picks}
    pkg.muon_orthogonalize(X, ns_method="gram")
    torch.cuda.synchronize()
    assert pkg.default_handle().check() == 0
    for k in picks:
        got = X[k].double().cpu().numpy()
        ref = oracle.gram_newton_schulz(inputs[k])
        err = record(f"gram orthogonalize {m}x{n} matrix {k}", _rel(got, ref), TOL_BF16)
        assert err < TOL_BF16, (m, n, k, err)
        if k == 0:
            std = oracle.newton_schulz(inputs[k])
            assert _rel(ref, std) < 1e-9          # the two oracles agree (exact arithmetic)
    del X
    torch.cuda.empty_cache()


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
        W_prev = [w.double().cpu().numpy() for w in Wd]
        pkg.muon_step(Wd, G, Md, lr=lr, wd=wd, mu=0.95, nesterov=True)
        pkg.adamw_step(Pd, Ga, Ad, Vd, step=t, lr=lr_adam, beta1=0.9, beta2=0.95, eps=1e-8, wd=wd)
        worst = (0.0, None)
        for i in range(len(ws.muon)):
            # the oracle takes this step from the parameter the GPU held before it
            w_ref, M_ref[i] = oracle.muon_step(W_prev[i], G[i].double().cpu().numpy(), M_ref[i], lr=lr, wd=wd)
            err = cell_err(Wd[i].double().cpu().numpy(), w_ref, W_prev[i] * (1 - lr * wd))
            assert err < TOL_BF16, (t, ws.muon[i].name, err)
            worst = max(worst, (err, ws.muon[i].name), key=lambda x: x[0])
        record(f"gpt2-small step {t}: worst of 48 matrices ({worst[1]}, cell bound)", worst[0], TOL_BF16)
        P_ref = [oracle.adamw_step(p, g.double().cpu().numpy(), m, v, t, lr=lr_adam, beta1=0.9, beta2=0.95,
                                   eps=1e-8, wd=wd) for (p, m, v), g in zip(P_ref, Ga)]
    assert pkg.default_handle().check() == 0
    for i in range(len(ws.muon)):
        assert _rel(Md[i].double().cpu().numpy(), M_ref[i]) < TOL_EXACT
    for (p, m, v), pd, md, vd in zip(P_ref, Pd, Ad, Vd):
        assert _rel(md.double().cpu().numpy(), m) < TOL_EXACT
        assert _rel(vd.double().cpu().numpy(), v) < TOL_EXACT
        assert np.linalg.norm(pd.double().cpu().numpy() - p) <= 3 * _budget(p) + TOL_EXACT * np.linalg.norm(p)
