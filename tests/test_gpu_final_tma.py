"""FINAL through per-matrix tensor maps (FINAL_T, and G_FINAL_T for the Gram
method's last product) against the generic FINAL.

When every destination of a chunk is bf16 with a 16-byte aligned base and
row stride, the last update product loads each destination block by TMA
beside the master-X planes, applies W = alpha W + beta O in shared memory
and stores it back by TMA; otherwise (fp32, misaligned, odd row strides) the
destinations are read and written element-wise.  Both evaluate the same fp32
expression and round once to bf16, so their results must agree bit for bit;
a handle created with MUON_FINAL_TMA=0 always takes the generic path.
Shapes cover the CTA-pair and one-CTA kernels, transposed destinations,
ragged tiles, Muon-Split head blocks and alpha = 0 (orthogonalize in place).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from newton_schulz_orthogonalized_muon_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


def _handle(pkg, **env):
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        return pkg.MuonHandle(0)
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


@pytest.fixture(scope="module")
def handles():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    torch.cuda.set_device(0)
    return pkg, {
        # pairs from m = 256, so that the 512-row group runs on them too
        "pair": (_handle(pkg, MUON_TC_PAIR_MIN_M="256"), _handle(pkg, MUON_TC_PAIR_MIN_M="256", MUON_FINAL_TMA="0")),
        "single": (_handle(pkg, MUON_TC_PAIR="0"), _handle(pkg, MUON_TC_PAIR="0", MUON_FINAL_TMA="0")),
    }


SPECS = [
    ("a", (512, 1536), 1),
    ("b", (1536, 512), 1),      # transposed destination
    ("c", (2176, 2400), 1),     # ragged last 256-row tile
    ("d", (1408, 2048), 1),     # the MoE expert shape
    ("e", (2048, 1408), 1),     # its transposed partner, same group
    ("f", (256, 768), 2),       # two head blocks of 128 x 768
    ("g", (96, 200), 1),        # one ragged tile in both directions
    ("h", (300, 136), 1),       # transposed, ragged, n = 136 (stride 272 bytes)
]


def _inputs(seed):
    W = [torch.tensor(wl.weight(seed + i, s)).to(torch.bfloat16).cuda() for i, (_, s, _) in enumerate(SPECS)]
    G = [torch.tensor(wl.lowrank_grad(seed + 50 + i, s[0], s[1], 64)).to(torch.bfloat16).cuda()
         for i, (_, s, _) in enumerate(SPECS)]
    return W, G


@pytest.mark.parametrize("kernel,method", [("pair", "standard"), ("single", "standard"), ("pair", "gram")])
def test_final_tma_matches_generic_bitwise(handles, kernel, method):
    pkg, hs = handles
    h_tma, h_gen = hs[kernel]
    W, G = _inputs(300)
    split = [k for _, _, k in SPECS]
    outs = []
    for h in (h_tma, h_gen):
        w = [x.clone() for x in W]
        m = [torch.zeros(x.shape, device="cuda") for x in W]
        pkg.muon_step(w, G, m, lr=0.02, wd=0.1, split_heads=split, ns_method=method, handle=h)
        assert h.check() == 0
        outs.append(w)
    for (name, shape, _), a, b in zip(SPECS, outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name


def test_final_tma_matches_oracle(handles):
    pkg, hs = handles
    h = hs["pair"][0]
    W, G = _inputs(400)
    split = [k for _, _, k in SPECS]
    W0 = [w.double().cpu().numpy() for w in W]
    M = [torch.zeros(x.shape, device="cuda") for x in W]
    pkg.muon_step(W, G, M, lr=0.02, wd=0.1, split_heads=split, handle=h)
    assert h.check() == 0
    for i, (name, shape, heads) in enumerate(SPECS):
        w_ref, _ = oracle.muon_step(W0[i], G[i].double().cpu().numpy(), np.zeros(shape), lr=0.02, wd=0.1,
                                    split_heads=heads)
        base = W0[i] * (1 - 0.02 * 0.1)
        w = np.abs(w_ref)
        # one bf16 rounding of W itself is allowed on top of the NS tolerance
        budget = float(np.linalg.norm(0.5 * np.exp2(np.floor(np.log2(np.maximum(w, 1e-30))) - 7)))
        err = (np.linalg.norm(W[i].double().cpu().numpy() - w_ref) - budget) / np.linalg.norm(w_ref - base)
        assert err < TOL_BF16, name


def test_misaligned_destination_falls_back(handles):
    """A destination whose base is not 16-byte aligned takes the generic path
    for its whole chunk; the result is the same bits either way."""
    pkg, hs = handles
    h_tma, h_gen = hs["pair"]
    shape = (512, 1536)
    outs = []
    for h in (h_tma, h_gen):
        store = torch.zeros(2 * shape[0] * shape[1] + 8, dtype=torch.bfloat16, device="cuda")
        w_al = store[:shape[0] * shape[1]].view(shape)
        w_mis = store[shape[0] * shape[1] + 1:2 * shape[0] * shape[1] + 1].view(shape)   # 2-byte offset
        w_al.copy_(torch.tensor(wl.weight(500, shape)).to(torch.bfloat16))
        w_mis.copy_(torch.tensor(wl.weight(501, shape)).to(torch.bfloat16))
        G = [torch.tensor(wl.lowrank_grad(510 + i, shape[0], shape[1], 64)).to(torch.bfloat16).cuda() for i in range(2)]
        M = [torch.zeros(shape, device="cuda") for _ in range(2)]
        pkg.muon_step([w_al, w_mis], G, M, lr=0.02, wd=0.1, handle=h)
        assert h.check() == 0
        outs.append((w_al.clone(), w_mis.clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("shape,method", [((2048, 2304), "standard"), ((1408, 2048), "standard"),
                                          ((2048, 1408), "standard"), ((130, 512), "standard"),
                                          ((256, 4096), "gram"), ((1024, 700), "gram")])
def test_orthogonalize_in_place_matches_generic(handles, shape, method):
    """alpha = 0: the destination block is not read, only written."""
    pkg, hs = handles
    X = torch.tensor(wl.lowrank_grad(600, shape[0], shape[1], 64)).to(torch.bfloat16).cuda()
    outs = []
    for h in hs["pair"]:
        y = X.clone()
        pkg.muon_orthogonalize(y, ns_method=method, handle=h)
        assert h.check() == 0
        outs.append(y)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref = oracle.newton_schulz(X.double().cpu().numpy())
    got = outs[0].double().cpu().numpy()
    assert float(np.linalg.norm(got - ref) / np.linalg.norm(ref)) < TOL_BF16


def test_chunked_group_matches_one_chunk_bitwise(handles):
    """A workspace limit that splits a group into several chunks gives each
    chunk its own tensor-map array; the matrices are independent, so the
    result is the same bits as one chunk."""
    pkg, _ = handles
    shape, count = (512, 1536), 6
    W = [torch.tensor(wl.weight(700 + i, shape)).to(torch.bfloat16).cuda() for i in range(count)]
    G = [torch.tensor(wl.lowrank_grad(720 + i, shape[0], shape[1], 64)).to(torch.bfloat16).cuda() for i in range(count)]
    big, small = pkg.MuonHandle(0), pkg.MuonHandle(0)
    need = pkg.workspace_size([shape] * count, handle=small)
    small.set_workspace_limit(need // 3)
    assert pkg.workspace_size([shape] * count, handle=small) < need
    outs = []
    for h in (big, small):
        w = [x.clone() for x in W]
        m = [torch.zeros(shape, device="cuda") for _ in range(count)]
        pkg.muon_step(w, G, m, lr=0.02, wd=0.1, handle=h)
        assert h.check() == 0
        outs.append(w)
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
