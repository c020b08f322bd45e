"""CTA-pair tensor-core kernels (tcgen05 cta_group::2, 256 x 256 tiles).

A handle created with MUON_TC_PAIR_MIN_M=256 runs every product of a group
with m >= 256 on the pair kernels (UPDATE / FINAL when m is a multiple of
256 or m >= 2048); a handle created with MUON_TC_PAIR=0 runs the one-CTA
kernels.  Both are
compared with the fp64 oracle, and with each other, on the same inputs,
including ragged n, a ragged last 256-row tile (m = 2176), transposed
matrices and batches.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from newton_schulz_orthogonalized_muon_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.fixture(scope="module")
def handles():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    torch.cuda.set_device(0)
    # pairs from m = 256 (the default starts them at m = 1024, and at 256)
    old_min = os.environ.get("MUON_TC_PAIR_MIN_M")
    os.environ["MUON_TC_PAIR_MIN_M"] = "256"
    try:
        pair = pkg.MuonHandle(0)
    finally:
        if old_min is None:
            del os.environ["MUON_TC_PAIR_MIN_M"]
        else:
            os.environ["MUON_TC_PAIR_MIN_M"] = old_min
    old = os.environ.get("MUON_TC_PAIR")
    os.environ["MUON_TC_PAIR"] = "0"
    try:
        single = pkg.MuonHandle(0)
    finally:
        if old is None:
            del os.environ["MUON_TC_PAIR"]
        else:
            os.environ["MUON_TC_PAIR"] = old
    return pkg, pair, single


@pytest.mark.parametrize("shape", [(256, 1024), (512, 700), (768, 3072), (3072, 768), (2048, 2304), (512, 512),
                                   (2176, 2400)])
def test_pair_kernels_match_oracle_and_single(handles, shape):
    pkg, pair, single = handles
    X = wl.lowrank_grad(70, shape[0], shape[1], 64)
    t = torch.tensor(X).to(torch.bfloat16).cuda()
    ref = oracle.newton_schulz(t.double().cpu().numpy())
    a, b = t.clone(), t.clone()
    pkg.muon_orthogonalize(a, handle=pair)
    pkg.muon_orthogonalize(b, handle=single)
    torch.cuda.synchronize()
    assert pair.check() == 0 and single.check() == 0
    ga, gb = a.double().cpu().numpy(), b.double().cpu().numpy()
    assert _rel(ga, ref) < TOL_BF16
    assert _rel(gb, ref) < TOL_BF16
    assert _rel(ga, gb) < TOL_BF16


def test_pair_kernels_batched_step(handles):
    pkg, pair, _ = handles
    specs = [wl.ParamSpec("a", (512, 1536)), wl.ParamSpec("b", (1536, 512)), wl.ParamSpec("c", (512, 1536))]
    W = [torch.tensor(wl.weight(80 + i, s.shape)).to(torch.bfloat16).cuda() for i, s in enumerate(specs)]
    G = [torch.tensor(wl.lowrank_grad(90 + i, s.shape[0], s.shape[1], 64)).to(torch.bfloat16).cuda()
         for i, s in enumerate(specs)]
    M = [torch.zeros(s.shape, device="cuda") for s in specs]
    W0 = [w.double().cpu().numpy() for w in W]
    pkg.muon_step(W, G, M, lr=0.02, wd=0.1, handle=pair)
    assert pair.check() == 0
    for i in range(len(specs)):
        w_ref, _ = oracle.muon_step(W0[i], G[i].double().cpu().numpy(), np.zeros(specs[i].shape), lr=0.02, wd=0.1)
        base = W0[i] * (1 - 0.02 * 0.1)
        w = np.abs(w_ref)
        budget = float(np.linalg.norm(0.5 * np.exp2(np.floor(np.log2(np.maximum(w, 1e-30))) - 7)))
        err = (np.linalg.norm(W[i].double().cpu().numpy() - w_ref) - budget) / np.linalg.norm(w_ref - base)
        assert err < TOL_BF16


@pytest.mark.parametrize("shape", [(256, 2048), (512, 4100), (1024, 768), (256, 512), (2176, 2400)])
def test_pair_gram_matches_oracle_and_single(handles, shape):
    pkg, pair, single = handles
    rank = min(shape) if shape == (256, 512) else 64
    X = wl.lowrank_grad(71, shape[0], shape[1], rank)
    t = torch.tensor(X).to(torch.bfloat16).cuda()
    ref = oracle.gram_newton_schulz(t.double().cpu().numpy())
    a, b = t.clone(), t.clone()
    pkg.muon_orthogonalize(a, ns_method="gram", handle=pair)
    pkg.muon_orthogonalize(b, ns_method="gram", handle=single)
    torch.cuda.synchronize()
    assert pair.check() == 0 and single.check() == 0
    ga, gb = a.double().cpu().numpy(), b.double().cpu().numpy()
    assert _rel(ga, ref) < TOL_BF16
    assert _rel(gb, ref) < TOL_BF16
    assert _rel(ga, gb) < TOL_BF16


@pytest.fixture(scope="module")
def ragged_handle(handles):
    """A handle that runs the symmetric products of groups with m >= 1024 on
    pairs even when m is not a multiple of 256 (the last 256-row tile is
    ragged); the threshold is the default, set explicitly here."""
    pkg = handles[0]
    old = os.environ.get("MUON_TC_PAIR_MIN_M")
    os.environ["MUON_TC_PAIR_MIN_M"] = "1024"
    try:
        return pkg.MuonHandle(0)
    finally:
        if old is None:
            del os.environ["MUON_TC_PAIR_MIN_M"]
        else:
            os.environ["MUON_TC_PAIR_MIN_M"] = old


@pytest.mark.parametrize("shape", [(1408, 2048), (1152, 1600), (2048, 1408)])
def test_ragged_pair_tiles_match_oracle_and_single(handles, ragged_handle, shape):
    pkg, _, single = handles
    X = wl.lowrank_grad(72, shape[0], shape[1], 64)
    t = torch.tensor(X).to(torch.bfloat16).cuda()
    ref = oracle.newton_schulz(t.double().cpu().numpy())
    a, b = t.clone(), t.clone()
    pkg.muon_orthogonalize(a, handle=ragged_handle)
    pkg.muon_orthogonalize(b, handle=single)
    torch.cuda.synchronize()
    assert ragged_handle.check() == 0 and single.check() == 0
    ga, gb = a.double().cpu().numpy(), b.double().cpu().numpy()
    assert _rel(ga, ref) < TOL_BF16
    assert _rel(ga, gb) < TOL_BF16

