"""The other schedules of the same arithmetic, against the serial one bit
for bit (parameters and momenta, two steps).

* Overlapped (MUON_OVERLAP=1): each unit's preparation (momentum, Nesterov,
  norm partials, the master's planes) runs on the handle's side stream while
  the previous unit's products run, the two units using the two halves of
  the workspace; the cases force several chunks per group (a small
  workspace limit) and several groups, so that a unit's half is reused.
* Concurrent groups (the default for small sets, MUON_CONCURRENT=1 forces
  it): every same-shape group on a stream of its own, the regions side by
  side; bf16 parameters (tensor-core path) and fp32 parameters (the fp32
  tensor-core path), and a workspace limit too small for the side-by-side
  layout, which falls back to the serial order."""
import os

import pytest
import torch

from newton_schulz_orthogonalized_muon_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("limit_mb", [8, 64, 4096])
def test_overlapped_schedule_matches_serial_bitwise(limit_mb):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    torch.cuda.set_device(0)
    serial, ovl = _handle(pkg, MUON_CONCURRENT="0"), _handle(pkg, MUON_OVERLAP="1")
    specs = [wl.ParamSpec("a", (512, 1536)), wl.ParamSpec("b", (1536, 512)), wl.ParamSpec("c", (256, 768)),
             wl.ParamSpec("d", (1408, 2048)), wl.ParamSpec("q", (512, 512), split_heads=4),
             wl.ParamSpec("e", (512, 1536)), wl.ParamSpec("f", (96, 200))]
    W0 = [torch.tensor(wl.weight(600 + i, s.shape)).to(torch.bfloat16) for i, s in enumerate(specs)]
    G = [[torch.tensor(wl.lowrank_grad(700 + 10 * k + i, s.shape[0], s.shape[1], 32)).to(torch.bfloat16).cuda()
          for i, s in enumerate(specs)] for k in range(2)]
    outs = []
    for h in (serial, ovl):
        h.set_workspace_limit(limit_mb << 20)
        W = [w.clone().cuda() for w in W0]
        M = [torch.zeros(s.shape, device="cuda") for s in specs]
        for k in range(2):
            pkg.muon_step(W, G[k], M, lr=0.02, wd=0.1, split_heads=[s.split_heads for s in specs], handle=h)
        torch.cuda.synchronize()
        assert h.check() == 0
        outs.append(([w.cpu() for w in W], [m.cpu() for m in M]))
    for a, b in zip(outs[0][0] + outs[0][1], outs[1][0] + outs[1][1]):
        assert torch.equal(a, b)


def _set(dtype):
    specs = [wl.ParamSpec("a", (512, 1536)), wl.ParamSpec("b", (1536, 512)), wl.ParamSpec("c", (256, 768)),
             wl.ParamSpec("d", (704, 1024)), wl.ParamSpec("q", (512, 512), split_heads=4),
             wl.ParamSpec("e", (512, 1536)), wl.ParamSpec("f", (96, 200)), wl.ParamSpec("g", (768, 768))]
    W0 = [torch.tensor(wl.weight(900 + i, s.shape)).to(dtype) for i, s in enumerate(specs)]
    G = [[torch.tensor(wl.lowrank_grad(950 + 10 * k + i, s.shape[0], s.shape[1], 32)).to(dtype).cuda()
          for i, s in enumerate(specs)] for k in range(2)]
    return specs, W0, G


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("limit_mb", [2, 4096])
def test_concurrent_groups_match_serial_bitwise(dtype, limit_mb):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    torch.cuda.set_device(0)
    serial, conc = _handle(pkg, MUON_CONCURRENT="0"), _handle(pkg, MUON_CONCURRENT="1")
    specs, W0, G = _set(dtype)
    split = [s.split_heads for s in specs]
    outs = []
    for h in (serial, conc):
        h.set_workspace_limit(limit_mb << 20)
        W = [w.clone().cuda() for w in W0]
        M = [torch.zeros(s.shape, device="cuda") for s in specs]
        for k in range(2):
            pkg.muon_step(W, G[k], M, lr=0.02, wd=0.1, split_heads=split, handle=h)
        torch.cuda.synchronize()
        assert h.check() == 0
        outs.append(([w.cpu() for w in W], [m.cpu() for m in M]))
    for a, b in zip(outs[0][0] + outs[0][1], outs[1][0] + outs[1][1]):
        assert torch.equal(a, b)
    # the size the concurrent handle plans is what its step allocated
    shapes = [s.shape for s in specs]
    need = pkg.workspace_size(shapes, split_heads=split, ns_dtype=dtype, handle=conc)
    assert need > 0
    if limit_mb == 4096:                 # regions side by side
        assert need > pkg.workspace_size(shapes, split_heads=split, ns_dtype=dtype, handle=serial)



@pytest.mark.parametrize("limit_mb", [2, 4096])
def test_auto_method_matches_the_two_methods_bitwise(limit_mb):
    # ns_method="auto": the wide groups (n >= 4m) take the Gram method and
    # the others the standard one; each must equal a call with that method
    # alone bit for bit, and the workspace planned for auto covers both
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    torch.cuda.set_device(0)
    h = pkg.MuonHandle(0)
    h.set_workspace_limit(limit_mb << 20)
    wide = [wl.ParamSpec("w1", (256, 1024)), wl.ParamSpec("w2", (1536, 384)), wl.ParamSpec("w3", (128, 1024))]
    square = [wl.ParamSpec("s1", (512, 1024)), wl.ParamSpec("s2", (384, 384)), wl.ParamSpec("s3", (700, 1400))]
    specs = wide + square
    W0 = [torch.tensor(wl.weight(1200 + i, s.shape)).to(torch.bfloat16) for i, s in enumerate(specs)]
    G = [torch.tensor(wl.lowrank_grad(1300 + i, s.shape[0], s.shape[1], 16)).to(torch.bfloat16).cuda()
         for i, s in enumerate(specs)]

    def run(idx, method):
        W = [W0[i].clone().cuda() for i in idx]
        M = [torch.zeros(specs[i].shape, device="cuda") for i in idx]
        pkg.muon_step(W, [G[i] for i in idx], M, lr=0.02, wd=0.1, ns_method=method, handle=h)
        torch.cuda.synchronize()
        assert h.check() == 0
        return [w.cpu() for w in W], [m.cpu() for m in M]

    n_w = len(wide)
    w_all, m_all = run(list(range(len(specs))), "auto")
    w_g, m_g = run(list(range(n_w)), "gram")
    w_s, m_s = run(list(range(n_w, len(specs))), "standard")
    for a, b in zip(w_all + m_all, w_g + w_s + m_g + m_s):
        assert torch.equal(a, b)
    shapes = [s.shape for s in specs]
    need = pkg.workspace_size(shapes, ns_method="auto", handle=h)
    assert need == max(pkg.workspace_size([s.shape for s in wide], ns_method="gram", handle=h),
                       pkg.workspace_size([s.shape for s in square], ns_method="standard", handle=h))
