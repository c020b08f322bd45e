"""Wide-matrix sweep at full size: batches of 64 Gaussian bf16 matrices for
m in {256, 1024, 2048} and n in {4096, 16384}, orthogonalised with the
standard and the Gram method in one batched call each; two sampled matrices
per shape are checked against the fp64 oracle (which equals the SVD closed
form of the quintic, see tests/test_oracle_pins.py)."""
import numpy as np
import pytest
import torch

import oracle
from newton_schulz_orthogonalized_muon_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.mark.parametrize("m,n", wl.WIDE_SWEEP)
def test_wide_sweep_standard_and_gram(m, n):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    torch.cuda.set_device(0)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(wl.matrix_seed(7, m * 100000 + n))
    X = torch.randn(wl.WIDE_BATCH, m, n, generator=gen, device="cuda").to(torch.bfloat16)
    picks = [0, wl.WIDE_BATCH - 1]
    refs = {k: oracle.newton_schulz(X[k].double().cpu().numpy()) for k in picks}
    for method in ("standard", "gram"):
        Y = X.clone()
        pkg.muon_orthogonalize(Y, ns_method=method)
        torch.cuda.synchronize()
        assert pkg.default_handle().check() == 0
        for k in picks:
            got = Y[k].double().cpu().numpy()
            err = np.linalg.norm(got - refs[k]) / np.linalg.norm(refs[k])
            assert err < TOL_BF16, (method, m, n, k, err)
        del Y
    del X
    torch.cuda.empty_cache()
