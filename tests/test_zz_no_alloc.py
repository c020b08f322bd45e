"""The allocation-free entry point, muon_orthogonalize_noalloc.

Callers that cannot allocate device memory (inside an allocation-free graph
capture, under a fixed memory budget, or behind a custom allocator) use this
entry point: it runs the same kernels as muon_orthogonalize but takes all its
scratch from a static array inside the library.  The test calls it through
the C ABI twice in a row, on two different matrices, and checks each result
against the handle-based muon_orthogonalize within the parity tolerances
used by the other GPU tests (bf16 2e-2, fp32 1e-4).  This file is collected
last so that a failure here never hides another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

from newton_schulz_orthogonalized_muon_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, 2e-2), (torch.float32, 1e-4)])
def test_noalloc_matches_handle_path_twice(dtype, tol):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    lib = pkg.load_library()
    torch.cuda.set_device(0)
    code = 1 if dtype == torch.bfloat16 else 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, shape in enumerate([(256, 1024), (700, 300)]):
        X = torch.tensor(wl.lowrank_grad(60 + call, shape[0], shape[1], 32)).to(dtype).cuda()
        ref = X.clone()
        pkg.muon_orthogonalize(ref)                     # existing entry point (handle workspace)
        st = lib.muon_orthogonalize_noalloc(ctypes.c_void_p(X.data_ptr()), code, shape[0], shape[1], 5, None, stream)
        assert st == 0
        torch.cuda.synchronize()
        assert _rel(X, ref) < tol, (call, shape)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    lib = pkg.load_library()
    X = torch.zeros(2048, 2048, dtype=torch.bfloat16, device="cuda")
    assert lib.muon_orthogonalize_noalloc(ctypes.c_void_p(X.data_ptr()), 1, 2048, 2048, 5, None, None) == 1
    assert lib.muon_orthogonalize_noalloc(ctypes.c_void_p(X.data_ptr()), 1, 1, 2 ** 21, 5, None, None) == 1
