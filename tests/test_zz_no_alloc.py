"""The allocation-free entry point, muon_orthogonalize_noalloc.

Callers that cannot allocate device memory (inside an allocation-free graph
capture, under a fixed memory budget, or behind a custom allocator) use this
entry point: it runs the same kernels as muon_orthogonalize but takes all its
scratch from a static array inside the library.  The tests call it through
the C ABI twice in a row, on two different matrices, and check each result
against the handle-based muon_orthogonalize and against the fp64 oracle
within the parity tolerances used by the other GPU tests (bf16 2e-2, fp32
1e-4); they check that a NaN input is reported by muon_noalloc_check and
that the check clears the word.  This file is collected last so that a
failure here never hides another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from newton_schulz_orthogonalized_muon_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _host(t):
    return t.double().cpu().numpy()


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    torch.cuda.set_device(0)
    return pkg.load_library()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, 2e-2), (torch.float32, 1e-4)])
def test_noalloc_matches_handle_path_and_oracle_twice(lib, dtype, tol):
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    code = 1 if dtype == torch.bfloat16 else 0
    errs = []
    for call, shape in enumerate([(256, 1024), (700, 300)]):
        X = torch.tensor(wl.lowrank_grad(60 + call, shape[0], shape[1], 32)).to(dtype).cuda()
        ref64 = oracle.newton_schulz(_host(X))          # oracle on the same (rounded) input
        ref = X.clone()
        pkg.muon_orthogonalize(ref)                     # existing entry point (handle workspace)
        st = lib.muon_orthogonalize_noalloc(ctypes.c_void_p(X.data_ptr()), code, shape[0], shape[1], 5, None,
                                            _stream())
        assert st == 0
        assert lib.muon_noalloc_check(_stream()) == 0
        e_handle, e_oracle = _rel(_host(X), _host(ref)), _rel(_host(X), ref64)
        errs.append((shape, e_handle, e_oracle))
        assert e_handle < tol, (call, shape, e_handle)
        assert e_oracle < tol, (call, shape, e_oracle)
    print(f"noalloc {dtype}: (shape, rel err vs handle path, rel err vs fp64 oracle) = {errs}")


def test_noalloc_reports_a_nonfinite_input_and_clears_it(lib):
    X = torch.tensor(wl.lowrank_grad(70, 128, 512, 16)).to(torch.bfloat16).cuda()
    X[5, 7] = float("nan")
    assert lib.muon_orthogonalize_noalloc(ctypes.c_void_p(X.data_ptr()), 1, 128, 512, 5, None, _stream()) == 0
    assert lib.muon_noalloc_check(_stream()) == 5       # MUON_ERR_NONFINITE
    assert lib.muon_noalloc_check(_stream()) == 0       # read and cleared
    # a clean call afterwards reports nothing and still matches the oracle
    Y = torch.tensor(wl.lowrank_grad(71, 128, 512, 16)).to(torch.bfloat16).cuda()
    ref = oracle.newton_schulz(_host(Y))
    assert lib.muon_orthogonalize_noalloc(ctypes.c_void_p(Y.data_ptr()), 1, 128, 512, 5, None, _stream()) == 0
    assert lib.muon_noalloc_check(_stream()) == 0
    assert _rel(_host(Y), ref) < 2e-2


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    X = torch.zeros(2048, 2048, dtype=torch.bfloat16, device="cuda")
    assert lib.muon_orthogonalize_noalloc(ctypes.c_void_p(X.data_ptr()), 1, 2048, 2048, 5, None, None) == 1
    assert lib.muon_orthogonalize_noalloc(ctypes.c_void_p(X.data_ptr()), 1, 1, 2 ** 21, 5, None, None) == 1
    assert lib.muon_noalloc_set_timeout_ns(0) == 1
    assert lib.muon_noalloc_set_timeout_ns(4_000_000_000) == 0
