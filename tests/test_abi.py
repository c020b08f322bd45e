"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every function include/muon.h declares, and rejects bad
arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "muon.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from newton_schulz_orthogonalized_muon_gb300 import _build
    if not os.path.exists(_build.LIB_PATH):
        _build.build()
    import newton_schulz_orthogonalized_muon_gb300 as pkg
    return pkg.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("muon_orthogonalize", "muon_step", "adamw_step", "muon_handle_create", "muon_handle_check"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_lists_every_declared_symbol():
    from newton_schulz_orthogonalized_muon_gb300 import _binding
    assert sorted(_binding.EXPORTS) == declared_functions()


def test_status_strings_and_version(lib):
    assert lib.muon_version() == 10000
    assert lib.muon_status_string(0) == b"ok"
    assert lib.muon_status_string(6) == b"device wait timed out"
    assert lib.muon_status_string(99) == b"unknown status"


def test_null_handle_is_rejected_without_a_device(lib):
    assert lib.muon_orthogonalize(None, None, 1, 1, 4, 4, 5, None, 0, None) == 1
    assert lib.muon_step(None, None, 0, 0.02, 0.1, 0.95, 1, 0, 5, None, 0.2, 1, None) == 1
    assert lib.muon_handle_check(None, None) == 1
    assert lib.muon_handle_destroy(None) == 0
    assert lib.muon_last_error(None) == b"null handle"
    assert lib.muon_handle_create(None, 0) == 1


def test_create_without_a_gb300_reports_unsupported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the gpu tests")
    h = ctypes.c_void_p()
    assert lib.muon_handle_create(ctypes.byref(h), 0) == 2
    assert not h.value


def test_param_struct_layout_matches_header():
    from newton_schulz_orthogonalized_muon_gb300._binding import MuonParamC
    # void* x3, int64 x2, int32 x4, int64
    assert ctypes.sizeof(MuonParamC) == 3 * 8 + 2 * 8 + 4 * 4 + 8
    assert MuonParamC.scale_dim.offset == 56


def test_struct_layouts_match_the_c_compiler(tmp_path):
    """sizeof / offsetof of the ABI structs as gcc lays them out from the
    header, against the ctypes mirrors the binding passes."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from newton_schulz_orthogonalized_muon_gb300._binding import MuonParamC, MuonStepOptionsC
    src = tmp_path / "layout.c"
    src.write_text(
        "#include <stdio.h>\n#include <stddef.h>\n#include \"muon.h\"\n"
        "int main(void) { printf(\"%zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(muon_param_t),"
        " offsetof(muon_param_t, scale_dim), sizeof(muon_step_options_t), offsetof(muon_step_options_t, coeffs),"
        " offsetof(muon_step_options_t, ns_dtype), offsetof(muon_step_options_t, update_rms),"
        " offsetof(muon_step_options_t, extra_scale)); printf(\"%zu\\n\", offsetof(muon_step_options_t, coeffs_per_step));"
        " return 0; }\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    want = [ctypes.sizeof(MuonParamC), MuonParamC.scale_dim.offset, ctypes.sizeof(MuonStepOptionsC),
            MuonStepOptionsC.coeffs.offset, MuonStepOptionsC.ns_dtype.offset, MuonStepOptionsC.update_rms.offset,
            MuonStepOptionsC.extra_scale.offset, MuonStepOptionsC.coeffs_per_step.offset]
    assert got == want


def test_workspace_size_rejects_a_null_handle(lib):
    out = ctypes.c_uint64(7)
    assert lib.muon_workspace_size(None, None, 0, 0, 5, 1, ctypes.byref(out)) == 1


def test_step_ex_rejects_bad_arguments_without_a_device(lib):
    from newton_schulz_orthogonalized_muon_gb300._binding import MuonStepOptionsC
    opts = MuonStepOptionsC(0.02, 0.1, 0.95, 1, 0, 5, None, 1, 0, 0.2, 1.0, 0)
    assert lib.muon_step_ex(None, None, 0, ctypes.byref(opts), None) == 1


def test_product_path_does_not_import_the_oracle():
    pkg_dir = os.path.join(ROOT, "newton_schulz_orthogonalized_muon_gb300")
    for dirpath, _, files in os.walk(pkg_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
