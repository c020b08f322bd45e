"""GB300-native (sm_103a) Muon optimizer step.

The compute runs in ``libmuon_gb300.so`` (hand-written CUDA: tcgen05/TMA/TMEM
Newton-Schulz GEMMs, fused momentum/norm and AdamW kernels) behind the C ABI
in ``include/muon.h``.  This package is a thin ctypes binding over it; the
binding is loaded on first use and raises if the library was not built.
"""
__version__ = "1.0.0"

_BINDING_NAMES = ("MuonHandle", "MuonError", "muon_orthogonalize", "muon_orthogonalize_noalloc", "noalloc_check", "muon_step", "adamw_step",
                  "workspace_size", "default_handle", "MUON_SCALE_RMS", "MUON_SCALE_MUP",
                  "load_library", "selftest_timeout", "MUON_F32", "MUON_BF16", "MUON_NS_STANDARD", "MUON_NS_GRAM",
                  "MUON_NS_AUTO",
                  "QUINTIC", "EXPORTS")


_OPTIM_NAMES = ("Muon", "split_params", "takes_muon")


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import _binding
        return getattr(_binding, name)
    if name in _OPTIM_NAMES:
        from . import optim
        return getattr(optim, name)
    raise AttributeError(name)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library in-tree for sm_103a; returns its path."""
    from ._build import build as _b
    return _b(force=force, verbose=verbose)
