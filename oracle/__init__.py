"""fp64 CPU oracle for the Muon step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package; the product path never does.
"""
from .muon_oracle import *  # noqa: F401,F403
from .muon_oracle import (QUINTIC, NS_STEPS, NORM_EPS, UPDATE_RMS, is_muon_param,
                          momentum_update, frobenius_normalize, newton_schulz,
                          gram_newton_schulz, orthogonalize, update_scale, apply_update,
                          orthogonalize_split, muon_step, adamw_step)
