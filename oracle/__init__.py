"""Oracle for the Muon step: plain float64 CPU code (NumPy, and a plain-C
cross-check).  TEST INFRASTRUCTURE ONLY — imported by ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg, never by the
library.  It shares no code with the CUDA path."""
from .muon_ref import (  # noqa: F401
    DEFAULT_GAMMA, DEFAULT_LR, DEFAULT_MU, DEFAULT_WD, FAST_COEFFS, HYBRID_STAGES,
    SCALE_NONE, SCALE_SPECTRAL, SCALE_UNIT_RMS_NORM, STABLE_COEFFS, MuonHyper,
    bias_correct, decoupled_update, expand_stages, frobenius_normalize, group_by_shape,
    head_slices, lookahead_ema, lookahead_sgd, momentum_ema, momentum_sgd, muon_step,
    newton_schulz, newton_schulz_literal, ns_iteration, row_blocks, update_scale,
)
