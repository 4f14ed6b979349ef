"""Tolerances shared by the CPU calibration and the GPU parity tests (no torch, no GPU)."""
import numpy as np

# Regression guard on the relative error of every output row (the contract is the
# max-abs tolerance; this catches what max-abs cannot see at long contexts).
# Calibrated in tests/test_parity_power.py: honest bf16 results stay below a third
# of it, a dropped 64-row tile or a split merged twice lands above twice it.
REL_GUARD = 1e-2


def rel_err(got, ref):
    """Largest over rows (the last axis is the head dimension) of ||got - ref|| / ||ref||."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.linalg.norm((got - ref).reshape(-1, ref.shape[-1]), axis=-1)
    den = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=-1)
    return float((num / np.maximum(den, 1e-300)).max())
