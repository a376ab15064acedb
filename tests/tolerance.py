"""Error metrics used by the parity tests.

The block's outputs and gradients (Y, dX, dW_gu, dW_down, and the stage outputs
H and O) must satisfy, per tensor, ||gpu - ref||_F / ||ref||_F <= 2e-2 and
max|gpu - ref| / rms(ref) <= 5e-2, rms(ref) = ||ref||_F / sqrt(n): the bf16-input
bound for the block's floating-point results.
"""
import numpy as np

NORM_REL = 2e-2
MAX_REL_RMS = 5e-2
# routing weights: fp32 exp, an fp32 sum of k terms and one fp32 divide against the
# fp64 value; each step is a few ulps of 2^-24, so 2e-6 relative is a safe bound.
W_REL = 2e-6


def errors(got, ref) -> tuple[float, float]:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    diff = got - ref
    nref = np.linalg.norm(ref)
    if nref == 0.0:
        return float(np.linalg.norm(diff)), float(np.abs(diff).max(initial=0.0))
    rms = nref / np.sqrt(ref.size)
    return float(np.linalg.norm(diff) / nref), float(np.abs(diff).max(initial=0.0) / rms)


def assert_close(got, ref, name: str = "", norm_rel: float = NORM_REL,
                 max_rel_rms: float = MAX_REL_RMS) -> tuple[float, float]:
    nr, mr = errors(got, ref)
    assert nr <= norm_rel and mr <= max_rel_rms, (
        f"{name}: normwise rel {nr:.3e} (limit {norm_rel}), max/rms {mr:.3e} (limit {max_rel_rms})")
    return nr, mr
