"""Error metrics used by the parity tests.

The block's outputs and gradients (Y, dX, dW_gu, dW_down, and the stage outputs
H, GU and O) must satisfy, per tensor:
  normwise   ||gpu - ref||_F / ||ref||_F <= 2e-2
  elementwise max_i |gpu_i - ref_i| / max(|ref_i|, rms(ref)) <= 5e-2,
              rms(ref) = ||ref||_F / sqrt(n).
Each element's error is normalised by its own magnitude, floored at the tensor's
rms: a single bf16 rounding (relative 2^-9) can never break the element bound, a
wrong term or index does. Normalising every element by rms alone fails on
heavy-tailed tensors (a skewed expert load makes dW mostly zeros plus a few large
experts) from output rounding alone.
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
    scale = np.maximum(np.abs(ref), rms)
    return float(np.linalg.norm(diff) / nref), float((np.abs(diff) / scale).max(initial=0.0))


def assert_close(got, ref, name: str = "", norm_rel: float = NORM_REL,
                 max_rel_rms: float = MAX_REL_RMS) -> tuple[float, float]:
    nr, mr = errors(got, ref)
    assert nr <= norm_rel and mr <= max_rel_rms, (
        f"{name}: normwise rel {nr:.3e} (limit {norm_rel}), elementwise {mr:.3e} (limit {max_rel_rms})")
    return nr, mr
