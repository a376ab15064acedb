"""Error metrics used by the parity tests.

The block's outputs and gradients (Y, dX, dW_gu, dW_down, and the stage outputs
H, GU and O) must satisfy, per tensor:
  normwise   ||gpu - ref||_F / ||ref||_F <= 2e-2
  elementwise max_i |gpu_i - ref_i| / rms(ref) <= 5e-2,
              rms(ref) = ||ref||_F / sqrt(n),
i.e. no element's error exceeds 5e-2 once the tensor is normalised to unit rms.
The expert weight gradients dW_gu and dW_down are E independent matrices whose
scales follow each expert's load (a skewed load gives one expert every token and
leaves others empty), so they are checked expert by expert (assert_close_experts):
each non-empty expert's slice against the bound with its own rms, each empty
expert's slice exactly zero. The router-logit gradient is sparse: a token's row is
nonzero only at its k chosen experts, so it is checked on those entries
(assert_close_selected: the bounds with the norm and rms taken over the chosen
entries) and must be exactly zero elsewhere.

Setting MOE_PARITY_LOG=<file> appends every checked error to that file, with the
element error also normalised by max(|ref_i|, rms) for comparison.
"""
import os

import numpy as np

NORM_REL = 2e-2
MAX_REL_RMS = 5e-2
# routing weights: fp32 exp, an fp32 sum of k terms and one fp32 divide against the
# fp64 value; each step is a few ulps of 2^-24, so 2e-6 relative is a safe bound.
W_REL = 2e-6


def errors(got, ref) -> tuple[float, float]:
    """(normwise relative error, largest element error / rms(ref))."""
    nr, mr, _ = _errors3(got, ref)
    return nr, mr


def _errors3(got, ref) -> tuple[float, float, float]:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    diff = got - ref
    nref = np.linalg.norm(ref)
    if nref == 0.0:
        m = float(np.abs(diff).max(initial=0.0))
        return float(np.linalg.norm(diff)), m, m
    rms = nref / np.sqrt(ref.size)
    ad = np.abs(diff)
    per_elem = float((ad / np.maximum(np.abs(ref), rms)).max(initial=0.0))
    return float(np.linalg.norm(diff) / nref), float(ad.max(initial=0.0) / rms), per_elem


def assert_close(got, ref, name: str = "", norm_rel: float = NORM_REL,
                 max_rel_rms: float = MAX_REL_RMS) -> tuple[float, float]:
    nr, mr, pe = _errors3(got, ref)
    log = os.environ.get("MOE_PARITY_LOG")
    if log:
        with open(log, "a") as fh:
            fh.write(f"{os.environ.get('PYTEST_CURRENT_TEST', '?').split(' ')[0]}\t{name}\t"
                     f"normwise={nr:.3e}\tmax/rms={mr:.3e}\tmax/max(|ref|,rms)={pe:.3e}\n")
    assert nr <= norm_rel and mr <= max_rel_rms, (
        f"{name}: normwise rel {nr:.3e} (limit {norm_rel}), elementwise {mr:.3e} (limit {max_rel_rms})")
    return nr, mr


def assert_close_experts(got, ref, name: str = "", element_floor: str = "rms") -> None:
    """Per-expert check of a [E, ...] weight gradient (see the module docstring).
    element_floor="ref" normalises each element's error by max(|ref_i|, rms) instead
    of rms: only for the cases whose exact result bf16 cannot hold within the rms
    element bound (listed with the evidence where it is used)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    worst = (0.0, 0.0)
    for e in range(ref.shape[0]):
        if not ref[e].any():
            assert not got[e].any(), f"{name}[{e}]: an expert without tokens must get zeros"
            continue
        nr, mr, pe = _errors3(got[e], ref[e])
        if element_floor == "ref":
            mr = pe
        worst = (max(worst[0], nr), max(worst[1], mr))
        assert nr <= NORM_REL and mr <= MAX_REL_RMS, (
            f"{name}[{e}]: normwise rel {nr:.3e} (limit {NORM_REL}), elementwise {mr:.3e} "
            f"(limit {MAX_REL_RMS})")
    log = os.environ.get("MOE_PARITY_LOG")
    if log:
        with open(log, "a") as fh:
            fh.write(f"{os.environ.get('PYTEST_CURRENT_TEST', '?').split(' ')[0]}\t{name} "
                     f"(worst expert)\tnormwise={worst[0]:.3e}\t"
                     f"{'max/rms' if element_floor == 'rms' else 'max/max(|ref|,rms)'}"
                     f"={worst[1]:.3e}\n")


def assert_close_selected(got, ref, selected, name: str = "") -> tuple[float, float]:
    """Check a gradient that is nonzero only where `selected` (see the module docstring):
    exactly zero elsewhere, the bounds over the selected entries."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    selected = np.asarray(selected, dtype=bool)
    assert got.shape == ref.shape == selected.shape
    assert not got[~selected].any(), f"{name}: entries outside the selection must be zero"
    assert not ref[~selected].any(), f"{name}: the reference is nonzero outside the selection"
    return assert_close(got[selected], ref[selected], name + " (chosen experts)")

