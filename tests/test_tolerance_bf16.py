"""What bf16 can hold within the parity bound (CPU only, no GPU).

The element bound of the parity tests is max_i |gpu_i - ref_i| / rms(ref) <= 5e-2.
For a weight gradient of an expert with few rows the exact result is heavy-tailed
(a sum of few products of near-Gaussian values), and an element 18x the rms sits so
high that rounding it to bf16 (relative 2^-9) alone uses most of the bound. These
tests pin that fact on the exact oracle result, and show that an implementation
whose rounding points are the block's (bf16 GEMM operands GU, G and dGU, fp32
accumulation, bf16 dW) misses the bound on those experts by itself: the cases the
GPU parity tests list as limited by bf16 (DW_BF16_LIMITED) are limited by the
arithmetic the method fixes, not by the kernels.
"""
import numpy as np
import torch

import oracle
import workloads
from tolerance import MAX_REL_RMS


def _bf16(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


def _case(T, d, E, k, f, seed, zipf):
    wl = workloads.Workload("t", T=T, d=d, E=E, k=k, f=f, seed=seed, backward=True,
                            zipf_bias=zipf)
    inp = workloads.make_inputs(wl)
    X, L = inp.x.double().numpy(), inp.logits.numpy()
    Wg, Wd, DY = inp.w_gu.double().numpy(), inp.w_down.double().numpy(), inp.dy.double().numpy()
    ref = oracle.forward(X, L, Wg, Wd, k)
    return wl, X, Wg, Wd, DY, ref, oracle.backward(DY, ref, Wg, Wd)


def _rms(a):
    return np.linalg.norm(a) / np.sqrt(a.size)


def test_rounding_the_exact_dw_to_bf16_uses_most_of_the_bound():
    # 96 tokens over 4 experts of 46-51 rows, d = f = 2880
    wl, *_, g = _case(96, 2880, 4, 2, 2880, 43, False)
    worst = 0.0
    for e in range(wl.E):
        ref = g["dw_gu"][e]
        worst = max(worst, np.abs(_bf16(ref) - ref).max() / _rms(ref))
    assert worst > 0.8 * MAX_REL_RMS          # 4.8e-2 of the 5e-2 budget


def test_rounding_the_exact_dw_down_to_bf16_breaks_the_bound():
    # skewed load: experts of 1-140 rows; one expert's dW_down cannot be held in bf16
    # within the rms element bound at all
    wl, *_, g = _case(512, 256, 32, 4, 256, 42, True)
    worst = 0.0
    for e in range(wl.E):
        ref = g["dw_down"][e]
        if ref.any():
            worst = max(worst, np.abs(_bf16(ref) - ref).max() / _rms(ref))
    assert worst > MAX_REL_RMS                # 6.2e-2


def test_bf16_rounding_points_alone_miss_the_rms_bound():
    """dW_gu[e] = Xp_e^T dGU_e with dGU formed from the bf16-saved gate/up values and
    the bf16 G = w dY, rounded to bf16 as the grouped GEMM's operand, and the result
    rounded to bf16: exact arithmetic otherwise. Expert 4 (140 rows) misses the bound."""
    wl, X, Wg, Wd, DY, ref, g = _case(512, 256, 32, 4, 256, 42, True)
    f, e = wl.f, 4
    r0, r1 = ref["offsets"][e], ref["offsets"][e + 1]
    toks = ref["tok_of"][r0:r1]
    slot = [list(ref["ids"][t]).index(e) for t in toks]
    w = ref["w"][toks, slot]
    xe = X[toks]
    gu = _bf16(xe @ Wg[e])
    dh = _bf16(w[:, None] * DY[toks]) @ Wd[e].T
    gg, uu = gu[:, :f], gu[:, f:]
    s = 1.0 / (1.0 + np.exp(-gg))
    dgu = _bf16(np.concatenate([dh * uu * s * (1 + gg * (1 - s)), dh * gg * s], axis=1))
    dw = _bf16(xe.T @ dgu)
    exact = g["dw_gu"][e]
    err = np.abs(dw - exact).max() / _rms(exact)
    assert err > MAX_REL_RMS                  # 5.85e-2: the value the kernel reaches too
    assert np.linalg.norm(dw - exact) / np.linalg.norm(exact) < 5e-3   # normwise is fine
