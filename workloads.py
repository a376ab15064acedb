"""Seeded synthetic inputs for the MoE expert block.

This module is shared by the CUDA path (tests, bench) and by the CPU oracle, and
therefore holds none of the block's arithmetic: it only draws random numbers,
rounds them to bf16 the way any bf16 input is rounded (round-to-nearest-even),
and describes the five workload shapes.

Shapes follow the pages' workloads (the gpt-oss-20b and Qwen3-30B-A3B models
trained in "Halo: Frontier-Lab Training for Everyone", section "Halo vs. stock
TRL", and in "Halo's 2.8x over TRL is not a kernel", section "Where the gap
actually is"), reduced to one MoE expert block. Values are synthetic; no
dataset or trained weight is involved.

Recipe (per seed, numpy PCG64, in this draw order): x ~ N(0,1) [T,d];
logits ~ N(0,1) [T,E] fp32; W_gu ~ N(0, 0.02^2) [E,d,2f]; W_down ~ N(0, 0.02^2)
[E,f,d]; dY ~ N(0,1) [T,d] (backward configs only). x, W_gu, W_down and dY are
rounded to bf16; logits stay fp32. The skewed workload adds a per-expert bias
3*ln(p_e) to every logit row, p_e the Zipf(s=1.2) probability of rank e+1 over
E ranks, so expert 0 is the most popular. Where the router GEMM computes the
logits from x, its weight W_r ~ N(0, 1/d) [E,d] (unit-variance logits) is rounded
to bf16 and drawn from a stream of its own (seed sequence [seed, 7]), so adding it
changes none of the draws above.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    d: int            # hidden size
    E: int            # experts
    k: int            # experts per token
    f: int            # expert FFN width (W_gu is d x 2f, W_down is f x d)
    seed: int
    backward: bool    # the workload includes the backward pass
    zipf_bias: bool = False
    description: str = ""

    @property
    def A(self) -> int:
        """Rows after dispatch: one per (token, chosen expert)."""
        return self.T * self.k

    def gemm_flops(self, backward: bool | None = None) -> int:
        """Algorithmic GEMM FLOPs: 6*A*d*f forward, 18*A*d*f forward+backward."""
        bwd = self.backward if backward is None else backward
        return (18 if bwd else 6) * self.A * self.d * self.f

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", T=512, d=256, E=8, k=2, f=512, seed=0, backward=False,
                     description="tiny MoE forward, T=512 d=256 E=8 k=2 f=512"),
    "qwen3_moe": Workload("qwen3_moe", T=4096, d=2048, E=128, k=8, f=768, seed=1,
                          backward=False,
                          description="Qwen3-MoE-like forward, T=4096 d=2048 E=128 k=8 f=768"),
    "gpt_oss_20b": Workload("gpt_oss_20b", T=4096, d=2880, E=32, k=4, f=2880, seed=2,
                            backward=True,
                            description="gpt-oss-20b-like forward+backward, T=4096 d=2880 E=32 k=4 f=2880"),
    "skewed": Workload("skewed", T=4096, d=2880, E=32, k=4, f=2880, seed=3, backward=True,
                       zipf_bias=True,
                       description="skewed-load gpt-oss-20b-like forward+backward, Zipf(1.2) expert bias"),
    "long": Workload("long", T=65536, d=2880, E=32, k=4, f=2880, seed=4, backward=True,
                     description="long-sequence gpt-oss-20b-like forward+backward, T=65536"),
}


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """fp32 numpy -> torch bf16 (CPU), round-to-nearest-even."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _normal_bf16(rng: np.random.Generator, shape: tuple, scale: float | None = None,
                 chunk_elems: int = 1 << 24) -> torch.Tensor:
    """N(0,1) (times scale) drawn in fp32 and rounded to bf16, in slabs along dim 0.

    Drawing slab by slab consumes the generator in the same order as one call over
    the whole shape (element by element), so the values equal a single draw; the
    slabs only keep the fp32 staging buffer small.
    """
    out = torch.empty(shape, dtype=torch.bfloat16)
    inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    rows = max(1, chunk_elems // max(inner, 1))
    flat = out.view(shape[0], inner)
    buf = np.empty((min(rows, shape[0]), inner), dtype=np.float32)
    for r0 in range(0, shape[0], rows):
        n = min(rows, shape[0] - r0)
        b = buf[:n]
        rng.standard_normal(out=b, dtype=np.float32)
        if scale is not None:
            b *= np.float32(scale)
        flat[r0:r0 + n].copy_(torch.from_numpy(b))
    return out


def zipf_bias(E: int, s: float = 1.2, scale: float = 3.0) -> np.ndarray:
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    return (scale * np.log(p)).astype(np.float32)


@dataclasses.dataclass
class Inputs:
    """CPU tensors of one workload: bf16 where the block takes bf16, fp32 logits."""
    x: torch.Tensor         # [T, d] bf16
    logits: torch.Tensor    # [T, E] fp32
    w_gu: torch.Tensor      # [E, d, 2f] bf16 (gate columns [0,f), up columns [f,2f))
    w_down: torch.Tensor    # [E, f, d] bf16
    dy: torch.Tensor | None  # [T, d] bf16


def make_inputs(wl: Workload, with_dy: bool | None = None) -> Inputs:
    rng = np.random.default_rng(wl.seed)
    T, d, E, f = wl.T, wl.d, wl.E, wl.f
    x = _normal_bf16(rng, (T, d))
    logits = rng.standard_normal((T, E), dtype=np.float32)
    if wl.zipf_bias:
        logits = logits + zipf_bias(E)[None, :]
    w_gu = _normal_bf16(rng, (E, d, 2 * f), 0.02)
    w_down = _normal_bf16(rng, (E, f, d), 0.02)
    want_dy = wl.backward if with_dy is None else with_dy
    dy = _normal_bf16(rng, (T, d)) if want_dy else None
    return Inputs(x=x, logits=torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)),
                  w_gu=w_gu, w_down=w_down, dy=dy)


def make_router_weight(wl: Workload) -> torch.Tensor:
    """Router weight [E, d] bf16, one row per expert, N(0, 1/d)."""
    rng = np.random.default_rng([wl.seed, 7])
    return _normal_bf16(rng, (wl.E, wl.d), 1.0 / np.sqrt(wl.d))


def small_case(T: int, d: int, E: int, k: int, f: int, seed: int, backward: bool = True,
               logit_scale: float = 1.0) -> tuple[Workload, Inputs]:
    """An ad-hoc shape drawn with the same recipe (for parity and edge-case tests)."""
    wl = Workload(f"case_T{T}_d{d}_E{E}_k{k}_f{f}_s{seed}", T=T, d=d, E=E, k=k, f=f,
                  seed=seed, backward=backward)
    inp = make_inputs(wl)
    if logit_scale != 1.0:
        inp.logits = inp.logits * logit_scale
    return wl, inp


__all__ = ["Workload", "WORKLOADS", "Inputs", "make_inputs", "small_case", "to_bf16",
           "zipf_bias", "make_router_weight"]
