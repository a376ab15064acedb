"""Where the grouped GEMMs' time goes: the stage timing of the diagnostic build.

    python -m moe_expert_layer_route_gb300.stage_timing [workload]
    python -m moe_expert_layer_route_gb300.stage_timing --check

Builds (if needed) and loads the diagnostic variant of the library, which carries the
grouped GEMMs' stage timing (compiled with MOE_STAGE_TIMING; the shipped library has
none of it, the stamps cost ~2% of the GEMMs' time even unarmed), then runs one forward
+ backward of a seeded workload (after a warm-up step) once per GEMM kind with the
timing armed for that kind, and prints, from CTA 0's stamps (SM clock cycles): the
spacing of the MMA issuer's stages (a stage is two 64-wide K-blocks, 8 MMAs of
256 x 256 x 16 per SM pair: 1024 cycles of tensor work per SM), how long the issuer
waited for each stage's operands after issuing the previous one, the latency from the
producer's TMA issue to the issuer seeing the data, and the epilogue's time per tile.
--check runs a small case and checks the stamps' order and that an armed launch computes
what an unarmed one does.

It must be the process's entry point: the diagnostic library replaces the shipped one
for the whole process.
"""
from __future__ import annotations

import json
import sys

import numpy as np


def _load():
    import moe_expert_layer_route_gb300 as moe
    from moe_expert_layer_route_gb300 import _build
    if moe._lib is not None and moe.LIB_PATH != _build.TIMING_LIB:
        raise RuntimeError("the shipped library is already loaded in this process; run "
                           "`python -m moe_expert_layer_route_gb300.stage_timing` on its own")
    moe.LIB_PATH = _build.build(timing=True)
    moe.lib()
    return moe


def _summary(st: np.ndarray, tl: np.ndarray, kt: int | None = None) -> dict:
    """kt: stages per tile when every tile of the kind has the same K (the ragged-M
    kinds), to split the spacing into the first stage of a tile and the others."""
    t0 = st[0, 0]
    pe, pi, mf, mi = (st[:, j] - t0 for j in range(4))
    out = {"stages": int(len(st)), "cycles": int(mi[-1]),
           "issue_spacing_median": float(np.median(np.diff(mi))),
           "issue_spacing_mean": float(np.diff(mi).mean()),
           "waited_for_data_median": float(np.median(mf[1:] - mi[:-1])),
           "tma_issue_to_data_median": float(np.median(mf - pi)),
           "tiles": int(len(tl))}
    if kt and len(mi) > kt:
        first = (np.arange(1, len(mi)) % kt) == 0  # spacing that ends at a tile's first stage
        sp, wait, lat = np.diff(mi), mf[1:] - mi[:-1], (mf - pi)[1:]
        out.update({
            "stages_per_tile": int(kt),
            "tile_first_stage_spacing_mean": float(sp[first].mean()),
            "other_stage_spacing_mean": float(sp[~first].mean()),
            "tile_first_stage_wait_mean": float(wait[first].mean()),
            "tile_first_stage_tma_latency_mean": float(lat[first].mean()),
            "other_stage_tma_latency_mean": float(lat[~first].mean()),
            # the producer's wait for a free slot before each of those stages
            "tile_first_stage_producer_slot_wait_mean": float((pi - pe)[1:][first].mean()),
        })
    if len(tl):
        out["epilogue_per_tile_median"] = float(np.median(tl[:, 1] - tl[:, 0]))
    if len(tl) > 1:
        out["accumulator_ready_spacing_median"] = float(np.median(np.diff(tl[:, 0])))
    return out


def run(workload: str = "gpt_oss_20b") -> dict:
    import torch

    import workloads  # the seeded input recipe (repository root)
    moe = _load()
    wl = workloads.WORKLOADS[workload]
    inp = workloads.make_inputs(wl, with_dy=True)
    dev = "cuda"
    x, lg, dy = inp.x.to(dev), inp.logits.to(dev), inp.dy.to(dev)
    wgu, wd = inp.w_gu.to(dev), inp.w_down.to(dev)

    def step():
        y, ws, s = moe.forward(x, lg, wgu, wd, wl.k, training=True)
        moe.backward(s, dy, wgu, wd, ws)

    step()
    torch.cuda.synchronize()
    # stages per tile of the ragged-M kinds: K / (K per stage), 128 on SM pairs, 64 on
    # single CTAs (pairs from 256 rows per expert)
    bks = 128 if wl.T * wl.k // wl.E >= 256 else 64
    kts = {"gate_up": -(-wl.d // bks), "down": -(-wl.f // bks), "dgrad_h": -(-wl.d // bks),
           "dgrad_x": -(-2 * wl.f // bks)}
    res = {}
    try:
        for kind in ("gate_up", "down", "dgrad_h", "dgrad_x", "wgrad"):
            moe.stage_timing_arm(kind)
            step()
            st, tl = moe.stage_timing_read()
            if len(st) > 1:
                res[kind] = _summary(st, tl, kts.get(kind))
    finally:
        moe.stage_timing_arm(None)
    return res


def check() -> None:
    """Stamps in order; an armed launch computes exactly what an unarmed one does;
    disarmed, nothing is stamped."""
    import torch

    import workloads
    moe = _load()
    wl = workloads.Workload("timing", T=1024, d=256, E=4, k=2, f=320, seed=90, backward=False)
    inp = workloads.make_inputs(wl)
    s = moe.shape(wl.T, wl.d, wl.E, wl.k, wl.f)
    ids, _ = moe.route(inp.logits.cuda(), wl.k)
    disp = moe.dispatch(s, inp.x.cuda(), ids)
    args = (s, disp["xp"], disp["counts"], inp.w_gu.cuda(), inp.w_down.cuda())
    _, _, o_plain = moe.expert_ffn(*args)
    try:
        moe.stage_timing_arm("down")
        _, _, o_timed = moe.expert_ffn(*args)
        st, tl = moe.stage_timing_read()
        assert torch.equal(o_timed, o_plain), "an armed launch changed the result"
        assert len(st) > 1 and len(tl) >= 1, "nothing stamped"
        p_free, p_issued, m_full, m_issued = st.T
        assert (p_issued >= p_free).all() and (m_issued >= m_full).all()
        assert (np.diff(m_issued) > 0).all(), "stages not consumed in order"
        assert (m_full >= p_issued).all(), "data seen before it was requested"
        assert (tl[:, 1] >= tl[:, 0]).all()
        moe.stage_timing_arm(None)
        moe.expert_ffn(*args)
        st2, tl2 = moe.stage_timing_read()
        assert len(st2) == 0 and len(tl2) == 0, "stamped while disarmed"
    finally:
        moe.stage_timing_arm(None)
    print("stage timing check ok")


if __name__ == "__main__":
    if len(sys.argv) > 1 and sys.argv[1] == "--check":
        check()
    else:
        print(json.dumps(run(sys.argv[1] if len(sys.argv) > 1 else "gpt_oss_20b"), indent=1))
