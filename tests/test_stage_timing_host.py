"""The stage timing summary on the host: from synthetic stamps whose spacing is known,
the summary returns that spacing, the producer's and the issuer's waits, and, given the
stages per tile, the extra delay of each tile's first stage."""
import numpy as np

from moe_expert_layer_route_gb300.stage_timing import _summary


def _stamps(n, kt, period, first_extra, tma, slot_wait):
    """n stages: the MMA issuer issues stage i at mi[i]; a tile's first stage (i % kt == 0,
    i > 0) comes first_extra cycles later; its data was seen 100 cycles before it was
    issued and requested tma cycles before that; the producer waited slot_wait cycles
    between its free slot and its issued loads."""
    mi = np.zeros(n, dtype=np.int64)
    for i in range(1, n):
        mi[i] = mi[i - 1] + period + (first_extra if i % kt == 0 else 0)
    mf = mi - 100
    pi = mf - tma
    pe = pi - slot_wait
    return np.stack([pe, pi, mf, mi], axis=1) + 10_000


def test_summary_splits_tile_first_stages():
    kt, period, extra = 23, 1200, 600
    st = _stamps(230, kt, period, extra, tma=1900, slot_wait=20)
    tl = np.array([[0, 5000], [30000, 35000], [60000, 65000]], dtype=np.int64)
    s = _summary(st, tl, kt)
    assert s["stages"] == 230 and s["tiles"] == 3 and s["stages_per_tile"] == kt
    assert s["issue_spacing_median"] == period
    assert s["other_stage_spacing_mean"] == period
    assert s["tile_first_stage_spacing_mean"] == period + extra
    # from the previous stage's issue to this stage's data: the spacing less 100
    assert s["waited_for_data_median"] == period - 100
    assert s["tile_first_stage_wait_mean"] == period + extra - 100
    assert s["tma_issue_to_data_median"] == 1900
    assert s["tile_first_stage_tma_latency_mean"] == 1900 == s["other_stage_tma_latency_mean"]
    assert s["tile_first_stage_producer_slot_wait_mean"] == 20
    assert s["epilogue_per_tile_median"] == 5000
    assert s["accumulator_ready_spacing_median"] == 30000


def test_summary_without_stages_per_tile_has_no_split():
    st = _stamps(50, 10, 1000, 0, tma=1500, slot_wait=5)
    s = _summary(st, np.zeros((0, 2), dtype=np.int64))
    assert "stages_per_tile" not in s and "epilogue_per_tile_median" not in s
    assert s["issue_spacing_mean"] == 1000
