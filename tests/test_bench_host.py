"""Host-side checks of bench.py's bookkeeping (no GPU): the per-kernel work figures it
divides by launch times must follow the library's own rules and the stated formulas."""
import pytest

import bench
import workloads


@pytest.fixture(scope="module")
def moe():
    from moe_expert_layer_route_gb300 import _build
    _build.build()
    import moe_expert_layer_route_gb300 as m
    return m


@pytest.mark.parametrize("T,d,E", [(4096, 2880, 32), (4096, 2048, 128), (65536, 2880, 32),
                                   (512, 256, 8), (100, 520, 40), (33, 64, 256)])
def test_router_splits_match_the_library_scratch(moe, T, d, E):
    splits = bench.router_splits(T, d, E)
    size = moe.lib().moe_router_backward_scratch_size(moe.shape(T, d, E, 2, 8))
    assert size == (splits * E * d * 4 if splits > 1 else 16)


def test_gemm_bytes_are_weights_plus_rows():
    wl = workloads.WORKLOADS["gpt_oss_20b"]
    A, d, f, E = wl.A, wl.d, wl.f, wl.E
    gb = bench.gemm_bytes(wl, training=True)
    w_gu, w_down = E * d * 2 * f * 2, E * f * d * 2
    assert gb["gemm_gate_up_swiglu"] == w_gu + A * (d + f + 2 * f) * 2
    assert gb["gemm_wgrad_gu"] == w_gu + A * (d + 2 * f) * 2
    assert gb["gemm_down"] == gb["gemm_wgrad_down"] == w_down + A * (f + d) * 2
    # forward-only: no saved gate/up pre-activations
    assert bench.gemm_bytes(wl, training=False)["gemm_gate_up_swiglu"] == \
        w_gu + A * (d + f) * 2


def test_kernel_work_flops_sum_to_the_block():
    wl = workloads.WORKLOADS["gpt_oss_20b"]
    work = bench.kernel_work(wl)
    gemm = sum(v for k, (kind, v) in work.items() if kind == "flop")
    assert gemm == wl.gemm_flops(backward=True)          # 18 A d f
    assert work["router_route_count"] == ("alu_flop", 2 * wl.T * wl.E * wl.d)


def test_fused_route_scan_moves_the_bytes_of_both_stages():
    """The forward's route launch runs the scan in its last block: its algorithmic bytes
    are those of route + count plus those of the scan."""
    wl = workloads.WORKLOADS["qwen3_moe"]
    work = bench.kernel_work(wl)
    assert work["route_count_scan"][0] == "byte"
    assert work["route_count_scan"][1] == work["route_count"][1] + work["scan"][1]
