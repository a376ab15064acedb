"""Failure detection on the GPU without a fault: a pipeline wait that nothing will
ever satisfy runs out of time, the kernel records MOE_ERR_TIMEOUT in the workspace
status word and returns, the host reads it, and the context stays usable.

The stall is made by withholding the loads of each CTA's first k-block in the gate_up
GEMM (moe_debug_gate_up_withheld), with a 20 ms wait limit, for the single-CTA engine
(256 rows per expert) and the SM-pair engine (512 rows per expert)."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_route_gb300 as m
    return m


@pytest.mark.parametrize("T,E", [(512, 4), (1024, 4)], ids=["single", "pair"])
def test_withheld_loads_time_out_and_the_context_survives(moe, T, E):
    wl = workloads.Workload("stall", T=T, d=256, E=E, k=2, f=192, seed=90, backward=False)
    inp = workloads.make_inputs(wl)
    s = moe.shape(wl.T, wl.d, wl.E, wl.k, wl.f)
    ids, _ = moe.route(inp.logits.cuda(), wl.k)
    disp = moe.dispatch(s, inp.x.cuda(), ids)
    w_gu, w_down = inp.w_gu.cuda(), inp.w_down.cuda()
    ws = moe.new_workspace(s, False)
    h0, _, o0 = moe.expert_ffn(s, disp["xp"], disp["counts"], w_gu, w_down, ws=ws)
    moe.check_device_status(ws)                       # a normal call leaves MOE_OK

    moe.debug_gate_up_withheld(s, disp["xp"], disp["counts"], w_gu, ws, wait_limit_us=20000)
    with pytest.raises(moe.MoEError) as err:
        moe.check_device_status(ws)
    assert err.value.status == -7                     # MOE_ERR_TIMEOUT
    moe.check_device_status(ws)                       # reading it cleared it

    h1, _, o1 = moe.expert_ffn(s, disp["xp"], disp["counts"], w_gu, w_down, ws=ws)
    torch.cuda.synchronize()
    moe.check_device_status(ws)
    # rows at and past padded_offsets[E] belong to no expert and are never written
    P = int(disp["padded_offsets"][-1])
    assert torch.equal(h0[:P], h1[:P]) and torch.equal(o0[:P], o1[:P])
