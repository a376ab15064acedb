"""The library's calls can be captured in a CUDA graph: they allocate nothing, never
synchronise the host, and the router GEMM gradient's fork to the library's second
stream and join back are events, which capture as graph edges. A captured training step
(router GEMM forward, expert backward, load-balancing gradient, router GEMM gradient)
replayed twice gives the eager step's results bit for bit (every kernel is
deterministic)."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_route_gb300 as m
    return m


def test_captured_training_step_replays_bit_exactly(moe):
    T, d, E, k, f = 1000, 256, 16, 4, 192
    wl = workloads.Workload("graph", T=T, d=d, E=E, k=k, f=f, seed=31, backward=True)
    inp = workloads.make_inputs(wl)
    x, dy = inp.x.to(DEV), inp.dy.to(DEV)
    w_gu, w_down = inp.w_gu.to(DEV), inp.w_down.to(DEV)
    w_r = workloads.make_router_weight(wl).to(DEV)
    s = moe.shape(T, d, E, k, f)
    ws, scratch = moe.new_workspace(s, True, DEV), moe.new_scratch(s, DEV)
    r_scratch = torch.empty(max(16, moe.lib().moe_router_backward_scratch_size(s)),
                            dtype=torch.uint8, device=DEV)
    y = torch.empty_like(x)
    logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
    grads = (torch.empty_like(x), torch.empty_like(w_gu), torch.empty_like(w_down))
    dl = torch.empty((T, E), dtype=torch.float32, device=DEV)
    dw_r = torch.empty((E, d), dtype=torch.float32, device=DEV)
    counts = moe.workspace_views(s, True, ws)["counts"]

    def step():
        moe.forward_router(x, w_r, w_gu, w_down, k, training=True, ws=ws, y=y, logits=logits)
        moe.backward(s, dy, w_gu, w_down, ws, scratch, out=grads, dlogits=dl)
        moe.aux_loss_backward(s, logits, counts, 0.01, dl)
        moe.router_backward(s, x, w_r, dl, grads[0], dw_r, r_scratch)

    outs = (y, logits, *grads, dl, dw_r)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        step()                                   # eager (also sets up kernel attributes)
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs]
    for t in outs:
        t.zero_()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(2):
        for t in outs:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        moe.check_device_status(ws)
        moe.check_device_status(scratch)
        for got, want in zip(outs, eager):
            assert torch.equal(got, want)
