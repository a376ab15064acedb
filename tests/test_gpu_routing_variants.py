"""Routing variants on the GPU against the oracle: the selection bias (choose on
logit + bias, weight on the unbiased logits), the load-balancing statistics
(f_e, P_e, E * sum f_e P_e) and the gradient of the load-balancing loss."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import check_dispatch_exact, inputs_np, to_np
from tolerance import W_REL, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_route_gb300 as m
    return m


def _bias(E, seed, kind):
    rng = np.random.default_rng(seed)
    if kind == "zipf":
        return workloads.zipf_bias(E)
    if kind == "coarse":  # ties between biased scores
        return (rng.integers(-4, 5, size=E) * 0.25).astype(np.float32)
    return (rng.standard_normal(E) * 0.5).astype(np.float32)


@pytest.mark.parametrize("T,E,k,kind", [(512, 8, 2, "normal"), (4096, 128, 8, "normal"),
                                        (300, 32, 4, "zipf"), (777, 40, 5, "coarse"),
                                        (130, 256, 16, "normal"), (64, 8, 1, "zipf")])
def test_route_with_selection_bias(moe, T, E, k, kind):
    wl = workloads.Workload("b", T=T, d=64, E=E, k=k, f=64, seed=T + E, backward=False)
    inp = workloads.make_inputs(wl)
    logits = inp.logits.numpy()
    if kind == "coarse":
        logits = (np.round(logits * 4) / 4).astype(np.float32)
    bias = _bias(E, T, kind)
    ids, w = moe.route(torch.from_numpy(logits).to(DEV), k, torch.from_numpy(bias).to(DEV))
    rid, rw = oracle.route(logits, k, bias)
    assert np.array_equal(to_np(ids), rid)
    np.testing.assert_allclose(to_np(w), rw, rtol=W_REL, atol=0)


def test_forward_with_bias_and_aux_statistics(moe):
    wl, inp = None, None
    wl = workloads.Workload("fa", T=1000, d=256, E=16, k=4, f=192, seed=81, backward=False)
    inp = workloads.make_inputs(wl)
    X, L, Wg, Wd, _ = inputs_np(inp)
    bias = _bias(16, 82, "normal")
    ref = oracle.forward(X, L, Wg, Wd, wl.k, bias)
    st = oracle.aux_stats(L, ref["counts"], wl.k)
    aux = torch.empty(2 * 16 + 1, dtype=torch.float32, device=DEV)
    y, ws, s = moe.forward(inp.x.to(DEV), inp.logits.to(DEV), inp.w_gu.to(DEV),
                           inp.w_down.to(DEV), wl.k, bias=torch.from_numpy(bias).to(DEV),
                           aux_stats=aux)
    torch.cuda.synchronize()
    views = moe.workspace_views(s, False, ws)
    check_dispatch_exact(views, ref, inp.x, wl.k)
    assert_close(to_np(y), ref["y"], "Y")
    a = to_np(aux)
    np.testing.assert_allclose(a[:16], st["f"], rtol=1e-6, atol=0)
    np.testing.assert_allclose(a[16:32], st["P"], rtol=1e-5, atol=0)
    np.testing.assert_allclose(a[32], st["aux"], rtol=1e-5)


@pytest.mark.parametrize("T,E,k", [(4096, 32, 4), (333, 128, 8), (1, 8, 2)])
def test_aux_statistics_at_scale_and_edges(moe, T, E, k):
    wl = workloads.Workload("a", T=T, d=64, E=E, k=k, f=64, seed=T * 3 + E, backward=False)
    inp = workloads.make_inputs(wl)
    aux = torch.empty(2 * E + 1, dtype=torch.float32, device=DEV)
    _, ws, s = moe.forward(inp.x.to(DEV), inp.logits.to(DEV), inp.w_gu.to(DEV),
                           inp.w_down.to(DEV), k, aux_stats=aux)
    counts = to_np(moe.workspace_views(s, False, ws)["counts"])
    st = oracle.aux_stats(inp.logits.numpy(), counts, k)
    a = to_np(aux)
    np.testing.assert_allclose(a[:E], st["f"], rtol=1e-6, atol=0)
    np.testing.assert_allclose(a[E:2 * E], st["P"], rtol=1e-5, atol=1e-9)
    np.testing.assert_allclose(a[2 * E], st["aux"], rtol=1e-5)


def test_aux_loss_gradient_adds_into_dlogits(moe):
    wl = workloads.Workload("g", T=700, d=128, E=24, k=3, f=64, seed=91, backward=True)
    inp = workloads.make_inputs(wl)
    X, L, Wg, Wd, DY = inputs_np(inp)
    ref = oracle.forward(X, L, Wg, Wd, wl.k)
    w_gu, w_down = inp.w_gu.to(DEV), inp.w_down.to(DEV)
    logits = inp.logits.to(DEV)
    y, ws, s = moe.forward(inp.x.to(DEV), logits, w_gu, w_down, wl.k, training=True)
    _, _, _, dl = moe.backward(s, inp.dy.to(DEV), w_gu, w_down, ws, router_grad=True)
    counts = moe.workspace_views(s, True, ws)["counts"]
    moe.aux_loss_backward(s, logits, counts, 0.01, dl)
    torch.cuda.synchronize()
    want = oracle.router_backward(DY, ref) + 0.01 * oracle.aux_loss_grad(L, ref["counts"], wl.k)
    assert_close(to_np(dl), want, "dlogits + aux gradient")
    only = torch.zeros_like(logits)
    moe.aux_loss_backward(s, logits, counts, 1.0, only)
    assert_close(to_np(only), oracle.aux_loss_grad(L, ref["counts"], wl.k), "aux gradient")
    assert np.abs(to_np(only).sum(axis=1)).max() < 1e-6
