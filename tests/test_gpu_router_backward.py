"""The gradient through the router GEMM against the oracle (fp64).

dW_r = dlogits^T x and the dX term dlogits W_r are fp32 sums, so they are checked
against bounds derived from their summation length (n terms in fp32: at most about
n * 2^-24 of the sum of |terms|) plus, for dX, the one bf16 rounding of the result.
The last test runs a whole training step through the router (forward from x,
backward with the router-logit and load-balancing gradients, then the router GEMM's
gradient) and checks dX and dW_r against the oracle's step."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import inputs_np, to_np
from tolerance import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -24


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_route_gb300 as m
    return m


def _inputs(T, d, E, seed):
    wl = workloads.Workload("rb", T=T, d=d, E=E, k=min(2, E), f=8, seed=seed, backward=True)
    inp = workloads.make_inputs(wl)
    wr = workloads.make_router_weight(wl)
    dl = np.random.default_rng(seed + 1).standard_normal((T, E)).astype(np.float32)
    return wl, inp, wr, dl


def _check(moe, T, d, E, seed):
    wl, inp, wr, dl = _inputs(T, d, E, seed)
    s = moe.shape(T, d, E, wl.k, 8)
    dx = inp.dy.to(DEV).clone()            # any bf16 dX on entry
    dx_in = inp.dy.double().numpy()
    dw = moe.router_backward(s, inp.x.to(DEV), wr.to(DEV), torch.from_numpy(dl).to(DEV), dx)
    torch.cuda.synchronize()
    X, W = inp.x.double().numpy(), wr.double().numpy()
    want_dw, want_dx = oracle.router_weight_backward(X, W, dl)
    got_dw = to_np(dw).astype(np.float64)
    bound_dw = 2 * T * U * (np.abs(dl).T.astype(np.float64) @ np.abs(X)) + 1e-30
    assert (np.abs(got_dw - want_dw) <= bound_dw).all(), \
        f"dW_r off by {np.max(np.abs(got_dw - want_dw) / bound_dw):.2f} of its bound"
    ref = dx_in + want_dx
    got = to_np(dx).astype(np.float64)
    bound_dx = 2.0 ** -8 * np.abs(ref) + 2 * (E + 1) * U * (np.abs(dl) @ np.abs(W) + np.abs(dx_in))
    assert (np.abs(got - ref) <= bound_dx + 1e-30).all(), \
        f"dX off by {np.max(np.abs(got - ref) / (bound_dx + 1e-30)):.2f} of its bound"


@pytest.mark.parametrize("T,d,E", [
    (100, 256, 8),       # one column block, one token split
    (333, 520, 40),      # ragged columns (520 = 2 x 256 + 8), E not a multiple of 32
    (64, 2880, 32),      # the gpt-oss-20b row length
    (130, 2048, 128),    # four expert blocks in dW, two 64-expert stages in dX
    (70, 136, 256),
    (1, 8, 4),
])
def test_router_backward_matches_the_oracle(moe, T, d, E):
    _check(moe, T, d, E, seed=T + d + E)


def test_router_backward_full_size_token_splits(moe):
    # 4096 tokens: dW_r is summed in about 26 token splits, then the splits in order
    _check(moe, 4096, 2880, 32, seed=5)


def test_router_backward_is_deterministic(moe):
    wl, inp, wr, dl = _inputs(1000, 512, 32, 9)
    s = moe.shape(1000, 512, 32, 2, 8)
    outs = []
    for _ in range(2):
        dx = inp.dy.to(DEV).clone()
        dw = moe.router_backward(s, inp.x.to(DEV), wr.to(DEV), torch.from_numpy(dl).to(DEV), dx)
        outs.append((dx, dw))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_router_backward_no_tokens(moe):
    s = moe.shape(0, 64, 8, 2, 8)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    wr = torch.ones((8, 64), dtype=torch.bfloat16, device=DEV)
    dw = torch.full((8, 64), 7.0, device=DEV)
    moe.router_backward(s, x, wr, torch.empty((0, 8), device=DEV), x.clone(), dw)
    torch.cuda.synchronize()
    assert not dw.any()


def test_training_step_through_the_router(moe):
    T, d, E, k, f = 700, 256, 16, 4, 192
    wl = workloads.Workload("rt", T=T, d=d, E=E, k=k, f=f, seed=23, backward=True)
    inp = workloads.make_inputs(wl)
    wr = workloads.make_router_weight(wl)
    X, _, Wg, Wd, DY = inputs_np(inp)
    L = oracle.router_logits(inp.x.float().numpy(), wr.float().numpy())
    ref = oracle.forward(X, L, Wg, Wd, k)
    g = oracle.backward(DY, ref, Wg, Wd)
    dl_ref = oracle.router_backward(DY, ref) + 0.01 * oracle.aux_loss_grad(L, ref["counts"], k)
    dwr_ref, dxr_ref = oracle.router_weight_backward(X, wr.double().numpy(), dl_ref)

    x, w_gu, w_down, w_r = inp.x.to(DEV), inp.w_gu.to(DEV), inp.w_down.to(DEV), wr.to(DEV)
    y, logits, ws, s = moe.forward_router(x, w_r, w_gu, w_down, k, training=True)
    dx, dwg, dwd, dl = moe.backward(s, inp.dy.to(DEV), w_gu, w_down, ws, router_grad=True)
    moe.aux_loss_backward(s, logits, moe.workspace_views(s, True, ws)["counts"], 0.01, dl)
    dwr = moe.router_backward(s, x, w_r, dl, dx)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(logits), L)
    assert_close(to_np(y), ref["y"], "Y")
    assert_close(to_np(dl), dl_ref, "dlogits")
    assert_close(to_np(dx), g["dx"] + dxr_ref, "dX (experts + router)")
    assert_close(to_np(dwr), dwr_ref, "dW_r")
