"""The router GEMM with the route in its epilogue, against the oracle.

The logits are one fp32 chain per (token, expert) in ascending i on both sides, so
they are compared bit for bit, and so are the chosen experts; the routing weights
(a softmax through expf) within the route tests' relative bound. Shapes span several
32-token chunks with a ragged last chunk, d not a multiple of the 32-wide staging
block, every thread-tile configuration (E up to 8, 16, 32, 64, 128, 256), k = 1 and
k = 16, and T = 0."""
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


def _case(T, d, E, k, seed):
    wl = workloads.Workload("r", T=T, d=d, E=E, k=k, f=64, seed=seed, backward=False)
    return wl, workloads.make_inputs(wl), workloads.make_router_weight(wl)


def _check_route(moe, x, wr, k, bias=None):
    logits, ids, w = moe.router_route(x.to(DEV), wr.to(DEV), k,
                                      None if bias is None else torch.from_numpy(bias).to(DEV))
    torch.cuda.synchronize()
    want = oracle.router_logits(x.float().numpy(), wr.float().numpy())
    got = to_np(logits)
    assert np.array_equal(got, want), \
        f"logits differ at {np.argwhere(got != want)[:5].tolist()}"
    rid, rw = oracle.route(want, k, bias)
    assert np.array_equal(to_np(ids), rid)
    np.testing.assert_allclose(to_np(w), rw, rtol=W_REL, atol=0)


@pytest.mark.parametrize("T,d,E,k", [
    (100, 256, 8, 2),       # E <= 8 tile, ragged last chunk
    (333, 200, 32, 4),      # d = 6 blocks of 32 + 8: ragged k block
    (64, 2880, 32, 4),      # the gpt-oss-20b router row length
    (130, 2048, 128, 8),    # Qwen3-MoE-like
    (70, 136, 256, 16),     # widest tile, k = 16
    (33, 64, 16, 3),
    (97, 520, 64, 6),
    (45, 8, 5, 1),          # one 8-wide vector per row, E not a tile multiple, k = 1
    (1, 24, 40, 2),
])
def test_router_route_bit_exact(moe, T, d, E, k):
    _, inp, wr = _case(T, d, E, k, seed=T * 7 + d + E)
    _check_route(moe, inp.x, wr, k)


def test_router_route_with_selection_bias(moe):
    _, inp, wr = _case(500, 384, 32, 4, seed=5)
    _check_route(moe, inp.x, wr, 4, workloads.zipf_bias(32))


def test_router_route_ties_go_to_the_lower_index(moe):
    # integer-valued inputs make many logits exactly equal
    rng = np.random.default_rng(6)
    x = torch.from_numpy(rng.integers(-2, 3, size=(96, 64)).astype(np.float32)).to(torch.bfloat16)
    wr = torch.from_numpy(rng.integers(-1, 2, size=(24, 64)).astype(np.float32)).to(torch.bfloat16)
    _check_route(moe, x, wr, 5)


@pytest.mark.parametrize("name", ["gpt_oss_20b", "qwen3_moe"])
def test_router_route_full_size(moe, name):
    wl = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(wl.scaled(backward=False))
    _check_route(moe, inp.x, workloads.make_router_weight(wl), wl.k)


def test_router_route_long_sampled(moe):
    wl = workloads.WORKLOADS["long"]
    inp = workloads.make_inputs(wl.scaled(backward=False))
    wr = workloads.make_router_weight(wl)
    logits, ids, w = moe.router_route(inp.x.to(DEV), wr.to(DEV), wl.k)
    rows = np.random.default_rng(8).choice(wl.T, 512, replace=False)
    rows[:2] = [0, wl.T - 1]
    want = oracle.router_logits(inp.x[rows].float().numpy(), wr.float().numpy())
    assert np.array_equal(to_np(logits)[rows], want)
    rid, rw = oracle.route(want, wl.k)
    assert np.array_equal(to_np(ids)[rows], rid)
    np.testing.assert_allclose(to_np(w)[rows], rw, rtol=W_REL, atol=0)


def test_router_route_no_tokens(moe):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    wr = torch.zeros((8, 64), dtype=torch.bfloat16, device=DEV)
    logits, ids, w = moe.router_route(x, wr, 2)
    assert logits.shape == (0, 8) and ids.shape == (0, 2)


@pytest.mark.parametrize("T,d,E,k,f", [(1000, 256, 16, 4, 192), (600, 520, 40, 3, 136)])
def test_forward_router_matches_the_oracle(moe, T, d, E, k, f):
    wl = workloads.Workload("fr", T=T, d=d, E=E, k=k, f=f, seed=T + E, backward=False)
    inp = workloads.make_inputs(wl)
    wr = workloads.make_router_weight(wl)
    X, _, Wg, Wd, _ = inputs_np(inp)
    L = oracle.router_logits(inp.x.float().numpy(), wr.float().numpy())
    ref = oracle.forward(X, L, Wg, Wd, k)
    y, logits, ws, s = moe.forward_router(inp.x.to(DEV), wr.to(DEV), inp.w_gu.to(DEV),
                                          inp.w_down.to(DEV), k)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(logits), L)
    check_dispatch_exact(moe.workspace_views(s, False, ws), ref, inp.x, k)
    assert_close(to_np(y), ref["y"], "Y")
    # the same block fed the same logits from memory gives the same bits
    y2, _, _ = moe.forward(inp.x.to(DEV), logits, inp.w_gu.to(DEV), inp.w_down.to(DEV), k)
    assert torch.equal(y, y2)


def test_forward_router_bias_and_aux_statistics(moe):
    T, d, E, k = 777, 256, 32, 4
    wl = workloads.Workload("fa", T=T, d=d, E=E, k=k, f=128, seed=17, backward=False)
    inp = workloads.make_inputs(wl)
    wr = workloads.make_router_weight(wl)
    bias = workloads.zipf_bias(E)
    L = oracle.router_logits(inp.x.float().numpy(), wr.float().numpy())
    X, _, Wg, Wd, _ = inputs_np(inp)
    ref = oracle.forward(X, L, Wg, Wd, k, bias)
    st = oracle.aux_stats(L, ref["counts"], k)
    aux = torch.empty(2 * E + 1, dtype=torch.float32, device=DEV)
    y, logits, ws, s = moe.forward_router(inp.x.to(DEV), wr.to(DEV), inp.w_gu.to(DEV),
                                          inp.w_down.to(DEV), k, bias=torch.from_numpy(bias).to(DEV),
                                          aux_stats=aux)
    torch.cuda.synchronize()
    check_dispatch_exact(moe.workspace_views(s, False, ws), ref, inp.x, k)
    assert_close(to_np(y), ref["y"], "Y")
    a = to_np(aux)
    np.testing.assert_allclose(a[:E], st["f"], rtol=1e-6, atol=0)
    np.testing.assert_allclose(a[E:2 * E], st["P"], rtol=1e-5, atol=0)
    np.testing.assert_allclose(a[2 * E], st["aux"], rtol=1e-5)
