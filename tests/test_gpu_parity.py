"""Parity of the CUDA path (through the C ABI) with the CPU oracle on GB300.

Indices, counts, offsets and the permutation are compared bit-exactly; routing
weights within 2e-6 relative (fp32 exp and sum against fp64); outputs and
gradients with the normwise bound of tests/tolerance.py. Shapes span several
tiles with ragged tails in M, N and K, empty experts, and the degenerate cases
(k = 1, k = E, E = 1, T = 1, T = 0)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import check_dispatch_exact, inputs_np, row_maps, to_np
from tolerance import W_REL, assert_close, assert_close_experts, assert_close_selected

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_route_gb300 as m
    assert torch.cuda.is_available()
    return m


DEV = "cuda"

# (T, d, E, k, f, seed, zipf)
ROUTE_CASES = [
    (512, 256, 8, 2, 512, 0, False),     # the tiny workload's shape
    (4096, 64, 128, 8, 64, 1, False),    # Qwen3-MoE-like routing (E=128, k=8)
    (77, 64, 33, 5, 64, 2, False),       # E just above a warp, T not a multiple of 32
    (300, 64, 3, 3, 64, 3, False),       # k = E < 32
    (130, 64, 256, 16, 64, 4, False),    # the largest E and k
    (64, 64, 8, 1, 64, 5, False),        # k = 1
    (1, 64, 4, 2, 64, 6, False),         # one token
    (2048, 64, 32, 4, 64, 7, True),      # skewed load with empty experts
]

FFN_CASES = [
    (512, 256, 8, 2, 512, 0, False),
    (300, 200, 5, 2, 200, 11, False),    # ragged K (200 = 3*64+8) and ragged N
    (1000, 320, 16, 4, 136, 12, False),  # N tail of 8 columns
    (96, 2880, 4, 2, 2880, 13, False),   # gpt-oss-20b-like widths
    (256, 2048, 128, 8, 768, 14, False), # Qwen3-MoE-like widths, many near-empty experts
    (512, 256, 32, 4, 256, 15, True),    # skewed: empty experts, one expert gets every token
    (200, 128, 1, 1, 64, 16, False),     # E = 1: a dense SwiGLU MLP
    # >= 256 rows per expert: the GEMMs run on SM pairs (256-row pair-tiles; an odd
    # tile count leaves the second half of an expert's last pair-tile unused)
    (1024, 256, 4, 2, 320, 17, False),
    (640, 256, 5, 2, 320, 22, False),    # 256 rows per expert: the smallest that pairs
    (900, 200, 3, 2, 200, 18, False),
    (300, 64, 256, 16, 64, 19, False),   # the largest E and k: 256 experts of ~19 rows
    (200, 64, 4, 2, 24, 20, False),      # f = 24: gate and up N tiles of 24 columns
    (300, 2048, 16, 6, 64, 21, False),   # combine: 4 warps per row, k = 6 (loads staged for k <= 8)
]


def _case(T, d, E, k, f, seed, zipf, backward=True):
    wl = workloads.Workload(f"c{T}_{d}_{E}_{k}_{f}", T=T, d=d, E=E, k=k, f=f, seed=seed,
                            backward=backward, zipf_bias=zipf)
    return wl, workloads.make_inputs(wl)


def _ids(c):
    return "T{}_d{}_E{}_k{}_f{}".format(*c[:5]) + ("_zipf" if c[6] else "")


@pytest.mark.parametrize("c", ROUTE_CASES, ids=_ids)
def test_route_bit_exact(moe, c):
    wl, inp = _case(*c)
    ids, w = moe.route(inp.logits.to(DEV), wl.k)
    rid, rw = oracle.route(inp.logits.numpy(), wl.k)
    assert np.array_equal(to_np(ids), rid)
    np.testing.assert_allclose(to_np(w), rw, rtol=W_REL, atol=0)


@pytest.mark.parametrize("E", [40, 200])
def test_route_ties_take_the_lower_index(moe, E):
    rng = np.random.default_rng(21 + E)
    logits = (rng.integers(-2, 3, size=(999, E)).astype(np.float32) * np.float32(0.25))
    logits[:5] = 0.0
    logits[5, :] = -0.0
    logits[5, 7] = 0.0
    # +0 and -0 mixed among negative scores: the two zeros are equal scores
    zeros = rng.random((999, E)) < 0.3
    signs = np.where(rng.random((999, E)) < 0.5, np.float32(-0.0), np.float32(0.0))
    logits[6:] = np.where(zeros[6:], signs[6:], -np.abs(logits[6:]) - np.float32(0.25))
    for k in (1, 3, 8, 16):
        ids, w = moe.route(torch.from_numpy(logits).to(DEV), k)
        rid, rw = oracle.route(logits, k)
        assert np.array_equal(to_np(ids), rid)
        np.testing.assert_allclose(to_np(w), rw, rtol=W_REL, atol=0)


@pytest.mark.parametrize("c", ROUTE_CASES, ids=_ids)
def test_dispatch_bit_exact(moe, c):
    wl, inp = _case(*c)
    s = moe.shape(wl.T, wl.d, wl.E, wl.k, wl.f)
    rid, _ = oracle.route(inp.logits.numpy(), wl.k)
    ref = oracle.dispatch(rid, wl.E)
    ref["ids"] = rid
    ids, _ = moe.route(inp.logits.to(DEV), wl.k)
    out = moe.dispatch(s, inp.x.to(DEV), ids)
    torch.cuda.synchronize()
    check_dispatch_exact(out, ref, inp.x, wl.k)


@pytest.mark.parametrize("k", [1, 2, 4, 8, 16])
def test_identity_experts_round_trip_is_k_times_x(moe, k):
    """dispatch -> identity experts -> combine with unit weights returns bf16(k * x) exactly."""
    wl, inp = _case(333, 136, 24, k, 64, 30 + k, False)
    s = moe.shape(wl.T, wl.d, wl.E, wl.k, wl.f)
    x = inp.x.to(DEV)
    ids, _ = moe.route(inp.logits.to(DEV), k)
    out = moe.dispatch(s, x, ids)
    ones = torch.ones((wl.T, k), dtype=torch.float32, device=DEV)
    y = moe.combine(s, out["xp"], ones, out["row_of"])
    want = (inp.x.float() * k).to(torch.bfloat16)
    assert torch.equal(y.cpu(), want)


@pytest.mark.parametrize("c", FFN_CASES, ids=_ids)
def test_expert_ffn_parity(moe, c):
    wl, inp = _case(*c, backward=False)
    s = moe.shape(wl.T, wl.d, wl.E, wl.k, wl.f)
    X, L, Wg, Wd, _ = inputs_np(inp)
    ref = oracle.forward(X, L, Wg, Wd, wl.k)
    ids, _ = moe.route(inp.logits.to(DEV), wl.k)
    disp = moe.dispatch(s, inp.x.to(DEV), ids)
    h, gu, o = moe.expert_ffn(s, disp["xp"], disp["counts"], inp.w_gu.to(DEV),
                              inp.w_down.to(DEV), save_gu=True)
    torch.cuda.synchronize()
    grow, orow = row_maps(to_np(disp["counts"]), to_np(disp["padded_offsets"]),
                          to_np(disp["offsets"]))
    assert_close(to_np(gu)[grow], ref["gu"][orow], "GU")
    assert_close(to_np(h)[grow], ref["h"][orow], "H")
    assert_close(to_np(o)[grow], ref["o"][orow], "O")
    # padding rows of every segment compute exactly zero
    pad = np.ones(int(to_np(disp["padded_offsets"])[-1]), dtype=bool)
    pad[grow] = False
    if pad.any():
        for t in (o, h, gu):
            assert not to_np(t)[:len(pad)][pad].any()


@pytest.mark.parametrize("c", FFN_CASES, ids=_ids)
def test_forward_parity(moe, c):
    wl, inp = _case(*c, backward=False)
    X, L, Wg, Wd, _ = inputs_np(inp)
    ref = oracle.forward(X, L, Wg, Wd, wl.k)
    y, ws, s = moe.forward(inp.x.to(DEV), inp.logits.to(DEV), inp.w_gu.to(DEV),
                           inp.w_down.to(DEV), wl.k, training=False)
    torch.cuda.synchronize()
    moe.check_device_status(ws)
    views = moe.workspace_views(s, False, ws)
    check_dispatch_exact(views, ref, inp.x, wl.k)
    np.testing.assert_allclose(to_np(views["w"]), ref["w"], rtol=W_REL, atol=0)
    assert_close(to_np(y), ref["y"], "Y")


BWD_CASES = [
    (512, 256, 8, 2, 512, 40, False),
    (300, 200, 5, 2, 200, 41, False),
    (512, 256, 32, 4, 256, 42, True),    # empty experts get dW = 0
    (96, 2880, 4, 2, 2880, 43, False),
    (200, 128, 1, 1, 64, 44, False),
    (1, 64, 4, 2, 64, 45, False),
    (1024, 256, 4, 2, 320, 46, False),   # SM-pair GEMMs (see FFN_CASES)
    (640, 256, 5, 2, 320, 52, False),    # 256 rows per expert, about half in 3 tiles
    (900, 200, 3, 2, 200, 47, False),
    (1024, 384, 4, 2, 576, 48, False),   # pairs with N tails in every GEMM (384, 576, 1152)
    (300, 64, 256, 16, 64, 49, False),   # the largest E and k
    (333, 72, 3, 2, 40, 50, False),      # K tail of 8 (d = 72) and N tails of 40 (f = 40)
    (600, 1536, 8, 4, 128, 51, False),   # combine and dX gather: 2 warps per row (d = 1536)
]


# The weight gradients of these cases hold experts of 1-140 rows whose dW is
# heavy-tailed (the largest element 13-20x the expert's rms). Rounding the exact result
# to bf16 alone costs up to 4.8e-2 of the 5e-2 rms element bound on dW_gu there, and
# 6.2e-2 (over the bound) on dW_down of the skewed case; the bf16 GEMM operands (H, G,
# dGU) add as much again, so no implementation with bf16 operands and bf16 dW meets that
# bound on them: a CPU emulation of the block's bf16 rounding points reproduces the
# kernel's errors exactly (5.848e-2 on dW_gu[4] of the first case, 6.820e-2 on
# dW_down[88] of the third). Their dW is checked below with the normwise bound and each
# element against its own magnitude; test_dw_rms_bound_small_experts records (strict
# xfail) that the rms element bound is missed.
DW_BF16_LIMITED = [(512, 256, 32, 4, 256, 42, True), (96, 2880, 4, 2, 2880, 43, False),
                   (300, 64, 256, 16, 64, 49, False)]


def _bwd_run(moe, c):
    wl, inp = _case(*c)
    X, L, Wg, Wd, DY = inputs_np(inp)
    ref = oracle.forward(X, L, Wg, Wd, wl.k)
    g = oracle.backward(DY, ref, Wg, Wd)
    w_gu, w_down = inp.w_gu.to(DEV), inp.w_down.to(DEV)
    y, ws, s = moe.forward(inp.x.to(DEV), inp.logits.to(DEV), w_gu, w_down, wl.k, training=True)
    dx, dw_gu, dw_down, dl = moe.backward(s, inp.dy.to(DEV), w_gu, w_down, ws, router_grad=True)
    torch.cuda.synchronize()
    moe.check_device_status(ws)
    return wl, ref, g, DY, (y, dx, dw_gu, dw_down, dl)


@pytest.mark.xfail(strict=True, reason="bf16 operands and bf16 dW cannot meet the rms element "
                   "bound on heavy-tailed experts of 1-140 rows (see DW_BF16_LIMITED)")
@pytest.mark.parametrize("which", ["dw_gu", "dw_down"])
@pytest.mark.parametrize("c", DW_BF16_LIMITED, ids=_ids)
def test_dw_rms_bound_small_experts(moe, c, which):
    _, _, g, _, out = _bwd_run(moe, c)
    got = out[2] if which == "dw_gu" else out[3]
    assert_close_experts(to_np(got), g[which], which)


@pytest.mark.parametrize("c", BWD_CASES, ids=_ids)
def test_backward_parity(moe, c):
    wl, ref, g, DY, (y, dx, dw_gu, dw_down, dl) = _bwd_run(moe, c)
    assert_close(to_np(y), ref["y"], "Y")
    assert_close(to_np(dx), g["dx"], "dX")
    dl_ref = oracle.router_backward(DY, ref)
    chosen = np.zeros(dl_ref.shape, dtype=bool)
    np.put_along_axis(chosen, ref["ids"].astype(np.int64), True, axis=1)
    if wl.k == 1:
        assert not dl.any()                         # weight 1 whatever the logit
    else:                                           # unchosen experts get exactly 0
        assert_close_selected(to_np(dl), dl_ref, chosen, "dlogits")
    floor = "ref" if c in DW_BF16_LIMITED else "rms"
    assert_close_experts(to_np(dw_gu), g["dw_gu"], "dW_gu", element_floor=floor)
    assert_close_experts(to_np(dw_down), g["dw_down"], "dW_down", element_floor=floor)
    empty = np.nonzero(ref["counts"] == 0)[0]
    for e in empty:
        assert not dw_gu[int(e)].any() and not dw_down[int(e)].any()


def test_no_tokens(moe):
    """T = 0: nothing routed; the backward still writes dW = 0 for every expert."""
    wl, inp = _case(0, 64, 4, 2, 64, 50, False)
    w_gu, w_down = inp.w_gu.to(DEV), inp.w_down.to(DEV)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    logits = torch.empty((0, 4), dtype=torch.float32, device=DEV)
    y, ws, s = moe.forward(x, logits, w_gu, w_down, 2, training=True)
    out = (torch.empty((0, 64), dtype=torch.bfloat16, device=DEV),
           torch.full_like(w_gu, 7.0), torch.full_like(w_down, 7.0))
    dx, dw_gu, dw_down = moe.backward(s, x, w_gu, w_down, ws, out=out)
    torch.cuda.synchronize()
    assert y.shape == (0, 64) and not dw_gu.any() and not dw_down.any()


def test_determinism(moe):
    """Two runs give bit-identical indices, outputs and gradients."""
    wl, inp = _case(700, 320, 16, 4, 200, 60, False)
    w_gu, w_down = inp.w_gu.to(DEV), inp.w_down.to(DEV)
    outs = []
    for _ in range(2):
        y, ws, s = moe.forward(inp.x.to(DEV), inp.logits.to(DEV), w_gu, w_down, wl.k,
                               training=True)
        dx, dwg, dwd, dl = moe.backward(s, inp.dy.to(DEV), w_gu, w_down, ws, router_grad=True)
        v = moe.workspace_views(s, True, ws)
        outs.append([t.clone() for t in (y, dx, dwg, dwd, dl, v["ids"], v["row_of"],
                                          v["tok_of"])])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
