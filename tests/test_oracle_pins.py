"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something it does not compute the same way:
hand-derived worked examples (tests/golden), closed forms, library routines for
special cases (a stable argsort, bincount, scipy's softmax, torch's silu), brute
force in pure-Python loops on tiny shapes, invariants of the method, and central
finite differences for the backward. The mutation tests at the end plant a
plausible mistake in a copy of the oracle and check that a pin catches it.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import moe_oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "route_dispatch_worked.json")


def _closed_form(expr) -> float:
    if isinstance(expr, (int, float)):
        return float(expr)
    return float(eval(expr.replace("ln3", "log(3)"), {"__builtins__": {}},
                      {"exp": math.exp, "log": math.log}))


def _tiny(T=24, d=16, E=6, k=3, f=8, seed=11, logit_scale=1.0):
    wl, inp = workloads.small_case(T, d, E, k, f, seed, logit_scale=logit_scale)
    return (inp.x.double().numpy(), inp.logits.numpy(), inp.w_gu.double().numpy(),
            inp.w_down.double().numpy(), inp.dy.double().numpy(), k)


# ------------------------------------------------------------------------ route pins
def test_route_golden_worked_examples():
    g = json.load(open(GOLDEN))
    for case in g["route"]:
        ids, w = oracle.route(np.array([case["logits"]], dtype=np.float32), case["k"])
        assert ids[0].tolist() == case["ids"], case["why"]
        want = np.array([_closed_form(s) for s in case["w"]])
        np.testing.assert_allclose(w[0], want, rtol=1e-14, atol=0, err_msg=case["why"])


def test_route_bias_golden_worked_examples():
    g = json.load(open(GOLDEN))
    for case in g["route_bias"]:
        ids, w = oracle.route(np.array([case["logits"]], dtype=np.float32), case["k"],
                              np.array(case["bias"], dtype=np.float32))
        assert ids[0].tolist() == case["ids"], case["why"]
        want = np.array([_closed_form(x) for x in case["w"]])
        np.testing.assert_allclose(w[0], want, rtol=1e-14, atol=0, err_msg=case["why"])


def test_route_bias_zero_and_dominance():
    rng = np.random.default_rng(31)
    logits = rng.standard_normal((200, 16)).astype(np.float32)
    for k in (1, 4):
        a = oracle.route(logits, k)
        b = oracle.route(logits, k, np.zeros(16, dtype=np.float32))
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    bias = (rng.integers(-4, 5, size=16) * 0.5).astype(np.float32)
    ids, w = oracle.route(logits, 4, bias)
    score = logits + bias
    for t in range(200):
        chosen = set(ids[t].tolist())
        for i in chosen:
            for j in set(range(16)) - chosen:
                assert score[t, i] > score[t, j] or (score[t, i] == score[t, j] and i < j)
        lc = logits[t, ids[t]].astype(np.float64)       # weights ignore the bias
        np.testing.assert_allclose(w[t], scipy.special.softmax(lc), rtol=1e-13)


def test_aux_stats_golden_worked_examples():
    g = json.load(open(GOLDEN))
    for case in g["aux"]:
        logits = np.array([[_closed_form(v) for v in row] for row in case["logits"]],
                          dtype=np.float64)
        st = oracle.aux_stats(logits, np.array(case["counts"]), case["k"])
        np.testing.assert_allclose(st["f"], [_closed_form(v) for v in case["f"]], atol=1e-15)
        np.testing.assert_allclose(st["P"], [_closed_form(v) for v in case["P"]], rtol=1e-14)
        assert abs(st["aux"] - _closed_form(case["aux"])) < 1e-14, case["why"]
    # the counts of the golden examples are what the router chooses on those logits
    for case in g["aux"]:
        logits = np.array([[_closed_form(v) for v in row] for row in case["logits"]],
                          dtype=np.float32)
        ids, _ = oracle.route(logits, case["k"])
        assert np.bincount(ids.ravel(), minlength=len(case["counts"])).tolist() == case["counts"]


def test_aux_loss_grad_matches_finite_differences():
    rng = np.random.default_rng(32)
    logits = rng.standard_normal((7, 5))
    counts = np.array([3, 0, 5, 4, 2])
    g = oracle.aux_loss_grad(logits, counts, 2)
    h = 1e-6
    for t in range(7):
        for e in range(5):
            lp, lm = logits.copy(), logits.copy()
            lp[t, e] += h
            lm[t, e] -= h
            fd = (oracle.aux_stats(lp, counts, 2)["aux"] - oracle.aux_stats(lm, counts, 2)["aux"]) / (2 * h)
            assert abs(fd - g[t, e]) <= 1e-8, (t, e, fd, g[t, e])
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-15)


def test_router_logits_sequential_fp32_definition():
    """The fp32 sum runs in index order: 2^24 + 1 rounds back to 2^24 (ties to even),
    so [1, 1, 1] . [2^24, 1, -2^24] is 0, not the exact 1; the reverse order gives 1."""
    x = np.ones((1, 3), dtype=np.float32)
    w = np.array([[2.0 ** 24, 1.0, -(2.0 ** 24)]], dtype=np.float32)
    assert oracle.router_logits(x, w)[0, 0] == 0.0
    assert oracle.router_logits(x, w[:, ::-1])[0, 0] == 1.0


def test_router_logits_addition_rounds_half_to_even():
    """(1 + 2^-7)^2 = 1 + 2^-6 + 2^-14 (exact: two 8-bit significands); added to 2^10 the
    2^-14 bit is half of the fp32 ulp there (2^-13), a tie that rounds to the even
    neighbour, so the logit is 2^10 + 1 + 2^-6."""
    v = np.float32(1 + 2.0 ** -7)
    x = np.array([[1.0, v]], dtype=np.float32)
    w = np.array([[2.0 ** 10, v]], dtype=np.float32)
    assert oracle.router_logits(x, w)[0, 0] == np.float32(2.0 ** 10 + 1 + 2.0 ** -6)
    assert oracle.router_logits(x, w * 2)[0, 0] == np.float32(2.0 ** 11 + 2 + 2.0 ** -5)


def test_router_logits_exact_on_integers_and_close_to_fp64():
    rng = np.random.default_rng(41)
    x = rng.integers(-8, 9, size=(20, 64)).astype(np.float32)     # small integers: every
    w = rng.integers(-8, 9, size=(6, 64)).astype(np.float32)      # partial sum is exact
    assert np.array_equal(oracle.router_logits(x, w), x.astype(np.int64) @ w.astype(np.int64).T)
    wl, inp = workloads.small_case(50, 256, 8, 2, 64, seed=42)
    xb = inp.x.float().numpy()
    wr = workloads.to_bf16(np.random.default_rng(43).standard_normal((8, 256)) * 0.05).float().numpy()
    got = oracle.router_logits(xb, wr).astype(np.float64)
    ref = xb.astype(np.float64) @ wr.astype(np.float64).T
    bound = 256 * 2.0 ** -24 * (np.abs(xb).astype(np.float64) @ np.abs(wr).astype(np.float64).T)
    assert (np.abs(got - ref) <= bound).all()
    assert not np.array_equal(got, ref.astype(np.float32))   # the order does show


def test_router_weight_backward_is_the_gemm_gradient():
    rng = np.random.default_rng(44)
    x, w = rng.standard_normal((9, 7)), rng.standard_normal((4, 7))
    dl = rng.standard_normal((9, 4))
    dw, dx = oracle.router_weight_backward(x, w, dl)
    assert dw.shape == (4, 7) and dx.shape == (9, 7)
    h = 1e-6
    loss = lambda xx, ww: (xx @ ww.T * dl).sum()
    for e in range(4):
        for i in range(7):
            wp, wm = w.copy(), w.copy()
            wp[e, i] += h
            wm[e, i] -= h
            assert abs((loss(x, wp) - loss(x, wm)) / (2 * h) - dw[e, i]) < 1e-7
    for t in range(9):
        for i in range(7):
            xp, xm = x.copy(), x.copy()
            xp[t, i] += h
            xm[t, i] -= h
            assert abs((loss(xp, w) - loss(xm, w)) / (2 * h) - dx[t, i]) < 1e-7


def test_route_selection_property():
    """Every chosen logit beats every unchosen one (ties: lower index wins)."""
    rng = np.random.default_rng(5)
    # coarse values so ties are frequent
    logits = rng.integers(-3, 4, size=(300, 12)).astype(np.float32) * np.float32(0.5)
    for k in (1, 2, 5, 12):
        ids, w = oracle.route(logits, k)
        for t in range(logits.shape[0]):
            chosen = set(ids[t].tolist())
            assert len(chosen) == k
            for i in chosen:
                for j in set(range(12)) - chosen:
                    li, lj = logits[t, i], logits[t, j]
                    assert li > lj or (li == lj and i < j)
            # slots in descending logit, equal logits in ascending index
            for a in range(k - 1):
                la, lb = logits[t, ids[t, a]], logits[t, ids[t, a + 1]]
                assert la > lb or (la == lb and ids[t, a] < ids[t, a + 1])
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-14)


def test_route_weights_match_library_softmax():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((64, 16)).astype(np.float32)
    for k in (1, 3, 8, 16):
        ids, w = oracle.route(logits, k)
        chosen = np.take_along_axis(logits, ids, 1).astype(np.float64)
        np.testing.assert_allclose(w, scipy.special.softmax(chosen, axis=1), rtol=1e-13)
    # k = E: the weights are the full softmax, read through the permutation
    ids, w = oracle.route(logits, 16)
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, ids, 1), rtol=1e-13)


def test_route_special_cases():
    logits = np.zeros((7, 9), dtype=np.float32)
    ids, w = oracle.route(logits, 4)
    assert (ids == np.arange(4)).all()
    np.testing.assert_allclose(w, 0.25, rtol=0, atol=0)
    rng = np.random.default_rng(7)
    ids, w = oracle.route(rng.standard_normal((50, 8)).astype(np.float32), 1)
    assert (w == 1.0).all()


def test_route_rejects_nonfinite():
    with pytest.raises(ValueError):
        oracle.route(np.array([[0.0, np.nan]], dtype=np.float32), 1)


# --------------------------------------------------------------------- dispatch pins
def test_dispatch_golden_worked_example():
    g = json.load(open(GOLDEN))["dispatch"]
    r = oracle.dispatch(np.array(g["ids"]), g["E"])
    for key in ("counts", "offsets", "row_of", "tok_of"):
        assert r[key].tolist() == g[key], key


@pytest.mark.parametrize("T,E,k,scale", [(1, 4, 1, 1.0), (37, 8, 2, 1.0), (500, 32, 4, 1.0),
                                         (300, 128, 8, 1.0), (200, 16, 4, 0.0)])
def test_dispatch_is_stable_sort_by_expert(T, E, k, scale):
    rng = np.random.default_rng(T + E)
    logits = (rng.standard_normal((T, E)) * scale).astype(np.float32)
    ids, _ = oracle.route(logits, k)
    r = oracle.dispatch(ids, E)
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    assert (r["counts"] == counts).all()
    assert r["counts"].sum() == T * k
    assert (r["offsets"] == np.concatenate([[0], np.cumsum(counts)])).all()
    perm = np.argsort(flat, kind="stable")           # library stable sort of the assignments
    assert (r["tok_of"] == perm // k).all()
    inv = np.empty_like(perm)
    inv[perm] = np.arange(T * k)
    assert (r["row_of"].reshape(-1) == inv).all()
    for e in range(E):                                 # ascending tokens inside a segment
        seg = r["tok_of"][r["offsets"][e]:r["offsets"][e + 1]]
        assert (np.diff(seg) > 0).all()


def test_identity_experts_return_k_times_x():
    """dispatch -> identity experts -> combine with unit weights = k * x."""
    x, logits, _, _, _, k = _tiny(T=40, E=7, k=3)
    ids, _ = oracle.route(logits, k)
    r = oracle.dispatch(ids, 7)
    xp = oracle.permute_rows(x, r["tok_of"])
    y = oracle.combine(xp, np.ones(ids.shape), r["row_of"])
    assert np.array_equal(y, k * x)


def test_combine_one_hot_weights_select_a_slot():
    rng = np.random.default_rng(8)
    o = rng.standard_normal((12, 5))
    row_of = rng.permutation(12).reshape(4, 3)
    for j in range(3):
        w = np.zeros((4, 3))
        w[:, j] = 1.0
        assert np.array_equal(oracle.combine(o, w, row_of), o[row_of[:, j]])


# ---------------------------------------------------------------------- expert pins
def _brute_force_y(x, logits, w_gu, w_down, k):
    """Pure-Python per-token loops: no matmul, no sort, no numpy reductions."""
    T, E = logits.shape
    d = x.shape[1]
    f = w_down.shape[1]
    y = [[0.0] * d for _ in range(T)]
    for t in range(T):
        row = [float(v) for v in logits[t]]
        chosen = []
        for _ in range(k):                     # k passes of "largest, lowest index on ties"
            best = None
            for e in range(E):
                if e in chosen:
                    continue
                if best is None or row[e] > row[best]:
                    best = e
            chosen.append(best)
        z = [math.exp(row[e] - row[chosen[0]]) for e in chosen]
        s = sum(z)
        for e, ze in zip(chosen, z):
            wt = ze / s
            h = []
            for c in range(f):
                g = sum(float(x[t, i]) * float(w_gu[e, i, c]) for i in range(d))
                u = sum(float(x[t, i]) * float(w_gu[e, i, f + c]) for i in range(d))
                h.append(g / (1.0 + math.exp(-g)) * u)
            for n in range(d):
                y[t][n] += wt * sum(h[c] * float(w_down[e, c, n]) for c in range(f))
    return np.array(y)


def test_forward_matches_pure_python_brute_force():
    x, logits, w_gu, w_down, _, k = _tiny(T=10, d=8, E=5, k=2, f=6)
    ref = _brute_force_y(x, logits, w_gu, w_down, k)
    y = oracle.forward(x, logits, w_gu, w_down, k)["y"]
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)


def test_single_expert_is_dense_swiglu_mlp():
    """E = 1, k = 1: the block is a dense SwiGLU MLP (torch silu, torch matmul)."""
    wl, inp = workloads.small_case(33, 24, 1, 1, 40, seed=3)
    y = oracle.forward(inp.x.double().numpy(), inp.logits.numpy(), inp.w_gu.double().numpy(),
                       inp.w_down.double().numpy(), 1)["y"]
    X, Wgu, Wd = inp.x.double(), inp.w_gu[0].double(), inp.w_down[0].double()
    ref = (torch.nn.functional.silu(X @ Wgu[:, :40]) * (X @ Wgu[:, 40:])) @ Wd
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-15)


def test_swiglu_closed_form_with_identity_weights():
    """W_gate = c*I, W_up = I, W_down = I (d = f): y = sum_j w_j * silu(c x) * x."""
    d = 12
    rng = np.random.default_rng(9)
    x = rng.standard_normal((20, d))
    logits = rng.standard_normal((20, 3)).astype(np.float32)
    c = 1.7
    w_gu = np.concatenate([c * np.eye(d), np.eye(d)], axis=1)[None].repeat(3, 0)
    w_down = np.eye(d)[None].repeat(3, 0)
    out = oracle.forward(x, logits, w_gu, w_down, 2)
    expect = (c * x) / (1.0 + np.exp(-c * x)) * x            # same for every expert
    np.testing.assert_allclose(out["y"], expect, rtol=1e-13)


def test_empty_experts_are_legal():
    x, logits, w_gu, w_down, dy, k = _tiny(T=16, E=6, k=2)
    logits[:, 4:] -= 100.0                                   # experts 4, 5 never chosen
    out = oracle.forward(x, logits, w_gu, w_down, k)
    assert out["counts"][4] == 0 and out["counts"][5] == 0
    g = oracle.backward(dy, out, w_gu, w_down)
    assert not g["dw_gu"][4:].any() and not g["dw_down"][4:].any()


# --------------------------------------------------------------------- backward pins
def _loss(x, logits, w_gu, w_down, k, dy):
    return float((oracle.forward(x, logits, w_gu, w_down, k)["y"] * dy).sum())


def test_backward_matches_central_finite_differences():
    x, logits, w_gu, w_down, dy, k = _tiny(T=8, d=16, E=4, k=2, f=32, seed=12)
    # scale weights up so the SwiGLU is well outside its linear region
    w_gu = w_gu * 20.0
    w_down = w_down * 20.0
    out = oracle.forward(x, logits, w_gu, w_down, k)
    grads = oracle.backward(dy, out, w_gu, w_down)
    rng = np.random.default_rng(13)
    h = 1e-6
    for name, arr, grad in (("x", x, grads["dx"]), ("w_gu", w_gu, grads["dw_gu"]),
                            ("w_down", w_down, grads["dw_down"])):
        flat = arr.reshape(-1)
        for idx in rng.choice(flat.size, size=60, replace=False):
            old = flat[idx]
            flat[idx] = old + h
            lp = _loss(x, logits, w_gu, w_down, k, dy)
            flat[idx] = old - h
            lm = _loss(x, logits, w_gu, w_down, k, dy)
            flat[idx] = old
            fd = (lp - lm) / (2 * h)
            an = grad.reshape(-1)[idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, an)


def test_backward_directional_derivative():
    """<dY, J v> = <J^T dY, v> along a random direction in (x, W_gu, W_down)."""
    x, logits, w_gu, w_down, dy, k = _tiny(T=12, d=16, E=4, k=2, f=24, seed=14)
    out = oracle.forward(x, logits, w_gu, w_down, k)
    g = oracle.backward(dy, out, w_gu, w_down)
    rng = np.random.default_rng(15)
    vx, vg, vd = (rng.standard_normal(a.shape) for a in (x, w_gu, w_down))
    h = 1e-5
    lp = _loss(x + h * vx, logits, w_gu + h * vg, w_down + h * vd, k, dy)
    lm = _loss(x - h * vx, logits, w_gu - h * vg, w_down - h * vd, k, dy)
    fd = (lp - lm) / (2 * h)
    an = (g["dx"] * vx).sum() + (g["dw_gu"] * vg).sum() + (g["dw_down"] * vd).sum()
    assert abs(fd - an) <= 1e-7 * max(1.0, abs(fd))


def test_router_backward_matches_finite_differences():
    """d<dY, Y>/d logits by central differences. The logits are multiples of 2^-6 and
    the step is 2^-12, so every perturbed fp32 logit is exact and no top-k choice
    changes (the gaps between distinct logits are at least 2^-6)."""
    x, _, w_gu, w_down, dy, k = _tiny(T=6, d=12, E=5, k=3, f=10, seed=17)
    rng = np.random.default_rng(18)
    logits = (rng.integers(-128, 128, size=(6, 5)) / 64.0).astype(np.float32)
    out = oracle.forward(x, logits, w_gu, w_down, k)
    dl = oracle.router_backward(dy, out)
    h = 2.0 ** -12
    for t in range(6):
        for e in range(5):
            lp, lm = logits.copy(), logits.copy()
            lp[t, e] += np.float32(h)
            lm[t, e] -= np.float32(h)
            fd = (_loss(x, lp, w_gu, w_down, k, dy) - _loss(x, lm, w_gu, w_down, k, dy)) / (2 * h)
            assert abs(fd - dl[t, e]) <= 1e-6 * max(1.0, abs(fd)), (t, e, fd, dl[t, e])
    chosen = np.zeros_like(dl, dtype=bool)
    np.put_along_axis(chosen, out["ids"].astype(np.int64), True, axis=1)
    assert not dl[~chosen].any()
    np.testing.assert_allclose(dl.sum(axis=1), 0.0, atol=1e-12)   # softmax Jacobian rows sum to 0


def test_router_backward_k1_is_zero():
    """With one expert per token the weight is 1 whatever the logit: no gradient."""
    x, logits, w_gu, w_down, dy, _ = _tiny(T=9, d=8, E=4, k=1, f=8, seed=19)
    out = oracle.forward(x, logits, w_gu, w_down, 1)
    assert not oracle.router_backward(dy, out).any()


# ----------------------------------------------- one-at-a-time outputs vs the full oracle
def test_single_output_helpers_agree_with_full_oracle():
    x, logits, w_gu, w_down, dy, k = _tiny(T=30, d=16, E=5, k=2, f=12, seed=16)
    out = oracle.forward(x, logits, w_gu, w_down, k)
    g = oracle.backward(dy, out, w_gu, w_down)
    for t in (0, 7, 29):
        np.testing.assert_allclose(
            oracle.forward_token(x[t], out["ids"][t], out["w"][t], w_gu, w_down), out["y"][t],
            rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(
            oracle.backward_token(x[t], dy[t], out["ids"][t], out["w"][t], w_gu, w_down),
            g["dx"][t], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(
            oracle.router_backward_token(x[t], dy[t], out["ids"][t], out["w"][t], 5, w_gu, w_down),
            oracle.router_backward(dy, out)[t], rtol=1e-12, atol=1e-15)
    for e in range(5):
        rows = np.array([0, 3, 11])
        np.testing.assert_allclose(
            oracle.dw_down_rows(e, rows, x, dy, out["ids"], out["w"], w_gu, w_down),
            g["dw_down"][e][rows], rtol=1e-12, atol=1e-15)
        cols = np.array([0, 5, 12, 23])
        np.testing.assert_allclose(
            oracle.dw_gu_cols(e, cols, x, dy, out["ids"], out["w"], w_gu, w_down),
            g["dw_gu"][e][:, cols], rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------- planted mistakes (CPU)
def _swapped_gate_up(xr, w_gu_e, w_down_e):
    w_gu_e = np.asarray(w_gu_e, dtype=np.float64)
    f = np.asarray(w_down_e).shape[0]
    gu = np.asarray(xr, dtype=np.float64) @ w_gu_e
    g, u = gu[:, f:], gu[:, :f]                                  # gate and up swapped
    h = g / (1 + np.exp(-g)) * u
    return {"gu": gu, "h": h, "o": h @ np.asarray(w_down_e, dtype=np.float64)}


def _reversed_down_rows(xr, w_gu_e, w_down_e):
    w_gu_e = np.asarray(w_gu_e, dtype=np.float64)
    f = np.asarray(w_down_e).shape[0]
    gu = np.asarray(xr, dtype=np.float64) @ w_gu_e
    g, u = gu[:, :f], gu[:, f:]
    h = g / (1 + np.exp(-g)) * u
    wd = np.asarray(w_down_e, dtype=np.float64)
    return {"gu": gu, "h": h, "o": h @ wd[::-1]}                  # wrong row index of W_down


def _route_ties_high(logits, k):
    logits = np.asarray(logits, dtype=np.float32)
    order = np.argsort(-logits[:, ::-1], axis=1, kind="stable")
    ids = (logits.shape[1] - 1 - order[:, :k]).astype(np.int32)  # ties -> higher index
    chosen = np.take_along_axis(logits, ids, 1).astype(np.float64)
    z = np.exp(chosen - chosen[:, :1])
    return ids, z / z.sum(1, keepdims=True)


def _bwd_missing_term(dh, g, u):
    s = 1 / (1 + np.exp(-g))
    return dh * u * s, dh * g * s                               # drops (1 + g(1 - s))


def _router_bwd_uncentred(dy, fwd):
    dy = np.asarray(dy, dtype=np.float64)
    dw = np.einsum("td,tjd->tj", dy, np.asarray(fwd["o"], dtype=np.float64)[fwd["row_of"]])
    dl = np.zeros((dy.shape[0], int(fwd["counts"].shape[0])))
    np.put_along_axis(dl, fwd["ids"].astype(np.int64), fwd["w"] * dw, axis=1)  # no centring
    return dl


@pytest.mark.parametrize("mutant", ["swapped_gate_up", "reversed_down_rows", "ties_high",
                                    "bwd_missing_term", "router_uncentred"])
def test_pins_catch_planted_mistakes(monkeypatch, mutant):
    caught = False
    if mutant == "swapped_gate_up":
        monkeypatch.setattr(moe_oracle, "swiglu_expert", _swapped_gate_up)
        try:
            test_single_expert_is_dense_swiglu_mlp()
        except AssertionError:
            caught = True
    elif mutant == "reversed_down_rows":
        monkeypatch.setattr(moe_oracle, "swiglu_expert", _reversed_down_rows)
        try:
            test_forward_matches_pure_python_brute_force()
        except AssertionError:
            caught = True
    elif mutant == "ties_high":
        monkeypatch.setattr(moe_oracle, "route", _route_ties_high)
        monkeypatch.setattr(oracle, "route", _route_ties_high)
        try:
            test_route_golden_worked_examples()
        except AssertionError:
            caught = True
    elif mutant == "bwd_missing_term":
        monkeypatch.setattr(moe_oracle, "swiglu_backward", _bwd_missing_term)
        try:
            test_backward_matches_central_finite_differences()
        except AssertionError:
            caught = True
    elif mutant == "router_uncentred":
        monkeypatch.setattr(oracle, "router_backward", _router_bwd_uncentred)
        try:
            test_router_backward_matches_finite_differences()
        except AssertionError:
            caught = True
    assert caught, f"no pin caught the planted mistake {mutant}"
