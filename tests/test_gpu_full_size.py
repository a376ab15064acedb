"""Parity at the five workloads' full sizes, in the launch configuration the bench
times (moe_forward / moe_backward through the C ABI). Indices, counts and the
permutation are compared in full and bit-exactly; Y, dX and dW on seeded samples
that the oracle computes one at a time (whole token rows of Y and dX, whole rows
of dW_down and whole columns of dW_gu)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import check_dispatch_exact, to_np
from tolerance import W_REL, assert_close, assert_close_selected

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_route_gb300 as m
    return m


@pytest.mark.parametrize("name", ["tiny", "qwen3_moe", "gpt_oss_20b", "skewed", "long"])
def test_workload_full_size(moe, name):
    wl = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(wl)
    dev = "cuda"
    w_gu, w_down = inp.w_gu.to(dev), inp.w_down.to(dev)
    y, ws, s = moe.forward(inp.x.to(dev), inp.logits.to(dev), w_gu, w_down, wl.k,
                           training=wl.backward)
    if wl.backward:
        dx, dw_gu, dw_down, dl = moe.backward(s, inp.dy.to(dev), w_gu, w_down, ws,
                                              router_grad=True)
    torch.cuda.synchronize()
    moe.check_device_status(ws)

    logits = inp.logits.numpy()
    rid, rw = oracle.route(logits, wl.k)
    ref = oracle.dispatch(rid, wl.E)
    ref["ids"] = rid
    views = moe.workspace_views(s, wl.backward, ws)
    assert np.array_equal(to_np(views["ids"]), rid)
    np.testing.assert_allclose(to_np(views["w"]), rw, rtol=W_REL, atol=0)
    check_dispatch_exact(views, ref, inp.x, wl.k)
    if name == "skewed":
        # the top expert takes every token (the 1/k ceiling), and at least 4 are empty
        assert ref["counts"].max() == wl.T and (ref["counts"] == 0).sum() >= 4

    rng = np.random.default_rng(1000 + wl.seed)
    toks = np.unique(np.concatenate([[0, wl.T - 1], rng.choice(wl.T, size=40, replace=False)]))
    x64 = inp.x[torch.from_numpy(toks)].double().numpy()
    Wg, Wd = inp.w_gu, inp.w_down            # bf16 CPU tensors, widened per expert below

    class _PerExpert:
        def __init__(self, t):
            self.t = t

        def __getitem__(self, e):
            return self.t[int(e)].double().numpy()

    WG, WD = _PerExpert(Wg), _PerExpert(Wd)
    y_ref = np.stack([oracle.forward_token(x64[i], rid[t], rw[t], WG, WD)
                      for i, t in enumerate(toks)])
    assert_close(to_np(y[torch.from_numpy(toks).to(dev)]), y_ref, "Y (sampled tokens)")
    if not wl.backward:
        return
    dy64 = inp.dy[torch.from_numpy(toks)].double().numpy()
    dx_ref = np.stack([oracle.backward_token(x64[i], dy64[i], rid[t], rw[t], WG, WD)
                       for i, t in enumerate(toks)])
    assert_close(to_np(dx[torch.from_numpy(toks).to(dev)]), dx_ref, "dX (sampled tokens)")
    dl_ref = np.stack([oracle.router_backward_token(x64[i], dy64[i], rid[t], rw[t], wl.E, WG, WD)
                       for i, t in enumerate(toks)])
    chosen = np.zeros(dl_ref.shape, dtype=bool)
    np.put_along_axis(chosen, rid[toks].astype(np.int64), True, axis=1)
    assert_close_selected(to_np(dl[torch.from_numpy(toks).to(dev)]), dl_ref, chosen,
                          "dlogits (sampled tokens)")

    counts = ref["counts"]
    experts = {int(np.argmax(counts)), int(np.argmin(counts)), int(rng.integers(wl.E))}
    for e in sorted(experts):
        # the oracle needs only the expert's own token rows: pass that subset, re-indexed
        toks_e, _ = oracle.expert_members(rid, rw, e)
        sel = torch.from_numpy(toks_e)
        xs, dys = inp.x[sel].double().numpy(), inp.dy[sel].double().numpy()
        sub_ids, sub_w = rid[toks_e], rw[toks_e]
        # whole rows of dW_down [f x d] and whole columns of dW_gu [d x 2f]: every
        # sample spans the last (partial) tile along the other axis (d = 2880 = 11.25
        # tiles of 256), and the samples include rows and columns in the first and the
        # last tile along their own axis, plus a few at random
        rows = np.unique(np.concatenate([[0, 1, wl.f // 2, wl.f - 65, wl.f - 1],
                                         rng.integers(0, wl.f, size=3)]))
        cols = np.unique(np.concatenate([[0, wl.f - 1, wl.f, 2 * wl.f - 65, 2 * wl.f - 1],
                                         rng.integers(0, 2 * wl.f, size=3)]))
        dwd = oracle.dw_down_rows(e, rows, xs, dys, sub_ids, sub_w, WG, WD)
        dwg = oracle.dw_gu_cols(e, cols, xs, dys, sub_ids, sub_w, WG, WD)
        got_d = to_np(dw_down[e][torch.from_numpy(rows).to(dev)])
        got_g = to_np(dw_gu[e][:, torch.from_numpy(cols).to(dev)])
        if counts[e] == 0:
            assert not got_d.any() and not got_g.any()
        else:
            assert_close(got_d, dwd, f"dW_down[{e}] rows")
            assert_close(got_g, dwg, f"dW_gu[{e}] cols")
