"""Expert parallelism and token data parallelism across CPU ranks (gloo, no GPU).

The product's multi-rank logic -- moe_expert_layer_route_gb300.ep.ep_forward /
ep_backward (the count exchange, the row splits, the two all-to-all-v's of each
direction and the order of the stages around them) and dp.allreduce_weight_grads --
runs here in 2 and 4 spawned gloo ranks with the real torch.distributed collectives.
The per-rank device stages are replaced by CPU stand-ins written from the definitions
(the oracle's route, counting sort, SwiGLU experts and combine, and the regroup
permutation written out from its definition), so the test checks the exchange and
layout logic, and that every rank's Y, dX, router-logit gradient and its experts'
dW equal the single-process oracle on the whole batch. A third test makes one rank
never join the exchange: the other rank's collective fails on its process-group
timeout with an error on the host, and the process stays usable."""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import workloads


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


# ------------------------------------------------------------------ CPU stand-in stages
def _t(a, dtype=torch.float64):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype)


class OracleStages:
    """Each stage of ep_forward / ep_backward on CPU tensors in float64, from the
    oracle's functions and the layout definitions (see moe_ep_regroup's header)."""

    @staticmethod
    def route(logits, k):
        ids, w = oracle.route(logits.numpy(), k)
        return _t(ids, torch.int32), _t(w)

    @staticmethod
    def dispatch(s, x, ids):
        d = oracle.dispatch(ids.numpy(), s.E)
        xs = x.double()[torch.from_numpy(d["tok_of"])]
        return {"xs": xs, "counts": _t(d["counts"], torch.int32),
                "offsets": _t(d["offsets"], torch.int32), "row_of": _t(d["row_of"], torch.int64)}

    @staticmethod
    def regroup(s_loc, G, recv_counts, n, xr):
        rc = recv_counts.numpy().astype(np.int64)          # [G, El], source-major blocks
        El = rc.shape[1]
        cnt = rc.sum(axis=0)
        pad = np.concatenate([[0], np.cumsum((cnt + 127) // 128 * 128)])
        dest_of = np.empty(n, dtype=np.int64)
        i = 0
        for s_ in range(G):                                # received order: [s][e][rows]
            for e in range(El):
                before = rc[:s_, e].sum()                  # earlier sources of this expert
                for j in range(rc[s_, e]):
                    dest_of[i] = pad[e] + before + j
                    i += 1
        assert i == n
        R = int(pad[-1])
        xp = torch.zeros((R, xr.shape[1]), dtype=torch.float64)
        xp[torch.from_numpy(dest_of)] = xr.double()
        return {"xp": xp, "counts": _t(cnt, torch.int64), "pad": pad,
                "dest_of": torch.from_numpy(dest_of)}

    @staticmethod
    def check(reg):
        pass

    @staticmethod
    def expert_ffn(s_loc, xp, counts, w_gu, w_down, training):
        f = w_down.shape[1]
        pad = np.concatenate([[0], np.cumsum((counts.numpy() + 127) // 128 * 128)])
        h = torch.zeros((xp.shape[0], f), dtype=torch.float64)
        gu = torch.zeros((xp.shape[0], 2 * f), dtype=torch.float64)
        o = torch.zeros_like(xp)
        for e in range(len(counts)):
            lo, hi = int(pad[e]), int(pad[e] + counts[e])
            if hi > lo:
                r = oracle.swiglu_expert(xp[lo:hi].numpy(), w_gu[e].double().numpy(),
                                         w_down[e].double().numpy())
                gu[lo:hi], h[lo:hi], o[lo:hi] = _t(r["gu"]), _t(r["h"]), _t(r["o"])
        return h, gu, o

    @staticmethod
    def unregroup(s_loc, n, o, dest_of):
        return o[dest_of]

    @staticmethod
    def combine(s, ob, w, row_of):
        y = torch.zeros((s.T, ob.shape[1]), dtype=torch.float64)
        for j in range(s.k):
            wj = 1.0 if w is None else w[:, j:j + 1]
            y += wj * ob[row_of[:, j]]
        return y

    @staticmethod
    def grad_scatter(s, dy, w, ids, disp, ob, router_grad):
        dy = dy.double()
        row_of = disp["row_of"]
        gs = torch.zeros((s.T * s.k, s.d), dtype=torch.float64)
        for j in range(s.k):
            gs[row_of[:, j]] = w[:, j:j + 1] * dy
        dl = None
        if router_grad:
            fwd = {"ids": ids.numpy(), "w": w.numpy(), "row_of": row_of.numpy(),
                   "o": ob.numpy(), "counts": np.zeros(s.E)}
            dl = _t(oracle.router_backward(dy.numpy(), fwd))
        return gs, dl

    @staticmethod
    def expert_backward(s_loc, g, xp, gu, h, counts, w_gu, w_down):
        f = w_down.shape[1]
        pad = np.concatenate([[0], np.cumsum((counts.numpy() + 127) // 128 * 128)])
        dxp = torch.zeros_like(xp)
        dwg = torch.zeros(w_gu.shape, dtype=torch.float64)
        dwd = torch.zeros(w_down.shape, dtype=torch.float64)
        for e in range(len(counts)):
            lo, hi = int(pad[e]), int(pad[e] + counts[e])
            if hi == lo:
                continue
            Ge, He, GUe, Xe = (t[lo:hi].numpy() for t in (g, h, gu, xp))
            wd, wg = w_down[e].double().numpy(), w_gu[e].double().numpy()
            dg, du = oracle.swiglu_backward(Ge @ wd.T, GUe[:, :f], GUe[:, f:])
            dgu = np.concatenate([dg, du], axis=1)
            dwd[e], dwg[e] = _t(He.T @ Ge), _t(Xe.T @ dgu)
            dxp[lo:hi] = _t(dgu @ wg.T)
        return dxp, dwg, dwd


# ----------------------------------------------------------------------------- ranks
def _init(rank, world, port, timeout_s=60):
    import torch.distributed as dist
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=timeout_s))
    return dist


def _case(c):
    T, d, E, k, f, seed, zipf = c
    wl = workloads.Workload("ep", T=T, d=d, E=E, k=k, f=f, seed=seed, backward=True,
                            zipf_bias=zipf)
    return wl, workloads.make_inputs(wl)


def _ep_rank(rank, world, port, c, q):
    dist = _init(rank, world, port)
    try:
        from moe_expert_layer_route_gb300 import ep
        wl, inp = _case(c)
        El = wl.E // world
        toks = np.array_split(np.arange(wl.T), world)[rank]
        sel = torch.from_numpy(toks)
        ex = ep.DistExchange()
        w_gu = inp.w_gu[rank * El:(rank + 1) * El]
        w_down = inp.w_down[rank * El:(rank + 1) * El]
        y, ctx = ep.ep_forward(inp.x[sel], inp.logits[sel], w_gu, w_down, wl.k, wl.E, ex,
                               training=True, stages=OracleStages)
        dx, dwg, dwd, dl = ep.ep_backward(ctx, inp.dy[sel], w_gu, w_down, ex, router_grad=True,
                                          stages=OracleStages)
        q.put((rank, toks, y.numpy(), dx.numpy(), dl.numpy(), dwg.numpy(), dwd.numpy(),
               ctx.send_splits, ctx.recv_splits))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,c", [
    (2, (96, 64, 8, 2, 48, 0, False)),
    (4, (130, 40, 16, 4, 24, 1, False)),     # ragged token split, 4 experts per rank
    (4, (128, 32, 8, 3, 16, 2, True)),       # skewed: some ranks' experts get few or no rows
    (2, (64, 32, 4, 3, 16, 3, False)),       # k > experts per rank: a token sends 2 rows to a rank
])
def test_ep_over_gloo_ranks_matches_the_oracle(world, c):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ep_rank, args=(r, world, port, c, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl, inp = _case(c)
    X, L = inp.x.double().numpy(), inp.logits.numpy()
    Wg, Wd, DY = inp.w_gu.double().numpy(), inp.w_down.double().numpy(), inp.dy.double().numpy()
    ref = oracle.forward(X, L, Wg, Wd, wl.k)
    g = oracle.backward(DY, ref, Wg, Wd)
    dl_ref = oracle.router_backward(DY, ref)
    El = wl.E // world
    sent = np.zeros((world, world), dtype=np.int64)
    for rank, toks, y, dx, dl, dwg, dwd, send_splits, recv_splits in got:
        np.testing.assert_allclose(y, ref["y"][toks], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dx, g["dx"][toks], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dl, dl_ref[toks], rtol=1e-9, atol=1e-12)
        sl = slice(rank * El, (rank + 1) * El)
        np.testing.assert_allclose(dwg, g["dw_gu"][sl], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dwd, g["dw_down"][sl], rtol=1e-10, atol=1e-12)
        sent[rank] = send_splits
        # rows received by this rank = rows routed to its experts from every rank
        assert sum(recv_splits) == int(ref["counts"][sl].sum())
    assert sent.sum() == wl.T * wl.k


def _silent_rank(rank, world, port, q):
    dist = _init(rank, world, port, timeout_s=2)
    try:
        if rank == 1:       # never joins the exchange; leaves once rank 0 has reported
            q.get(timeout=60)
            return
        from moe_expert_layer_route_gb300 import ep
        wl, inp = _case((32, 32, 4, 2, 16, 4, False))
        ex = ep.DistExchange()
        try:
            ep.ep_forward(inp.x[:16], inp.logits[:16], inp.w_gu[:2], inp.w_down[:2], 2, 4, ex,
                          stages=OracleStages)
            outcome = "returned"
        except RuntimeError as err:  # the collective's timeout, raised on the host
            outcome = "raised: " + str(err)[:80]
        q.put(outcome)
        q.put("done")
    finally:
        try:
            dist.destroy_process_group()
        except Exception:  # noqa: BLE001 - the group may already be broken by the timeout
            pass


def test_a_rank_that_never_joins_fails_the_exchange_on_the_host():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_silent_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    outcome = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
    assert outcome.startswith("raised"), outcome
    assert procs[0].exitcode == 0


def _dp_rank(rank, world, port, c, q):
    dist = _init(rank, world, port)
    try:
        from moe_expert_layer_route_gb300 import dp
        wl, inp = _case(c)
        toks = np.array_split(np.arange(wl.T), world)[rank]
        X = inp.x.double().numpy()[toks]
        L = inp.logits.numpy()[toks]
        Wg, Wd = inp.w_gu.double().numpy(), inp.w_down.double().numpy()
        ref = oracle.forward(X, L, Wg, Wd, wl.k)
        g = oracle.backward(inp.dy.double().numpy()[toks], ref, Wg, Wd)
        # fp32 and bf16 gradient tensors, as the library writes them
        dwg32, dwd32 = _t(g["dw_gu"], torch.float32), _t(g["dw_down"], torch.float32)
        dwg16 = _t(g["dw_gu"], torch.float32).to(torch.bfloat16)
        dp.allreduce_weight_grads((dwg32, dwd32))
        dp.allreduce_weight_grads((dwg16,))
        q.put((rank, dwg32.numpy(), dwd32.numpy(), dwg16.float().numpy()))
    finally:
        dist.destroy_process_group()


def test_token_dp_allreduce_reproduces_the_whole_batch_weight_gradients():
    c = (100, 48, 8, 2, 32, 5, False)
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_dp_rank, args=(r, world, port, c, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl, inp = _case(c)
    ref = oracle.forward(inp.x.double().numpy(), inp.logits.numpy(), inp.w_gu.double().numpy(),
                         inp.w_down.double().numpy(), wl.k)
    g = oracle.backward(inp.dy.double().numpy(), ref, inp.w_gu.double().numpy(),
                        inp.w_down.double().numpy())
    for rank, dwg, dwd, dwg16 in got:
        np.testing.assert_allclose(dwg, g["dw_gu"], rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(dwd, g["dw_down"], rtol=1e-5, atol=1e-6)
        # bf16 shares summed in fp32 and rounded once: within two bf16 roundings
        err = np.abs(dwg16 - g["dw_gu"]).max() / np.abs(g["dw_gu"]).max()
        assert err < 2 * 2.0 ** -8
    assert np.array_equal(got[0][1], got[1][1])          # every rank holds the same sum
