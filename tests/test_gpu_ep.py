"""Expert parallelism on one GPU: G emulated ranks through the library's CUDA stages.

Each rank is a host thread running moe_expert_layer_route_gb300.ep.ep_forward /
ep_backward on its own share of the tokens and its own E/G experts, with per-rank
buffers on the one GPU. The exchanges are stood in for by a host rendezvous: at each
all-to-all every thread synchronises its stream, publishes its pieces, waits for the
others, and copies what it receives (device-to-device copies). No kernel waits on
another rank; the threads only meet on the host between launches.

Checked against the CPU oracle on the whole batch: every rank's Y, dX and
router-logit gradient, and the weight gradients of its experts, with the bounds of
tests/tolerance.py; the stage calls themselves (compact dispatch, regroup, unregroup)
bit-exactly against their definitions; and a regroup given counts that do not add up
writes nothing and reports it through the device status word."""
import threading

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import to_np
from tolerance import assert_close, assert_close_experts, assert_close_selected

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_route_gb300 as m
    assert torch.cuda.is_available()
    return m


class _Rendezvous:
    def __init__(self, G):
        self.G = G
        self.barrier = threading.Barrier(G, timeout=300)
        self.slots = [None] * G


class ThreadExchange:
    """The two exchanges of ep.DistExchange between G threads of one process."""

    def __init__(self, rv: _Rendezvous, rank: int):
        self.rv, self.rank, self.G = rv, rank, rv.G

    def _all_to_all(self, pieces):
        torch.cuda.current_stream().synchronize()      # the pieces are computed
        self.rv.slots[self.rank] = pieces
        self.rv.barrier.wait()
        got = [self.rv.slots[s][self.rank].clone() for s in range(self.G)]
        torch.cuda.current_stream().synchronize()      # copied before senders reuse them
        self.rv.barrier.wait()
        return got

    def counts(self, send):
        return torch.stack(self._all_to_all([send[r] for r in range(self.G)]))

    def rows(self, buf, send_splits, recv_splits):
        got = self._all_to_all(list(torch.split(buf, send_splits)))
        assert [g.shape[0] for g in got] == list(recv_splits)
        return torch.cat(got) if got else buf[:0]


def _run_ranks(G, fn):
    rv = _Rendezvous(G)
    out, errs = [None] * G, []

    def body(r):
        try:
            out[r] = fn(r, ThreadExchange(rv, r))
        except BaseException as e:  # noqa: BLE001 - re-raised in the test's thread
            errs.append(e)
            rv.barrier.abort()

    th = [threading.Thread(target=body, args=(r,)) for r in range(G)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    if errs:
        raise errs[0]
    return out


def _case(c):
    T, d, E, k, f, seed, zipf = c
    wl = workloads.Workload("ep", T=T, d=d, E=E, k=k, f=f, seed=seed, backward=True,
                            zipf_bias=zipf)
    return wl, workloads.make_inputs(wl)


# (G, (T, d, E, k, f, seed, zipf)); every expert here has >= 256 rows except in the
# skewed case, whose small experts' dW is checked as in the single-GPU parity tests
EP_CASES = [
    (2, (1024, 256, 8, 2, 512, 80, False)),
    (4, (2048, 256, 16, 4, 320, 81, False)),   # SM-pair GEMMs on every rank
    (4, (1202, 200, 8, 3, 136, 82, False)),    # ragged token split, K and N tails
    (2, (512, 2880, 4, 2, 2880, 83, False)),   # gpt-oss-20b-like widths
    (4, (2048, 256, 32, 4, 256, 84, True)),    # skewed: empty experts on some ranks
    (2, (256, 64, 4, 3, 64, 85, False)),       # k = 3 > 2 experts per rank
    (1, (512, 128, 4, 2, 64, 86, False)),      # one rank: no exchange partner
]


def _ids(p):
    G, c = p
    return f"G{G}_T{c[0]}_d{c[1]}_E{c[2]}_k{c[3]}_f{c[4]}" + ("_zipf" if c[6] else "")


@pytest.mark.parametrize("p", EP_CASES, ids=_ids)
def test_ep_emulated_ranks_match_the_oracle(moe, p):
    from moe_expert_layer_route_gb300 import ep
    G, c = p
    wl, inp = _case(c)
    El = wl.E // G
    splits = np.array_split(np.arange(wl.T), G)

    def rank_fn(r, ex):
        sel = torch.from_numpy(splits[r])
        w_gu = inp.w_gu[r * El:(r + 1) * El].to(DEV)
        w_down = inp.w_down[r * El:(r + 1) * El].to(DEV)
        y, ctx = ep.ep_forward(inp.x[sel].to(DEV), inp.logits[sel].to(DEV), w_gu, w_down, wl.k,
                               wl.E, ex, training=True)
        dx, dwg, dwd, dl = ep.ep_backward(ctx, inp.dy[sel].to(DEV), w_gu, w_down, ex,
                                          router_grad=True)
        torch.cuda.synchronize()
        return [to_np(t) for t in (y, dx, dl, dwg, dwd)]

    got = _run_ranks(G, rank_fn)
    X, L = inp.x.double().numpy(), inp.logits.numpy()
    Wg, Wd, DY = inp.w_gu.double().numpy(), inp.w_down.double().numpy(), inp.dy.double().numpy()
    ref = oracle.forward(X, L, Wg, Wd, wl.k)
    g = oracle.backward(DY, ref, Wg, Wd)
    dl_ref = oracle.router_backward(DY, ref)
    y = np.concatenate([o[0] for o in got])
    dx = np.concatenate([o[1] for o in got])
    dl = np.concatenate([o[2] for o in got])
    assert_close(y, ref["y"], "Y (EP)")
    assert_close(dx, g["dx"], "dX (EP)")
    chosen = np.zeros(dl_ref.shape, dtype=bool)
    np.put_along_axis(chosen, ref["ids"].astype(np.int64), True, axis=1)
    assert_close_selected(dl, dl_ref, chosen, "dlogits (EP)")
    floor = "ref" if c[6] else "rms"   # skewed: experts of a few rows (see DW_BF16_LIMITED)
    dwg = np.concatenate([o[3] for o in got])
    dwd = np.concatenate([o[4] for o in got])
    assert_close_experts(dwg, g["dw_gu"], "dW_gu (EP)", element_floor=floor)
    assert_close_experts(dwd, g["dw_down"], "dW_down (EP)", element_floor=floor)


def test_ep_dispatch_is_the_compact_counting_sort(moe):
    wl, inp = _case((777, 136, 12, 3, 64, 87, False))
    s = moe.shape(wl.T, wl.d, wl.E, wl.k, wl.f)
    x = inp.x.to(DEV)
    ids, _ = moe.route(inp.logits.to(DEV), wl.k)
    disp = moe.ep_dispatch(s, x, ids)
    torch.cuda.synchronize()
    rid, _ = oracle.route(inp.logits.numpy(), wl.k)
    ref = oracle.dispatch(rid, wl.E)
    assert np.array_equal(to_np(disp["counts"]), ref["counts"])
    assert np.array_equal(to_np(disp["offsets"]), ref["offsets"])
    assert np.array_equal(to_np(disp["row_of"]), ref["row_of"])
    assert torch.equal(disp["xs"].cpu(), inp.x[torch.from_numpy(ref["tok_of"])])


def _regroup_definition(rc: np.ndarray):
    """dest_of and the padded segment starts of a received layout, from the definition."""
    G, El = rc.shape
    cnt = rc.sum(axis=0)
    pad = np.concatenate([[0], np.cumsum((cnt + 127) // 128 * 128)])
    dest = []
    for s in range(G):
        for e in range(El):
            dest += [pad[e] + rc[:s, e].sum() + j for j in range(rc[s, e])]
    return np.asarray(dest, dtype=np.int64), cnt, pad


@pytest.mark.parametrize("G,El,d", [(3, 5, 72), (4, 64, 256), (2, 1, 2880), (8, 32, 64)])
def test_ep_regroup_and_unregroup_follow_their_definition(moe, G, El, d):
    rng = np.random.default_rng(G * 100 + El)
    rc = rng.integers(0, 300, size=(G, El)).astype(np.int32)
    rc[rng.random((G, El)) < 0.2] = 0                 # empty blocks
    n = int(rc.sum())
    s_loc = moe.ep_local_shape(moe.shape(max(1, -(-n // G)), d, El * G, 1, 64), G)
    s_loc.T = max(s_loc.T, n)                         # room for every received row
    xr = workloads.to_bf16(rng.standard_normal((n, d), dtype=np.float32)).to(DEV)
    reg = moe.ep_regroup(s_loc, G, torch.from_numpy(rc).to(DEV), n, xr)
    torch.cuda.synchronize()
    moe.check_device_status(reg["ws"])
    dest, cnt, pad = _regroup_definition(rc.astype(np.int64))
    assert np.array_equal(to_np(reg["dest_of"]), dest)
    assert np.array_equal(to_np(reg["counts"]), cnt)
    assert np.array_equal(to_np(reg["padded_offsets"]), pad)
    xp = reg["xp"]
    assert torch.equal(xp[torch.from_numpy(dest).to(DEV)], xr)
    used = np.zeros(int(pad[-1]), dtype=bool)
    used[dest] = True
    assert not xp[:int(pad[-1])][torch.from_numpy(~used).to(DEV)].any()   # padding rows zero
    back = moe.ep_unregroup(s_loc, n, xp, reg["dest_of"])
    assert torch.equal(back, xr)


def test_ep_regroup_rejects_counts_that_do_not_add_up(moe):
    G, El, d = 2, 3, 64
    rc = torch.tensor([[5, 0, 7], [1, 2, 3]], dtype=torch.int32, device=DEV)
    s_loc = moe.ep_local_shape(moe.shape(32, d, G * El, 2, 64), G)
    xr = torch.ones((17, d), dtype=torch.bfloat16, device=DEV)
    reg = moe.ep_regroup(s_loc, G, rc, 17, xr)        # the counts add up to 18, not 17
    torch.cuda.synchronize()
    with pytest.raises(moe.MoEError) as ex:
        moe.check_device_status(reg["ws"])
    assert ex.value.status == -1                      # MOE_ERR_INVALID_ARG
    moe.check_device_status(reg["ws"])                # cleared; the context is usable
    good = moe.ep_regroup(s_loc, G, rc, 18, torch.ones((18, d), dtype=torch.bfloat16,
                                                       device=DEV))
    torch.cuda.synchronize()
    moe.check_device_status(good["ws"])
