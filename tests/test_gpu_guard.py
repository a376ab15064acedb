"""Guard regions around every buffer the library writes (the bounds check that stands
in for a memory checker).

Each output, workspace and scratch buffer handed to the C ABI sits inside a larger
allocation whose slack before and after it is filled with a sentinel byte. After the
calls (the stages one by one, the whole forward and backward, the router GEMM and its
gradient) every slack byte must still hold the sentinel: no kernel, and no TMA store
clipped at a tensor edge, writes outside the buffer it was given. The shapes are the
edge cases of the tile schedule: ragged M, N and K tails, the largest E and k, empty
experts, one token and no token."""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

PAD = 4096          # slack bytes on each side (a multiple of the 256-byte alignment)
SENTINEL = 0xA5
DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import moe_expert_layer_route_gb300 as m
    assert torch.cuda.is_available()
    return m


class Guarded:
    """A buffer of `nbytes` with sentinel-filled slack on both sides."""

    def __init__(self, nbytes: int, name: str):
        self.n = int(nbytes)
        self.name = name
        self.buf = torch.full((PAD + self.n + PAD,), SENTINEL, dtype=torch.uint8, device=DEV)

    def tensor(self, dtype, shape):
        return self.buf[PAD:PAD + self.n].view(dtype).view(*shape)

    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr() + PAD)

    def check(self):
        lo, hi = self.buf[:PAD], self.buf[PAD + self.n:]
        bad_lo = int((lo != SENTINEL).sum())
        bad_hi = int((hi != SENTINEL).sum())
        assert bad_lo == 0 and bad_hi == 0, (
            f"{self.name}: {bad_lo} bytes written before and {bad_hi} after the buffer")


def _g(nbytes, name, reg):
    g = Guarded(max(int(nbytes), 16), name)
    reg.append(g)
    return g


def _ok(rc, where):
    assert rc == 0, f"{where} returned {rc}"


CASES = [
    (300, 200, 5, 2, 200, 1, False),     # ragged K (200 = 3*64 + 8) and N tails
    (333, 72, 3, 2, 40, 2, False),       # K tail of 8, N tails of 40
    (1024, 384, 4, 2, 576, 3, False),    # SM pairs with N tails in every GEMM
    (300, 64, 256, 16, 64, 4, False),    # the largest E and k
    (512, 256, 32, 4, 256, 5, True),     # skewed: empty experts, one expert gets every token
    (96, 2880, 4, 2, 2880, 6, False),    # gpt-oss-20b-like widths (11.25 tiles of 256)
    (1, 64, 4, 2, 64, 7, False),         # one token
    (0, 64, 4, 2, 64, 8, False),         # no token
]


def _ids(c):
    return "T{}_d{}_E{}_k{}_f{}".format(*c[:5]) + ("_zipf" if c[6] else "")


@pytest.mark.parametrize("c", CASES, ids=_ids)
def test_no_write_outside_any_buffer(moe, c):
    T, d, E, k, f, seed, zipf = c
    wl = workloads.Workload("guard", T=T, d=d, E=E, k=k, f=f, seed=seed, backward=True,
                            zipf_bias=zipf)
    inp = workloads.make_inputs(wl)
    L = moe.lib()
    s = moe.shape(T, d, E, k, f)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    R = moe.padded_rows(s)
    x, logits = inp.x.to(DEV), inp.logits.to(DEV)
    w_gu, w_down, dy = inp.w_gu.to(DEV), inp.w_down.to(DEV), inp.dy.to(DEV)
    w_r = workloads.make_router_weight(wl).to(DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    reg = []

    # ---- the stages one by one, each output in its own guarded buffer
    ws0 = _g(L.moe_workspace_size(s, 0), "stage workspace", reg)
    ids, w = _g(T * k * 4, "ids", reg), _g(T * k * 4, "w", reg)
    _ok(L.moe_route(s, p(logits), ids.ptr(), w.ptr(), None, st), "moe_route")
    xp = _g(R * d * 2, "xp", reg)
    counts, offsets = _g(E * 4, "counts", reg), _g((E + 1) * 4, "offsets", reg)
    padded, row_of = _g((E + 1) * 4, "padded_offsets", reg), _g(T * k * 4, "row_of", reg)
    tok_of = _g(R * 4, "tok_of", reg)
    _ok(L.moe_dispatch(s, p(x), ids.ptr(), xp.ptr(), counts.ptr(), offsets.ptr(), padded.ptr(),
                       row_of.ptr(), tok_of.ptr(), ws0.ptr(), ws0.n, st), "moe_dispatch")
    h, gu, o = _g(R * f * 2, "h", reg), _g(R * 2 * f * 2, "gu", reg), _g(R * d * 2, "o", reg)
    _ok(L.moe_expert_ffn(s, xp.ptr(), counts.ptr(), p(w_gu), p(w_down), h.ptr(), gu.ptr(),
                         o.ptr(), ws0.ptr(), ws0.n, st), "moe_expert_ffn")
    y0 = _g(T * d * 2, "y (combine)", reg)
    _ok(L.moe_combine(s, o.ptr(), w.ptr(), row_of.ptr(), y0.ptr(), st), "moe_combine")
    xp2 = _g(R * d * 2, "xp (no-alloc dispatch)", reg)
    c2, o2 = _g(E * 4, "counts (no-alloc)", reg), _g((E + 1) * 4, "offsets (no-alloc)", reg)
    p2, r2 = _g((E + 1) * 4, "padded (no-alloc)", reg), _g(T * k * 4, "row_of (no-alloc)", reg)
    t2 = _g(R * 4, "tok_of (no-alloc)", reg)
    _ok(L.moe_dispatch_noalloc(s, p(x), ids.ptr(), xp2.ptr(), c2.ptr(), o2.ptr(), p2.ptr(),
                               r2.ptr(), t2.ptr(), st), "moe_dispatch_noalloc")

    # ---- the whole block, forward and backward, with the router-logit gradient
    ws = _g(L.moe_workspace_size(s, 1), "forward workspace", reg)
    y = _g(T * d * 2, "y", reg)
    _ok(L.moe_forward(s, p(x), p(logits), p(w_gu), p(w_down), y.ptr(), 1, None, ws.ptr(), ws.n,
                      st), "moe_forward")
    sc = _g(L.moe_backward_scratch_size(s), "backward scratch", reg)
    dx, dwg = _g(T * d * 2, "dx", reg), _g(E * d * 2 * f * 2, "dw_gu", reg)
    dwd, dl = _g(E * f * d * 2, "dw_down", reg), _g(T * E * 4, "dlogits", reg)
    _ok(L.moe_backward(s, p(dy), p(w_gu), p(w_down), ws.ptr(), ws.n, dx.ptr(), dwg.ptr(),
                       dwd.ptr(), dl.ptr(), sc.ptr(), sc.n, st), "moe_backward")

    # ---- the router GEMM in front, its gradient, and the load-balancing statistics
    wsr = _g(L.moe_workspace_size(s, 1), "router forward workspace", reg)
    yr, lg = _g(T * d * 2, "y (router)", reg), _g(T * E * 4, "logits (router)", reg)
    aux = _g((2 * E + 1) * 4, "aux_stats", reg)
    bias = torch.from_numpy(workloads.zipf_bias(E)).to(DEV)
    opts = moe._RouteOptions(p(bias), aux.ptr())
    _ok(L.moe_forward_router(s, p(x), p(w_r), lg.ptr(), p(w_gu), p(w_down), yr.ptr(), 1,
                             ctypes.byref(opts), wsr.ptr(), wsr.n, st), "moe_forward_router")
    scr = _g(L.moe_backward_scratch_size(s), "router backward scratch", reg)
    dxr, dlr = _g(T * d * 2, "dx (router)", reg), _g(T * E * 4, "dlogits (router)", reg)
    dwg2, dwd2 = _g(E * d * 2 * f * 2, "dw_gu (router)", reg), _g(E * f * d * 2, "dw_down (r)", reg)
    _ok(L.moe_backward(s, p(dy), p(w_gu), p(w_down), wsr.ptr(), wsr.n, dxr.ptr(), dwg2.ptr(),
                       dwd2.ptr(), dlr.ptr(), scr.ptr(), scr.n, st), "moe_backward (router)")
    fwd_counts = moe.workspace_views(s, True, wsr.tensor(torch.uint8, (wsr.n,)))["counts"]
    _ok(L.moe_aux_loss_backward(s, lg.ptr(), p(fwd_counts), ctypes.c_float(0.01), dlr.ptr(), st),
        "moe_aux_loss_backward")
    rs = _g(L.moe_router_backward_scratch_size(s), "router GEMM scratch", reg)
    dwr = _g(E * d * 4, "dw_router", reg)
    _ok(L.moe_router_backward(s, p(x), p(w_r), dlr.ptr(), dxr.ptr(), dwr.ptr(), rs.ptr(), rs.n,
                              st), "moe_router_backward")
    ids3, w3 = _g(T * k * 4, "ids (router route)", reg), _g(T * k * 4, "w (router route)", reg)
    lg3 = _g(T * E * 4, "logits (router route)", reg)
    opts3 = moe._RouteOptions(p(bias), None)
    _ok(L.moe_router_route(s, p(x), p(w_r), lg3.ptr(), ids3.ptr(), w3.ptr(), ctypes.byref(opts3),
                           st), "moe_router_route")

    torch.cuda.synchronize()
    moe.check_device_status(ws.tensor(torch.uint8, (ws.n,)))
    moe.check_device_status(sc.tensor(torch.uint8, (sc.n,)))
    for g in reg:
        g.check()
    if T > 0:   # the guarded calls computed the same block as the unguarded binding
        y_ref, _, _ = moe.forward(x, logits, w_gu, w_down, k, training=False)
        assert torch.equal(y.tensor(torch.bfloat16, (T, d)), y_ref)
        assert torch.equal(y0.tensor(torch.bfloat16, (T, d)), y_ref)
        assert np.array_equal(t2.tensor(torch.int32, (R,)).cpu().numpy(),
                              tok_of.tensor(torch.int32, (R,)).cpu().numpy())
