"""Python binding of libmoe_gb300.so, the C ABI of the MoE expert block on GB300.

Argument marshalling only: every function checks tensor placement and dtypes,
allocates the outputs and the workspace with torch (device memory is PyTorch's
job here), and passes raw pointers plus the current CUDA stream to the C entry
point of the same name. Every step of the block runs in the library's CUDA
kernels; there is no fallback of any kind. If the library has not been built,
or no GB300 is present, the calls raise.

The C header (include/moe_gb300.h) documents each operation, its layout and its
error behaviour; names and argument order here follow it.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmoe_gb300.so")

_c_i64 = ctypes.c_int64
_c_vp = ctypes.c_void_p


class MoEShape(ctypes.Structure):
    _fields_ = [("T", _c_i64), ("d", _c_i64), ("E", _c_i64), ("k", _c_i64), ("f", _c_i64)]


class _Views(ctypes.Structure):
    _fields_ = [(n, _c_vp) for n in ("ids", "w", "counts", "offsets", "padded_offsets", "row_of",
                                     "tok_of", "xp", "gu", "h", "o")]


class _RouteOptions(ctypes.Structure):
    _fields_ = [("selection_bias", _c_vp), ("aux_stats", _c_vp)]


class _LaunchTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("ms", ctypes.c_float)]


STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED",
          -3: "MOE_ERR_ALIGNMENT", -4: "MOE_ERR_WORKSPACE", -5: "MOE_ERR_OVERFLOW",
          -6: "MOE_ERR_CUDA", -7: "MOE_ERR_TIMEOUT"}

# every exported entry point: (name, restype, argtypes)
_SIG = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_padded_rows": (_c_i64, [MoEShape]),
    "moe_workspace_size": (ctypes.c_size_t, [MoEShape, ctypes.c_int]),
    "moe_backward_scratch_size": (ctypes.c_size_t, [MoEShape]),
    "moe_workspace_views": (ctypes.c_int, [MoEShape, ctypes.c_int, _c_vp, ctypes.c_size_t,
                                           ctypes.POINTER(_Views)]),
    "moe_route": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, ctypes.POINTER(_RouteOptions),
                                 _c_vp]),
    "moe_dispatch": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                    _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "moe_expert_ffn": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                      _c_vp, ctypes.c_size_t, _c_vp]),
    "moe_combine": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "moe_dispatch_noalloc": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                            _c_vp, _c_vp, _c_vp]),
    "moe_forward": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_int,
                                   ctypes.POINTER(_RouteOptions), _c_vp, ctypes.c_size_t, _c_vp]),
    "moe_router_route": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                        ctypes.POINTER(_RouteOptions), _c_vp]),
    "moe_forward_router": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                          ctypes.c_int, ctypes.POINTER(_RouteOptions), _c_vp,
                                          ctypes.c_size_t, _c_vp]),
    "moe_router_backward_scratch_size": (ctypes.c_size_t, [MoEShape]),
    "moe_router_backward": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                           ctypes.c_size_t, _c_vp]),
    "moe_aux_loss_backward": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, ctypes.c_float, _c_vp, _c_vp]),
    "moe_backward": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_vp,
                                    _c_vp, _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "moe_expert_ffn_backward": (ctypes.c_int, [MoEShape] + [_c_vp] * 10 +
                                [_c_vp, ctypes.c_size_t, _c_vp, ctypes.c_size_t, _c_vp]),
    "moe_ep_local_shape": (ctypes.c_int, [MoEShape, ctypes.c_int, ctypes.POINTER(MoEShape)]),
    "moe_ep_dispatch": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                       ctypes.c_size_t, _c_vp]),
    "moe_ep_regroup": (ctypes.c_int, [MoEShape, ctypes.c_int, _c_vp, _c_i64, _c_vp, _c_vp, _c_vp,
                                      _c_vp, _c_vp, _c_vp, ctypes.c_size_t, _c_vp]),
    "moe_ep_unregroup": (ctypes.c_int, [MoEShape, _c_i64, _c_vp, _c_vp, _c_vp, _c_vp]),
    "moe_ep_grad_scatter": (ctypes.c_int, [MoEShape] + [_c_vp] * 9 + [_c_vp]),
    "moe_check_device_status": (ctypes.c_int, [_c_vp, _c_vp]),
    "moe_debug_gate_up_withheld": (ctypes.c_int, [MoEShape, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                                  ctypes.c_size_t, ctypes.c_int, _c_vp]),
    "moe_profile_start": (ctypes.c_int, [ctypes.c_int]),
    "moe_profile_stop": (ctypes.c_int, [ctypes.POINTER(_LaunchTime), ctypes.c_int]),
    "moe_launch_count": (_c_i64, []),
    "moe_stage_timing_arm": (ctypes.c_int, [ctypes.c_int]),
    "moe_stage_timing_read": (ctypes.c_int, [_c_vp, ctypes.c_int, _c_vp, ctypes.c_int]),
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_status_text(status)})")


def _status_text(status: int) -> str:
    try:
        return lib().moe_status_string(status).decode()
    except Exception:  # noqa: BLE001 - the library itself may be what is missing
        return "?"


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()'); there is no non-CUDA path")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIG.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MoEError(status, where)


def shape(T: int, d: int, E: int, k: int, f: int) -> MoEShape:
    return MoEShape(int(T), int(d), int(E), int(k), int(f))


def _p(t: torch.Tensor | None) -> _c_vp:
    if t is None:
        return _c_vp(None)
    if not t.is_cuda:
        raise ValueError("tensors passed to the MoE library must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return _c_vp(t.data_ptr())


def _stream() -> _c_vp:
    return _c_vp(torch.cuda.current_stream().cuda_stream)


def _dev(*ts: torch.Tensor) -> torch.device:
    return next(t.device for t in ts if t is not None)


def _want(t: torch.Tensor, dtype: torch.dtype, name: str) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


# ------------------------------------------------------------------ sizes and views
def padded_rows(s: MoEShape) -> int:
    r = lib().moe_padded_rows(s)
    if r < 0:
        raise MoEError(-1, "moe_padded_rows")
    return int(r)


def workspace_size(s: MoEShape, training: bool) -> int:
    n = lib().moe_workspace_size(s, int(bool(training)))
    if n == 0:
        raise MoEError(-1, "moe_workspace_size")
    return int(n)


def backward_scratch_size(s: MoEShape) -> int:
    n = lib().moe_backward_scratch_size(s)
    if n == 0:
        raise MoEError(-1, "moe_backward_scratch_size")
    return int(n)


def new_workspace(s: MoEShape, training: bool, device="cuda") -> torch.Tensor:
    return torch.empty(workspace_size(s, training), dtype=torch.uint8, device=device)


def new_scratch(s: MoEShape, device="cuda") -> torch.Tensor:
    return torch.empty(backward_scratch_size(s), dtype=torch.uint8, device=device)


def workspace_views(s: MoEShape, training: bool, ws: torch.Tensor) -> dict:
    """Tensor views of the intermediates a forward call leaves in its workspace."""
    v = _Views()
    _check(lib().moe_workspace_views(s, int(bool(training)), _p(ws), ws.numel(), ctypes.byref(v)),
           "moe_workspace_views")
    base = ws.data_ptr()
    R = padded_rows(s)
    T, d, E, k, f = s.T, s.d, s.E, s.k, s.f
    spec = {"ids": ((T, k), torch.int32), "w": ((T, k), torch.float32),
            "counts": ((E,), torch.int32), "offsets": ((E + 1,), torch.int32),
            "padded_offsets": ((E + 1,), torch.int32), "row_of": ((T, k), torch.int32),
            "tok_of": ((R,), torch.int32), "xp": ((R, d), torch.bfloat16),
            "gu": ((R, 2 * f), torch.bfloat16), "h": ((R, f), torch.bfloat16),
            "o": ((R, d), torch.bfloat16)}
    out = {}
    for name, (shp, dt) in spec.items():
        ptr = getattr(v, name)
        if ptr is None:
            out[name] = None
            continue
        off = ptr - base
        n = 1
        for x in shp:
            n *= x
        nbytes = n * torch.empty((), dtype=dt).element_size()
        out[name] = ws[off:off + nbytes].view(dt).view(*shp)
    return out


# ------------------------------------------------------------------------- the stages
def _options(bias: torch.Tensor | None, aux: torch.Tensor | None):
    if bias is None and aux is None:
        return None
    if bias is not None:
        _want(bias, torch.float32, "selection bias")
    if aux is not None:
        _want(aux, torch.float32, "aux_stats")
    return ctypes.byref(_RouteOptions(_p(bias), _p(aux)))


def route(logits: torch.Tensor, k: int, bias: torch.Tensor | None = None
          ) -> tuple[torch.Tensor, torch.Tensor]:
    """moe_route: ids [T,k] int32, w [T,k] fp32 (bias: optional [E] selection bias)."""
    _want(logits, torch.float32, "logits")
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    s = shape(T, 8, E, k, 8)
    _check(lib().moe_route(s, _p(logits), _p(ids), _p(w), _options(bias, None), _stream()),
           "moe_route")
    return ids, w


def router_route(x: torch.Tensor, w_router: torch.Tensor, k: int,
                 bias: torch.Tensor | None = None, logits: torch.Tensor | None = None
                 ) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """moe_router_route: fp32 logits = x w_router^T, then the route of moe_route.
    x [T,d] bf16, w_router [E,d] bf16; returns (logits [T,E] fp32, ids, w)."""
    _want(x, torch.bfloat16, "x")
    _want(w_router, torch.bfloat16, "w_router")
    T, d = x.shape
    E = w_router.shape[0]
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    s = shape(T, d, E, k, 8)
    _check(lib().moe_router_route(s, _p(x), _p(w_router), _p(logits), _p(ids), _p(w),
                                  _options(bias, None), _stream()), "moe_router_route")
    return logits, ids, w


def dispatch(s: MoEShape, x: torch.Tensor, ids: torch.Tensor, ws: torch.Tensor | None = None) -> dict:
    """moe_dispatch: the stable counting sort of the assignments by expert."""
    _want(x, torch.bfloat16, "x")
    _want(ids, torch.int32, "ids")
    dev = x.device
    R = padded_rows(s)
    if ws is None:
        ws = new_workspace(s, False, dev)
    out = {"xp": torch.empty((R, s.d), dtype=torch.bfloat16, device=dev),
           "counts": torch.empty((s.E,), dtype=torch.int32, device=dev),
           "offsets": torch.empty((s.E + 1,), dtype=torch.int32, device=dev),
           "padded_offsets": torch.empty((s.E + 1,), dtype=torch.int32, device=dev),
           "row_of": torch.empty((s.T, s.k), dtype=torch.int32, device=dev),
           "tok_of": torch.empty((R,), dtype=torch.int32, device=dev)}
    _check(lib().moe_dispatch(s, _p(x), _p(ids), _p(out["xp"]), _p(out["counts"]),
                              _p(out["offsets"]), _p(out["padded_offsets"]), _p(out["row_of"]),
                              _p(out["tok_of"]), _p(ws), ws.numel(), _stream()), "moe_dispatch")
    return out


def dispatch_noalloc(s: MoEShape, x: torch.Tensor, ids: torch.Tensor) -> dict:
    """moe_dispatch_noalloc: moe_dispatch without a workspace (fixed 4 MiB device scratch)."""
    _want(x, torch.bfloat16, "x")
    _want(ids, torch.int32, "ids")
    dev = x.device
    R = padded_rows(s)
    out = {"xp": torch.empty((R, s.d), dtype=torch.bfloat16, device=dev),
           "counts": torch.empty((s.E,), dtype=torch.int32, device=dev),
           "offsets": torch.empty((s.E + 1,), dtype=torch.int32, device=dev),
           "padded_offsets": torch.empty((s.E + 1,), dtype=torch.int32, device=dev),
           "row_of": torch.empty((s.T, s.k), dtype=torch.int32, device=dev),
           "tok_of": torch.empty((R,), dtype=torch.int32, device=dev)}
    _check(lib().moe_dispatch_noalloc(s, _p(x), _p(ids), _p(out["xp"]), _p(out["counts"]),
                                      _p(out["offsets"]), _p(out["padded_offsets"]),
                                      _p(out["row_of"]), _p(out["tok_of"]), _stream()),
           "moe_dispatch_noalloc")
    return out


def expert_ffn(s: MoEShape, xp: torch.Tensor, counts: torch.Tensor, w_gu: torch.Tensor,
               w_down: torch.Tensor, save_gu: bool = False, ws: torch.Tensor | None = None
               ) -> tuple[torch.Tensor, torch.Tensor | None, torch.Tensor]:
    """moe_expert_ffn: h [R,f], gu [R,2f] (if save_gu), o [R,d]."""
    for t, n in ((xp, "xp"), (w_gu, "w_gu"), (w_down, "w_down")):
        _want(t, torch.bfloat16, n)
    _want(counts, torch.int32, "counts")
    dev = xp.device
    R = padded_rows(s)
    if ws is None:
        ws = new_workspace(s, False, dev)
    h = torch.empty((R, s.f), dtype=torch.bfloat16, device=dev)
    gu = torch.empty((R, 2 * s.f), dtype=torch.bfloat16, device=dev) if save_gu else None
    o = torch.empty((R, s.d), dtype=torch.bfloat16, device=dev)
    _check(lib().moe_expert_ffn(s, _p(xp), _p(counts), _p(w_gu), _p(w_down), _p(h), _p(gu), _p(o),
                                _p(ws), ws.numel(), _stream()), "moe_expert_ffn")
    return h, gu, o


def combine(s: MoEShape, o: torch.Tensor, w: torch.Tensor | None, row_of: torch.Tensor
            ) -> torch.Tensor:
    """moe_combine: y [T,d] bf16 (w None: unit weights, the plain gather-sum)."""
    _want(o, torch.bfloat16, "o")
    if w is not None:
        _want(w, torch.float32, "w")
    _want(row_of, torch.int32, "row_of")
    y = torch.empty((s.T, s.d), dtype=torch.bfloat16, device=o.device)
    _check(lib().moe_combine(s, _p(o), _p(w), _p(row_of), _p(y), _stream()), "moe_combine")
    return y


def forward(x: torch.Tensor, logits: torch.Tensor, w_gu: torch.Tensor, w_down: torch.Tensor,
            k: int, training: bool = False, ws: torch.Tensor | None = None,
            y: torch.Tensor | None = None, bias: torch.Tensor | None = None,
            aux_stats: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor, MoEShape]:
    """moe_forward: returns (y, workspace, shape); the workspace feeds backward().
    bias: optional [E] selection bias; aux_stats: optional [2E+1] fp32 output."""
    _want(x, torch.bfloat16, "x")
    _want(logits, torch.float32, "logits")
    T, d = x.shape
    E, _, f2 = w_gu.shape
    s = shape(T, d, E, k, f2 // 2)
    if ws is None:
        ws = new_workspace(s, training, x.device)
    if y is None:
        y = torch.empty((T, d), dtype=torch.bfloat16, device=x.device)
    _check(lib().moe_forward(s, _p(x), _p(logits), _p(w_gu), _p(w_down), _p(y), int(bool(training)),
                             _options(bias, aux_stats), _p(ws), ws.numel(), _stream()),
           "moe_forward")
    return y, ws, s


def forward_router(x: torch.Tensor, w_router: torch.Tensor, w_gu: torch.Tensor,
                   w_down: torch.Tensor, k: int, training: bool = False,
                   ws: torch.Tensor | None = None, y: torch.Tensor | None = None,
                   logits: torch.Tensor | None = None, bias: torch.Tensor | None = None,
                   aux_stats: torch.Tensor | None = None
                   ) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor, MoEShape]:
    """moe_forward_router: the block with the router GEMM in front.
    Returns (y, logits [T,E] fp32, workspace, shape)."""
    _want(x, torch.bfloat16, "x")
    _want(w_router, torch.bfloat16, "w_router")
    T, d = x.shape
    E, _, f2 = w_gu.shape
    s = shape(T, d, E, k, f2 // 2)
    if ws is None:
        ws = new_workspace(s, training, x.device)
    if y is None:
        y = torch.empty((T, d), dtype=torch.bfloat16, device=x.device)
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    _check(lib().moe_forward_router(s, _p(x), _p(w_router), _p(logits), _p(w_gu), _p(w_down),
                                    _p(y), int(bool(training)), _options(bias, aux_stats), _p(ws),
                                    ws.numel(), _stream()), "moe_forward_router")
    return y, logits, ws, s


def router_backward(s: MoEShape, x: torch.Tensor, w_router: torch.Tensor,
                    dlogits: torch.Tensor, dx: torch.Tensor, dw_router: torch.Tensor | None = None,
                    scratch: torch.Tensor | None = None) -> torch.Tensor:
    """moe_router_backward: adds dlogits w_router into dx (in place); returns dW_r [E,d] fp32."""
    _want(x, torch.bfloat16, "x")
    _want(w_router, torch.bfloat16, "w_router")
    _want(dlogits, torch.float32, "dlogits")
    _want(dx, torch.bfloat16, "dx")
    if dw_router is None:
        dw_router = torch.empty(w_router.shape, dtype=torch.float32, device=x.device)
    need = int(lib().moe_router_backward_scratch_size(s))
    if scratch is None or scratch.numel() < need:
        scratch = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _check(lib().moe_router_backward(s, _p(x), _p(w_router), _p(dlogits), _p(dx), _p(dw_router),
                                     _p(scratch), scratch.numel(), _stream()),
           "moe_router_backward")
    return dw_router


def aux_loss_backward(s: MoEShape, logits: torch.Tensor, counts: torch.Tensor, coeff: float,
                      dlogits: torch.Tensor) -> torch.Tensor:
    """moe_aux_loss_backward: adds coeff * d aux / d logits into dlogits (in place)."""
    _want(logits, torch.float32, "logits")
    _want(counts, torch.int32, "counts")
    _want(dlogits, torch.float32, "dlogits")
    _check(lib().moe_aux_loss_backward(s, _p(logits), _p(counts), float(coeff), _p(dlogits),
                                       _stream()), "moe_aux_loss_backward")
    return dlogits


def backward(s: MoEShape, dy: torch.Tensor, w_gu: torch.Tensor, w_down: torch.Tensor,
             ws: torch.Tensor, scratch: torch.Tensor | None = None,
             out: tuple | None = None, router_grad: bool = False,
             dlogits: torch.Tensor | None = None):
    """moe_backward: (dx, dw_gu, dw_down) for the forward that filled ws (training=True),
    plus dlogits [T, E] fp32 as a fourth element when router_grad (or dlogits) is given."""
    _want(dy, torch.bfloat16, "dy")
    dev = dy.device
    if scratch is None:
        scratch = new_scratch(s, dev)
    if out is None:
        dx = torch.empty((s.T, s.d), dtype=torch.bfloat16, device=dev)
        dw_gu = torch.empty(tuple(w_gu.shape), dtype=torch.bfloat16, device=dev)
        dw_down = torch.empty(tuple(w_down.shape), dtype=torch.bfloat16, device=dev)
    else:
        dx, dw_gu, dw_down = out
    if router_grad and dlogits is None:
        dlogits = torch.empty((s.T, s.E), dtype=torch.float32, device=dev)
    if dlogits is not None:
        _want(dlogits, torch.float32, "dlogits")
    _check(lib().moe_backward(s, _p(dy), _p(w_gu), _p(w_down), _p(ws), ws.numel(), _p(dx),
                              _p(dw_gu), _p(dw_down), _p(dlogits), _p(scratch), scratch.numel(),
                              _stream()),
           "moe_backward")
    if dlogits is not None:
        return dx, dw_gu, dw_down, dlogits
    return dx, dw_gu, dw_down


def expert_ffn_backward(s: MoEShape, g: torch.Tensor, xp: torch.Tensor, gu: torch.Tensor,
                        h: torch.Tensor, counts: torch.Tensor, w_gu: torch.Tensor,
                        w_down: torch.Tensor, ws: torch.Tensor | None = None,
                        scratch: torch.Tensor | None = None):
    """moe_expert_ffn_backward: (dxp [R,d], dw_gu [E,d,2f], dw_down [E,f,d]) for the row
    gradient g [R,d] (segment-padded, zero padding rows)."""
    for t, n in ((g, "g"), (xp, "xp"), (gu, "gu"), (h, "h"), (w_gu, "w_gu"), (w_down, "w_down")):
        _want(t, torch.bfloat16, n)
    _want(counts, torch.int32, "counts")
    dev = g.device
    if ws is None:
        ws = new_workspace(s, False, dev)
    if scratch is None:
        scratch = new_scratch(s, dev)
    dxp = torch.empty((padded_rows(s), s.d), dtype=torch.bfloat16, device=dev)
    dw_gu = torch.empty(tuple(w_gu.shape), dtype=torch.bfloat16, device=dev)
    dw_down = torch.empty(tuple(w_down.shape), dtype=torch.bfloat16, device=dev)
    _check(lib().moe_expert_ffn_backward(s, _p(g), _p(xp), _p(gu), _p(h), _p(counts), _p(w_gu),
                                         _p(w_down), _p(dxp), _p(dw_gu), _p(dw_down), _p(ws),
                                         ws.numel(), _p(scratch), scratch.numel(), _stream()),
           "moe_expert_ffn_backward")
    return dxp, dw_gu, dw_down


# ----------------------------------------------------------- expert parallelism
def ep_local_shape(s: MoEShape, G: int) -> MoEShape:
    """moe_ep_local_shape: the shape of one rank's expert work among G ranks."""
    out = MoEShape()
    _check(lib().moe_ep_local_shape(s, int(G), ctypes.byref(out)), "moe_ep_local_shape")
    return out


def ep_dispatch(s: MoEShape, x: torch.Tensor, ids: torch.Tensor,
                ws: torch.Tensor | None = None) -> dict:
    """moe_ep_dispatch: the compact send buffer xs [T k, d] sorted by expert, counts [E],
    offsets [E+1] and row_of [T, k] (compact rows)."""
    _want(x, torch.bfloat16, "x")
    _want(ids, torch.int32, "ids")
    dev = x.device
    if ws is None:
        ws = new_workspace(s, False, dev)
    out = {"xs": torch.empty((s.T * s.k, s.d), dtype=torch.bfloat16, device=dev),
           "counts": torch.empty((s.E,), dtype=torch.int32, device=dev),
           "offsets": torch.empty((s.E + 1,), dtype=torch.int32, device=dev),
           "row_of": torch.empty((s.T, s.k), dtype=torch.int32, device=dev)}
    _check(lib().moe_ep_dispatch(s, _p(x), _p(ids), _p(out["xs"]), _p(out["counts"]),
                                 _p(out["offsets"]), _p(out["row_of"]), _p(ws), ws.numel(),
                                 _stream()), "moe_ep_dispatch")
    return out


def ep_regroup(s_loc: MoEShape, G: int, recv_counts: torch.Tensor, n_recv: int,
               xr: torch.Tensor, ws: torch.Tensor | None = None) -> dict:
    """moe_ep_regroup: received rows xr [n_recv, d] (source-major) to the local experts'
    segment-padded rows xp [R_loc, d]; also counts [El], padded_offsets [El+1], dest_of
    [n_recv] and the workspace holding the status word."""
    _want(recv_counts, torch.int32, "recv_counts")
    _want(xr, torch.bfloat16, "xr")
    dev = xr.device
    if ws is None:
        ws = new_workspace(s_loc, False, dev)
    out = {"xp": torch.empty((padded_rows(s_loc), s_loc.d), dtype=torch.bfloat16, device=dev),
           "counts": torch.empty((s_loc.E,), dtype=torch.int32, device=dev),
           "padded_offsets": torch.empty((s_loc.E + 1,), dtype=torch.int32, device=dev),
           "dest_of": torch.empty((max(int(n_recv), 1),), dtype=torch.int32, device=dev),
           "ws": ws}
    _check(lib().moe_ep_regroup(s_loc, int(G), _p(recv_counts.contiguous()), int(n_recv),
                                _p(xr) if n_recv else _c_vp(None), _p(out["xp"]),
                                _p(out["counts"]), _p(out["padded_offsets"]), _p(out["dest_of"]),
                                _p(ws), ws.numel(), _stream()), "moe_ep_regroup")
    out["dest_of"] = out["dest_of"][:int(n_recv)]
    return out


def ep_unregroup(s_loc: MoEShape, n_recv: int, o: torch.Tensor, dest_of: torch.Tensor
                 ) -> torch.Tensor:
    """moe_ep_unregroup: out [n_recv, d] = o[dest_of]."""
    _want(o, torch.bfloat16, "o")
    _want(dest_of, torch.int32, "dest_of")
    out = torch.empty((int(n_recv), s_loc.d), dtype=torch.bfloat16, device=o.device)
    if n_recv:
        _check(lib().moe_ep_unregroup(s_loc, int(n_recv), _p(o), _p(dest_of), _p(out),
                                      _stream()), "moe_ep_unregroup")
    return out


def ep_grad_scatter(s: MoEShape, dy: torch.Tensor, w: torch.Tensor, ids: torch.Tensor,
                    disp: dict, ob: torch.Tensor | None = None, router_grad: bool = False):
    """moe_ep_grad_scatter: gs [T k, d] = w dY in the compact send order; with
    router_grad also dlogits [T, E] from the returned expert outputs ob."""
    _want(dy, torch.bfloat16, "dy")
    dev = dy.device
    gs = torch.empty((s.T * s.k, s.d), dtype=torch.bfloat16, device=dev)
    dl = torch.empty((s.T, s.E), dtype=torch.float32, device=dev) if router_grad else None
    if router_grad and ob is None:
        raise ValueError("the router-logit gradient needs the returned expert outputs ob")
    _check(lib().moe_ep_grad_scatter(s, _p(dy), _p(w), _p(ids), _p(disp["counts"]),
                                     _p(disp["offsets"]), _p(disp["row_of"]), _p(ob), _p(gs),
                                     _p(dl), _stream()), "moe_ep_grad_scatter")
    return gs, dl


def debug_gate_up_withheld(s: MoEShape, xp: torch.Tensor, counts: torch.Tensor,
                           w_gu: torch.Tensor, ws: torch.Tensor, wait_limit_us: int) -> None:
    """moe_debug_gate_up_withheld: the gate_up GEMM with its first loads withheld."""
    h = torch.empty((padded_rows(s), s.f), dtype=torch.bfloat16, device=xp.device)
    _check(lib().moe_debug_gate_up_withheld(s, _p(xp), _p(counts), _p(w_gu), _p(h), _p(ws),
                                            ws.numel(), int(wait_limit_us), _stream()),
           "moe_debug_gate_up_withheld")


def check_device_status(ws_or_scratch: torch.Tensor) -> None:
    _check(lib().moe_check_device_status(_p(ws_or_scratch), _stream()), "moe_check_device_status")


# ------------------------------------------------------------------------ measurement
def profile_start(capacity: int = 256) -> None:
    _check(lib().moe_profile_start(int(capacity)), "moe_profile_start")


def profile_stop(capacity: int = 4096) -> list[tuple[str, float]]:
    buf = (_LaunchTime * capacity)()
    n = lib().moe_profile_stop(buf, capacity)
    if n < 0:
        raise MoEError(n, "moe_profile_stop")
    return [(buf[i].name.decode(), float(buf[i].ms)) for i in range(min(n, capacity))]


STAGE_TIMING_STAGES, STAGE_TIMING_TILES = 8192, 2048
GEMM_KINDS = {"gate_up": 0, "down": 1, "dgrad_h": 2, "dgrad_x": 3, "wgrad": 4}


def stage_timing_arm(kind: str | None) -> None:
    """moe_stage_timing_arm: stamp CTA 0's pipeline stages of one GEMM kind (None: off)."""
    _check(lib().moe_stage_timing_arm(-1 if kind is None else GEMM_KINDS[kind]),
           "moe_stage_timing_arm")


def stage_timing_read():
    """moe_stage_timing_read: (stages [n, 4], tiles [m, 2]) int64 SM-clock stamps."""
    import numpy as np
    st = np.zeros((STAGE_TIMING_STAGES, 4), dtype=np.uint64)
    tl = np.zeros((STAGE_TIMING_TILES, 2), dtype=np.uint64)
    n = lib().moe_stage_timing_read(_c_vp(st.ctypes.data), STAGE_TIMING_STAGES,
                                    _c_vp(tl.ctypes.data), STAGE_TIMING_TILES)
    if n < 0:
        raise MoEError(n, "moe_stage_timing_read")
    m = int((tl[:, 1] > 0).sum())
    return st[:n].astype(np.int64), tl[:m].astype(np.int64)


def launch_count() -> int:
    return int(lib().moe_launch_count())


__all__ = ["MoEShape", "MoEError", "lib", "shape", "padded_rows", "workspace_size",
           "backward_scratch_size", "new_workspace", "new_scratch", "workspace_views", "route",
           "router_route", "dispatch", "dispatch_noalloc", "expert_ffn", "aux_loss_backward",
           "combine", "forward", "forward_router", "backward", "router_backward", "check_device_status",
           "expert_ffn_backward", "ep_local_shape", "ep_dispatch", "ep_regroup", "ep_unregroup",
           "ep_grad_scatter", "stage_timing_arm", "stage_timing_read",
           "debug_gate_up_withheld", "profile_start", "profile_stop", "launch_count", "LIB_PATH"]
