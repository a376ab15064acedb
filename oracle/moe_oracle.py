"""CPU oracle of the MoE expert block (route, dispatch, SwiGLU experts, combine, backward).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module. The product path (the CUDA library and its Python binding) never
touches it, and it shares no code with that path.

Plain numpy, float64 throughout, no blocking or fusion beyond what each step's
definition states; a library matmul or sort stands in for a step where noted.
Inputs are the exact values of the block's inputs (bf16 tensors widened to
fp32/fp64, fp32 logits), so every result here is the exact-arithmetic value up to
fp64 rounding.

What the method computes, and where it is stated:

* Route -- "Halo's 2.8x over TRL is not a kernel, and its own benchmark proves
  it", section "Where the gap actually is": fp32 router logits feed a per-token
  top-k router (Figure 3, "EP token routing"), and the expert outputs come back
  "weighted by the top-k probabilities". Readings: the k experts with the largest
  logits, ties to the lower expert index, slots in descending-logit order, weights
  the softmax over the k chosen logits (equal to softmax-then-renormalise).
* Dispatch -- same figure: a grouped matmul "over tokens sorted by expert".
  Reading: a stable counting sort of the assignments a = t*k + j by expert id.
* Experts -- "Halo: Frontier-Lab Training for Everyone", section "Novel model
  integration" (Laguna caption: grouped GEMM and fused SwiGLU) and section "One
  trainer architecture" (fused experts are single 3-D weight tensors). Reading:
  W_gu[e] is d x 2f with gate columns [0, f) and up columns [f, 2f);
  h = silu(g) * u; o = h @ W_down[e].
* Combine -- Figure 3 again: rows return to their origin, weighted by the top-k
  probabilities. Y[t] = sum_j w[t, j] * O[row_of[t, j]].
* Backward -- "Halo: Frontier-Lab Training for Everyone", section "The hard
  problems along the way" (atomic-free routing backward) and the LoRA paragraph
  of "One trainer architecture" (expert gradients). Gradients of Y with respect
  to x, W_gu and W_down with the routing weights held constant, and (router_backward)
  the gradient with respect to the router logits through the routing weights, the
  top-k selection held fixed.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _sigmoid(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


# ----------------------------------------------------------------------------- route
def route(logits: np.ndarray, k: int, bias: np.ndarray | None = None
          ) -> tuple[np.ndarray, np.ndarray]:
    """Per-token top-k over the router logits, then softmax over the k chosen.

    Follows Figure 3 ("per-token top-k router") and the fp32 router of "Where the
    gap actually is" in "Halo's 2.8x over TRL is not a kernel". Experts are ordered
    by (score descending, expert index ascending); the first k are the token's
    slots. The score is the fp32 logit, or, with a selection bias (the
    "bias_update" balancing of the LFM2 recipe in the same article: balancing
    "through the expert-selection bias"), the fp32 sum logit + bias[e]. The
    selection compares fp32 values, so it is exact. The weights use the unbiased
    logits of the chosen experts: w[t, j] = exp(l_j - m) / sum_i exp(l_i - m),
    m the largest chosen logit.

    Returns ids [T, k] int32 and w [T, k] float64.
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    if not np.all(np.isfinite(logits)):
        raise ValueError("router logits must be finite")
    score = logits
    if bias is not None:
        bias = np.asarray(bias, dtype=np.float32)
        if bias.shape != (E,) or not np.all(np.isfinite(bias)):
            raise ValueError("selection bias must be E finite values")
        score = logits + bias[None, :]          # fp32 addition, as the score is defined
    # a stable sort on the negated scores keeps equal scores in index order
    order = np.argsort(-score, axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    chosen = np.take_along_axis(logits, ids, axis=1).astype(F64)
    z = np.exp(chosen - chosen.max(axis=1, keepdims=True))
    w = z / z.sum(axis=1, keepdims=True)
    return ids, w


def aux_stats(logits: np.ndarray, counts: np.ndarray, k: int) -> dict:
    """Load-balancing statistics of one routing.

    The TorchTurbo adapter (its "Adapter" section) has routers apply an auxiliary
    loss (moe.aux_loss_coeff) and report aux_loss. Reading: the usual balancing loss
    aux = E * sum_e f_e * P_e with f_e = counts_e / (T k), the fraction of the
    assignments that went to expert e, and P_e the mean over tokens of the softmax
    over all E unbiased logits.
    """
    logits = np.asarray(logits, dtype=F64)
    T, E = logits.shape
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    f = np.asarray(counts, dtype=F64) / (T * k)
    P = p.mean(axis=0)
    return {"f": f, "P": P, "aux": float(E * (f * P).sum())}


def aux_loss_grad(logits: np.ndarray, counts: np.ndarray, k: int) -> np.ndarray:
    """d aux / d logits with f held constant (it counts discrete choices):
    d aux / d l[t, e] = (E / T) * p[t, e] * (f_e - sum_e' f_e' p[t, e'])."""
    logits = np.asarray(logits, dtype=F64)
    T, E = logits.shape
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    f = np.asarray(counts, dtype=F64) / (T * k)
    return (E / T) * p * (f[None, :] - (p * f[None, :]).sum(axis=1, keepdims=True))


def router_logits(x: np.ndarray, w_r: np.ndarray) -> np.ndarray:
    """fp32 router logits: logits[t, e] = sum over i of x[t, i] * w_r[e, i].

    "Halo's 2.8x over TRL is not a kernel, and its own benchmark proves it" computes
    the router's logits in fp32 ("Where the gap actually is"; `fp32_router: true` in
    the LFM2 recipe of "The small-hardware end"). Reading: x [T, d] and the router
    weight w_r [E, d] (one row per expert) are bf16 values taken as fp32; the sum runs
    over i = 0 .. d-1 in order, each step adding the exact product x[t, i] * w_r[e, i]
    (exact in fp64: two 8-bit significands) to the fp32 partial sum with one rounding
    to fp32. Returns [T, E] float32.
    """
    x = np.asarray(x, dtype=np.float32).astype(F64)
    w_r = np.asarray(w_r, dtype=np.float32).astype(F64)
    T, d = x.shape
    acc = np.zeros((T, w_r.shape[0]), dtype=np.float32)
    for i in range(d):
        acc = (acc.astype(F64) + x[:, i:i + 1] * w_r[:, i][None, :]).astype(np.float32)
    return acc


def router_weight_backward(x: np.ndarray, w_r: np.ndarray, dlogits: np.ndarray
                           ) -> tuple[np.ndarray, np.ndarray]:
    """Gradients through the router GEMM logits = x w_r^T: dW_r = dlogits^T x [E, d]
    and the contribution dlogits w_r [T, d] to dX (float64)."""
    x = np.asarray(x, dtype=F64)
    w_r = np.asarray(w_r, dtype=F64)
    dl = np.asarray(dlogits, dtype=F64)
    return dl.T @ x, dl @ w_r


# -------------------------------------------------------------------------- dispatch
def dispatch(ids: np.ndarray, E: int) -> dict:
    """Counting-sort dispatch of the T*k assignments into per-expert segments.

    Follows Figure 3 of "Halo's 2.8x over TRL is not a kernel" ("tokens sorted by
    expert"). The steps of a counting sort: count each expert, take the exclusive
    prefix sum of the counts as segment starts, then walk the assignments in order
    a = t*k + j and give each the next free row of its expert's segment.

    Returns counts [E], offsets [E+1] (offsets[E] = T*k), row_of [T, k] (the row of
    assignment (t, j) in the sorted order) and tok_of [T*k] (the token of each row).
    """
    ids = np.asarray(ids)
    T, k = ids.shape
    flat = [int(e) for e in ids.reshape(-1)]
    counts = [0] * E
    for e in flat:
        if not (0 <= e < E):
            raise ValueError("expert id out of range")
        counts[e] += 1
    offsets = [0] * (E + 1)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:E]
    row_of = [0] * (T * k)
    tok_of = [0] * (T * k)
    for a, e in enumerate(flat):
        r = cursor[e]
        cursor[e] += 1
        row_of[a] = r
        tok_of[r] = a // k
    return {
        "counts": np.asarray(counts, dtype=np.int64),
        "offsets": np.asarray(offsets, dtype=np.int64),
        "row_of": np.asarray(row_of, dtype=np.int64).reshape(T, k),
        "tok_of": np.asarray(tok_of, dtype=np.int64),
    }


def permute_rows(x: np.ndarray, tok_of: np.ndarray) -> np.ndarray:
    """Xp[r] = x[tok_of[r]]: the token rows in dispatch order."""
    return np.asarray(x, dtype=F64)[np.asarray(tok_of)]


# --------------------------------------------------------------------------- experts
def swiglu_expert(xr: np.ndarray, w_gu_e: np.ndarray, w_down_e: np.ndarray) -> dict:
    """One expert's SwiGLU MLP on the rows xr [m, d].

    "Halo: Frontier-Lab Training for Everyone", section "Novel model integration":
    grouped GEMM with a fused SwiGLU. gu = xr @ W_gu[e] (library matmul),
    g = gu[:, :f], u = gu[:, f:], h = g * sigmoid(g) * u, o = h @ W_down[e].
    """
    w_gu_e = np.asarray(w_gu_e, dtype=F64)
    w_down_e = np.asarray(w_down_e, dtype=F64)
    f = w_down_e.shape[0]
    gu = np.asarray(xr, dtype=F64) @ w_gu_e
    g, u = gu[:, :f], gu[:, f:]
    h = g * _sigmoid(g) * u
    o = h @ w_down_e
    return {"gu": gu, "h": h, "o": o}


def expert_ffn(xp: np.ndarray, offsets: np.ndarray, w_gu: np.ndarray,
               w_down: np.ndarray) -> dict:
    """All experts over their segments of the dispatched rows (the grouped GEMM).

    Segment e is rows [offsets[e], offsets[e+1]) of xp; empty segments are legal.
    """
    E = len(offsets) - 1
    A, d = xp.shape
    f = np.asarray(w_down).shape[1]
    GU = np.zeros((A, 2 * f), dtype=F64)
    H = np.zeros((A, f), dtype=F64)
    O = np.zeros((A, d), dtype=F64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        r = swiglu_expert(xp[lo:hi], w_gu[e], w_down[e])
        GU[lo:hi], H[lo:hi], O[lo:hi] = r["gu"], r["h"], r["o"]
    return {"gu": GU, "h": H, "o": O}


# --------------------------------------------------------------------------- combine
def combine(o: np.ndarray, w: np.ndarray, row_of: np.ndarray) -> np.ndarray:
    """Y[t] = sum_j w[t, j] * O[row_of[t, j]].

    Figure 3 of "Halo's 2.8x over TRL is not a kernel": the rows come back to the
    token they left, weighted by the top-k probabilities.
    """
    o = np.asarray(o, dtype=F64)
    w = np.asarray(w, dtype=F64)
    T, k = row_of.shape
    y = np.zeros((T, o.shape[1]), dtype=F64)
    for j in range(k):
        y += w[:, j:j + 1] * o[row_of[:, j]]
    return y


# --------------------------------------------------------------------------- forward
def forward(x, logits, w_gu, w_down, k: int, bias=None) -> dict:
    """The whole block: route, dispatch, experts, combine. Returns every stage."""
    x = np.asarray(x, dtype=F64)
    E = np.asarray(w_gu).shape[0]
    ids, w = route(logits, k, bias)
    disp = dispatch(ids, E)
    xp = permute_rows(x, disp["tok_of"])
    ffn = expert_ffn(xp, disp["offsets"], w_gu, w_down)
    y = combine(ffn["o"], w, disp["row_of"])
    out = {"ids": ids, "w": w, "xp": xp, "y": y}
    out.update(disp)
    out.update(ffn)
    return out


# -------------------------------------------------------------------------- backward
def swiglu_backward(dh: np.ndarray, g: np.ndarray, u: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """d/dg and d/du of h = silu(g) * u: silu'(g) = s * (1 + g * (1 - s)), s = sigmoid(g)."""
    s = _sigmoid(g)
    dg = dh * u * s * (1.0 + g * (1.0 - s))
    du = dh * g * s
    return dg, du


def backward(dy, fwd: dict, w_gu, w_down) -> dict:
    """Gradients of the block for dY, the routing weights held constant.

    Per assignment (t, j) with row r = row_of[t, j]: G[r] = w[t, j] * dY[t]. Per
    expert e on its segment: dW_down[e] = H_e^T G_e, dH_e = G_e W_down[e]^T,
    (dg, du) = SwiGLU backward, dGU_e = [dg, du], dW_gu[e] = Xp_e^T dGU_e,
    dXp_e = dGU_e W_gu[e]^T. Finally dX[t] = sum_j dXp[row_of[t, j]]: a gather per
    token, so no two writers touch one output (the atomic-free backward of "The
    hard problems along the way").
    """
    dy = np.asarray(dy, dtype=F64)
    T, d = dy.shape
    E, _, f2 = np.asarray(w_gu).shape
    f = f2 // 2
    row_of, w, offsets = fwd["row_of"], fwd["w"], fwd["offsets"]
    A = int(offsets[-1])
    G = np.zeros((A, d), dtype=F64)
    k = row_of.shape[1]
    for j in range(k):
        G[row_of[:, j]] = w[:, j:j + 1] * dy
    dW_gu = np.zeros((E, d, 2 * f), dtype=F64)
    dW_down = np.zeros((E, f, d), dtype=F64)
    dGU = np.zeros((A, 2 * f), dtype=F64)
    dXp = np.zeros((A, d), dtype=F64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        Ge, He = G[lo:hi], fwd["h"][lo:hi]
        GUe, Xe = fwd["gu"][lo:hi], fwd["xp"][lo:hi]
        wd = np.asarray(w_down[e], dtype=F64)
        wgu = np.asarray(w_gu[e], dtype=F64)
        dW_down[e] = He.T @ Ge
        dHe = Ge @ wd.T
        dg, du = swiglu_backward(dHe, GUe[:, :f], GUe[:, f:])
        dGUe = np.concatenate([dg, du], axis=1)
        dGU[lo:hi] = dGUe
        dW_gu[e] = Xe.T @ dGUe
        dXp[lo:hi] = dGUe @ wgu.T
    dX = np.zeros((T, d), dtype=F64)
    for j in range(k):
        dX += dXp[row_of[:, j]]
    return {"g": G, "dgu": dGU, "dxp": dXp, "dx": dX, "dw_gu": dW_gu, "dw_down": dW_down}


def router_backward(dy, fwd: dict) -> np.ndarray:
    """Gradient of the loss <dY, Y> with respect to the router logits.

    "The hard problems along the way" ("Halo: Frontier-Lab Training for Everyone")
    credits a routing backward without atomics. Y[t] = sum_j w[t, j] O[row_of[t, j]]
    with w the softmax over the k chosen logits, so with dw_j = <dY[t], O[row_of[t, j]]>
    the chain rule through that softmax gives, for the chosen experts,
    dlogit[t, ids[t, j]] = w_j * (dw_j - sum_i w_i dw_i); the others get 0 (the
    selection itself is piecewise constant). Returns [T, E] float64.
    """
    dy = np.asarray(dy, dtype=F64)
    T = dy.shape[0]
    ids, w, row_of, o = fwd["ids"], fwd["w"], fwd["row_of"], fwd["o"]
    E = int(fwd["counts"].shape[0])
    dw = np.einsum("td,tjd->tj", dy, np.asarray(o, dtype=F64)[row_of])
    centred = dw - (w * dw).sum(axis=1, keepdims=True)
    dl = np.zeros((T, E), dtype=F64)
    np.put_along_axis(dl, np.asarray(ids, dtype=np.int64), w * centred, axis=1)
    return dl


def router_backward_token(x_t, dy_t, ids_t, w_t, E: int, w_gu, w_down) -> np.ndarray:
    """dlogit[t, :] for one token from its own routing (one-at-a-time form)."""
    x_t = np.asarray(x_t, dtype=F64)
    dy_t = np.asarray(dy_t, dtype=F64)
    dw = np.array([dy_t @ swiglu_expert(x_t[None, :], w_gu[int(e)], w_down[int(e)])["o"][0]
                   for e in ids_t])
    w_t = np.asarray(w_t, dtype=F64)
    dl = np.zeros(E, dtype=F64)
    dl[np.asarray(ids_t, dtype=np.int64)] = w_t * (dw - (w_t * dw).sum())
    return dl


# ------------------------------------------------------- single outputs, one at a time
def forward_token(x_t: np.ndarray, ids_t: np.ndarray, w_t: np.ndarray, w_gu, w_down) -> np.ndarray:
    """Y[t] for one token from its own routing, without the dispatch."""
    y = np.zeros(np.asarray(x_t).shape[-1], dtype=F64)
    for e, wj in zip(ids_t, w_t):
        r = swiglu_expert(np.asarray(x_t, dtype=F64)[None, :], w_gu[int(e)], w_down[int(e)])
        y += wj * r["o"][0]
    return y


def backward_token(x_t, dy_t, ids_t, w_t, w_gu, w_down) -> np.ndarray:
    """dX[t] for one token: sum over its k slots of dGU_r W_gu[e]^T."""
    x_t = np.asarray(x_t, dtype=F64)
    dy_t = np.asarray(dy_t, dtype=F64)
    dx = np.zeros_like(x_t)
    for e, wj in zip(ids_t, w_t):
        wgu = np.asarray(w_gu[int(e)], dtype=F64)
        wd = np.asarray(w_down[int(e)], dtype=F64)
        f = wd.shape[0]
        gu = x_t @ wgu
        dh = (wj * dy_t) @ wd.T
        dg, du = swiglu_backward(dh, gu[:f], gu[f:])
        dx += np.concatenate([dg, du]) @ wgu.T
    return dx


def expert_members(ids: np.ndarray, w: np.ndarray, e: int) -> tuple[np.ndarray, np.ndarray]:
    """Tokens routed to expert e (ascending) and their routing weight for e."""
    hit = np.asarray(ids) == e
    toks = np.nonzero(hit.any(axis=1))[0]
    wts = (np.asarray(w) * hit).sum(axis=1)[toks]
    return toks, wts


def dw_down_rows(e: int, rows: np.ndarray, x, dy, ids, w, w_gu, w_down) -> np.ndarray:
    """Rows i of dW_down[e] = sum over the expert's tokens of H[r, i] * G[r, :]."""
    toks, wts = expert_members(ids, w, e)
    f = np.asarray(w_down[e]).shape[0]
    d = np.asarray(dy).shape[1]
    rows = np.asarray(rows)
    if len(toks) == 0:
        return np.zeros((len(rows), d), dtype=F64)
    wgu = np.asarray(w_gu[e], dtype=F64)
    X = np.asarray(x[toks], dtype=F64)
    g = X @ wgu[:, rows]
    u = X @ wgu[:, f + rows]
    h = g * _sigmoid(g) * u                       # [m, len(rows)]
    G = wts[:, None] * np.asarray(dy[toks], dtype=F64)
    return h.T @ G


def dw_gu_cols(e: int, cols: np.ndarray, x, dy, ids, w, w_gu, w_down) -> np.ndarray:
    """Columns c of dW_gu[e] = sum over the expert's tokens of Xp[r, :] * dGU[r, c]."""
    toks, wts = expert_members(ids, w, e)
    f = np.asarray(w_down[e]).shape[0]
    d = np.asarray(x).shape[1]
    cols = np.asarray(cols)
    if len(toks) == 0:
        return np.zeros((d, len(cols)), dtype=F64)
    wgu = np.asarray(w_gu[e], dtype=F64)
    wd = np.asarray(w_down[e], dtype=F64)
    X = np.asarray(x[toks], dtype=F64)
    G = wts[:, None] * np.asarray(dy[toks], dtype=F64)
    c0 = cols % f                                  # the hidden unit each column belongs to
    g = X @ wgu[:, c0]
    u = X @ wgu[:, f + c0]
    dh = G @ wd[c0, :].T
    dg, du = swiglu_backward(dh, g, u)
    dgu = np.where(cols[None, :] < f, dg, du)
    return X.T @ dgu
