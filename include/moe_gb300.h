/*
 * moe_gb300.h -- C ABI of the MoE expert block on one GB300 (sm_103a).
 *
 * The block has four steps, each a hand-written CUDA kernel (or a few):
 *   route     per-token top-k over fp32 router logits, softmax over the k chosen;
 *   dispatch  stable counting sort of the T*k (token, slot) assignments by expert,
 *             copying each token row into its expert's contiguous segment;
 *   experts   grouped SwiGLU MLPs over the segments on the tcgen05 tensor cores
 *             (bf16 in, fp32 accumulate in TMEM);
 *   combine   per-token gather of its k expert rows, weighted by the routing weights;
 * plus the backward pass for dX, dW_gu and dW_down.
 *
 * Where the method is stated: "Halo's 2.8x over TRL is not a kernel, and its own
 * benchmark proves it", section "Where the gap actually is" and its Figure 3 ("EP
 * token routing": fp32 router logits, per-token top-k router, grouped matmul over
 * tokens sorted by expert, rows returned in order weighted by the top-k
 * probabilities); "Halo: Frontier-Lab Training for Everyone", sections "Novel model
 * integration" (grouped GEMM with fused SwiGLU), "One trainer architecture" (fused
 * experts as 3-D weight tensors) and "The hard problems along the way" (atomic-free
 * routing backward; a fused SwiGLU kernel that overflowed at 745k tokens on one GPU,
 * which is why every byte offset here is 64-bit).
 *
 * Conventions for every call:
 *   - Shapes: T tokens, d hidden, E experts, k experts per token, f expert FFN width.
 *     A = T*k assignments. All matrices are row-major and densely packed.
 *   - Types: bf16 is IEEE bfloat16 passed as uint16_t bit patterns (moe_bf16);
 *     router logits and routing weights are fp32; indices are int32.
 *   - Pointers are DEVICE pointers owned by the caller unless stated. The library
 *     allocates no device memory and keeps no per-call state; scratch lives in the
 *     caller's workspace. Every pointer must be 16-byte aligned.
 *   - All calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and return a status for errors the host can see: argument, shape,
 *     alignment, workspace size, 32-bit index overflow, or a failed launch. Device
 *     faults surface at the caller's next synchronisation. Nothing aborts the process.
 *   - Preconditions checked on the host: 1 <= k <= min(E, 16), 1 <= E <= 256,
 *     T >= 0, d >= 8 and f >= 8 with d % 8 == 0 and f % 8 == 0 (16-byte rows),
 *     T*k and the padded row count below 2^31. Router logits must be finite
 *     (not checked; the result for NaN/Inf logits is unspecified).
 *
 * Segment-padded row space. The dispatched rows (Xp, H, GU, O) live in a row space
 * of R = moe_padded_rows(shape) rows where expert e's segment starts at row
 *   P_e = 128 * sum_{e' < e} ceil(counts[e'] / 128)
 * and holds its counts[e] rows in ascending token order (the stable sort), followed
 * by zero rows up to the next multiple of 128. The compact layout of the method
 * (segment e at offsets[e] = sum_{e'<e} counts[e']) is recovered as
 *   compact row = row - P_e + offsets[e].
 * Padding keeps every 128-row GEMM tile inside one expert.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;   /* IEEE bfloat16 bit pattern */
typedef void *moe_stream;    /* cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,  /* null pointer, bad shape or k > E */
  MOE_ERR_UNSUPPORTED = -2,  /* shape outside the supported range (E > 256, k > 16, no sm_103 GPU) */
  MOE_ERR_ALIGNMENT = -3,    /* a pointer is not 16-byte aligned, or d or f is not a multiple of 8 */
  MOE_ERR_WORKSPACE = -4,    /* workspace or scratch smaller than the size query returns */
  MOE_ERR_OVERFLOW = -5,     /* an index would not fit in int32 */
  MOE_ERR_CUDA = -6,         /* a CUDA call or kernel launch failed */
  MOE_ERR_TIMEOUT = -7       /* a kernel gave up waiting on its own pipeline (see moe_check_device_status) */
} moe_status;

typedef struct {
  int64_t T; /* tokens */
  int64_t d; /* hidden size */
  int64_t E; /* experts */
  int64_t k; /* experts per token */
  int64_t f; /* expert FFN width: W_gu is E x d x 2f, W_down is E x f x d */
} moe_shape;

/* Text of a status code. Never NULL. */
const char *moe_status_string(moe_status s);

/* Rows R of the segment-padded row space (see above): 128 * (ceil(T*k/128) + E). */
int64_t moe_padded_rows(moe_shape s);

/* Bytes of the workspace that moe_forward (and any single-stage call) needs.
 * training != 0 adds the saved pre-activations GU (R x 2f bf16) used by moe_backward. */
size_t moe_workspace_size(moe_shape s, int training);

/* Bytes of the scratch that moe_backward needs (G, dGU and dXp, R rows each). */
size_t moe_backward_scratch_size(moe_shape s);

/* Device pointers into a forward workspace, for callers that want the intermediate
 * results of moe_forward. Layout is fixed by the shape and `training`.
 * Fills every field; gu is NULL when training == 0. */
typedef struct {
  int32_t *ids;     /* T x k   chosen experts, slots in descending-logit order */
  float *w;         /* T x k   routing weights (softmax over the k chosen logits) */
  int32_t *counts;  /* E       rows per expert */
  int32_t *offsets; /* E + 1   compact segment starts (exclusive prefix of counts) */
  int32_t *padded_offsets; /* E + 1   segment starts P_e in the padded row space */
  int32_t *row_of;  /* T x k   padded row of assignment (t, j) */
  int32_t *tok_of;  /* R       token of each padded row, -1 on padding rows and past P_E */
  moe_bf16 *xp;     /* R x d   dispatched token rows */
  moe_bf16 *gu;     /* R x 2f  gate|up pre-activations (training only) */
  moe_bf16 *h;      /* R x f   SwiGLU activations */
  moe_bf16 *o;      /* R x d   expert outputs */
} moe_forward_views;
moe_status moe_workspace_views(moe_shape s, int training, void *ws, size_t ws_bytes,
                               moe_forward_views *out);

/* Options of the routing step; a NULL options pointer or NULL fields give the plain
 * top-k.
 *   selection_bias [E] fp32 in: the experts are chosen by the fp32 score
 *     logit + selection_bias[e] (descending, ties to the lower index) while the
 *     weights stay the softmax over the chosen experts' unbiased logits; the
 *     "bias_update" balancing of the LFM2 recipe in "Halo's 2.8x over TRL is not a
 *     kernel" ("The small-hardware end": LFM2 balances "through the expert-selection
 *     bias").
 *   aux_stats [2E + 1] fp32 out (moe_forward only): load-balancing statistics for the
 *     TorchTurbo adapter's auxiliary loss ("Adapter": aux_loss_coeff, aux_loss):
 *     aux_stats[e] = f_e = counts_e / (T k), aux_stats[E + e] = P_e = the mean over
 *     tokens of the softmax over all E logits, aux_stats[2E] = E * sum_e f_e P_e.
 *     Reduced in a fixed order (deterministic). */
typedef struct {
  const float *selection_bias;
  float *aux_stats;
} moe_route_options;

/* Route. "Halo's 2.8x over TRL is not a kernel", Figure 3 and "Where the gap
 * actually is": per-token top-k router on fp32 logits, outputs weighted by the
 * top-k probabilities.
 *   logits [T x E] fp32 in; ids [T x k] int32 out; w [T x k] fp32 out;
 *   opts: see moe_route_options (aux_stats is ignored here) or NULL.
 * ids[t][0..k-1] are the k experts with the largest scores (the logits, or
 * logits + selection bias), ordered by descending score, equal scores by ascending
 * expert index (the lower index wins a tie). w[t][j] = exp(l_j - m) / sum_i exp(l_i - m)
 * over the k chosen unbiased logits, m their largest. One warp per token. */
moe_status moe_route(moe_shape s, const float *logits, int32_t *ids, float *w,
                     const moe_route_options *opts, moe_stream stream);

/* Dispatch. Figure 3 of "Halo's 2.8x over TRL is not a kernel": tokens sorted by
 * expert for a grouped matmul. A stable counting sort of the assignments
 * a = t*k + j by ids: block histograms, an exclusive scan of the per-expert counts,
 * and a 16-byte vectorised row scatter.
 *   x [T x d] bf16 in; ids [T x k] int32 in (each row k distinct experts in [0, E));
 *   xp [R x d] bf16 out (padding rows zeroed); counts [E], offsets [E+1] int32 out
 *   (compact, offsets[E] = T*k); padded_offsets [E+1] int32 out (P_e);
 *   row_of [T x k] int32 out (padded row of (t, j)); tok_of [R] int32 out (-1 on padding
 *   rows and on the rows at and past padded_offsets[E], which belong to no expert; xp is
 *   not written there).
 * Uses ws (at least moe_workspace_size(s, 0) bytes) for the block histograms. */
moe_status moe_dispatch(moe_shape s, const moe_bf16 *x, const int32_t *ids, moe_bf16 *xp,
                        int32_t *counts, int32_t *offsets, int32_t *padded_offsets,
                        int32_t *row_of, int32_t *tok_of, void *ws, size_t ws_bytes,
                        moe_stream stream);

/* Experts. "Halo: Frontier-Lab Training for Everyone", "Novel model integration":
 * grouped GEMM with fused SwiGLU over 3-D expert weights. For every expert e and
 * every row r of its segment:
 *   gu = xp[r] @ W_gu[e]  (gate = columns [0, f), up = columns [f, 2f))
 *   h[r] = silu(gate) * up,  o[r] = h[r] @ W_down[e]
 * on tcgen05 tensor cores: bf16 operands, fp32 accumulation in TMEM, the SwiGLU in
 * the epilogue of the first GEMM, h and o rounded to bf16 once.
 *   xp [R x d] bf16 in, segment-padded as moe_dispatch writes it; counts [E] int32 in;
 *   w_gu [E x d x 2f] bf16 in; w_down [E x f x d] bf16 in;
 *   h [R x f] bf16 out; gu [R x 2f] bf16 out or NULL (saved for the backward);
 *   o [R x d] bf16 out.
 * Uses ws (at least moe_workspace_size(s, 0) bytes) for the tile plan. */
moe_status moe_expert_ffn(moe_shape s, const moe_bf16 *xp, const int32_t *counts,
                          const moe_bf16 *w_gu, const moe_bf16 *w_down, moe_bf16 *h,
                          moe_bf16 *gu, moe_bf16 *o, void *ws, size_t ws_bytes,
                          moe_stream stream);

/* Combine. Figure 3 of "Halo's 2.8x over TRL is not a kernel": rows return to
 * their token weighted by the top-k probabilities.
 *   y[t] = bf16( sum_{j=0..k-1} w[t][j] * o[row_of[t][j]] ), an fp32 sum in slot
 *   order, one rounding. A gather per token: deterministic, no atomics.
 *   o [rows x d] bf16 in (any row space row_of indexes: the padded one of moe_dispatch,
 *   or the compact one of moe_ep_dispatch); w [T x k] fp32 in, or NULL for unit
 *   weights (the plain sum, e.g. the dX gather of an expert-parallel backward);
 *   row_of [T x k] int32 in; y [T x d] bf16 out. */
moe_status moe_combine(moe_shape s, const moe_bf16 *o, const float *w, const int32_t *row_of,
                       moe_bf16 *y, moe_stream stream);

/* The whole block: route, dispatch, experts, combine, with every intermediate in ws
 * (see moe_workspace_views). training != 0 also keeps GU for moe_backward; ws must
 * then hold moe_workspace_size(s, 1) bytes and outlive the matching moe_backward.
 *   x [T x d] bf16; logits [T x E] fp32; w_gu [E x d x 2f] bf16; w_down [E x f x d] bf16;
 *   y [T x d] bf16 out; opts: see moe_route_options, or NULL. */
moe_status moe_forward(moe_shape s, const moe_bf16 *x, const float *logits, const moe_bf16 *w_gu,
                       const moe_bf16 *w_down, moe_bf16 *y, int training,
                       const moe_route_options *opts, void *ws, size_t ws_bytes,
                       moe_stream stream);

/* Router GEMM with the route in its epilogue. "Halo's 2.8x over TRL is not a kernel":
 * the router logits are computed in fp32 ("Where the gap actually is"; the LFM2 recipe's
 * `fp32_router: true` in "The small-hardware end") in front of the per-token top-k of
 * Figure 3.
 *   logits[t][e] = sum_{i=0..d-1} x[t][i] * w_router[e][i]
 * as one fp32 chain per logit in ascending i, each step adding the exact product of
 * the two bf16 values with one rounding (an fmaf chain), so the logits, and the top-k
 * taken on them exactly as moe_route does, are bit-reproducible. One block per 32
 * tokens computes all E logits of its tokens on the fp32 SIMT pipes (the fixed order
 * rules out tensor cores), stores them and routes the chunk.
 *   x [T x d] bf16 in; w_router [E x d] bf16 in (one row per expert);
 *   logits [T x E] fp32 out; ids [T x k] int32 out; w [T x k] fp32 out;
 *   opts: see moe_route_options (aux_stats is ignored here) or NULL. */
moe_status moe_router_route(moe_shape s, const moe_bf16 *x, const moe_bf16 *w_router,
                            float *logits, int32_t *ids, float *w, const moe_route_options *opts,
                            moe_stream stream);

/* moe_forward with the router GEMM of moe_router_route in front: the first kernel
 * computes the logits (written to `logits`, [T x E] fp32 out) and routes and counts
 * the tokens in one pass; the rest is moe_forward. w_router [E x d] bf16 in; every
 * other argument as in moe_forward. */
moe_status moe_forward_router(moe_shape s, const moe_bf16 *x, const moe_bf16 *w_router,
                              float *logits, const moe_bf16 *w_gu, const moe_bf16 *w_down,
                              moe_bf16 *y, int training, const moe_route_options *opts, void *ws,
                              size_t ws_bytes, moe_stream stream);

/* Bytes of scratch moe_router_backward needs (token-split partial sums of dW_r). */
size_t moe_router_backward_scratch_size(moe_shape s);

/* Gradient through the router GEMM of moe_router_route / moe_forward_router, for a
 * router-logit gradient dlogits (for instance moe_backward's, plus
 * moe_aux_loss_backward's):
 *   dw_router[e][i] = sum_t dlogits[t][e] * x[t][i]          (fp32, the fp32 router)
 *   dx[t][i] = bf16( dx[t][i] + sum_e dlogits[t][e] * w_router[e][i] )
 * so that dx, holding moe_backward's dX on entry, holds the whole input gradient on
 * return (one more bf16 rounding of dx). fp32 sums on the SIMT pipes; dW_r sums token
 * splits in order and then adds the splits in order (no atomics, bit-reproducible).
 *   x [T x d] bf16 in; w_router [E x d] bf16 in; dlogits [T x E] fp32 in;
 *   dx [T x d] bf16 in/out; dw_router [E x d] fp32 out;
 *   scratch: at least moe_router_backward_scratch_size(s) bytes. */
moe_status moe_router_backward(moe_shape s, const moe_bf16 *x, const moe_bf16 *w_router,
                               const float *dlogits, moe_bf16 *dx, float *dw_router,
                               void *scratch, size_t scratch_bytes, moe_stream stream);

/* Gradient of the load-balancing loss coeff * aux (see moe_route_options) with respect
 * to the router logits, ADDED into dlogits, with the assignment fractions f held
 * fixed (they count discrete choices):
 *   dlogits[t][e] += coeff * (E / T) * p[t][e] * (f_e - sum_e' f_e' p[t][e'])
 * where p[t] is the softmax over all E logits of token t and f_e = counts[e] / (T k).
 * One warp per token; every element read and written by one thread.
 *   logits [T x E] fp32 in; counts [E] int32 in (from the forward); dlogits [T x E]
 *   fp32 in/out. */
moe_status moe_aux_loss_backward(moe_shape s, const float *logits, const int32_t *counts,
                                 float coeff, float *dlogits, moe_stream stream);

/* Backward of the block for dY ("Halo: Frontier-Lab Training for Everyone", "The hard
 * problems along the way": an atomic-free routing backward). With
 * G[r] = w[t][j] * dY[t] for r = row_of[t][j]:
 *   dW_down[e] = H_e^T G_e;  dH = G W_down[e]^T;  dgate = dH * up * silu'(gate),
 *   dup = dH * silu(gate);   dW_gu[e] = Xp_e^T [dgate | dup];
 *   dXp = [dgate | dup] W_gu[e]^T;  dX[t] = sum_j dXp[row_of[t][j]] (a gather);
 * and, when dlogits is not NULL, the router-logit gradient through the routing
 * weights (the top-k choice held fixed): with dw_j = <dY[t], O[row_of[t][j]]>,
 *   dlogits[t][ids[t][j]] = w_j * (dw_j - sum_i w_i dw_i), 0 for the other experts.
 * Every gradient is written by exactly one thread (no atomics, bit-reproducible);
 * experts with no rows get dW = 0.
 *   dy [T x d] bf16 in; w_gu, w_down as in moe_forward; ws: the workspace of a
 *   moe_forward(training = 1) call with the same shape and weights;
 *   dx [T x d], dw_gu [E x d x 2f], dw_down [E x f x d] bf16 out;
 *   dlogits [T x E] fp32 out or NULL;
 *   scratch: at least moe_backward_scratch_size(s) bytes. */
moe_status moe_backward(moe_shape s, const moe_bf16 *dy, const moe_bf16 *w_gu,
                        const moe_bf16 *w_down, const void *ws, size_t ws_bytes, moe_bf16 *dx,
                        moe_bf16 *dw_gu, moe_bf16 *dw_down, float *dlogits, void *scratch,
                        size_t scratch_bytes, moe_stream stream);

/* Backward of the experts alone (moe_expert_ffn's gradient), for a caller that forms
 * the row gradient G itself (the expert-parallel backward: G arrives from other
 * ranks). For every expert e and its segment rows, as in moe_backward:
 *   dH = G W_down[e]^T;  dgate = dH * up * silu'(gate),  dup = dH * silu(gate);
 *   dW_down[e] = H_e^T G_e;  dW_gu[e] = Xp_e^T [dgate | dup];  dXp = [dgate | dup] W_gu[e]^T
 * on the tcgen05 tensor cores (bf16 operands, fp32 accumulation, dGU rounded to bf16
 * as the GEMM operand, outputs rounded once). Experts with no rows get dW = 0.
 *   g [R x d] bf16 in, segment-padded like xp with zero padding rows; xp [R x d],
 *   gu [R x 2f], h [R x f] bf16 in (from moe_expert_ffn on the same counts);
 *   counts [E] int32 in; w_gu, w_down as in moe_expert_ffn;
 *   dxp [R x d] bf16 out (padding rows zero); dw_gu [E x d x 2f], dw_down [E x f x d] out;
 *   ws: at least moe_workspace_size(s, 0) bytes (tile plan, status word);
 *   scratch: at least moe_backward_scratch_size(s) bytes (dGU). */
moe_status moe_expert_ffn_backward(moe_shape s, const moe_bf16 *g, const moe_bf16 *xp,
                                   const moe_bf16 *gu, const moe_bf16 *h, const int32_t *counts,
                                   const moe_bf16 *w_gu, const moe_bf16 *w_down, moe_bf16 *dxp,
                                   moe_bf16 *dw_gu, moe_bf16 *dw_down, void *ws, size_t ws_bytes,
                                   void *scratch, size_t scratch_bytes, moe_stream stream);

/* ----------------------------------------------------------- expert parallelism
 * "Halo's 2.8x over TRL is not a kernel, and its own benchmark proves it", Figure 3
 * ("EP token routing") and section "Where the gap actually is": with the experts
 * sharded over G ranks, tokens are sorted by expert, each row is sent to the rank
 * that owns its expert (the dispatch all-to-all), the owners run their experts, and
 * the rows return (the combine all-to-all) to be summed at their token, weighted by
 * the top-k probabilities. The TorchTurbo README's expert-parallel plan shards the
 * fused expert weights Shard(0): rank g owns experts [g E/G, (g+1) E/G), E % G == 0.
 *
 * One rank's forward, around the caller's two exchanges (all-to-all over the ranks,
 * e.g. NCCL; these calls never wait on another rank):
 *   1. moe_route, then moe_ep_dispatch: the rows sorted by expert into a compact send
 *      buffer xs [T k x d] whose rows for rank r are [offsets[r El], offsets[(r+1) El]),
 *      El = E / G, and counts [E] (rank r receives counts[r El .. (r+1) El)).
 *   2. exchange the counts: recv_counts [G x El], row s from source rank s; then the
 *      rows: xr [n_recv x d], source-major ([s][local expert][rows]).
 *   3. moe_ep_regroup into the local segment-padded layout of the local shape
 *      (moe_ep_local_shape), moe_expert_ffn over the El local experts, moe_ep_unregroup
 *      back to the received order.
 *   4. exchange the rows back (the reverse splits): ob [T k x d] in xs's order, then
 *      moe_combine(s, ob, w, row_of, y).
 * The backward mirrors it: moe_ep_grad_scatter (G = w dY in xs's order, and the
 * router-logit gradient from ob), the exchange, moe_ep_regroup of G,
 * moe_expert_ffn_backward, moe_ep_unregroup of dXp, the exchange back, and
 * moe_combine with w = NULL (dX[t] = sum_j dXs[row_of[t][j]]). Every rank gets the
 * complete dW of its own experts (they saw every token routed to them). */

/* The local shape of rank-side expert work: E/G experts, T*G tokens (a bound on the
 * tokens that can reach one rank when every rank holds T), min(k, E/G) experts per
 * token; its padded row space holds every row a rank can receive. Needs E % G == 0. */
moe_status moe_ep_local_shape(moe_shape s, int G, moe_shape *out);

/* The dispatch of moe_dispatch into the compact layout of the method: xs row
 * offsets[e] + (rank of token t among expert e's tokens) = x[t], no padding rows.
 *   x [T x d] bf16 in; ids [T x k] int32 in; xs [T k x d] bf16 out; counts [E],
 *   offsets [E+1] int32 out; row_of [T x k] int32 out (compact row of (t, j));
 *   ws: at least moe_workspace_size(s, 0) bytes. */
moe_status moe_ep_dispatch(moe_shape s, const moe_bf16 *x, const int32_t *ids, moe_bf16 *xs,
                           int32_t *counts, int32_t *offsets, int32_t *row_of, void *ws,
                           size_t ws_bytes, moe_stream stream);

/* Received rows to the local experts' segment-padded layout. Received row i of block
 * (source s, local expert e) goes to row P_e + sum_{s'<s} recv_counts[s'][e] + (its
 * index in the block), P_e = 128 * sum_{e'<e} ceil(counts_loc[e'] / 128): per expert,
 * the sources in rank order, each in its sender's token order. Padding rows are zeroed.
 *   s_loc: the local shape (moe_ep_local_shape); recv_counts [G x El] int32 in (device);
 *   n_recv: the number of received rows (the sum of recv_counts), at most s_loc.T *
 *   s_loc.k; xr [n_recv x d] bf16 in; xp [R_loc x d] bf16 out, R_loc =
 *   moe_padded_rows(s_loc); counts_loc [El], padded_loc [El+1] int32 out;
 *   dest_of [n_recv] int32 out (the padded row of each received row);
 *   ws: at least moe_workspace_size(s_loc, 0) bytes. If the device counts do not add up
 *   to n_recv (or are negative), nothing is written and moe_check_device_status(ws)
 *   returns MOE_ERR_INVALID_ARG. */
moe_status moe_ep_regroup(moe_shape s_loc, int G, const int32_t *recv_counts, int64_t n_recv,
                          const moe_bf16 *xr, moe_bf16 *xp, int32_t *counts_loc,
                          int32_t *padded_loc, int32_t *dest_of, void *ws, size_t ws_bytes,
                          moe_stream stream);

/* The inverse gather of moe_ep_regroup: out[i] = o[dest_of[i]] for i < n_recv (expert
 * outputs, or dXp in the backward, back in the received order for the return exchange).
 *   o [R_loc x d] bf16 in; dest_of [n_recv] int32 in (from moe_ep_regroup; an entry
 *   outside [0, R_loc) is skipped); out [n_recv x d] bf16 out. */
moe_status moe_ep_unregroup(moe_shape s_loc, int64_t n_recv, const moe_bf16 *o,
                            const int32_t *dest_of, moe_bf16 *out, moe_stream stream);

/* The row gradient of an expert-parallel backward in the compact send order:
 * gs[row_of[t][j]] = bf16(w[t][j] * dy[t]); with dlogits, also the router-logit
 * gradient of moe_backward from the returned expert outputs ob (dw_j =
 * <dy[t], ob[row_of[t][j]]>, dlogits[t][ids[t][j]] = w_j (dw_j - sum_i w_i dw_i), 0
 * elsewhere). dy [T x d] bf16; w, ids, row_of [T x k]; counts [E], offsets [E+1] from
 * moe_ep_dispatch; ob [T k x d] bf16 (may be NULL without dlogits); gs [T k x d] bf16
 * out; dlogits [T x E] fp32 out or NULL. */
moe_status moe_ep_grad_scatter(moe_shape s, const moe_bf16 *dy, const float *w,
                               const int32_t *ids, const int32_t *counts, const int32_t *offsets,
                               const int32_t *row_of, const moe_bf16 *ob, moe_bf16 *gs,
                               float *dlogits, moe_stream stream);

/* Dispatch without a workspace, for callers that cannot allocate device memory.
 * The pages have no counterpart of this call: it exists for callers that have no
 * way to obtain device memory for a workspace (code running under a runtime that
 * owns every allocation, or that must not call cudaMalloc at that point). It
 * computes exactly what moe_dispatch computes, with the same arguments minus ws and
 * ws_bytes, and allocates nothing: its scratch (local ranks, chunk histograms, the
 * tile-to-expert table) is a file-scope __device__ array of 4 MiB (2^20 int32) that
 * every GPU loading the library holds until exit.
 *   Limit: round64(T*k) + round64(E*ceil(T/32)) + round64(R/128) <= 2^20 int32,
 *   round64(n) = n rounded up to a multiple of 64 and R = moe_padded_rows(s)
 *   (T = 65536 with E = 32 and k = 4 fits). Larger shapes return MOE_ERR_WORKSPACE.
 *   The first call on a device looks up the array's device address (set-up, once
 *   per device, with that device current); make that first call before any stream
 *   capture. The address is kept for the life of the process: do not use this call
 *   on a device after a cudaDeviceReset of that device. Every call shares the one array and it keeps the last call's contents:
 *   each call writes every entry it reads, so nothing needs clearing, but calls that
 *   overlap on the GPU (other streams or host threads) race and must be ordered by
 *   the caller. */
moe_status moe_dispatch_noalloc(moe_shape s, const moe_bf16 *x, const int32_t *ids, moe_bf16 *xp,
                                int32_t *counts, int32_t *offsets, int32_t *padded_offsets,
                                int32_t *row_of, int32_t *tok_of, moe_stream stream);

/* Failure test of the GEMM pipeline (no counterpart on the pages): runs the planning
 * kernel and the gate_up GEMM of moe_expert_ffn with the TMA loads of every CTA's first
 * k-block withheld, so that stage is never filled and every pipeline wait of the kernel
 * gives up after wait_limit_us microseconds (1 .. 10^6). The kernel then records
 * MOE_ERR_TIMEOUT in the status word of ws, waits (bounded) for its own copies, frees
 * its tensor memory and returns; moe_check_device_status(ws) reports it and the CUDA
 * context stays usable. h receives undefined values. Arguments as moe_expert_ffn. */
moe_status moe_debug_gate_up_withheld(moe_shape s, const moe_bf16 *xp, const int32_t *counts,
                                      const moe_bf16 *w_gu, moe_bf16 *h, void *ws,
                                      size_t ws_bytes, int wait_limit_us, moe_stream stream);

/* Device-side status of a workspace or scratch: synchronises `stream`, reads the
 * status word that the kernels set when a pipeline wait runs past its time limit (or,
 * for moe_ep_regroup, when the received counts are inconsistent), and clears it.
 * Returns MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_INVALID_ARG. */
moe_status moe_check_device_status(const void *ws_or_scratch, moe_stream stream);

/* Launch timing for measurement. While enabled, the library brackets each kernel
 * it launches with a pair of CUDA events recorded on that kernel's stream.
 * moe_profile_stop synchronises those events and writes, for each launch in order,
 * a static kernel name and its duration in milliseconds; it returns the number of
 * launches recorded (at most `capacity` given to moe_profile_start) or a negative
 * moe_status. Not thread-safe: for one host thread at a time. */
typedef struct {
  const char *name;
  float ms;
} moe_launch_time;
moe_status moe_profile_start(int capacity);
int moe_profile_stop(moe_launch_time *out, int out_capacity);

/* Stage timing of the grouped GEMMs (a measurement aid with no counterpart on the pages).
 * Only the diagnostic build of the library (compiled with MOE_STAGE_TIMING,
 * lib/libmoe_gb300_timing.so, built by `python -m moe_expert_layer_route_gb300.stage_timing`)
 * has it; in the shipped library both calls return MOE_ERR_UNSUPPORTED (the stamps cost ~2%
 * of the GEMMs' time even unarmed). Armed for one GEMM kind (0 gate_up, 1 down, 2 dgrad_h, 3 dgrad_x,
 * 4 the weight gradients; -1 disarms), the next launches of that kind have their CTA 0
 * stamp the SM clock (clock64) at each pipeline stage and each tile into device arrays that
 * every GPU loading the library holds (8192 stages, 2048 tiles; later launches overwrite
 * earlier ones). Arming clears the stamps; calls that overlap on the GPU race on them.
 * moe_stage_timing_read synchronises the device and copies them out:
 *   stages [8192 x 4] out: per stage, the producer's free-slot wait ended, its loads
 *     issued, the MMA issuer's full-stage wait ended, its MMAs and commit issued;
 *   tiles [2048 x 2] out: per tile of CTA 0, accumulator seen ready by its first epilogue
 *     warp, accumulator released;
 * and returns the number of stages stamped, or a negative moe_status. */
moe_status moe_stage_timing_arm(int kind);
int moe_stage_timing_read(uint64_t *stages, int stage_capacity, uint64_t *tiles,
                          int tile_capacity);

/* Number of kernels the library has launched since it was loaded. */
int64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
