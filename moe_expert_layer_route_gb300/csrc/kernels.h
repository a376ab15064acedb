// Internal interface between the C-ABI layer (moe_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"
#include "common.cuh"

namespace moe {

// Host-side checks shared by the entry points (moe_api.cu): the shape rules of the
// C ABI header, and that the current device is an sm_103 GPU (MOE_ERR_UNSUPPORTED
// otherwise).
moe_status check_shape(const moe_shape &s);
moe_status check_device();

constexpr int kTileRows = 128;  // rows of one GEMM tile; expert segments are padded to it

// Launch bookkeeping (moe_api.cu): launch_begin() before a kernel launch records a
// start event when profiling is on; note_launch() after it records the end event,
// counts the launch and returns cudaGetLastError().
void launch_begin(cudaStream_t st);
cudaError_t note_launch(const char *name, cudaStream_t st);

// route_dispatch.cu
// bias [E] (selection bias) and prob_part [E x ceil(T/32)] (per-chunk softmax sums for
// the load-balancing statistics) may be null
// Outputs of the scan that the fused route + count + scan launch writes; done is a
// zeroed int32 the launch's blocks take tickets from (left zeroed again).
struct ScanOut {
  int32_t *counts = nullptr, *offsets = nullptr, *padded = nullptr, *tile_expert = nullptr,
          *pair_start = nullptr, *pair_expert = nullptr;
  float *aux = nullptr;
  int *done = nullptr;
};
cudaError_t launch_route_count_scan(const float *logits, const float *bias, int32_t *ids,
                                   float *w, int32_t *rank, int32_t *hist, float *prob_part,
                                   int T, int E, int k, const ScanOut &so, cudaStream_t st);
cudaError_t launch_route(const float *logits, const float *bias, int32_t *ids, float *w,
                         int32_t *rank, int32_t *hist, float *prob_part, int T, int E, int k,
                         bool with_count, cudaStream_t st);
// router.cu: logits = x W_r^T (fp32) and the route of launch_route from them; status
// (may be null) records a staging load that timed out
cudaError_t launch_router_route(const void *x, const void *w_r, const float *bias, float *logits,
                                int32_t *ids, float *w, int32_t *rank, int32_t *hist,
                                float *prob_part, int *status, int T, int d, int E, int k,
                                bool with_count, cudaStream_t st);
// dX += dlogits W_r (bf16 in/out) and dW_r = dlogits^T x (fp32), the latter through
// router_dw_splits(T, d, E) token splits whose partials (E*d floats each) go to part
int router_dw_splits(int T, int d, int E);
cudaError_t launch_router_dx(const void *w_r, const float *dlogits, void *dx, int T, int d,
                             int E, cudaStream_t st);
cudaError_t launch_router_dw(const void *x, const float *dlogits, float *dw, float *part, int T,
                             int d, int E, cudaStream_t st);
cudaError_t launch_aux_grad(const float *logits, const int32_t *counts, float coeff,
                            float *dlogits, int T, int E, int k, cudaStream_t st);
cudaError_t launch_count(const int32_t *ids, int32_t *rank, int32_t *hist, int T, int E, int k,
                         cudaStream_t st);
// pair_start / pair_expert may be null (then only the 128-row tile table is written);
// with prob_part also aux = [f_e (E), P_e (E), E * sum f_e P_e]
cudaError_t launch_scan(int32_t *hist, int T, int E, int k, int32_t *counts, int32_t *offsets,
                        int32_t *padded, int32_t *tile_expert, int32_t *pair_start,
                        int32_t *pair_expert, const float *prob_part, float *aux,
                        cudaStream_t st);
cudaError_t launch_plan(const int32_t *counts, int E, int32_t *offsets, int32_t *padded,
                        int32_t *tile_expert, int32_t *pair_start, int32_t *pair_expert,
                        cudaStream_t st);
cudaError_t launch_scatter(const void *x, const int32_t *ids, const int32_t *rank,
                           const int32_t *hist, const int32_t *padded, const int32_t *counts,
                           int32_t *row_of, int32_t *tok_of, void *xp, int T, int d, int E, int k,
                           int R, cudaStream_t st);
cudaError_t launch_combine(const void *o, const float *w, const int32_t *row_of, void *y, int T,
                           int d, int k, cudaStream_t st);
cudaError_t launch_gather_sum(const void *dxp, const int32_t *row_of, void *dx, int T, int d,
                              int k, cudaStream_t st);
// with dlogits (T x E fp32, may be null) also the router-logit gradient from o and ids
cudaError_t launch_scale_scatter(const void *dy, const float *w, const int32_t *row_of,
                                 const int32_t *padded, const int32_t *counts, void *g, int T,
                                 int d, int E, int k, const void *o, const int32_t *ids,
                                 float *dlogits, cudaStream_t st);

// grouped_gemm.cu -- the tcgen05 grouped GEMM engine.
//
// Ragged-M problems (one per expert, rows = the expert's padded segment):
//   GATE_UP   : H = swiglu(Xp W_gu[e]) [+ GU saved]      A = Xp   [R x d]   K-major
//                                                        B = W_gu [E x d x 2f] MN-major
//   DOWN      : O = H W_down[e]                          A = H    [R x f]   K-major
//                                                        B = W_down [E x f x d] MN-major
//   DGRAD_H   : dGU = swiglu_bwd(G W_down[e]^T, GU)      A = G    [R x d]   K-major
//                                                        B = W_down [E x f x d] K-major
//   DGRAD_X   : dXp = dGU W_gu[e]^T                      A = dGU  [R x 2f]  K-major
//                                                        B = W_gu [E x d x 2f] K-major
// Ragged-K problems (one per expert, K = the expert's padded segment):
//   WGRAD     : dW[e] = X_e^T Y_e                        A = X [R x M] MN-major
//                                                        B = Y [R x N] MN-major
struct GemmPlan {
  const int32_t *padded;       // [E+1] padded segment starts
  const int32_t *counts;       // [E] rows per expert
  const int32_t *tile_expert;  // [R/128] expert of each 128-row tile
  const int32_t *pair_start;   // [E+1] first 256-row pair-tile of each expert
  const int32_t *pair_expert;  // [R/128] expert of each pair-tile
  int E;
  int64_t R;                   // rows of the padded space
  int64_t rows_per_expert;     // T*k / E, the mean segment length (picks the tile order)
  unsigned long long wait_ns = 0;  // pipeline wait limit (0 = the default kWaitLimitNs)
  int withhold_kblock = -1;        // failure test: k-block whose loads are withheld
};

cudaError_t gemm_gate_up(const GemmPlan &p, const void *xp, const void *w_gu, void *h, void *gu,
                         int d, int f, int *status, cudaStream_t st);
cudaError_t gemm_down(const GemmPlan &p, const void *h, const void *w_down, void *o, int d, int f,
                      int *status, cudaStream_t st);
cudaError_t gemm_dgrad_h(const GemmPlan &p, const void *g, const void *w_down, const void *gu,
                         void *dgu, int d, int f, int *status, cudaStream_t st);
cudaError_t gemm_dgrad_x(const GemmPlan &p, const void *dgu, const void *w_gu, void *dxp, int d,
                         int f, int *status, cudaStream_t st);
// dW[e] (M x N, bf16, row-major, experts contiguous) = X_e^T Y_e over the padded
// segment rows of expert e; X is R x M, Y is R x N.
cudaError_t gemm_wgrad(const GemmPlan &p, const void *x, const void *y, void *dw, int M, int N,
                       int *status, const char *name, cudaStream_t st);

// cuTensorMapEncodeTiled through the driver entry point (resolved once): bf16
// elements, zero fill out of bounds, swizzle 128 or 64 (bytes).
cudaError_t encode_tensor_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                              const uint64_t *strides_bytes, const uint32_t *box, int swizzle);

// ep.cu: the received rows (source-major [s][e][rows], recv_counts [G][El]) to the
// segment-padded expert-major layout of the local experts (zero padding rows), with
// dest_of[i] the padded row of received row i; status records kDevBadCounts when the
// counts do not add up to n_recv or overflow the R padded rows (then nothing is written)
cudaError_t launch_ep_regroup(const int32_t *recv_counts, const void *xr, void *xp,
                              int32_t *counts_loc, int32_t *padded_loc, int32_t *dest_of,
                              int *status, int G, int El, int n_recv, int R, int d,
                              cudaStream_t st);
// out[i] = o[dest_of[i]] (rows of d bf16), i < n_recv; dest_of outside [0, R) is skipped
cudaError_t launch_ep_unregroup(const void *o, const int32_t *dest_of, void *out, int n_recv,
                                int R, int d, cudaStream_t st);

// Stage timing of the grouped GEMMs (grouped_gemm.cu): arm for one kind (0 gate_up, 1
// down, 2 dgrad_h, 3 dgrad_x, 4 weight gradients; -1 disarms), clearing the stamps; read
// kTimingStages x 4 and kTimingTiles x 2 stamps (synchronises the device)
constexpr int kTimingStages = 8192;
constexpr int kTimingTiles = 2048;
cudaError_t stage_timing_arm(int kind);
cudaError_t stage_timing_read(unsigned long long *stages, unsigned long long *tiles);

int num_sms();

}  // namespace moe
