// C ABI of the MoE expert block: argument checks, workspace layout, and the launch
// sequences of each entry point. The arithmetic is in route_dispatch.cu and
// grouped_gemm.cu; this file only validates, carves workspaces and orders launches.
#include <atomic>
#include <mutex>
#include <set>
#include <string>
#include <vector>

#include "../../include/moe_gb300.h"
#include "kernels.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct FwdLayout {
  size_t status, ids, w, rank, hist, prob_part, counts, offsets, padded, tile_expert, pair_start,
      pair_expert, row_of, tok_of, xp, gu, h, o, total;
};

struct BwdLayout {
  size_t status, g, dgu, dxp, total;
};

int64_t padded_rows(const moe_shape &s) {
  const int64_t A = s.T * s.k;
  return (int64_t)kTileRows * ((A + kTileRows - 1) / kTileRows + s.E);
}

FwdLayout fwd_layout(const moe_shape &s, int training) {
  FwdLayout L{};
  const int64_t A = s.T * s.k, R = padded_rows(s);
  const int64_t C = (s.T + 31) / 32 > 0 ? (s.T + 31) / 32 : 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  L.status = take(kAlign);
  L.ids = take(A * 4);
  L.w = take(A * 4);
  L.rank = take(A * 4);
  L.hist = take((size_t)s.E * C * 4);
  L.prob_part = take((size_t)s.E * C * 4);
  L.counts = take(s.E * 4);
  L.offsets = take((s.E + 1) * 4);
  L.padded = take((s.E + 1) * 4);
  L.tile_expert = take(R / kTileRows * 4);
  L.pair_start = take((s.E + 1) * 4);
  L.pair_expert = take(R / kTileRows * 4);
  L.row_of = take(A * 4);
  L.tok_of = take(R * 4);
  L.xp = take((size_t)R * s.d * 2);
  L.gu = training ? take((size_t)R * 2 * s.f * 2) : 0;
  L.h = take((size_t)R * s.f * 2);
  L.o = take((size_t)R * s.d * 2);
  L.total = off;
  return L;
}

BwdLayout bwd_layout(const moe_shape &s) {
  BwdLayout L{};
  const int64_t R = padded_rows(s);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  L.status = take(kAlign);
  L.g = take((size_t)R * s.d * 2);
  L.dgu = take((size_t)R * 2 * s.f * 2);
  L.dxp = take((size_t)R * s.d * 2);
  L.total = off;
  return L;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <typename... P>
moe_status check_ptrs(P... ptrs) {
  const void *a[] = {static_cast<const void *>(ptrs)...};
  for (const void *p : a) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_ALIGNMENT;
  }
  return MOE_OK;
}

// A second stream per device for independent kernels of one call that run side by
// side (the router GEMM's two gradients). Each use is a fork (event on the caller's
// stream, waited by the side stream) and a join (event on the side stream, waited by
// the caller's stream) enqueued under one lock, so the calls of several host threads
// do not interleave their event records.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool tried = false;
};
std::mutex g_side_mu;
SideStream g_side[64];

// The side stream of the current device, or null (then the work stays on the caller's
// stream). Call with g_side_mu held.
SideStream *side_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  SideStream &sd = g_side[dev & 63];
  if (!sd.tried) {
    sd.tried = true;
    if (cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) {
      sd.s = nullptr;
      cudaGetLastError();
    }
  }
  return sd.s ? &sd : nullptr;
}

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                   \
  do {                                  \
    const moe_status _s = (expr);       \
    if (_s != MOE_OK) return _s;        \
  } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

template <typename T>
T *at(void *base, size_t off) {
  return reinterpret_cast<T *>(static_cast<uint8_t *>(base) + off);
}

// ----------------------------------------------------------------- profiling state
std::atomic<int64_t> g_launches{0};
struct Prof {
  bool on = false;
  int cap = 0, used = 0;
  std::vector<cudaEvent_t> start, stop;
  std::vector<const char *> names;
  bool pending = false;
} g_prof;


bool on_side_stream(cudaStream_t st) {
  if (!st) return false;
  for (const SideStream &sd : g_side)
    if (sd.s == st) return true;
  return false;
}

// "<name> (overlapped)", interned (the profile keeps the pointers)
const char *overlapped_name(const char *name) {
  static std::mutex mu;
  static std::set<std::string> names;
  std::lock_guard<std::mutex> lock(mu);
  return names.insert(std::string(name) + " (overlapped)").first->c_str();
}

}  // namespace

namespace moe {

// Host-side checks shared by every entry point (declared in kernels.h).
moe_status check_shape(const moe_shape &s) {
  if (s.T < 0 || s.d <= 0 || s.E <= 0 || s.k <= 0 || s.f <= 0) return MOE_ERR_INVALID_ARG;
  if (s.k > s.E) return MOE_ERR_INVALID_ARG;
  if (s.E > 256 || s.k > 16) return MOE_ERR_UNSUPPORTED;
  if (s.d % 8 != 0 || s.f % 8 != 0) return MOE_ERR_ALIGNMENT;
  if (s.d > (1 << 20) || s.f > (1 << 20)) return MOE_ERR_UNSUPPORTED;
  const int64_t lim = (int64_t)1 << 31;
  if (s.T >= lim / s.k) return MOE_ERR_OVERFLOW;            // T*k fits int32
  if (padded_rows(s) >= lim) return MOE_ERR_OVERFLOW;       // padded rows fit int32
  return MOE_OK;
}

moe_status check_device() {
  static int ok[64] = {};  // 0 unknown, 1 good, -1 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int &v = ok[dev & 63];
  if (v == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    v = (major == 10 && minor == 3) ? 1 : -1;
  }
  return v == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

}  // namespace moe

namespace moe {

void launch_begin(cudaStream_t st) {
  if (g_prof.on && g_prof.used < g_prof.cap) {
    cudaEventRecord(g_prof.start[g_prof.used], st);
    g_prof.pending = true;
  }
}

cudaError_t note_launch(const char *name, cudaStream_t st) {
  const cudaError_t e = cudaGetLastError();
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (g_prof.on && g_prof.pending) {
    cudaEventRecord(g_prof.stop[g_prof.used], st);
    // a launch on the side stream overlaps others: its events span them too
    g_prof.names[g_prof.used] = on_side_stream(st) ? overlapped_name(name) : name;
    ++g_prof.used;
    g_prof.pending = false;
  }
  return e;
}

}  // namespace moe

extern "C" {

const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or device";
    case MOE_ERR_ALIGNMENT: return "misaligned pointer or dimension";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_OVERFLOW: return "index overflow";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
  }
  return "unknown status";
}

int64_t moe_padded_rows(moe_shape s) {
  if (check_shape(s) != MOE_OK) return -1;
  return padded_rows(s);
}

size_t moe_workspace_size(moe_shape s, int training) {
  if (check_shape(s) != MOE_OK) return 0;
  return fwd_layout(s, training).total;
}

size_t moe_backward_scratch_size(moe_shape s) {
  if (check_shape(s) != MOE_OK) return 0;
  return bwd_layout(s).total;
}

moe_status moe_workspace_views(moe_shape s, int training, void *ws, size_t ws_bytes,
                               moe_forward_views *out) {
  MOE_TRY(check_shape(s));
  if (!ws || !out) return MOE_ERR_INVALID_ARG;
  const FwdLayout L = fwd_layout(s, training);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  out->ids = at<int32_t>(ws, L.ids);
  out->w = at<float>(ws, L.w);
  out->counts = at<int32_t>(ws, L.counts);
  out->offsets = at<int32_t>(ws, L.offsets);
  out->padded_offsets = at<int32_t>(ws, L.padded);
  out->row_of = at<int32_t>(ws, L.row_of);
  out->tok_of = at<int32_t>(ws, L.tok_of);
  out->xp = at<moe_bf16>(ws, L.xp);
  out->gu = training ? at<moe_bf16>(ws, L.gu) : nullptr;
  out->h = at<moe_bf16>(ws, L.h);
  out->o = at<moe_bf16>(ws, L.o);
  return MOE_OK;
}

moe_status moe_route(moe_shape s, const float *logits, int32_t *ids, float *w,
                     const moe_route_options *opts, moe_stream stream) {
  MOE_TRY(check_shape(s));
  const float *bias = opts ? opts->selection_bias : nullptr;
  if (bias && !aligned16(bias)) return MOE_ERR_ALIGNMENT;
  if (s.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs(logits, ids, w));
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_CUDA(launch_route(logits, bias, ids, w, nullptr, nullptr, nullptr, (int)s.T, (int)s.E,
                        (int)s.k, false, st));
  return MOE_OK;
}

moe_status moe_dispatch(moe_shape s, const moe_bf16 *x, const int32_t *ids, moe_bf16 *xp,
                        int32_t *counts, int32_t *offsets, int32_t *padded_offsets,
                        int32_t *row_of, int32_t *tok_of, void *ws, size_t ws_bytes,
                        moe_stream stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_ptrs(xp, counts, offsets, padded_offsets, tok_of, ws));
  if (s.T > 0) MOE_TRY(check_ptrs(x, ids, row_of));
  const FwdLayout L = fwd_layout(s, 0);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = (int)s.T, E = (int)s.E, k = (int)s.k, d = (int)s.d;
  int32_t *rank = at<int32_t>(ws, L.rank), *hist = at<int32_t>(ws, L.hist);
  MOE_CUDA(launch_count(ids, rank, hist, T, E, k, st));
  MOE_CUDA(launch_scan(hist, T, E, k, counts, offsets, padded_offsets,
                       at<int32_t>(ws, L.tile_expert), nullptr, nullptr, nullptr, nullptr, st));
  MOE_CUDA(launch_scatter(x, ids, rank, hist, padded_offsets, counts, row_of, tok_of, xp, T, d, E,
                          k, (int)padded_rows(s), st));
  return MOE_OK;
}

moe_status moe_expert_ffn(moe_shape s, const moe_bf16 *xp, const int32_t *counts,
                          const moe_bf16 *w_gu, const moe_bf16 *w_down, moe_bf16 *h,
                          moe_bf16 *gu, moe_bf16 *o, void *ws, size_t ws_bytes,
                          moe_stream stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_ptrs(xp, counts, w_gu, w_down, h, o, ws));
  if (gu && !aligned16(gu)) return MOE_ERR_ALIGNMENT;
  const FwdLayout L = fwd_layout(s, 0);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int *status = at<int>(ws, L.status);
  MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  int32_t *padded = at<int32_t>(ws, L.padded), *tiles = at<int32_t>(ws, L.tile_expert);
  int32_t *pstart = at<int32_t>(ws, L.pair_start), *pexp = at<int32_t>(ws, L.pair_expert);
  MOE_CUDA(launch_plan(counts, (int)s.E, at<int32_t>(ws, L.offsets), padded, tiles, pstart, pexp,
                       st));
  const GemmPlan p{padded, counts, tiles, pstart, pexp, (int)s.E, padded_rows(s), s.T * s.k / s.E};
  MOE_CUDA(gemm_gate_up(p, xp, w_gu, h, gu, (int)s.d, (int)s.f, status, st));
  MOE_CUDA(gemm_down(p, h, w_down, o, (int)s.d, (int)s.f, status, st));
  return MOE_OK;
}

moe_status moe_combine(moe_shape s, const moe_bf16 *o, const float *w, const int32_t *row_of,
                       moe_bf16 *y, moe_stream stream) {
  MOE_TRY(check_shape(s));
  if (s.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs(o, row_of, y));
  if (w && !aligned16(w)) return MOE_ERR_ALIGNMENT;
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (w) MOE_CUDA(launch_combine(o, w, row_of, y, (int)s.T, (int)s.d, (int)s.k, st));
  else MOE_CUDA(launch_gather_sum(o, row_of, y, (int)s.T, (int)s.d, (int)s.k, st));
  return MOE_OK;
}

}  // extern "C"

namespace {

// The forward from router logits in memory (w_router null) or from the router GEMM
// (w_router set: logits is then written).
moe_status forward_impl(moe_shape s, const moe_bf16 *x, const float *logits_in,
                        const moe_bf16 *w_router, float *logits_out, const moe_bf16 *w_gu,
                        const moe_bf16 *w_down, moe_bf16 *y, int training,
                        const moe_route_options *opts, void *ws, size_t ws_bytes,
                        moe_stream stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_ptrs(w_gu, w_down, ws));
  const float *bias = opts ? opts->selection_bias : nullptr;
  float *aux = opts ? opts->aux_stats : nullptr;
  if ((bias && !aligned16(bias)) || (aux && !aligned16(aux))) return MOE_ERR_ALIGNMENT;
  if (s.T > 0) {
    MOE_TRY(check_ptrs(x, y));
    MOE_TRY(w_router ? check_ptrs(w_router, logits_out) : check_ptrs(logits_in));
  }
  const FwdLayout L = fwd_layout(s, training);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = (int)s.T, E = (int)s.E, k = (int)s.k, d = (int)s.d, f = (int)s.f;
  int *status = at<int>(ws, L.status);
  int32_t *ids = at<int32_t>(ws, L.ids), *rank = at<int32_t>(ws, L.rank);
  int32_t *hist = at<int32_t>(ws, L.hist), *counts = at<int32_t>(ws, L.counts);
  int32_t *padded = at<int32_t>(ws, L.padded), *tiles = at<int32_t>(ws, L.tile_expert);
  int32_t *row_of = at<int32_t>(ws, L.row_of), *tok_of = at<int32_t>(ws, L.tok_of);
  float *w = at<float>(ws, L.w);
  void *xp = at<void>(ws, L.xp), *h = at<void>(ws, L.h), *o = at<void>(ws, L.o);
  void *gu = training ? at<void>(ws, L.gu) : nullptr;
  // the status word and, after it, the ticket counter of the fused route + scan launch
  MOE_CUDA(cudaMemsetAsync(status, 0, 2 * sizeof(int), st));
  float *prob_part = aux ? at<float>(ws, L.prob_part) : nullptr;
  int32_t *pstart = at<int32_t>(ws, L.pair_start), *pexp = at<int32_t>(ws, L.pair_expert);
  if (w_router) {
    MOE_CUDA(launch_router_route(x, w_router, bias, logits_out, ids, w, rank, hist, prob_part,
                                 status, T, d, E, k, true, st));
    MOE_CUDA(launch_scan(hist, T, E, k, counts, at<int32_t>(ws, L.offsets), padded, tiles,
                         pstart, pexp, prob_part, aux, st));
  } else {
    ScanOut so;
    so.counts = counts;
    so.offsets = at<int32_t>(ws, L.offsets);
    so.padded = padded;
    so.tile_expert = tiles;
    so.pair_start = pstart;
    so.pair_expert = pexp;
    so.aux = aux;
    so.done = status + 1;
    MOE_CUDA(launch_route_count_scan(logits_in, bias, ids, w, rank, hist, prob_part, T, E, k, so,
                                     st));
  }
  if (aux && T == 0) MOE_CUDA(cudaMemsetAsync(aux, 0, (2 * E + 1) * sizeof(float), st));
  MOE_CUDA(launch_scatter(x, ids, rank, hist, padded, counts, row_of, tok_of, xp, T, d, E, k,
                          (int)padded_rows(s), st));
  const GemmPlan p{padded, counts, tiles, pstart, pexp, E, padded_rows(s), s.T * s.k / s.E};
  MOE_CUDA(gemm_gate_up(p, xp, w_gu, h, gu, d, f, status, st));
  MOE_CUDA(gemm_down(p, h, w_down, o, d, f, status, st));
  MOE_CUDA(launch_combine(o, w, row_of, y, T, d, k, st));
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_forward(moe_shape s, const moe_bf16 *x, const float *logits, const moe_bf16 *w_gu,
                       const moe_bf16 *w_down, moe_bf16 *y, int training,
                       const moe_route_options *opts, void *ws, size_t ws_bytes,
                       moe_stream stream) {
  return forward_impl(s, x, logits, nullptr, nullptr, w_gu, w_down, y, training, opts, ws,
                      ws_bytes, stream);
}

moe_status moe_forward_router(moe_shape s, const moe_bf16 *x, const moe_bf16 *w_router,
                              float *logits, const moe_bf16 *w_gu, const moe_bf16 *w_down,
                              moe_bf16 *y, int training, const moe_route_options *opts, void *ws,
                              size_t ws_bytes, moe_stream stream) {
  if (s.T > 0 && !w_router) return MOE_ERR_INVALID_ARG;
  return forward_impl(s, x, nullptr, w_router, logits, w_gu, w_down, y, training, opts, ws,
                      ws_bytes, stream);
}

moe_status moe_router_route(moe_shape s, const moe_bf16 *x, const moe_bf16 *w_router,
                            float *logits, int32_t *ids, float *w, const moe_route_options *opts,
                            moe_stream stream) {
  MOE_TRY(check_shape(s));
  const float *bias = opts ? opts->selection_bias : nullptr;
  if (bias && !aligned16(bias)) return MOE_ERR_ALIGNMENT;
  if (s.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs(x, w_router, logits, ids, w));
  MOE_TRY(check_device());
  MOE_CUDA(launch_router_route(x, w_router, bias, logits, ids, w, nullptr, nullptr, nullptr,
                               nullptr, (int)s.T, (int)s.d, (int)s.E, (int)s.k, false,
                               static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_backward(moe_shape s, const moe_bf16 *dy, const moe_bf16 *w_gu,
                        const moe_bf16 *w_down, const void *ws, size_t ws_bytes, moe_bf16 *dx,
                        moe_bf16 *dw_gu, moe_bf16 *dw_down, float *dlogits, void *scratch,
                        size_t scratch_bytes, moe_stream stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_ptrs(w_gu, w_down, ws, dw_gu, dw_down, scratch));
  if (s.T > 0) MOE_TRY(check_ptrs(dy, dx));
  if (dlogits && !aligned16(dlogits)) return MOE_ERR_ALIGNMENT;
  const FwdLayout L = fwd_layout(s, 1);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  const BwdLayout B = bwd_layout(s);
  if (scratch_bytes < B.total) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = (int)s.T, E = (int)s.E, k = (int)s.k, d = (int)s.d, f = (int)s.f;
  void *fws = const_cast<void *>(ws);
  const float *w = at<float>(fws, L.w);
  const int32_t *row_of = at<int32_t>(fws, L.row_of), *counts = at<int32_t>(fws, L.counts);
  const int32_t *padded = at<int32_t>(fws, L.padded), *tiles = at<int32_t>(fws, L.tile_expert);
  const int32_t *pstart = at<int32_t>(fws, L.pair_start), *pexp = at<int32_t>(fws, L.pair_expert);
  const void *xp = at<void>(fws, L.xp), *gu = at<void>(fws, L.gu), *h = at<void>(fws, L.h);
  const void *o = at<void>(fws, L.o);
  const int32_t *ids = at<int32_t>(fws, L.ids);
  int *status = at<int>(scratch, B.status);
  void *g = at<void>(scratch, B.g), *dgu = at<void>(scratch, B.dgu), *dxp = at<void>(scratch, B.dxp);
  const GemmPlan p{padded, counts, tiles, pstart, pexp, E, padded_rows(s), s.T * s.k / s.E};
  MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  MOE_CUDA(launch_scale_scatter(dy, w, row_of, padded, counts, g, T, d, E, k, o, ids,
                                s.T > 0 ? dlogits : nullptr, st));
  // dX first (the input gradient is what the layer below waits for), its gather right
  // after dgrad_x so that it reads dXp while the L2 still holds much of it (at
  // gpt_oss_20b 22 us against 27 us after the weight gradients), then the weight gradients
  MOE_CUDA(gemm_dgrad_h(p, g, w_down, gu, dgu, d, f, status, st));
  MOE_CUDA(gemm_dgrad_x(p, dgu, w_gu, dxp, d, f, status, st));
  MOE_CUDA(launch_gather_sum(dxp, row_of, dx, T, d, k, st));
  MOE_CUDA(gemm_wgrad(p, h, g, dw_down, f, d, status, "gemm_wgrad_down", st));
  MOE_CUDA(gemm_wgrad(p, xp, dgu, dw_gu, d, 2 * f, status, "gemm_wgrad_gu", st));
  return MOE_OK;
}

moe_status moe_expert_ffn_backward(moe_shape s, const moe_bf16 *g, const moe_bf16 *xp,
                                   const moe_bf16 *gu, const moe_bf16 *h, const int32_t *counts,
                                   const moe_bf16 *w_gu, const moe_bf16 *w_down, moe_bf16 *dxp,
                                   moe_bf16 *dw_gu, moe_bf16 *dw_down, void *ws, size_t ws_bytes,
                                   void *scratch, size_t scratch_bytes, moe_stream stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_ptrs(g, xp, gu, h, counts, w_gu, w_down, dxp, dw_gu, dw_down, ws, scratch));
  const FwdLayout L = fwd_layout(s, 0);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  const BwdLayout B = bwd_layout(s);
  if (scratch_bytes < B.total) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int E = (int)s.E, d = (int)s.d, f = (int)s.f;
  int *status = at<int>(ws, L.status);
  int32_t *padded = at<int32_t>(ws, L.padded), *tiles = at<int32_t>(ws, L.tile_expert);
  int32_t *pstart = at<int32_t>(ws, L.pair_start), *pexp = at<int32_t>(ws, L.pair_expert);
  void *dgu = at<void>(scratch, B.dgu);
  MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  MOE_CUDA(launch_plan(counts, E, at<int32_t>(ws, L.offsets), padded, tiles, pstart, pexp, st));
  const GemmPlan p{padded, counts, tiles, pstart, pexp, E, padded_rows(s), s.T * s.k / s.E};
  MOE_CUDA(gemm_dgrad_h(p, g, w_down, gu, dgu, d, f, status, st));
  MOE_CUDA(gemm_wgrad(p, h, g, dw_down, f, d, status, "gemm_wgrad_down", st));
  MOE_CUDA(gemm_dgrad_x(p, dgu, w_gu, dxp, d, f, status, st));
  MOE_CUDA(gemm_wgrad(p, xp, dgu, dw_gu, d, 2 * f, status, "gemm_wgrad_gu", st));
  return MOE_OK;
}

moe_status moe_ep_local_shape(moe_shape s, int G, moe_shape *out) {
  MOE_TRY(check_shape(s));
  if (!out || G < 1 || G > s.E || s.E % G != 0) return MOE_ERR_INVALID_ARG;
  moe_shape l = s;
  l.E = s.E / G;
  l.T = s.T * G;
  l.k = s.k < l.E ? s.k : l.E;
  MOE_TRY(check_shape(l));
  *out = l;
  return MOE_OK;
}

moe_status moe_ep_dispatch(moe_shape s, const moe_bf16 *x, const int32_t *ids, moe_bf16 *xs,
                           int32_t *counts, int32_t *offsets, int32_t *row_of, void *ws,
                           size_t ws_bytes, moe_stream stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_ptrs(counts, offsets, ws));
  if (s.T > 0) MOE_TRY(check_ptrs(x, ids, xs, row_of));
  const FwdLayout L = fwd_layout(s, 0);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = (int)s.T, E = (int)s.E, k = (int)s.k, d = (int)s.d;
  int32_t *rank = at<int32_t>(ws, L.rank), *hist = at<int32_t>(ws, L.hist);
  MOE_CUDA(launch_count(ids, rank, hist, T, E, k, st));
  MOE_CUDA(launch_scan(hist, T, E, k, counts, offsets, at<int32_t>(ws, L.padded),
                       at<int32_t>(ws, L.tile_expert), nullptr, nullptr, nullptr, nullptr, st));
  // the compact layout: the segment starts are the compact offsets (no padding rows),
  // and the row space ends at A = T k
  if (T > 0)
    MOE_CUDA(launch_scatter(x, ids, rank, hist, offsets, counts, row_of, at<int32_t>(ws, L.tok_of),
                            xs, T, d, E, k, T * k, st));
  return MOE_OK;
}

moe_status moe_ep_regroup(moe_shape s_loc, int G, const int32_t *recv_counts, int64_t n_recv,
                          const moe_bf16 *xr, moe_bf16 *xp, int32_t *counts_loc,
                          int32_t *padded_loc, int32_t *dest_of, void *ws, size_t ws_bytes,
                          moe_stream stream) {
  MOE_TRY(check_shape(s_loc));
  if (G < 1 || G * s_loc.E > 256 || n_recv < 0) return MOE_ERR_INVALID_ARG;
  if (n_recv > s_loc.T * s_loc.k) return MOE_ERR_WORKSPACE;  // beyond the local row space
  MOE_TRY(check_ptrs(recv_counts, xp, counts_loc, padded_loc, ws));
  if (n_recv > 0) MOE_TRY(check_ptrs(xr, dest_of));
  const FwdLayout L = fwd_layout(s_loc, 0);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int *status = at<int>(ws, L.status);
  MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  MOE_CUDA(launch_ep_regroup(recv_counts, xr, xp, counts_loc, padded_loc, dest_of, status, G,
                             (int)s_loc.E, (int)n_recv, (int)padded_rows(s_loc), (int)s_loc.d,
                             st));
  return MOE_OK;
}

moe_status moe_ep_unregroup(moe_shape s_loc, int64_t n_recv, const moe_bf16 *o,
                            const int32_t *dest_of, moe_bf16 *out, moe_stream stream) {
  MOE_TRY(check_shape(s_loc));
  if (n_recv < 0) return MOE_ERR_INVALID_ARG;
  if (n_recv > s_loc.T * s_loc.k) return MOE_ERR_WORKSPACE;
  if (n_recv == 0) return MOE_OK;
  MOE_TRY(check_ptrs(o, dest_of, out));
  MOE_TRY(check_device());
  MOE_CUDA(launch_ep_unregroup(o, dest_of, out, (int)n_recv, (int)padded_rows(s_loc),
                               (int)s_loc.d, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_ep_grad_scatter(moe_shape s, const moe_bf16 *dy, const float *w,
                               const int32_t *ids, const int32_t *counts, const int32_t *offsets,
                               const int32_t *row_of, const moe_bf16 *ob, moe_bf16 *gs,
                               float *dlogits, moe_stream stream) {
  MOE_TRY(check_shape(s));
  if (s.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs(dy, w, ids, counts, offsets, row_of, gs));
  if (dlogits) MOE_TRY(check_ptrs(dlogits, ob));
  MOE_TRY(check_device());
  // compact rows: the segment starts are the compact offsets, so no padding row exists
  MOE_CUDA(launch_scale_scatter(dy, w, row_of, offsets, counts, gs, (int)s.T, (int)s.d, (int)s.E,
                                (int)s.k, ob, ids, dlogits, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

size_t moe_router_backward_scratch_size(moe_shape s) {
  if (check_shape(s) != MOE_OK) return 0;
  const int splits = router_dw_splits((int)s.T, (int)s.d, (int)s.E);
  return splits > 1 ? (size_t)splits * s.E * s.d * sizeof(float) : 16;
}

moe_status moe_router_backward(moe_shape s, const moe_bf16 *x, const moe_bf16 *w_router,
                               const float *dlogits, moe_bf16 *dx, float *dw_router,
                               void *scratch, size_t scratch_bytes, moe_stream stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_ptrs(w_router, dw_router, scratch));
  if (s.T > 0) MOE_TRY(check_ptrs(x, dlogits, dx));
  if (scratch_bytes < moe_router_backward_scratch_size(s)) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (s.T == 0) {
    MOE_CUDA(cudaMemsetAsync(dw_router, 0, (size_t)s.E * s.d * sizeof(float), st));
    return MOE_OK;
  }
  // dW_r (token splits, then their sum) runs beside the dX term on the side stream
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream *sd = side_stream();
  cudaStream_t wst = st;
  if (sd) {
    MOE_CUDA(cudaEventRecord(sd->fork, st));
    MOE_CUDA(cudaStreamWaitEvent(sd->s, sd->fork, 0));
    wst = sd->s;
  }
  const cudaError_t ew = launch_router_dw(x, dlogits, dw_router, static_cast<float *>(scratch),
                                          (int)s.T, (int)s.d, (int)s.E, wst);
  if (sd) MOE_CUDA(cudaEventRecord(sd->join, sd->s));
  const cudaError_t ex = launch_router_dx(w_router, dlogits, dx, (int)s.T, (int)s.d, (int)s.E, st);
  if (sd) MOE_CUDA(cudaStreamWaitEvent(st, sd->join, 0));
  MOE_CUDA(ew);
  MOE_CUDA(ex);
  return MOE_OK;
}

moe_status moe_aux_loss_backward(moe_shape s, const float *logits, const int32_t *counts,
                                 float coeff, float *dlogits, moe_stream stream) {
  MOE_TRY(check_shape(s));
  if (s.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs(logits, counts, dlogits));
  MOE_TRY(check_device());
  MOE_CUDA(launch_aux_grad(logits, counts, coeff, dlogits, (int)s.T, (int)s.E, (int)s.k,
                           static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_debug_gate_up_withheld(moe_shape s, const moe_bf16 *xp, const int32_t *counts,
                                      const moe_bf16 *w_gu, moe_bf16 *h, void *ws,
                                      size_t ws_bytes, int wait_limit_us, moe_stream stream) {
  MOE_TRY(check_shape(s));
  MOE_TRY(check_ptrs(xp, counts, w_gu, h, ws));
  if (wait_limit_us <= 0 || wait_limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  const FwdLayout L = fwd_layout(s, 0);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  MOE_TRY(check_device());
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int *status = at<int>(ws, L.status);
  MOE_CUDA(cudaMemsetAsync(status, 0, sizeof(int), st));
  int32_t *padded = at<int32_t>(ws, L.padded), *tiles = at<int32_t>(ws, L.tile_expert);
  int32_t *pstart = at<int32_t>(ws, L.pair_start), *pexp = at<int32_t>(ws, L.pair_expert);
  MOE_CUDA(launch_plan(counts, (int)s.E, at<int32_t>(ws, L.offsets), padded, tiles, pstart, pexp,
                       st));
  GemmPlan p{padded, counts, tiles, pstart, pexp, (int)s.E, padded_rows(s), s.T * s.k / s.E};
  p.wait_ns = 1000ull * (unsigned long long)wait_limit_us;
  p.withhold_kblock = 0;
  MOE_CUDA(gemm_gate_up(p, xp, w_gu, h, nullptr, (int)s.d, (int)s.f, status, st));
  return MOE_OK;
}

moe_status moe_check_device_status(const void *ws_or_scratch, moe_stream stream) {
  if (!ws_or_scratch) return MOE_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  MOE_CUDA(cudaMemcpyAsync(&v, ws_or_scratch, sizeof(int), cudaMemcpyDeviceToHost, st));
  MOE_CUDA(cudaStreamSynchronize(st));
  if (v != kDevOk) {
    MOE_CUDA(cudaMemsetAsync(const_cast<void *>(ws_or_scratch), 0, sizeof(int), st));
    MOE_CUDA(cudaStreamSynchronize(st));
    return v == kDevBadCounts ? MOE_ERR_INVALID_ARG : MOE_ERR_TIMEOUT;
  }
  return MOE_OK;
}

moe_status moe_profile_start(int capacity) {
  if (capacity <= 0) return MOE_ERR_INVALID_ARG;
  for (cudaEvent_t e : g_prof.start) cudaEventDestroy(e);
  for (cudaEvent_t e : g_prof.stop) cudaEventDestroy(e);
  g_prof = Prof{};
  g_prof.start.resize(capacity);
  g_prof.stop.resize(capacity);
  g_prof.names.resize(capacity);
  for (int i = 0; i < capacity; ++i) {
    if (cudaEventCreate(&g_prof.start[i]) != cudaSuccess ||
        cudaEventCreate(&g_prof.stop[i]) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  g_prof.cap = capacity;
  g_prof.on = true;
  return MOE_OK;
}

int moe_profile_stop(moe_launch_time *out, int out_capacity) {
  if (!g_prof.on) return 0;
  g_prof.on = false;
  const int n = g_prof.used;
  for (int i = 0; i < n && i < out_capacity; ++i) {
    if (cudaEventSynchronize(g_prof.stop[i]) != cudaSuccess) return MOE_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof.start[i], g_prof.stop[i]) != cudaSuccess)
      return MOE_ERR_CUDA;
    out[i].name = g_prof.names[i];
    out[i].ms = ms;
  }
  return n;
}

moe_status moe_stage_timing_arm(int kind) {
  if (kind < -1 || kind > 4) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_device());
  const cudaError_t e = stage_timing_arm(kind);
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;  // not the diagnostic build
  MOE_CUDA(e);
  return MOE_OK;
}

int moe_stage_timing_read(uint64_t *stages, int stage_capacity, uint64_t *tiles,
                          int tile_capacity) {
  if (!stages || !tiles || stage_capacity < kTimingStages || tile_capacity < kTimingTiles)
    return MOE_ERR_INVALID_ARG;
  const moe_status dev = check_device();
  if (dev != MOE_OK) return dev;
  const cudaError_t e = stage_timing_read(reinterpret_cast<unsigned long long *>(stages),
                                          reinterpret_cast<unsigned long long *>(tiles));
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  int n = 0;
  while (n < kTimingStages && stages[4 * n + 3] != 0) ++n;
  return n;
}

int64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
