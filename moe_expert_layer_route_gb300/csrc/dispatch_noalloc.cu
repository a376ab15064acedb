// moe_dispatch_noalloc: moe_dispatch for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory for a workspace: code running
// under a runtime that owns every allocation (a fixed memory pool handed out by
// someone else, a plugin inside a host framework with no allocator hook), or code
// that must not call cudaMalloc at all at that point. For them this entry point
// takes only the dispatch's own inputs and outputs; its scratch (per-assignment
// local ranks, per-chunk expert histograms, the tile-to-expert table) lives in
// the file-scope device array below instead of a caller workspace.
//
// The array is part of the library's device image, so every GPU that loads the
// library holds its 4 MiB until the process exits. All calls share it: calls
// that overlap on the GPU (two streams, two host threads) race on it, so the
// caller must order them. Each call writes every scratch entry it later reads
// (the histogram of every (expert, chunk), the rank of every assignment, the
// expert of every tile), so nothing needs clearing between calls even though the
// array keeps the previous call's contents.
#include <mutex>

#include "../../include/moe_gb300.h"
#include "kernels.h"

namespace {

// Capacity of the shared scratch, in int32 entries (4 MiB).
constexpr int64_t kScratchInts = int64_t(1) << 20;

static __device__ __align__(256) int32_t g_dispatch_scratch[kScratchInts];

std::mutex g_setup_mu;
int32_t *g_scratch_addr[64] = {};  // device address of g_dispatch_scratch, per device

// Set-up, once per device, with that device current: the host-side name of a
// __device__ array is only a stand-in, the kernels need its device address. The
// address is cached for the life of the process, so the library must not be used on
// a device across a cudaDeviceReset (the cached address would then be stale).
moe_status scratch_address(int32_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<int32_t *>(p);
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

inline int64_t round64(int64_t n) { return (n + 63) / 64 * 64; }  // 256-byte steps

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" moe_status moe_dispatch_noalloc(moe_shape s, const moe_bf16 *x, const int32_t *ids,
                                           moe_bf16 *xp, int32_t *counts, int32_t *offsets,
                                           int32_t *padded_offsets, int32_t *row_of,
                                           int32_t *tok_of, moe_stream stream) {
  // the same shape rules and device check as every other entry point
  const moe_status shape_ok = moe::check_shape(s);
  if (shape_ok != MOE_OK) return shape_ok;
  const void *always[] = {xp, counts, offsets, padded_offsets, tok_of};
  for (const void *p : always) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_ALIGNMENT;
  }
  if (s.T > 0) {
    const void *tokens[] = {x, ids, row_of};
    for (const void *p : tokens) {
      if (!p) return MOE_ERR_INVALID_ARG;
      if (!aligned16(p)) return MOE_ERR_ALIGNMENT;
    }
  }
  const int64_t A = s.T * s.k;
  const int64_t C = (s.T + 31) / 32 > 0 ? (s.T + 31) / 32 : 1;
  const int64_t R = moe_padded_rows(s);
  const int64_t rank_at = 0;
  const int64_t hist_at = rank_at + round64(A);
  const int64_t tiles_at = hist_at + round64(s.E * C);
  const int64_t need = tiles_at + round64(R / moe::kTileRows);
  if (need > kScratchInts) return MOE_ERR_WORKSPACE;  // beyond the fixed 4 MiB scratch
  const moe_status dev_ok = moe::check_device();
  if (dev_ok != MOE_OK) return dev_ok;

  int32_t *scratch = nullptr;
  const moe_status st0 = scratch_address(&scratch);
  if (st0 != MOE_OK) return st0;
  int32_t *rank = scratch + rank_at, *hist = scratch + hist_at, *tiles = scratch + tiles_at;

  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = (int)s.T, E = (int)s.E, k = (int)s.k, d = (int)s.d;
  if (moe::launch_count(ids, rank, hist, T, E, k, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (moe::launch_scan(hist, T, E, k, counts, offsets, padded_offsets, tiles, nullptr, nullptr,
                       nullptr, nullptr, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_scatter(x, ids, rank, hist, padded_offsets, counts, row_of, tok_of, xp, T, d, E,
                          k, (int)R, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
