// Expert parallelism: the row permutations on either side of the token exchange.
//
// "Halo's 2.8x over TRL is not a kernel, and its own benchmark proves it", Figure 3
// ("EP token routing") and section "Where the gap actually is": with the experts
// sharded over G ranks (the TorchTurbo README's expert-parallel plan shards the fused
// expert tensors Shard(0) over ep_size ranks), each rank sorts its tokens by expert,
// sends every row to the rank that owns its expert (a dispatch all-to-all), runs its
// own experts, and the rows travel back (a combine all-to-all) to be summed, weighted
// by the top-k probabilities, at their token.
//
// Rank g owns experts [g E_loc, (g+1) E_loc), E_loc = E / G. The sender's stable sort
// by expert already makes each destination's rows contiguous, in (local expert,
// token) order, so the rows a rank receives arrive source-major: [source s][local
// expert e][rows]. The grouped GEMMs want them expert-major in the segment-padded row
// space, so a received row of block (s, e) goes to
//   P_e + sum_{s' < s} recv_counts[s'][e] + (its index within the block),
// P_e the 128-row-aligned segment start of local expert e over all sources: within an
// expert the rows stay in source order, and within a source in the sender's token
// order. ep_regroup_kernel performs that copy (and zeroes the padding rows); the
// inverse gather ep_unregroup_kernel puts the expert outputs (or dXp) back in the
// received order for the return exchange. Both are row copies bound by HBM.
#include "route_common.cuh"

namespace moe {

constexpr int kEpVec = 4;  // 16-byte vectors each lane keeps in flight

// Tables of the received layout, built in shared memory by every block from the G x E_loc
// received counts (at most kMaxE entries: G * E_loc = E).
struct EpTables {
  int32_t roff[kMaxE + 1];  // first received row of block j = s * E_loc + e (source-major)
  int32_t base[kMaxE];      // first padded row of block j
  int32_t cnt[kMaxE];       // rows of local expert e over all sources
  int32_t pad[kMaxE + 1];   // segment start P_e, and P_{E_loc}
  int ok;                   // the counts are non-negative, add up to n_recv and fit R rows
};

__device__ void ep_build_tables(const int32_t *__restrict__ recv_counts, int G, int El,
                                int n_recv, int R, EpTables &tb) {
  if (threadIdx.x == 0) {
    const int n = G * El;
    bool ok = true;
    int64_t run = 0;  // 64-bit sums: a corrupt count cannot wrap around into a valid total
    for (int j = 0; j < n; ++j) {
      const int32_t c = recv_counts[j];
      ok = ok && c >= 0;
      tb.roff[j] = (int32_t)min(run, (int64_t)INT32_MAX);
      run += c;
    }
    ok = ok && run == n_recv;
    tb.roff[n] = (int32_t)min(run, (int64_t)INT32_MAX);
    int64_t p = 0;
    for (int e = 0; e < El && ok; ++e) {
      int64_t c = 0;
      for (int s = 0; s < G; ++s) {
        tb.base[s * El + e] = (int32_t)(p + c);
        c += recv_counts[s * El + e];
      }
      tb.cnt[e] = (int32_t)c;
      tb.pad[e] = (int32_t)p;
      p += (c + kTileRows - 1) / kTileRows * kTileRows;
      ok = ok && p <= R;
    }
    tb.pad[El] = (int32_t)min(p, (int64_t)INT32_MAX);
    tb.ok = ok;
  }
  __syncthreads();
}

// last block j < n with roff[j] <= i (blocks may be empty: roff is non-decreasing)
__device__ __forceinline__ int ep_block_of(const int32_t *roff, int n, int32_t i) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (roff[mid] <= i) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Blocks [0, row_blocks): one warp per received row i < n_recv: dest_of[i] = its padded
// row, xp[dest_of[i]] = xr[i]. Blocks [row_blocks, row_blocks + El kPadParts) zero the
// local experts' padding rows, kPadParts blocks per expert. Block 0 also writes counts_loc and padded_loc. When the
// received counts do not add up to n_recv, or their segments do not fit the R padded
// rows, nothing is written and status (if given) records kDevBadCounts.
__global__ void __launch_bounds__(256) ep_regroup_kernel(
    const int32_t *__restrict__ recv_counts, const uint4 *__restrict__ xr, uint4 *__restrict__ xp,
    int32_t *__restrict__ counts_loc, int32_t *__restrict__ padded_loc,
    int32_t *__restrict__ dest_of, int *status, int G, int El, int n_recv, int R, int nvec,
    int row_blocks) {
  __shared__ EpTables tb;
  ep_build_tables(recv_counts, G, El, n_recv, R, tb);
  const int n = G * El;
  if (!tb.ok) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && status) atomicExch(status, kDevBadCounts);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x < row_blocks) {
    if (blockIdx.x == 0) {
      for (int e = threadIdx.x; e < El; e += blockDim.x) counts_loc[e] = tb.cnt[e];
      for (int e = threadIdx.x; e <= El; e += blockDim.x) padded_loc[e] = tb.pad[e];
    }
    const int i = blockIdx.x * 8 + warp;
    if (i >= n_recv) return;
    const int j = ep_block_of(tb.roff, n, i);
    const int64_t dst = tb.base[j] + (i - tb.roff[j]);
    if (lane == 0) dest_of[i] = (int32_t)dst;
    const uint4 *src = xr + (int64_t)i * nvec;
    uint4 *out = xp + dst * nvec;
    for (int v0 = lane; v0 < nvec; v0 += 32 * kEpVec) {
      uint4 val[kEpVec];
#pragma unroll
      for (int u = 0; u < kEpVec; ++u)
        if (v0 + 32 * u < nvec) val[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kEpVec; ++u)
        if (v0 + 32 * u < nvec) out[v0 + 32 * u] = val[u];
    }
  } else {
    const int e = (blockIdx.x - row_blocks) / kPadParts;
    zero_pad_part(xp, tb.pad[e] + tb.cnt[e], tb.pad[e + 1], (blockIdx.x - row_blocks) % kPadParts,
                  nvec);
  }
}

// out[i] = o[dest_of[i]] for i < n_recv, one warp per row. A row index outside the R
// padded rows (a dest_of that no successful regroup wrote) is skipped, not followed.
__global__ void __launch_bounds__(256) ep_unregroup_kernel(const uint4 *__restrict__ o,
                                                           const int32_t *__restrict__ dest_of,
                                                           uint4 *__restrict__ out, int n_recv,
                                                           int R, int nvec) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + warp;
  if (i >= n_recv) return;
  const int32_t r = dest_of[i];
  if (r < 0 || r >= R) return;
  const uint4 *src = o + (int64_t)r * nvec;
  uint4 *dst = out + (int64_t)i * nvec;
  for (int v0 = lane; v0 < nvec; v0 += 32 * kEpVec) {
    uint4 val[kEpVec];
#pragma unroll
    for (int u = 0; u < kEpVec; ++u)
      if (v0 + 32 * u < nvec) val[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
    for (int u = 0; u < kEpVec; ++u)
      if (v0 + 32 * u < nvec) dst[v0 + 32 * u] = val[u];
  }
}

static inline int ep_cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

cudaError_t launch_ep_regroup(const int32_t *recv_counts, const void *xr, void *xp,
                              int32_t *counts_loc, int32_t *padded_loc, int32_t *dest_of,
                              int *status, int G, int El, int n_recv, int R, int d,
                              cudaStream_t st) {
  const int row_blocks = ep_cdiv(n_recv, 8) > 0 ? ep_cdiv(n_recv, 8) : 1;
  launch_begin(st);
  ep_regroup_kernel<<<row_blocks + El * kPadParts, 256, 0, st>>>(
      recv_counts, (const uint4 *)xr, (uint4 *)xp, counts_loc, padded_loc, dest_of, status, G,
      El, n_recv, R, d / 8, row_blocks);
  return note_launch("ep_regroup", st);
}

cudaError_t launch_ep_unregroup(const void *o, const int32_t *dest_of, void *out, int n_recv,
                                int R, int d, cudaStream_t st) {
  if (n_recv == 0) return cudaSuccess;
  launch_begin(st);
  ep_unregroup_kernel<<<ep_cdiv(n_recv, 8), 256, 0, st>>>((const uint4 *)o, dest_of,
                                                          (uint4 *)out, n_recv, R, d / 8);
  return note_launch("ep_unregroup", st);
}

}  // namespace moe
