// Bandwidth-bound stages of the MoE expert block: route, dispatch (histogram, scan,
// scatter), combine, and the two backward gathers.
//
// Route and combine follow Figure 3 ("EP token routing") of "Halo's 2.8x over TRL
// is not a kernel, and its own benchmark proves it": a per-token top-k router on
// fp32 logits, a grouped matmul over tokens sorted by expert, and rows returned to
// their token weighted by the top-k probabilities. Every output element here is
// written by one thread and every sum runs in a fixed order, so results are
// bit-reproducible without atomics ("The hard problems along the way" in "Halo:
// Frontier-Lab Training for Everyone" credits an atomic-free routing backward).
#include "route_common.cuh"

namespace moe {

constexpr int kVec = 4;           // 16-byte vectors each lane keeps in flight in the row copies

__device__ void scan_block(int32_t *__restrict__ hist, int C, int E, int32_t *__restrict__ counts,
                           int32_t *__restrict__ offsets, int32_t *__restrict__ padded,
                           int32_t *__restrict__ tile_expert, int32_t *__restrict__ pair_start,
                           int32_t *__restrict__ pair_expert, const float *__restrict__ prob_part,
                           float *__restrict__ aux, int T, int k);

// Block c routes tokens [32c, 32c+32), one warp per token, and, when COUNT, also
// writes the chunk histogram and local ranks for the dispatch. With prob_part it also
// writes prob_part[e][c], the sum over the chunk's tokens (in token order) of the
// softmax of all E logits, for the load-balancing statistics.
// With SCAN (and COUNT), the block that finishes last also runs the scan of the chunk
// counts (scan_block): each block publishes its counts with a fence before taking a
// ticket from *done, so the block with the last ticket sees every block's counts; it
// resets *done for the next launch. No block waits for another.
template <bool COUNT, int Q, bool SCAN>
__global__ void __launch_bounds__(1024) route_kernel(const float *__restrict__ logits,
                                                     const float *__restrict__ bias,
                                                     int32_t *__restrict__ ids,
                                                     float *__restrict__ w,
                                                     int32_t *__restrict__ rank,
                                                     int32_t *__restrict__ hist,
                                                     float *__restrict__ prob_part, int T, int E,
                                                     int k, int C, ScanOut so) {
  __shared__ int32_t s_ids[kChunk][kMaxK];
  __shared__ float s_prob[kChunk][kMaxE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  for (int i = warp; i < kChunk; i += 32) {
    const int t = c * kChunk + i;
    if (t >= T) {
      if (prob_part)
        for (int e = lane; e < E; e += 32) s_prob[i][e] = 0.f;
      break;
    }
    int sid[1];
    float sw[1], pr[1][Q];
    route_tokens<Q, 1, false>(logits + (int64_t)t * E, E, bias, E, k, lane, sid, sw,
                              prob_part != nullptr, pr);
    if (lane < k) {
      ids[(int64_t)t * k + lane] = sid[0];
      w[(int64_t)t * k + lane] = sw[0];
      s_ids[i][lane] = sid[0];
    }
    if (prob_part) {
#pragma unroll
      for (int q = 0; q < Q; ++q)
        if (lane + 32 * q < E) s_prob[i][lane + 32 * q] = pr[0][q];
    }
  }
  if (COUNT || prob_part) __syncthreads();
  if (prob_part) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      float acc = 0.f;
      for (int i = 0; i < kChunk; ++i) acc += s_prob[i][e];
      prob_part[(int64_t)e * C + c] = acc;
    }
  }
  if constexpr (COUNT) count_chunk(s_ids, c, T, E, k, C, warp, 32, lane, rank, hist);
  if constexpr (COUNT && SCAN) {
    __shared__ int s_last;
    __threadfence();  // this thread's hist and prob_part stores, device-wide
    __syncthreads();  // every thread of the block has stored
    if (threadIdx.x == 0) {
      __threadfence();  // cumulative: the block's stores before its ticket
      s_last = atomicAdd(so.done, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();  // the other blocks' stores before this block's reads
      scan_block(hist, C, E, so.counts, so.offsets, so.padded, so.tile_expert, so.pair_start,
                 so.pair_expert, prob_part, so.aux, T, k);
      if (threadIdx.x == 0) *so.done = 0;
    }
  }
}

// Histogram and local ranks from ids already in memory (standalone dispatch).
__global__ void __launch_bounds__(256) count_kernel(const int32_t *__restrict__ ids,
                                                    int32_t *__restrict__ rank,
                                                    int32_t *__restrict__ hist, int T, int E,
                                                    int k, int C) {
  __shared__ int32_t s_ids[kChunk][kMaxK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  for (int i = threadIdx.x; i < kChunk * k; i += blockDim.x) {
    const int t = c * kChunk + i / k;
    s_ids[i / k][i % k] = (t < T) ? ids[(int64_t)t * k + i % k] : -1;
  }
  __syncthreads();
  count_chunk(s_ids, c, T, E, k, C, warp, 8, lane, rank, hist);
}

// --------------------------------------------------------------------------- scan
// One block. Warp w scans the chunk counts of experts w, w+32, ... in chunk order,
// turning hist[e][c] into the exclusive prefix within expert e; then the per-expert
// totals give counts, compact offsets, padded offsets (segments rounded up to whole
// 128-row tiles), the expert of every 128-row tile and, for the GEMMs that run on
// pairs of SMs, the pairs of consecutive tiles of one expert: pair_start[e] is the
// first pair of expert e (ceil(tiles_e / 2) pairs each) and pair_expert[p] the
// expert of pair p. The pair tables are skipped when their pointers are null.
__device__ int last_le(const int32_t *v, int n, int x) {  // last i < n with v[i] <= x
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (v[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ void plan_from_counts(const int32_t *s_cnt, int E, int32_t *__restrict__ offsets,
                                 int32_t *__restrict__ padded, int32_t *__restrict__ tile_expert,
                                 int32_t *__restrict__ pair_start,
                                 int32_t *__restrict__ pair_expert, int32_t *s_pad,
                                 int32_t *s_pair) {
  if (threadIdx.x < 32) {
    // warp 0: lane l takes experts [l kPer, (l+1) kPer); exclusive prefixes over the
    // lanes by shuffles, then each lane walks its experts in order
    constexpr int kPer = kMaxE / 32;
    const int lane = threadIdx.x;
    int32_t n_rows = 0, n_tiles = 0, n_pairs = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane * kPer + i;
      if (e < E) {
        const int tiles = (s_cnt[e] + kTileRows - 1) / kTileRows;
        n_rows += s_cnt[e];
        n_tiles += tiles;
        n_pairs += (tiles + 1) / 2;
      }
    }
    int32_t rows = n_rows, tiles_in = n_tiles, pairs_in = n_pairs;  // inclusive over lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t a = __shfl_up_sync(0xffffffffu, rows, o);
      const int32_t b = __shfl_up_sync(0xffffffffu, tiles_in, o);
      const int32_t c = __shfl_up_sync(0xffffffffu, pairs_in, o);
      if (lane >= o) {
        rows += a;
        tiles_in += b;
        pairs_in += c;
      }
    }
    int32_t off = rows - n_rows, til = tiles_in - n_tiles, pairs = pairs_in - n_pairs;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane * kPer + i;
      if (e < E) {
        offsets[e] = off;
        padded[e] = til * kTileRows;
        s_pad[e] = til * kTileRows;
        s_pair[e] = pairs;
        const int tiles = (s_cnt[e] + kTileRows - 1) / kTileRows;
        off += s_cnt[e];
        til += tiles;
        pairs += (tiles + 1) / 2;
      }
    }
    if (lane == 31) {
      offsets[E] = rows;
      padded[E] = tiles_in * kTileRows;
      s_pad[E] = tiles_in * kTileRows;
      s_pair[E] = pairs_in;
    }
  }
  __syncthreads();
  const int ntiles = s_pad[E] / kTileRows;
  for (int mt = threadIdx.x; mt < ntiles; mt += blockDim.x)
    tile_expert[mt] = last_le(s_pad, E, mt * kTileRows);
  if (pair_start) {
    for (int e = threadIdx.x; e <= E; e += blockDim.x) pair_start[e] = s_pair[e];
    for (int p = threadIdx.x; p < s_pair[E]; p += blockDim.x)
      pair_expert[p] = last_le(s_pair, E, p);
  }
}

// With prob_part, also the load-balancing statistics: aux[e] = f_e = counts_e / (T k),
// aux[E + e] = P_e = (sum over chunks, in chunk order, of prob_part[e][c]) / T and
// aux[2E] = E * sum_e f_e P_e (summed in expert order).
// The scan of one block of 1024 threads (the scan kernel's, or the fused route kernel's
// last block's). hist and prob_part are read through L2 (.cg): in the fused kernel other
// blocks wrote them during the same launch.
__device__ void scan_block(int32_t *__restrict__ hist, int C, int E, int32_t *__restrict__ counts,
                           int32_t *__restrict__ offsets, int32_t *__restrict__ padded,
                           int32_t *__restrict__ tile_expert, int32_t *__restrict__ pair_start,
                           int32_t *__restrict__ pair_expert, const float *__restrict__ prob_part,
                           float *__restrict__ aux, int T, int k) {
  __shared__ int32_t s_cnt[kMaxE];
  __shared__ float s_p[kMaxE];
  __shared__ int32_t s_pad[kMaxE + 1];
  __shared__ int32_t s_pair[kMaxE + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The warp's work items are (expert, group of 128 chunks) in order: experts warp,
  // warp + 32, ..., each group by group. Lane l takes the group's chunks 4l .. 4l+3: a
  // running sum over its four, one warp scan of the lane totals, then the four exclusive
  // prefixes (one 5-step shuffle scan per 128 chunks; a scan per 32-chunk slice took ~4x
  // the instructions). The next item's chunks are loaded before the current one is
  // scanned, so a load's latency overlaps the previous scan.
  constexpr int kPer = 4, kGroup = 32 * kPer;
  // (one empty group when C = 0, so that every expert's count is still written)
  const int ngroups = max(1, (C + kGroup - 1) / kGroup);
  const int items = (warp < E ? (E - warp + 31) / 32 : 0) * ngroups;
  int32_t v[kPer], vn[kPer];
  auto load = [&](int it, int32_t(&dst)[kPer]) {
    const int e = warp + 32 * (it / ngroups), c0 = (it % ngroups) * kGroup + kPer * lane;
    const int32_t *h = hist + (int64_t)e * C;
#pragma unroll
    for (int u = 0; u < kPer; ++u) dst[u] = (c0 + u < C) ? __ldcg(h + c0 + u) : 0;
  };
  if (items > 0) load(0, v);
  int32_t running = 0;
  for (int it = 0; it < items; ++it) {
    if (it + 1 < items) load(it + 1, vn);
    const int e = warp + 32 * (it / ngroups), g0 = (it % ngroups) * kGroup;
    const int c0 = g0 + kPer * lane;
    int32_t *h = hist + (int64_t)e * C;
    int32_t p[kPer];  // inclusive sums within the lane's four chunks
    p[0] = v[0];
#pragma unroll
    for (int u = 1; u < kPer; ++u) p[u] = p[u - 1] + v[u];
    int32_t incl = p[kPer - 1];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const int32_t base = running + incl - p[kPer - 1];
#pragma unroll
    for (int u = 0; u < kPer; ++u)
      if (c0 + u < C) h[c0 + u] = base + p[u] - v[u];
    running += __shfl_sync(0xffffffffu, incl, 31);
    if (g0 + kGroup >= C) {  // the expert's last group
      if (lane == 0) {
        s_cnt[e] = running;
        counts[e] = running;
      }
      running = 0;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) v[u] = vn[u];
  }
  if (prob_part) {
    for (int e = warp; e < E; e += 32) {
      float acc = 0.f;  // lane-strided chunks, then a fixed butterfly: a fixed order
      for (int c = lane; c < C; c += 32) acc += __ldcg(prob_part + (int64_t)e * C + c);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) s_p[e] = acc / (float)T;
    }
  }
  __syncthreads();
  if (prob_part && threadIdx.x == 0) {
    float l = 0.f;
    for (int e = 0; e < E; ++e) {
      const float f = (float)s_cnt[e] / ((float)T * (float)k);
      aux[e] = f;
      aux[E + e] = s_p[e];
      l += f * s_p[e];
    }
    aux[2 * E] = (float)E * l;
  }
  plan_from_counts(s_cnt, E, offsets, padded, tile_expert, pair_start, pair_expert, s_pad, s_pair);
}

__global__ void __launch_bounds__(1024) scan_kernel(int32_t *__restrict__ hist, int C, int E,
                                                    int32_t *__restrict__ counts,
                                                    int32_t *__restrict__ offsets,
                                                    int32_t *__restrict__ padded,
                                                    int32_t *__restrict__ tile_expert,
                                                    int32_t *__restrict__ pair_start,
                                                    int32_t *__restrict__ pair_expert,
                                                    const float *__restrict__ prob_part,
                                                    float *__restrict__ aux, int T, int k) {
  scan_block(hist, C, E, counts, offsets, padded, tile_expert, pair_start, pair_expert, prob_part,
             aux, T, k);
}

// The same plan from counts alone (standalone expert FFN calls).
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t *__restrict__ counts, int E,
                                                    int32_t *__restrict__ offsets,
                                                    int32_t *__restrict__ padded,
                                                    int32_t *__restrict__ tile_expert,
                                                    int32_t *__restrict__ pair_start,
                                                    int32_t *__restrict__ pair_expert) {
  __shared__ int32_t s_cnt[kMaxE];
  __shared__ int32_t s_pad[kMaxE + 1];
  __shared__ int32_t s_pair[kMaxE + 1];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = counts[e];
  __syncthreads();
  plan_from_counts(s_cnt, E, offsets, padded, tile_expert, pair_start, pair_expert, s_pad, s_pair);
}

// ------------------------------------------------------------------------- scatter
// Blocks [0, token_blocks): one warp per token; lane j < k computes the padded row of
// slot j (segment start + chunk base + local rank), then the warp copies x[t] to each
// of its k rows in 16-byte vectors (read once, written k times).
// Blocks [token_blocks, token_blocks + E kPadParts): expert e's padding rows are zeroed
// (and marked tok_of = -1) by kPadParts blocks. The last block marks the rows past the
// last segment (up to R) with tok_of = -1.
__global__ void __launch_bounds__(256) scatter_kernel(
    const uint4 *__restrict__ x, const int32_t *__restrict__ ids,
    const int32_t *__restrict__ rank, const int32_t *__restrict__ hist,
    const int32_t *__restrict__ padded, const int32_t *__restrict__ counts,
    int32_t *__restrict__ row_of, int32_t *__restrict__ tok_of, uint4 *__restrict__ xp, int T,
    int nvec, int E, int k, int C, int token_blocks, int R) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x < token_blocks) {
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    int row = 0;
    if (lane < k) {
      const int e = ids[(int64_t)t * k + lane];
      row = padded[e] + hist[(int64_t)e * C + t / kChunk] + rank[(int64_t)t * k + lane];
      row_of[(int64_t)t * k + lane] = row;
      tok_of[row] = t;
    }
    int rows[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) rows[j] = __shfl_sync(0xffffffffu, row, j);
    // kVec 16-byte loads in flight per lane, then their k stores each
    const uint4 *src = x + (int64_t)t * nvec;
    for (int v0 = lane; v0 < nvec; v0 += 32 * kVec) {
      uint4 val[kVec];
#pragma unroll
      for (int u = 0; u < kVec; ++u)
        if (v0 + 32 * u < nvec) val[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          uint4 *dst = xp + (int64_t)rows[j] * nvec;
#pragma unroll
          for (int u = 0; u < kVec; ++u)
            if (v0 + 32 * u < nvec) dst[v0 + 32 * u] = val[u];
        }
      }
    }
  } else if ((int)blockIdx.x < token_blocks + E * kPadParts) {
    const int e = (blockIdx.x - token_blocks) / kPadParts;
    const int part = (blockIdx.x - token_blocks) % kPadParts;
    const int r0 = padded[e] + counts[e], r1 = padded[e + 1];
    zero_pad_part(xp, r0, r1, part, nvec);
    const int a = (int)pad_part_begin(r0, r1, part), b = (int)pad_part_end(r0, r1, part);
    for (int r = a + threadIdx.x; r < b; r += blockDim.x) tok_of[r] = -1;
  } else {
    // rows past the last segment belong to no expert
    for (int r = padded[E] + threadIdx.x; r < R; r += blockDim.x) tok_of[r] = -1;
  }
}

// ------------------------------------------------------------------------- combine
// WPT warps per token, each on every WPT-th 32-vector slice of the row:
// y[t] = sum_j w[t][j] * o[row_of[t][j]], fp32 FMA in slot order, one bf16 rounding.
// With unit weights it is the backward's dX gather-sum. Several warps per row shorten
// each warp's chain of dependent row loads (the kernel is latency-bound below ~1 GB).
// KT > 0 (k <= KT): the k row loads of a vector are all issued before the sum uses
// them (measured on GB300: 15-23% faster than loading inside the sum at k = 4);
// KT = 0: any k <= 16, each load consumed as it arrives.
template <bool WEIGHTED, int WPT, int KT>
__global__ void __launch_bounds__(256) gather_sum_kernel(const uint4 *__restrict__ o,
                                                         const float *__restrict__ w,
                                                         const int32_t *__restrict__ row_of,
                                                         uint4 *__restrict__ y, int T, int nvec,
                                                         int k) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (8 / WPT) + warp / WPT;
  const int seg = warp % WPT;
  if (t >= T) return;
  int row = 0;
  float wt = 1.f;
  if (lane < k) {
    row = row_of[(int64_t)t * k + lane];
    if (WEIGHTED) wt = w[(int64_t)t * k + lane];
  }
  int rows[kMaxK];
  float wts[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    rows[j] = __shfl_sync(0xffffffffu, row, j);
    wts[j] = __shfl_sync(0xffffffffu, wt, j);
  }
  for (int v = seg * 32 + lane; v < nvec; v += 32 * WPT) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    if (KT > 0) {
      uint4 raw[KT > 0 ? KT : 1];
#pragma unroll
      for (int j = 0; j < KT; ++j)
        if (j < k) raw[j] = __ldg(o + (int64_t)rows[j] * nvec + v);
#pragma unroll
      for (int j = 0; j < KT; ++j) {
        if (j < k) {
          float f[8];
          unpack8(raw[j], f);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            acc[i] = WEIGHTED ? fmaf(wts[j], f[i], acc[i]) : acc[i] + f[i];
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          float f[8];
          unpack8(__ldg(o + (int64_t)rows[j] * nvec + v), f);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            acc[i] = WEIGHTED ? fmaf(wts[j], f[i], acc[i]) : acc[i] + f[i];
        }
      }
    }
    y[(int64_t)t * nvec + v] = pack8(acc);
  }
}

// ------------------------------------------------------------------ backward scatter
// G[row_of[t][j]] = bf16(w[t][j] * dY[t]) (one warp per token); the extra E kPadParts
// blocks zero the experts' padding rows of G so the GEMMs read zeros there.
//
// With dlogits, the same pass also forms the router-logit gradient of the token
// ("The hard problems along the way" in "Halo: Frontier-Lab Training for Everyone":
// a routing backward without atomics): dw_j = <dY[t], O[row_of[t][j]]> in fp32 (each
// lane's partial sums, then a fixed-order warp reduction), then
// dlogits[t][ids[t][j]] = w_j (dw_j - sum_i w_i dw_i) and 0 for the other experts. The
// whole row of each token is written by its warp.
//
// KT bounds k (4, 8 or 16: the per-slot arrays are sized by it) and ROUTER says whether
// the router-logit gradient is formed, so the plain G scatter carries no register for it
// (the kernel is latency-bound at a few thousand tokens, where occupancy decides).
template <bool ROUTER, int KT>
__global__ void __launch_bounds__(256) scale_scatter_kernel(
    const uint4 *__restrict__ dy, const float *__restrict__ w, const int32_t *__restrict__ row_of,
    const int32_t *__restrict__ padded, const int32_t *__restrict__ counts,
    uint4 *__restrict__ g, int T, int nvec, int E, int k, int token_blocks,
    const uint4 *__restrict__ o, const int32_t *__restrict__ ids, float *__restrict__ dlogits) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((int)blockIdx.x < token_blocks) {
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    int row = 0;
    float wt = 0.f;
    if (lane < k) {
      row = row_of[(int64_t)t * k + lane];
      wt = w[(int64_t)t * k + lane];
    }
    int rows[KT];
    float wts[KT], dot[ROUTER ? KT : 1];
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      rows[j] = __shfl_sync(0xffffffffu, row, j);
      wts[j] = __shfl_sync(0xffffffffu, wt, j);
      if (ROUTER) dot[j] = 0.f;
    }
    const uint4 *src = dy + (int64_t)t * nvec;
    for (int v0 = lane; v0 < nvec; v0 += 32 * kVec) {
      uint4 val[kVec];
#pragma unroll
      for (int u = 0; u < kVec; ++u)
        if (v0 + 32 * u < nvec) val[u] = __ldg(src + v0 + 32 * u);
      if (ROUTER) {
        // the dot products first: kVec output-row loads in flight per slot
#pragma unroll
        for (int j = 0; j < KT; ++j) {
          if (j < k) {
            const uint4 *orow = o + (int64_t)rows[j] * nvec;
            uint4 ov[kVec];
#pragma unroll
            for (int u = 0; u < kVec; ++u)
              if (v0 + 32 * u < nvec) ov[u] = __ldg(orow + v0 + 32 * u);
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
              if (v0 + 32 * u < nvec) {
                float f[8], of[8];
                unpack8(val[u], f);
                unpack8(ov[u], of);
#pragma unroll
                for (int i = 0; i < 8; ++i) dot[j] = fmaf(f[i], of[i], dot[j]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < KT; ++j) {
        if (j < k) {
          uint4 *dst = g + (int64_t)rows[j] * nvec;
#pragma unroll
          for (int u = 0; u < kVec; ++u) {
            if (v0 + 32 * u < nvec) {
              float f[8], sc[8];
              unpack8(val[u], f);
#pragma unroll
              for (int i = 0; i < 8; ++i) sc[i] = wts[j] * f[i];
              dst[v0 + 32 * u] = pack8(sc);
            }
          }
        }
      }
    }
    if (ROUTER) {
      float s = 0.f;
      int eid[KT];
      const int my_id = (lane < k) ? ids[(int64_t)t * k + lane] : -1;
#pragma unroll
      for (int j = 0; j < KT; ++j) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot[j] += __shfl_xor_sync(0xffffffffu, dot[j], off);
        eid[j] = __shfl_sync(0xffffffffu, my_id, j);
        if (j < k) s = fmaf(wts[j], dot[j], s);
      }
      float *out = dlogits + (int64_t)t * E;
      for (int e = lane; e < E; e += 32) {
        float val = 0.f;
#pragma unroll
        for (int j = 0; j < KT; ++j)
          if (j < k && eid[j] == e) val = wts[j] * (dot[j] - s);
        out[e] = val;
      }
    }
  } else {
    const int e = (blockIdx.x - token_blocks) / kPadParts;
    zero_pad_part(g, padded[e] + counts[e], padded[e + 1], (blockIdx.x - token_blocks) % kPadParts,
                  nvec);
  }
}

// ---------------------------------------------------------- load-balancing gradient
// dlogits[t][e] += coeff * (E / T) * p[t][e] * (f_e - sum_e' f_e' p[t][e']), the
// gradient of coeff * aux with the assignment fractions f held fixed (they count
// discrete choices); p is the softmax over all E logits of token t. One warp per
// token, each element read and written by one lane.
__global__ void __launch_bounds__(256) aux_grad_kernel(const float *__restrict__ logits,
                                                       const int32_t *__restrict__ counts,
                                                       float coeff, float *__restrict__ dlogits,
                                                       int T, int E, int k) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float *row = logits + (int64_t)t * E;
  float v[8], f[8];
  float mx = -INFINITY;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int e = lane + 32 * q;
    v[q] = (e < E) ? __ldg(row + e) : -INFINITY;
    f[q] = (e < E) ? (float)__ldg(counts + e) / ((float)T * (float)k) : 0.f;
    mx = fmaxf(mx, v[q]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float sum = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    v[q] = (lane + 32 * q < E) ? expf(v[q] - mx) : 0.f;
    sum += v[q];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  float fp = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    v[q] /= sum;
    fp += f[q] * v[q];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) fp += __shfl_xor_sync(0xffffffffu, fp, off);
  const float scale = coeff * (float)E / (float)T;
  float *out = dlogits + (int64_t)t * E;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int e = lane + 32 * q;
    if (e < E) out[e] += scale * v[q] * (f[q] - fp);
  }
}

// ------------------------------------------------------------------------ launchers
static inline int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

cudaError_t launch_route(const float *logits, const float *bias, int32_t *ids, float *w,
                         int32_t *rank, int32_t *hist, float *prob_part, int T, int E, int k,
                         bool with_count, cudaStream_t st) {
  const int C = ceil_div(T, kChunk);
  if (C == 0) return cudaSuccess;
  // Q = logits per lane: the smallest of 1, 2, 4, 8 with E <= 32 Q
#define MOE_ROUTE(Q)                                                                        \
  do {                                                                                     \
    launch_begin(st);                                                                      \
    if (with_count)                                                                        \
      route_kernel<true, Q, false><<<C, 1024, 0, st>>>(logits, bias, ids, w, rank, hist,   \
                                                       prob_part, T, E, k, C, ScanOut{});  \
    else                                                                                   \
      route_kernel<false, Q, false><<<C, 1024, 0, st>>>(logits, bias, ids, w, rank, hist,  \
                                                        prob_part, T, E, k, C, ScanOut{}); \
    return note_launch(with_count ? "route_count" : "route", st);                         \
  } while (0)
  if (E <= 32) MOE_ROUTE(1);
  if (E <= 64) MOE_ROUTE(2);
  if (E <= 128) MOE_ROUTE(4);
  MOE_ROUTE(8);
#undef MOE_ROUTE
}

cudaError_t launch_route_count_scan(const float *logits, const float *bias, int32_t *ids,
                                   float *w, int32_t *rank, int32_t *hist, float *prob_part,
                                   int T, int E, int k, const ScanOut &so, cudaStream_t st) {
  const int C = ceil_div(T, kChunk);
  if (C == 0)  // no token: the scan alone writes the empty plan
    return launch_scan(hist, T, E, k, so.counts, so.offsets, so.padded, so.tile_expert,
                       so.pair_start, so.pair_expert, prob_part, so.aux, st);
#define MOE_ROUTE_SCAN(Q)                                                                   \
  do {                                                                                     \
    launch_begin(st);                                                                      \
    route_kernel<true, Q, true><<<C, 1024, 0, st>>>(logits, bias, ids, w, rank, hist,      \
                                                    prob_part, T, E, k, C, so);            \
    return note_launch("route_count_scan", st);                                           \
  } while (0)
  if (E <= 32) MOE_ROUTE_SCAN(1);
  if (E <= 64) MOE_ROUTE_SCAN(2);
  if (E <= 128) MOE_ROUTE_SCAN(4);
  MOE_ROUTE_SCAN(8);
#undef MOE_ROUTE_SCAN
}

cudaError_t launch_aux_grad(const float *logits, const int32_t *counts, float coeff,
                            float *dlogits, int T, int E, int k, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  launch_begin(st);
  aux_grad_kernel<<<ceil_div(T, 8), 256, 0, st>>>(logits, counts, coeff, dlogits, T, E, k);
  return note_launch("aux_grad", st);
}

cudaError_t launch_count(const int32_t *ids, int32_t *rank, int32_t *hist, int T, int E, int k,
                         cudaStream_t st) {
  const int C = ceil_div(T, kChunk);
  if (C == 0) return cudaSuccess;
  launch_begin(st);
  count_kernel<<<C, 256, 0, st>>>(ids, rank, hist, T, E, k, C);
  return note_launch("count", st);
}

cudaError_t launch_scan(int32_t *hist, int T, int E, int k, int32_t *counts, int32_t *offsets,
                        int32_t *padded, int32_t *tile_expert, int32_t *pair_start,
                        int32_t *pair_expert, const float *prob_part, float *aux,
                        cudaStream_t st) {
  const int C = ceil_div(T, kChunk);
  launch_begin(st);
  scan_kernel<<<1, 1024, 0, st>>>(hist, C, E, counts, offsets, padded, tile_expert, pair_start,
                                  pair_expert, T > 0 ? prob_part : nullptr, aux, T, k);
  return note_launch("scan", st);
}

cudaError_t launch_plan(const int32_t *counts, int E, int32_t *offsets, int32_t *padded,
                        int32_t *tile_expert, int32_t *pair_start, int32_t *pair_expert,
                        cudaStream_t st) {
  launch_begin(st);
  plan_kernel<<<1, 1024, 0, st>>>(counts, E, offsets, padded, tile_expert, pair_start,
                                  pair_expert);
  return note_launch("plan", st);
}

cudaError_t launch_scatter(const void *x, const int32_t *ids, const int32_t *rank,
                           const int32_t *hist, const int32_t *padded, const int32_t *counts,
                           int32_t *row_of, int32_t *tok_of, void *xp, int T, int d, int E, int k,
                           int R, cudaStream_t st) {
  const int C = ceil_div(T, kChunk);
  const int token_blocks = ceil_div(T, 8);
  launch_begin(st);
  scatter_kernel<<<token_blocks + E * kPadParts + 1, 256, 0, st>>>(
      (const uint4 *)x, ids, rank, hist, padded, counts, row_of, tok_of, (uint4 *)xp, T, d / 8,
      E, k, C, token_blocks, R);
  return note_launch("scatter", st);
}

// warps per token of the gather kernels: more for longer rows (at least 64 vectors each)
template <bool WEIGHTED, int KT>
static void launch_gather_kt(const void *o, const float *w, const int32_t *row_of, void *y,
                             int T, int nvec, int k, cudaStream_t st) {
  if (nvec >= 256)
    gather_sum_kernel<WEIGHTED, 4, KT><<<ceil_div(T, 2), 256, 0, st>>>(
        (const uint4 *)o, w, row_of, (uint4 *)y, T, nvec, k);
  else if (nvec >= 128)
    gather_sum_kernel<WEIGHTED, 2, KT><<<ceil_div(T, 4), 256, 0, st>>>(
        (const uint4 *)o, w, row_of, (uint4 *)y, T, nvec, k);
  else
    gather_sum_kernel<WEIGHTED, 1, KT><<<ceil_div(T, 8), 256, 0, st>>>(
        (const uint4 *)o, w, row_of, (uint4 *)y, T, nvec, k);
}

template <bool WEIGHTED>
static void launch_gather(const void *o, const float *w, const int32_t *row_of, void *y, int T,
                          int nvec, int k, cudaStream_t st) {
  if (k <= 4) launch_gather_kt<WEIGHTED, 4>(o, w, row_of, y, T, nvec, k, st);
  else if (k <= 8) launch_gather_kt<WEIGHTED, 8>(o, w, row_of, y, T, nvec, k, st);
  else launch_gather_kt<WEIGHTED, 0>(o, w, row_of, y, T, nvec, k, st);
}

cudaError_t launch_combine(const void *o, const float *w, const int32_t *row_of, void *y, int T,
                           int d, int k, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  launch_begin(st);
  launch_gather<true>(o, w, row_of, y, T, d / 8, k, st);
  return note_launch("combine", st);
}

cudaError_t launch_gather_sum(const void *dxp, const int32_t *row_of, void *dx, int T, int d,
                              int k, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  launch_begin(st);
  launch_gather<false>(dxp, nullptr, row_of, dx, T, d / 8, k, st);
  return note_launch("dx_gather", st);
}

cudaError_t launch_scale_scatter(const void *dy, const float *w, const int32_t *row_of,
                                 const int32_t *padded, const int32_t *counts, void *g, int T,
                                 int d, int E, int k, const void *o, const int32_t *ids,
                                 float *dlogits, cudaStream_t st) {
  const int token_blocks = ceil_div(T, 8);
  launch_begin(st);
#define MOE_SCALE_SCATTER(R, KT)                                                             \
  scale_scatter_kernel<R, KT><<<token_blocks + E * kPadParts, 256, 0, st>>>(                \
      (const uint4 *)dy, w, row_of, padded, counts, (uint4 *)g, T, d / 8, E, k, token_blocks, \
      (const uint4 *)o, ids, dlogits)
  if (dlogits) {
    if (k <= 4) MOE_SCALE_SCATTER(true, 4);
    else if (k <= 8) MOE_SCALE_SCATTER(true, 8);
    else MOE_SCALE_SCATTER(true, 16);
  } else {
    if (k <= 4) MOE_SCALE_SCATTER(false, 4);
    else if (k <= 8) MOE_SCALE_SCATTER(false, 8);
    else MOE_SCALE_SCATTER(false, 16);
  }
#undef MOE_SCALE_SCATTER
  return note_launch(dlogits ? "g_scatter_router_grad" : "g_scatter", st);
}

}  // namespace moe
