// Per-token top-k routing and per-chunk counting shared by the route kernels
// (logits from memory in route_dispatch.cu, logits from the router GEMM in
// router.cu).
#pragma once

#include "kernels.h"

namespace moe {

constexpr int kChunk = 32;        // tokens per histogram chunk (one per lane of a warp)
constexpr int kMaxK = 16;
constexpr int kMaxE = 256;

// ----------------------------------------------------------------- padding rows
// An expert segment's padding rows [r0, r1) (fewer than kTileRows of them) are zeroed by
// kPadParts blocks of 256 threads, part p taking rows [r0 + p kPadRows, r0 + (p+1) kPadRows)
// and the last part also whatever lies beyond. One block per segment left the SMs that
// held those blocks with up to 0.7 MB of stores each (d = 2880) against ~0.2 MB for a
// block of row copies.
constexpr int kPadRows = 32;
constexpr int kPadParts = kTileRows / kPadRows;
static_assert(kPadParts * kPadRows == kTileRows, "padding parts must cover a tile");

__device__ __forceinline__ int64_t pad_part_begin(int64_t r0, int64_t r1, int part) {
  return min(r1, r0 + (int64_t)part * kPadRows);
}
__device__ __forceinline__ int64_t pad_part_end(int64_t r0, int64_t r1, int part) {
  return part == kPadParts - 1 ? r1 : min(r1, r0 + (int64_t)(part + 1) * kPadRows);
}

__device__ __forceinline__ void zero_pad_part(uint4 *__restrict__ base, int64_t r0, int64_t r1,
                                              int part, int nvec) {
  const int64_t a = pad_part_begin(r0, r1, part), b = pad_part_end(r0, r1, part);
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int64_t q = a * nvec + threadIdx.x; q < b * nvec; q += blockDim.x) base[q] = zero;
}

// ---------------------------------------------------------------------------- route
// An unsigned key with the order of the fp32 scores: non-negative values above negative
// ones, magnitudes in the right direction on each side; -0 is taken as +0 so that the two
// zeros tie, as they compare equal.
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t b = (x == 0.f) ? 0u : __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// One warp routes NTOK tokens at once (their shuffle chains interleave, which hides
// the shuffle latency). Lane l holds logits l, l+32, ..., l+32(Q-1) of each token
// (E <= 32 Q). k rounds of a warp arg-max of the score under the order (score
// descending, index ascending); lane j keeps slot j. The score is the logit, or
// logit + bias[e] in fp32 with a selection bias. Weights: softmax over the k chosen
// unbiased logits in fp32. With want_prob (aux statistics) the lane also returns in
// prob the full softmax over all E unbiased logits for its experts. Token n's row
// starts at row0 + n * row_stride; SMEM_ROW: the rows are in shared memory.
template <int Q, int NTOK, bool SMEM_ROW>
__device__ __forceinline__ void route_tokens(const float *__restrict__ row0, int row_stride,
                                             const float *__restrict__ bias, int E, int k,
                                             int lane, int (&slot_id)[NTOK],
                                             float (&slot_w)[NTOK], bool want_prob,
                                             float (&prob)[NTOK][Q]) {
  float v[NTOK][Q], sc[NTOK][Q], bq[Q];
  uint32_t taken[NTOK];
  uint32_t invalid = 0;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int e = lane + 32 * q;
    bq[q] = (e < E && bias) ? __ldg(bias + e) : 0.f;
    if (e >= E) invalid |= 1u << q;
  }
#pragma unroll
  for (int n = 0; n < NTOK; ++n) {
    const float *row = row0 + (int64_t)n * row_stride;
    taken[n] = invalid;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const int e = lane + 32 * q;
      v[n][q] = (e < E) ? (SMEM_ROW ? row[e] : __ldg(row + e)) : 0.f;
      sc[n][q] = (e < E && bias) ? v[n][q] + bq[q] : v[n][q];
    }
  }
  float my_l[NTOK];
  int my_i[NTOK];
#pragma unroll
  for (int n = 0; n < NTOK; ++n) {
    my_l[n] = 0.f;
    my_i[n] = -1;
  }
  // Each score as an order-preserving unsigned key (equal scores, +0 and -0 included,
  // give equal keys; every finite score maps above 0, which marks "none"). A round's
  // arg-max is then two warp reductions: the largest key, and the lowest expert index
  // among the lanes whose own best candidate has it.
  uint32_t key[NTOK][Q];
#pragma unroll
  for (int n = 0; n < NTOK; ++n)
#pragma unroll
    for (int q = 0; q < Q; ++q)
      key[n][q] = ((taken[n] >> q) & 1u) ? 0u : order_key(sc[n][q]);
  for (int j = 0; j < k; ++j) {
    uint32_t best[NTOK];
    int bi[NTOK];
#pragma unroll
    for (int n = 0; n < NTOK; ++n) {
      best[n] = 0u;
      bi[n] = 0x7fffffff;  // "none"
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        // candidates in ascending index: strict '>' keeps the lower index on ties
        if (!((taken[n] >> q) & 1u) && key[n][q] > best[n]) {
          best[n] = key[n][q];
          bi[n] = lane + 32 * q;
        }
      }
    }
    uint32_t top[NTOK];
#pragma unroll
    for (int n = 0; n < NTOK; ++n) top[n] = __reduce_max_sync(0xffffffffu, best[n]);
#pragma unroll
    for (int n = 0; n < NTOK; ++n)
      bi[n] = __reduce_min_sync(0xffffffffu, best[n] == top[n] ? bi[n] : 0x7fffffff);
    float lv[NTOK];
#pragma unroll
    for (int n = 0; n < NTOK; ++n) {
      const bool mine = (bi[n] & 31) == lane;
      lv[n] = 0.f;
#pragma unroll
      for (int q = 0; q < Q; ++q)
        if (mine && (bi[n] >> 5) == q) lv[n] = v[n][q];
      if (mine) taken[n] |= 1u << (bi[n] >> 5);
    }
#pragma unroll
    for (int n = 0; n < NTOK; ++n)  // the chosen expert's unbiased logit
      lv[n] = __shfl_sync(0xffffffffu, lv[n], bi[n] & 31);
#pragma unroll
    for (int n = 0; n < NTOK; ++n) {
      if (lane == j) {
        my_l[n] = lv[n];
        my_i[n] = bi[n];
      }
    }
  }
  float m[NTOK], z[NTOK], s[NTOK];
#pragma unroll
  for (int n = 0; n < NTOK; ++n) m[n] = (lane < k) ? my_l[n] : -INFINITY;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float o[NTOK];
#pragma unroll
    for (int n = 0; n < NTOK; ++n) o[n] = __shfl_xor_sync(0xffffffffu, m[n], off);
#pragma unroll
    for (int n = 0; n < NTOK; ++n) m[n] = fmaxf(m[n], o[n]);
  }
#pragma unroll
  for (int n = 0; n < NTOK; ++n) {
    z[n] = (lane < k) ? expf(my_l[n] - m[n]) : 0.f;
    s[n] = z[n];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float o[NTOK];
#pragma unroll
    for (int n = 0; n < NTOK; ++n) o[n] = __shfl_xor_sync(0xffffffffu, s[n], off);
#pragma unroll
    for (int n = 0; n < NTOK; ++n) s[n] += o[n];
  }
#pragma unroll
  for (int n = 0; n < NTOK; ++n) {
    slot_id[n] = my_i[n];
    slot_w[n] = z[n] / s[n];
  }
  if (want_prob) {
    float mx[NTOK], sum[NTOK];
#pragma unroll
    for (int n = 0; n < NTOK; ++n) {
      mx[n] = -INFINITY;
#pragma unroll
      for (int q = 0; q < Q; ++q)
        if (!((invalid >> q) & 1u)) mx[n] = fmaxf(mx[n], v[n][q]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float o[NTOK];
#pragma unroll
      for (int n = 0; n < NTOK; ++n) o[n] = __shfl_xor_sync(0xffffffffu, mx[n], off);
#pragma unroll
      for (int n = 0; n < NTOK; ++n) mx[n] = fmaxf(mx[n], o[n]);
    }
#pragma unroll
    for (int n = 0; n < NTOK; ++n) {
      sum[n] = 0.f;
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        prob[n][q] = ((invalid >> q) & 1u) ? 0.f : expf(v[n][q] - mx[n]);
        sum[n] += prob[n][q];
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float o[NTOK];
#pragma unroll
      for (int n = 0; n < NTOK; ++n) o[n] = __shfl_xor_sync(0xffffffffu, sum[n], off);
#pragma unroll
      for (int n = 0; n < NTOK; ++n) sum[n] += o[n];
    }
#pragma unroll
    for (int n = 0; n < NTOK; ++n)
#pragma unroll
      for (int q = 0; q < Q; ++q) prob[n][q] = prob[n][q] / sum[n];
  }
}

// Ballot count of one chunk of 32 tokens: for each expert, the number of tokens of
// the chunk that chose it (hist[e][c]) and, for each (token, slot), the number of
// earlier tokens of the chunk that chose the same expert (the stable local rank).
__device__ __forceinline__ void count_chunk(const int32_t (*s_ids)[kMaxK], int c, int T, int E,
                                            int k, int C, int warp, int nwarps, int lane,
                                            int32_t *__restrict__ rank,
                                            int32_t *__restrict__ hist) {
  const int t = c * kChunk + lane;
  const bool valid = t < T;
  for (int e = warp; e < E; e += nwarps) {
    int slot = -1;
    if (valid) {
      for (int j = 0; j < k; ++j)
        if (s_ids[lane][j] == e) slot = j;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, slot >= 0);
    if (slot >= 0) rank[(int64_t)t * k + slot] = __popc(m & lanemask_lt());
    if (lane == 0) hist[(int64_t)e * C + c] = __popc(m);
  }
}

}  // namespace moe
