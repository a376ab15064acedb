// The router in front of the expert block: fp32 logits = x W_r^T computed from the
// bf16 hidden states and router weight, with the top-k route, the chunk histogram and
// the local ranks of the dispatch taken from those logits in the same kernel.
//
// "Halo's 2.8x over TRL is not a kernel, and its own benchmark proves it" computes the
// router logits in fp32 ("Where the gap actually is"; `fp32_router: true` in the LFM2
// recipe of "The small-hardware end") ahead of the per-token top-k router of Figure 3.
// Each logit here is one fp32 chain over i = 0 .. d-1 in order: fmaf adds the exact
// product of two bf16 values (two 8-bit significands fit fp32) with one rounding, so
// the logits, and every top-k decision taken on them, are reproducible bit for bit.
#include "route_common.cuh"

namespace moe {

namespace {

constexpr int kSub = 2;          // 64-column TMA boxes (one 128-byte row each) per stage
constexpr int kKB = 64 * kSub;   // k per staged block

// acc = a * b + acc for the bf16 in the low (HI = false) or high half of a and b: the
// exact product of two bf16 values added to the fp32 accumulator with one rounding
// (the same value as fmaf on the widened operands), without unpacking the operands.
template <bool HI>
__device__ __forceinline__ float fma_bf16(uint32_t a, uint32_t b, float acc) {
  float d;
  if (HI)
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
        : "=f"(d) : "r"(a), "r"(b), "f"(acc));
  else
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
        : "=f"(d) : "r"(a), "r"(b), "f"(acc));
  return d;
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Route of the block's 32 tokens from shared-memory logits, one lane per token (no
// shuffles: the k rounds of warp arg-max in route_kernel are chains of dependent
// shuffles, which a few warps cannot hide). Every warp scans a contiguous range of
// experts for all 32 tokens, keeping a sorted top-KP list per lane (score descending;
// a later expert replaces an entry only with a strictly larger score, so equal scores
// keep the lower index); a merge tree over the warps, always the lower expert range
// first on ties, gives the top-k. The softmax sums repeat, term for term, the
// butterfly association of route_kernel's warp reductions, so ids, weights and the
// load-balancing rows are bit-identical to routing the same logits from memory.
// Rows are padded to LS = E + 1 floats so that lane-per-token reads hit distinct banks.
template <int KP, int NW>
__device__ __forceinline__ void route_chunk_lanes(const float *s_log, int LS, float *s_prob,
                                                  float *s_work, const float *__restrict__ bias,
                                                  int E, int k, int nt, int warp, int lane,
                                                  int64_t t0, int32_t *__restrict__ ids,
                                                  float *__restrict__ w,
                                                  int32_t (*s_ids)[kMaxK], bool want_prob) {
  const int i = lane;
  const float *row = s_log + i * LS;
  float *L_s = s_work;                                          // [NW][KP][32]
  float *L_l = L_s + NW * KP * 32;
  int *L_i = reinterpret_cast<int *>(L_l + NW * KP * 32);
  float *s_mx = reinterpret_cast<float *>(L_i + NW * KP * 32);  // [NW][32]
  float *s_part = s_mx + NW * 32;                               // [32][32]
  float *s_tot = s_part + 32 * 32;                              // [32]
  const int e0 = (E * warp) / NW, e1 = (E * (warp + 1)) / NW;

  float sv[KP], lv[KP];
  int si[KP];
#pragma unroll
  for (int j = 0; j < KP; ++j) {
    sv[j] = 0.f;
    lv[j] = 0.f;
    si[j] = -1;  // empty
  }
  for (int e = e0; e < e1; ++e) {
    const float lg = row[e];
    const float sc = bias ? lg + __ldg(bias + e) : lg;
#pragma unroll
    for (int j = KP - 1; j >= 0; --j) {  // slot j - 1 is read before it changes
      const bool here = si[j] < 0 || sc > sv[j];
      const bool up = j > 0 && (si[j - 1] < 0 || sc > sv[j - 1]);
      if (up) {
        sv[j] = sv[j - 1];
        lv[j] = lv[j - 1];
        si[j] = si[j - 1];
      } else if (here) {
        sv[j] = sc;
        lv[j] = lg;
        si[j] = e;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < KP; ++j) {
    const int o = (warp * KP + j) * 32 + lane;
    L_s[o] = sv[j];
    L_l[o] = lv[j];
    L_i[o] = si[j];
  }
  __syncthreads();
#pragma unroll
  for (int half = 1; half < NW; half *= 2) {
    if (warp % (2 * half) == 0 && warp + half < NW) {
      const int A = warp * KP * 32 + lane, B = (warp + half) * KP * 32 + lane;
      int ia = 0, ib = 0;
#pragma unroll
      for (int j = 0; j < KP; ++j) {
        const bool av = ia < KP && L_i[A + ia * 32] >= 0;
        const bool bv = ib < KP && L_i[B + ib * 32] >= 0;
        const float as = av ? L_s[A + ia * 32] : 0.f, bs = bv ? L_s[B + ib * 32] : 0.f;
        if (bv && (!av || bs > as)) {
          sv[j] = bs;
          lv[j] = L_l[B + ib * 32];
          si[j] = L_i[B + ib * 32];
          ++ib;
        } else {
          sv[j] = as;
          lv[j] = av ? L_l[A + ia * 32] : 0.f;
          si[j] = av ? L_i[A + ia * 32] : -1;
          ia += av ? 1 : 0;
        }
      }
#pragma unroll
      for (int j = 0; j < KP; ++j) {  // every read of the two lists is done
        L_s[A + j * 32] = sv[j];
        L_l[A + j * 32] = lv[j];
        L_i[A + j * 32] = si[j];
      }
    }
    __syncthreads();
  }
  if (warp == 0 && i < nt) {
    // warp 0 holds the final list (it took part in every merge level)
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < KP; ++j)
      if (j < k) m = fmaxf(m, lv[j]);
    float z[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) z[j] = (j < KP && j < k) ? expf(lv[j] - m) : 0.f;
    // route_kernel's butterfly over lanes (xor 16, 8, 4, 2, 1), lanes >= k holding 0
    float t8[8], t4[4];
#pragma unroll
    for (int l = 0; l < 8; ++l) t8[l] = z[l] + z[l + 8];
#pragma unroll
    for (int l = 0; l < 4; ++l) t4[l] = t8[l] + t8[l + 4];
    const float sum = (t4[0] + t4[2]) + (t4[1] + t4[3]);
    const int64_t t = t0 + i;
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      if (j < k) {
        ids[t * k + j] = si[j];
        w[t * k + j] = z[j] / sum;
        s_ids[i][j] = si[j];
      }
    }
  }
  if (want_prob) {
    // softmax over all E logits, with route_kernel's sums: per lane l of that kernel
    // the experts l, l + 32, ... in order, then the xor butterfly over the 32 lanes
    float pm = -INFINITY;
    for (int e = e0; e < e1; ++e) pm = fmaxf(pm, row[e]);
    s_mx[warp * 32 + lane] = pm;
    __syncthreads();
    float mx = -INFINITY;
#pragma unroll
    for (int v = 0; v < NW; ++v) mx = fmaxf(mx, s_mx[v * 32 + lane]);
    for (int e = e0; e < e1; ++e) s_prob[i * LS + e] = expf(row[e] - mx);
    __syncthreads();
    constexpr int LPW = 32 / NW;
    for (int l = warp * LPW; l < (warp + 1) * LPW; ++l) {
      float acc = 0.f;
      for (int e = l; e < E; e += 32) acc += s_prob[i * LS + e];
      s_part[l * 32 + lane] = acc;
    }
    __syncthreads();
    if (warp == 0) {
      float p[32];
#pragma unroll
      for (int l = 0; l < 32; ++l) p[l] = s_part[l * 32 + lane];
#pragma unroll
      for (int h = 16; h > 0; h >>= 1)
#pragma unroll
        for (int l = 0; l < h; ++l) p[l] = p[l] + p[l + h];
      s_tot[lane] = p[0];
    }
    __syncthreads();
    const float tot = s_tot[lane];
    for (int e = e0; e < e1; ++e)
      s_prob[i * LS + e] = (i < nt) ? s_prob[i * LS + e] / tot : 0.f;
  }
}

// shared-memory bytes the route of a chunk needs past the two [32][E+1] float arrays
template <int NW>
__host__ __device__ constexpr size_t route_lanes_work() {
  return (size_t)NW * 16 * 32 * 12 + NW * 32 * 4 + 32 * 32 * 4 + 32 * 4;
}

// Block c computes the logits of tokens [32c, 32c+32) for all experts, stores them,
// then routes the chunk exactly as route_kernel does (warp per token) and, with COUNT,
// writes the chunk histogram and local ranks.
//
// Thread tile: TT tokens x TE experts. Lane bits: token group tg fastest (32/TT of
// them), then expert group eg; the thread owns tokens tg + (32/TT) j and experts
// eg + EG j. EP = EG * TE >= E.
//
// Staging, per block of 128 k: one thread issues TMA loads of two 64-column boxes each
// of the x rows [32c, 32c+32) and of the W_r rows [0, EP) (128-byte swizzle: 16-byte
// chunk j of row r lands at chunk j ^ (r % 8)) into a ring of S stages; rows past T or E and columns past d arrive as
// zeros. The arithmetic reads its bf16 operands straight from the stage, 8 k per
// 16-byte load (the swizzle spreads the few rows a warp reads over distinct banks), and
// runs the chains with the mixed-precision fma. A barrier per block frees the stage
// for the next load. A wait for a TMA load that does not complete within the limit
// sets *status (when given), marks the chunk's ids -1 and ends the block.
template <int TT, int TE, int EG, int S, bool COUNT>
__global__ void __launch_bounds__((32 / TT) * EG, 1) router_route_kernel(
    const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
    const float *__restrict__ bias, float *__restrict__ logits, int32_t *__restrict__ ids,
    float *__restrict__ w, int32_t *__restrict__ rank, int32_t *__restrict__ hist,
    float *__restrict__ prob_part, int *__restrict__ status, int T, int d, int E, int k, int C) {
  constexpr int TG = 32 / TT;
  constexpr int NT = TG * EG;
  constexpr int EP = EG * TE;
  constexpr int ROWS = kChunk + EP;
  constexpr int SUB = ROWS * 128;           // bytes of one 64-column sub-block
  constexpr int STAGE = SUB * kSub;         // bytes of one ring stage
  static_assert(kChunk % TT == 0 && NT % 32 == 0 && EP % 8 == 0, "tile");
  static_assert((size_t)S * STAGE >= 2 * sizeof(float) * kChunk * (EP + 1) +
                    route_lanes_work<NT / 32>(), "epilogue space");

  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t full[S];
  __shared__ int32_t s_ids[kChunk][kMaxK];
  const int tid = threadIdx.x;
  const int tg = tid % TG, eg = tid / TG;
  const int c = blockIdx.x;
  const int t0 = c * kChunk;
  const int nblk = (d + kKB - 1) / kKB;

  if (tid == 0) {
    for (int i = 0; i < S; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
  }
  __syncthreads();
  auto issue = [&](int b) {  // thread 0: block b into stage b % S
    uint8_t *dst = smem + (b % S) * STAGE;
    mbar_arrive_expect_tx(&full[b % S], STAGE);
#pragma unroll
    for (int u = 0; u < kSub; ++u) {
      tma_load_2d(dst + u * SUB, &tm_x, &full[b % S], b * kKB + 64 * u, t0);
      tma_load_2d(dst + u * SUB + kChunk * 128, &tm_w, &full[b % S], b * kKB + 64 * u, 0);
    }
  };
  if (tid == 0)
    for (int b = 0; b < S && b < nblk; ++b) issue(b);

  // byte offset of this thread's rows in a stage, with the row's swizzle folded in:
  // chunk j of row r is at (r * 128 + (r % 8) * 16) ^ (j * 16)
  int xo[TT], wo[TE];
#pragma unroll
  for (int a = 0; a < TT; ++a) {
    const int r = tg + TG * a;
    xo[a] = r * 128 + ((r & 7) << 4);
  }
#pragma unroll
  for (int e = 0; e < TE; ++e) {
    const int r = kChunk + eg + EG * e;
    wo[e] = r * 128 + ((r & 7) << 4);
  }

  float acc[TT][TE];
#pragma unroll
  for (int a = 0; a < TT; ++a)
#pragma unroll
    for (int e = 0; e < TE; ++e) acc[a][e] = 0.f;
  // one 16-byte chunk (k = 8j .. 8j+7) of every operand row: chains in ascending k
  auto fma_chunk = [&](const uint4 (&xv)[TT], const uint4 (&wv)[TE]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int a = 0; a < TT; ++a)
#pragma unroll
        for (int e = 0; e < TE; ++e)
          acc[a][e] = fma_bf16<false>(word(xv[a], i), word(wv[e], i), acc[a][e]);
#pragma unroll
      for (int a = 0; a < TT; ++a)
#pragma unroll
        for (int e = 0; e < TE; ++e)
          acc[a][e] = fma_bf16<true>(word(xv[a], i), word(wv[e], i), acc[a][e]);
    }
  };

  // The wait for a block and the barrier that frees the previous stage are one step:
  // every thread waits for block b, then __syncthreads_or both frees stage b - 1 and
  // makes the give-up decision the same in every thread.
  bool fail = __syncthreads_or(!mbar_wait(&full[0], 0, status)) != 0;
  int b = 0;
  for (; b < nblk && !fail; ++b) {
    const uint8_t *sbase = smem + (b % S) * STAGE;
#pragma unroll 1
    for (int u = 0; u < kSub; ++u) {  // the stage's 64-column sub-blocks in k order
      const uint8_t *sb = sbase + u * SUB;
      uint4 xA[TT], wA[TE], xB[TT], wB[TE];  // two register sets: the next chunk loads early
#pragma unroll
      for (int a = 0; a < TT; ++a) xA[a] = *reinterpret_cast<const uint4 *>(sb + xo[a]);
#pragma unroll
      for (int e = 0; e < TE; ++e) wA[e] = *reinterpret_cast<const uint4 *>(sb + wo[e]);
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
#pragma unroll
        for (int a = 0; a < TT; ++a)
          xB[a] = *reinterpret_cast<const uint4 *>(sb + (xo[a] ^ ((j + 1) << 4)));
#pragma unroll
        for (int e = 0; e < TE; ++e)
          wB[e] = *reinterpret_cast<const uint4 *>(sb + (wo[e] ^ ((j + 1) << 4)));
        fma_chunk(xA, wA);
        if (j + 2 < 8) {
#pragma unroll
          for (int a = 0; a < TT; ++a)
            xA[a] = *reinterpret_cast<const uint4 *>(sb + (xo[a] ^ ((j + 2) << 4)));
#pragma unroll
          for (int e = 0; e < TE; ++e)
            wA[e] = *reinterpret_cast<const uint4 *>(sb + (wo[e] ^ ((j + 2) << 4)));
        }
        fma_chunk(xB, wB);
      }
    }
    const bool ok = b + 1 >= nblk || mbar_wait(&full[(b + 1) % S], ((b + 1) / S) & 1, status);
    fail = __syncthreads_or(!ok) != 0;
    if (tid == 0 && !fail && b + S < nblk) issue(b + S);  // into the stage of block b
  }
  if (fail) {
    // block b timed out; let the loads already issued (b .. b + S - 1) land, bounded,
    // before the block's shared memory goes away
    if (tid == 0)
      for (int bb = b; bb < nblk && bb < b + S; ++bb)
        mbar_wait(&full[bb % S], (bb / S) & 1, status, 100000000ull);
    const int nt = min(kChunk, T - t0);
    for (int i = tid; i < nt * k; i += NT) ids[(int64_t)t0 * k + i] = -1;
    return;
  }

  // (the last barrier of the loop: every thread is done with the ring)
  // logits [32][E+1] and the softmax rows [32][E+1] for the statistics, then the
  // route's work area, over the ring
  const int LS = E + 1;
  float *s_log = reinterpret_cast<float *>(smem);
  float *s_prob = s_log + kChunk * LS;
  float *s_work = s_prob + kChunk * LS;
#pragma unroll
  for (int a = 0; a < TT; ++a)
#pragma unroll
    for (int e = 0; e < TE; ++e) {
      const int ex = eg + EG * e;
      if (ex < E) s_log[(tg + TG * a) * LS + ex] = acc[a][e];
    }
  __syncthreads();
  const int nt = min(kChunk, T - t0);
  for (int i = tid; i < nt * E; i += NT) {
    const int r = i / E;
    logits[(int64_t)t0 * E + i] = s_log[r * LS + (i - r * E)];
  }

  const int warp = tid >> 5, lane = tid & 31;
  constexpr int NW = NT / 32;
  const bool want_prob = prob_part != nullptr;
  if (k <= 1)
    route_chunk_lanes<1, NW>(s_log, LS, s_prob, s_work, bias, E, k, nt, warp, lane, t0, ids, w,
                             s_ids, want_prob);
  else if (k <= 2)
    route_chunk_lanes<2, NW>(s_log, LS, s_prob, s_work, bias, E, k, nt, warp, lane, t0, ids, w,
                             s_ids, want_prob);
  else if (k <= 4)
    route_chunk_lanes<4, NW>(s_log, LS, s_prob, s_work, bias, E, k, nt, warp, lane, t0, ids, w,
                             s_ids, want_prob);
  else if (k <= 8)
    route_chunk_lanes<8, NW>(s_log, LS, s_prob, s_work, bias, E, k, nt, warp, lane, t0, ids, w,
                             s_ids, want_prob);
  else
    route_chunk_lanes<16, NW>(s_log, LS, s_prob, s_work, bias, E, k, nt, warp, lane, t0, ids, w,
                              s_ids, want_prob);
  if (COUNT || prob_part) __syncthreads();
  if (prob_part) {
    for (int e = tid; e < E; e += NT) {
      float s = 0.f;
      for (int i = 0; i < kChunk; ++i) s += s_prob[i * LS + e];
      prob_part[(int64_t)e * C + c] = s;
    }
  }
  if constexpr (COUNT) count_chunk(s_ids, c, T, E, k, C, warp, NW, lane, rank, hist);
}

template <int TT, int TE, int EG, int S>
constexpr size_t router_smem() {
  return (size_t)S * (kChunk + EG * TE) * 128 * kSub + 1024;  // + alignment slack
}

template <int TT, int TE, int EG, int S, bool COUNT>
cudaError_t launch_router_as(const void *x, const void *w_r, const float *bias, float *logits,
                             int32_t *ids, float *w, int32_t *rank, int32_t *hist,
                             float *prob_part, int *status, int T, int d, int E, int k, int C,
                             cudaStream_t st) {
  constexpr int NT = (32 / TT) * EG;
  constexpr int EP = EG * TE;
  constexpr size_t smem = router_smem<TT, TE, EG, S>();
  static_assert(smem <= 227 * 1024, "shared memory");
  auto kernel = router_route_kernel<TT, TE, EG, S, COUNT>;
  static bool attr_set[64] = {};  // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set[dev & 63] = true;
  }
  CUtensorMap tm_x, tm_w;
  const uint64_t sx[1] = {(uint64_t)d * 2};
  const uint64_t dx[2] = {(uint64_t)d, (uint64_t)T}, dw[2] = {(uint64_t)d, (uint64_t)E};
  const uint32_t bx[2] = {64u, (uint32_t)kChunk}, bw[2] = {64u, (uint32_t)EP};
  cudaError_t e = encode_tensor_map(&tm_x, x, 2, dx, sx, bx, 128);
  if (e == cudaSuccess) e = encode_tensor_map(&tm_w, w_r, 2, dw, sx, bw, 128);
  if (e != cudaSuccess) return e;
  launch_begin(st);
  kernel<<<C, NT, smem, st>>>(tm_x, tm_w, bias, logits, ids, w, rank, hist, prob_part, status, T,
                              d, E, k, C);
  return note_launch(COUNT ? "router_route_count" : "router_route", st);
}

template <bool COUNT>
cudaError_t launch_router_cfg(const void *x, const void *w_r, const float *bias, float *logits,
                              int32_t *ids, float *w, int32_t *rank, int32_t *hist,
                              float *prob_part, int *status, int T, int d, int E, int k, int C,
                              cudaStream_t st) {
#define MOE_ROUTER(TT, TE, EG, S)                                                             \
  return launch_router_as<TT, TE, EG, S, COUNT>(x, w_r, bias, logits, ids, w, rank, hist,    \
                                                prob_part, status, T, d, E, k, C, st)
  if (E <= 8) MOE_ROUTER(4, 1, 8, 6);
  if (E <= 16) MOE_ROUTER(4, 2, 8, 6);
  if (E <= 32) MOE_ROUTER(4, 2, 16, 3);
  if (E <= 64) MOE_ROUTER(4, 4, 16, 3);
  if (E <= 128) MOE_ROUTER(4, 4, 32, 3);
  MOE_ROUTER(8, 4, 64, 2);
#undef MOE_ROUTER
}

// ------------------------------------------------------------------- router backward
// The gradient through logits = x W_r^T for a given dlogits [T][E] (fp32):
//   dW_r[e][i] = sum_t dlogits[t][e] x[t][i]       dX[t][i] += sum_e dlogits[t][e] W_r[e][i]
// Both in fp32 on the SIMT pipes (dlogits is fp32; bf16 operands are widened exactly).
// A thread owns 4 rows x 8 columns (one 16-byte bf16 vector of the wide operand); per
// step of the reduction it loads 4 fp32 values (the same for the whole warp) and 8 bf16.

constexpr int kRbCols = 256;     // columns of d per block (8 per lane)
constexpr int kRbRows = 32;      // tokens (dX) or experts (dW) per block: 4 per warp

// dX: block (token chunk, column block). dl and W_r staged 64 experts at a time.
__global__ void __launch_bounds__(256) router_dx_kernel(const float *__restrict__ dl,
                                                        const uint4 *__restrict__ w_r,
                                                        uint4 *__restrict__ dx, int T, int d,
                                                        int E) {
  constexpr int EB = 64;
  __shared__ __align__(16) float s_dl[EB][kRbRows + 4];    // [e][token], padded rows
  __shared__ __align__(16) uint4 s_w[EB][kRbCols / 8];     // [e][8-column vector]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRbRows, c0 = blockIdx.y * kRbCols;
  const int nvr = d >> 3, v = (c0 >> 3) + lane;            // this lane's column vector
  float acc[4][8];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[a][j] = 0.f;
  for (int e0 = 0; e0 < E; e0 += EB) {
    const int ne = min(EB, E - e0);
    __syncthreads();  // the previous tiles are consumed
    for (int idx = threadIdx.x; idx < EB * kRbRows; idx += 256) {
      const int t = idx / EB, e = idx % EB;  // consecutive threads: consecutive experts
      s_dl[e][t] = (e < ne && t0 + t < T) ? dl[(int64_t)(t0 + t) * E + e0 + e] : 0.f;
    }
    for (int idx = threadIdx.x; idx < EB * (kRbCols / 8); idx += 256) {
      const int e = idx / (kRbCols / 8), c = idx % (kRbCols / 8);
      const int vv = (c0 >> 3) + c;
      s_w[e][c] = (e < ne && vv < nvr) ? ldg_nc(w_r + (int64_t)(e0 + e) * nvr + vv)
                                       : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    for (int e = 0; e < ne; ++e) {
      const float4 g = *reinterpret_cast<const float4 *>(&s_dl[e][4 * warp]);
      float wv[8];
      unpack8(s_w[e][lane], wv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[0][j] = fmaf(g.x, wv[j], acc[0][j]);
        acc[1][j] = fmaf(g.y, wv[j], acc[1][j]);
        acc[2][j] = fmaf(g.z, wv[j], acc[2][j]);
        acc[3][j] = fmaf(g.w, wv[j], acc[3][j]);
      }
    }
  }
  if (v >= nvr) return;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int t = t0 + 4 * warp + a;
    if (t >= T) break;
    uint4 *p = dx + (int64_t)t * nvr + v;
    float f[8];
    unpack8(*p, f);
#pragma unroll
    for (int j = 0; j < 8; ++j) f[j] += acc[a][j];
    *p = pack8(f);
  }
}

// dW partials: block (column block, expert block, token split). Token tiles of 32;
// each split sums its tokens in order into part[split][e][i] (or straight into dW when
// there is one split). The next tile's loads wait in registers while the current tile
// is summed (two shared-memory buffers, one barrier per tile).
__global__ void __launch_bounds__(256) router_dw_kernel(const float *__restrict__ dl,
                                                        const uint4 *__restrict__ x,
                                                        float *__restrict__ part, int T, int d,
                                                        int E, int split_tokens) {
  constexpr int TB = 32;
  constexpr int XV = TB * (kRbCols / 8) / 256;             // x vectors per thread per tile
  __shared__ __align__(16) float s_dl[2][TB][kRbRows];     // [buf][token][expert]
  __shared__ __align__(16) uint4 s_x[2][TB][kRbCols / 8];  // [buf][token][8-column vector]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * kRbCols, e0 = blockIdx.y * kRbRows;
  const int ts = blockIdx.z;
  const int tbeg = ts * split_tokens, tend = min(T, tbeg + split_tokens);
  const int nvr = d >> 3, v = (c0 >> 3) + lane;
  // this thread's staging work: dl value (token dt, expert de), x vectors (token xt[i],
  // column vector xc)
  const int dt = threadIdx.x / kRbRows, de = threadIdx.x % kRbRows;  // 8 tokens x 32 experts
  const int xc = threadIdx.x % (kRbCols / 8), xt0 = threadIdx.x / (kRbCols / 8);
  float rdl[TB * kRbRows / 256];
  uint4 rx[XV];
  auto fetch = [&](int t0) {
    const int nt = min(TB, tend - t0);
#pragma unroll
    for (int i = 0; i < TB * kRbRows / 256; ++i) {
      const int t = dt + 8 * i;
      rdl[i] = (t < nt && e0 + de < E) ? dl[(int64_t)(t0 + t) * E + e0 + de] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < XV; ++i) {
      const int t = xt0 + (256 / (kRbCols / 8)) * i;
      const int vv = (c0 >> 3) + xc;
      rx[i] = (t < nt && vv < nvr) ? ldg_nc(x + (int64_t)(t0 + t) * nvr + vv)
                                   : make_uint4(0, 0, 0, 0);
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int i = 0; i < TB * kRbRows / 256; ++i) s_dl[buf][dt + 8 * i][de] = rdl[i];
#pragma unroll
    for (int i = 0; i < XV; ++i) s_x[buf][xt0 + (256 / (kRbCols / 8)) * i][xc] = rx[i];
  };
  float acc[4][8];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[a][j] = 0.f;
  if (tbeg < tend) {
    fetch(tbeg);
    stash(0);
  }
  __syncthreads();
  int buf = 0;
  for (int t0 = tbeg; t0 < tend; t0 += TB, buf ^= 1) {
    const int nt = min(TB, tend - t0);
    const bool more = t0 + TB < tend;
    if (more) fetch(t0 + TB);
    for (int t = 0; t < nt; ++t) {
      const float4 g = *reinterpret_cast<const float4 *>(&s_dl[buf][t][4 * warp]);
      float xv[8];
      unpack8(s_x[buf][t][lane], xv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[0][j] = fmaf(g.x, xv[j], acc[0][j]);
        acc[1][j] = fmaf(g.y, xv[j], acc[1][j]);
        acc[2][j] = fmaf(g.z, xv[j], acc[2][j]);
        acc[3][j] = fmaf(g.w, xv[j], acc[3][j]);
      }
    }
    if (more) stash(buf ^ 1);  // the other buffer was last read before the previous barrier
    __syncthreads();
  }
  if (v >= nvr) return;
  float *out = part + (int64_t)ts * E * d;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int e = e0 + 4 * warp + a;
    if (e >= E) break;
    float4 *p = reinterpret_cast<float4 *>(out + (int64_t)e * d + 8 * (int64_t)v);
    p[0] = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    p[1] = make_float4(acc[a][4], acc[a][5], acc[a][6], acc[a][7]);
  }
}

// dW = sum of the splits' partials, in split order.
__global__ void __launch_bounds__(256) router_dw_reduce_kernel(const float4 *__restrict__ part,
                                                               float4 *__restrict__ dw,
                                                               int64_t n4, int splits) {
  for (int64_t i = blockIdx.x * 256ll + threadIdx.x; i < n4; i += (int64_t)gridDim.x * 256) {
    float4 s = part[i];
    for (int p = 1; p < splits; ++p) {
      const float4 q = part[(int64_t)p * n4 + i];
      s.x += q.x;
      s.y += q.y;
      s.z += q.z;
      s.w += q.w;
    }
    dw[i] = s;
  }
}

}  // namespace

cudaError_t launch_router_route(const void *x, const void *w_r, const float *bias, float *logits,
                                int32_t *ids, float *w, int32_t *rank, int32_t *hist,
                                float *prob_part, int *status, int T, int d, int E, int k,
                                bool with_count, cudaStream_t st) {
  const int C = (T + kChunk - 1) / kChunk;
  if (C == 0) return cudaSuccess;
  if (with_count)
    return launch_router_cfg<true>(x, w_r, bias, logits, ids, w, rank, hist, prob_part, status, T,
                                   d, E, k, C, st);
  return launch_router_cfg<false>(x, w_r, bias, logits, ids, w, rank, hist, prob_part, status, T,
                                  d, E, k, C, st);
}

// The token splits of dW_r: about two waves of blocks on the 152 SMs of a GB300, fixed
// by the shape alone so that the scratch size and the order of the sums are the same on
// every machine.
int router_dw_splits(int T, int d, int E) {
  const int cells = ((d + kRbCols - 1) / kRbCols) * ((E + kRbRows - 1) / kRbRows);
  const int chunks = (T + 31) / 32;
  const int splits = (2 * 152 + cells - 1) / cells;
  return max(1, min(splits, chunks));
}

cudaError_t launch_router_dx(const void *w_r, const float *dlogits, void *dx, int T, int d,
                             int E, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const dim3 bdx((T + kRbRows - 1) / kRbRows, (d + kRbCols - 1) / kRbCols);
  launch_begin(st);
  router_dx_kernel<<<bdx, 256, 0, st>>>(dlogits, static_cast<const uint4 *>(w_r),
                                        static_cast<uint4 *>(dx), T, d, E);
  return note_launch("router_dx", st);
}

cudaError_t launch_router_dw(const void *x, const float *dlogits, float *dw, float *part, int T,
                             int d, int E, cudaStream_t st) {
  const int splits = router_dw_splits(T, d, E);
  const int chunks = max(1, (T + 31) / 32);
  const int split_tokens = ((chunks + splits - 1) / splits) * 32;
  const int nsplit = T > 0 ? (T + split_tokens - 1) / split_tokens : 1;  // <= splits
  const dim3 bdw((d + kRbCols - 1) / kRbCols, (E + kRbRows - 1) / kRbRows, nsplit);
  launch_begin(st);
  router_dw_kernel<<<bdw, 256, 0, st>>>(dlogits, static_cast<const uint4 *>(x),
                                        nsplit == 1 ? dw : part, T, d, E, split_tokens);
  cudaError_t e = note_launch("router_dw", st);
  if (e != cudaSuccess || nsplit == 1) return e;
  const int64_t n4 = (int64_t)E * d / 4;
  const int64_t blocks = (n4 + 255) / 256, cap = 4 * (int64_t)num_sms();
  launch_begin(st);
  router_dw_reduce_kernel<<<(int)(blocks < cap ? blocks : cap), 256, 0, st>>>(
      reinterpret_cast<const float4 *>(part), reinterpret_cast<float4 *>(dw), n4, nsplit);
  return note_launch("router_dw_reduce", st);
}

}  // namespace moe
