// Grouped GEMM engine of the MoE expert block on the sm_103a tensor cores.
//
// The experts of "Halo: Frontier-Lab Training for Everyone" ("Novel model
// integration": grouped GEMM with a fused SwiGLU; "One trainer architecture": fused
// experts as 3-D weight tensors) run as one persistent kernel per GEMM over all
// experts. Design:
//   * one CTA per SM: warp 0 issues TMA loads, warp 1 issues tcgen05.mma (one elected
//     lane), the other warps run the epilogue out of TMEM (per kind 8, two per TMEM lane
//     quarter each on half of the tile's columns, or 4, one per quarter);
//   * two forms: a CTA alone on a 128 x 256 (M x N) tile, or a 2-CTA cluster on a
//     256 x 256 tile through the cta_group::2 MMA (each CTA loads its 128 A rows and
//     half of B, the even CTA issues the MMAs);
//   * 128-byte swizzled operands brought by cp.async.bulk.tensor into an mbarrier ring
//     of 192 KB per CTA (pairs: 3 stages of two K-blocks of 64; single CTAs: 4 stages
//     of one);
//   * the fp32 accumulator lives in TMEM, two 256-column buffers so the epilogue of
//     one tile overlaps the main loop of the next;
//   * ragged per-expert M: expert segments are padded to 128 rows, so every M tile
//     belongs to one expert and a device-side table maps tile -> expert (no host
//     sync, the schedule reads the routing result from device memory);
//   * ragged per-expert K (weight gradients): the K loop runs over the expert's rows
//     and stops at the last 16-row slice that holds one.
// Every output element is written by exactly one thread; nothing uses atomics.
#include "kernels.h"

#include <cudaTypedefs.h>
#include <mutex>

namespace moe {
namespace {

// Two forms of the engine, chosen per launch. Single: one CTA per 128 x 256 tile.
// Pair: two SMs (a 2-CTA cluster) share one 256 x 256 tile through the cta_group::2
// MMA: each CTA loads its own 128 rows of A and half of the B tile, the even CTA
// issues the MMA, and each CTA keeps its 128 rows of the accumulator in its TMEM. Per
// CTA a k-block then moves 32 KB instead of 48 KB, which leaves room for 6 K-blocks in flight.
constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kABytes = BM * BK * 2;  // 16 KB

template <bool PAIR>
struct Cfg {
  static constexpr int kMTile = PAIR ? 2 * BM : BM;  // rows of one (pair-)tile
  static constexpr int kBRows = PAIR ? BN / 2 : BN;  // B rows (N) each CTA loads
  // A pipeline stage holds kSub K-blocks of 64 (each its own 128-byte-swizzled A and
  // B tiles): the MMA issuer waits for, and commits, one stage of kSub * 4 MMAs at a
  // time. Measured on GB300: a barrier round costs about as much as two or three MMAs,
  // so the pairs run faster on 3 stages of 128 K than on 6 of 64 K (same bytes in
  // flight); the single-CTA form, whose K-blocks are 48 KB, keeps 4 stages of one.
  static constexpr int kSub = PAIR ? 2 : 1;
  static constexpr int kBKS = BK * kSub;  // K per stage
  static constexpr int kStages = (PAIR ? 6 : 4) / kSub;
  static constexpr int kBBytes = kBRows * BK * 2;    // 16 or 32 KB
  static constexpr int kSubBytes = kABytes + kBBytes;  // one K-block of 64
  static constexpr int kStageBytes = kSub * kSubBytes;
};
constexpr int kBoxBytes = 64 * 64 * 2;  // one 64 x 64 bf16 box (MN-major tiles are built of these)
constexpr int kEpiWarps = 8;  // at most: two per TMEM lane quarter, each on half of the columns
constexpr int kTmemCols = 512;
// epilogue staging: per epilogue warp two 32-row x 32-column bf16 buffers (2 KB each,
// 64-byte swizzled like the TMA store expects)
constexpr int kStageOutBytes = 32 * 32 * 2;
constexpr int kEpiSmem = kEpiWarps * 2 * kStageOutBytes;
template <bool PAIR>
constexpr int smem_bytes() {
  return Cfg<PAIR>::kStages * Cfg<PAIR>::kStageBytes + kEpiSmem + 1024;
}
// ragged-M GEMMs run on pairs when experts average at least this many rows. Measured on
// GB300 at 256 rows per expert (qwen3_moe-like: 217-304 rows, so about half the experts end
// in a half-empty pair-tile): pairs 206 / 118 us for gate_up / down against 213 / 122 us
// for single CTAs, whose 128 x 256 tiles need 1.5x the operand bytes per MMA.
constexpr int64_t kPairMinRows = 256;
// Ragged-M tile order (see decode): weight-stationary when experts have few rows
// (each weight tile is then shared by only a few CTAs, which should run together),
// m-tile major when they have many (the activation rows are then the reused operand).
// Measured on GB300: weight-stationary is faster at 512 rows per expert, m-major at 8192.
constexpr int64_t kWeightStationaryMaxRows = 2048;

enum Kind { GATE_UP = 0, DOWN = 1, DGRAD_H = 2, DGRAD_X = 3, WGRAD = 4 };

// Epilogue warps of a kind: 8 (two per TMEM lane quarter, each on half of the tile's
// columns) or 4 (one per quarter, both halves in turn). Four leave fewer warps beside
// the producer and MMA lanes on their SMSPs; measured on GB300 at gpt_oss_20b they made
// gate_up, down and dgrad_x 3-5 us faster each, but wgrad_down slower and dgrad_h (whose
// SwiGLU-backward epilogue is the heaviest) 60 us slower.
template <int KIND>
constexpr int epi_warps() {
  return (KIND == GATE_UP || KIND == DOWN || KIND == DGRAD_X) ? 4 : 8;
}
// The DGRAD_H epilogue gives each warp one half of the tile's columns (ch_own >= 0).
static_assert(epi_warps<DGRAD_H>() == 8, "the DGRAD_H epilogue needs two warps per lane quarter");
template <int KIND>
constexpr int threads_of() {
  return 64 + 32 * epi_warps<KIND>();
}

struct Args {
  const int32_t *padded;       // [E+1]
  const int32_t *counts;       // [E] rows of each expert (WGRAD: the K extent)
  const int32_t *tile_expert;  // [R/128]
  const int32_t *pair_start;   // [E+1] (pair mode)
  const int32_t *pair_expert;  // pair-tile -> expert (pair mode)
  int E;
  int n_tiles;  // tiles along N
  int m_tiles;  // WGRAD: (pair-)tiles along M of one expert's dW
  int k_tiles;  // ragged-M kinds: K / (K per stage), rounded up
  int k_last;   // ragged-M kinds: 16-wide K slices of the last stage that hold columns
  int weight_stationary;  // short experts: ragged-M and weight-gradient tile orders
  int M_out;    // WGRAD: rows of dW[e]
  int N_out;    // valid output columns
  int f;        // SwiGLU width (GATE_UP, DGRAD_H)
  void *out2;       // GATE_UP: GU saved (null when not training)
  const void *aux;  // DGRAD_H: GU
  int64_t ld_aux;
  int *status;
  unsigned long long wait_ns;  // limit of every pipeline wait
  int withhold_kblock;         // failure test only: the producer's k-block whose loads
                               // are withheld (its stage never fills); -1 otherwise
};

// One CTA's share of a (pair-)tile: its 128 rows start at m0; valid is false when a
// pair-tile's second 128-row block lies past the expert's segment (its rows then
// feed the MMA but nothing is stored).
struct Tile {
  int e, m0, n0, kt, kr0;
  int n;      // accumulator columns (the MMA's N): BN, or BN / split in a split last wave
  int klast;  // 16-wide K slices of the last stage that hold data (at most 4 * kSub)
  bool valid;
};

template <int KIND, bool PAIR>
__device__ __forceinline__ int total_tiles(const Args &a) {
  if (KIND == WGRAD) return a.E * a.m_tiles * a.n_tiles;
  if (PAIR) return a.pair_start[a.E] * a.n_tiles;
  return (a.padded[a.E] / BM) * a.n_tiles;
}

// The last wave of a pair launch of DGRAD_H: when the tiles do not fill the final
// round of the persistent loop, the tiles of that round (from `first` on) are cut into
// `split` narrower tiles along N (the MMA's N = BN / split; each CTA of the pair takes
// N / 2 of its K-major B rows), so the round runs on more pairs. Measured on GB300 at
// gpt_oss_20b: dgrad_h 269 -> 263 us; the same split left down and dgrad_x unchanged
// (a narrow tile still pays the full per-stage barrier cost), so it is not used there.
struct Tail {
  int first;  // tiles before the split round
  int split;  // 1, 2 or 4
};

template <int KIND, bool PAIR>
__device__ __forceinline__ Tail tail_split(int total, int pairs) {
  Tail tl{total, 1};
  if (!PAIR || KIND != DGRAD_H) return tl;
  const int rem = total % pairs;
  if (rem == 0) return tl;
  tl.split = 4 * rem <= pairs ? 4 : (2 * rem <= pairs ? 2 : 1);
  tl.first = total - rem;
  return tl;
}

template <int KIND, bool PAIR>
__device__ __forceinline__ Tile decode_tile(const Args &a, int tile, int rank);

template <int KIND, bool PAIR>
__device__ __forceinline__ Tile decode(const Args &a, const Tail &tl, int tile, int rank) {
  if (tile < tl.first || tl.split == 1) return decode_tile<KIND, PAIR>(a, tile, rank);
  const int sub = tile - tl.first;
  Tile t = decode_tile<KIND, PAIR>(a, tl.first + sub / tl.split, rank);
  t.n = BN / tl.split;
  t.n0 += (sub % tl.split) * t.n;
  return t;
}

template <int KIND, bool PAIR>
__device__ __forceinline__ Tile decode_tile(const Args &a, int tile, int rank) {
  constexpr int kMTile = Cfg<PAIR>::kMTile;
  Tile t;
  t.valid = true;
  t.n = BN;
  t.klast = Cfg<PAIR>::kBKS / 16;
  if (KIND == WGRAD) {
    // Long experts (more rows than kWeightStationaryMaxRows): (expert, n-tile, m-tile)
    // with the m-tile fastest, so a round of the persistent CTAs covers every m-tile of a
    // few n-tiles and each n panel of the expert (dGU for dW_gu, G for dW_down: K rows x
    // N columns) is fetched from DRAM fewer times, the m panels being re-read from round
    // to round. Measured on GB300 at 8192 rows per expert: dW_gu 1.6-3.5% faster, its DRAM
    // reads 19.9 -> 17.6 GB on one GPU. Short experts keep the n-tile fastest (at 512 rows
    // the m-fastest order was 3% slower).
    const int per = a.m_tiles * a.n_tiles;
    t.e = tile / per;
    const int r = tile - t.e * per;
    const bool m_fast = !a.weight_stationary;
    const int fast = m_fast ? a.m_tiles : a.n_tiles;  // one division either way
    const int slow_i = r / fast, fast_i = r - slow_i * fast;
    t.m0 = (m_fast ? fast_i : slow_i) * kMTile + rank * BM;
    t.n0 = (m_fast ? slow_i : fast_i) * BN;
    t.kr0 = a.padded[t.e];
    constexpr int kBKS = Cfg<PAIR>::kBKS;
    t.kt = (a.counts[t.e] + kBKS - 1) / kBKS;  // stages holding the expert's rows
    // the last stage's rows past the count are zero padding or other experts' rows:
    // its MMAs stop at the last 16-row slice that holds a row of this expert
    t.klast = (a.counts[t.e] - (t.kt - 1) * kBKS + 15) / 16;
    return t;
  }
  // ragged M: "units" are 128-row tiles (single) or pairs of them (pair mode);
  // unit_start[e] / unit_expert[u] locate them.
  int u, nt;
  if (!a.weight_stationary) {
    // unit major: consecutive tiles share the activation rows
    u = tile / a.n_tiles;
    nt = tile - u * a.n_tiles;
    t.e = PAIR ? a.pair_expert[u] : a.tile_expert[u];
  } else {
    // weight-stationary: within an expert, (n-tile, unit) with the unit fastest, so
    // the CTAs that read one weight tile run together. Expert e owns tiles
    // [n_tiles * start_e, n_tiles * start_(e+1)).
    t.e = PAIR ? a.pair_expert[tile / a.n_tiles] : a.tile_expert[tile / a.n_tiles];
    const int base = PAIR ? a.pair_start[t.e] : a.padded[t.e] / BM;
    const int units = (PAIR ? a.pair_start[t.e + 1] : a.padded[t.e + 1] / BM) - base;
    const int local = tile - base * a.n_tiles;
    nt = local / units;
    u = base + (local - nt * units);
  }
  int mt = u;
  if (PAIR) {
    mt = a.padded[t.e] / BM + 2 * (u - a.pair_start[t.e]) + rank;
    t.valid = mt < a.padded[t.e + 1] / BM;
  }
  t.m0 = mt * BM;
  t.n0 = nt * (KIND == GATE_UP ? BN / 2 : BN);
  t.kt = a.k_tiles;
  t.klast = a.k_last;
  t.kr0 = 0;
  return t;
}

// The loads of one k-block into this CTA's stage. Single: everything, completing on
// the local barrier. Pair: this CTA's A rows and its half of B, completing on the
// even CTA's barrier (bar_pair, a shared::cluster address).
template <int KIND, bool PAIR>
__device__ __forceinline__ void issue_loads(const CUtensorMap *tmA, const CUtensorMap *tmB,
                                            uint8_t *sA, uint8_t *sB, uint64_t *bar,
                                            uint32_t bar_pair, const Tile &t, int kb, int rank) {
  constexpr bool kPair = PAIR;
  constexpr int kBRows = Cfg<PAIR>::kBRows;
  const int k0 = kb * BK;
  auto ld2 = [&](void *dst, const CUtensorMap *m, int c0, int c1) {
    if (kPair) tma_load_2d_pair(dst, m, bar_pair, c0, c1);
    else tma_load_2d(dst, m, bar, c0, c1);
  };
  auto ld3 = [&](void *dst, const CUtensorMap *m, int c0, int c1, int c2) {
    if (kPair) tma_load_3d_pair(dst, m, bar_pair, c0, c1, c2);
    else tma_load_3d(dst, m, bar, c0, c1, c2);
  };
  auto ld4 = [&](void *dst, const CUtensorMap *m, int c0, int c1, int c2, int c3) {
    if (kPair) tma_load_4d_pair(dst, m, bar_pair, c0, c1, c2, c3);
    else tma_load_4d(dst, m, bar, c0, c1, c2, c3);
  };
  // A operand: this CTA's 128 rows
  if (KIND == WGRAD) {
    // X^T tile: columns m0..m0+127 of X, rows kr0+k0 .. +63 (MN-major)
    ld2(sA, tmA, t.m0, t.kr0 + k0);
    ld2(sA + kBoxBytes, tmA, t.m0 + 64, t.kr0 + k0);
  } else {
    ld2(sA, tmA, k0, t.m0);  // rows m0..m0+127, K columns k0..k0+63
  }
  // B operand: N columns [n_lo, n_lo + kBRows) of the tile
  if (KIND == GATE_UP) {
    // W_gu viewed as [E][d][2][f]: the tile's N = 128 gate columns then the same 128
    // up columns; a pair splits them, the even CTA loading gate and the odd one up
    if (kPair) {
#pragma unroll
      for (int i = 0; i < 2; ++i) ld4(sB + i * kBoxBytes, tmB, t.n0 + 64 * i, rank, k0, t.e);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) ld4(sB + i * kBoxBytes, tmB, t.n0 + 64 * (i & 1), i >> 1, k0, t.e);
    }
  } else if (KIND == DOWN) {
    // a pair's MMA takes N / 2 B columns from each CTA (N = t.n)
    const int n_lo = t.n0 + rank * (kPair ? t.n / 2 : 0);
#pragma unroll
    for (int i = 0; i < kBRows / 64; ++i) ld3(sB + i * kBoxBytes, tmB, n_lo + 64 * i, k0, t.e);
  } else if (KIND == DGRAD_H || KIND == DGRAD_X) {
    // kBRows N-rows x 64 K, K-major; the MMA uses the first N / 2 of each CTA's rows
    ld3(sB, tmB, k0, t.n0 + rank * (kPair ? t.n / 2 : 0), t.e);
  } else {
    const int n_lo = t.n0 + rank * kBRows;
#pragma unroll
    for (int i = 0; i < kBRows / 64; ++i) ld2(sB + i * kBoxBytes, tmB, n_lo + 64 * i, t.kr0 + k0);
  }
}

__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// One epilogue warp's two staging buffers, used as a ring: each staged output chunk
// (32 rows x 32 columns) takes the next buffer once the bulk store that last read it
// is done, then leaves smem by one TMA store.
struct Stager {
  uint8_t *base;
  int n;
  __device__ __forceinline__ uint8_t *next(int lane) {
    uint8_t *b = base + (n & 1) * kStageOutBytes;
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
    return b;
  }
  // both buffers at once (two outputs from one pass over the accumulator)
  __device__ __forceinline__ void both(int lane) {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  }
  // lane's row (64 bytes), 16-byte chunk j (columns 8j..8j+7), 64-byte swizzle: the
  // chunk index is XORed with bits 7..8 of the offset, i.e. (row / 2) % 4
  static __device__ __forceinline__ void put(uint8_t *b, int lane, int j, const float (&v)[8]) {
    *reinterpret_cast<uint4 *>(b + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = pack8(v);
  }
  __device__ __forceinline__ void publish() {
    fence_proxy_async_shared();
    __syncwarp();
  }
};

__device__ __forceinline__ void put32(uint8_t *b, int lane, const float *x) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = x[8 * v + i];
    Stager::put(b, lane, v, o);
  }
}

// Write one 32 x 32 chunk of bf16 values (this lane's row: x[0..31]) through the next
// staging buffer and a TMA store at coordinates c (clipped at the tensor's edges).
template <int NC>
__device__ __forceinline__ void emit_chunk(Stager &st, int lane, const float *x,
                                           const CUtensorMap *tm, const int (&c)[NC]) {
  uint8_t *b = st.next(lane);
  put32(b, lane, x);
  st.publish();
  if (lane == 0) {
    if (NC == 2) tma_store_2d(tm, b, c[0], c[1]);
    else tma_store_3d(tm, b, c[0], c[1], c[NC - 1]);
    bulk_commit();
  }
  ++st.n;
}

// Hand the accumulator buffer back to the MMA issuer (once this warp's TMEM reads are
// complete).
__device__ __forceinline__ void release_acc(int lane, uint64_t *bar_local, uint32_t bar_pair,
                                            bool pair) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if (pair) mbar_arrive_cluster(bar_pair);
    else mbar_arrive(bar_local);
  }
}

// Epilogue of one tile for one warp: TMEM lanes of quarter q (rows m0+32q ..), the
// accumulator columns of half ch of the tile. Except for DGRAD_H, the warp reads all
// its accumulator columns into registers first and releases the accumulator (rel_*)
// before it converts and stores, so the next tile's MMAs need not wait for the stores.
// Returns whether it released the accumulator.
template <int KIND>
__device__ __forceinline__ bool epilogue_tile(const Args &a, const Tile &t, uint32_t taddr,
                                              bool last_half,
                                              int q, int ch, int lane, Stager &st,
                                              const CUtensorMap *tmO, const CUtensorMap *tmO2,
                                              uint64_t *rel_local, uint32_t rel_pair,
                                              bool pair) {
  const int row0 = t.m0 + 32 * q;  // first row of this warp's 32-row slab
  if (KIND == GATE_UP) {
    // accumulator columns [0,128) gate, [128,256) up; this warp: h columns ch*64 ..+63
    float g[64], u[64];
    tmem_ld64x2(taddr + ch * 64, taddr + BN / 2 + ch * 64, g, u);
    if (last_half) release_acc(lane, rel_local, rel_pair, pair);
    if (!t.valid) return last_half;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col = t.n0 + ch * 64 + 32 * c;
      if (col < a.f) {
        if (a.out2) {  // the saved pre-activations first, then h in place over gate
          const int cg[3] = {col, 0, row0}, cu[3] = {col, 1, row0};
          emit_chunk<3>(st, lane, g + 32 * c, tmO2, cg);
          emit_chunk<3>(st, lane, u + 32 * c, tmO2, cu);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) g[32 * c + i] = silu(g[32 * c + i]) * u[32 * c + i];
        const int ch2[2] = {col, row0};
        emit_chunk<2>(st, lane, g + 32 * c, tmO, ch2);
      }
    }
    return true;
  } else if (KIND == DOWN || KIND == DGRAD_X || KIND == WGRAD) {
    float x[128];
    if (KIND == WGRAD && t.kt == 0) {
#pragma unroll
      for (int i = 0; i < 128; ++i) x[i] = 0.f;
    } else {
      tmem_ld128(taddr + ch * 128, x);
    }
    if (last_half) release_acc(lane, rel_local, rel_pair, pair);
    if (!t.valid) return last_half;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int col = t.n0 + ch * 128 + 32 * c;
      const bool ok = col < a.N_out && ch * 128 + 32 * c < t.n &&
                      (KIND != WGRAD || row0 < a.M_out);
      if (ok) {
        if (KIND == WGRAD) {
          const int cw[3] = {col, row0, t.e};
          emit_chunk<3>(st, lane, x + 32 * c, tmO, cw);
        } else {
          const int co[2] = {col, row0};
          emit_chunk<2>(st, lane, x + 32 * c, tmO, co);
        }
      }
    }
    return true;
  } else {  // DGRAD_H
    if (!t.valid) return false;
    // dH -> (dgate, dup) with the saved gate/up pre-activations of this row; the
    // gate/up values of the next 32 columns are loaded while these are computed.
    const int64_t row = row0 + lane;
    const uint16_t *gu = reinterpret_cast<const uint16_t *>(a.aux) + row * a.ld_aux;
    uint4 cg[4], cu[4], ng[4], nu[4];
    auto load = [&](int c, uint4 (&g4)[4], uint4 (&u4)[4]) {
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        if (c + 8 * v < a.f) {
          g4[v] = ldg_nc(gu + c + 8 * v);
          u4[v] = ldg_nc(gu + a.f + c + 8 * v);
        } else {
          g4[v] = make_uint4(0, 0, 0, 0);
          u4[v] = make_uint4(0, 0, 0, 0);
        }
      }
    };
    const int c_begin = ch * 128, c_end = min(ch * 128 + 128, t.n);
    if (c_begin >= c_end) return false;  // a narrow last-wave tile: no columns here
    load(t.n0 + c_begin, cg, cu);
#pragma unroll 1
    for (int c32 = c_begin; c32 < c_end; c32 += 32) {
      const int col = t.n0 + c32;
      if (col >= a.f) break;
      if (c32 + 32 < c_end) load(col + 32, ng, nu);
      float dh[32];
      tmem_ld32(taddr + c32, dh);
      st.both(lane);
      uint8_t *bg = st.base, *bu = st.base + kStageOutBytes;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        float g[8], u[8], dg[8], du[8];
        unpack8(cg[v], g);
        unpack8(cu[v], u);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float s = 1.f / (1.f + __expf(-g[i]));
          const float x = dh[8 * v + i];
          dg[i] = x * u[i] * s * (1.f + g[i] * (1.f - s));
          du[i] = x * g[i] * s;
        }
        Stager::put(bg, lane, v, dg);
        Stager::put(bu, lane, v, du);
      }
      st.publish();
      if (lane == 0) {
        tma_store_3d(tmO, bg, col, 0, row0);
        tma_store_3d(tmO, bu, col, 1, row0);
        bulk_commit();
      }
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        cg[v] = ng[v];
        cu[v] = nu[v];
      }
    }
    return false;
  }
}

// Before a DGRAD_H tile's accumulator is ready: pull this thread's row of the saved
// gate/up values for the tile's columns into L2, so the epilogue's loads hit L2.
__device__ __forceinline__ void prefetch_gu_row(const Args &a, const Tile &t, int row, int ch) {
  const char *base = reinterpret_cast<const char *>(a.aux) + (int64_t)row * a.ld_aux * 2;
  const int c_end = min(t.n0 + min(ch * 128 + 128, t.n), a.f);
#pragma unroll 1
  for (int c = t.n0 + ch * 128; c < c_end; c += 64) {  // 64 bf16 = one 128-byte line
    asm volatile("prefetch.global.L2 [%0];" ::"l"(base + 2 * (int64_t)c));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(base + 2 * ((int64_t)a.f + c)));
  }
}

// Stage timing (a measurement aid, only in the diagnostic build compiled with
// MOE_STAGE_TIMING, where it costs ~2% even unarmed; the shipped build has none of it):
// CTA 0 of the armed GEMM kind stamps clock64() at each pipeline stage -- when the
// producer's wait for the free slot ended and when its loads were issued, when the MMA
// issuer's wait for the full stage ended and when its MMAs and commit were issued -- and,
// per tile, when its first epilogue warp saw the accumulator and when it released it.
#ifdef MOE_STAGE_TIMING
#define MOE_STAMP(...) __VA_ARGS__
__device__ int g_timing_kind = -1;
__device__ unsigned long long g_stage_times[kTimingStages][4];
__device__ unsigned long long g_tile_times[kTimingTiles][2];
#else
#define MOE_STAMP(...)
#endif

// Launched with a cluster of 2 when PAIR (see launch_kind).
template <int KIND, bool PAIR>
__global__ void __launch_bounds__(threads_of<KIND>(), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO,
                        const __grid_constant__ CUtensorMap tmO2, const Args a) {
  constexpr bool kPair = PAIR;
  constexpr int kStages = Cfg<PAIR>::kStages, kStageBytes = Cfg<PAIR>::kStageBytes;
  constexpr int kMTile = Cfg<PAIR>::kMTile;
  constexpr int A_MN = (KIND == WGRAD) ? 1 : 0;
  constexpr int B_MN = (KIND == DGRAD_H || KIND == DGRAD_X) ? 0 : 1;
  constexpr uint32_t kIdesc = idesc_bf16_f32(kMTile, BN, A_MN, B_MN);
  // descriptor strides: K-major SW128 tiles use SBO = 1024 (8 rows of 128 B) and step
  // 32 B per 16-element K slice; MN-major SW128 tiles use LBO = one 64x64 box (the
  // next 64 M/N columns), SBO = 1024 (8 K rows) and step 16 rows = 2048 B per K slice.
  constexpr uint32_t kALbo = A_MN ? kBoxBytes : 16, kBLbo = B_MN ? kBoxBytes : 16;
  constexpr uint32_t kAStep = A_MN ? 2048 : 32, kBStep = B_MN ? 2048 : 32;

  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar[2], acce_bar[2], drain_bar;
  __shared__ uint32_t tmem_slot;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = kPair ? (int)cluster_ctarank() : 0;     // 0 = the CTA issuing MMAs
  const int unit0 = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // this pair's first tile
  const int units = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);   // the even CTA's producer; bytes from both CTAs
      mbar_init(&empty_bar[s], 1);  // one (multicast) commit per consumed stage
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], (kPair ? 2 : 1) * epi_warps<KIND>());  // both CTAs' epilogues
    }
    mbar_init(&drain_bar, 1);
    fence_barrier_init();
    fence_proxy_async_shared();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmO);
    if (KIND == GATE_UP) tma_prefetch_desc(&tmO2);
  }
  if (warp == 1) {
    if (kPair) {
      tmem_alloc_pair(&tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  const int full = total_tiles<KIND, PAIR>(a);
  const Tail tl = tail_split<KIND, PAIR>(full, units);
  const int total = tl.first + (full - tl.first) * tl.split;
  bool failed = false;
  MOE_STAMP(const bool timing = blockIdx.x == 0 && g_timing_kind == KIND;)

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      int issued = 0;
      for (int tile = unit0; tile < total && ok; tile += units) {
        const Tile t = decode<KIND, PAIR>(a, tl, tile, rank);
        for (int kb = 0; kb < t.kt; ++kb) {
          if (!mbar_wait(&empty_bar[s], ph ^ 1, a.status, a.wait_ns)) {
            ok = false;
            break;
          }
          MOE_STAMP(const bool stamp = timing && issued < kTimingStages;
                    if (stamp) g_stage_times[issued][0] = clock64();)
          uint8_t *sA = smem + s * kStageBytes;
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[s], (kPair ? 2 : 1) * kStageBytes);
          const uint32_t bar_pair = kPair ? mapa_shared(&full_bar[s], 0) : 0;
          if (issued != a.withhold_kblock) {
#pragma unroll
            for (int j = 0; j < Cfg<PAIR>::kSub; ++j) {
              uint8_t *sj = sA + j * Cfg<PAIR>::kSubBytes;
              issue_loads<KIND, PAIR>(&tmA, &tmB, sj, sj + kABytes, &full_bar[s], bar_pair, t,
                                      kb * Cfg<PAIR>::kSub + j, rank);
            }
          }
          MOE_STAMP(if (stamp) g_stage_times[issued][1] = clock64();)
          ++issued;
          if (++s == kStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok) {
        failed = true;
        if (rank == 0) {
          // wait (bounded) for the copies in flight: the even CTA's full barriers
          // count the bytes of both CTAs
          int n = issued < kStages ? issued : kStages;
          int ss = s;
          uint32_t pp = ph;
          for (int i = 0; i < n; ++i) {
            if (--ss < 0) {
              ss = kStages - 1;
              pp ^= 1;
            }
            mbar_wait(&full_bar[ss], pp, nullptr, 100000000ull);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // -------------------------------------------------------------- MMA issuer
      int s = 0;
      uint32_t ph = 0;
      int buf = 0;
      uint32_t aph = 0;
      bool ok = true, any = false;
      MOE_STAMP(int staged = 0;)  // stages consumed (for the stage timing)
      const uint32_t smem_base = smem_u32(smem);
      for (int tile = unit0; tile < total && ok; tile += units) {
        const Tile t = decode<KIND, PAIR>(a, tl, tile, 0);
        const uint32_t idesc = t.n == BN ? kIdesc : idesc_bf16_f32(kMTile, t.n, A_MN, B_MN);
        if (!mbar_wait(&acce_bar[buf], aph ^ 1, a.status, a.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        if (t.kt == 0) {
          // nothing to accumulate (an expert without rows): release the epilogues
          mbar_arrive(&accf_bar[buf]);
          if (kPair) mbar_arrive_cluster(mapa_shared(&accf_bar[buf], 1));
        } else {
          for (int kb = 0; kb < t.kt; ++kb) {
            if (!mbar_wait(&full_bar[s], ph, a.status, a.wait_ns)) {
              ok = false;
              break;
            }
            MOE_STAMP(const bool stamp = timing && staged < kTimingStages;
                      if (stamp) g_stage_times[staged][2] = clock64();)
            tc_fence_after();
            const int nk = (kb == t.kt - 1) ? t.klast : Cfg<PAIR>::kBKS / 16;
#pragma unroll
            for (int j = 0; j < Cfg<PAIR>::kSub; ++j) {
              const uint32_t a_addr = smem_base + s * kStageBytes + j * Cfg<PAIR>::kSubBytes;
              const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                if (j * (BK / 16) + kk < nk) {
                  const uint64_t ad = smem_desc_sw128(a_addr + kk * kAStep, kALbo, 1024);
                  const uint64_t bd = smem_desc_sw128(b_addr + kk * kBStep, kBLbo, 1024);
                  const uint32_t acc = (kb | j | kk) != 0;
                  if (kPair) tc_mma_bf16_pair(d_tmem, ad, bd, idesc, acc);
                  else tc_mma_bf16(d_tmem, ad, bd, idesc, acc);
                }
              }
            }
            any = true;
            if (kPair) tc_commit_pair(&empty_bar[s]);
            else tc_commit(&empty_bar[s]);
            MOE_STAMP(if (stamp) g_stage_times[staged][3] = clock64(); ++staged;)
            if (++s == kStages) {
              s = 0;
              ph ^= 1;
            }
          }
          if (!ok) break;
          if (kPair) tc_commit_pair(&accf_bar[buf]);
          else tc_commit(&accf_bar[buf]);
        }
        buf ^= 1;
        if (buf == 0) aph ^= 1;
      }
      if (!ok) {
        failed = true;
        if (any) {
          // let every issued MMA finish before the accumulator is freed
          if (kPair) tc_commit_pair(&drain_bar);
          else tc_commit(&drain_bar);
          mbar_wait(&drain_bar, 0, nullptr, 100000000ull);
        }
      }
    }
  } else {
    // --------------------------------------------------------------- epilogue
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    // which half of the tile's columns it handles (-1: both, one after the other)
    const int ch_own = epi_warps<KIND>() == 8 ? (warp - 2) >> 2 : -1;
    Stager st{smem + kStages * kStageBytes + (warp - 2) * 2 * kStageOutBytes, 0};
    const uint32_t acce_pair0 = kPair ? mapa_shared(&acce_bar[0], 0) : 0;
    const uint32_t acce_pair1 = kPair ? mapa_shared(&acce_bar[1], 0) : 0;
    int buf = 0;
    uint32_t aph = 0;
    for (int tile = unit0; tile < total; tile += units) {
      const Tile t = decode<KIND, PAIR>(a, tl, tile, rank);
      if (KIND == DGRAD_H && t.valid) prefetch_gu_row(a, t, t.m0 + 32 * q + lane, ch_own);
      bool ok = mbar_wait(&accf_bar[buf], aph, a.status, a.wait_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        failed = true;
        break;
      }
      tc_fence_after();
      MOE_STAMP(const int tile_no = (tile - unit0) / units;
                const bool stamp = timing && warp == 2 && lane == 0 && tile_no < kTimingTiles;
                if (stamp) g_tile_times[tile_no][0] = clock64();)
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN;
      bool released = false;
      for (int ch = ch_own < 0 ? 0 : ch_own; ch < (ch_own < 0 ? 2 : ch_own + 1); ++ch)
        released = epilogue_tile<KIND>(a, t, taddr, ch_own >= 0 || ch == 1, q, ch, lane, st,
                                       &tmO, &tmO2, &acce_bar[buf],
                                       buf ? acce_pair1 : acce_pair0, kPair);
      if (!released) release_acc(lane, &acce_bar[buf], buf ? acce_pair1 : acce_pair0, kPair);
      MOE_STAMP(if (stamp) g_tile_times[tile_no][1] = clock64();)
      buf ^= 1;
      if (buf == 0) aph ^= 1;
    }
    if (lane == 0) bulk_wait_all();  // the staged stores have left smem and landed
  }

  __syncwarp();
  if (__syncthreads_or(failed)) {
    // a wait gave up: give copies that may still target this CTA's smem time to land
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < 200000ull) __nanosleep(1000);
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();  // no signal or MMA of the pair still targets this CTA
  if (warp == 1) {
    tc_fence_after();
    if (kPair) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

template <int KIND, bool PAIR>
cudaError_t launch_kind_as(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmO,
                           const CUtensorMap &tmO2, const Args &a, int64_t max_tiles,
                           const char *name, cudaStream_t st) {
  static bool attr_set[64] = {};  // per device
  static int slots_cache[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  auto kernel = grouped_gemm_kernel<KIND, PAIR>;
  if (!attr_set[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes<PAIR>());
    if (e != cudaSuccess) return e;
    attr_set[dev & 63] = true;
  }
  if (max_tiles <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = PAIR ? 2 : 1;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.blockDim = dim3(threads_of<KIND>(), 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<PAIR>();
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  // persistent: as many CTAs (or CTA pairs) as can be resident at once, never more
  // than there are tiles
  int &slots = slots_cache[dev & 63];
  if (slots == 0) {
    slots = num_sms();
    if (PAIR) {
      cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
      int clusters = 0;
      const cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
      if (e != cudaSuccess) return e;
      if (clusters <= 0) return cudaErrorInvalidConfiguration;
      slots = clusters;
    }
  }
  cfg.gridDim = dim3((int)(max_tiles < slots ? max_tiles : slots) * (PAIR ? 2 : 1), 1, 1);
  launch_begin(st);
  cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmO, tmO2, a);
  return note_launch(name, st);
}

inline int cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Operand maps use 64-column boxes with the 128-byte swizzle; output maps (TMA
// stores from the epilogue staging) use 32-column boxes with the 64-byte swizzle.
cudaError_t map2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                  uint32_t box_rows, int swizzle = 128) {
  const uint64_t dims[2] = {inner, rows};
  const uint64_t strides[1] = {inner * 2};
  const uint32_t box[2] = {box_inner, box_rows};
  return encode_tensor_map(m, base, 2, dims, strides, box, swizzle);
}

cudaError_t map3d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t mid, uint64_t outer,
                  uint32_t box_inner, uint32_t box_mid, int swizzle = 128) {
  const uint64_t dims[3] = {inner, mid, outer};
  const uint64_t strides[2] = {inner * 2, inner * mid * 2};
  const uint32_t box[3] = {box_inner, box_mid, 1};
  return encode_tensor_map(m, base, 3, dims, strides, box, swizzle);
}

// [outer][2][inner] viewed as 3-D with one 32-row slab of one half per box: the
// gate|up layout of GU and dGU (inner = f).
cudaError_t map_halves(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows) {
  const uint64_t dims[3] = {inner, 2, rows};
  const uint64_t strides[2] = {inner * 2, inner * 4};
  const uint32_t box[3] = {32, 1, 32};
  return encode_tensor_map(m, base, 3, dims, strides, box, 64);
}

// Upper bound of the ragged-M units (128-row tiles, or pairs of them in one expert).
int64_t max_units(const GemmPlan &p, bool pair) {
  return pair ? p.R / (2 * BM) + p.E : p.R / BM;
}

// pairs of SMs for the ragged-M GEMMs when experts are long enough (kPairMinRows)
bool pair_for_rows(const GemmPlan &p) { return p.rows_per_expert >= kPairMinRows; }

template <int KIND>
cudaError_t launch_kind(bool pair, const CUtensorMap &tmA, const CUtensorMap &tmB,
                        const CUtensorMap &tmO, const CUtensorMap &tmO2, const Args &a,
                        int64_t max_tiles, const char *name, cudaStream_t st) {
  return pair ? launch_kind_as<KIND, true>(tmA, tmB, tmO, tmO2, a, max_tiles, name, st)
              : launch_kind_as<KIND, false>(tmA, tmB, tmO, tmO2, a, max_tiles, name, st);
}

// K extent of a ragged-M GEMM: its stages (of the form's K per stage) and the 16-wide
// slices of the last one that hold columns (the MMAs past them would only add the
// TMA's zero fill).
void set_k(Args &a, int64_t K, bool pair) {
  const int bks = pair ? Cfg<true>::kBKS : Cfg<false>::kBKS;
  a.k_tiles = cdiv(K, bks);
  a.k_last = cdiv(K - (int64_t)(a.k_tiles - 1) * bks, 16);
}

Args base_args(const GemmPlan &p, int *status) {
  Args a{};
  a.padded = p.padded;
  a.counts = p.counts;
  a.tile_expert = p.tile_expert;
  a.pair_start = p.pair_start;
  a.pair_expert = p.pair_expert;
  a.E = p.E;
  a.status = status;
  a.weight_stationary = p.rows_per_expert <= kWeightStationaryMaxRows;
  a.wait_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
  a.withhold_kblock = p.withhold_kblock;
  return a;
}

}  // namespace

#ifdef MOE_STAGE_TIMING
cudaError_t stage_timing_arm(int kind) {
  void *p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_stage_times);
  if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(g_stage_times));
  if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, g_tile_times);
  if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(g_tile_times));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_timing_kind, &kind, sizeof(int));
  return e;
}

cudaError_t stage_timing_read(unsigned long long *stages, unsigned long long *tiles) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(stages, g_stage_times, sizeof(g_stage_times));
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(tiles, g_tile_times, sizeof(g_tile_times));
  return e;
}
#else
cudaError_t stage_timing_arm(int) { return cudaErrorNotSupported; }
cudaError_t stage_timing_read(unsigned long long *, unsigned long long *) {
  return cudaErrorNotSupported;
}
#endif

cudaError_t encode_tensor_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                              const uint64_t *strides_bytes, const uint32_t *box, int swizzle) {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return cudaErrorNotSupported;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i < rank - 1) gstride[i] = strides_bytes[i];
  }
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                        const_cast<void *>(base), gdim, gstride, bdim, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int num_sms() {
  static int cache[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  int &c = cache[dev & 63];
  if (c == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    c = n > 0 ? n : 1;
  }
  return c;
}

cudaError_t gemm_gate_up(const GemmPlan &p, const void *xp, const void *w_gu, void *h, void *gu,
                         int d, int f, int *status, cudaStream_t st) {
  CUtensorMap tA, tB, tO, tO2;
  cudaError_t e = map2d(&tA, xp, d, p.R, 64, BM);
  if (e != cudaSuccess) return e;
  {
    const uint64_t dims[4] = {(uint64_t)f, 2, (uint64_t)d, (uint64_t)p.E};
    const uint64_t strides[3] = {(uint64_t)f * 2, (uint64_t)f * 4, (uint64_t)d * f * 4};
    const uint32_t box[4] = {64, 1, 64, 1};
    e = encode_tensor_map(&tB, w_gu, 4, dims, strides, box, 128);
    if (e != cudaSuccess) return e;
  }
  e = map2d(&tO, h, f, p.R, 32, 32, 64);
  if (e != cudaSuccess) return e;
  e = gu ? map_halves(&tO2, gu, f, p.R) : map2d(&tO2, h, f, p.R, 32, 32, 64);
  if (e != cudaSuccess) return e;
  const bool pair = pair_for_rows(p);
  Args a = base_args(p, status);
  a.n_tiles = cdiv(f, BN / 2);
  set_k(a, d, pair);
  a.N_out = f;
  a.f = f;
  a.out2 = gu;
  return launch_kind<GATE_UP>(pair, tA, tB, tO, tO2, a, max_units(p, pair) * a.n_tiles,
                              "gemm_gate_up_swiglu", st);
}

cudaError_t gemm_down(const GemmPlan &p, const void *h, const void *w_down, void *o, int d, int f,
                      int *status, cudaStream_t st) {
  CUtensorMap tA, tB, tO;
  cudaError_t e = map2d(&tA, h, f, p.R, 64, BM);
  if (e != cudaSuccess) return e;
  e = map3d(&tB, w_down, d, f, p.E, 64, 64);
  if (e != cudaSuccess) return e;
  e = map2d(&tO, o, d, p.R, 32, 32, 64);
  if (e != cudaSuccess) return e;
  const bool pair = pair_for_rows(p);
  Args a = base_args(p, status);
  a.n_tiles = cdiv(d, BN);
  set_k(a, f, pair);
  a.N_out = d;
  return launch_kind<DOWN>(pair, tA, tB, tO, tO, a, max_units(p, pair) * a.n_tiles, "gemm_down",
                           st);
}

cudaError_t gemm_dgrad_h(const GemmPlan &p, const void *g, const void *w_down, const void *gu,
                         void *dgu, int d, int f, int *status, cudaStream_t st) {
  CUtensorMap tA, tB, tO;
  const bool pair = pair_for_rows(p);
  cudaError_t e = map2d(&tA, g, d, p.R, 64, BM);
  if (e != cudaSuccess) return e;
  // [E][f][d]: K = d inner, N = f rows; each CTA of a pair loads half the N rows
  e = map3d(&tB, w_down, d, f, p.E, 64, pair ? BN / 2 : BN);
  if (e != cudaSuccess) return e;
  e = map_halves(&tO, dgu, f, p.R);
  if (e != cudaSuccess) return e;
  Args a = base_args(p, status);
  a.n_tiles = cdiv(f, BN);
  set_k(a, d, pair);
  a.N_out = f;
  a.f = f;
  a.aux = gu;
  a.ld_aux = 2 * (int64_t)f;
  return launch_kind<DGRAD_H>(pair, tA, tB, tO, tO, a, max_units(p, pair) * a.n_tiles,
                              "gemm_dgrad_h_swiglu_bwd", st);
}

cudaError_t gemm_dgrad_x(const GemmPlan &p, const void *dgu, const void *w_gu, void *dxp, int d,
                         int f, int *status, cudaStream_t st) {
  CUtensorMap tA, tB, tO;
  const bool pair = pair_for_rows(p);
  cudaError_t e = map2d(&tA, dgu, 2 * (uint64_t)f, p.R, 64, BM);
  if (e != cudaSuccess) return e;
  // [E][d][2f]: K = 2f inner, N = d rows; each CTA of a pair loads half the N rows
  e = map3d(&tB, w_gu, 2 * (uint64_t)f, d, p.E, 64, pair ? BN / 2 : BN);
  if (e != cudaSuccess) return e;
  e = map2d(&tO, dxp, d, p.R, 32, 32, 64);
  if (e != cudaSuccess) return e;
  Args a = base_args(p, status);
  a.n_tiles = cdiv(d, BN);
  set_k(a, 2 * (int64_t)f, pair);
  a.N_out = d;
  return launch_kind<DGRAD_X>(pair, tA, tB, tO, tO, a, max_units(p, pair) * a.n_tiles,
                              "gemm_dgrad_x", st);
}

cudaError_t gemm_wgrad(const GemmPlan &p, const void *x, const void *y, void *dw, int M, int N,
                       int *status, const char *name, cudaStream_t st) {
  CUtensorMap tA, tB, tO;
  cudaError_t e = map2d(&tA, x, M, p.R, 64, 64);
  if (e != cudaSuccess) return e;
  e = map2d(&tB, y, N, p.R, 64, 64);
  if (e != cudaSuccess) return e;
  e = map3d(&tO, dw, N, M, p.E, 32, 32, 64);
  if (e != cudaSuccess) return e;
  Args a = base_args(p, status);
  const bool pair = true;  // measured faster on pairs at 512 and 8192 rows per expert
  a.m_tiles = cdiv(M, pair ? 2 * BM : BM);
  a.n_tiles = cdiv(N, BN);
  a.M_out = M;
  a.N_out = N;
  return launch_kind<WGRAD>(pair, tA, tB, tO, tO, a, (int64_t)p.E * a.m_tiles * a.n_tiles, name,
                            st);
}

}  // namespace moe
