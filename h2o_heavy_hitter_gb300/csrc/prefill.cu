// Prefill attention of the H2O policy on the 5th-generation tensor cores:
// causal softmax attention of a prompt and the column sums of its probability
// matrix, the prompt tokens' accumulated scores (H2O: Heavy-Hitter Oracle ...,
// summary page, section 3.2 and appendix A, Pseudocode).
//
// Two passes over the causal (query, key) tile pairs, 128 x 128 tiles:
//   forward: one item per (row, query tile). S = Q K^T in TMEM (tcgen05.mma, bf16
//            operands staged by TMA with 128-byte swizzle), online softmax in
//            registers (one thread per query row, base-2 logits), P written
//            back to TMEM as bf16 (its own double buffer, never aliased with
//            S) and O += P V issued with P as the TMEM operand. The running
//            max is only raised when it grows by more than 2^8, so O is rarely
//            rescaled. Writes O (fp32) and the base-2 log-sum-exp of every
//            query row.
//   colsum:  one item per (row, key tile). S^T = K Q^T in TMEM (one thread per
//            key row), P = 2^(s - lse2) with the finished row statistics, and
//            each thread sums its key's probabilities over all later queries.
// The column sums need every row's final normaliser, so the second pass
// recomputes QK^T (1.5x the algorithmic flops) rather than storing T^2 values.
//
// Both kernels are persistent (one CTA per SM walking a longest-first item
// list). Warp roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM
// and issues the MMAs, warps 2-5 (one per TMEM lane quadrant) do the softmax.
// Every mbarrier wait is bounded; a wait that gives up sets the device error
// word and the CTA unwinds, always freeing its Tensor Memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "h2o.h"
#include "kernels.h"
#include "tc.cuh"

namespace h2o {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 320;        // 10 warps: TMA, MMA, 8 softmax
constexpr int kSoftmaxThreads = 256;
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16

template <int D>
struct FwdCfg {
  static constexpr int KST = D == 128 ? 3 : 4;  // K tiles in flight
  static constexpr int VST = D == 128 ? 2 : 3;  // V tiles in flight
  static constexpr int TILE = BM * D * 2;
  static constexpr uint32_t S_COL = 0;    // two S buffers: columns [0, 128) and [128, 256)
  static constexpr uint32_t O_COL = 256;  // O: columns [256, 256 + D)
  static constexpr uint32_t P_COL = 384;  // two bf16 P buffers: columns [384, 448) and [448, 512)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr size_t SMEM = static_cast<size_t>(1 + KST + VST) * TILE + 1024 + 4096;
};

struct FwdBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4];
  uint64_t v_full[4], v_empty[4];
  uint64_t s_full[2], p_ready[2];
  uint64_t o_done;  // one phase per PV (waited only by the rare O rescale)
  uint64_t o_last;  // one phase per item: its last PV has completed
  uint64_t o_free;  // one phase per item: the epilogue has read O out of TMEM
  uint64_t xbar[4];  // per lane quadrant, one phase per tile: both halves' maxima posted
  uint64_t ebar[4];  // per lane quadrant, one phase per item: both halves' sums posted
  float xmax[2][2][128];  // [tile parity][half][row]
  float xsum[2][128];     // [half][row]
  uint32_t tmem;
};

static_assert(sizeof(FwdBars) <= 4096, "FwdBars must fit the space reserved in FwdCfg::SMEM");

struct FwdParams {
  float* O;
  float* lse2;
  int rows, T, Tp, nqt, items;
  int rb;  // rows per L2 block of the item order
  float qscale;
  int32_t* err;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D>
__device__ __forceinline__ void load_tile(void* dst, const CUtensorMap* map, int tile, int row,
                                          uint64_t* bar) {
#pragma unroll
  for (int b = 0; b < D / 64; ++b)
    tma_load_3d(static_cast<uint8_t*>(dst) + b * kBoxBytes, map, b * 64, tile * 128, row, bar);
}

// Wait used by the softmax warps: the result is made warp-uniform, so a wait
// that gives up in one lane never leaves the warp to run a warp-collective
// tcgen05.ld / st divergently.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* err) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, err));
}

// Item order shared by both kernels. Rows are taken in blocks of `rb` rows
// whose K/V (forward) or Q (column sums) fit comfortably in L2, so the several
// tiles of a row that read the same operand tiles run close together in time;
// inside a block, items with more tiles come first. Returns the row and the
// tile rank (0 = the item with the most tiles).
__device__ __forceinline__ void item_coords(int it, int rows, int nqt, int rb, int& row,
                                            int& rank) {
  const int per_block = rb * nqt;
  const int b = it / per_block;
  const int r0 = b * rb;
  const int nb = min(rb, rows - r0);
  const int w = it - b * per_block;
  rank = w / nb;
  row = r0 + w % nb;
}

// K-major operand (rows x D, D contiguous): k-step kk covers columns [16kk, 16kk + 16).
template <int D>
__device__ __forceinline__ uint64_t desc_kmajor(const uint8_t* tile, int kk) {
  return smem_desc(tile + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024);
}

// Persistent: CTA b takes work items b, b + grid, ... of a list ordered by
// decreasing work (query tile nqt-1 of every row first). Barrier phases run on
// per-CTA counters that every role advances identically: g = K/V tiles so far,
// j = items so far.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::TILE;
  uint8_t* sV = smem + (1 + C::KST) * C::TILE;
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + (1 + C::KST + C::VST) * C::TILE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < C::KST; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < C::VST; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_ready[i], kSoftmaxThreads);
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->o_last, 1);
    mbar_init(&bars->o_free, kSoftmaxThreads);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars->xbar[i], 2);
      mbar_init(&bars->ebar[i], 2);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tq);
    tma_prefetch_map(&tk);
    tma_prefetch_map(&tv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      int j = 0;
      for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x, ++j) {
        int row, rank;
        item_coords(it, p.rows, p.nqt, p.rb, row, rank);
        const int qt = p.nqt - 1 - rank;
        if (j > 0 && !mbar_wait(&bars->q_empty, (j - 1) & 1, p.err)) break;  // last QK^T done
        mbar_arrive_expect_tx(&bars->q_full, C::TILE);
        load_tile<D>(sQ, &tq, qt, row, &bars->q_full);
        for (int kt = 0; kt <= qt; ++kt, ++g) {
          const int ks = g % C::KST, vs = g % C::VST;
          if (g >= C::KST && !mbar_wait(&bars->k_empty[ks], ((g / C::KST) - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->k_full[ks], C::TILE);
          load_tile<D>(sK + ks * C::TILE, &tk, kt, row, &bars->k_full[ks]);
          if (g >= C::VST && !mbar_wait(&bars->v_empty[vs], ((g / C::VST) - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->v_full[vs], C::TILE);
          load_tile<D>(sV + vs * C::TILE, &tv, kt, row, &bars->v_full[vs]);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, 0, 1);
      uint32_t g = 0;
      bool ok = true;
      int j = 0;
      for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x, ++j) {
        int row, rank;
        item_coords(it, p.rows, p.nqt, p.rb, row, rank);
        const int nkt = p.nqt - rank;
        if (!mbar_wait(&bars->q_full, j & 1, p.err)) break;
        for (int kt = 0; kt <= nkt; ++kt) {
          if (kt < nkt) {
            const uint32_t gk = g + kt;
            const int ks = gk % C::KST, sb = gk & 1;
            if (!mbar_wait(&bars->k_full[ks], (gk / C::KST) & 1, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint8_t* k_tile = sK + ks * C::TILE;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              umma_ss(tmem + C::S_COL + sb * 128, desc_kmajor<D>(sQ, kk), desc_kmajor<D>(k_tile, kk),
                      idesc_qk, kk > 0);
            umma_commit(&bars->s_full[sb]);
            umma_commit(&bars->k_empty[ks]);
            if (kt == nkt - 1) umma_commit(&bars->q_empty);
          }
          if (kt >= 1) {
            const uint32_t gp = g + kt - 1;
            const int pb = gp & 1, vs = gp % C::VST;
            if (!mbar_wait(&bars->p_ready[pb], (gp >> 1) & 1, p.err) ||
                !mbar_wait(&bars->v_full[vs], (gp / C::VST) & 1, p.err) ||
                (kt == 1 && j > 0 && !mbar_wait(&bars->o_free, (j - 1) & 1, p.err))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint8_t* v_tile = sV + vs * C::TILE;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              // B = V tile, MN-major: 16 keys = two 8-row swizzle atoms (2048 B);
              // the two 64-column halves of d sit one TMA box (16 KB) apart.
              const uint64_t bdesc = smem_desc(v_tile + kk * 2048, kBoxBytes, 1024);
              umma_ts(tmem + C::O_COL, tmem + C::P_COL + pb * 64 + kk * 8, bdesc, idesc_pv,
                      (kt > 1 || kk > 0) ? 1u : 0u);
            }
            umma_commit(&bars->v_empty[vs]);
            umma_commit(&bars->o_done);
            if (kt == nkt) umma_commit(&bars->o_last);
          }
        }
        g += nkt;
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax
    // Two warps per TMEM lane quadrant, one per half of the 128 S columns; a
    // thread owns one query row's half. The halves share the row's running max
    // (tile maxima exchanged through shared memory every tile) and add their
    // row sums at the end of the item.
    const int sw = warp - 2;
    const int quad = warp & 3, half = sw >> 2;
    const int r = quad * 32 + lane;
    const int cb = half * 64;  // first S column of this half
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t g = 0;
    bool ok = true;
    int j = 0;
    for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x, ++j) {
      int row, rank;
      item_coords(it, p.rows, p.nqt, p.rb, row, rank);
      const int qt = p.nqt - 1 - rank;
      const int nkt = qt + 1, qrow = qt * BM + r;
      float m = -INFINITY, l = 0.f;
      for (int kt = 0; kt < nkt; ++kt) {
        const uint32_t gs = g + kt;
        const int sb = gs & 1;
        if (!warp_wait(&bars->s_full[sb], (gs >> 1) & 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[64];
        tmem_ld32(tmem + lane_off + C::S_COL + sb * 128 + cb, s);
        tmem_ld32(tmem + lane_off + C::S_COL + sb * 128 + cb + 32, s + 32);
        tmem_wait_ld();
        if (kt == qt) {  // diagonal tile: key c is visible to query r iff c <= r
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (cb + c > r) s[c] = __float_as_uint(-INFINITY);
        }
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = __uint_as_float(s[e]);
#pragma unroll
        for (int c = 8; c < 64; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], __uint_as_float(s[c]));
        float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                         fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        // exchange the half maxima of this row with the partner warp
        bars->xmax[gs & 1][half][r] = mx;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->xbar[quad]);
        if (!warp_wait(&bars->xbar[quad], gs & 1, p.err)) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, bars->xmax[gs & 1][half ^ 1][r]) * p.qscale;
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m + 8.f) {
          alpha = ex2(m - mx);
          rescale = kt > 0;
          m = mx;
        }
        float rs8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) rs8[e] = 0.f;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2(fmaf(__uint_as_float(s[cc * 32 + 2 * e]), p.qscale, -m));
            const float p1 = ex2(fmaf(__uint_as_float(s[cc * 32 + 2 * e + 1]), p.qscale, -m));
            rs8[e & 7] += p0 + p1;
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tmem + lane_off + C::P_COL + sb * 64 + half * 32 + cc * 16, pk);
        }
        const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        l = fmaf(l, alpha, rs);
        // tcgen05.ld / st are warp-collective: the whole warp rescales its O rows
        // when any of its rows raised the max (the others multiply by alpha = 1).
        if (__any_sync(0xffffffffu, rescale)) {
          if (!warp_wait(&bars->o_done, (gs - 1) & 1, p.err)) {  // PV of the previous tile done
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t o[32];
            const uint32_t oc = tmem + lane_off + C::O_COL + half * (D / 2) + c * 32;
            tmem_ld32(oc, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(oc, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_ready[sb]);
      }
      // o_done cannot be used here: when the softmax of the last tile ends, the
      // PV of the tile before may still run, and a parity wait two phases back
      // would return at once. o_last completes exactly once per item.
      if (!ok || !warp_wait(&bars->o_last, j & 1, p.err)) break;
      tc_fence_after();
      uint32_t o[D / 2];
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tmem_ld32(tmem + lane_off + C::O_COL + half * (D / 2) + c * 32, o + c * 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->o_free);  // O may be overwritten by the next item
      // the row's sum is the sum of both halves
      bars->xsum[half][r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ebar[quad]);
      if (!warp_wait(&bars->ebar[quad], j & 1, p.err)) break;
      l += bars->xsum[half ^ 1][r];
      if (qrow < p.T) {
        const float inv = 1.f / l;
        float* orow = p.O + (static_cast<size_t>(row) * p.T + qrow) * D + half * (D / 2);
#pragma unroll
        for (int e = 0; e < D / 2; e += 4)
          *reinterpret_cast<float4*>(orow + e) =
              make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                          __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
        if (half == 0) p.lse2[static_cast<size_t>(row) * p.Tp + qrow] = m + log2f(l);
      }
      g += nkt;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ column sums
template <int D>
struct ColCfg {
  static constexpr int QST = D == 128 ? 4 : 6;  // query tiles in flight
  static constexpr int TILE = BM * D * 2;
  static constexpr uint32_t TMEM_COLS = 256;   // two S^T buffers
  static constexpr size_t SMEM =
      static_cast<size_t>(1 + QST) * TILE + QST * BM * sizeof(float) + 1024 + 2048;
};

struct ColBars {
  uint64_t k_full, k_empty;
  uint64_t q_full[8], q_empty[8];
  uint64_t s_full[2], s_free[2];
  uint64_t ebar[4];     // per lane quadrant, one phase per item: both halves' sums posted
  float xsum[2][128];   // [half][key row]
  uint32_t tmem;
};

static_assert(sizeof(ColBars) <= 2048, "ColBars must fit the space reserved in ColCfg::SMEM");

struct ColParams {
  const float* lse2;
  float* colsum;
  int rows, T, Tp, nqt, items;
  int rb;  // rows per L2 block of the item order
  float qscale;
  int32_t* err;
};

// Persistent like the forward kernel; items are (row, key tile), key tile 0
// (the most query tiles) first. g counts query tiles so far, j items so far.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_colsum_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const ColParams p) {
  using C = ColCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sK = smem;
  uint8_t* sQ = smem + C::TILE;
  float* sL = reinterpret_cast<float*>(smem + (1 + C::QST) * C::TILE);
  ColBars* bars = reinterpret_cast<ColBars*>(smem + (1 + C::QST) * C::TILE + C::QST * BM * 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->k_full, 1);
    mbar_init(&bars->k_empty, 1);
    for (int i = 0; i < C::QST; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1 + 8);  // MMA commit + one arrival per softmax warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 8);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&bars->ebar[i], 2);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tq);
    tma_prefetch_map(&tk);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      int j = 0;
      for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x, ++j) {
        int row, kt;
        item_coords(it, p.rows, p.nqt, p.rb, row, kt);
        const int nq = p.nqt - kt;
        if (j > 0 && !mbar_wait(&bars->k_empty, (j - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&bars->k_full, C::TILE);
        load_tile<D>(sK, &tk, kt, row, &bars->k_full);
        for (int i = 0; i < nq; ++i, ++g) {
          const int st = g % C::QST, qt = kt + i;
          if (g >= C::QST && !mbar_wait(&bars->q_empty[st], ((g / C::QST) - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->q_full[st], C::TILE + BM * 4);
          load_tile<D>(sQ + st * C::TILE, &tq, qt, row, &bars->q_full[st]);
          bulk_copy_g2s(sL + st * BM, p.lse2 + static_cast<size_t>(row) * p.Tp + qt * BM, BM * 4,
                        &bars->q_full[st]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BN, BM, 0, 0);  // M = keys, N = queries
      uint32_t g = 0;
      bool ok = true;
      int j = 0;
      for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x, ++j) {
        int row, kt;
        item_coords(it, p.rows, p.nqt, p.rb, row, kt);
        const int nq = p.nqt - kt;
        if (!mbar_wait(&bars->k_full, j & 1, p.err)) break;
        for (int i = 0; i < nq; ++i) {
          const uint32_t gq = g + i;
          const int st = gq % C::QST, sb = gq & 1;
          if (!mbar_wait(&bars->q_full[st], (gq / C::QST) & 1, p.err) ||
              (gq >= 2 && !mbar_wait(&bars->s_free[sb], ((gq >> 1) - 1) & 1, p.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* q_tile = sQ + st * C::TILE;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + sb * 128, desc_kmajor<D>(sK, kk), desc_kmajor<D>(q_tile, kk), idesc,
                    kk > 0);
          umma_commit(&bars->s_full[sb]);
          umma_commit(&bars->q_empty[st]);
        }
        umma_commit(&bars->k_empty);
        g += nq;
      }
    }
  } else {
    // Two warps per TMEM lane quadrant, one per half of the 128 query columns;
    // a thread sums its key's probabilities over its half, and the halves are
    // added once per item.
    const int sw = warp - 2;
    const int quad = warp & 3, half = sw >> 2;
    const int r = quad * 32 + lane;  // key row within the tile
    const int cb = half * 64;        // first query column of this half
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t g = 0;
    bool ok = true;
    int j = 0;
    for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x, ++j) {
      int row, kt;
      item_coords(it, p.rows, p.nqt, p.rb, row, kt);
      const int nq = p.nqt - kt;
      float acc = 0.f;
      for (int i = 0; i < nq; ++i) {
        const uint32_t gq = g + i;
        const int st = gq % C::QST, sb = gq & 1, qt = kt + i;
        if (!warp_wait(&bars->s_full[sb], (gq >> 1) & 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[64];
        tmem_ld32(tmem + lane_off + sb * 128 + cb, s);
        tmem_ld32(tmem + lane_off + sb * 128 + cb + 32, s + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[sb]);
        if (!warp_wait(&bars->q_full[st], (gq / C::QST) & 1, p.err)) {
          ok = false;
          break;
        }
        const float* L = sL + st * BM + cb;
        const int qvalid = min(BM, p.T - qt * BM) - cb;  // queries past the prompt end are padding
        // Eight independent sums; the LSE values come as float4 loads.
        float a8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) a8[e] = 0.f;
        if (i == 0 || qvalid < 64) {
          const int c0 = i == 0 ? r - cb : 0;  // diagonal tile: queries >= key r only
#pragma unroll
          for (int c4 = 0; c4 < 64; c4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(L + c4);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = c4 + e;
              const float x = ex2(fmaf(__uint_as_float(s[c]), p.qscale, -lv[e]));
              a8[c & 7] += (c >= c0 && c < qvalid) ? x : 0.f;
            }
          }
        } else {
#pragma unroll
          for (int c4 = 0; c4 < 64; c4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(L + c4);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = c4 + e;
              a8[c & 7] += ex2(fmaf(__uint_as_float(s[c]), p.qscale, -lv[e]));
            }
          }
        }
        acc += ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->q_empty[st]);
      }
      if (!ok) break;
      // add the two halves
      bars->xsum[half][r] = acc;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ebar[quad]);
      if (!warp_wait(&bars->ebar[quad], j & 1, p.err)) break;
      const int key = kt * BN + r;
      if (half == 0 && key < p.T)
        p.colsum[static_cast<size_t>(row) * p.T + key] = acc + bars->xsum[1][r];
      g += nq;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Rows per block of the item order: `tensors` bf16 [T, D] operands re-read by
// every item of a row (K and V for the forward pass, Q for the column sums)
// should total about 24 MB per block, well inside the 129 MB L2.
int rows_per_l2_block(int T, int D, int tensors) {
  const double per_row = static_cast<double>(tensors) * T * D * 2;
  const int rb = static_cast<int>(24.0e6 / per_row);
  return rb < 1 ? 1 : rb;
}

// SM count of the current device (one persistent CTA per SM).
int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// [rows, T, D] bf16, boxes of 128 tokens x 64 channels, 128-byte swizzle,
// zero fill past the prompt end.
cudaError_t make_map(CUtensorMap* m, const void* base, int rows, int T, int D) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(T) * D * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t forward_t(const void* Q, const void* K, const void* V, int rows, int T, float* O,
                      float* lse2, int32_t* err, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  cudaError_t e;
  if ((e = make_map(&mq, Q, rows, T, D)) != cudaSuccess) return e;
  if ((e = make_map(&mk, K, rows, T, D)) != cudaSuccess) return e;
  if ((e = make_map(&mv, V, rows, T, D)) != cudaSuccess) return e;
  static bool attr = false;
  if (!attr) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(FwdCfg<D>::SMEM));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int nqt = (T + BM - 1) / BM;
  FwdParams p{O, lse2, rows, T, lse_stride(T), nqt, rows * nqt, rows_per_l2_block(T, D, 2),
              kLog2e / sqrtf(float(D)), err};
  const unsigned grid = static_cast<unsigned>(std::min(p.items, num_sms()));
  attn_fwd_kernel<D><<<grid, kThreads, FwdCfg<D>::SMEM, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t colsum_t(const void* Q, const void* K, const float* lse2, int rows, int T,
                     float* colsum, int32_t* err, cudaStream_t stream) {
  CUtensorMap mq, mk;
  cudaError_t e;
  if ((e = make_map(&mq, Q, rows, T, D)) != cudaSuccess) return e;
  if ((e = make_map(&mk, K, rows, T, D)) != cudaSuccess) return e;
  static bool attr = false;
  if (!attr) {
    e = cudaFuncSetAttribute(attn_colsum_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(ColCfg<D>::SMEM));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int nqt = (T + BM - 1) / BM;
  ColParams p{lse2, colsum, rows, T, lse_stride(T), nqt, rows * nqt, rows_per_l2_block(T, D, 1),
              kLog2e / sqrtf(float(D)), err};
  const unsigned grid = static_cast<unsigned>(std::min(p.items, num_sms()));
  attn_colsum_kernel<D><<<grid, kThreads, ColCfg<D>::SMEM, stream>>>(mq, mk, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_forward(const void* Q, const void* K, const void* V, int rows, int T, int d,
                            float* O, float* lse2, int32_t* err, cudaStream_t stream) {
  if (static_cast<long>(rows) * T == 0) return cudaSuccess;
  return d == 128 ? forward_t<128>(Q, K, V, rows, T, O, lse2, err, stream)
                  : forward_t<64>(Q, K, V, rows, T, O, lse2, err, stream);
}

cudaError_t prefill_colsum(const void* Q, const void* K, const float* lse2, int rows, int T,
                           int d, float* colsum, int32_t* err, cudaStream_t stream) {
  if (static_cast<long>(rows) * T == 0) return cudaSuccess;
  return d == 128 ? colsum_t<128>(Q, K, lse2, rows, T, colsum, err, stream)
                  : colsum_t<64>(Q, K, lse2, rows, T, colsum, err, stream);
}

// ------------------------------------------------------------------ allocation-free scratch
// Per-row log-sum-exp for h2o_prefill_attention_noalloc lives in this fixed
// file-scope device array instead of an allocation. Host code must not pass
// the symbol itself to a kernel (on the host it is only a stand-in); its
// device address is looked up per device below.
static __device__ __align__(256) float g_noalloc_lse[H2O_NOALLOC_MAX_LSE];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
float* g_noalloc_ptr[kMaxDevices] = {};
}  // namespace

cudaError_t noalloc_lse_scratch(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_lse);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace h2o
