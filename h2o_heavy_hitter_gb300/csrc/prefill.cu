// Prefill attention of the H2O policy on the 5th-generation tensor cores:
// causal softmax attention of a prompt and the column sums of its probability
// matrix, the prompt tokens' accumulated scores (H2O: Heavy-Hitter Oracle ...,
// summary page, section 3.2 and appendix A, Pseudocode).
//
// Two passes over the causal (query, key) tile pairs, 128 x 128 tiles:
//   forward: one item per (row, block of two query tiles A and B). Every K/V
//            tile loaded serves both query tiles. S_t = Q_t K^T in TMEM
//            (tcgen05.mma, bf16 operands staged by TMA with 128-byte swizzle),
//            online softmax in registers (one thread per query row, base-2
//            logits), P written back as bf16 over the S columns it came from,
//            and O_t += P_t V issued with P as the TMEM operand; the softmax of
//            one tile overlaps the MMAs of the other. The running max is only
//            raised when it grows by more than 2^8, so O is rarely rescaled.
//            The softmax warps read the finished O out of TMEM, release it,
//            and write it normalised with TMA stores through small staging
//            tiles. Writes O (fp32) and the base-2 log-sum-exp of every query.
//   colsum:  one item per (row, key tile). S^T = K Q^T in TMEM (one thread per
//            key row) with the key tile held in TMEM as the A operand, so each
//            MMA reads only the query tile from shared memory; P = 2^(s - lse2)
//            with the finished row statistics, and each thread sums its key's
//            probabilities over all later queries.
// The column sums need every row's final normaliser, so the second pass
// recomputes QK^T (1.5x the algorithmic flops) rather than storing T^2 values.
//
// Both kernels are persistent (one CTA per SM walking a longest-first item
// list) and warp-specialised: TMA producer warps, one MMA warp that owns the
// TMEM, and softmax warps (one per TMEM lane quadrant and query tile in the
// forward pass, two per lane quadrant in the column sums). Every mbarrier wait
// is bounded; a wait that gives up sets the device error word and the CTA
// unwinds, always freeing its Tensor Memory.
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
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16

// ---- bulk async stores (TMA engine, shared -> global) ---------------------------
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// At most one committed store has not yet read its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Every committed store has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ forward
// An item of the forward kernel is a block of 256 query rows of one row:
// query tiles A = 2 qb and B = 2 qb + 1. Every K/V tile loaded serves both
// query tiles, which halves the K/V traffic out of L2 per flop.
// Warp roles (11 warps):
constexpr int kWarpQK = 0;        // TMA loads of Q and K
constexpr int kWarpMMA = 1;       // owns TMEM, issues every tcgen05.mma
constexpr int kWarpV = 2;         // TMA loads of V
constexpr int kWarpSoftmax0 = 3;  // warps 3..6: tile A, 7..10: tile B, one per TMEM lane quadrant
constexpr int kFwdThreads = 11 * 32;
constexpr int kTileThreads = 128;  // softmax threads of one query tile (one per query row)

template <int D>
struct FwdCfg {
  static constexpr int KST = D == 128 ? 2 : 3;  // K tiles in flight
  static constexpr int VST = D == 128 ? 2 : 3;  // V tiles in flight
  static constexpr int TILE = BM * D * 2;
  // TMEM: S of tile t at columns [128 t, 128 t + 128); the bf16 P of a tile
  // overwrites its own S (keys [16 i, 16 i + 16) at columns [8 i, 8 i + 8));
  // O of tile t at 256 + 128 t.
  static constexpr uint32_t O_COL = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int STAGE_BYTES = 32 * 16 * 4;  // one staging tile: 32 rows x 16 fp32
  static constexpr size_t TILES = static_cast<size_t>(2 + KST + VST) * TILE;
  // two staging tiles per softmax warp; barriers; slack for 1024-byte alignment
  static constexpr size_t SMEM = TILES + 8 * 2 * STAGE_BYTES + 1024 + 2048;
};

struct FwdBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4];
  uint64_t v_full[4], v_empty[4];
  uint64_t s_full[2], p_ready[2];  // per query tile, one phase per key tile
  uint64_t o_last[2];  // per query tile, one phase per item: the tile's last PV completed
  uint64_t o_free[2];  // per query tile, one phase per item: its O has been read out of TMEM
  uint32_t tmem;
};

static_assert(sizeof(FwdBars) <= 2048, "FwdBars must fit the space reserved in FwdCfg::SMEM");

struct FwdParams {
  float* lse2;
  const int32_t* lens;  // per batch entry prompt lengths (ragged batch) or null
  int heads;            // rows per batch entry (row / heads indexes lens)
  int rows, T, Tp, nqt, nqb, items;  // T padded length; nqb = blocks of two query tiles per row
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

// Wait used by warps that go on to run warp-collective tcgen05.ld / st: the
// result is made warp-uniform, so a wait that gives up in one lane never
// leaves the warp to run them divergently.
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

// Persistent: CTA b takes items b, b + grid, ... of a list ordered by
// decreasing work (the last query block of every row first). Barrier phases
// run on per-CTA counters that every role advances identically: g = K/V tiles
// so far, n[t] = key tiles processed by query tile t so far, e[t] = items in
// which tile t took part. The MMA issue order per key tile kt is
//   PV_A(kt-1), S_A(kt), PV_B(kt-1), S_B(kt),
// so the softmax of one tile overlaps the two MMAs of the other, and S_t(kt)
// (which overwrites P_t(kt-1)) follows the PV that reads it. The MMAs of one
// thread run in issue order; when the softmax sees S_t(kt) complete, every PV
// of tile t before it has completed too, so O_t can be rescaled right away.
template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                    const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;  // tile A, then tile B
  uint8_t* sK = smem + 2 * C::TILE;
  uint8_t* sV = smem + (2 + C::KST) * C::TILE;
  uint8_t* sStage = smem + C::TILES;
  FwdBars* bars = reinterpret_cast<FwdBars*>(sStage + 16 * C::STAGE_BYTES);
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
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_ready[t], kTileThreads);
      mbar_init(&bars->o_last[t], 1);
      mbar_init(&bars->o_free[t], kTileThreads / 32);
    }
    fence_barrier_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(&bars->tmem, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == kWarpQK && lane == 0) {
    tma_prefetch_map(&tq);
    tma_prefetch_map(&tk);
  }
  if (warp == kWarpV && lane == 0) tma_prefetch_map(&tv);
  if (warp == kWarpSoftmax0 && lane == 0) tma_prefetch_map(&to);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  if (warp == kWarpQK || warp == kWarpV) {
    // ---------------------------------------------------------------- TMA loads
    // Warp 0 loads the item's query tiles and its K tiles, warp 2 its V tiles,
    // so K tiles are never held back by a wait for a V stage.
    if (lane == 0) {
      const bool is_k = warp == kWarpQK;
      const int nst = is_k ? C::KST : C::VST;
      uint64_t* full = is_k ? bars->k_full : bars->v_full;
      uint64_t* empty = is_k ? bars->k_empty : bars->v_empty;
      uint8_t* ring = is_k ? sK : sV;
      const CUtensorMap* map = is_k ? &tk : &tv;
      uint32_t g = 0;
      bool ok = true;
      int j = 0;  // items processed (query loads)
      for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x) {
        int row, rank;
        item_coords(it, p.rows, p.nqb, p.rb, row, rank);
        const int nqt = (row_len(p.lens, p.heads, row, p.T) + BM - 1) / BM;
        const int qa = 2 * (p.nqb - 1 - rank);
        if (qa >= nqt) continue;  // past the end of this row's prompt
        const bool has_b = qa + 1 < nqt;
        const int nk = has_b ? qa + 2 : qa + 1;
        if (is_k) {
          if (j > 0 && !mbar_wait(&bars->q_empty, (j - 1) & 1, p.err)) break;  // last S done
          mbar_arrive_expect_tx(&bars->q_full, (has_b ? 2 : 1) * C::TILE);
          load_tile<D>(sQ, &tq, qa, row, &bars->q_full);
          if (has_b) load_tile<D>(sQ + C::TILE, &tq, qa + 1, row, &bars->q_full);
        }
        for (int kt = 0; kt < nk; ++kt, ++g) {
          const int st = g % nst;
          if (g >= static_cast<uint32_t>(nst) &&
              !mbar_wait(&empty[st], ((g / nst) - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], C::TILE);
          load_tile<D>(ring + st * C::TILE, map, kt, row, &full[st]);
        }
        ++j;
      }
    }
  } else if (warp == kWarpMMA) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, 0, 1);
      uint32_t g = 0, n0 = 0, n1 = 0, e1 = 0;
      bool ok = true;
      int j = 0;
      // Descriptors of the operand tiles are computed once; a stage or k-step
      // only adds its byte offset (>> 4) to the start-address field, so each
      // MMA costs one 64-bit add and the instruction.
      const uint64_t dq0 = desc_kmajor<D>(sQ, 0), dk0 = desc_kmajor<D>(sK, 0);
      const uint64_t dv0 = smem_desc(sV, kBoxBytes, 1024);
      auto pv = [&](int t, uint32_t gp, bool first) {
        // B = V tile, MN-major: 16 keys = two 8-row swizzle atoms (2048 B);
        // the two 64-column halves of d sit one TMA box (16 KB) apart.
        const uint64_t vb = dv0 + static_cast<uint64_t>((gp % C::VST) * (C::TILE >> 4));
        const uint32_t d_tm = tmem + C::O_COL + t * 128, a_tm = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_ts(d_tm, a_tm + kk * 8, vb + kk * (2048 >> 4), idesc_pv, (!first || kk > 0) ? 1u : 0u);
      };
      auto qk = [&](int t, uint32_t gk) {
        const uint64_t kb = dk0 + static_cast<uint64_t>((gk % C::KST) * (C::TILE >> 4));
        const uint64_t qb = dq0 + static_cast<uint64_t>(t * (C::TILE >> 4));
        const uint32_t d_tm = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
          umma_ss(d_tm, qb + off, kb + off, idesc_qk, kk > 0);
        }
      };
      for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x) {
        int row, rank;
        item_coords(it, p.rows, p.nqb, p.rb, row, rank);
        const int nqt = (row_len(p.lens, p.heads, row, p.T) + BM - 1) / BM;
        const int qa = 2 * (p.nqb - 1 - rank);
        if (qa >= nqt) continue;
        const bool has_b = qa + 1 < nqt;
        const int nk = has_b ? qa + 2 : qa + 1;
        const int last_a = qa, last_b = qa + 1;
        if (!mbar_wait(&bars->q_full, j & 1, p.err)) break;
        for (int kt = 0; ok && kt <= nk; ++kt) {
          const uint32_t gp = g + kt - 1, gk = g + kt;
          bool v_ready = false, k_ready = false;
          // ---- tile A: PV_A(kt - 1), then S_A(kt)
          if (kt >= 1 && kt - 1 <= last_a) {
            if (!mbar_wait(&bars->p_ready[0], (n0 + kt - 1) & 1, p.err) ||
                !mbar_wait(&bars->v_full[gp % C::VST], (gp / C::VST) & 1, p.err) ||
                (kt == 1 && j > 0 && !mbar_wait(&bars->o_free[0], (j - 1) & 1, p.err))) {
              ok = false;
              break;
            }
            v_ready = true;
            tc_fence_after();
            pv(0, gp, kt == 1);
            if (kt - 1 == last_a) umma_commit(&bars->o_last[0]);
            if (!has_b) umma_commit(&bars->v_empty[gp % C::VST]);
          }
          if (kt < nk && kt <= last_a) {
            if (!mbar_wait(&bars->k_full[gk % C::KST], (gk / C::KST) & 1, p.err)) {
              ok = false;
              break;
            }
            k_ready = true;
            tc_fence_after();
            qk(0, gk);
            umma_commit(&bars->s_full[0]);
            if (!has_b) {
              umma_commit(&bars->k_empty[gk % C::KST]);
              if (kt == nk - 1) umma_commit(&bars->q_empty);
            }
          }
          if (!has_b) continue;
          // ---- tile B: PV_B(kt - 1), then S_B(kt)
          if (kt >= 1) {
            if (!mbar_wait(&bars->p_ready[1], (n1 + kt - 1) & 1, p.err) ||
                (!v_ready && !mbar_wait(&bars->v_full[gp % C::VST], (gp / C::VST) & 1, p.err)) ||
                (kt == 1 && e1 > 0 && !mbar_wait(&bars->o_free[1], (e1 - 1) & 1, p.err))) {
              ok = false;
              break;
            }
            tc_fence_after();
            pv(1, gp, kt == 1);
            umma_commit(&bars->v_empty[gp % C::VST]);
            if (kt - 1 == last_b) umma_commit(&bars->o_last[1]);
          }
          if (kt < nk) {
            if (!k_ready && !mbar_wait(&bars->k_full[gk % C::KST], (gk / C::KST) & 1, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            qk(1, gk);
            umma_commit(&bars->s_full[1]);
            umma_commit(&bars->k_empty[gk % C::KST]);
            if (kt == nk - 1) umma_commit(&bars->q_empty);
          }
        }
        g += nk;
        n0 += last_a + 1;
        if (has_b) {
          n1 += last_b + 1;
          ++e1;
        }
        ++j;
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax + epilogue
    // Four warps per query tile, one per TMEM lane quadrant; a thread owns one
    // query row and all 128 keys of each S tile.
    const int sw = warp - kWarpSoftmax0;  // 0..7
    const int t = sw >> 2;                // query tile: 0 = A, 1 = B
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + t * 128;
    const uint32_t o_tm = tmem + lane_off + C::O_COL + t * 128;
    uint32_t n = 0, e = 0, rounds = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < p.items; it += gridDim.x) {
      int row, rank;
      item_coords(it, p.rows, p.nqb, p.rb, row, rank);
      const int tlen = row_len(p.lens, p.heads, row, p.T);
      const int qt = 2 * (p.nqb - 1 - rank) + t;
      if (qt * BM >= tlen) continue;  // past the prompt (tile B of a last block, or a short row)
      const int qrow = qt * BM + r;
      float m = -INFINITY, l = 0.f;
      for (int kt = 0; kt <= qt; ++kt) {
        if (!warp_wait(&bars->s_full[t], (n + kt) & 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_tm + c * 32, s + c * 32);
        tmem_wait_ld();
        if (kt == qt) {  // diagonal tile: key c is visible to query r iff c <= r
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > r) s[c] = __float_as_uint(-INFINITY);
        }
        float mx8[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) mx8[x] = fmaxf(__uint_as_float(s[x]), __uint_as_float(s[x + 8]));
#pragma unroll
        for (int c = 16; c < 128; c += 16)
#pragma unroll
          for (int x = 0; x < 8; ++x)
            mx8[x] = fmax3(mx8[x], __uint_as_float(s[c + x]), __uint_as_float(s[c + 8 + x]));
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7])) *
                         p.qscale;
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m + 8.f) {
          alpha = ex2(m - mx);
          rescale = kt > 0;
          m = mx;
        }
        // p = 2^(s * qscale - m), two keys per packed fma / add
        const uint64_t sc2 = f2_pack(p.qscale, p.qscale), nm2 = f2_pack(-m, -m);
        uint64_t rs2[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) rs2[x] = f2_pack(0.f, 0.f);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t pk[8];
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            float a, b;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[cc * 16 + 2 * x]),
                                     __uint_as_float(s[cc * 16 + 2 * x + 1])),
                             sc2, nm2),
                      a, b);
            const float p0 = ex2(a), p1 = ex2(b);
            rs2[x & 3] = f2_add(rs2[x & 3], f2_pack(p0, p1));
            pk[x] = pack_bf16x2(p0, p1);
          }
          tmem_st8(s_tm + cc * 8, pk);  // P over the S columns already read
        }
        float rsv[8];
#pragma unroll
        for (int x = 0; x < 4; ++x) f2_unpack(rs2[x], rsv[2 * x], rsv[2 * x + 1]);
        const float rs =
            ((rsv[0] + rsv[1]) + (rsv[2] + rsv[3])) + ((rsv[4] + rsv[5]) + (rsv[6] + rsv[7]));
        l = fmaf(l, alpha, rs);
        // tcgen05.ld / st are warp-collective: the whole warp rescales its O rows
        // when any of its rows raised the max (the others multiply by alpha = 1).
        // Every PV of this tile issued so far has completed (see above).
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(o_tm + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
            tmem_st32(o_tm + c * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_ready[t]);
      }
      if (!ok) break;
      // ---- epilogue: O out of TMEM (then the next item's PVs may use it),
      // normalised and written with TMA stores through two 2 KB staging tiles
      // per warp (64-byte swizzle: chunk q of row i at ((q ^ ((i >> 1) & 3)) * 16),
      // which keeps the shared-memory writes conflict free).
      if (!warp_wait(&bars->o_last[t], e & 1, p.err)) break;
      tc_fence_after();
      uint32_t o[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(o_tm + c * 32, o + c * 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free[t]);
      const float inv = 1.f / l;
      if (qrow < tlen) p.lse2[static_cast<size_t>(row) * p.Tp + qrow] = -(m + log2f(l));
      const int tok0 = qt * BM + quad * 32;  // first token of this warp's rows
#pragma unroll
      for (int c = 0; c < D / 16; ++c, ++rounds) {
        uint8_t* stg = sStage + (sw * 2 + (rounds & 1)) * C::STAGE_BYTES;
        if (lane == 0) bulk_wait_read_1();  // the store that last used this tile has read it
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<float4*>(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) = make_float4(
              __uint_as_float(o[16 * c + 4 * q]) * inv, __uint_as_float(o[16 * c + 4 * q + 1]) * inv,
              __uint_as_float(o[16 * c + 4 * q + 2]) * inv,
              __uint_as_float(o[16 * c + 4 * q + 3]) * inv);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // rows past the padded length are clipped; rows of the last box past
          // a shorter row's prompt land in its padding, which holds no result
          if (tok0 < tlen) tma_store_3d(&to, stg, c * 16, tok0, row);
          bulk_commit();
        }
      }
      n += qt + 1;
      ++e;
    }
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ column sums
constexpr int kColParts = 4;  // softmax warps per TMEM lane quadrant, each 128 / 4 query columns
constexpr int kColCols = BM / kColParts;
constexpr int kColWarps = 4 * kColParts;
constexpr int kColThreads = (2 + kColWarps) * 32;  // warps: 0 TMA, 1 MMA, the rest softmax

template <int D>
struct ColCfg {
  static constexpr int KST = 2;                 // key tiles staged in shared memory
  static constexpr int QST = D == 128 ? 4 : 8;  // query tiles in flight
  static constexpr int LST = 8;                 // LSE slices in flight
  static constexpr int TILE = BM * D * 2;
  // TMEM: S^T buffers at columns [0, 128) and [128, 256); the key tile as the
  // MMA's A operand (bf16 pairs, one key per lane) in two buffers of D/2
  // columns from column 256, by item parity.
  static constexpr uint32_t KA_COL = 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr size_t SMEM =
      static_cast<size_t>(KST + QST) * TILE + LST * BM * sizeof(float) + 1024 + 8192;
};

struct ColBars {
  uint64_t k_full[2], k_empty[2];  // key tile staged in shared memory / copied out of it
  uint64_t ka_full[2];             // key tile written into TMEM (A operand), by item parity
  uint64_t q_full[8], q_empty[8];
  uint64_t l_full[8], l_empty[8];
  uint64_t s_full[2], s_free[2];
  uint64_t ebar[4];     // per lane quadrant, one phase per item: every part's sum posted
  float xsum[2][kColParts][128];  // [item parity][part][key row]
  uint32_t tmem;
};

static_assert(sizeof(ColBars) <= 8192, "ColBars must fit the space reserved in ColCfg::SMEM");

struct ColParams {
  const float* lse2;
  float* colsum;
  const int32_t* lens;  // per batch entry prompt lengths (ragged batch) or null
  int heads;            // rows per batch entry
  int rows, T, Tp, nqt, items;  // T padded length
  int rb;  // rows per L2 block of the item order
  float qscale;
  int32_t* err;
};

// Persistent like the forward kernel; items are (row, key tile), key tile 0
// (the most query tiles) first. g counts query tiles so far, j items so far.
// The key tile of an item is the A operand of all its MMAs, so it is read out
// of shared memory once and kept in TMEM: the softmax warps copy the key tile
// of item j + 1 into TMEM when they start item j (item j - 1's MMAs, the last
// readers of that TMEM buffer, have completed by then).
template <int D>
__global__ void __launch_bounds__(kColThreads, 1)
    attn_colsum_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const ColParams p) {
  using C = ColCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sK = smem;
  uint8_t* sQ = smem + C::KST * C::TILE;
  float* sL = reinterpret_cast<float*>(smem + (C::KST + C::QST) * C::TILE);
  ColBars* bars = reinterpret_cast<ColBars*>(smem + (C::KST + C::QST) * C::TILE + C::LST * BM * 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = blockIdx.x < p.items ? (p.items - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], kColWarps);  // one arrival per softmax warp after its copy
      mbar_init(&bars->ka_full[i], kColWarps);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], kColWarps);
    }
    for (int i = 0; i < C::QST; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    for (int i = 0; i < C::LST; ++i) {
      mbar_init(&bars->l_full[i], 1);
      mbar_init(&bars->l_empty[i], kColWarps);
    }
    for (int i = 0; i < 4; ++i) mbar_init(&bars->ebar[i], kColParts);
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
    // ---------------------------------------------------------------- TMA producer
    // Key tiles run two items ahead: items 0 and 1 first, then the key tile of
    // item j + 2 once the query tiles of item j are issued.
    if (lane == 0) {
      auto load_k = [&](int n) -> bool {
        int row, kt;
        item_coords(blockIdx.x + n * gridDim.x, p.rows, p.nqt, p.rb, row, kt);
        const int ks = n & 1;
        if (n >= 2 && !mbar_wait(&bars->k_empty[ks], ((n >> 1) - 1) & 1, p.err)) return false;
        mbar_arrive_expect_tx(&bars->k_full[ks], C::TILE);
        load_tile<D>(sK + ks * C::TILE, &tk, kt, row, &bars->k_full[ks]);
        return true;
      };
      bool ok = true;
      for (int n = 0; ok && n < min(2, n_items); ++n) ok = load_k(n);
      uint32_t g = 0;
      for (int j = 0; ok && j < n_items; ++j) {
        int row, kt;
        item_coords(blockIdx.x + j * gridDim.x, p.rows, p.nqt, p.rb, row, kt);
        const int nq = max(0, (row_len(p.lens, p.heads, row, p.T) + BM - 1) / BM - kt);
        for (int i = 0; i < nq; ++i, ++g) {
          const int st = g % C::QST, ls = g % C::LST, qt = kt + i;
          if (g >= C::QST && !mbar_wait(&bars->q_empty[st], ((g / C::QST) - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->q_full[st], C::TILE);
          load_tile<D>(sQ + st * C::TILE, &tq, qt, row, &bars->q_full[st]);
          if (g >= C::LST && !mbar_wait(&bars->l_empty[ls], ((g / C::LST) - 1) & 1, p.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->l_full[ls], BM * 4);
          bulk_copy_g2s(sL + ls * BM, p.lse2 + static_cast<size_t>(row) * p.Tp + qt * BM, BM * 4,
                        &bars->l_full[ls]);
        }
        if (ok && j + 2 < n_items) ok = load_k(j + 2);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // S^T = K Q^T with K from TMEM (A) and the query tile from shared memory (B).
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BN, BM, 0, 0);  // M = keys, N = queries
      const uint64_t dq0 = desc_kmajor<D>(sQ, 0);  // query stage s adds s * TILE >> 4
      uint32_t g = 0;
      for (int j = 0; j < n_items; ++j) {
        int row, kt;
        item_coords(blockIdx.x + j * gridDim.x, p.rows, p.nqt, p.rb, row, kt);
        const int nq = max(0, (row_len(p.lens, p.heads, row, p.T) + BM - 1) / BM - kt);
        const int kb = j & 1;
        if (!mbar_wait(&bars->ka_full[kb], (j >> 1) & 1, p.err)) break;
        bool ok = true;
        for (int i = 0; i < nq; ++i) {
          const uint32_t gq = g + i;
          const int st = gq % C::QST, sb = gq & 1;
          if (!mbar_wait(&bars->q_full[st], (gq / C::QST) & 1, p.err) ||
              (gq >= 2 && !mbar_wait(&bars->s_free[sb], ((gq >> 1) - 1) & 1, p.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t qd = dq0 + static_cast<uint64_t>(st * (C::TILE >> 4));
          const uint32_t d_tm = tmem + sb * 128, a_tm = tmem + C::KA_COL + kb * (D / 2);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ts(d_tm, a_tm + kk * 8, qd + (((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4), idesc,
                    kk > 0);
          umma_commit(&bars->s_full[sb]);
          umma_commit(&bars->q_empty[st]);
        }
        if (!ok) break;
        g += nq;
      }
    }
  } else {
    // kColParts warps per TMEM lane quadrant, each on kColCols of the 128 query
    // columns; a thread sums its key's probabilities over its columns, and the
    // parts are added once per item.
    const int sw = warp - 2;
    const int quad = warp & 3, part = sw >> 2;
    const int r = quad * 32 + lane;  // key row within the tile
    const int cb = part * kColCols;  // first query column of this part
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    // Copies this thread's key row, this warp's part of the channels
    // (D / (2 kColParts) bf16 pairs), from the staged key tile into TMEM
    // buffer n & 1.
    auto copy_k = [&](int n) -> bool {
      const int ks = n & 1;
      if (!warp_wait(&bars->k_full[ks], (n >> 1) & 1, p.err)) return false;
      const uint8_t* tile = sK + ks * C::TILE;
      constexpr int CH = D / (8 * kColParts);  // 16-byte chunks of 8 channels per part
      uint32_t w[4 * CH];
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int cg = part * CH + c;
        const uint4 v = *reinterpret_cast<const uint4*>(tile + (cg >> 3) * kBoxBytes + r * 128 +
                                                        (((cg & 7) ^ (r & 7)) << 4));
        w[4 * c] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
      }
      const uint32_t dst = tmem + lane_off + C::KA_COL + (n & 1) * (D / 2) + part * (4 * CH);
      if constexpr (4 * CH == 16)
        tmem_st16(dst, w);
      else
        tmem_st8(dst, w);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->ka_full[n & 1]);
        mbar_arrive(&bars->k_empty[ks]);
      }
      return true;
    };
    uint32_t g = 0;
    bool ok = n_items == 0 || copy_k(0);
    for (int j = 0; ok && j < n_items; ++j) {
      int row, kt;
      item_coords(blockIdx.x + j * gridDim.x, p.rows, p.nqt, p.rb, row, kt);
      const int tlen = row_len(p.lens, p.heads, row, p.T);
      // items past a short row's prompt have no queries: the key tile still
      // passes through TMEM so that every barrier phase stays in step
      const int nq = max(0, (tlen + BM - 1) / BM - kt);
      if (j + 1 < n_items && !copy_k(j + 1)) break;
      float acc = 0.f;
      for (int i = 0; i < nq; ++i) {
        const uint32_t gq = g + i;
        const int ls = gq % C::LST, sb = gq & 1, qt = kt + i;
        if (!warp_wait(&bars->s_full[sb], (gq >> 1) & 1, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s[kColCols];
        tmem_ld32(tmem + lane_off + sb * 128 + cb, s);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[sb]);
        if (!warp_wait(&bars->l_full[ls], (gq / C::LST) & 1, p.err)) {
          ok = false;
          break;
        }
        const float* L = sL + ls * BM + cb;
        const int qvalid = min(BM, tlen - qt * BM) - cb;  // queries past the prompt end are padding
        // L holds -lse2 of each query: p = 2^(s * qscale - lse2), two queries per
        // packed fma / add; the LSE values come as float4 loads.
        const uint64_t sc2 = f2_pack(p.qscale, p.qscale);
        uint64_t a2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) a2[e] = f2_pack(0.f, 0.f);
        if (i == 0 || qvalid < kColCols) {
          const int c0 = i == 0 ? r - cb : 0;  // diagonal tile: queries >= key r only
#pragma unroll
          for (int c4 = 0; c4 < kColCols; c4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(L + c4);
            float x[4];
            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[c4]), __uint_as_float(s[c4 + 1])), sc2,
                             f2_pack(l4.x, l4.y)),
                      x[0], x[1]);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(s[c4 + 2]), __uint_as_float(s[c4 + 3])), sc2,
                             f2_pack(l4.z, l4.w)),
                      x[2], x[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = c4 + e;
              x[e] = (c >= c0 && c < qvalid) ? ex2(x[e]) : 0.f;
            }
            a2[(c4 >> 2) & 3] = f2_add(a2[(c4 >> 2) & 3], f2_add(f2_pack(x[0], x[1]), f2_pack(x[2], x[3])));
          }
        } else {
          float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c4 = 0; c4 < kColCols; c4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(L + c4);
            a4[0] += ex2(fmaf(__uint_as_float(s[c4]), p.qscale, l4.x));
            a4[1] += ex2(fmaf(__uint_as_float(s[c4 + 1]), p.qscale, l4.y));
            a4[2] += ex2(fmaf(__uint_as_float(s[c4 + 2]), p.qscale, l4.z));
            a4[3] += ex2(fmaf(__uint_as_float(s[c4 + 3]), p.qscale, l4.w));
          }
          a2[0] = f2_pack(a4[0], a4[1]);
          a2[1] = f2_pack(a4[2], a4[3]);
        }
        float a8[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) f2_unpack(a2[e], a8[2 * e], a8[2 * e + 1]);
        acc += ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->l_empty[ls]);
      }
      if (!ok) break;
      // add the parts
      bars->xsum[j & 1][part][r] = acc;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ebar[quad]);
      if (!warp_wait(&bars->ebar[quad], j & 1, p.err)) break;
      const int key = kt * BN + r;
      if (part == 0 && key < tlen) {
        float total = acc;
#pragma unroll
        for (int q = 1; q < kColParts; ++q) total += bars->xsum[j & 1][q][r];
        p.colsum[static_cast<size_t>(row) * p.T + key] = total;
      }
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

// Per-device state of this file (kernel attributes, looked-up symbol
// addresses) is kept for devices 0 .. kMaxDevices - 1 under one mutex.
// forget_device_state() starts a new epoch, which invalidates all of it.
constexpr int kMaxDevices = 64;
std::mutex g_device_state_mutex;
int g_device_state_epoch = 1;

// Lets `kernel` use `bytes` of dynamic shared memory on the current device.
// The attribute is per device, so it is set once per device and epoch;
// opted_in[dev] records the epoch in which it was set (guarded by the mutex,
// so concurrent first calls are safe).
template <typename Kernel>
cudaError_t raise_smem_limit(Kernel kernel, size_t bytes, int (&opted_in)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_device_state_mutex);
  if (opted_in[dev] != g_device_state_epoch) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    opted_in[dev] = g_device_state_epoch;
  }
  return cudaSuccess;
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

// Output [rows, T, D] fp32 as the target of the epilogue's TMA stores: boxes
// of 32 tokens x 16 channels (64 bytes, 64-byte swizzle); tokens past T are
// clipped, so the last tile of a row never writes into the next row.
cudaError_t make_store_map(CUtensorMap* m, void* base, int rows, int T, int D) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(T) * D * 4};
  cuuint32_t box[3] = {16, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t forward_t(const void* Q, const void* K, const void* V, int rows, int T,
                      const int32_t* lens, int heads, float* O, float* lse2, int32_t* err,
                      cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mo;
  cudaError_t e;
  if ((e = make_map(&mq, Q, rows, T, D)) != cudaSuccess) return e;
  if ((e = make_map(&mk, K, rows, T, D)) != cudaSuccess) return e;
  if ((e = make_map(&mv, V, rows, T, D)) != cudaSuccess) return e;
  if ((e = make_store_map(&mo, O, rows, T, D)) != cudaSuccess) return e;
  static int opted_in[kMaxDevices] = {};
  if ((e = raise_smem_limit(attn_fwd_kernel<D>, FwdCfg<D>::SMEM, opted_in)) != cudaSuccess) return e;
  const int nqt = (T + BM - 1) / BM, nqb = (nqt + 1) / 2;
  FwdParams p{lse2, lens, heads, rows, T, lse_stride(T), nqt, nqb, rows * nqb,
              rows_per_l2_block(T, D, 2), kLog2e / sqrtf(float(D)), err};
  const unsigned grid = static_cast<unsigned>(std::min(p.items, num_sms()));
  attn_fwd_kernel<D><<<grid, kFwdThreads, FwdCfg<D>::SMEM, stream>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t colsum_t(const void* Q, const void* K, const float* lse2, int rows, int T,
                     const int32_t* lens, int heads, float* colsum, int32_t* err,
                     cudaStream_t stream) {
  CUtensorMap mq, mk;
  cudaError_t e;
  if ((e = make_map(&mq, Q, rows, T, D)) != cudaSuccess) return e;
  if ((e = make_map(&mk, K, rows, T, D)) != cudaSuccess) return e;
  static int opted_in[kMaxDevices] = {};
  if ((e = raise_smem_limit(attn_colsum_kernel<D>, ColCfg<D>::SMEM, opted_in)) != cudaSuccess)
    return e;
  const int nqt = (T + BM - 1) / BM;
  ColParams p{lse2, colsum, lens, heads, rows, T, lse_stride(T), nqt, rows * nqt,
              rows_per_l2_block(T, D, 1), kLog2e / sqrtf(float(D)), err};
  const unsigned grid = static_cast<unsigned>(std::min(p.items, num_sms()));
  attn_colsum_kernel<D><<<grid, kColThreads, ColCfg<D>::SMEM, stream>>>(mq, mk, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prefill_forward(const void* Q, const void* K, const void* V, int rows, int T,
                            const int32_t* lens, int heads, int d, float* O, float* lse2,
                            int32_t* err, cudaStream_t stream) {
  if (static_cast<long>(rows) * T == 0) return cudaSuccess;
  return d == 128 ? forward_t<128>(Q, K, V, rows, T, lens, heads, O, lse2, err, stream)
                  : forward_t<64>(Q, K, V, rows, T, lens, heads, O, lse2, err, stream);
}

cudaError_t prefill_colsum(const void* Q, const void* K, const float* lse2, int rows, int T,
                           const int32_t* lens, int heads, int d, float* colsum, int32_t* err,
                           cudaStream_t stream) {
  if (static_cast<long>(rows) * T == 0) return cudaSuccess;
  return d == 128 ? colsum_t<128>(Q, K, lse2, rows, T, lens, heads, colsum, err, stream)
                  : colsum_t<64>(Q, K, lse2, rows, T, lens, heads, colsum, err, stream);
}

// ------------------------------------------------------------------ allocation-free scratch
// Per-row log-sum-exp for h2o_prefill_attention_noalloc lives in this fixed
// file-scope device array instead of an allocation, and the cache-free entry
// points report bounded waits that gave up through the error word next to it.
// Host code must not pass either symbol itself to a kernel (on the host it is
// only a stand-in); their device addresses are looked up per device below.
static __device__ __align__(256) float g_noalloc_lse[H2O_NOALLOC_MAX_LSE];
static __device__ __align__(16) int32_t g_attention_err[4];

namespace {
float* g_noalloc_ptr[kMaxDevices] = {};
int32_t* g_attention_err_ptr[kMaxDevices] = {};

// Device address of `symbol` on the current device, looked up once per device
// with that device current and cached in slot[dev].
template <typename T, typename Sym>
cudaError_t device_symbol(T* (&slot)[kMaxDevices], const Sym& symbol, T** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_device_state_mutex);
  if (slot[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess) return e;
    slot[dev] = static_cast<T*>(p);
  }
  *out = slot[dev];
  return cudaSuccess;
}
}  // namespace

cudaError_t noalloc_lse_scratch(float** out) { return device_symbol(g_noalloc_ptr, g_noalloc_lse, out); }

cudaError_t attention_error_word(int32_t** out) {
  return device_symbol(g_attention_err_ptr, g_attention_err, out);
}

void forget_device_state() {
  std::lock_guard<std::mutex> lock(g_device_state_mutex);
  for (int i = 0; i < kMaxDevices; ++i) {
    g_noalloc_ptr[i] = nullptr;
    g_attention_err_ptr[i] = nullptr;
  }
  ++g_device_state_epoch;
}

}  // namespace h2o
