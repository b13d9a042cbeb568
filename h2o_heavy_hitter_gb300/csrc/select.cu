// Prefill selection and compaction of the H2O policy (H2O: Heavy-Hitter
// Oracle ..., summary page, appendix A: Pseudocode and System Details).
//
// select:  per row, keep the r most recent prompt tokens and the h other
//          tokens with the largest (score, position) keys (every token when
//          T <= h + r). The h-th largest key is found by an MSB-first radix
//          select over the fp32 score bits (scores are non-negative, so their
//          bit patterns order like the values); ties at the boundary score
//          keep the later positions. The kept positions are compacted in
//          ascending order into the row's cache slots with block-wide scans.
// gather:  copy the K/V rows of the kept positions into their slots.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace h2o {
namespace {

constexpr int kSelectThreads = 1024;

// Block-wide exclusive scan of one int per thread; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int x, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < nw ? wsum[lane] : 0;
    int vi = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, vi, off);
      if (lane >= off) vi += y;
    }
    wsum[lane] = vi - v;
    if (lane == 31) wsum[32] = vi;
  }
  __syncthreads();
  const int r = wsum[warp] + incl - x;
  *total = wsum[32];
  __syncthreads();
  return r;
}

// colsum rows are `stride` floats apart (the padded prompt length); the row's
// own prompt length T is `stride`, or its batch entry's length in `lens`.
__global__ void __launch_bounds__(kSelectThreads) select_kernel(const float* __restrict__ colsum,
                                                               int stride,
                                                               const int32_t* __restrict__ lens,
                                                               int heads, int h, int r, int k,
                                                               bool ring,
                                                               float* __restrict__ score,
                                                               int32_t* __restrict__ pos,
                                                               int32_t* __restrict__ meta,
                                                               int32_t* __restrict__ err) {
  __shared__ unsigned hist[256];
  __shared__ int wsum[33];
  __shared__ unsigned s_prefix;
  __shared__ int s_rank;
  const int row = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const int T = row_len(lens, heads, row, stride);
  if (lens && tid == 0 && row % heads == 0 && T != lens[row / heads] && err)
    atomicOr(err, kErrBadLength);
  const float* cs = colsum + static_cast<size_t>(row) * stride;
  float* sc = score + static_cast<size_t>(row) * k;
  int32_t* ps = pos + static_cast<size_t>(row) * k;

  const bool keep_all = T <= k;
  const int n_cand = keep_all ? 0 : T - r;
  // Keep candidate p iff bits(score_p) > tau, or == tau and p is not among the
  // first `skip` candidates holding that exact score.
  unsigned tau = 0xffffffffu;
  int skip = 0x7fffffff;
  if (!keep_all && h > 0) {
    unsigned prefix = 0, mask = 0;
    int rank = n_cand - h;  // index, in ascending (score, position) order, of the smallest kept key
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += nt) hist[i] = 0;
      __syncthreads();
      for (int p = tid; p < n_cand; p += nt) {
        const unsigned u = __float_as_uint(cs[p]);
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // Warp 0 finds the bin holding the rank-th key: each lane sums eight
        // bins, a shuffle scan places the lanes, and the one lane whose range
        // contains the rank walks its eight bins.
        unsigned c[8];
        int local = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = hist[tid * 8 + j];
          local += static_cast<int>(c[j]);
        }
        int incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, off);
          if (tid >= off) incl += y;
        }
        int cum = incl - local;
        if (cum <= rank && rank < incl) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (cum + static_cast<int>(c[j]) > rank) {
              s_prefix = prefix | (static_cast<unsigned>(tid * 8 + j) << shift);
              s_rank = rank - cum;
              break;
            }
            cum += static_cast<int>(c[j]);
          }
        }
      }
      __syncthreads();
      prefix = s_prefix;
      rank = s_rank;
      mask |= 0xffu << shift;
    }
    tau = prefix;
    skip = rank;
  }

  const int seg = (T + nt - 1) / nt;
  const int p0 = min(T, tid * seg), p1 = min(T, p0 + seg);
  int eq = 0;
  if (!keep_all && h > 0)
    for (int p = p0; p < min(p1, n_cand); ++p) eq += __float_as_uint(cs[p]) == tau;
  int dummy;
  const int eq_base = block_exclusive_scan(eq, wsum, &dummy);

  auto keep = [&](int p, int& e) -> bool {
    if (keep_all || p >= n_cand) return true;
    if (h == 0) return false;
    const unsigned u = __float_as_uint(cs[p]);
    if (u > tau) return true;
    if (u == tau) return (e++) >= skip;
    return false;
  };
  int kept = 0;
  {
    int e = eq_base;
    for (int p = p0; p < p1; ++p) kept += keep(p, e);
  }
  int total;
  int s = block_exclusive_scan(kept, wsum, &total);
  if (ring) {  // every slot empty first: the window's slots need not be contiguous
    for (int j = tid; j < k; j += nt) {
      ps[j] = -1;
      sc[j] = 0.f;
    }
    __syncthreads();
  }
  {
    // Kept tokens in ascending position order take slots 0, 1, ...; in the
    // ring layout the window's tokens (all after the older kept ones) take
    // slot h + p mod r instead.
    int e = eq_base;
    for (int p = p0; p < p1; ++p)
      if (keep(p, e)) {
        const int slot = ring && p >= T - r ? h + p % r : s;
        ps[slot] = p;
        sc[slot] = cs[p];
        ++s;
      }
  }
  if (!ring)
    for (int j = total + tid; j < k; j += nt) {
      ps[j] = -1;
      sc[j] = 0.f;
    }
  if (tid == 0) {
    int32_t* mr = meta + static_cast<size_t>(row) * 4;
    mr[0] = total;
    mr[1] = T;
    mr[2] = -1;
    mr[3] = 0;
  }
}

// One warp per kGatherSlots slots: every lane loads its 16-byte chunks of all
// of them before it stores any, so that several loads per lane are in flight.
constexpr int kGatherSlots = 4;

template <int D>
__global__ void __launch_bounds__(256) gather_kernel(const __nv_bfloat16* __restrict__ K,
                                                    const __nv_bfloat16* __restrict__ V, int T,
                                                    int k, const int32_t* __restrict__ pos,
                                                    __nv_bfloat16* __restrict__ Kc,
                                                    __nv_bfloat16* __restrict__ Vc,
                                                    int32_t* __restrict__ err) {
  constexpr int CH = D / 8;                    // 16-byte chunks per K or V row
  constexpr int PER_SLOT = 2 * CH;             // chunks of a slot: K row, then V row
  constexpr int N = PER_SLOT * kGatherSlots / 32;  // chunks per lane
  const int row = blockIdx.x;
  const int slot0 = (blockIdx.y * 8 + (threadIdx.x >> 5)) * kGatherSlots;
  const int lane = threadIdx.x & 31;
  uint4 v[N];
  size_t dst[N];
  bool isv[N], live[N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const int q = lane + 32 * i;
    const int slot = slot0 + q / PER_SLOT;
    const int c = q % PER_SLOT;
    isv[i] = c >= CH;
    live[i] = false;
    if (slot >= k) continue;
    const int p = pos[static_cast<size_t>(row) * k + slot];
    if (p < 0) continue;
    if (p >= T) {  // never written by the selection; reported, nothing is read
      if (c == 0 && err) atomicOr(err, kErrBadState);
      continue;
    }
    const int cc = isv[i] ? c - CH : c;
    v[i] = *reinterpret_cast<const uint4*>((isv[i] ? V : K) +
                                           (static_cast<size_t>(row) * T + p) * D + cc * 8);
    dst[i] = (static_cast<size_t>(row) * k + slot) * D + cc * 8;
    live[i] = true;
  }
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (live[i]) *reinterpret_cast<uint4*>((isv[i] ? Vc : Kc) + dst[i]) = v[i];
}

// E4M3 cache: eight lanes per slot, four slots per warp; every lane loads its
// D / 8 values of the kept token's K and V rows, then each row is quantised
// with one scale (the amax is reduced over the slot's eight lanes).
template <int D>
__global__ void __launch_bounds__(256) gather_fp8_kernel(const __nv_bfloat16* __restrict__ K,
                                                        const __nv_bfloat16* __restrict__ V, int T,
                                                        int k, const int32_t* __restrict__ pos,
                                                        uint8_t* __restrict__ Kc,
                                                        uint8_t* __restrict__ Vc,
                                                        float* __restrict__ kscale,
                                                        float* __restrict__ vscale,
                                                        int32_t* __restrict__ err) {
  constexpr int LPS = 8;          // lanes per slot
  constexpr int EPL = D / LPS;    // values per lane: 16 (d = 128) or 8 (d = 64)
  constexpr int NV = EPL / 8;     // 16-byte loads per lane and row
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int slot = (blockIdx.y * 8 + (threadIdx.x >> 5)) * kGatherSlots + lane / LPS;
  const int l = lane % LPS;
  const unsigned gmask = 0xffu << (lane & ~(LPS - 1));  // the slot's eight lanes
  // The eight lanes of a slot share slot and position, so they leave together
  // and the quantiser's shuffles below see whole groups.
  if (slot >= k) return;
  const int p = pos[static_cast<size_t>(row) * k + slot];
  if (p < 0) return;
  if (p >= T) {  // never written by the selection; reported, nothing is read
    if (l == 0 && err) atomicOr(err, kErrBadState);
    return;
  }
  const size_t src = (static_cast<size_t>(row) * T + p) * D + l * EPL;
  const size_t dst = (static_cast<size_t>(row) * k + slot) * D + l * EPL;
  uint4 raw[2][NV];
#pragma unroll
  for (int isv = 0; isv < 2; ++isv)
#pragma unroll
    for (int j = 0; j < NV; ++j)
      raw[isv][j] = *reinterpret_cast<const uint4*>((isv ? V : K) + src + 8 * j);
#pragma unroll
  for (int isv = 0; isv < 2; ++isv) {
    float f[EPL];
#pragma unroll
    for (int j = 0; j < NV; ++j) bf16x8_to_f32(raw[isv][j], f + 8 * j);
    uint32_t pairs[EPL / 2];
    const float sc = quantize_e4m3<EPL>(f, gmask, LPS, pairs);
    uint8_t* out = (isv ? Vc : Kc) + dst;
    if constexpr (EPL == 16)
      *reinterpret_cast<uint4*>(out) =
          make_uint4(pairs[0] | (pairs[1] << 16), pairs[2] | (pairs[3] << 16),
                     pairs[4] | (pairs[5] << 16), pairs[6] | (pairs[7] << 16));
    else
      *reinterpret_cast<uint2*>(out) = make_uint2(pairs[0] | (pairs[1] << 16), pairs[2] | (pairs[3] << 16));
    if (l == 0) (isv ? vscale : kscale)[static_cast<size_t>(row) * k + slot] = sc;
  }
}

__global__ void reset_kernel(int rows, int k, float* __restrict__ score, int32_t* __restrict__ pos,
                             int32_t* __restrict__ meta) {
  const size_t n = static_cast<size_t>(rows) * k;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    pos[i] = -1;
    score[i] = 0.f;
    if (i < static_cast<size_t>(rows)) {
      meta[4 * i + 0] = 0;
      meta[4 * i + 1] = 0;
      meta[4 * i + 2] = -1;
      meta[4 * i + 3] = 0;
    }
  }
}

// Failure-path probe: waits, with the library's bounded wait, on an mbarrier
// nothing ever arrives on. The wait gives up after the limit, sets the wait
// bit of the error word and the kernel returns, as a kernel of the hot path
// would when a producer never delivers.
__global__ void wait_limit_kernel(int32_t* err) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  fence_barrier_init();
  mbar_wait(&bar, 0, err);
}

}  // namespace

cudaError_t wait_limit_probe(int32_t* err, cudaStream_t stream) {
  wait_limit_kernel<<<1, 1, 0, stream>>>(err);
  return cudaGetLastError();
}

cudaError_t prefill_select(const float* colsum, int rows, int T, const int32_t* lens, int heads,
                           int h, int r, bool ring, float* score, int32_t* pos, int32_t* meta,
                           int32_t* err, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  // About four candidates per thread: a short prompt's row takes a small block,
  // so that many rows run at once (the result does not depend on the block
  // size: compaction and ties follow position order).
  const int threads = std::min(kSelectThreads, std::max(128, ((T + 3) / 4 + 31) / 32 * 32));
  select_kernel<<<rows, threads, 0, stream>>>(colsum, T, lens, heads, h, r, h + r, ring, score,
                                              pos, meta, err);
  return cudaGetLastError();
}

cudaError_t prefill_gather(const void* K, const void* V, int rows, int T, int d, int k,
                           const int32_t* pos, void* Kc, void* Vc, int32_t* err,
                           cudaStream_t stream) {
  if (rows == 0 || T == 0) return cudaSuccess;
  const int per_block = 8 * kGatherSlots;
  const dim3 grid(static_cast<unsigned>(rows), static_cast<unsigned>((k + per_block - 1) / per_block));
  auto kk = static_cast<const __nv_bfloat16*>(K);
  auto vv = static_cast<const __nv_bfloat16*>(V);
  auto kc = static_cast<__nv_bfloat16*>(Kc);
  auto vc = static_cast<__nv_bfloat16*>(Vc);
  if (d == 128)
    gather_kernel<128><<<grid, 256, 0, stream>>>(kk, vv, T, k, pos, kc, vc, err);
  else
    gather_kernel<64><<<grid, 256, 0, stream>>>(kk, vv, T, k, pos, kc, vc, err);
  return cudaGetLastError();
}

cudaError_t prefill_gather_fp8(const void* K, const void* V, int rows, int T, int d, int k,
                               const int32_t* pos, void* Kc, void* Vc, float* kscale,
                               float* vscale, int32_t* err, cudaStream_t stream) {
  if (rows == 0 || T == 0) return cudaSuccess;
  const int per_block = 8 * kGatherSlots;
  const dim3 grid(static_cast<unsigned>(rows), static_cast<unsigned>((k + per_block - 1) / per_block));
  auto kk = static_cast<const __nv_bfloat16*>(K);
  auto vv = static_cast<const __nv_bfloat16*>(V);
  auto kc = static_cast<uint8_t*>(Kc);
  auto vc = static_cast<uint8_t*>(Vc);
  if (d == 128)
    gather_fp8_kernel<128><<<grid, 256, 0, stream>>>(kk, vv, T, k, pos, kc, vc, kscale, vscale,
                                                     err);
  else
    gather_fp8_kernel<64><<<grid, 256, 0, stream>>>(kk, vv, T, k, pos, kc, vc, kscale, vscale, err);
  return cudaGetLastError();
}

cudaError_t cache_reset(int rows, int k, float* score, int32_t* pos, int32_t* meta,
                        cudaStream_t stream) {
  const size_t n = static_cast<size_t>(rows) * k;
  if (n == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((n + 255) / 256, 4096));
  reset_kernel<<<blocks, 256, 0, stream>>>(rows, k, score, pos, meta);
  return cudaGetLastError();
}

}  // namespace h2o
