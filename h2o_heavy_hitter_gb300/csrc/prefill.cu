// Prefill attention of the H2O policy: causal softmax attention of a prompt
// and the column sums of its probability matrix, the prompt tokens'
// accumulated scores (H2O: Heavy-Hitter Oracle ..., summary page, section 3.2
// and appendix A, Pseudocode).
//
// Two passes over the causal (query, key) pairs:
//   forward: per query row, online softmax over keys 0..i -> O_i and the
//            base-2 log-sum-exp lse2_i of the scaled logits;
//   colsum:  per key column j, sum_{i >= j} 2^(s_ij - lse2_i).
// Both passes compute s_ij with the same lane mapping and reduction order, so
// the logits of the second pass equal the first pass's bit for bit.
//
// This is the CUDA-core form: one warp per query row (forward) or key column
// (colsum), d/32 elements per lane.
#include "common.cuh"
#include "kernels.h"

namespace h2o {
namespace {

template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16* p, float* f) {
  constexpr int E = D / 32;
  if constexpr (E == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(u << 16);
    f[1] = __uint_as_float(u & 0xffff0000u);
  }
}

template <int D>
__device__ __forceinline__ float warp_dot(const float* q, const float* k) {
  constexpr int E = D / 32;
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) s = fmaf(q[e], k[e], s);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

template <int D>
__global__ void __launch_bounds__(256) forward_warp_kernel(const __nv_bfloat16* __restrict__ Q,
                                                          const __nv_bfloat16* __restrict__ K,
                                                          const __nv_bfloat16* __restrict__ V,
                                                          int rows, int T, float qscale,
                                                          float* __restrict__ O,
                                                          float* __restrict__ lse2) {
  constexpr int E = D / 32;
  const long w = static_cast<long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long>(rows) * T) return;
  const int row = static_cast<int>(w / T), i = static_cast<int>(w % T);
  const size_t base = static_cast<size_t>(row) * T * D;
  float q[E];
  load_row<D>(Q + base + static_cast<size_t>(i) * D + lane * E, q);
#pragma unroll
  for (int e = 0; e < E; ++e) q[e] *= qscale;
  float m = -INFINITY, l = 0.f, o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) o[e] = 0.f;
  for (int j = 0; j <= i; ++j) {
    float kf[E], vf[E];
    load_row<D>(K + base + static_cast<size_t>(j) * D + lane * E, kf);
    load_row<D>(V + base + static_cast<size_t>(j) * D + lane * E, vf);
    const float s = warp_dot<D>(q, kf);
    const float mn = fmaxf(m, s);
    const float corr = ex2(m - mn);
    const float p = ex2(s - mn);
    l = fmaf(l, corr, p);
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = fmaf(p, vf[e], o[e] * corr);
    m = mn;
  }
  const float inv = 1.f / l;
  float* orow = O + base + static_cast<size_t>(i) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; ++e) orow[e] = o[e] * inv;
  if (lane == 0) lse2[static_cast<size_t>(row) * T + i] = m + log2f(l);
}

template <int D>
__global__ void __launch_bounds__(256) colsum_warp_kernel(const __nv_bfloat16* __restrict__ Q,
                                                         const __nv_bfloat16* __restrict__ K,
                                                         const float* __restrict__ lse2, int rows,
                                                         int T, float qscale,
                                                         float* __restrict__ colsum) {
  constexpr int E = D / 32;
  const long w = static_cast<long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long>(rows) * T) return;
  const int row = static_cast<int>(w / T), j = static_cast<int>(w % T);
  const size_t base = static_cast<size_t>(row) * T * D;
  float kf[E];
  load_row<D>(K + base + static_cast<size_t>(j) * D + lane * E, kf);
  float acc = 0.f;
  for (int i = j; i < T; ++i) {
    float q[E];
    load_row<D>(Q + base + static_cast<size_t>(i) * D + lane * E, q);
#pragma unroll
    for (int e = 0; e < E; ++e) q[e] *= qscale;
    const float s = warp_dot<D>(q, kf);
    acc += ex2(s - lse2[static_cast<size_t>(row) * T + i]);
  }
  if (lane == 0) colsum[static_cast<size_t>(row) * T + j] = acc;
}

}  // namespace

cudaError_t prefill_forward(const void* Q, const void* K, const void* V, int rows, int T, int d,
                            float* O, float* lse2, int32_t* /*err*/, cudaStream_t stream) {
  const long warps = static_cast<long>(rows) * T;
  if (warps == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  const float qscale = kLog2e / sqrtf(static_cast<float>(d));
  auto q = static_cast<const __nv_bfloat16*>(Q);
  auto k = static_cast<const __nv_bfloat16*>(K);
  auto v = static_cast<const __nv_bfloat16*>(V);
  if (d == 128)
    forward_warp_kernel<128><<<blocks, 256, 0, stream>>>(q, k, v, rows, T, qscale, O, lse2);
  else
    forward_warp_kernel<64><<<blocks, 256, 0, stream>>>(q, k, v, rows, T, qscale, O, lse2);
  return cudaGetLastError();
}

cudaError_t prefill_colsum(const void* Q, const void* K, const float* lse2, int rows, int T,
                           int d, float* colsum, int32_t* /*err*/, cudaStream_t stream) {
  const long warps = static_cast<long>(rows) * T;
  if (warps == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((warps + 7) / 8);
  const float qscale = kLog2e / sqrtf(static_cast<float>(d));
  auto q = static_cast<const __nv_bfloat16*>(Q);
  auto k = static_cast<const __nv_bfloat16*>(K);
  if (d == 128)
    colsum_warp_kernel<128><<<blocks, 256, 0, stream>>>(q, k, lse2, rows, T, qscale, colsum);
  else
    colsum_warp_kernel<64><<<blocks, 256, 0, stream>>>(q, k, lse2, rows, T, qscale, colsum);
  return cudaGetLastError();
}

}  // namespace h2o
