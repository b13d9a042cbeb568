// Device helpers shared by the H2O kernels (sm_103a): shared-memory barriers,
// 1-D bulk async copies, bounded waits and small numeric utilities.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace h2o {

// Bits of the device error word (int32 in device memory, OR-ed by kernels).
enum DeviceError : int {
  kErrWaitTimeout = 1,  // an mbarrier wait gave up
  kErrBadState = 2,     // a kernel found inconsistent row metadata
  kErrBadLength = 4,    // a ragged batch's prompt length was outside [0, T_max]
};

// Prompt length of `row` (= batch * heads + head) in a prefill launch over
// prompts padded to T tokens: T, or the length of the row's batch entry when
// per-entry lengths are given, clamped to [0, T] so that no access leaves the
// padded tensors (the selection kernel reports lengths out of range).
__device__ __forceinline__ int row_len(const int32_t* lens, int heads, int row, int T) {
  if (!lens) return T;
  const int n = lens[row / heads];
  return n < 0 ? 0 : (n > T ? T : n);
}

// Wall-clock bound of every device-side wait, in nanoseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async proxy and the cluster.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Gives up after
// kWaitLimitNs, OR-ing kErrWaitTimeout into *err (if err is not null) and
// returning false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      if (err) atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
}

// ---- 1-D bulk copy (TMA engine, no tensor map) ------------------------------
// Copies `bytes` (multiple of 16; both addresses 16-byte aligned) from global
// memory into this CTA's shared memory; completion is signalled as
// transaction bytes on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Asks the TMA engine to pull `bytes` (multiple of 16; address 16-byte aligned)
// of global memory into L2. Nothing is read into the SM, and L2 is where every
// write to global memory lands, so the lines can never be stale.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---- numerics ----------------------------------------------------------------
// 2^x with the MUFU.EX2 unit (PTX ex2.approx.ftz.f32); ex2(-inf) = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- packed fp32 pairs (sm_100+ f32x2 instructions) ---------------------------
// Two fp32 values in one 64-bit register, element 0 in the low half. fma and
// add round each element exactly as the scalar instructions do.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max(a, b, c) in one instruction (sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---- E4M3 (OCP FP8) codes ------------------------------------------------------
// Eight codes (one per byte, element 0 in the lowest byte) to fp32; exact.
__device__ __forceinline__ void e4m3x8_to_f32(const uint2& v, float* f) {
  const uint32_t w[2] = {v.x, v.y};
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
          static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * h)) & 0xFFFFu), __NV_E4M3);
      const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      f[4 * i + 2 * h] = f2.x;
      f[4 * i + 2 * h + 1] = f2.y;
    }
}
// Two fp32 values to E4M3 codes (lo in the low byte): round to nearest even,
// saturated to +-448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  return __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}
// Quantises the values x[0..n) of this thread, part of a token vector spread
// over the lanes in `mask` (`lanes` of them, a power of two, adjacent): scale =
// amax / 448 and code = E4M3(x * (448 / amax)), fp32 with one rounding per
// operation; a zero vector gets scale 0 and zero codes. Writes the codes
// (n / 2 pairs) and returns the scale.
template <int N>
__device__ __forceinline__ float quantize_e4m3(const float* x, unsigned mask, int lanes,
                                               uint32_t* pairs) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) amax = fmaxf(amax, fabsf(x[i]));
  for (int off = lanes / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(mask, amax, off));
  if (amax == 0.f) {
#pragma unroll
    for (int j = 0; j < N / 2; ++j) pairs[j] = 0u;
    return 0.f;
  }
  const float inv = __fdiv_rn(448.f, amax);
#pragma unroll
  for (int j = 0; j < N / 2; ++j)
    pairs[j] = f32x2_to_e4m3x2(__fmul_rn(x[2 * j], inv), __fmul_rn(x[2 * j + 1], inv));
  return __fdiv_rn(amax, 448.f);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

}  // namespace h2o
