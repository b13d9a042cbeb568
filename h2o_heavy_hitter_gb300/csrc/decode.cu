// Fused H2O decode step, one launch per layer and step: instantiation of the
// kernel in decode_kernel.cuh, its launch shape and its launcher.
#include "decode_kernel.cuh"

namespace h2o {
namespace {

using KernelFn = void (*)(DecodeArgs);

template <int D, int NT, bool F8, bool PIPE>
KernelFn pick_p(const DecodeConfig& c) {
  if (c.unroll == 2) return decode_kernel<D, NT, 2, PIPE, F8>;
  if (F8 && c.unroll == 8) return decode_kernel<D, NT, 8, PIPE, F8>;
  return decode_kernel<D, NT, 4, PIPE, F8>;
}

template <int D, int NT, bool F8>
KernelFn pick_u(const DecodeConfig& c) {
  return c.pipe ? pick_p<D, NT, F8, true>(c) : pick_p<D, NT, F8, false>(c);
}

template <bool F8>
KernelFn pick_f(const DecodeConfig& c, int d) {
  if (d == 128) return c.threads == 256 ? pick_u<128, 256, F8>(c) : pick_u<128, 128, F8>(c);
  return c.threads == 256 ? pick_u<64, 256, F8>(c) : pick_u<64, 128, F8>(c);
}

KernelFn pick(const DecodeConfig& c, int d, bool f8) { return f8 ? pick_f<true>(c, d) : pick_f<false>(c, d); }

}  // namespace

DecodeConfig decode_config(int rows, int k, int d, int num_sms, const DecodeTuning& tune,
                           bool fp8, long long l2_bytes) {
  DecodeConfig c{};
  const bool few_rows = rows < num_sms;
  const bool many_rows = rows >= 4 * num_sms;
  // An E4M3 slot is half the bytes of a bf16 one: with many rows (one
  // unpipelined batch per group) twice as many slots per batch keep the same
  // bytes in flight (measured: batch 256 x 32 heads, 194 us against 213 us).
  c.unroll = tune.unroll == 2 || tune.unroll == 4 || (fp8 && tune.unroll == 8)
                 ? tune.unroll
                 : (fp8 && many_rows ? 8 : 4);
  c.pdl = tune.pdl >= 0;
  // The L2 prefetch before the dependency wait pays only when a launch's K/V
  // fits comfortably in L2: a larger sweep evicts the prefetched lines before
  // it reads them, and HBM moves them twice (measured: 128 rows x 4096 slots,
  // 275 MB, 49 -> 66 us per step with the prefetch; 8192 rows x 410 slots,
  // 262 -> 303 us).
  const long long kv_bytes = 2LL * rows * k * d * (fp8 ? 1 : 2);
  c.prefetch = tune.prefetch > 0 || (tune.prefetch == 0 && 5 * kv_bytes <= 3 * l2_bytes);
  // Measured on GB300 (decode sweeps over the workload shapes):
  //  * many rows (>= 4 per SM): one 128-thread CTA per row, one batch in flight;
  //  * fewer rows than that: 256-thread CTAs with two batches in flight per
  //    group (software pipelining), which keeps memory busy across the serial
  //    batches of a long row; below one row per SM the rows are split into
  //    segments until the grid is one wave of about two CTAs per SM (128 rows
  //    of 4096 slots: 49 us per step with two segments per row, against 61 us
  //    for eight segments of 128-thread CTAs and 61 us for three).
  // Short rows (under 256 slots) are latency-bound: 128 threads, one batch.
  const bool small = many_rows || (few_rows && k < 256);
  c.threads = tune.threads == 128 || tune.threads == 256 ? tune.threads : (small ? 128 : 256);
  c.pipe = tune.pipe > 0 || (tune.pipe == 0 && !small);
  const int groups = c.threads / (d / 8);
  int segs = 1;
  if (tune.segs > 0) {
    segs = tune.segs;
  } else if (few_rows) {
    while (segs < kMaxDecodeSegs && static_cast<long>(rows) * segs * 2 <= 2L * num_sms &&
           (k + 2 * segs - 1) / (2 * segs) >= 2 * groups * c.unroll)
      segs *= 2;
  }
  if (segs < 1) segs = 1;
  if (segs > kMaxDecodeSegs) segs = kMaxDecodeSegs;
  c.seg_len = (k + segs - 1) / segs;
  c.segs = (k + c.seg_len - 1) / c.seg_len;  // no empty trailing segment
  c.smem = c.segs == 1 && k <= kSoloSlots ? static_cast<size_t>(k) * sizeof(float) : 0;
  return c;
}

cudaError_t decode_launch(const DecodeArgs& a, const DecodeConfig& cfg, int rows, int d,
                          cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(rows) * static_cast<unsigned>(cfg.segs));
  lc.blockDim = dim3(static_cast<unsigned>(cfg.threads));
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = cfg.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, pick(cfg, d, a.kscale != nullptr), a);
}

}  // namespace h2o
