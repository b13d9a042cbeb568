// Several H2O decode steps of every row in one launch: the kernel of
// decode_kernel.cuh with MULTI set, one CTA per row looping over the steps.
//
// Rows are independent, so a row's steps need no grid-wide synchronisation:
// its CTA runs step s + 1 as soon as its own step s has written the new slot.
// This removes the per-step launch and drain (the fixed cost of one launch per
// step) for callers that hold the inputs of several steps at once, e.g. a
// teacher-forced pass over a known continuation, layer by layer.
#include "decode_kernel.cuh"

namespace h2o {
namespace {

using KernelFn = void (*)(DecodeArgs);

template <int D, bool F8>
KernelFn pick_multi_d(const DecodeConfig& c) {
  if (c.threads == 256) return decode_kernel<D, 256, 4, true, F8, true>;
  if constexpr (F8) {
    if (c.unroll == 8) return decode_kernel<D, 128, 8, false, F8, true>;
  }
  return decode_kernel<D, 128, 4, false, F8, true>;
}

KernelFn pick_multi(const DecodeConfig& c, int d, bool f8) {
  if (d == 128) return f8 ? pick_multi_d<128, true>(c) : pick_multi_d<128, false>(c);
  return f8 ? pick_multi_d<64, true>(c) : pick_multi_d<64, false>(c);
}

}  // namespace

DecodeConfig decode_multi_config(int rows, int k, int d, int num_sms, bool fp8) {
  DecodeConfig c{};
  const bool many_rows = rows >= 4 * num_sms;
  c.threads = many_rows ? 128 : 256;
  c.pipe = !many_rows;
  c.unroll = fp8 && many_rows ? 8 : 4;
  c.pdl = false;
  c.segs = 1;
  c.seg_len = k;
  c.smem = static_cast<size_t>(k) * sizeof(float);
  (void)d;
  return c;
}

cudaError_t decode_multi_launch(const DecodeArgs& a, const DecodeConfig& cfg, int rows, int d,
                                cudaStream_t stream) {
  if (rows == 0 || a.steps == 0) return cudaSuccess;
  if (cfg.segs != 1 || a.segs != 1 || a.k > kMultiMaxSlots) return cudaErrorInvalidValue;
  KernelFn fn = pick_multi(cfg, d, a.kscale != nullptr);
  fn<<<static_cast<unsigned>(rows), static_cast<unsigned>(cfg.threads), cfg.smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace h2o
