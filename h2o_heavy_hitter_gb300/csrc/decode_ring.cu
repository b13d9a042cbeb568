// Decode step for a cache in the ring layout (the pages' implementation: a
// heavy-hitter region plus the recent window as a circular queue): the kernel
// of decode_kernel.cuh with RING set, bf16 cache, four slots per group batch.
#include "decode_kernel.cuh"

namespace h2o {
namespace {

using KernelFn = void (*)(DecodeArgs);

template <int D, int NT>
KernelFn pick_ring_t(const DecodeConfig& c) {
  return c.pipe ? decode_kernel<D, NT, 4, true, false, false, true>
                : decode_kernel<D, NT, 4, false, false, false, true>;
}

KernelFn pick_ring(const DecodeConfig& c, int d) {
  if (d == 128) return c.threads == 256 ? pick_ring_t<128, 256>(c) : pick_ring_t<128, 128>(c);
  return c.threads == 256 ? pick_ring_t<64, 256>(c) : pick_ring_t<64, 128>(c);
}

}  // namespace

cudaError_t decode_ring_launch(const DecodeArgs& a, const DecodeConfig& cfg, int rows, int d,
                               cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (a.r < 1 || a.kscale != nullptr) return cudaErrorInvalidValue;
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
  return cudaLaunchKernelEx(&lc, pick_ring(cfg, d), a);
}

}  // namespace h2o
