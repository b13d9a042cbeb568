// Fused H2O decode step (one launch per layer and step).
//
// Policy (H2O: Heavy-Hitter Oracle ..., summary page, sections 2 and 4.1): for
// every (batch, head) row, append the new token, attend over the cached tokens
// plus the new one, add each softmax probability to the token's accumulated
// score, evict at most one token -- the smallest (score, position) among those
// at positions <= t - r -- and write the new token into the freed slot.
//
// GB300 mapping. The step is a GEMV over k cached rows: HBM-bound, no tensor
// cores. A row is split over a thread-block cluster of C CTAs; each CTA owns a
// contiguous chunk of the row's slots and streams its K/V chunk into shared
// memory with 1-D bulk async copies (TMA engine) in stages of SPS slots, NST
// stages in flight. Inside a CTA, a group of d/8 lanes handles one slot (16 B
// per lane, conflict-free shared loads), computes the logit with group
// shuffles and keeps an online softmax (max, sum, partial output) per group.
// The CTAs of a cluster combine (max, sum) through distributed shared memory,
// so every CTA knows the exact normaliser before it updates its scores; the
// argmin over eviction candidates is a packed u64 key (score bits, position),
// reduced in the warp, the CTA and then the cluster. The slot holding the
// argmin is overwritten in place by the CTA that owns it. Row metadata (fill
// count, next position) lives in device memory and is advanced here, so a
// CUDA graph of many steps replays correctly.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace h2o {
namespace {

constexpr int kNewSlot = -2;  // argmin slot value meaning "the new token itself"
constexpr int kMaxCluster = 16;
constexpr size_t kMaxSmem = 220 * 1024;  // below the 227 KB per-CTA limit of sm_103a

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int D, int NT, int SPS, int NST>
struct DecodeSmem {
  static constexpr int LPS = D / 8;  // lanes per slot (16 bytes each)
  static constexpr int G = NT / LPS; // slot groups per CTA
  static constexpr int NW = NT / 32;
  uint64_t bar[NST];
  unsigned long long xkey;  // this CTA's smallest candidate key (read by peers)
  unsigned long long kmin;  // cluster-wide smallest key (broadcast in the CTA)
  int my_slot;              // slot of xkey (kNewSlot for the new token)
  int pad_;
  float xml[4];             // {max, sum, new token logit, 0} of this CTA (read by peers)
  float peer_ml[kMaxCluster][2];
  float snew;               // logit of the new token (copied from rank 0)
  float xo[D];              // partial output scaled to this CTA's max (read by rank 0)
  float red_ml[G][2];
  float red_o[G][D];
  unsigned long long wkey[NW];
  int wslot[NW];
  alignas(128) __nv_bfloat16 Kst[NST][SPS * D];
  alignas(128) __nv_bfloat16 Vst[NST][SPS * D];
};

template <int D, int NT, int SPS, int NST>
__global__ void __launch_bounds__(NT) decode_kernel(const DecodeArgs a) {
  using Sm = DecodeSmem<D, NT, SPS, NST>;
  constexpr int LPS = Sm::LPS;
  constexpr int G = Sm::G;
  constexpr int NW = Sm::NW;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
  float* s_log = reinterpret_cast<float*>(smem_raw + sizeof(Sm));  // [chunk] logits (base 2)
  float* s_sc = s_log + a.chunk;                                  // [chunk] scores
  int* s_pos = reinterpret_cast<int*>(s_sc + a.chunk);            // [chunk] positions

  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int crank = static_cast<int>(cluster.block_rank());
  const int row = blockIdx.x / C;
  const int tid = threadIdx.x;
  const int g = tid / LPS, l = tid % LPS;
  const int warp = tid >> 5, lane = tid & 31;
  const unsigned gmask = ((LPS == 32) ? 0xffffffffu : ((1u << LPS) - 1u)) << ((lane / LPS) * LPS);

  const int32_t* meta = a.meta + static_cast<size_t>(row) * 4;
  const int count = meta[0];
  const int t = meta[1];
  const int s0 = crank * a.chunk;
  const int n = max(0, min(a.chunk, count - s0));
  const int nst = (n + SPS - 1) / SPS;
  const size_t slot0 = static_cast<size_t>(row) * a.k + s0;
  const __nv_bfloat16* Kg = static_cast<const __nv_bfloat16*>(a.Kc) + slot0 * D;
  const __nv_bfloat16* Vg = static_cast<const __nv_bfloat16*>(a.Vc) + slot0 * D;

  auto issue = [&](int st) {
    const int buf = st % NST;
    const int ns = min(SPS, n - st * SPS);
    const uint32_t bytes = static_cast<uint32_t>(ns) * D * 2;
    mbar_arrive_expect_tx(&sm.bar[buf], 2 * bytes);
    bulk_copy_g2s(sm.Kst[buf], Kg + static_cast<size_t>(st) * SPS * D, bytes, &sm.bar[buf]);
    bulk_copy_g2s(sm.Vst[buf], Vg + static_cast<size_t>(st) * SPS * D, bytes, &sm.bar[buf]);
  };

  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < NST; ++i) mbar_init(&sm.bar[i], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int st = 0; st < min(NST, nst); ++st) issue(st);
  }

  // q, pre-scaled so that logits come out in base 2.
  float qf[8];
  {
    const uint4 qv = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                     static_cast<size_t>(row) * D + l * 8);
    bf16x8_to_f32(qv, qf);
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[i] *= a.qscale;
  }
  for (int i = tid; i < n; i += NT) {
    s_sc[i] = a.score[slot0 + i];
    s_pos[i] = a.pos[slot0 + i];
  }

  // Online softmax state of this lane's group.
  float m = -INFINITY, lsum = 0.f, o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = 0.f;
  auto consume = [&](const uint4& kv, const uint4& vv) -> float {
    float kf[8], vf[8];
    bf16x8_to_f32(kv, kf);
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) dot = fmaf(qf[i], kf[i], dot);
#pragma unroll
    for (int off = LPS / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(gmask, dot, off);
    const float mn = fmaxf(m, dot);
    const float corr = ex2(m - mn);
    const float p = ex2(dot - mn);
    lsum = fmaf(lsum, corr, p);
    bf16x8_to_f32(vv, vf);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = fmaf(p, vf[i], o[i] * corr);
    m = mn;
    return dot;
  };

  // The new token counts as one more slot of cluster rank 0, group 0.
  if (crank == 0 && g == 0) {
    const size_t off = static_cast<size_t>(row) * D + l * 8;
    const uint4 kv = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.k_new) + off);
    const uint4 vv = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.v_new) + off);
    const float sn = consume(kv, vv);
    if (l == 0) sm.xml[2] = sn;
  }

  bool failed = false;
  for (int st = 0; st < nst; ++st) {
    const int buf = st % NST;
    if (!mbar_wait(&sm.bar[buf], (st / NST) & 1, a.err)) failed = true;
    const int ns = min(SPS, n - st * SPS);
    const __nv_bfloat16* kb = sm.Kst[buf];
    const __nv_bfloat16* vb = sm.Vst[buf];
    for (int j = g; j < ns; j += G) {
      const uint4 kv = *reinterpret_cast<const uint4*>(kb + j * D + l * 8);
      const uint4 vv = *reinterpret_cast<const uint4*>(vb + j * D + l * 8);
      const float dot = consume(kv, vv);
      if (l == 0) s_log[st * SPS + j] = dot;
    }
    __syncthreads();
    if (tid == 0 && st + NST < nst) issue(st + NST);
  }

  // Combine the groups of this CTA.
  if (l == 0) {
    sm.red_ml[g][0] = m;
    sm.red_ml[g][1] = lsum;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) sm.red_o[g][l * 8 + i] = o[i];
  failed = __syncthreads_or(failed);
  if (tid < D) {
    float mc = -INFINITY;
#pragma unroll 4
    for (int gg = 0; gg < G; ++gg) mc = fmaxf(mc, sm.red_ml[gg][0]);
    float lc = 0.f, oc = 0.f;
    for (int gg = 0; gg < G; ++gg) {
      const float mg = sm.red_ml[gg][0];
      if (mg != -INFINITY) {
        const float w = ex2(mg - mc);
        lc = fmaf(sm.red_ml[gg][1], w, lc);
        oc = fmaf(sm.red_o[gg][tid], w, oc);
      }
    }
    sm.xo[tid] = oc;
    if (tid == 0) {
      sm.xml[0] = mc;
      sm.xml[1] = lc;
    }
  }
  cluster.sync();  // (1) every CTA's (max, sum, partial output) is published

  if (tid < C) {
    const float* pml = cluster.map_shared_rank(sm.xml, tid);
    sm.peer_ml[tid][0] = pml[0];
    sm.peer_ml[tid][1] = pml[1];
    if (tid == 0) sm.snew = pml[2];
  }
  __syncthreads();
  float M = -INFINITY;
  for (int c = 0; c < C; ++c) M = fmaxf(M, sm.peer_ml[c][0]);
  float L = 0.f;
  for (int c = 0; c < C; ++c)
    if (sm.peer_ml[c][0] != -INFINITY) L = fmaf(sm.peer_ml[c][1], ex2(sm.peer_ml[c][0] - M), L);
  const float invL = 1.f / L;
  const float p_new = ex2(sm.snew - M) * invL;

  if (crank == 0 && tid < D) {
    float acc = 0.f;
    for (int c = 0; c < C; ++c) {
      const float mc = sm.peer_ml[c][0];
      if (mc != -INFINITY) acc = fmaf(cluster.map_shared_rank(sm.xo, c)[tid], ex2(mc - M), acc);
    }
    if (!failed) a.out[static_cast<size_t>(row) * D + tid] = acc * invL;
  }

  // Accumulate scores; find this CTA's smallest eviction candidate.
  const int thr = t - a.r;  // candidates: positions <= t - r
  unsigned long long best = ~0ull;
  int bslot = -1;
  for (int i = tid; i < n; i += NT) {
    const float ns = s_sc[i] + ex2(s_log[i] - M) * invL;
    s_sc[i] = ns;
    const int ps = s_pos[i];
    if (ps <= thr) {
      const unsigned long long key =
          (static_cast<unsigned long long>(__float_as_uint(ns)) << 32) | static_cast<uint32_t>(ps);
      if (key < best) {
        best = key;
        bslot = s0 + i;
      }
    }
  }
  if (crank == 0 && tid == 0 && a.r == 0) {
    const unsigned long long key =
        (static_cast<unsigned long long>(__float_as_uint(p_new)) << 32) | static_cast<uint32_t>(t);
    if (key < best) {
      best = key;
      bslot = kNewSlot;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long ok = __shfl_xor_sync(0xffffffffu, best, off);
    const int os = __shfl_xor_sync(0xffffffffu, bslot, off);
    if (ok < best) {
      best = ok;
      bslot = os;
    }
  }
  if (lane == 0) {
    sm.wkey[warp] = best;
    sm.wslot[warp] = bslot;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long b = ~0ull;
    int bs = -1;
    for (int w = 0; w < NW; ++w)
      if (sm.wkey[w] < b) {
        b = sm.wkey[w];
        bs = sm.wslot[w];
      }
    sm.xkey = b;
    sm.my_slot = bs;
  }
  cluster.sync();  // (2) every CTA's smallest key is published
  if (tid == 0) {
    unsigned long long km = ~0ull;
    for (int c = 0; c < C; ++c) km = min(km, *cluster.map_shared_rank(&sm.xkey, c));
    sm.kmin = km;
  }
  cluster_arrive();  // (3) this thread has finished all reads of peer shared memory
  __syncthreads();

  const unsigned long long kmin = sm.kmin;
  const bool full = count >= a.k;
  int target = -1;  // slot that receives the new token, if this CTA owns it
  int evict_pos = -1;
  if (full) {
    evict_pos = static_cast<int>(kmin & 0xffffffffu);
    if (sm.xkey == kmin && sm.my_slot != kNewSlot) target = sm.my_slot;
  } else if (count >= s0 && count < s0 + a.chunk) {
    target = count;  // append into the next empty slot
  }

  if (!failed) {
    for (int i = tid; i < n; i += NT) a.score[slot0 + i] = (s0 + i == target) ? p_new : s_sc[i];
    if (target >= 0) {
      const size_t dst = (static_cast<size_t>(row) * a.k + target) * D;
      const size_t src = static_cast<size_t>(row) * D;
      if (g == 0) {
        const uint4 kv = *reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(a.k_new) + src + l * 8);
        const uint4 vv = *reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(a.v_new) + src + l * 8);
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.Kc) + dst + l * 8) = kv;
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.Vc) + dst + l * 8) = vv;
      }
      if (tid == 0) {
        a.pos[static_cast<size_t>(row) * a.k + target] = t;
        if (target >= s0 + n) a.score[static_cast<size_t>(row) * a.k + target] = p_new;
      }
    }
    if (crank == 0 && tid == 0) {
      int32_t* mw = a.meta + static_cast<size_t>(row) * 4;
      mw[0] = full ? a.k : count + 1;
      mw[1] = t + 1;
      mw[2] = evict_pos;
    }
  }
  cluster_wait();  // (3) no CTA exits while a peer may still read its shared memory
}

template <int D, int NT, int SPS, int NST>
size_t smem_bytes(int chunk) {
  return sizeof(DecodeSmem<D, NT, SPS, NST>) + static_cast<size_t>(chunk) * 12;
}

// Compile-time shapes: (threads, slots per stage) per head dim; stages 2 or 4.
template <int D>
struct Shape;
template <>
struct Shape<128> {
  static constexpr int NT = 256, SPS = 32;
};
template <>
struct Shape<64> {
  static constexpr int NT = 128, SPS = 32;
};

template <int D, int NST>
auto kernel_ptr() {
  return decode_kernel<D, Shape<D>::NT, Shape<D>::SPS, NST>;
}

template <int D, int NST>
cudaError_t prepare_t(const DecodeConfig& cfg) {
  auto k = kernel_ptr<D, NST>();
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(cfg.smem));
  if (e != cudaSuccess) return e;
  if (cfg.cluster > 8) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <int D, int NST>
cudaError_t launch_t(const DecodeArgs& a, const DecodeConfig& cfg, int rows, cudaStream_t stream) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(rows * cfg.cluster));
  lc.blockDim = dim3(Shape<D>::NT);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cfg.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel_ptr<D, NST>(), a);
}

}  // namespace

DecodeConfig decode_config(int rows, int k, int d, int num_sms, int cluster_override,
                           int stages_override) {
  DecodeConfig c{};
  const int sps = 32;
  int cl = 1;
  if (cluster_override > 0) {
    cl = cluster_override;
  } else {
    // Enough CTAs to cover every SM twice, but no chunk shorter than one stage.
    while (cl < 8 && static_cast<long>(rows) * cl < 2L * num_sms && (k + 2 * cl - 1) / (2 * cl) >= sps)
      cl *= 2;
  }
  c.stages = stages_override > 0 ? stages_override : 4;
  if (c.stages != 2 && c.stages != 4) c.stages = 4;
  auto smem_for = [&](int chunk) -> size_t {
    if (d == 128)
      return c.stages == 4 ? smem_bytes<128, 256, 32, 4>(chunk) : smem_bytes<128, 256, 32, 2>(chunk);
    return c.stages == 4 ? smem_bytes<64, 128, 32, 4>(chunk) : smem_bytes<64, 128, 32, 2>(chunk);
  };
  // The per-slot logit/score/position arrays must fit beside the stage ring.
  if (cl < 1) cl = 1;
  while (cl < kMaxCluster && smem_for((k + cl - 1) / cl) > kMaxSmem) cl *= 2;
  if (cl > kMaxCluster) cl = kMaxCluster;
  c.cluster = cl;
  c.chunk = (k + cl - 1) / cl;
  c.smem = smem_for(c.chunk);
  return c;
}

cudaError_t decode_prepare(const DecodeConfig& cfg, int d) {
  if (d == 128) return cfg.stages == 4 ? prepare_t<128, 4>(cfg) : prepare_t<128, 2>(cfg);
  return cfg.stages == 4 ? prepare_t<64, 4>(cfg) : prepare_t<64, 2>(cfg);
}

cudaError_t decode_launch(const DecodeArgs& a, const DecodeConfig& cfg, int rows, int d,
                          cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (d == 128)
    return cfg.stages == 4 ? launch_t<128, 4>(a, cfg, rows, stream) : launch_t<128, 2>(a, cfg, rows, stream);
  return cfg.stages == 4 ? launch_t<64, 4>(a, cfg, rows, stream) : launch_t<64, 2>(a, cfg, rows, stream);
}

}  // namespace h2o
