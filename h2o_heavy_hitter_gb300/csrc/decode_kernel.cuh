// Fused H2O decode step (one launch per layer and step).
//
// Policy (H2O: Heavy-Hitter Oracle ..., summary page, sections 2 and 4.1): for
// every (batch, head) row, append the new token, attend over the cached tokens
// plus the new one, add each softmax probability to the token's accumulated
// score, evict at most one token -- the smallest (score, position) among those
// at positions <= t - r -- and write the new token into the freed slot.
//
// GB300 mapping. The step is a GEMV over the k cached slots of every row:
// HBM-bound, no tensor cores. A row is split into `segs` segments of
// consecutive slots, one CTA each. Inside a CTA a group of d/8 lanes owns a
// slot (16 bytes per lane: one coalesced 256-byte K row and V row for d = 128);
// every group loads U slots' K/V straight into registers with 16-byte
// non-caching loads, computes the U logits together (independent shuffle
// chains) and keeps an online softmax (max, sum, partial output). A CTA writes
// its slots' logits and its (max, sum, output) partial to per-layer scratch,
// then the last CTA of the row to arrive (global atomic counter, fence-based
// message passing, nobody waits) combines the partials into the exact
// normaliser, writes the output, adds p_j to every slot's score, finds the
// eviction as the minimum packed u64 key (score bits << 32 | position) over
// the candidates, and overwrites that slot with the new token. Row metadata
// (fill count, next position) and the arrival counters live in device memory
// and are advanced / reset here, so a CUDA graph of many steps replays
// correctly. The launch uses programmatic dependent launch: the next step's
// CTAs are scheduled while this step drains and read nothing before their
// dependency wait.
//
// This header holds the kernel template; decode.cu instantiates it for one
// step per launch, decode_multi.cu for several steps of a row per launch.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace h2o {
namespace {

constexpr int kNewSlot = -2;  // argmin slot value meaning "the new token itself"
constexpr int kSoloSlots = 8192;  // longest row whose logits stay in shared memory
constexpr int kSoloRegs = 4;      // slots per thread whose score/position is preloaded

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ldg_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// Coherent variants, for a launch that reads cache slots it wrote itself in an
// earlier step: the non-coherent path promises nothing for such data.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ float dot8(const uint2& kv, const float* qf) {  // E4M3 codes
  float kf[8];
  e4m3x8_to_f32(kv, kf);
  float d = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) d = fmaf(qf[i], kf[i], d);
  return d;
}

__device__ __forceinline__ void accum8(float* o, float p, const uint2& vv) {  // E4M3 codes
  float vf[8];
  e4m3x8_to_f32(vv, vf);
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = fmaf(p, vf[i], o[i]);
}

// U slots' keys and values of one group batch: bf16 vectors (16 bytes per
// lane), or E4M3 codes (8 bytes per lane) with one scale per slot.
template <bool F8, int U>
struct KVBatch {
  using Vec = typename std::conditional<F8, uint2, uint4>::type;
  Vec k[U], v[U];
  float ks[U], vs[U];
};

__device__ __forceinline__ float dot8(const uint4& kv, const float* qf) {
  float kf[8];
  bf16x8_to_f32(kv, kf);
  float d = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) d = fmaf(qf[i], kf[i], d);
  return d;
}

__device__ __forceinline__ void accum8(float* o, float p, const uint4& vv) {
  float vf[8];
  bf16x8_to_f32(vv, vf);
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = fmaf(p, vf[i], o[i]);
}

__device__ __forceinline__ unsigned long long pack_key(float score, int pos) {
  return (static_cast<unsigned long long>(__float_as_uint(score)) << 32) |
         static_cast<uint32_t>(pos);
}

template <int D, int NT>
struct DecodeShared {
  static constexpr int LPS = D / 8;   // lanes per slot (16 bytes each)
  static constexpr int G = NT / LPS;  // slot groups per CTA
  static constexpr int NW = NT / 32;
  float red_ml[NW][2];
  float red_o[NW][D];  // element i of lane l of warp w's merged group at [w][i * LPS + l]
  float vnew[D];       // the new token's value vector
  float seg_w[kMaxDecodeSegs];
  float s_new;
  float M, invL, w_new, p_new;
  unsigned long long wkey[NW];
  int wslot[NW];
  int is_last;
  int target;
  int bad;         // a slot of the row held a position outside [0, t)
  float lv_score;  // ring layout: updated score of the token leaving the recent window
};

// PIPE: two batches of U slots per group in flight (software pipelining).
// F8: the cache holds E4M3 codes with per-slot scales; the new token is
// quantised (amax / 448 scale, fp32) before it is attended to and stored.
// MULTI: one CTA per row (segs = 1) runs a.steps consecutive steps of its row
// in one launch, with step s's inputs and output at offset s * rows * d; the
// steps are separated by block barriers and the cache is read with coherent
// loads, since a step reads the slot the previous step wrote.
// RING (bf16 cache, r >= 1): the layout of the pages' implementation -- heavy
// slots [0, h) filled from 0, and the recent window as a circular queue, the
// token at position p in slot h + p mod r. The recent slots' positions are
// implied by t and never read; the eviction candidates are the heavy slots
// and the token leaving the window (position t - r, in the slot the new token
// takes). When a heavy slot is evicted the leaving token moves into it.
template <int D, int NT, int U, bool PIPE, bool F8, bool MULTI = false, bool RING = false>
__global__ void __launch_bounds__(NT) decode_kernel(const DecodeArgs a) {
  static_assert(!(RING && F8), "the ring layout is built for the bf16 cache");
  using Sm = DecodeShared<D, NT>;
  constexpr int LPS = Sm::LPS, G = Sm::G, NW = Sm::NW;
  constexpr int PS = D + 4;  // partial stride: {max, sum, -, -, output[D]}
  __shared__ Sm sm;
  const int tid = threadIdx.x, g = tid / LPS, l = tid % LPS;
  const int warp = tid >> 5, lane = tid & 31;
  const unsigned gmask = ((1u << LPS) - 1u) << ((lane / LPS) * LPS);
  const int row = blockIdx.x / a.segs, seg = blockIdx.x % a.segs;
  const int s0 = seg * a.seg_len;
  const int cap = max(0, min(a.seg_len, a.k - s0));
  const size_t rk = static_cast<size_t>(row) * a.k;

  constexpr int EB = F8 ? 1 : 2;  // bytes per cached element
  if constexpr (!MULTI) {
    // This CTA's K and V slots start moving from HBM into L2 while the
    // previous kernel in the stream drains: a bulk L2 prefetch reads nothing
    // into the SM, so it is allowed before the dependency wait below (the
    // previous kernel may still write one slot of the row; that write lands in
    // L2 as well). Warp 0's lanes take 256-byte-aligned pieces of each range.
    if (warp == 0 && cap > 0 && a.prefetch) {
      const uint32_t bytes = static_cast<uint32_t>(cap) * D * EB;
      const uint32_t piece = ((bytes + 31) / 32 + 255) & ~255u;
      const uint32_t off = static_cast<uint32_t>(lane) * piece;
      if (off < bytes) {
        const uint32_t n = min(piece, bytes - off);
        const size_t base = (rk + s0) * D * EB + off;
        bulk_prefetch_l2(static_cast<const uint8_t*>(a.Kc) + base, n);
        bulk_prefetch_l2(static_cast<const uint8_t*>(a.Vc) + base, n);
      }
    }
  }
  // Everything before this wait overlaps the previous kernel's tail.
  grid_dependency_wait();  // the cache, scores and metadata are written by the previous step
  const int nsteps = MULTI ? a.steps : 1;
#pragma unroll 1
  for (int step = 0; step < nsteps; ++step) {
  const size_t io = static_cast<size_t>(step) * a.rows * D;  // this step's inputs and output
  // ---- inputs. They are read after the dependency wait: the kernel before
  // this one in the stream may have written q, k_new or v_new.
  float qf[8];
  {
    const uint4 qv = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) + io +
                                                     static_cast<size_t>(row) * D + l * 8);
    bf16x8_to_f32(qv, qf);
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[i] *= a.qscale;
  }
  uint4 knew = make_uint4(0, 0, 0, 0), vnew = make_uint4(0, 0, 0, 0);
  if (g == 0) {
    const size_t off = io + static_cast<size_t>(row) * D + l * 8;
    knew = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.k_new) + off);
    vnew = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.v_new) + off);
    if constexpr (!F8) {
      float vf[8];
      bf16x8_to_f32(vnew, vf);
#pragma unroll
      for (int i = 0; i < 8; ++i) sm.vnew[l * 8 + i] = vf[i];
    }
  }

  const int32_t* meta = a.meta + static_cast<size_t>(row) * 4;
  const int count = meta[0];
  const int t = meta[1];
  // A row holds 0 .. k tokens at distinct positions below t. Metadata that
  // says otherwise (a cache state installed through the cache view, say) is
  // reported and the row is left untouched: every CTA of the row reads the
  // same values and leaves together, so no slot outside the row is written.
  if (count < 0 || count > a.k || t < count) {
    if (tid == 0 && seg == 0 && a.err) atomicOr(a.err, kErrBadState);
    return;
  }
  if (tid == 0) sm.bad = 0;
  const int n = max(0, min(cap, count - s0));
  // ring layout: recent slots in use, heavy slots in use, the slot of position t - r (and t)
  const int nring = RING ? min(t, a.r) : 0;
  const int nh = RING ? count - nring : 0;
  const int lv = RING ? a.h + t % a.r : -1;
  // slot gi of the row holds a token (ring layout)
  auto occ_g = [&](int gi) -> bool { return gi < nh || (gi >= a.h && gi < a.h + nring); };
  // slot s0 + i of this segment holds a token (a batch may reach past the
  // segment's last slot: those lanes loaded nothing)
  const bool ring_full = RING && count >= a.k;  // every slot in use: no per-slot test
  auto occ = [&](int i) -> bool {
    if constexpr (RING)
      return i < cap && (ring_full || occ_g(s0 + i));
    else
      return i < n;
  };
  {  // the row's finishing CTA reads these scores and positions: warm L2 now
    const int lines = (cap * 4 + 127) / 128 + 1;
    for (int i = tid; i < 2 * lines; i += NT) {
      const char* base = i < lines ? reinterpret_cast<const char*>(a.score + rk + s0)
                                   : reinterpret_cast<const char*>(a.pos + rk + s0);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(base + (i % lines) * 128));
    }
  }

  // ---- sweep this segment's slots: group g takes slots g, g + G, ...; U per batch.
  float m = -INFINITY, lsum = 0.f, o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = 0.f;
  const uint8_t* Kg = static_cast<const uint8_t*>(a.Kc) + ((rk + s0) * D + l * 8) * EB;
  const uint8_t* Vg = static_cast<const uint8_t*>(a.Vc) + ((rk + s0) * D + l * 8) * EB;
  // A row handled by a single CTA keeps its logits in shared memory; split rows
  // hand them to the finishing CTA through the per-layer scratch.
  extern __shared__ float solo_logits[];
  const bool solo = a.segs == 1 && a.k <= kSoloSlots;
  float* lg_out = solo ? solo_logits : a.logits + rk + s0;
  // Single-CTA rows: this thread's slots' scores and positions, loaded now so
  // that their latency hides behind the K/V sweep.
  const int filled = min(count, a.k);
  const int slot_end = RING ? a.k : filled;  // slots the finish visits (occupied or not)
  float sc_r[kSoloRegs];
  int ps_r[kSoloRegs];
#pragma unroll
  for (int jj = 0; jj < kSoloRegs; ++jj) {
    const int i = tid + jj * NT;
    if (solo && i < slot_end && (!RING || occ_g(i))) {
      sc_r[jj] = a.score[rk + i];
      ps_r[jj] = !RING || i < a.h ? a.pos[rk + i] : 0;  // recent positions are implied
    }
  }
  // One batch: U slots of this group, loaded by capacity (slots past the fill
  // count are masked when consumed).
  using Batch = KVBatch<F8, U>;
  auto load = [&](Batch& b, int base) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * G;
      if (i < cap) {
        if constexpr (F8 && MULTI) {
          b.k[u] = ld_stream8(Kg + static_cast<size_t>(i) * D);
          b.v[u] = ld_stream8(Vg + static_cast<size_t>(i) * D);
          b.ks[u] = a.kscale[rk + s0 + i];
          b.vs[u] = a.vscale[rk + s0 + i];
        } else if constexpr (F8) {
          b.k[u] = ldg_stream8(Kg + static_cast<size_t>(i) * D);
          b.v[u] = ldg_stream8(Vg + static_cast<size_t>(i) * D);
          b.ks[u] = __ldg(a.kscale + rk + s0 + i);
          b.vs[u] = __ldg(a.vscale + rk + s0 + i);
        } else if constexpr (MULTI) {
          b.k[u] = ld_stream(Kg + static_cast<size_t>(i) * D * 2);
          b.v[u] = ld_stream(Vg + static_cast<size_t>(i) * D * 2);
        } else {
          b.k[u] = ldg_stream(Kg + static_cast<size_t>(i) * D * 2);
          b.v[u] = ldg_stream(Vg + static_cast<size_t>(i) * D * 2);
        }
      }
    }
  };
  auto consume = [&](const Batch& b, int base) {
    float s[U];
#pragma unroll
    for (int u = 0; u < U; ++u) s[u] = dot8(b.k[u], qf);
#pragma unroll
    for (int off = LPS / 2; off > 0; off >>= 1)
#pragma unroll
      for (int u = 0; u < U; ++u) s[u] += __shfl_xor_sync(gmask, s[u], off);
    if constexpr (F8) {
#pragma unroll
      for (int u = 0; u < U; ++u) s[u] *= b.ks[u];
    }
    float bm = m;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (occ(base + u * G)) bm = fmaxf(bm, s[u]);
    const float corr = ex2(m - bm);
    lsum *= corr;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] *= corr;
    m = bm;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * G;
      if (occ(i)) {
        const float p = ex2(s[u] - bm);
        lsum += p;
        if constexpr (F8)
          accum8(o, p * b.vs[u], b.v[u]);
        else
          accum8(o, p, b.v[u]);
        if (l == 0) lg_out[i] = s[u];
      }
    }
  };
  constexpr int STEP = G * U;
  if constexpr (PIPE) {
    // Two batches in flight: the next batch's loads are issued before the
    // current batch is consumed, so memory is never idle between batches.
    Batch ba, bb;
    if (g < cap) load(ba, g);
    for (int base = g; base < cap; base += 2 * STEP) {
      if (base + STEP < cap) load(bb, base + STEP);
      consume(ba, base);
      if (base + STEP >= cap) break;
      if (base + 2 * STEP < cap) load(ba, base + 2 * STEP);
      consume(bb, base + STEP);
    }
  } else {
    for (int base = g; base < cap; base += STEP) {
      Batch b;
      load(b, base);
      consume(b, base);
    }
  }
  grid_launch_dependents();

  // ---- this CTA's partial. The groups of a warp are merged with shuffles,
  // so shared memory holds one (max, sum, output) per warp. A group that saw
  // no filled slot has m = -inf and undefined sums: it contributes nothing.
  if (m == -INFINITY) {
    lsum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.f;
  }
#pragma unroll
  for (int off = LPS; off < 32; off <<= 1) {
    const float mp = __shfl_xor_sync(0xffffffffu, m, off);
    const float lp = __shfl_xor_sync(0xffffffffu, lsum, off);
    const float mn = fmaxf(m, mp);
    const float w = m == -INFINITY ? 0.f : ex2(m - mn);
    const float wp = mp == -INFINITY ? 0.f : ex2(mp - mn);
    lsum = lsum * w + lp * wp;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = o[i] * w + __shfl_xor_sync(0xffffffffu, o[i], off) * wp;
    m = mn;
  }
  if (lane < LPS) {
    if (lane == 0) {
      sm.red_ml[warp][0] = m;
      sm.red_ml[warp][1] = lsum;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) sm.red_o[warp][i * LPS + lane] = o[i];
  }
  uint2 kcode = make_uint2(0, 0), vcode = make_uint2(0, 0);  // E4M3 cache: the new token
  float kq_scale = 0.f, vq_scale = 0.f;
  if (g == 0) {  // logit of the new token (group 0 holds k_new)
    float sn;
    if constexpr (F8) {
      // quantise the new token as it will be stored; attend to the stored values
      float kf[8], vf[8], deq[8];
      uint32_t pr[4];
      bf16x8_to_f32(knew, kf);
      kq_scale = quantize_e4m3<8>(kf, gmask, LPS, pr);
      kcode = make_uint2(pr[0] | (pr[1] << 16), pr[2] | (pr[3] << 16));
      e4m3x8_to_f32(kcode, deq);
      sn = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) sn = fmaf(qf[i], deq[i] * kq_scale, sn);
      bf16x8_to_f32(vnew, vf);
      vq_scale = quantize_e4m3<8>(vf, gmask, LPS, pr);
      vcode = make_uint2(pr[0] | (pr[1] << 16), pr[2] | (pr[3] << 16));
      e4m3x8_to_f32(vcode, deq);
#pragma unroll
      for (int i = 0; i < 8; ++i) sm.vnew[l * 8 + i] = deq[i] * vq_scale;
    } else {
      sn = dot8(knew, qf);
    }
#pragma unroll
    for (int off = LPS / 2; off > 0; off >>= 1) sn += __shfl_xor_sync(gmask, sn, off);
    if (l == 0) sm.s_new = sn;
  }
  __syncthreads();
  // Every thread merges the warps' partials (max mc, sum lc); threads tid < D
  // also their output element oc, scaled to mc.
  float mc = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) mc = fmaxf(mc, sm.red_ml[w][0]);
  float lc = 0.f, oc = 0.f;
  const int gi = ((tid & (D - 1)) % 8) * LPS + (tid & (D - 1)) / 8;  // element tid % 8 of lane tid / 8
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const float mg = sm.red_ml[w][0];
    if (mg != -INFINITY) {
      const float wt = ex2(mg - mc);
      lc = fmaf(sm.red_ml[w][1], wt, lc);
      if (tid < D) oc = fmaf(sm.red_o[w][gi], wt, oc);
    }
  }
  const float s_new = sm.s_new;

  // ---- exact normaliser over the row and the new token.
  float M, invL, w_new, p_new, w_self = 0.f;
  if (a.segs > 1) {
    // hand the partial to the row's last CTA
    float* part = a.partial + (static_cast<size_t>(row) * a.segs + seg) * PS;
    if (tid < D) part[4 + tid] = oc;
    if (tid == 0) {
      part[0] = mc;
      part[1] = lc;
    }
    __threadfence();  // logits and partial visible before the arrival is counted
    __syncthreads();
    if (tid == 0) sm.is_last = atomicAdd(a.counter + row, 1) == a.segs - 1;
    __syncthreads();
    if (!sm.is_last) return;
    __threadfence();  // every other segment's writes are visible from here on
    if (tid == 0) {
      float Mx = s_new;
      for (int c = 0; c < a.segs; ++c)
        Mx = fmaxf(Mx, __ldcg(a.partial + (static_cast<size_t>(row) * a.segs + c) * PS));
      float L = ex2(s_new - Mx);
      for (int c = 0; c < a.segs; ++c) {
        const float* pc = a.partial + (static_cast<size_t>(row) * a.segs + c) * PS;
        const float mcs = __ldcg(pc);
        const float w = mcs == -INFINITY ? 0.f : ex2(mcs - Mx);
        sm.seg_w[c] = w;
        L = fmaf(__ldcg(pc + 1), w, L);
      }
      sm.M = Mx;
      sm.invL = 1.f / L;
      sm.w_new = ex2(s_new - Mx);
      sm.p_new = sm.w_new * sm.invL;
    }
    __syncthreads();
    M = sm.M;
    invL = sm.invL;
    w_new = sm.w_new;
    p_new = sm.p_new;
  } else {  // one CTA holds the whole row: every thread finishes from its own registers
    M = fmaxf(s_new, mc);
    w_self = mc == -INFINITY ? 0.f : ex2(mc - M);
    w_new = ex2(s_new - M);
    invL = 1.f / fmaf(lc, w_self, w_new);
    p_new = w_new * invL;
  }
  if (tid < D) {
    float acc = 0.f;
    if (a.segs > 1) {
      for (int c = 0; c < a.segs; ++c)
        acc = fmaf(__ldcg(a.partial + (static_cast<size_t>(row) * a.segs + c) * PS + 4 + tid),
                   sm.seg_w[c], acc);
    } else {
      acc = oc * w_self;
    }
    a.out[io + static_cast<size_t>(row) * D + tid] = fmaf(sm.vnew[tid], w_new, acc) * invL;
  }

  // Scores of every occupied slot of the row; this CTA's smallest candidate key.
  const int thr = t - a.r;  // candidates: positions <= t - r
  unsigned long long best = ~0ull;
  int bslot = -1;
#pragma unroll 1
  for (int jj = 0, i = tid; i < slot_end; ++jj, i += NT) {
    if (RING && !ring_full && !occ_g(i)) continue;
    float sc;
    int ps;
    if (solo && jj < kSoloRegs) {
#pragma unroll
      for (int q = 0; q < kSoloRegs; ++q)  // register arrays need static indices
        if (q == jj) {
          sc = sc_r[q];
          ps = ps_r[q];
        }
    } else {
      sc = a.score[rk + i];
      ps = !RING || i < a.h ? a.pos[rk + i] : 0;
    }
    if ((!RING || i < a.h) && (ps < 0 || ps >= t)) sm.bad = 1;  // reported below
    const float lg = solo ? solo_logits[i] : __ldcg(a.logits + rk + i);
    const float ns = sc + ex2(lg - M) * invL;
    a.score[rk + i] = ns;
    if constexpr (RING) {
      if (i == lv) sm.lv_score = ns;  // read by thread 0 after the barrier below
      if (i >= a.h) {
        if (i == lv && t >= a.r) ps = thr;  // the leaving token competes, position t - r
        else continue;                      // the rest of the window never does
      }
    }
    if (ps <= thr) {
      const unsigned long long key = pack_key(ns, ps);
      if (key < best) {
        best = key;
        bslot = i;
      }
    }
  }
  if (tid == 0 && a.r == 0) {  // with no recent window the new token competes too
    const unsigned long long key = pack_key(p_new, t);
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
    if (sm.bad && a.err) atomicOr(a.err, kErrBadState);
    const bool full = count >= a.k;
    int target, evict_pos = -1;
    if constexpr (RING) {
      // target: the heavy slot the leaving token moves into, or -1; the new
      // token always takes ring slot lv
      if (full) {
        evict_pos = static_cast<int>(b & 0xffffffffu);
        target = bs == lv ? -1 : bs;
      } else {
        target = t >= a.r ? nh : -1;  // not full: the leaving token joins the heavy slots
      }
    } else if (full) {
      evict_pos = b == ~0ull ? -1 : static_cast<int>(b & 0xffffffffu);
      target = bs == kNewSlot ? -1 : bs;  // a dropped new token leaves the cache unchanged
    } else {
      target = count;  // not full: append into the next empty slot
    }
    sm.target = target;
    int32_t* mw = a.meta + static_cast<size_t>(row) * 4;
    mw[0] = full ? a.k : count + 1;
    mw[1] = t + 1;
    mw[2] = evict_pos;
    if (a.evicted) a.evicted[static_cast<size_t>(step) * a.rows + row] = evict_pos;
    if constexpr (RING) {
      if (target >= 0) {
        a.pos[rk + target] = t - a.r;
        a.score[rk + target] = sm.lv_score;
      }
      a.pos[rk + lv] = t;  // written for readback; the kernel never reads it
      a.score[rk + lv] = p_new;
    } else if (target >= 0) {
      a.pos[rk + target] = t;
      a.score[rk + target] = p_new;  // after the score loop's write of this slot (barrier above)
    }
    if (a.segs > 1) a.counter[row] = 0;  // ready for the next step
  }
  __syncthreads();
  const int target = sm.target;
  if constexpr (RING) {
    if (g == 0) {
      __nv_bfloat16* Kc = static_cast<__nv_bfloat16*>(a.Kc);
      __nv_bfloat16* Vc = static_cast<__nv_bfloat16*>(a.Vc);
      const size_t src = (rk + lv) * D + l * 8;
      if (target >= 0) {  // the leaving token moves into the freed heavy slot first
        const uint4 kl = *reinterpret_cast<const uint4*>(Kc + src);
        const uint4 vl = *reinterpret_cast<const uint4*>(Vc + src);
        const size_t dst = (rk + target) * D + l * 8;
        *reinterpret_cast<uint4*>(Kc + dst) = kl;
        *reinterpret_cast<uint4*>(Vc + dst) = vl;
      }
      *reinterpret_cast<uint4*>(Kc + src) = knew;
      *reinterpret_cast<uint4*>(Vc + src) = vnew;
    }
  } else if (target >= 0 && g == 0) {
    const size_t dst = (rk + target) * D + l * 8;
    if constexpr (F8) {
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.Kc) + dst) = kcode;
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.Vc) + dst) = vcode;
      if (l == 0) {
        a.kscale[rk + target] = kq_scale;
        a.vscale[rk + target] = vq_scale;
      }
    } else {
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.Kc) + dst) = knew;
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.Vc) + dst) = vnew;
    }
  }
  // the slot, score and metadata writes of this step before the next reads them
  if constexpr (MULTI) __syncthreads();
  }  // step
}

}  // namespace
}  // namespace h2o
