// Host-side launchers of the H2O kernels. Plain C++ types only; every launcher
// enqueues on `stream` and returns the launch status.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace h2o {

// log2(e): logits are carried in base 2 so that softmax uses exp2.
constexpr float kLog2e = 1.4426950408889634f;

// ---- decode ------------------------------------------------------------------
constexpr int kMaxDecodeSegs = 64;  // most CTAs one row's decode step is split over

struct DecodeArgs {
  void* Kc;           // [rows][k][d] cached keys of one layer: bf16, or E4M3 codes
  void* Vc;           // [rows][k][d] cached values (same format)
  float* kscale;      // E4M3 cache only: [rows][k] per-slot key scales (null for bf16)
  float* vscale;      // E4M3 cache only: [rows][k] per-slot value scales
  float* score;       // [rows][k] accumulated scores
  int32_t* pos;       // [rows][k] positions (-1 empty)
  int32_t* meta;      // [rows][4] {filled, next position, last evicted, 0}
  float* logits;      // [rows][k] scratch: this step's base-2 logits
  float* partial;     // [rows][segs][d + 4] scratch: {max, sum, -, -, output[d]} per segment
  int32_t* counter;   // [rows] scratch: segments arrived this step (0 between steps)
  const void* q;      // bf16 [steps][rows][d]
  const void* k_new;  // bf16 [steps][rows][d]
  const void* v_new;  // bf16 [steps][rows][d]
  float* out;         // [steps][rows][d]
  int32_t* evicted;   // [steps][rows] evicted position (-1 none) of each step, or null
  int32_t* err;       // device error word: kErrBadState when a row's cache state is inconsistent
  int rows;           // rows of the layer
  int steps;          // steps per launch (1 except for the multi-step launcher)
  int k;              // slots per row (h + r)
  int h;              // heavy slots (ring layout: slots [0, h), the window after them)
  int r;              // recent window
  int segs;           // CTAs per row
  int seg_len;        // slots per segment (the last may be shorter)
  float qscale;       // log2(e) / sqrt(d)
  int prefetch;       // pull the CTA's K/V slots into L2 before the dependency wait
};

// Launch shape of the decode kernel. Zero / out-of-range values pick defaults.
struct DecodeTuning {
  int threads;  // 128 or 256 threads per CTA
  int unroll;   // slots per group per batch (2 or 4; 8 with an E4M3 cache)
  int segs;     // CTAs per row; 0 = automatic
  int pdl;      // < 0: launch without programmatic dependent launch
  int pipe;     // > 0: two batches per group in flight; < 0: one; 0: automatic
  int prefetch; // > 0: L2 prefetch before the dependency wait; < 0: none; 0: automatic
};

struct DecodeConfig {
  bool pdl;     // programmatic dependent launch (overlaps the previous kernel's tail)
  bool pipe;    // two batches per group in flight
  bool prefetch;  // K/V slots pulled into L2 before the dependency wait
  int threads, unroll;
  int segs;     // CTAs per row
  int seg_len;  // slots per segment
  size_t smem;  // dynamic shared memory per CTA (logits of a single-CTA row)
};

// Picks the launch shape for (rows, k, d) on a device with `num_sms` SMs and
// an L2 of `l2_bytes`.
DecodeConfig decode_config(int rows, int k, int d, int num_sms, const DecodeTuning& tune,
                           bool fp8, long long l2_bytes);
cudaError_t decode_launch(const DecodeArgs& a, const DecodeConfig& cfg, int rows, int d,
                          cudaStream_t stream);
// The same step for a cache in the ring layout (bf16, r >= 1): heavy slots
// [0, h), the token at recent position p in slot h + p mod r.
cudaError_t decode_ring_launch(const DecodeArgs& a, const DecodeConfig& cfg, int rows, int d,
                               cudaStream_t stream);

// Several steps in one launch: one CTA per row runs a.steps consecutive steps
// (needs k <= kMultiMaxSlots, whose logits stay in shared memory). The launch
// shape follows decode_config with one segment per row: 128 threads for many
// rows, else 256 with two batches in flight.
constexpr int kMultiMaxSlots = 8192;
DecodeConfig decode_multi_config(int rows, int k, int d, int num_sms, bool fp8);
cudaError_t decode_multi_launch(const DecodeArgs& a, const DecodeConfig& cfg, int rows, int d,
                                cudaStream_t stream);

// ---- prefill -----------------------------------------------------------------
// Row stride (floats) of the per-row log-sum-exp scratch: T rounded up to a
// whole 128-token tile, so every tile's slice is 512-byte aligned.
inline int lse_stride(int T) { return (T + 127) / 128 * 128; }

// Causal attention over `rows` rows of T tokens: O (fp32 [rows][T][d]) and the
// negated base-2 log-sum-exp of each query row's scaled logits, -lse2
// (fp32 [rows][lse_stride(T)]). Ragged batch: with `lens` (device int32, one
// length per batch entry of `heads` rows) row i holds a prompt of
// lens[i / heads] tokens padded to T; results past a row's length are not
// written (O rows of the last 32-token box may be) and the padding of Q, K, V
// must be finite (padded keys enter the MMAs with probability 0).
cudaError_t prefill_forward(const void* Q, const void* K, const void* V, int rows, int T,
                            const int32_t* lens, int heads, int d, float* O, float* lse2,
                            int32_t* err, cudaStream_t stream);
// Column sums of the causal probability matrix (fp32 [rows][T]), given -lse2.
cudaError_t prefill_colsum(const void* Q, const void* K, const float* lse2, int rows, int T,
                           const int32_t* lens, int heads, int d, float* colsum, int32_t* err,
                           cudaStream_t stream);
// Device address of the library's fixed log-sum-exp array used by
// h2o_prefill_attention_noalloc (H2O_NOALLOC_MAX_LSE floats). Looked up once
// per device, with that device current, and cached.
cudaError_t noalloc_lse_scratch(float** out);
// Device address of the library-level error word (int32) that the cache-free
// prefill entry points pass to their kernels; looked up like the array above.
cudaError_t attention_error_word(int32_t** out);
// Drops every cached per-device address and kernel attribute, so that the
// next call looks them up again (after a device reset).
void forget_device_state();

// Top-h plus recent selection of every row into the cache's pos/score/meta
// (colsum rows T floats apart; per-row lengths as for prefill_forward; a
// length outside [0, T] is clamped and sets kErrBadLength in *err). `ring`:
// kept tokens older than the window fill slots [0, h) in ascending order and
// a window token at position p goes to slot h + p mod r; otherwise every kept
// token is compacted in ascending order from slot 0.
cudaError_t prefill_select(const float* colsum, int rows, int T, const int32_t* lens, int heads,
                           int h, int r, bool ring, float* score, int32_t* pos, int32_t* meta,
                           int32_t* err, cudaStream_t stream);
// Copies the selected prompt K/V rows into the cache slots (a position outside
// [0, T) is skipped and sets kErrBadState in *err).
cudaError_t prefill_gather(const void* K, const void* V, int rows, int T, int d, int k,
                           const int32_t* pos, void* Kc, void* Vc, int32_t* err,
                           cudaStream_t stream);
// Resets rows to an empty cache (pos -1, score 0, meta {0, 0, -1, 0}).
// E4M3 cache: the kept tokens quantised into their slots, codes plus one fp32
// scale per slot for K and for V.
cudaError_t prefill_gather_fp8(const void* K, const void* V, int rows, int T, int d, int k,
                               const int32_t* pos, void* Kc, void* Vc, float* kscale,
                               float* vscale, int32_t* err, cudaStream_t stream);
cudaError_t cache_reset(int rows, int k, float* score, int32_t* pos, int32_t* meta,
                        cudaStream_t stream);
// One kernel whose bounded wait is never satisfied: it gives up after the
// wait limit and sets kErrWaitTimeout in *err (the failure path, on demand).
cudaError_t wait_limit_probe(int32_t* err, cudaStream_t stream);

}  // namespace h2o
