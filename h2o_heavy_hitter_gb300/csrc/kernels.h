// Host-side launchers of the H2O kernels. Plain C++ types only; every launcher
// enqueues on `stream` and returns the launch status.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace h2o {

// log2(e): logits are carried in base 2 so that softmax uses exp2.
constexpr float kLog2e = 1.4426950408889634f;

// ---- decode ------------------------------------------------------------------
struct DecodeArgs {
  void* Kc;           // bf16 [rows][k][d] cached keys of one layer
  void* Vc;           // bf16 [rows][k][d] cached values
  float* score;       // [rows][k] accumulated scores
  int32_t* pos;       // [rows][k] positions (-1 empty)
  int32_t* meta;      // [rows][4] {filled, next position, last evicted, 0}
  const void* q;      // bf16 [rows][d]
  const void* k_new;  // bf16 [rows][d]
  const void* v_new;  // bf16 [rows][d]
  float* out;         // [rows][d]
  int32_t* err;       // device error word
  int k;              // slots per row (h + r)
  int r;              // recent window
  int chunk;          // slots handled by one CTA of a row's cluster
  float qscale;       // log2(e) / sqrt(d)
};

struct DecodeConfig {
  int cluster;  // CTAs per row (1, 2, 4, 8 or 16)
  int chunk;    // ceil(k / cluster)
  int stages;   // bulk-copy stages in flight per CTA
  size_t smem;  // dynamic shared memory per CTA
};

// Picks the launch shape for (rows, k, d) on a device with `num_sms` SMs.
// `cluster_override` / `stages_override` > 0 force a value.
DecodeConfig decode_config(int rows, int k, int d, int num_sms, int cluster_override,
                           int stages_override);
// Sets the kernel attributes a configuration needs (call once, outside capture).
cudaError_t decode_prepare(const DecodeConfig& cfg, int d);
cudaError_t decode_launch(const DecodeArgs& a, const DecodeConfig& cfg, int rows, int d,
                          cudaStream_t stream);

// ---- prefill -----------------------------------------------------------------
// Causal attention over `rows` rows of T tokens: O (fp32 [rows][T][d]) and the
// base-2 log-sum-exp of each query row's scaled logits (fp32 [rows][T]).
cudaError_t prefill_forward(const void* Q, const void* K, const void* V, int rows, int T, int d,
                            float* O, float* lse2, int32_t* err, cudaStream_t stream);
// Column sums of the causal probability matrix (fp32 [rows][T]), given lse2.
cudaError_t prefill_colsum(const void* Q, const void* K, const float* lse2, int rows, int T,
                           int d, float* colsum, int32_t* err, cudaStream_t stream);
// Top-h plus recent selection of every row into the cache's pos/score/meta.
cudaError_t prefill_select(const float* colsum, int rows, int T, int h, int r, float* score,
                           int32_t* pos, int32_t* meta, cudaStream_t stream);
// Copies the selected prompt K/V rows into the cache slots.
cudaError_t prefill_gather(const void* K, const void* V, int rows, int T, int d, int k,
                           const int32_t* pos, void* Kc, void* Vc, cudaStream_t stream);
// Resets rows to an empty cache (pos -1, score 0, meta {0, 0, -1, 0}).
cudaError_t cache_reset(int rows, int k, float* score, int32_t* pos, int32_t* meta,
                        cudaStream_t stream);

}  // namespace h2o
