// C ABI of the H2O heavy-hitter KV-cache library (declared in include/h2o.h).
//
// Host side only: argument checks, the per-layer state machine, cache
// allocation from PyTorch's CUDA caching allocator, and kernel launches on the
// current PyTorch stream. Every step of the policy runs in the CUDA kernels.
#include "h2o.h"

#include <c10/cuda/CUDACachingAllocator.h>
#include <c10/cuda/CUDAFunctions.h>
#include <c10/cuda/CUDAStream.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "kernels.h"

namespace {

thread_local std::string g_error;

int fail(int code, const std::string& msg) {
  g_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(H2O_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

cudaStream_t current_stream() { return c10::cuda::getCurrentCUDAStream().stream(); }

int env_int(const char* name) {
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : 0;
}

// Allocation-failure injection (h2o_test_fail_allocations): the next n device
// allocations of the library throw as an exhausted allocator would.
std::atomic<int> g_fail_allocs{0};

void* device_alloc(size_t bytes, cudaStream_t s) {
  for (int n = g_fail_allocs.load(); n > 0; n = g_fail_allocs.load())
    if (g_fail_allocs.compare_exchange_weak(n, n - 1)) throw std::bad_alloc();
  return c10::cuda::CUDACachingAllocator::raw_alloc_with_stream(bytes, s);
}

// One device allocation from PyTorch's caching allocator, freed on scope exit.
struct Scratch {
  void* p = nullptr;
  explicit Scratch(size_t bytes, cudaStream_t s) {
    if (bytes) p = device_alloc(bytes, s);
  }
  ~Scratch() {
    if (p) c10::cuda::CUDACachingAllocator::raw_delete(p);
  }
  Scratch(const Scratch&) = delete;
  Scratch& operator=(const Scratch&) = delete;
};

}  // namespace

struct h2o_ctx {
  int layers, batch, heads, d, h, r, k, rows;
  int device;
  int kv_format;              // H2O_KV_BF16 or H2O_KV_FP8
  bool ring = false;          // H2O_LAYOUT_RING: heavy slots, then the window as a circular queue
  size_t kv_elems_per_layer;  // rows * k * d
  size_t kv_elem_bytes;       // 2 (bf16) or 1 (E4M3 code)
  void* base = nullptr;       // single cache allocation
  uint8_t* K = nullptr;
  uint8_t* V = nullptr;
  float* kscale = nullptr;    // E4M3 cache: per-slot key scales [layers][rows][k]
  float* vscale = nullptr;    // E4M3 cache: per-slot value scales
  float* score = nullptr;
  int32_t* pos = nullptr;
  int32_t* meta = nullptr;
  float* logits = nullptr;    // decode scratch, per layer [rows][k]
  float* partial = nullptr;   // decode scratch, per layer [rows][segs][d + 4]
  int32_t* counter = nullptr; // decode scratch, per layer [rows], zero between steps
  int32_t* err = nullptr;     // device error word
  std::vector<int> prompt_len;  // per layer: -1 until prefilled
  int sms = 0;                // SMs of the device
  h2o::DecodeConfig dcfg{};   // one step per launch
  h2o::DecodeConfig mcfg{};   // several steps per launch (h2o_decode_steps)

  void* layer_K(int l) const { return K + static_cast<size_t>(l) * kv_elems_per_layer * kv_elem_bytes; }
  void* layer_V(int l) const { return V + static_cast<size_t>(l) * kv_elems_per_layer * kv_elem_bytes; }
  float* layer_kscale(int l) const { return kscale ? kscale + static_cast<size_t>(l) * rows * k : nullptr; }
  float* layer_vscale(int l) const { return vscale ? vscale + static_cast<size_t>(l) * rows * k : nullptr; }
  float* layer_score(int l) const { return score + static_cast<size_t>(l) * rows * k; }
  int32_t* layer_pos(int l) const { return pos + static_cast<size_t>(l) * rows * k; }
  int32_t* layer_meta(int l) const { return meta + static_cast<size_t>(l) * rows * 4; }
  float* layer_logits(int l) const { return logits + static_cast<size_t>(l) * rows * k; }
  float* layer_partial(int l) const {
    return partial + static_cast<size_t>(l) * rows * dcfg.segs * (d + 4);
  }
  int32_t* layer_counter(int l) const { return counter + static_cast<size_t>(l) * rows; }
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Prompt tensors and prefill outputs are read and written by TMA, which needs
// 16-byte aligned addresses.
bool tma_aligned(const void* a, const void* b, const void* c, const void* d) {
  auto ok = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; };
  return ok(a) && ok(b) && ok(c) && ok(d);
}

// A context's memory lives on the device that was current when it was
// created; its work must be enqueued there.
int check_device(const h2o_ctx* c) {
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (cur != c->device)
    return fail(H2O_EINVAL, "the context belongs to device " + std::to_string(c->device) +
                                " but device " + std::to_string(cur) + " is current");
  return H2O_OK;
}

int check_layer(const h2o_ctx* c, int layer) {
  if (!c) return fail(H2O_EINVAL, "null context");
  if (layer < 0 || layer >= c->layers) return fail(H2O_EINVAL, "layer out of range");
  return check_device(c);
}

int run_attention(const void* Q, const void* K, const void* V, int rows, int T,
                  const int32_t* lens, int heads, int d, float* out, float* colsum, int32_t* err,
                  cudaStream_t s) {
  Scratch lse(static_cast<size_t>(rows) * h2o::lse_stride(T) * sizeof(float), s);
  cudaError_t e = h2o::prefill_forward(Q, K, V, rows, T, lens, heads, d, out,
                                       static_cast<float*>(lse.p), err, s);
  if (e != cudaSuccess) return cuda_fail(e, "prefill forward launch");
  e = h2o::prefill_colsum(Q, K, static_cast<float*>(lse.p), rows, T, lens, heads, d, colsum, err, s);
  if (e != cudaSuccess) return cuda_fail(e, "prefill column-sum launch");
  return H2O_OK;
}

// Prefill of one layer over prompts padded to T tokens; `lens` (device, one
// length per batch entry) or null for prompts of exactly T tokens.
int prefill_layer(h2o_ctx* c, int layer, const void* Q, const void* K, const void* V, int T,
                  const int32_t* lens, float* out) {
  if (int rc = check_layer(c, layer)) return rc;
  if (T < 0 || T > H2O_MAX_T) return fail(H2O_EINVAL, "T out of range");
  if (c->prompt_len[layer] >= 0)
    return fail(H2O_ESTATE, "layer already prefilled: h2o_reset it before a new prompt");
  cudaStream_t s = current_stream();
  cudaError_t e;
  if (T == 0) {
    e = h2o::cache_reset(c->rows, c->k, c->layer_score(layer), c->layer_pos(layer),
                         c->layer_meta(layer), s);
    if (e != cudaSuccess) return cuda_fail(e, "cache reset");
    c->prompt_len[layer] = 0;
    return H2O_OK;
  }
  if (!Q || !K || !V || !out) return fail(H2O_EINVAL, "null Q, K, V or out");
  if (!tma_aligned(Q, K, V, out)) return fail(H2O_EINVAL, "Q, K, V and out must be 16-byte aligned");
  const int heads = c->heads;
  try {
    Scratch colsum(static_cast<size_t>(c->rows) * T * sizeof(float), s);
    int rc = run_attention(Q, K, V, c->rows, T, lens, heads, c->d, out,
                           static_cast<float*>(colsum.p), c->err, s);
    if (rc) return rc;
    e = h2o::prefill_select(static_cast<float*>(colsum.p), c->rows, T, lens, heads, c->h, c->r,
                            c->ring, c->layer_score(layer), c->layer_pos(layer),
                            c->layer_meta(layer), c->err, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill select launch");
    e = c->kv_format == H2O_KV_FP8
            ? h2o::prefill_gather_fp8(K, V, c->rows, T, c->d, c->k, c->layer_pos(layer),
                                      c->layer_K(layer), c->layer_V(layer),
                                      c->layer_kscale(layer), c->layer_vscale(layer), c->err, s)
            : h2o::prefill_gather(K, V, c->rows, T, c->d, c->k, c->layer_pos(layer),
                                  c->layer_K(layer), c->layer_V(layer), c->err, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill gather launch");
  } catch (const std::exception& ex) {
    return fail(H2O_ENOMEM, std::string("prefill scratch allocation failed: ") + ex.what());
  }
  c->prompt_len[layer] = T;
  return H2O_OK;
}

}  // namespace

extern "C" {

const char* h2o_last_error(void) { return g_error.c_str(); }

int h2o_create(int layers, int batch, int heads, int head_dim, int h, int r, h2o_ctx** out) {
  return h2o_create_ex(layers, batch, heads, head_dim, h, r, H2O_KV_BF16, out);
}

int h2o_create_ex(int layers, int batch, int heads, int head_dim, int h, int r, int kv_format,
                  h2o_ctx** out) {
  if (!out) return fail(H2O_EINVAL, "null output pointer");
  *out = nullptr;
  const bool ring = (kv_format & H2O_LAYOUT_RING) != 0;
  kv_format &= ~H2O_LAYOUT_RING;
  if (kv_format != H2O_KV_BF16 && kv_format != H2O_KV_FP8)
    return fail(H2O_EINVAL, "kv_format must be H2O_KV_BF16 or H2O_KV_FP8, optionally | H2O_LAYOUT_RING");
  if (ring && (kv_format != H2O_KV_BF16 || r < 1))
    return fail(H2O_EINVAL, "H2O_LAYOUT_RING needs the bf16 cache and r >= 1");
  if (layers < 1 || batch < 1 || heads < 1) return fail(H2O_EINVAL, "layers, batch and heads must be >= 1");
  if (head_dim != 64 && head_dim != 128) return fail(H2O_EINVAL, "head_dim must be 64 or 128");
  if (h < 0 || r < 0 || h + r < 1 || h + r > H2O_MAX_K)
    return fail(H2O_EINVAL, "need h >= 0, r >= 0 and 1 <= h + r <= H2O_MAX_K");
  const long rows_l = static_cast<long>(batch) * heads;
  if (rows_l > (1L << 30)) return fail(H2O_EINVAL, "batch * heads too large");

  auto* c = new h2o_ctx();
  c->layers = layers;
  c->batch = batch;
  c->heads = heads;
  c->d = head_dim;
  c->h = h;
  c->r = r;
  c->k = h + r;
  c->rows = static_cast<int>(rows_l);
  c->kv_format = kv_format;
  c->ring = ring;
  c->kv_elem_bytes = kv_format == H2O_KV_FP8 ? 1 : 2;
  c->prompt_len.assign(layers, -1);
  try {
    c->device = c10::cuda::current_device();
  } catch (const std::exception& ex) {
    delete c;
    return fail(H2O_ECUDA, std::string("no CUDA device: ") + ex.what());
  }
  int sms = 0, l2 = 0;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, c->device);
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e, "cudaDeviceGetAttribute");
  }

  h2o::DecodeTuning tune{env_int("H2O_DECODE_THREADS"), env_int("H2O_DECODE_UNROLL"),
                         env_int("H2O_DECODE_SEGS"), env_int("H2O_DECODE_PDL"),
                         env_int("H2O_DECODE_PIPE"), env_int("H2O_DECODE_PREFETCH")};
  c->sms = sms;
  c->dcfg = h2o::decode_config(c->rows, c->k, c->d, sms, tune, kv_format == H2O_KV_FP8, l2);
  c->mcfg = h2o::decode_multi_config(c->rows, c->k, c->d, sms, kv_format == H2O_KV_FP8);

  const size_t L = layers, R = c->rows, K = c->k, D = head_dim;
  c->kv_elems_per_layer = R * K * D;
  const size_t kv_bytes = align_up(L * R * K * D * c->kv_elem_bytes, 256);
  const size_t sc_bytes = align_up(L * R * K * 4, 256);
  const size_t qs_bytes = kv_format == H2O_KV_FP8 ? sc_bytes : 0;  // per-slot scales
  const size_t meta_bytes = align_up(L * R * 16, 256);
  const size_t part_bytes = align_up(L * R * c->dcfg.segs * (D + 4) * 4, 256);
  const size_t cnt_bytes = align_up(L * R * 4, 256);
  const size_t total =
      2 * kv_bytes + 3 * sc_bytes + 2 * qs_bytes + meta_bytes + part_bytes + cnt_bytes + 256;
  cudaStream_t s = current_stream();
  try {
    c->base = device_alloc(total, s);
  } catch (const std::exception& ex) {
    delete c;
    return fail(H2O_ENOMEM, std::string("cache allocation failed: ") + ex.what());
  }
  char* p = static_cast<char*>(c->base);
  c->K = reinterpret_cast<uint8_t*>(p);
  p += kv_bytes;
  c->V = reinterpret_cast<uint8_t*>(p);
  p += kv_bytes;
  c->score = reinterpret_cast<float*>(p);
  p += sc_bytes;
  c->pos = reinterpret_cast<int32_t*>(p);
  p += sc_bytes;
  c->logits = reinterpret_cast<float*>(p);
  p += sc_bytes;
  c->meta = reinterpret_cast<int32_t*>(p);
  p += meta_bytes;
  c->partial = reinterpret_cast<float*>(p);
  p += part_bytes;
  c->counter = reinterpret_cast<int32_t*>(p);
  p += cnt_bytes;
  if (qs_bytes) {
    c->kscale = reinterpret_cast<float*>(p);
    p += qs_bytes;
    c->vscale = reinterpret_cast<float*>(p);
    p += qs_bytes;
  }
  c->err = reinterpret_cast<int32_t*>(p);

  e = cudaMemsetAsync(c->err, 0, sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->K, 0, 2 * kv_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->counter, 0, cnt_bytes, s);
  if (e == cudaSuccess && qs_bytes) e = cudaMemsetAsync(c->kscale, 0, 2 * qs_bytes, s);
  for (int l = 0; l < layers && e == cudaSuccess; ++l)
    e = h2o::cache_reset(c->rows, c->k, c->layer_score(l), c->layer_pos(l), c->layer_meta(l), s);
  if (e != cudaSuccess) {
    h2o_destroy(c);
    return cuda_fail(e, "cache initialisation");
  }
  *out = c;
  return H2O_OK;
}

void h2o_destroy(h2o_ctx* c) {
  if (!c) return;
  if (c->base) {
    cudaStreamSynchronize(current_stream());
    c10::cuda::CUDACachingAllocator::raw_delete(c->base);
  }
  delete c;
}

int h2o_prefill(h2o_ctx* c, int layer, const void* Q, const void* K, const void* V, int T,
                float* out) {
  return prefill_layer(c, layer, Q, K, V, T, nullptr, out);
}

int h2o_prefill_ragged(h2o_ctx* c, int layer, const void* Q, const void* K, const void* V,
                       int T_max, const int32_t* lens, float* out) {
  if (T_max > 0 && !lens) return fail(H2O_EINVAL, "null lens");
  return prefill_layer(c, layer, Q, K, V, T_max, lens, out);
}

int h2o_prefill_attention(const void* Q, const void* K, const void* V, int rows, int T,
                          int head_dim, float* out, float* score) {
  if (rows < 0 || T < 0 || T > H2O_MAX_T) return fail(H2O_EINVAL, "rows or T out of range");
  if (head_dim != 64 && head_dim != 128) return fail(H2O_EINVAL, "head_dim must be 64 or 128");
  if (static_cast<long>(rows) * T == 0) return H2O_OK;
  if (!Q || !K || !V || !out || !score) return fail(H2O_EINVAL, "null pointer");
  if (!tma_aligned(Q, K, V, out)) return fail(H2O_EINVAL, "Q, K, V and out must be 16-byte aligned");
  int32_t* err = nullptr;
  cudaError_t e = h2o::attention_error_word(&err);
  if (e != cudaSuccess) return cuda_fail(e, "error word lookup");
  try {
    return run_attention(Q, K, V, rows, T, nullptr, 1, head_dim, out, score, err,
                         current_stream());
  } catch (const std::exception& ex) {
    return fail(H2O_ENOMEM, std::string("scratch allocation failed: ") + ex.what());
  }
}

int h2o_prefill_attention_noalloc(const void* Q, const void* K, const void* V, int rows, int T,
                                  int head_dim, float* out, float* score, void* stream) {
  if (rows < 0 || T < 0 || T > H2O_MAX_T) return fail(H2O_EINVAL, "rows or T out of range");
  if (head_dim != 64 && head_dim != 128) return fail(H2O_EINVAL, "head_dim must be 64 or 128");
  const long need = static_cast<long>(rows) * h2o::lse_stride(T);
  if (need > H2O_NOALLOC_MAX_LSE)
    return fail(H2O_EINVAL, "rows * ceil(T / 128) * 128 = " + std::to_string(need) +
                                " exceeds the fixed scratch of H2O_NOALLOC_MAX_LSE = " +
                                std::to_string(H2O_NOALLOC_MAX_LSE) + " floats");
  if (need == 0) return H2O_OK;
  if (!Q || !K || !V || !out || !score) return fail(H2O_EINVAL, "null pointer");
  if (!tma_aligned(Q, K, V, out)) return fail(H2O_EINVAL, "Q, K, V and out must be 16-byte aligned");
  float* lse = nullptr;
  cudaError_t e = h2o::noalloc_lse_scratch(&lse);
  if (e != cudaSuccess) return cuda_fail(e, "scratch address lookup");
  int32_t* err = nullptr;
  e = h2o::attention_error_word(&err);
  if (e != cudaSuccess) return cuda_fail(e, "error word lookup");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = h2o::prefill_forward(Q, K, V, rows, T, nullptr, 1, head_dim, out, lse, err, s);
  if (e != cudaSuccess) return cuda_fail(e, "prefill forward launch");
  e = h2o::prefill_colsum(Q, K, lse, rows, T, nullptr, 1, head_dim, score, err, s);
  if (e != cudaSuccess) return cuda_fail(e, "prefill column-sum launch");
  return H2O_OK;
}

// Reads, then clears, a device error word on `s` after the stream's work so
// far; H2O_EDEVICE if it was set. Allocates nothing.
static int check_error_word(int32_t* word_dev, cudaStream_t s) {
  int32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, word_dev, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
  if (word != 0) {
    cudaMemsetAsync(word_dev, 0, sizeof(int32_t), s);
    char buf[128];
    std::snprintf(buf, sizeof(buf), "device error word 0x%x (1 = wait timeout, 2 = bad state, 4 = length out of range)", word);
    return fail(H2O_EDEVICE, buf);
  }
  return H2O_OK;
}

int h2o_attention_sync_check(void* stream) {
  int32_t* err = nullptr;
  cudaError_t e = h2o::attention_error_word(&err);
  if (e != cudaSuccess) return cuda_fail(e, "error word lookup");
  return check_error_word(err, static_cast<cudaStream_t>(stream));
}

int h2o_attention_test_wait_limit(void* stream) {
  int32_t* err = nullptr;
  cudaError_t e = h2o::attention_error_word(&err);
  if (e != cudaSuccess) return cuda_fail(e, "error word lookup");
  e = h2o::wait_limit_probe(err, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait-limit probe launch");
  return H2O_OK;
}

void h2o_forget_device_state(void) { h2o::forget_device_state(); }

int h2o_test_fail_allocations(int n) {
  if (n < 0) return fail(H2O_EINVAL, "n must be >= 0");
  g_fail_allocs.store(n);
  return H2O_OK;
}

}  // extern "C"

namespace {

h2o::DecodeArgs decode_args(h2o_ctx* c, int layer) {
  h2o::DecodeArgs a{};
  a.Kc = c->layer_K(layer);
  a.Vc = c->layer_V(layer);
  a.kscale = c->layer_kscale(layer);  // null for a bf16 cache
  a.vscale = c->layer_vscale(layer);
  a.score = c->layer_score(layer);
  a.pos = c->layer_pos(layer);
  a.meta = c->layer_meta(layer);
  a.logits = c->layer_logits(layer);
  a.partial = c->layer_partial(layer);
  a.counter = c->layer_counter(layer);
  a.err = c->err;
  a.rows = c->rows;
  a.steps = 1;
  a.k = c->k;
  a.h = c->h;
  a.r = c->r;
  a.segs = c->dcfg.segs;
  a.seg_len = c->dcfg.seg_len;
  a.qscale = h2o::kLog2e / std::sqrt(static_cast<float>(c->d));
  a.prefetch = c->dcfg.prefetch ? 1 : 0;
  return a;
}

}  // namespace

extern "C" {

int h2o_decode_step(h2o_ctx* c, int layer, const void* q, const void* k_new, const void* v_new,
                    float* out) {
  if (int rc = check_layer(c, layer)) return rc;
  if (!q || !k_new || !v_new || !out) return fail(H2O_EINVAL, "null q, k_new, v_new or out");
  if (c->prompt_len[layer] < 0) return fail(H2O_ESTATE, "decode step before prefill of this layer");
  h2o::DecodeArgs a = decode_args(c, layer);
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.out = out;
  cudaError_t e = c->ring ? h2o::decode_ring_launch(a, c->dcfg, c->rows, c->d, current_stream())
                          : h2o::decode_launch(a, c->dcfg, c->rows, c->d, current_stream());
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return H2O_OK;
}

int h2o_decode_steps(h2o_ctx* c, int layer, int steps, const void* q, const void* k_new,
                     const void* v_new, float* out, int32_t* evicted) {
  if (int rc = check_layer(c, layer)) return rc;
  if (steps < 0) return fail(H2O_EINVAL, "steps must be >= 0");
  if (steps == 0) return H2O_OK;
  if (!q || !k_new || !v_new || !out) return fail(H2O_EINVAL, "null q, k_new, v_new or out");
  if (c->prompt_len[layer] < 0) return fail(H2O_ESTATE, "decode step before prefill of this layer");
  h2o::DecodeArgs a = decode_args(c, layer);
  cudaStream_t s = current_stream();
  cudaError_t e;
  // One launch for all steps needs one CTA per row; with fewer rows than SMs
  // and long rows, per-step launches that split the rows over several CTAs
  // move the bytes faster (128 rows of 4096 slots: 49 against 53 us a step).
  const bool split_better = c->rows < c->sms && c->k >= 1024;
  if (c->k <= h2o::kMultiMaxSlots && !c->ring && !split_better) {
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.out = out;
    a.evicted = evicted;
    a.steps = steps;
    a.segs = 1;
    a.seg_len = c->k;
    e = h2o::decode_multi_launch(a, c->mcfg, c->rows, c->d, s);
    if (e != cudaSuccess) return cuda_fail(e, "multi-step decode launch");
    return H2O_OK;
  }
  // budgets too large for one CTA per row, long rows on few SMs, or the ring
  // layout: one launch per step
  const size_t in_step = static_cast<size_t>(c->rows) * c->d;
  for (int i = 0; i < steps; ++i) {
    a.q = static_cast<const uint16_t*>(q) + i * in_step;
    a.k_new = static_cast<const uint16_t*>(k_new) + i * in_step;
    a.v_new = static_cast<const uint16_t*>(v_new) + i * in_step;
    a.out = out + i * in_step;
    a.evicted = evicted ? evicted + static_cast<size_t>(i) * c->rows : nullptr;
    e = c->ring ? h2o::decode_ring_launch(a, c->dcfg, c->rows, c->d, s)
                : h2o::decode_launch(a, c->dcfg, c->rows, c->d, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  }
  return H2O_OK;
}

int h2o_reset(h2o_ctx* c, int layer) {
  if (!c) return fail(H2O_EINVAL, "null context");
  if (layer < -1 || layer >= c->layers) return fail(H2O_EINVAL, "layer out of range");
  if (int rc = check_device(c)) return rc;
  const int l0 = layer < 0 ? 0 : layer, l1 = layer < 0 ? c->layers : layer + 1;
  cudaStream_t s = current_stream();
  for (int l = l0; l < l1; ++l) {
    cudaError_t e = h2o::cache_reset(c->rows, c->k, c->layer_score(l), c->layer_pos(l),
                                     c->layer_meta(l), s);
    if (e != cudaSuccess) return cuda_fail(e, "cache reset");
    c->prompt_len[l] = -1;
  }
  return H2O_OK;
}

int h2o_cache_positions(h2o_ctx* c, int layer, int32_t* host_pos) {
  if (int rc = check_layer(c, layer)) return rc;
  if (!host_pos) return fail(H2O_EINVAL, "null host buffer");
  cudaStream_t s = current_stream();
  cudaError_t e = cudaMemcpyAsync(host_pos, c->layer_pos(layer),
                                  static_cast<size_t>(c->rows) * c->k * sizeof(int32_t),
                                  cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "positions copy");
  return h2o_sync_check(c);
}

int h2o_last_evicted(h2o_ctx* c, int layer, int32_t* host_pos) {
  if (int rc = check_layer(c, layer)) return rc;
  if (!host_pos) return fail(H2O_EINVAL, "null host buffer");
  cudaStream_t s = current_stream();
  cudaError_t e = cudaMemcpy2DAsync(host_pos, sizeof(int32_t), c->layer_meta(layer) + 2,
                                    4 * sizeof(int32_t), sizeof(int32_t), c->rows,
                                    cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "evicted-position copy");
  return h2o_sync_check(c);
}

int h2o_cache_view(h2o_ctx* c, int layer, void** K, void** V, float** score, int32_t** pos,
                   int32_t** meta) {
  if (int rc = check_layer(c, layer)) return rc;
  if (K) *K = c->layer_K(layer);
  if (V) *V = c->layer_V(layer);
  if (score) *score = c->layer_score(layer);
  if (pos) *pos = c->layer_pos(layer);
  if (meta) *meta = c->layer_meta(layer);
  return H2O_OK;
}

int h2o_cache_scales(h2o_ctx* c, int layer, float** k_scale, float** v_scale) {
  if (int rc = check_layer(c, layer)) return rc;
  if (c->kv_format != H2O_KV_FP8) return fail(H2O_EINVAL, "the cache of this context is bf16: no scales");
  if (k_scale) *k_scale = c->layer_kscale(layer);
  if (v_scale) *v_scale = c->layer_vscale(layer);
  return H2O_OK;
}

int h2o_cache_dims(h2o_ctx* c, int* k, int* rows) {
  if (!c) return fail(H2O_EINVAL, "null context");
  if (k) *k = c->k;
  if (rows) *rows = c->rows;
  return H2O_OK;
}

int h2o_test_wait_limit(h2o_ctx* c) {
  if (!c) return fail(H2O_EINVAL, "null context");
  if (int rc = check_device(c)) return rc;
  cudaError_t e = h2o::wait_limit_probe(c->err, current_stream());
  if (e != cudaSuccess) return cuda_fail(e, "wait-limit probe launch");
  return H2O_OK;
}

int h2o_sync_check(h2o_ctx* c) {
  if (!c) return fail(H2O_EINVAL, "null context");
  if (int rc = check_device(c)) return rc;
  return check_error_word(c->err, current_stream());
}

}  // extern "C"
