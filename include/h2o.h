/*
 * h2o.h - C ABI of the GB300 (sm_103a) H2O heavy-hitter KV-cache library.
 *
 * Sources (page title and section):
 *   [H2O] "H2O: Heavy-Hitter Oracle for Efficient Generative Inference of Large
 *         Language Models", section-by-section summary page of arXiv 2306.14048v3.
 *
 * The policy keeps, for every (layer, batch row, head) "row", at most
 * k = h + r cached tokens: h heavy hitters and the r most recent tokens
 * ([H2O] A, System Details). A token's accumulated score is the running sum of
 * the softmax probabilities it has received ([H2O] 1, 3.2). At most one token is
 * evicted per decoding step and the cache never exceeds k ([H2O] TL;DR, 2).
 *
 * Conventions shared by every entry point
 *   - Return value: H2O_OK (0) on success, a negative H2O_E* code on failure.
 *     h2o_last_error() then returns a message for the calling thread. No entry
 *     point traps or aborts; device kernels never trap. Bounded device waits
 *     that give up set a device error word that h2o_sync_check() reports.
 *   - Device pointers are CUDA device addresses on the current device; host
 *     pointers are ordinary CPU memory. Every buffer passed in stays owned by
 *     the caller and is only accessed by work the call enqueues. A context
 *     belongs to the device that was current when it was created: an entry
 *     point given a context returns H2O_EINVAL while another device is current.
 *   - All device work is enqueued, asynchronously, on the calling thread's
 *     current PyTorch CUDA stream (c10::cuda::getCurrentCUDAStream()). The
 *     caller must have initialised PyTorch's CUDA state on that device
 *     (torch.cuda.init() or any CUDA tensor). Only h2o_cache_positions,
 *     h2o_last_evicted and h2o_sync_check synchronise with the host.
 *   - The library owns the cache. It allocates it from PyTorch's CUDA caching
 *     allocator and frees it in h2o_destroy. PyTorch serves for nothing else.
 *   - Prompt tensors Q, K, V and prefill outputs `out` are moved by TMA and
 *     must be 16-byte aligned (any CUDA allocation is); otherwise H2O_EINVAL.
 *   - Layouts: Q, K, V of a prompt are bf16, contiguous [batch, heads, T, d];
 *     decode inputs q, k_new, v_new are bf16, contiguous [batch, heads, d];
 *     outputs are fp32 in the same layouts. head_dim d is 64 or 128. Logits
 *     are scaled by 1/sqrt(d).
 *   - Position t counts tokens of a row from 0: prompt tokens are 0 .. T-1 and
 *     decode step s processes position T + s.
 */
#ifndef H2O_H
#define H2O_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define H2O_OK 0
#define H2O_EINVAL (-1)  /* bad argument (null pointer, size out of range, layer out of range) */
#define H2O_ESTATE (-2)  /* call not valid in the current state (decode before prefill, or a
                            second prefill of a layer without h2o_reset) */
#define H2O_ENOMEM (-3)  /* device allocation failed */
#define H2O_ECUDA (-4)   /* a CUDA runtime call or kernel launch failed */
#define H2O_EDEVICE (-5) /* a kernel reported an error through the device error word */

#define H2O_MAX_T (1 << 20)  /* longest prompt accepted by h2o_prefill */
#define H2O_MAX_K 32768      /* largest budget h + r accepted by h2o_create */

#define H2O_KV_BF16 0  /* cache keys and values stored as bf16 (h2o_create) */
#define H2O_KV_FP8 1   /* cache keys and values stored as E4M3 codes with per-token scales */
#define H2O_LAYOUT_RING 0x100 /* OR into kv_format: heavy slots, then the window as a circular queue */

typedef struct h2o_ctx h2o_ctx; /* opaque; created by h2o_create, freed by h2o_destroy */

/*
 * h2o_create - allocate the cache of a model: `layers` layers of batch x heads
 * rows, each with a budget of h heavy-hitter plus r recent tokens ([H2O] A,
 * System Details: preallocated cache with a heavy-hitter and a recent region).
 *
 * Per layer the cache holds, for rows = batch * heads and k = h + r slots:
 *   K, V   bf16  [rows][k][d]   cached keys / values, slot-indexed (E4M3
 *                               codes, uint8, for an h2o_create_ex FP8 cache)
 *   score  fp32  [rows][k]      accumulated attention score of each slot
 *   pos    int32 [rows][k]      token position held by each slot (-1 = empty)
 *   meta   int32 [rows][4]      {filled slots, next position t, last evicted position (-1 none), 0}
 * Slots [0, filled) are occupied; slot order carries no meaning.
 *
 * Arguments: layers >= 1, batch >= 1, heads >= 1, head_dim in {64, 128},
 * h >= 0, r >= 0, 1 <= h + r <= H2O_MAX_K. *out receives the new context.
 * Errors: H2O_EINVAL, H2O_ENOMEM, H2O_ECUDA. On error *out is set to NULL.
 */
int h2o_create(int layers, int batch, int heads, int head_dim, int h, int r, h2o_ctx** out);

/*
 * h2o_create_ex - h2o_create with a choice of cache storage. The pages report
 * that H2O combines with quantisation of the KV cache and that the combination
 * beats either alone ([H2O] 5, Empirical Evaluation), without fixing a scheme.
 * kv_format H2O_KV_FP8 stores every cached token's key and value vectors as
 * E4M3 codes (OCP 8-bit floating point: 1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits, largest finite value 448) with one fp32 scale per vector:
 * scale = amax / 448 and code = E4M3(x * (448 / amax)), round to nearest even,
 * saturated; a zero vector has scale 0. The arithmetic is fp32 with one
 * rounding per operation. Prefill attention still runs on the full-precision
 * prompt and the kept tokens are quantised as they enter the cache; a decode
 * step quantises the new token first and attends to the stored (dequantised)
 * values of every cached token, the new one included. Per layer the cache then
 * holds K, V as uint8 [rows][k][d] and two fp32 [rows][k] scale arrays
 * (h2o_cache_scales), 2d + 8 bytes per slot instead of 4d.
 * kv_format H2O_KV_BF16 is h2o_create. Other arguments and errors as for
 * h2o_create; an unknown kv_format gives H2O_EINVAL.
 *
 * kv_format H2O_KV_BF16 | H2O_LAYOUT_RING (needs r >= 1) lays each row's
 * slots out as the pages' implementation does ([H2O] A, System Details: a
 * heavy-hitter region and the recent tokens in a circular queue): heavy slots
 * [0, h) in use from slot 0, and the token at recent position p in slot
 * h + p mod r. The decode step then reads no position of a recent slot (they
 * follow from t); its candidates are the heavy slots and the token leaving
 * the window, which moves into the heavy slot it displaces. Results are those
 * of the default slot-indexed layout (outputs, evictions, retained sets);
 * only the slot order differs. h2o_decode_steps takes one launch per step.
 */
int h2o_create_ex(int layers, int batch, int heads, int head_dim, int h, int r, int kv_format,
                  h2o_ctx** out);

/* h2o_destroy - free the cache and the context. Waits for the context's
 * stream work to finish first. NULL is accepted. */
void h2o_destroy(h2o_ctx* ctx);

/*
 * h2o_prefill - prompt pass of one layer ([H2O] A, Pseudocode: a prompt of at
 * least 2K tokens keeps K heavy hitters and K recent tokens).
 *
 * For every row: causal softmax attention of the T prompt queries over the
 * prompt keys, written to out; the accumulated score of prompt token j is the
 * column sum sum_{i >= j} P_ij of the causal probability matrix ([H2O] 3.2);
 * the cache then holds the r most recent tokens T-r .. T-1 plus the h other
 * tokens with the largest (score, position) keys, or every token if T <= h + r.
 * Ties in score keep the later position. Retained tokens keep their column
 * sums as accumulated scores.
 *
 * State: a layer takes one prompt ([H2O] A, Pseudocode: the prompt's heavy
 * hitters are selected once, then generation proceeds step by step). The
 * layer must be empty, as h2o_create or h2o_reset leaves it; a second prefill
 * without h2o_reset returns H2O_ESTATE and changes nothing. After a prefill
 * that fails the layer still counts as empty: decode returns H2O_ESTATE and
 * the next prefill is accepted.
 *
 * Q, K, V: device bf16 [batch, heads, T, d]; out: device fp32 [batch, heads, T, d].
 * 0 <= T <= H2O_MAX_T; with T = 0 the pointers may be NULL and the layer is
 * reset to an empty cache. Scratch (per-row log-sum-exp and column sums,
 * 8 bytes per prompt token) comes from PyTorch's caching allocator on the
 * current stream. Errors: H2O_EINVAL, H2O_ESTATE (layer not empty), H2O_ENOMEM,
 * H2O_ECUDA.
 */
int h2o_prefill(h2o_ctx* ctx, int layer, const void* Q, const void* K, const void* V, int T,
                float* out);

/*
 * h2o_reset - return one layer (layer >= 0) or every layer (layer = -1) to the
 * empty state h2o_create leaves: no token cached (positions -1, scores 0, fill
 * count and next position 0), ready for a new prompt (h2o_prefill). Enqueues
 * one small kernel per layer on the current stream; allocates nothing.
 * Errors: H2O_EINVAL (null context, layer out of range), H2O_ECUDA.
 */
int h2o_reset(h2o_ctx* ctx, int layer);

/*
 * h2o_prefill_ragged - h2o_prefill of a batch whose prompts differ in length
 * ([H2O] 5, Empirical Evaluation, Throughput and Latency: the gains come from
 * serving larger batches; entries of a batch are independent sequences, and
 * their prompts need not be equally long).
 *
 * Batch entry b holds a prompt of T_b = lens[b] tokens, stored right-padded
 * to T_max: Q, K, V device bf16 [batch, heads, T_max, d] with token t of entry
 * b at index t for t < T_b. Each row is processed exactly as h2o_prefill
 * processes a prompt of T_b tokens (attention, column sums, the r most recent
 * tokens T_b - r .. T_b - 1 plus the top-h others, or all T_b tokens when
 * T_b <= h + r), and its first decode step then processes position T_b.
 *
 * lens: device int32 [batch], 0 <= lens[b] <= T_max, read on the device (the
 * call can be captured in a CUDA graph with lengths written later). A length
 * outside that range is clamped into it and sets bit 4 of the device error
 * word (h2o_sync_check reports H2O_EDEVICE). The padding tokens t >= T_b of
 * Q, K and V must hold finite values (zeros, say): padded keys and values
 * enter the tensor-core products with probability 0, and 0 times a non-finite
 * value is not 0. out: device fp32 [batch, heads, T_max, d]; rows t >= T_b
 * hold no result (the call may write them). Scratch as for h2o_prefill, sized
 * by T_max. With T_max = 0 the pointers may be NULL and every row is reset to
 * an empty cache. The layer must be empty, as for h2o_prefill. Errors:
 * H2O_EINVAL (also for lens NULL with T_max > 0), H2O_ESTATE, H2O_ENOMEM,
 * H2O_ECUDA.
 */
int h2o_prefill_ragged(h2o_ctx* ctx, int layer, const void* Q, const void* K, const void* V,
                       int T_max, const int32_t* lens, float* out);

/*
 * h2o_decode_step - one generation step of one layer ([H2O] 4.1 and 2).
 *
 * For every row, with t its next position: append the new token (q, k_new,
 * v_new); attend over the cached tokens plus the new one, writing
 * out = sum_j p_j v_j with p = softmax(K q / sqrt(d)); add p_j to every cached
 * token's accumulated score and give the new token score p_t; if the row now
 * holds more than k tokens, evict the token with the smallest (score, position)
 * among those at positions <= t - r (the r most recent, t included, are never
 * evicted; with r = 0 the new token competes and may be dropped at once); the
 * new token's K/V, position and score go into the freed slot, or into the next
 * empty slot while the cache is not full.
 *
 * q, k_new, v_new: device bf16 [batch, heads, d]; out: device fp32 [batch, heads, d].
 * Allocates nothing and never synchronises. The step position and fill count
 * live in device memory and are advanced by the kernel, so the call can be
 * captured in a CUDA graph and replayed. Errors: H2O_EINVAL, H2O_ESTATE (layer
 * never prefilled), H2O_ECUDA.
 *
 * The kernel checks each row's state before it touches the row: a fill count
 * outside [0, k] or above the next position t, or an occupied slot whose
 * position is outside [0, t) (a state installed through h2o_cache_view that
 * no call of this library produces), sets bit 2 (bad state) of the device
 * error word, and a row with inconsistent counts is left unchanged.
 * h2o_sync_check then reports H2O_EDEVICE.
 */
int h2o_decode_step(h2o_ctx* ctx, int layer, const void* q, const void* k_new, const void* v_new,
                    float* out);

/*
 * h2o_decode_steps - `steps` consecutive h2o_decode_step calls of one layer
 * whose inputs are all known in advance ([H2O] 4.1: the policy is the same
 * greedy step repeated; 5, Ablation and Extended Evaluations: streaming over
 * long inputs), e.g. a teacher-forced pass over a known continuation, one
 * layer after the other. Results equal those of the single steps.
 *
 * q, k_new, v_new: device bf16 [steps, batch, heads, d]; out: device fp32
 * [steps, batch, heads, d]; evicted: device int32 [steps, batch * heads], the
 * position evicted by each row at each step (-1: none, the new token's own
 * position when it is dropped), or NULL. With h + r <= 8192 all steps run in
 * one launch, one CTA per row looping over its steps (no per-step launch and
 * drain); larger budgets, and rows of 1024 slots or more when there are fewer
 * rows than SMs (where splitting rows over several CTAs moves the bytes
 * faster), take one launch per step. steps >= 0 (0: nothing is
 * done). Allocates nothing and never synchronises; capturable in a CUDA
 * graph. Errors: H2O_EINVAL, H2O_ESTATE (layer never prefilled), H2O_ECUDA.
 */
int h2o_decode_steps(h2o_ctx* ctx, int layer, int steps, const void* q, const void* k_new,
                     const void* v_new, float* out, int32_t* evicted);

/*
 * h2o_prefill_attention - the attention part of prefill, without touching any
 * cache: causal attention of `rows` independent rows of T tokens, the output
 * and every token's column-sum score.
 *
 * Q, K, V: device bf16 [rows, T, d]; out: device fp32 [rows, T, d];
 * score: device fp32 [rows, T]. Scratch (per-row log-sum-exp, 4 bytes per
 * token) comes from PyTorch's caching allocator on the current stream.
 * A bounded device wait that gives up is reported through the library's own
 * error word (h2o_attention_sync_check), since no context is involved.
 * Errors: H2O_EINVAL, H2O_ENOMEM, H2O_ECUDA.
 */
int h2o_prefill_attention(const void* Q, const void* K, const void* V, int rows, int T,
                          int head_dim, float* out, float* score);

/*
 * h2o_prefill_attention_noalloc - the same computation as h2o_prefill_attention
 * (outputs and column-sum scores of `rows` cache-free rows), for callers that
 * must not allocate device memory during the call. The pages have no
 * counterpart to this entry point; it exists for the caller, not the policy.
 *
 * Who needs it: callers for which a device allocation during the call is not
 * an option. A serving process may reserve its device memory once at start-up
 * and forbid allocation on the request path, because cudaMalloc can block
 * until the device is idle and stall every stream. A process whose memory is
 * pre-reserved by another framework's arena (one that grabs most of the GPU up
 * front) has little free memory left, so an extra allocation can fail there.
 * Such callers cannot use h2o_prefill_attention, whose per-row log-sum-exp
 * scratch comes from PyTorch's caching allocator.
 *
 * Instead the scratch is a fixed device array inside the library
 * (H2O_NOALLOC_MAX_LSE floats, 4 MiB, held by every GPU that loads the
 * library until the process exits). This call allocates nothing, uses no
 * PyTorch state and enqueues its kernels on `stream` (a cudaStream_t; NULL is
 * the legacy default stream). The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture. All calls share the one array, so
 * calls whose work overlaps on the GPU (different streams, or different
 * threads without ordering between them) race on it; calls on one stream are
 * ordered and safe. Nothing in the array needs to start at zero: every entry a
 * call reads was written earlier by the same call.
 *
 * Where the array lives: CUDA loads a library's device code, and with it this
 * array, into a device on first use (lazy module loading is the default), so
 * the first call on each device may itself need 4 MiB of free device memory.
 * Make one small call on each device at start-up, before an arena reserves the
 * rest of the memory (and before any stream capture). The looked-up address
 * belongs to the device's context: after cudaDeviceReset on that device, call
 * h2o_forget_device_state() before the next call, which then looks it up
 * again.
 *
 * Errors inside the kernels: a bounded device wait that gives up sets the
 * library's error word, which h2o_attention_sync_check(stream) reports (the
 * word is also a fixed device variable, not an allocation).
 *
 * Q, K, V: device bf16 [rows, T, d]; out: device fp32 [rows, T, d];
 * score: device fp32 [rows, T]. Limit: rows * (T rounded up to a multiple of
 * 128) <= H2O_NOALLOC_MAX_LSE; larger calls are rejected with H2O_EINVAL and
 * a message. Errors: H2O_EINVAL, H2O_ECUDA.
 */
#define H2O_NOALLOC_MAX_LSE (1 << 20)
int h2o_prefill_attention_noalloc(const void* Q, const void* K, const void* V, int rows, int T,
                                  int head_dim, float* out, float* score, void* stream);

/*
 * h2o_attention_sync_check - synchronise `stream` (a cudaStream_t; NULL is the
 * legacy default stream) and report, then clear, the library-level device
 * error word of the current device that the cache-free entry points
 * (h2o_prefill_attention, h2o_prefill_attention_noalloc) write: bit 1 when
 * one of their bounded waits gave up (their outputs are then incomplete).
 * Allocates nothing. The word is shared by every such call on the device.
 * Errors: H2O_ECUDA, H2O_EDEVICE.
 */
int h2o_attention_sync_check(void* stream);

/*
 * h2o_attention_test_wait_limit - the failure path of the cache-free entry
 * points on demand: enqueues on `stream` one kernel whose bounded wait is
 * never satisfied; after the wait limit (2 s) it sets bit 1 of the
 * library-level error word and returns. The next h2o_attention_sync_check
 * reports H2O_EDEVICE. Errors: H2O_ECUDA.
 */
int h2o_attention_test_wait_limit(void* stream);

/*
 * h2o_forget_device_state - drop the per-device state the library caches (the
 * device addresses of its fixed arrays and its kernels' shared-memory
 * opt-ins), so that the next call on each device sets it up again. Needed
 * only after cudaDeviceReset (which discards a device's context, and with it
 * the library's loaded code and arrays); call it with no work of the library
 * in flight. Contexts made by h2o_create do not survive a device reset.
 */
void h2o_forget_device_state(void);

/*
 * h2o_test_fail_allocations - fault injection on the host: the next n device
 * allocations the library makes (a cache in h2o_create, prefill scratch) fail
 * as an exhausted allocator would, and the calls return H2O_ENOMEM with the
 * state unchanged (no context is created; a layer whose prefill failed stays
 * empty). n = 0 ends it. No GPU work is involved. Errors: H2O_EINVAL (n < 0).
 */
int h2o_test_fail_allocations(int n);

/*
 * h2o_cache_positions - copy the positions held by every slot of one layer to
 * host memory: host_pos int32 [batch * heads * k], row-major by (row, slot),
 * -1 for empty slots. Synchronises the current stream.
 * Errors: H2O_EINVAL, H2O_ECUDA, H2O_EDEVICE.
 */
int h2o_cache_positions(h2o_ctx* ctx, int layer, int32_t* host_pos);

/*
 * h2o_last_evicted - copy, per row, the position evicted by the layer's last
 * decode step (-1 when the step evicted nothing): host_pos int32
 * [batch * heads]. Synchronises the current stream.
 * Errors: H2O_EINVAL, H2O_ECUDA, H2O_EDEVICE.
 */
int h2o_last_evicted(h2o_ctx* ctx, int layer, int32_t* host_pos);

/*
 * h2o_cache_view - device addresses of one layer's cache arrays (layouts as in
 * h2o_create). The library keeps ownership; the addresses stay valid until
 * h2o_destroy. A caller may write through them (between calls, on the same
 * stream) to install a cache state; the fill count in meta must then match the
 * occupied slots, which are slots 0 .. filled-1 of the slot-indexed layout, or
 * for H2O_LAYOUT_RING the tokens older than the window from slot 0 and window
 * position p in slot h + p mod r. Any output pointer may be NULL.
 * Errors: H2O_EINVAL.
 */
int h2o_cache_view(h2o_ctx* ctx, int layer, void** K, void** V, float** score, int32_t** pos,
                   int32_t** meta);

/*
 * h2o_cache_scales - device addresses of one layer's per-slot scales of an
 * H2O_KV_FP8 cache: k_scale, v_scale fp32 [rows][k] (a slot's stored key is
 * E4M3(code) * k_scale). Same ownership and lifetime as h2o_cache_view; any
 * output pointer may be NULL. Errors: H2O_EINVAL (also for a bf16 cache).
 */
int h2o_cache_scales(h2o_ctx* ctx, int layer, float** k_scale, float** v_scale);

/* h2o_cache_dims - k (slots per row) and rows (batch * heads) per layer. */
int h2o_cache_dims(h2o_ctx* ctx, int* k, int* rows);

/*
 * h2o_test_wait_limit - the failure path on demand: enqueues one kernel whose
 * bounded mbarrier wait is never satisfied (nothing arrives on the barrier).
 * Like any kernel of the library whose producer never delivers, it gives up
 * after the wait limit (2 s), sets bit 1 (wait timeout) of the context's
 * device error word and returns; no kernel traps. The next h2o_sync_check
 * reports H2O_EDEVICE and clears the word, and the context stays usable.
 * Errors: H2O_EINVAL, H2O_ECUDA.
 */
int h2o_test_wait_limit(h2o_ctx* ctx);

/*
 * h2o_sync_check - synchronise the current stream and report, then clear, the
 * context's device error word. Errors: H2O_ECUDA, H2O_EDEVICE.
 */
int h2o_sync_check(h2o_ctx* ctx);

/* h2o_last_error - message of the calling thread's last failed call ("" if none). */
const char* h2o_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* H2O_H */
