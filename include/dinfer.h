/*
 * dinfer.h -- C-ABI of the GB300 (sm_103a) block-wise diffusion-LLM decoder.
 *
 * What it computes (dInfer: An Efficient Inference Framework for Diffusion
 * Language Models -- abstract: model, diffusion iteration manager, decoding
 * strategy and KV-cache manager; dInfer README, "Step 3: Use the model in
 * dInfer": BlockWiseDiffusionLLM(model, ThresholdParallelDecoder(0,
 * threshold, mask_id, eos_id), BlockIteratorFactory(True),
 * cache_factory=KVCacheFactory('dual')).generate(ids, gen_length,
 * block_length)):
 *
 *   x = prompt | mask_id * gen_length.  The generated part is decoded
 *   block_length positions at a time, left to right.  At a block boundary
 *   the model runs over the whole sequence and the per-layer keys/values of
 *   every position are stored (the dual cache: prefix and suffix); that
 *   forward's block rows are decoded as iteration 1.  Then, while the block
 *   still has masked positions, a denoising iteration recomputes only the
 *   block's rows, which attend bidirectionally over the cached prefix, the
 *   block's fresh keys/values and the cached suffix (the default dual cache;
 *   dinfer_set_cache_mode selects the other members of the family).  Each
 *   iteration the LM head gives, per block position, the top-1 token and its
 *   softmax probability (confidence); every masked position whose confidence exceeds
 *   the threshold is committed, or, if none does, the single most confident
 *   one (ties: lowest vocabulary index, lowest position).  The mask token's
 *   own logit is excluded from argmax and softmax.  eos_id is off unless
 *   dinfer_set_eos sets it (end of sequence after a completed block).
 *
 * Conventions
 *   - All calls are asynchronous on the context's stream unless stated.
 *   - The library owns the KV cache, workspaces and CUDA graphs; the caller
 *     owns weights, ids, masks and outputs.  Weights are borrowed: they must
 *     stay valid and unchanged until dinfer_destroy.
 *   - Errors are returned as dinfer_status; nothing is thrown across the
 *     ABI.  dinfer_last_error() describes the last failure of a context.
 *   - A context must be used by one host thread at a time.
 */
#ifndef DINFER_H
#define DINFER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dinfer_ctx dinfer_ctx;

typedef enum dinfer_status {
  DINFER_OK = 0,
  DINFER_EINVAL = -1,  /* bad argument: null pointer, size out of range, unsupported shape */
  DINFER_ENOMEM = -2,  /* device allocation failed */
  DINFER_ECUDA = -3,   /* a CUDA runtime / driver call failed (see dinfer_last_error) */
  DINFER_EDEVICE = -4, /* the device status word was set: token id out of range, NaN
                          confidence, iteration overflow or a pipeline wait timeout */
  DINFER_ESTATE = -5   /* call out of order (dinfer_block_step before dinfer_prefill_cache) */
} dinfer_status;

enum { DINFER_FP32 = 0, DINFER_BF16 = 1 };

/* Model description.  Dense models: n_experts = top_k = expert_ffn = 0.
 * bf16 models: head_dim 128, d_model and ffn multiples of 128 and 64, vocab
 * a multiple of 8.  max_batch / max_seq bound the dual cache and workspaces
 * allocated by dinfer_create (max_batch <= 64). */
typedef struct dinfer_model_desc {
  int32_t n_layers, d_model, n_heads, head_dim, ffn, vocab, mask_id;
  int32_t n_experts, top_k, expert_ffn;
  float rms_eps, rope_theta, logit_scale;
  int32_t dtype; /* DINFER_FP32 or DINFER_BF16: weights, K/V cache and GEMM inputs */
  int32_t max_batch, max_seq;
} dinfer_model_desc;

typedef struct dinfer_stats {
  int32_t n_blocks;        /* blocks of the generation (some skipped after end-of-sequence) */
  int32_t iterations;      /* denoising iterations, refreshes included */
  int32_t refreshes;       /* blocks run */
  float ms_device;         /* device time of the call (CUDA events on the stream) */
  int32_t* iters_per_block; /* optional caller array [n_blocks] (host), or NULL; 0 for a skipped block */
} dinfer_stats;

/* Number of weight pointers a model takes:
 *   1 + 9 * n_layers + 2, in this order, each row-major [out, in]:
 *   embed [V, d];
 *   per layer: attn_norm [d], wq [d, d], wk [d, d], wv [d, d], wo [d, d],
 *              ffn_norm [d], w_gate [f, d], w_up [f, d], w_down [d, f]
 *              (MoE: router [E, d], w13 [E, 2 fe, d] gate rows then up rows,
 *               w2 [E, d, fe] in place of the last three);
 *   final_norm [d]; lm_head [V, d].
 * Element type: bf16 for DINFER_BF16 models, fp32 for DINFER_FP32.
 * Returns -1 for an invalid description. */
int32_t dinfer_num_weights(const dinfer_model_desc* desc);

/* The model and its decoder (dInfer README, "Step 3": the model is built
 * from its configuration, its weights loaded in bf16, and wrapped with a
 * decoder and a dual KV-cache factory).  Validates the description, borrows
 * the device weight pointers (weights[i] as dinfer_num_weights orders them;
 * they stay owned by the caller and must outlive the context), allocates the
 * cache and workspaces for max_batch x max_seq and builds the weights' TMA
 * tensor maps.  stream: the cudaStream_t every call of the context is
 * ordered on (NULL = the legacy default stream).
 * Errors: DINFER_EINVAL (bad description, NULL or misaligned weight),
 * DINFER_ENOMEM (device allocation), DINFER_ECUDA (no device, a CUDA call
 * failed).  On failure *out is NULL and dinfer_last_error(NULL) explains why. */
dinfer_status dinfer_create(const dinfer_model_desc* desc, const void* const* weights, void* stream,
                            dinfer_ctx** out);

/* Waits for the context's stream, then frees the cache, workspaces and
 * graphs (not the borrowed weights).  NULL is ignored. */
void dinfer_destroy(dinfer_ctx* ctx);

/* Text of the last error of ctx (or of the last failed dinfer_create of this
 * thread when ctx is NULL).  Valid until the next call on the context. */
const char* dinfer_last_error(const dinfer_ctx* ctx);

/* KV-cache policy of the cached iterations (the README's cache factory names
 * the dual cache as one member of a family; its introduction adds a vicinity
 * refresh against cache staleness).  Every block starts with a refresh (a
 * forward over all positions that fills the cache); each later iteration of
 * the block recomputes a window of positions around the block, writing their
 * keys/values into the cache, and attends over the whole cached sequence:
 *   DINFER_CACHE_DUAL      the block only (default);
 *   DINFER_CACHE_NONE      every position (no cache: full recomputation);
 *   DINFER_CACHE_PREFIX    the block and everything after it (prefix-only cache);
 *   DINFER_CACHE_VICINITY  the block and `window` positions on each side of it
 *                          (clipped to the sequence).
 * Applies to dinfer_block_step and dinfer_generate.  Errors: DINFER_EINVAL for
 * an unknown mode or window < 0. */
enum { DINFER_CACHE_DUAL = 0, DINFER_CACHE_NONE = 1, DINFER_CACHE_PREFIX = 2, DINFER_CACHE_VICINITY = 3 };
dinfer_status dinfer_set_cache_mode(dinfer_ctx* ctx, int32_t mode, int32_t window);

/* End-of-sequence id of dinfer_generate (README "Step 3": the decoder takes
 * an eos_id): when a block completes and a sequence's block holds eos_id,
 * every later position of that sequence is set to eos_id (unmasked; tokens
 * already committed are kept), and the generation stops once no sequence has
 * masked positions left -- the remaining blocks' refreshes and iterations are
 * skipped on the device.  -1 (the default) disables it: every generated
 * position is decoded.  Errors: DINFER_EINVAL for an id outside [0, vocab)
 * or equal to mask_id. */
dinfer_status dinfer_set_eos(dinfer_ctx* ctx, int32_t eos_id);

/* Block boundary (cache refresh; dInfer README, "Step 3": the dual KV cache
 * of KVCacheFactory('dual'), the abstract's KV-cache manager): full forward
 * over ids[batch, seq_len] (device, int32, row-major), storing every layer's
 * K/V of all positions in the dual cache; then decodes the block
 * [block_start, block_start + block_len) and, if commit != 0, applies one
 * threshold commit (ThresholdParallelDecoder) to ids / mask (device, uint8,
 * 1 = masked) in place -- iteration 1 of the block.  committed: optional
 * device int32[batch] receiving the per-sequence commit count.  Asynchronous;
 * device-side errors surface at dinfer_sync or the next synchronising call.
 * Errors: DINFER_EINVAL (NULL or host ids / mask, batch > max_batch,
 * seq_len > max_seq, batch * block_len > 1024, block outside the sequence,
 * NaN threshold), DINFER_ECUDA. */
dinfer_status dinfer_prefill_cache(dinfer_ctx* ctx, int32_t* ids, uint8_t* mask, int32_t batch, int32_t seq_len,
                                   int32_t block_start, int32_t block_len, float threshold, int32_t commit,
                                   int32_t* committed);

/* One cached denoising iteration (dInfer README, "Step 3": the decoder's
 * threshold parallel commit; the abstract's diffusion iteration manager) of
 * the block set by the last dinfer_prefill_cache: the block rows of ids
 * [batch, seq_len] (device) -- or the window the cache policy recomputes --
 * are re-run against the cache (their fresh K/V overwrite their slots) and
 * one threshold commit updates ids / mask in place.  committed: optional
 * device int32[batch]; 0 for a sequence whose block had no mask.
 * Asynchronous like dinfer_prefill_cache.  Errors: DINFER_ESTATE before any
 * dinfer_prefill_cache, DINFER_EINVAL (NULL ids / mask, NaN threshold),
 * DINFER_ECUDA. */
dinfer_status dinfer_block_step(dinfer_ctx* ctx, int32_t* ids, uint8_t* mask, float threshold, int32_t* committed);

/* Whole generation (dInfer README, "Step 3": generate(input_ids,
 * gen_length, block_length) over BlockIteratorFactory's blocks; its
 * introduction: CUDA graphs and iteration loops without stream bubbles):
 * prompt [batch, prompt_len] int32 -> out [batch, prompt_len + gen_length]
 * int32 (prompt kept), both caller-owned.  prompt and out may be host or
 * device pointers; host buffers are copied inside the call.  Dual cache:
 * the block loop and the iteration loop run on the device (one CUDA graph
 * with conditional nodes).  Other cache policies: the host enqueues each
 * block (its refresh graph, then a graph whose conditional node runs the
 * block's iterations on the device) without waiting.  The call synchronises
 * once at the end.  gen_length must be a multiple of block_length.  stats may
 * be NULL.  Errors: DINFER_EINVAL (NULL buffers, gen_length not a positive
 * multiple of block_length, sizes beyond the context, NaN threshold),
 * DINFER_ECUDA, DINFER_EDEVICE (the device status word, read at the end: a
 * token id out of range, a NaN confidence, an iteration overflow or a timed
 * out pipeline wait; out is then not valid). */
dinfer_status dinfer_generate(dinfer_ctx* ctx, const int32_t* prompt, int32_t batch, int32_t prompt_len,
                              int32_t gen_length, int32_t block_length, float threshold, int32_t* out,
                              dinfer_stats* stats);

/* Test hook: while set, every decode also writes the fp32 logits [rows, V]
 * (mask token = -inf), tokens [rows] and confidences [rows] of the block
 * rows to these device buffers (each may be NULL); rows = batch * block_len.
 * Calls made while any is set run without CUDA graphs. */
dinfer_status dinfer_set_debug_outputs(dinfer_ctx* ctx, float* logits, int32_t* tok, float* conf);

/* Test hook for the per-layer parity diagnostics: while set, every
 * dinfer_prefill_cache / dinfer_block_step also writes the residual stream of
 * the block rows after each layer, hidden [n_layers][rows][d_model] fp32, and
 * the LM head's input (the final RMSNorm of the block rows, rounded to the
 * model's storage type), final_in [rows][d_model] (bf16 or fp32); rows =
 * batch * block_len, block rows in sequence order.  Either may be NULL.  Calls
 * made while any is set run without CUDA graphs; dinfer_generate writes
 * neither. */
dinfer_status dinfer_set_debug_hidden(dinfer_ctx* ctx, float* hidden, void* final_in);

/* Wait for the context's stream and report the device status word:
 * DINFER_OK, or DINFER_EDEVICE with the first failure described by
 * dinfer_last_error.  The word keeps its bits until the next
 * dinfer_prefill_cache or dinfer_generate clears it. */
dinfer_status dinfer_sync(dinfer_ctx* ctx);

/* Measurement hook for the byte count of a mixture-of-experts iteration (the
 * weights of the experts its rows select): *touched receives the number of
 * (MoE layer forward, expert) pairs that received at least one row since the
 * context was created or since the previous call, and the count restarts at
 * zero.  Waits for the context's stream.  Always 0 for dense models.
 * Errors: DINFER_EINVAL for NULL arguments, DINFER_ECUDA if the copy fails. */
dinfer_status dinfer_moe_experts_touched(dinfer_ctx* ctx, int64_t* touched);

#ifdef __cplusplus
}
#endif

#endif /* DINFER_H */
