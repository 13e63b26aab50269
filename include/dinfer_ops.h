/*
 * dinfer_ops.h -- kernel-level entry points of the same library, for parity
 * tests and per-kernel measurement at full model shapes.  Each runs exactly
 * one of the kernels that dinfer_block_step / dinfer_prefill_cache launch.
 *
 * All pointers are device pointers unless stated; all calls are asynchronous
 * on `stream` (a cudaStream_t, NULL = legacy default stream).  `workspace`
 * is caller-owned device memory of `workspace_bytes` bytes that must be
 * zero-filled once before its first use; the calls leave its counter region
 * zeroed again.  Calls sharing one workspace must not overlap on the GPU.
 * Errors: DINFER_EINVAL for bad sizes / NULL pointers / a too-small
 * workspace, DINFER_ECUDA for a failed launch.
 */
#ifndef DINFER_OPS_H
#define DINFER_OPS_H

#include "dinfer.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Workspace size that covers every op below for M <= 1024 rows, d <= 8192
 * and up to 64 query tiles x 64 heads of attention. */
size_t dinfer_op_workspace_bytes(void);

/* Every projection of the forward (QKV, O, gate/up, down, router) of the
 * bf16 model that dInfer README "Step 3" loads:
 * Y[m, n] = sum_k X[m, k] W[n, k]  (bf16 inputs, fp32 accumulate and output).
 * X [M, K] bf16, W [N, K] bf16 (row-major, 16-byte aligned), Y [M, N] fp32.
 * K % 64 == 0, N % 128 == 0, 1 <= M <= 1 << 20.  The tensor-core GEMM
 * (tcgen05, TMA, stream-K) used for every projection of the model: one-CTA
 * tiles of 128 weight rows for few rows (weight streaming), pair-CTA tiles
 * (tcgen05 cta_group::2, 256 weight rows x 256 rows per 2-CTA cluster) from
 * 384 rows on (tensor-bound), as the model's forward chooses them; the sum
 * order over k differs between the two, the results agree within fp32
 * accumulation rounding. */
dinfer_status dinfer_op_gemm_bf16(const void* X, const void* W, float* Y, int32_t M, int32_t N, int32_t K,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Fused LM head (the decoder of dInfer README "Step 3",
 * ThresholdParallelDecoder, needs per position the top-1 token and its
 * softmax probability; computed without materialising the logits):
 *   l[m, v] = scale * sum_k X[m, k] W[v, k], l[m, mask_id] = -inf,
 *   tok[m] = argmax_v l[m, v] (lowest index on ties),
 *   conf[m] = 1 / sum_v exp(l[m, v] - l[m, tok[m]]).
 * X [M, K] bf16 (M <= 1024), W [V, K] bf16, tok [M] int32, conf [M] fp32;
 * logits [M, V] fp32 optional (NULL = not written). K % 64 == 0, V % 8 == 0. */
dinfer_status dinfer_op_lmhead_bf16(const void* X, const void* W, int32_t M, int32_t V, int32_t K, int32_t mask_id,
                                    float scale, int32_t* tok, float* conf, float* logits, void* workspace,
                                    size_t workspace_bytes, void* stream);

/* Bidirectional attention of the block rows against the dual cache (dInfer
 * README, "Step 3": KVCacheFactory('dual'); no causal mask in a diffusion LM):
 *   o[r, h, :] = sum_j softmax_j(q[r, h, :] . k[b, j, h, :] / sqrt(128)) v[b, j, h, :]
 * over all j < L of sequence b = r / rows_per_seq, no mask.  q, o
 * [batch * rows_per_seq, heads * 128] bf16; k, v [batch, L, heads * 128] bf16.
 * One CTA per 128 query rows x head on the tcgen05 tensor cores; when that
 * grid has fewer CTAs than the GPU has SMs, the keys are split over up to 8
 * CTAs of a thread-block cluster.  All pointers 16-byte aligned.  The
 * workspace may be NULL; when given, a wait that timed out sets its status
 * word. */
dinfer_status dinfer_op_attention_bf16(const void* q, const void* k, const void* v, void* o, int32_t batch,
                                       int32_t rows_per_seq, int32_t L, int32_t heads, void* workspace,
                                       size_t workspace_bytes, void* stream);

/* Routed expert FFN of a mixture-of-experts layer (the LLaDA-MoE model of
 * dInfer README, "Step 3", an OLMoE-style model with fused experts), the
 * expert step of the denoising iteration's FFN:
 *   p = softmax(X router^T) over E experts; the K experts of highest p (ties
 *   to the lower index); out[m] = sum over them of p_e * SwiGLU_e(X[m]) with
 *   SwiGLU_e(x) = (silu(x W_g,e^T) * x W_u,e^T) W_d,e^T  (weights not renormalised).
 * X [M, d] bf16 (the normed FFN input); router [E, d]; w13 [E, 2 fe, d] (gate
 * rows then up rows); w2 [E, d, fe]; all bf16 row-major.  out [M, d] fp32.
 * topk_id [M, K] int32 / topk_w [M, K] fp32 optional (the routing decision).
 * d % 128 == 0, d <= 8192, E <= 64, K <= 8, fe % 64 == 0. */
dinfer_status dinfer_op_moe_ffn_bf16(const void* X, const void* router, const void* w13, const void* w2, int32_t M,
                                     int32_t d, int32_t E, int32_t K, int32_t fe, float* out, int32_t* topk_id,
                                     float* topk_w, void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free variant of dinfer_op_gemm_bf16 (no counterpart in the
 * method itself: it exists for callers that cannot allocate device memory
 * when they run a projection -- code inside another framework's memory pool,
 * real-time paths, plug-ins that must not grow their footprint).  Same
 * operands as dinfer_op_gemm_bf16 for M <= 64 token rows, and the same
 * schedule with its grid capped at 152 CTAs, so on a GPU of at most 152 SMs
 * (a GB300) the result is bitwise the same.  No workspace argument and no
 * allocation: the split-K partial tiles go to a fixed 9.5 MiB array in the
 * library's module, present on every GPU that loads the library until the
 * process exits.  The first call on a device looks the array's device address
 * up (cudaGetSymbolAddress, guarded so that concurrent first calls from
 * several host threads are safe); make that first call before any stream
 * capture.  All calls share the array, so calls that overlap on the GPU race
 * and must be serialised by the caller.  A pipeline wait that times out on the
 * device is not reported by this call (it returns before the kernels run):
 * it sets a status word that dinfer_op_gemm_bf16_noalloc_status reports.
 * Errors: DINFER_EINVAL for M > 64 or an unsupported shape, DINFER_ECUDA if
 * the set-up or a launch fails. */
dinfer_status dinfer_op_gemm_bf16_noalloc(const void* X, const void* W, float* Y, int32_t M, int32_t N, int32_t K,
                                          void* stream);

/* Device status of the allocation-free GEMM: waits for `stream`, reads the
 * status word its kernels share, and clears it.  DINFER_EDEVICE (with the
 * first timed-out wait's kernel, site, CTA and thread in dinfer_last_error)
 * means that the output of some call since the previous check is not valid;
 * DINFER_OK that no wait timed out.  Allocates nothing. */
dinfer_status dinfer_op_gemm_bf16_noalloc_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DINFER_OPS_H */
