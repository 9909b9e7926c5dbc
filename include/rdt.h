/*
 * rdt.h -- C ABI of librdt.so: one training step of a Qwen3-style decoder
 * block stack on one GB300 (sm_103a).
 *
 * Operations follow the aprender-train ("entrenar") pages:
 *   cuda_block.rs   (0.32.0): CudaTransformerBlock::forward, ::backward,
 *                   compute_attention_cuda, optimizer_step;
 *   cuda_trainer.rs (0.34.0): train_step_inner (fused cross-entropy),
 *                   gpu_forward / gpu_backward (final norm + LM head),
 *                   compute_workspace_clip_scale_gpu and
 *                   fused_clip_workspace_gradients (squared-sum clip),
 *                   run_nonblock_optimizer_step (AdamW).
 *
 * Conventions shared by every call:
 *  - Pointers are DEVICE pointers unless marked "host". The caller owns and
 *    allocates every buffer; the library never allocates, frees or
 *    synchronises (except rdt_device_error, which says so).
 *  - `stream` is a cudaStream_t passed as void*. Work is enqueued on it and
 *    the call returns before the GPU finishes.
 *  - Outputs are overwritten, never accumulated into.
 *  - Matrices are row-major. Weights are [out, in]; a projection computes
 *    y = x W^T. Activations are token-major [T, width] with T = batch*seq and
 *    token t = b*seq + s at position s of sequence b.
 *  - rdt_bf16 is the bit pattern of a bfloat16. Dense contractions take bf16
 *    operands (round-to-nearest-even copies of the fp32 masters) and
 *    accumulate in fp32; norms, softmax, loss and optimizer math are fp32.
 *  - Every call returns an rdt_status. Host-detectable problems (null
 *    pointers, unsupported shapes, misaligned pointers, buffers too small)
 *    return RDT_EINVAL before anything is enqueued; a failed launch returns
 *    RDT_ECUDA. rdt_last_error() gives a thread-local message for the last
 *    failure. Device-side waits in the kernels are bounded: one that gives up
 *    records RDT_ETIMEOUT in the device error word read by
 *    rdt_device_error().
 */
#ifndef RDT_H_
#define RDT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t rdt_bf16;

typedef enum rdt_status {
  RDT_OK = 0,
  RDT_EINVAL = 1,      /* bad argument, shape, alignment or buffer size */
  RDT_ECUDA = 2,       /* a CUDA runtime call or kernel launch failed */
  RDT_ETIMEOUT = 3,    /* a bounded device wait gave up (rdt_device_error) */
  RDT_ENONFINITE = 4,  /* reserved for callers: non-finite gradient norm */
  RDT_EINDEX = 5,      /* a token id outside [0, vocab) met on the device
                          (rdt_device_error; its row was zeroed / skipped) */
} rdt_status;

/* Model shape. hidden, head_dim and intermediate must be multiples of 16,
 * head_dim one of 16, 32, 64, 128; n_heads a multiple of n_kv_heads;
 * hidden <= 4096. rms_eps is used by every RMSNorm, forward and backward.
 * RoPE-neox rotates pairs (i, i + head_dim/2) by pos * rope_theta^(-2i/head_dim). */
typedef struct rdt_config {
  int32_t hidden;
  int32_t n_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t intermediate;
  int32_t vocab;
  float rms_eps;
  float rope_theta;
} rdt_config;

/* ---------------------------------------------------------------------------
 * Parameter layout of one block. A block's trainable tensors live in ONE flat
 * fp32 array (the masters) in this order, each starting at the offset
 * rdt_block_param_offsets() reports (multiples of 16 elements):
 *   WQ [nh*d, H], WK [nkv*d, H], WV [nkv*d, H], WO [H, nh*d],
 *   WG [I, H], WU [I, H], WD [H, I], G_ATTN [H], G_FFN [H], G_Q [d], G_K [d].
 * WQ/WK/WV are adjacent, so together they form the stacked [nh*d+2*nkv*d, H]
 * matrix; WG/WU likewise form [2I, H]. The matching bf16 shadow and the
 * gradient array use the same layout.
 * ------------------------------------------------------------------------- */
enum {
  RDT_WQ = 0, RDT_WK, RDT_WV, RDT_WO, RDT_WG, RDT_WU, RDT_WD,
  RDT_G_ATTN, RDT_G_FFN, RDT_G_Q, RDT_G_K, RDT_BLOCK_NTENSORS
};

/* Validates cfg (RDT_EINVAL on an unsupported shape). */
rdt_status rdt_check_config(const rdt_config* cfg);

/* Element count of one block's flat parameter array (fp32 or bf16), or -1. */
int64_t rdt_block_param_count(const rdt_config* cfg);

/* Host arrays of RDT_BLOCK_NTENSORS entries: element offset and element
 * count of each tensor inside the block's flat array. */
rdt_status rdt_block_param_offsets(const rdt_config* cfg, int64_t* offsets, int64_t* counts);

/* Bytes of the activations rdt_block_forward saves for rdt_block_backward
 * (opaque layout, caller-allocated, 256-byte aligned). */
size_t rdt_block_saved_bytes(const rdt_config* cfg, int32_t batch, int32_t seq);
/* Scratch bytes of rdt_block_forward / rdt_block_backward (256-byte aligned). */
size_t rdt_block_workspace_bytes(const rdt_config* cfg, int32_t batch, int32_t seq);
/* Scratch bytes of rdt_fused_cross_entropy for `tokens` tokens: O(tokens *
 * H) plus one vocabulary chunk of at most 256 MB; it does not grow with
 * tokens * V (the logits are never stored whole). */
size_t rdt_head_workspace_bytes(const rdt_config* cfg, int32_t tokens);
/* Scratch bytes of rdt_sq_sum. */
size_t rdt_sq_sum_workspace_bytes(void);

/* ---------------------------------------------------------------------------
 * Block forward (CudaTransformerBlock::forward with compute_attention_cuda;
 * the fused residual + RMSNorm of the NF4 block's forward):
 *   xn = RMSNorm(x, G_ATTN); q,k,v = xn Wq^T, xn Wk^T, xn Wv^T;
 *   per head: RMSNorm over head_dim (G_Q / G_K), then RoPE-neox at the
 *   token's position in its own sequence;
 *   o = causal softmax(q k^T / sqrt(d)) v, query head h reading kv head
 *       h / (nh/nkv); r1 = x + o Wo^T; xn2 = RMSNorm(r1, G_FFN);
 *   y = r1 + (silu(xn2 Wg^T) * (xn2 Wu^T)) Wd^T.
 * w      fp32 masters of this block (flat layout; the gains are read here)
 * w_bf16 bf16 shadow of the same layout (matrices are read here)
 * x, y   fp32 [batch*seq, hidden]; y must not alias x
 * saved  rdt_block_saved_bytes() bytes, written; keep for the backward
 * ws     rdt_block_workspace_bytes() bytes of scratch
 * ------------------------------------------------------------------------- */
rdt_status rdt_block_forward(const rdt_config* cfg, int32_t batch, int32_t seq,
                             const float* w, const rdt_bf16* w_bf16,
                             const float* x, float* y,
                             void* saved, size_t saved_bytes,
                             void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Block backward (CudaTransformerBlock::backward: backward_ffn,
 * backward_post_attn_norm, backward_attention with the GQA reduction and the
 * inverse RoPE, backward_residual_and_input_norm; the per-head QK-norm
 * backward and its gain gradients, which that path leaves out, are included).
 * x      the block's forward input, fp32 [T, H]
 * saved  what rdt_block_forward wrote for the same x and w
 * dy     upstream gradient fp32 [T, H]
 * dx     gradient w.r.t. x, fp32 [T, H] (overwritten; may alias dy)
 * grads  fp32 flat array in the block layout: every tensor overwritten
 *        (accumulate == 0) or added to (accumulate == 1: gradient
 *        accumulation over micro-batches, GpuGradientAccumulator in
 *        cuda_trainer.rs, here done in place by the gradient producers)
 * grad_sq  optional (may be null) fp64 device scalar: *grad_sq += the sum of
 *          the squares of every gradient this call leaves in grads (after
 *          the accumulation, so pass it on a step's last micro-batch only;
 *          the global-norm clip's squared sum, accumulated by the
 *          weight-gradient GEMMs' epilogues and the gain reductions as they
 *          produce the values; fixed summation order, so the same inputs give
 *          the same bits)
 * ------------------------------------------------------------------------- */
rdt_status rdt_block_backward(const rdt_config* cfg, int32_t batch, int32_t seq,
                              const float* w, const rdt_bf16* w_bf16,
                              const float* x, const void* saved, size_t saved_bytes,
                              const float* dy, float* dx, float* grads, int32_t accumulate,
                              double* grad_sq, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Final RMSNorm + LM head + cross-entropy, forward and backward in one call
 * (train_step_inner's fused cross-entropy; gpu_forward's final norm and LM
 * head; gpu_backward's LM-head and final-norm backward; KAIZEN-050/052's
 * fused CE). The logits are never stored whole, on the device or the host:
 * the vocabulary is walked in chunks of at most 256 MB of bf16 dz; each chunk's
 * logits are formed in the GEMMs' fp32 tensor-memory accumulators, once for
 * the log-sum-exp and the target's logit (forward) and once more for dz,
 * computed in fp32 from the saved log-sum-exp (backward). Nothing but the
 * caller's copy of loss_partials reaches the host.
 *   hn = RMSNorm(h, gamma_f); z = hn W_lm^T;
 *   loss_partials[t] = logsumexp(z_t) - z_t[targets[t]]   (unscaled NLL);
 *   dz = (softmax(z_t) - onehot(targets[t])) * loss_scale;
 *   dh, dgamma_f, dw_lm = gradients of sum_t loss_scale * loss_partials[t].
 * h        fp32 [tokens, H], the last block's output
 * gamma_f  fp32 [H]; w_lm bf16 [V, H]
 * targets  int32 [tokens], device; each must lie in [0, V) (not checked on
 *          the device: the caller validates ids before upload)
 * loss_scale  normally 1/tokens (loss = mean NLL); 1/(tokens * n) for each of
 *          n accumulated micro-batches (train_step_inner divides by
 *          accumulation_steps)
 * dh fp32 [tokens, H] (overwritten); dgamma_f fp32 [H] and dw_lm fp32 [V, H]
 *          overwritten (accumulate == 0) or added to (accumulate == 1)
 * grad_sq  optional (may be null) fp64 device scalar: *grad_sq = the sum of
 *          the squares of dgamma_f and dw_lm as this call leaves them (a
 *          step's backward starts here, so this call starts the clip's
 *          squared sum that each rdt_block_backward then adds to; pass it on
 *          the last micro-batch only when accumulating)
 * ------------------------------------------------------------------------- */
rdt_status rdt_fused_cross_entropy(const rdt_config* cfg, int32_t tokens,
                                   const float* h, const float* gamma_f,
                                   const rdt_bf16* w_lm, const int32_t* targets,
                                   float loss_scale, float* loss_partials,
                                   float* dh, float* dgamma_f, float* dw_lm, int32_t accumulate,
                                   double* grad_sq, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Squared-sum gradient clip (compute_workspace_clip_scale_gpu,
 * fused_clip_workspace_gradients; contract C-CLIP-001).
 * rdt_sq_sum: *sumsq = sum over the nbuf buffers of sum(g^2), accumulated in
 *   fp64 (fp32 within a thread's short run). bufs and lens are HOST arrays of
 *   device pointers / element counts; each buffer 16-byte aligned.
 * rdt_clip_scale: norm = sqrt(*sumsq) (the squared sums are not squared
 *   again); *scale = max_norm / norm if norm > max_norm else 1;
 *   *nonfinite = 1 if norm is not finite (then *scale = 1), else 0.
 * ------------------------------------------------------------------------- */
rdt_status rdt_sq_sum(const float* const* bufs, const int64_t* lens, int32_t nbuf,
                      double* sumsq, void* ws, size_t ws_bytes, void* stream);
rdt_status rdt_clip_scale(const double* sumsq, float max_norm, float* scale,
                          int32_t* nonfinite, void* stream);

/* rdt_sq_sum for callers that cannot allocate device memory (code inside an
 * allocator or pool callback, a runtime whose footprint is fixed once it
 * starts, a plugin whose host gives it no scratch buffer). The pages have no
 * counterpart of this call: it exists for those callers only. Same result as
 * rdt_sq_sum; no workspace argument and no allocation of any kind. Its
 * scratch is a fixed 32 KiB array (4096 fp64 partial sums) inside librdt.so
 * that every GPU loading the library keeps until the process exits; any total
 * length fits in it, and more than 64 buffers per call is rejected with
 * RDT_EINVAL. The first call on a device looks up the array's device address
 * (make that first call before any stream capture). Every call shares the one
 * array, so calls that may overlap on the GPU (different streams, or
 * different host threads on one device) race and must be serialised by the
 * caller; each call rewrites every partial it reads, so nothing needs
 * clearing in between. */
rdt_status rdt_sq_sum_noalloc(const float* const* bufs, const int64_t* lens, int32_t nbuf,
                              double* sumsq, void* stream);

/* ---------------------------------------------------------------------------
 * AdamW over n contiguous fp32 elements (optimizer_step's adamw_step_cuda;
 * step counted from 1 as run_nonblock_optimizer_step does):
 *   g' = scale * g; m = b1 m + (1-b1) g'; v = b2 v + (1-b2) g'^2;
 *   w = w - lr * ( (m/(1-b1^step)) / (sqrt(v/(1-b2^step)) + eps) + wd * w ).
 * scale     device fp32 scalar from rdt_clip_scale, or NULL for 1
 * skip_flag device int32, or NULL; when *skip_flag != 0 nothing is written
 * w_bf16    if not NULL, receives the bf16 (RNE) copy of the updated w
 * step_dev  if not NULL, a device int32 holding the step (>= 1) that the
 *           kernel reads instead of `step` (which is then ignored): a step
 *           count that lives on the device, so a captured CUDA graph of the
 *           training step can be replayed unchanged (see rdt_step_advance)
 * w, g, m, v, w_bf16 16-byte aligned. step >= 1 unless step_dev is given.
 * rdt_step_advance: *step += 1 on the device, in stream order.
 * ------------------------------------------------------------------------- */
rdt_status rdt_adamw_step(float* w, const float* g, float* m, float* v, int64_t n,
                          const float* scale, const int32_t* skip_flag, int32_t step,
                          const int32_t* step_dev, float lr, float beta1, float beta2,
                          float eps, float weight_decay, rdt_bf16* w_bf16, void* stream);
rdt_status rdt_step_advance(int32_t* step, void* stream);

/* The tensor-core GEMM every projection of the path runs on, exposed so it
 * can be tested on its own: C[M, N] (fp32, row stride ldc) = A' B'^T over K,
 * with A' = A ([M, K], row stride lda) when a_mn == 0, or the transpose of A
 * given as [K, M] when a_mn == 1; likewise B' = B ([N, K]) or B^T with B
 * given as [K, N]. A, B bf16; lda, ldb multiples of 8; ldc a multiple of 4.
 * split_ws (optional, 16-byte aligned, split_ws_floats fp32 elements): scratch
 * that lets a problem with too few 128 x 256 output tiles to fill the GPU run
 * as K-slices whose partials are then summed in slice order (the NF4 block's
 * adapter GEMMs take this path); null: one pass over K. */
rdt_status rdt_gemm(const rdt_bf16* A, int32_t a_mn, int64_t lda, const rdt_bf16* B,
                    int32_t b_mn, int64_t ldb, int32_t M, int32_t N, int32_t K, float* C,
                    int64_t ldc, float* split_ws, int64_t split_ws_floats, void* stream);

/* The NF4 GEMM of the NF4-frozen block (CudaNf4TransformerBlock in
 * cuda_block.rs: frozen projection weights stored as packed 4-bit NormalFloat
 * codes with one fp32 scale per 64-element block), exposed for tests:
 * C[M, N] (fp32, row stride ldc) = A [M, K1] (bf16, lda) times B^T, plus an
 * optional tail A2 [M, K2] times B2^T (K2 <= 64; the LoRA term folded in as
 * extra K). W is [w_rows, w_cols] row-major: codes uint8 [w_rows, w_cols/2]
 * (element 2j in the low nibble of byte j), scales fp32 [w_rows, w_cols/64];
 * W = level[code] * scale, levels the 16 NormalFloat-4 values of QLoRA.
 * b_mn == 0: B = W (N = w_rows, K1 = w_cols; y = x W^T), B2 [N, K2] (ldb2);
 * b_mn == 1: B = W^T (N = w_cols, K1 = w_rows; dX = dY W), B2 [K2, N].
 * w_cols % 256 == 0 and w_rows % 64 == 0; leading dimensions in elements,
 * bf16 ones multiples of 8, ldc a multiple of 4; 16-byte aligned pointers.
 * split_ws (optional, as in rdt_gemm): scratch for running the problem as
 * K-slices when its tiles would leave most of the GPU idle. */
rdt_status rdt_gemm_nf4(const rdt_bf16* A, int64_t lda, const uint8_t* codes,
                        const float* scales, int64_t w_rows, int64_t w_cols, int32_t b_mn,
                        const rdt_bf16* A2, int64_t lda2, const rdt_bf16* B2, int64_t ldb2,
                        int32_t K2, int32_t M, float* C, int64_t ldc, float* split_ws,
                        int64_t split_ws_floats, void* stream);

/* dst[i] = bf16(src[i]) with round-to-nearest-even; n elements, 16-byte aligned. */
rdt_status rdt_cast_bf16(const float* src, rdt_bf16* dst, int64_t n, void* stream);

/* ---------------------------------------------------------------------------
 * NF4-frozen block with LoRA adapters (CudaNf4TransformerBlock in
 * cuda_block.rs: the seven projection weights frozen as packed 4-bit
 * NormalFloat codes, one fp32 scale per block of 64 consecutive elements of
 * the row-major [out, in] weight; lora_scale = alpha / rank as in
 * cuda_trainer.rs; lora_forward in wgpu_trainer.rs: y = x W^T +
 * (alpha/rank) (x A^T) B^T with A [rank, in], B [out, rank]). The block is
 * the block above with every projection replaced by that LoRA projection on
 * the dequantized W = level[code] * scale (levels: the 16 NormalFloat-4
 * values of QLoRA); the norm gains are frozen and only the adapters get
 * gradients.
 *
 * Constraints (rdt_nf4_check): rdt_check_config's, hidden, n_heads*head_dim
 * and intermediate multiples of 256, n_kv_heads*head_dim a multiple of 64,
 * rank 8 or 16 (the stacked Q/K/V adapters, 3*rank columns, fit one 64-deep
 * GEMM step).
 *
 * codes   uint8, the seven projections' packed codes back to back in the
 *         order q, k, v, o, gate, up, down, each [out, in/2] row-major with
 *         element 2j in the low nibble of byte j (rdt_nf4_offsets: byte offsets)
 * scales  fp32, the seven projections' block scales in the same order, each
 *         [out, in/64] (rdt_nf4_offsets: element offsets)
 * gains   fp32 [hidden | hidden | head_dim | head_dim]: input-norm,
 *         post-attention-norm, q-norm and k-norm gains (frozen)
 * lora    fp32 adapters, tensors RDT_LORA_* back to back (rdt_lora_param_offsets);
 *         A's are [rank, in], B's [out, rank]
 * shadow  bf16 operand copy of the adapters the GEMMs read, rdt_lora_shadow_count
 *         elements, written by rdt_lora_shadow from lora (call it after every
 *         update of lora)
 * ------------------------------------------------------------------------- */
enum {
  RDT_LORA_A_Q, RDT_LORA_A_K, RDT_LORA_A_V, RDT_LORA_A_O, RDT_LORA_A_G, RDT_LORA_A_U,
  RDT_LORA_A_D, RDT_LORA_B_Q, RDT_LORA_B_K, RDT_LORA_B_V, RDT_LORA_B_O, RDT_LORA_B_G,
  RDT_LORA_B_U, RDT_LORA_B_D, RDT_LORA_NTENSORS
};

/* RDT_OK when cfg and rank meet the constraints above, else RDT_EINVAL. */
rdt_status rdt_nf4_check(const rdt_config* cfg, int32_t rank);
/* Total code bytes / scale elements of the seven projections (-1 if invalid). */
int64_t rdt_nf4_code_bytes(const rdt_config* cfg);
int64_t rdt_nf4_scale_count(const rdt_config* cfg);
/* Host arrays of 7 entries (q, k, v, o, gate, up, down): byte offsets into
 * codes and element offsets into scales. */
rdt_status rdt_nf4_offsets(const rdt_config* cfg, int64_t* code_offsets, int64_t* scale_offsets);
/* Adapter layout: element count; host arrays of RDT_LORA_NTENSORS offsets and counts. */
int64_t rdt_lora_param_count(const rdt_config* cfg, int32_t rank);
rdt_status rdt_lora_param_offsets(const rdt_config* cfg, int32_t rank, int64_t* offsets,
                                  int64_t* counts);
/* bf16 elements of the adapters' operand copy; rdt_lora_shadow writes it. */
int64_t rdt_lora_shadow_count(const rdt_config* cfg, int32_t rank);
rdt_status rdt_lora_shadow(const rdt_config* cfg, int32_t rank, const float* lora,
                           rdt_bf16* shadow, void* stream);
/* Saved-activation and scratch bytes of the NF4 block calls (256-byte aligned). */
size_t rdt_nf4_saved_bytes(const rdt_config* cfg, int32_t rank, int32_t batch, int32_t seq);
size_t rdt_nf4_workspace_bytes(const rdt_config* cfg, int32_t rank, int32_t batch, int32_t seq);

/* Forward of the NF4 + LoRA block: x, y fp32 [batch*seq, hidden] (y must not
 * alias x); saved written for rdt_nf4_block_backward. */
rdt_status rdt_nf4_block_forward(const rdt_config* cfg, int32_t rank, float alpha, int32_t batch,
                                 int32_t seq, const uint8_t* codes, const float* scales,
                                 const float* gains, const rdt_bf16* shadow, const float* x,
                                 float* y, void* saved, size_t saved_bytes, void* ws,
                                 size_t ws_bytes, void* stream);
/* Backward of the NF4 + LoRA block: dx fp32 [batch*seq, hidden] (may alias
 * dy); lora_grads fp32 in the adapter layout, every tensor overwritten;
 * grad_sq optional (may be null): *grad_sq += the sum of the squares of the
 * adapter gradients (fixed summation order). The frozen weights and gains get
 * no gradient. */
rdt_status rdt_nf4_block_backward(const rdt_config* cfg, int32_t rank, float alpha,
                                  int32_t batch, int32_t seq, const uint8_t* codes,
                                  const float* scales, const float* gains,
                                  const rdt_bf16* shadow, const float* x, const void* saved,
                                  size_t saved_bytes, const float* dy, float* dx,
                                  float* lora_grads, double* grad_sq, void* ws, size_t ws_bytes,
                                  void* stream);

/* ---------------------------------------------------------------------------
 * Measurement hooks (host-side bookkeeping only; no device memory).
 * rdt_gemm_timing_arm: while armed, the i-th tensor-core GEMM launch (any
 *   entry point) records the caller-created cudaEvent_t events[2i] on its
 *   stream just before the launch and events[2i+1] just after it, and stores
 *   its algorithmic FLOP count 2*M*N*K in flops[i] and, when kinds is not
 *   null, its kernel in kinds[i] (0: bf16 single-CTA tiles, 1: bf16 CTA-pair
 *   tiles, 2: NF4-decoding kernel; host arrays), for i < capacity. rdt_gemm_timing_disarm stops it and returns the number of
 *   launches seen (which may exceed capacity; only the first capacity are
 *   recorded).
 * rdt_launch_count: kernels this process has launched through the library
 *   so far (all entry points, all devices). */
rdt_status rdt_gemm_timing_arm(void* const* events, double* flops, int32_t* kinds,
                               int32_t capacity);
int64_t rdt_gemm_timing_disarm(void);
int64_t rdt_launch_count(void);

/* ---------------------------------------------------------------------------
 * Token embedding on the device (cuda_trainer.rs: gpu_forward's embedding
 * lookup and embed_backward's scatter-add, C-EMBED-GRAD-001, both of which
 * the pages run on the host).
 * rdt_embedding_forward: x[t, :] = table[ids[t], :]; table fp32 [vocab,
 *   hidden] (hidden % 4 == 0), ids int32 [tokens] on the device, x fp32
 *   [tokens, hidden]. An id outside [0, vocab) gives a zero row and records
 *   RDT_EINDEX in the device error word.
 * rdt_embedding_backward: dtable[id, :] = (accumulate == 0: every row first
 *   zeroed) or += scale * sum over the tokens t with ids[t] == id of
 *   dx[t, :], the sum taken in token order (deterministic, no atomics);
 *   scale an optional device fp32 scalar (null: 1), normally the activation
 *   gradient's own clip scale from rdt_sq_sum + rdt_clip_scale
 *   (C-EMBED-GRAD-001); ids outside [0, vocab) are skipped. ws: device
 *   scratch of rdt_embedding_workspace_bytes(tokens) bytes, 256-byte aligned.
 * ------------------------------------------------------------------------- */
size_t rdt_embedding_workspace_bytes(int32_t tokens);
rdt_status rdt_embedding_forward(const float* table, int64_t vocab, int32_t hidden,
                                 const int32_t* ids, int32_t tokens, float* x, void* stream);
rdt_status rdt_embedding_backward(const int32_t* ids, int32_t tokens, const float* dx,
                                  int32_t hidden, const float* scale, float* dtable,
                                  int64_t vocab, int32_t accumulate, void* ws, size_t ws_bytes,
                                  void* stream);

/* Thread-local description of the last failure on this thread ("" if none). */
const char* rdt_last_error(void);

/* Test hook for the bounded device waits (the error path the tensor-core
 * kernels take when a wait gives up; cuda_trainer.rs train_step_inner
 * reports a poisoned CUDA context after a device failure, which these bounds
 * avoid). Launches one warp on `stream` that holds 32 tensor-memory columns,
 * waits on an mbarrier with a limit of limit_ns nanoseconds (in [1e3, 1e10]),
 * then frees the columns and returns whatever the outcome. arrive != 0: the
 * warp arrives on the barrier first, so the wait completes at once;
 * arrive == 0: nothing arrives, the wait gives up after limit_ns and records
 * RDT_ETIMEOUT in the device error word (read it with rdt_device_error).
 * waited_ns: optional device uint64 that receives the wait's duration.
 * RDT_EINVAL for an out-of-range limit or a misaligned waited_ns. */
rdt_status rdt_wait_probe(int64_t limit_ns, int32_t arrive, uint64_t* waited_ns, void* stream);

/* Synchronises the current device, then reads and clears the device error
 * word of the current device (0 = none, else an rdt_status such as
 * RDT_ETIMEOUT). Writes it to *code (host). */
rdt_status rdt_device_error(int32_t* code);

#ifdef __cplusplus
}
#endif
#endif /* RDT_H_ */
