/*
 * sf.h -- C ABI of the layer-sliding fine-tuning step on one GB300 GPU.
 *
 * The method (SlideFormer, "An Efficient Heterogeneous Co-Design for
 * Fine-Tuning on a Single GPU"; abstract, and the gist.science technical
 * summary, section 2 "Methodologie") fine-tunes a decoder whose full state
 * stays in host memory:
 *   - the GPU holds only a fixed ring of identical layer buffers (section 2.B,
 *     "Pre-allocated GPU Cache Queue"); each layer's bf16 weights stream in
 *     from pinned host memory on a copy stream (section 2.A);
 *   - each layer's forward, and after the loss its recompute-and-backward,
 *     run on a compute stream; the LM-head projection and cross-entropy are
 *     fused and chunked so the full logits never exist (section 2.C, "Fused
 *     LinearCrossEntropy");
 *   - a finished layer's gradients stream back to host buffers that are
 *     shared with the bf16 weight copies (section 2.B, "Gedeelde
 *     CPU-buffers") while the next layer computes, and a per-layer Adam
 *     updates the fp32 master weights on host threads (section 2.A and 2.B,
 *     "Layer-Adam Optimizer").
 * The model is a pre-norm Llama-style decoder (section 4 names Llama, Qwen
 * and Mistral): RMSNorm, QKV projection with rotary embedding (rotate-half
 * pairs), causal grouped-query attention, output projection, RMSNorm, SwiGLU
 * FFN; embedding and LM head untied (options: Q/K/V biases and a tied LM
 * head, the Qwen layer); loss = mean token cross-entropy over labels !=
 * SF_IGNORE_INDEX.
 *
 * Conventions for every entry point:
 *   - Return value: SF_OK (0) or a negative status below.  No exception and
 *     no abort crosses this ABI.
 *   - The caller owns every pointer it passes.  Host inputs are copied
 *     before the call returns; host outputs are written before it returns.
 *   - The library owns all device memory, streams, events and pinned host
 *     memory of a context; sf_free releases them.
 *   - A context is used by one caller thread at a time.
 *   - Matrices are row-major; weights use the [out_features, in_features]
 *     layout of a linear layer; token t of a batch is t = b * seq + s.
 */
#ifndef SF_H_
#define SF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
#define SF_OK 0
#define SF_EINVAL (-1)   /* bad argument: null, size, range, unit, token or label */
#define SF_ENOMEM (-2)   /* device or host allocation failed */
#define SF_ECUDA (-3)    /* a CUDA call failed; the context is poisoned */
#define SF_ETIMEOUT (-4) /* a bounded wait (host event poll or device pipeline) ran out */
#define SF_ESTATE (-5)   /* call not valid in this state (poisoned ctx, grads not retained) */
#define SF_EDEVICE (-6)  /* a kernel recorded a device-side error (see sf_last_error) */

/* Units: decoder layers are 0 .. n_layers-1; the other tensors are: */
#define SF_UNIT_EMBED (-1)      /* token embedding [vocab, hidden] */
#define SF_UNIT_FINAL_NORM (-2) /* final RMSNorm gain [hidden] */
#define SF_UNIT_LM_HEAD (-3)    /* LM head [vocab, hidden] */

#define SF_IGNORE_INDEX (-100)

typedef struct sf_ctx sf_ctx;

/* Model and engine configuration.
 *   n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab: decoder shape.
 *     head_dim in {64, 128}; n_heads % n_kv_heads == 0; hidden, ffn, vocab
 *     multiples of 8; hidden <= 16384.  n_heads*head_dim may differ from hidden.
 *   max_batch, max_seq: the largest batch x seq a step may use (sizes buffers).
 *   ring_slots: R identical GPU layer buffers, 2 <= R <= n_layers (R ==
 *     n_layers keeps every layer resident: the non-offloaded reference mode).
 *   lce_chunk_rows: rows of the fused LM-head/cross-entropy per chunk
 *     (0 = automatic); the chunk's logits are the only logits ever stored.
 *   retain_grads: 1 keeps every unit's gradient of the last step on the host
 *     for sf_get_grads (costs a host copy per unit); 0 lets the gradient
 *     buffers be reused.
 *   rms_eps, rope_base: RMSNorm epsilon and RoPE base.
 *   device: CUDA device ordinal.
 *   adam_threads: host threads for Adam, gather and scatter (0 = all cores).
 *   wait_timeout_ms: bound of every host-side wait on the GPU (0 = 300000).
 *   async_update: 0 = sf_train_step returns after every host update of the
 *     step is done; 1 = it returns once the loss is ready and the updates
 *     still running overlap the next step (which waits for a unit's update
 *     just before that unit is needed).  Results are identical either way;
 *     sf_get_grads, sf_get_weights and sf_load_layer_weights wait for the
 *     pending updates first.
 *   offload_activations: 0 = every layer's input checkpoint (fp32 [T, d])
 *     stays in device memory; 1 = sliding activations: after a layer's
 *     forward its checkpoint is copied to pinned host memory and brought back
 *     just before that layer's backward, the device keeping a window of four
 *     (results are identical).
 *   deterministic: 0 = the attention backward adds the dQ contributions of
 *     its key blocks into one fp32 buffer in whatever order they arrive, so
 *     the last bits of a gradient can differ between two identical steps;
 *     1 = every key block writes its own slot and the slots are summed in key
 *     order (bit-reproducible steps, ~ceil(max_seq/128) x more dQ scratch in
 *     device memory and one extra pass over it).
 *   qkv_bias: 1 = the Q, K and V projections have biases (Qwen family); a
 *     layer unit then holds bq [Hq*hd], bk [Hkv*hd], bv [Hkv*hd] right after
 *     W_v, and the biases are added before the rotary embedding.
 *   tie_embeddings: 1 = the LM head is the embedding matrix; there is no
 *     SF_UNIT_LM_HEAD unit (its numel is 0) and the embedding's gradient is
 *     the sum of both uses.
 *   bf16_adam_state: 0 = the host keeps Adam's moments in fp32 (28 bytes of
 *     host memory traffic per parameter and step); 1 = it keeps them as
 *     bf16, rounded stochastically (random bits: the lowbias32 hash of the
 *     element's index in its unit, keyed by step and unit; the low half-word
 *     rounds the first moment, the high half-word the second), which
 *     cuts that traffic to 20 bytes and the host state from 14 to 10 bytes
 *     per parameter.  The update arithmetic stays fp32.
 *   fp16_grads: 0 = weight gradients leave the GPU as bf16; 1 = as fp16
 *     multiplied by a loss scale (3 more mantissa bits; the scale keeps small
 *     gradients out of fp16's subnormal range).  The host divides the scale
 *     out; a unit whose gradients overflowed keeps its weights and moments
 *     for that step (counted in sf_stats.skipped_updates).  The scale halves
 *     after a step in which an update was skipped and doubles after 1000
 *     steps without one (with async_update the count of a step is complete
 *     one step later).
 *   loss_scale: the initial scale for fp16_grads (0 = 65536; at most 2^24). */
typedef struct {
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int32_t max_batch, max_seq;
  int32_t ring_slots;
  int32_t lce_chunk_rows;
  int32_t retain_grads;
  float rms_eps, rope_base;
  int32_t device;
  int32_t adam_threads;
  int32_t wait_timeout_ms;
  int32_t async_update;
  int32_t offload_activations;
  int32_t deterministic;
  int32_t qkv_bias;
  int32_t tie_embeddings;
  int32_t bf16_adam_state;
  int32_t fp16_grads;
  float loss_scale;
} sf_config;

/* Adam hyper-parameters (bias-corrected; weight_decay is decoupled, AdamW). */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
} sf_adam;

/* Counters of the last sf_train_step (device times from CUDA events on the
 * stream each kernel was launched on). */
typedef struct {
  double step_ms;          /* compute stream, first to last operation of the step */
  double gemm_ms;          /* sum of tcgen05 GEMM launch durations */
  double gemm_flops;       /* algorithmic FLOPs of those launches (2*M*N*K each) */
  double attn_ms;          /* attention forward + backward kernels */
  double attn_flops;       /* algorithmic causal attention FLOPs */
  double h2d_bytes;        /* bytes copied host -> device during the step */
  double d2h_bytes;        /* bytes copied device -> host during the step */
  double host_adam_ms;     /* wall time the Adam workers spent updating */
  double host_wait_ms;     /* wall time sf_train_step blocked after the GPU finished */
  int64_t gemm_launches;
  int64_t kernel_launches; /* all kernels of this library launched in the step */
  int32_t timing_enabled;
  /* per decoder layer, averaged over the step (timing enabled): */
  double fwd_layer_ms;     /* forward compute (compute stream) */
  double bwd_layer_ms;     /* recompute + backward compute (compute stream) */
  double d2h_layer_ms;     /* gradient pack copy to the host (copy stream) */
  double update_layer_ms;  /* host Adam of one layer (wall time, update thread) */
  double loss_scale;       /* fp16_grads: the scale of this step's gradients; else 0 */
  int64_t skipped_updates; /* fp16_grads: unit updates skipped for overflow, in total */
  /* the compute stream's timeline (timing enabled): */
  double head_ms;          /* final norm + fused LM head / cross-entropy, forward and backward */
  double compute_ms;       /* all layer forwards, recompute-and-backwards and the head */
  double exposed_ms;       /* step_ms - compute_ms: time the compute stream waited, mostly
                              for weight / checkpoint copies that compute did not hide */
} sf_stats;

/* ---------------------------------------------------------------- model API */

/* Number of fp32 values of `unit` (see SF_UNIT_*): for a decoder layer the
 * concatenation g1[d], Wq[Hq*hd, d], Wk[Hkv*hd, d], Wv[Hkv*hd, d],
 * (with qkv_bias: bq[Hq*hd], bk[Hkv*hd], bv[Hkv*hd],) Wo[d, Hq*hd], g2[d],
 * Wg[F, d], Wu[F, d], Wd[d, F].  0 for a bad unit, and for SF_UNIT_LM_HEAD
 * when tie_embeddings is set. */
size_t sf_unit_numel(const sf_config* cfg, int32_t unit);

/* Validate cfg, allocate the ring slots, checkpoint and workspace buffers on
 * the device, pinned host buffers for every unit, fp32 master / Adam state in
 * host memory, streams, events and the host worker threads.  Every buffer the
 * step needs is allocated here (the step itself allocates nothing).
 * Source: gist.science summary, technical summary 2.B "Efficiënt Heterogeen
 * Geheugenbeheer", item "Pre-allocated GPU Cache Queue" (the
 * GPU holds a small window of layer units, reused without new allocation;
 * here ring_slots identical buffers of one layer's weights and gradients)
 * and "Layer-Adam Optimizer" (optimizer state in host memory); the
 * sciencestack abstract page, Abstract (state in CPU memory, GPU as a
 * compute engine over a window of layers).
 * Errors: SF_EINVAL (bad cfg), SF_ENOMEM, SF_ECUDA. */
int sf_init_model(const sf_config* cfg, sf_ctx** out);

/* Release everything the context owns.  NULL is a no-op. */
void sf_free(sf_ctx* ctx);

/* Message of the last error on ctx ("" if none); NULL ctx gives the message
 * of the last failed sf_init_model on this thread.  Owned by the library. */
const char* sf_last_error(const sf_ctx* ctx);

/* Set the fp32 master weights of `unit` (numel == sf_unit_numel) and reset
 * its Adam moments; the bf16 copy that streams to the GPU is rounded from it
 * (round-to-nearest-even).
 * Source: gist.science summary, technical summary 2.B "Gedeelde
 * CPU-buffers" (the fp32 -> bf16/fp16 conversion lives in fixed host
 * buffers that the layer's weights stream from) and 2.A (parameters of layer
 * L_i are fetched host-to-device ahead of their use).
 * Errors: SF_EINVAL, SF_ESTATE. */
int sf_load_layer_weights(sf_ctx* ctx, int32_t unit, const float* fp32_master, size_t numel);

/* One training step on tokens/labels [batch, seq] (int32, host memory):
 * forward over all layers through the GPU ring, fused LM-head cross-entropy,
 * recompute-and-backward over the layers in reverse order, gradient
 * streaming to the host and, if adam != NULL, the Adam update of every unit
 * (adam == NULL: gradients only, weights unchanged).
 * Source: gist.science summary, technical summary 2.A "Light-Weight
 * Asynchronous Engine" (after layer L_i's backward its gradients go to host
 * memory asynchronously while the GPU runs L_{i-1}'s backward and fetches
 * L_{i-2}; separate CUDA streams for copies and compute; the condition
 * T_compute >= T_transfer + T_update), 2.C "Fused LinearCrossEntropy" (the
 * projection and the loss fused so the full logits never exist, with no
 * loss of accuracy) and 2.B "Layer-Adam Optimizer"; the sciencestack
 * abstract page, figure 3 and 5 captions (the backward overlaps the
 * parameter updates and the GPU-CPU transfers).  On return the loss is
 * ready and, unless async_update is set, every update is done.  tokens in
 * [0, vocab); labels in [0, vocab) or SF_IGNORE_INDEX; batch*seq <=
 * max_batch*max_seq and seq <= max_seq.  With no valid label the loss and all
 * gradients are 0.  Errors: SF_EINVAL, SF_ECUDA, SF_ETIMEOUT, SF_EDEVICE,
 * SF_ESTATE. */
int sf_train_step(sf_ctx* ctx, const int32_t* tokens, const int32_t* labels, int32_t batch,
                  int32_t seq, const sf_adam* adam);

/* Gradient accumulation: one optimizer step over n_micro micro-batches of
 * batch x seq tokens each (tokens, labels: [n_micro, batch, seq] int32).  The
 * micro-batches run through the ring one after another; each one's gradients
 * are added into fp32 sums on the host (allocated on the first call with
 * n_micro > 1: 4 bytes per parameter), and the host update, overlapped with
 * the last micro-batch's backward as in sf_train_step, uses the sums.  The
 * result equals one sf_train_step over the n_micro * batch sequences: the
 * loss is the mean over every valid label of the step, and sf_get_grads
 * returns the summed gradients.  Same errors as sf_train_step; every
 * micro-batch is checked before the first one runs. */
int sf_train_step_accum(sf_ctx* ctx, const int32_t* tokens, const int32_t* labels,
                        int32_t n_micro, int32_t batch, int32_t seq, const sf_adam* adam);

/* Gradient of the last step for `unit`, in sf_unit_numel order, upcast from
 * the bf16 values that were streamed to the host (the embedding gradient is
 * accumulated in fp32).  Needs retain_grads = 1, else SF_ESTATE.
 * Source: gist.science summary, technical summary 2.B "Gedeelde CPU-buffers"
 * (gradients cast to bf16/fp16 and kept in shared fixed host buffers) and
 * 2.A (the d2h transfer of a finished layer's gradients). */
int sf_get_grads(sf_ctx* ctx, int32_t unit, float* out, size_t numel);

/* Current fp32 master weights of `unit`.  Errors: SF_EINVAL. */
int sf_get_weights(sf_ctx* ctx, int32_t unit, float* out, size_t numel);

/* Checkpointing of the optimizer.  sf_get_adam_state copies a unit's Adam
 * moments (first into m, second into v; fp32, the caller's order, numel =
 * sf_unit_numel) after waiting for pending updates; sf_set_adam_state
 * restores them (with bf16_adam_state they are rounded to nearest bf16).
 * sf_get_adam_step / sf_set_adam_step read and set the step count t of the
 * bias corrections (the next update uses t + 1).  Together with
 * sf_get_weights / sf_load_layer_weights (which zeroes the moments, so load
 * the weights first) they save and resume training exactly.  Errors:
 * SF_EINVAL (bad unit, numel or pointer), SF_ETIMEOUT / SF_ESTATE from the
 * wait for pending updates. */
int sf_get_adam_state(sf_ctx* ctx, int32_t unit, float* m, float* v, size_t numel);
int sf_set_adam_state(sf_ctx* ctx, int32_t unit, const float* m, const float* v, size_t numel);
int sf_get_adam_step(sf_ctx* ctx, int64_t* t);
int sf_set_adam_step(sf_ctx* ctx, int64_t t);

/* Wait (bounded by wait_timeout_ms) until every host update posted by the
 * steps so far is done; returns the first error a pending update reported.
 * A no-op when async_update is 0.  Errors: SF_ETIMEOUT, SF_ESTATE. */
int sf_sync(sf_ctx* ctx);

/* Loss of the last step: the mean token cross-entropy over the valid labels.
 * Source: gist.science summary, technical summary 2.C "Fused
 * LinearCrossEntropy" (the loss computed inside the fused output layer) and
 * section 4 "Betekenis en Impact" (standard training objectives).
 * Errors: SF_ESTATE before the first step. */
int sf_loss(sf_ctx* ctx, float* out);

/* The fused LM head + cross-entropy as a standalone call on host buffers (for
 * a head-only workload such as a large-vocabulary stress test): h bf16 [n, d],
 * w bf16 [v, d], labels int32 [n] where ignore_index marks ignored rows (any
 * other label must lie in [0, v)).  Writes loss (mean over valid rows), dh
 * bf16 [n, d] and dw fp32 [v, d], with the same kernels and chunked logits as
 * the training step.  ctx may be NULL (then the current device is used); the
 * call stages its inputs in device memory it allocates and frees.  Errors:
 * SF_EINVAL (sizes, pointers, labels), SF_ENOMEM, SF_ECUDA, SF_EDEVICE. */
int sf_lce_step(sf_ctx* ctx, const uint16_t* h, const uint16_t* w, const int32_t* labels,
                int64_t n, int32_t d, int32_t v, int32_t ignore_index, float* loss, uint16_t* dh,
                float* dw);

/* Per-kernel timing of the steps that follow: 1 records CUDA events around
 * every GEMM and attention launch (small overhead), 0 turns it off. */
int sf_set_timing(sf_ctx* ctx, int32_t enabled);

/* Counters of the last step. */
int sf_get_stats(const sf_ctx* ctx, sf_stats* out);

/* Host timeline of the engine, for showing overlap: one record per event,
 * t_ms from context creation (steady clock).  kind: 1 step begins, 2 batch
 * gathered, 3 wait for a unit's update begins, 4 that wait ends, 5 update task
 * begins (unit), 6 update task ends (unit), 7 the step's GPU work is done,
 * 8 step returns.  unit: layer index or SF_UNIT_*, -9 when not applicable.
 * The last 8192 records are kept; sf_get_trace copies up to cap of them
 * (oldest first) into out, sets *n and clears the record. */
typedef struct {
  double t_ms;
  int32_t kind;
  int32_t unit;
} sf_trace_event;
int sf_get_trace(sf_ctx* ctx, sf_trace_event* out, int32_t cap, int32_t* n);

/* Host memory bandwidth with the access pattern of the host Adam update:
 * per element, read 2 + 12 bytes and write 12 + 2 bytes, over `bytes` bytes
 * of freshly allocated host memory, on `threads` threads (0 = all cores);
 * best of three passes, in GB/s of read plus written bytes.  Allocates and
 * frees its own buffers.  Errors: SF_EINVAL, SF_ENOMEM. */
int sf_probe_host_bandwidth(int32_t threads, int64_t bytes, double* gbs);

/* Host-side fault injection for tests (no GPU fault is ever made):
 *   what = 1: the Adam worker fails on unit `arg` of the next step;
 *   what = 2: the Adam worker sleeps `arg` ms before each update;
 *   what = 0: clear.  */
int sf_debug_inject(sf_ctx* ctx, int32_t what, int32_t arg);

/* ---------------------------------------------------------------- kernel API
 * Single operations of the step on device pointers, launched on `stream`
 * (a cudaStream_t; NULL = the legacy default stream) and asynchronous like any
 * kernel launch.  Every scratch buffer is passed in by the caller; the first
 * call on a device also creates the 4-byte device error word that
 * sf_op_device_error reads.
 * Errors: SF_EINVAL for bad sizes / alignment (16-byte aligned bases and row
 * strides that are multiples of 8 elements), SF_ECUDA for a failed launch.
 * bf16 arguments are uint16 bit patterns of bfloat16. */

/* Dense bf16 GEMM on the tcgen05 tensor cores, fp32 accumulation.
 * layout 0 (NT): C[M,N] = alpha * A[M,K] * B[N,K]^T   (projection forward)
 * layout 1 (NN): C[M,N] = alpha * A[M,K] * B[K,N]     (input gradient)
 * layout 2 (TN): C[M,N] = alpha * A[K,M]^T * B[K,N]   (weight gradient)
 * epi 0: C bf16; 1: C fp32; 2: C fp32 = R + alpha*AB (R may alias C);
 * epi 3: C fp32 += alpha*AB.  lda/ldb/ldc/ldr are row strides in elements. */
int sf_op_gemm(int32_t layout, int32_t epi, int64_t M, int64_t N, int64_t K, const void* A,
               int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, const float* R,
               int64_t ldr, float alpha, void* stream);

/* C[M,N] bf16 = alpha * A[M,K] * B[N,K]^T + bias[N]: a projection forward with
 * a bias (the Q, K, V projections of Qwen-family models), the bias added to
 * the fp32 accumulator before the rounding.  bias bf16 [N], 64-byte aligned;
 * the other arguments as for sf_op_gemm with layout 0. */
int sf_op_gemm_bias(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                    int64_t ldb, void* C, int64_t ldc, const uint16_t* bias, float alpha,
                    void* stream);

/* Gradient of a bias: db[c] = sum over the rows r of dy[r, c], dy bf16 [rows,
 * cols] with row stride ld (cols even, ld even, 4-byte aligned), db bf16
 * [cols]; fp32 accumulation in a fixed order (bit-reproducible).  part: fp32
 * scratch of sf_op_bias_grad_scratch(rows, cols) floats. */
int sf_op_bias_grad(const uint16_t* dy, int64_t ld, int64_t rows, int32_t cols, float* part,
                    uint16_t* db, void* stream);
int64_t sf_op_bias_grad_scratch(int64_t rows, int32_t cols);

/* y[r] = bf16(g * x[r] / sqrt(mean(x[r]^2) + eps)), rstd[r] = 1/sqrt(...);
 * x fp32 [rows, d], g bf16 [d], y bf16 [rows, d], rstd fp32 [rows];
 * d a multiple of 8 in [8, 16384] (SF_EINVAL otherwise). */
int sf_op_rmsnorm_fwd(const float* x, const uint16_t* g, uint16_t* y, float* rstd, int64_t rows,
                      int32_t d, float eps, void* stream);

/* Backward of sf_op_rmsnorm_fwd given dy (fp32 [rows, d], the gradient of y):
 * dx = dres + rstd*(g*dy - xhat*mean(g*dy*xhat)) (fp32; dres may be NULL),
 * dxb = bf16(dx), dg = bf16(sum_r dy*xhat) [d].  scratch: fp32 of
 * sf_op_rmsnorm_bwd_scratch(rows, d) elements. */
int sf_op_rmsnorm_bwd(const float* x, const uint16_t* g, const float* rstd, const float* dy,
                      const float* dres, float* dx, uint16_t* dxb, uint16_t* dg, float* scratch,
                      int64_t rows, int32_t d, void* stream);
int64_t sf_op_rmsnorm_bwd_scratch(int64_t rows, int32_t d);

/* Host table of (cos, sin) of s * base^(-2j/head_dim), s < seq, j < head_dim/2,
 * written as float pairs [seq, head_dim/2, 2] to `out` (host memory). */
int sf_rope_table(int32_t seq, int32_t head_dim, float rope_base, float* out);

/* Rotary embedding in place on the first `heads` heads of each row of
 * x [tokens, ld] (bf16; position s = token % seq): pair (j, j + hd/2) rotated by
 * the table angle; inverse = 1 rotates by the opposite angle.  table: device
 * copy of sf_rope_table. */
int sf_op_rope(uint16_t* x, int64_t ld, int64_t tokens, int32_t seq, int32_t heads,
               int32_t head_dim, const float* table, int32_t inverse, void* stream);

/* Causal GQA attention forward.  qkv bf16 [B*S, (Hq+2Hkv)*hd] (Q heads, then K
 * heads, then V heads); o bf16 [B*S, Hq*hd]; lse fp32 [B, Hq, S] (natural
 * log-sum-exp of the scaled scores).  Scale 1/sqrt(hd). */
int sf_op_attn_fwd(const uint16_t* qkv, uint16_t* o, float* lse, int32_t B, int32_t S,
                   int32_t Hq, int32_t Hkv, int32_t hd, void* stream);

/* Backward of sf_op_attn_fwd: writes dQ, dK, dV into dqkv (same layout as qkv);
 * when table != NULL the inverse rotary embedding is applied to dQ and dK (the
 * gradient reaches the pre-rotation projections).  Scratch: delta fp32
 * [B*Hq*S]; dq_acc fp32 [B*S*Hq*hd] when deterministic == 0 (contributions
 * added in arrival order), or [ceil(S/128) * B*S*Hq*hd] when deterministic
 * != 0 (one slot per 128-key block, summed in key order: the result is
 * bit-reproducible).  dq_acc must be 16-byte aligned. */
int sf_op_attn_bwd(const uint16_t* qkv, const uint16_t* o, const uint16_t* dout,
                   const float* lse, float* delta, float* dq_acc, uint16_t* dqkv, int32_t B,
                   int32_t S, int32_t Hq, int32_t Hkv, int32_t hd, const float* table,
                   int32_t deterministic, void* stream);

/* m = silu(a) * b with ab = [a | b] bf16 [rows, 2*ffn]; m bf16 [rows, ffn]. */
int sf_op_swiglu_fwd(const uint16_t* ab, uint16_t* m, int64_t rows, int32_t ffn, void* stream);
/* dab = [dm * b * s(1 + a(1-s)) | dm * silu(a)], s = sigmoid(a). */
int sf_op_swiglu_bwd(const uint16_t* dm, const uint16_t* ab, uint16_t* dab, int64_t rows,
                     int32_t ffn, void* stream);

/* The Q/K/V projection with its rotary embedding, in one GEMM: the fp32
 * accumulator of A[M,K] * B[N,K]^T (plus bias[N] when bias != NULL, added
 * first, 64-byte aligned) is rotated on the columns [0, rope_cols) (heads of
 * head_dim columns, pair (j, j + head_dim/2) rotated by the table angle of
 * position row % seq, as sf_op_rope) and rounded to bf16 once into C[M,N].
 * head_dim in {64, 128}; N and rope_cols multiples of head_dim; table: device
 * copy of sf_rope_table (16-byte aligned).  Other arguments as sf_op_gemm. */
int sf_op_gemm_qkv(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                   int64_t ldb, uint16_t* C, int64_t ldc, const uint16_t* bias, const float* table,
                   int32_t seq, int32_t rope_cols, int32_t head_dim, void* stream);

/* The gate/up projection with SwiGLU, in one GEMM: B = [Wg; Wu] bf16 [2F, K]
 * (Wu starts F rows after Wg, same row stride ldb); a = A Wg^T and b = A Wu^T
 * (fp32 accumulators of the same tile), m[M,F] bf16 = silu(a) * b.  When
 * ab != NULL the fp32 a and b are also written: ab[r, j] = a, ab[r, F + j] = b
 * (row stride ldab >= 2F, 16-byte aligned), for the backward.  F multiple of
 * 8.  Other arguments as sf_op_gemm with layout 0. */
int sf_op_gemm_swiglu(int64_t M, int64_t F, int64_t K, const void* A, int64_t lda,
                      const void* B, int64_t ldb, uint16_t* m, int64_t ldm, float* ab,
                      int64_t ldab, void* stream);

/* The down projection's input gradient taken through SwiGLU, in one GEMM:
 * dm = dy[M,K] * wd[K,F] (layout 1, fp32 accumulator, never stored), then with
 * a = ab[r, j], b = ab[r, F + j] (fp32, from sf_op_gemm_swiglu) and
 * s = sigmoid(a): dab[r, j] = bf16(dm b s (1 + a (1 - s))),
 * dab[r, F + j] = bf16(dm a s).  ldab, lddab >= 2F; F multiple of 8. */
int sf_op_gemm_swiglu_bwd(int64_t M, int64_t F, int64_t K, const void* dy, int64_t lddy,
                          const void* wd, int64_t ldw, const float* ab, int64_t ldab,
                          uint16_t* dab, int64_t lddab, void* stream);

/* Fused chunked LM-head + cross-entropy forward and backward on device data:
 * z = h W^T in fp32 (never stored beyond one chunk of `chunk_rows` rows),
 * loss = (1/n_valid) sum_valid (logsumexp(z_t) - z_t[label_t]),
 * dh = dZ W (fp32 [n, d]), dw = dZ^T h (fp32 [v, d]) with
 * dZ = (softmax(z) - onehot)/n_valid on valid rows, 0 on ignored rows.
 * h bf16 [n, d], w bf16 [v, d], labels int32 [n] (device), loss fp32 [1].
 * A negative label (SF_IGNORE_INDEX among them) ignores its row; n_valid is
 * the number of labels in [0, v) (the caller counts it).  The labels live on
 * the device, so this call cannot check them: a label >= v sets the device
 * error word to 4 (sf_op_device_error) and its row is ignored.
 * workspace: sf_op_lce_workspace_bytes(n, v, chunk_rows) bytes, 256-aligned:
 * a chunk's fp32 logits and bf16 dZ (6 bytes per logit) and n fp32 row losses.
 * With c = min(chunk_rows, n) and r(x) = x rounded up to 256: fp32 logits
 * [c, v] at byte 0, bf16 dZ [c, v] at r(4cv), row losses [n] (lse - z[label],
 * 0 on ignored rows) at r(4cv) + r(2cv).  On return dZ holds the last chunk's
 * rows and the row losses all n rows; the logits area is overwritten. */
int sf_op_lce(const uint16_t* h, const uint16_t* w, const int32_t* labels, int64_t n, int32_t d,
              int32_t v, int64_t n_valid, int64_t chunk_rows, void* workspace, float* loss,
              float* dh, float* dw, void* stream);
int64_t sf_op_lce_workspace_bytes(int64_t n, int32_t v, int64_t chunk_rows);
/* The number of kernels the calling thread's last successful sf_op_lce call
 * launched (per chunk: the logits GEMM, the cross-entropy rows, the dH GEMM
 * and, when it ran as vocabulary ranges, their sum, the dW GEMM; then the loss
 * sum); 0 before any call.  No device work. */
int64_t sf_op_lce_launches(void);

/* sf_op_rmsnorm_bwd_noalloc: the same operation and results as
 * sf_op_rmsnorm_bwd, for callers that cannot allocate device memory (for
 * instance code inside a host application whose memory manager owns the
 * whole device budget, or a latency-critical loop where a cudaMalloc, which
 * can synchronise the device and can fail, is not acceptable).  It takes no
 * scratch argument and calls no allocating routine: the partial sums of the
 * gain gradient live in a fixed array of SF_STATIC_SCRATCH_FLOATS floats
 * (16 MiB) that the library reserves on every GPU that loads it, until the
 * process exits.  The paper has no counterpart to this entry point.
 *   - Size limit: returns SF_EINVAL when the row partition needs more than
 *     SF_STATIC_SCRATCH_FLOATS floats, i.e. when P * d > 4194304, with
 *     P = min(rows, 2 * number of SMs of the current device) (on a 152-SM
 *     GPU: any rows for d <= 13792, at most 256 rows for d = 16384).
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call shares the one array: calls whose kernels overlap on the GPU
 *     (other streams, other host threads) race and must not be issued.  Each
 *     call overwrites every partial it reads, so nothing has to be cleared.
 * Other arguments, layouts and errors: as sf_op_rmsnorm_bwd. */
#define SF_STATIC_SCRATCH_FLOATS 4194304
int sf_op_rmsnorm_bwd_noalloc(const float* x, const uint16_t* g, const float* rstd,
                              const float* dy, const float* dres, float* dx, uint16_t* dxb,
                              uint16_t* dg, int64_t rows, int32_t d, void* stream);

/* Read and clear the device error word of the kernel API on the current
 * device.  0: no error; 1, 2, 3: a bounded wait ran out in a GEMM, an
 * attention or a cross-entropy kernel; 4: sf_op_lce met a label at or beyond
 * the vocabulary.  The first code a launch writes stays.  Synchronises the
 * device. */
int sf_op_device_error(int32_t* out);

#ifdef __cplusplus
}
#endif
#endif /* SF_H_ */
