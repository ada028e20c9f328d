// Internal launchers of the CUDA kernels (host-side declarations).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace sf {

// Codes written to the device error word (the first one a launch meets).
enum DevErr : int {
  kDevOk = 0,
  kDevGemmTimeout = 1,
  kDevAttnTimeout = 2,
  kDevCeTimeout = 3,
  kDevCeBadLabel = 4,  // a label at or beyond the vocabulary (the row is ignored)
};

// Operand layouts of C[M,N] = A * B (all matrices row-major in memory):
//   kNT: A [M,K] (K contiguous), B [N,K] (K contiguous)   -> Y = X W^T
//   kNN: A [M,K] (K contiguous), B [K,N] (N contiguous)   -> dX = dY W
//   kTN: A [K,M] (M contiguous), B [K,N] (N contiguous)   -> dW = dY^T X
enum GemmLayout : int { kNT = 0, kNN = 1, kTN = 2 };
// Epilogues: C bf16 = alpha*acc | C f32 = alpha*acc | C f32 = R + alpha*acc | C f32 += alpha*acc
// | C bf16 = alpha*acc + bias[col] (bias bf16 [N], 64-byte aligned; layout kNT only)
// | C fp16 = alpha*acc (layout kTN only: scaled fp16 weight gradients)
// | kEpiQKV (layout kNT): y = alpha*acc (+ bias[col] when bias != null), then the
//   rotary embedding on the columns below rope_cols (heads of hd columns, pair
//   (j, j + hd/2), position row % seq, (cos, sin) from cs[pos * hd/2 + j]) and
//   one bf16 rounding: the Q/K/V projection with its rotation
// | kEpiGLU (layout kNT): B holds 2N rows, [Bg; Bu]; a = alpha*A Bg^T and
//   b = alpha*A Bu^T share one accumulator tile, C bf16 [M, N] = silu(a) * b;
//   when aux != null, a and b are also stored as fp32: aux[r, j] = a,
//   aux[r, N + j] = b (the SwiGLU forward of the gate/up projection)
// | kEpiGLUBwd (layout kNN): dm = alpha*acc, with a = R[r, j], b = R[r, N + j]
//   (fp32) C[r, j] = bf16(dm b s (1 + a (1 - s))), C[r, N + j] = bf16(dm a s),
//   s = sigmoid(a) (the down projection's input gradient through SwiGLU)
// | kEpiBF16Acc (layout kTN): C bf16 = alpha*acc + R (R fp32, may be null):
//   the last of a chunked sum of weight gradients, rounded once
enum GemmEpi : int {
  kEpiBF16 = 0, kEpiF32 = 1, kEpiF32Add = 2, kEpiF32Acc = 3, kEpiBF16Bias = 4, kEpiF16 = 5,
  kEpiQKV = 6, kEpiGLU = 7, kEpiGLUBwd = 8, kEpiBF16Acc = 9
};

struct GemmArgs {
  int layout = kNT, epi = kEpiBF16;
  int64_t M = 0, N = 0, K = 0;
  const void* A = nullptr;
  int64_t lda = 0;
  const void* B = nullptr;
  int64_t ldb = 0;
  void* C = nullptr;
  int64_t ldc = 0;
  const float* R = nullptr;
  int64_t ldr = 0;
  float alpha = 1.f;
  const void* bias = nullptr;  // kEpiBF16Bias; kEpiQKV (optional)
  // kEpiQKV: rotation table (cos, sin) [seq, hd/2], columns [0, rope_cols) rotated
  const float2* cs = nullptr;
  int seq = 0, rope_cols = 0, hd = 0;
  // kEpiGLU: optional fp32 copy of the gate and up outputs, row stride ldaux
  float* aux = nullptr;
  int64_t ldaux = 0;
  // kEpiF32 only: up to splitk_max ranges of K run as separate work units
  // when that fills the SMs better; split 0 writes C, split s > 0 the fp32
  // slice ws + (s - 1) * M * ldc, and a fixed-order sum adds the slices into
  // C (ws: (splitk_max - 1) * M * ldc floats, or null for no split)
  int splitk_max = 1;
  float* ws = nullptr;
  // when set, the number of kernels the call launched is added to it
  int* launched = nullptr;
};

// Returns 0, or a negative status with a message in `why` (64 chars at least).
int gemm(const GemmArgs& a, int* dev_err, cudaStream_t st, char* why);
// Host-side argument check only (no CUDA call): 0 or -1.
int gemm_check(const GemmArgs& a, char* why);

// ---- elementwise / normalisation kernels (elementwise.cu)
void rmsnorm_fwd(const float* x, const __nv_bfloat16* g, __nv_bfloat16* y, float* rstd,
                 int64_t rows, int d, float eps, cudaStream_t st);
// dx = dres + rstd*(g*dy - xhat*mean(g*dy*xhat)); dxb = bf16(dx); dg partials [parts, d]
void rmsnorm_bwd(const float* x, const __nv_bfloat16* g, const float* rstd, const float* dy,
                 const float* dres, float* dx, __nv_bfloat16* dxb, float* dg_part, int parts,
                 int64_t rows, int d, cudaStream_t st);
int rmsnorm_bwd_parts(int64_t rows, int d);
void reduce_parts_bf16(const float* part, int parts, int d, __nv_bfloat16* out, cudaStream_t st);
// The same sum as fp16 after multiplying by scale (a scaled fp16 gradient).
void reduce_parts_f16(const float* part, int parts, int d, uint16_t* out, float scale,
                      cudaStream_t st);
// out[c] = bf16(sum over rows of x[r, c]) for x bf16 [rows, cols] (cols even, row
// stride ld, 4-byte aligned rows); part: fp32 scratch [parts, cols]
void bias_grad(const __nv_bfloat16* x, int64_t ld, int64_t rows, int cols, float* part, int parts,
               __nv_bfloat16* out, cudaStream_t st);
// the column sums as fp16 times scale
void bias_grad_f16(const __nv_bfloat16* x, int64_t ld, int64_t rows, int cols, float* part,
                   int parts, uint16_t* out, float scale, cudaStream_t st);
void rope_inplace(__nv_bfloat16* qkv, int64_t ld, int64_t tokens, int seq, int heads,
                  int head_dim, const float2* cs, int inverse, cudaStream_t st);
// The fused cross-entropy rows on fp32 logits z [rows, vocab] (vocab % 8 == 0,
// z 16-byte aligned): loss_rows[r] = lse - z[r, label] (0 when ignored) and
// dz [rows, vocab] bf16 = (softmax(z) - onehot) * inv_n (0 on ignored rows).
// A cluster of CTAs shares a row held in shared memory, so z is read once;
// a wait that runs out writes kDevCeTimeout to *err, and a label >= vocab
// writes kDevCeBadLabel (its row is then ignored).  Returns 0, or -1 when the
// launch fails.
int ce_rows_f32(const float* z, __nv_bfloat16* dz, const int32_t* labels, int64_t rows,
                int64_t vocab, float inv_n, float* loss_rows, int* err, cudaStream_t st);
// CTAs per row of the cross-entropy kernel for this vocabulary (0: one CTA
// reading the row twice, for rows beyond the clusters' shared memory).
int ce_cluster_size(int64_t vocab);
void swiglu_fwd(const __nv_bfloat16* ab, __nv_bfloat16* m, int64_t rows, int ffn,
                cudaStream_t st);
void swiglu_bwd(const __nv_bfloat16* dm, const __nv_bfloat16* ab, __nv_bfloat16* dab,
                int64_t rows, int ffn, cudaStream_t st);
void sum_f32(const float* x, int64_t n, float scale, float* out, cudaStream_t st);
void cast_f32_bf16(const float* x, __nv_bfloat16* y, int64_t n, cudaStream_t st);
// y = fp16(scale * x)
void cast_f32_f16(const float* x, uint16_t* y, int64_t n, float scale, cudaStream_t st);
void cast_bf16_f32(const __nv_bfloat16* x, float* y, int64_t n, cudaStream_t st);

// ---- attention (attention.cu).  qkv [T, (Hq+2Hkv)*hd] bf16, token t = b*S + s.
// Forward on tcgen05 (attention_tc.cu); a bounded wait that runs out writes
// kDevAttnTimeout to *err.
int attn_fwd(const __nv_bfloat16* qkv, __nv_bfloat16* o, float* lse, int B, int S, int Hq,
             int Hkv, int hd, int* err, cudaStream_t st);
// Backward on tcgen05 (attention_tc.cu).  delta: fp32 scratch [B, Hq, S].
// dq_acc: fp32 scratch, [T, Hq*hd] (zeroed inside, partials added in the
// order they arrive) or, when deterministic, [ceil(S/128)][T, Hq*hd] (one slot
// per 128-key block, summed in key order: bit-reproducible).  Writes dQ and dK
// (inverse RoPE applied when cs != null) and dV into dqkv.
int attn_bwd(const __nv_bfloat16* qkv, const __nv_bfloat16* o, const __nv_bfloat16* dout,
             const float* lse, float* delta, float* dq_acc, __nv_bfloat16* dqkv, int B, int S,
             int Hq, int Hkv, int hd, const float2* cs, bool deterministic, int* err,
             cudaStream_t st);
// delta[b, h, s] = sum_j dO * O over one head's row (attention.cu)
void attn_delta(const __nv_bfloat16* o, const __nv_bfloat16* dout, float* delta, int B, int S,
                int Hq, int hd, cudaStream_t st);
// dQ = scale * (accumulated or slot-summed dq_acc), inverse RoPE, into the
// query columns of dqkv (attention.cu); slots = 0 for one accumulated buffer.
void attn_dq_finalize(const float* dq_acc, __nv_bfloat16* dqkv, int B, int S, int Hq, int Hkv,
                      int hd, float scale, const float2* cs, int slots, cudaStream_t st);

int num_sms();

}  // namespace sf
