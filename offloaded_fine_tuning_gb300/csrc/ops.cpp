// Kernel-level C ABI (sf.h, "kernel API"): single operations of the step on
// caller-owned device buffers.  Argument checks happen here, on the host,
// before any launch; the kernels themselves assume checked arguments.
#include <cuda_runtime.h>

#include <cmath>
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "sf.h"
#include "sf_internal.h"

namespace {

using bf16 = __nv_bfloat16;

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One device error word per device, created on first use.
constexpr int kMaxDev = 64;
int* g_err[kMaxDev] = {nullptr};
std::mutex g_err_m;

int* dev_err_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> l(g_err_m);
  if (!g_err[dev]) {
    int* p = nullptr;
    if (cudaMalloc(&p, sizeof(int)) != cudaSuccess) return nullptr;
    if (cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return nullptr;
    g_err[dev] = p;
  }
  return g_err[dev];
}

cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }
int launched() { return cudaGetLastError() == cudaSuccess ? SF_OK : SF_ECUDA; }

// Kernels launched by the calling thread's last sf_op_lce call.
thread_local int64_t lce_launches = 0;

}  // namespace

extern "C" {

int sf_op_gemm(int32_t layout, int32_t epi, int64_t M, int64_t N, int64_t K, const void* A,
               int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, const float* R,
               int64_t ldr, float alpha, void* stream) {
  if (epi < 0 || epi > 3 || layout < 0 || layout > 2) return SF_EINVAL;
  sf::GemmArgs g;
  g.layout = layout; g.epi = epi; g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = lda; g.B = B; g.ldb = ldb; g.C = C; g.ldc = ldc; g.R = R; g.ldr = ldr;
  g.alpha = alpha;
  char why[128];
  if (sf::gemm_check(g, why) != 0) return SF_EINVAL;
  if (M == 0 || N == 0) return SF_OK;
  int* err = dev_err_word();
  if (!err) return SF_ECUDA;
  const int st = sf::gemm(g, err, S(stream), why);
  if (st == -1) return SF_EINVAL;
  if (st != 0) return SF_ECUDA;
  return SF_OK;
}

int sf_op_gemm_bias(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                    int64_t ldb, void* C, int64_t ldc, const uint16_t* bias, float alpha,
                    void* stream) {
  sf::GemmArgs g;
  g.layout = sf::kNT; g.epi = sf::kEpiBF16Bias; g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = lda; g.B = B; g.ldb = ldb; g.C = C; g.ldc = ldc; g.alpha = alpha;
  g.bias = bias;
  char why[128];
  if (sf::gemm_check(g, why) != 0) return SF_EINVAL;
  if (M == 0 || N == 0) return SF_OK;
  int* err = dev_err_word();
  if (!err) return SF_ECUDA;
  const int st = sf::gemm(g, err, S(stream), why);
  if (st == -1) return SF_EINVAL;
  if (st != 0) return SF_ECUDA;
  return SF_OK;
}

int64_t sf_op_bias_grad_scratch(int64_t rows, int32_t cols) {
  if (rows < 0 || cols < 0) return -1;
  return (int64_t)sf::rmsnorm_bwd_parts(rows, cols) * cols;
}

int sf_op_bias_grad(const uint16_t* dy, int64_t ld, int64_t rows, int32_t cols, float* part,
                    uint16_t* db, void* stream) {
  if (rows < 0 || cols < 2 || cols % 2 || ld < cols || ld % 2) return SF_EINVAL;
  if (!dy || !part || !db || (reinterpret_cast<uintptr_t>(dy) & 3)) return SF_EINVAL;
  if (rows == 0) return SF_EINVAL;
  sf::bias_grad(reinterpret_cast<const bf16*>(dy), ld, rows, cols, part,
                sf::rmsnorm_bwd_parts(rows, cols), reinterpret_cast<bf16*>(db), S(stream));
  return cudaGetLastError() == cudaSuccess ? SF_OK : SF_ECUDA;
}

int sf_op_rmsnorm_fwd(const float* x, const uint16_t* g, uint16_t* y, float* rstd, int64_t rows,
                      int32_t d, float eps, void* stream) {
  if (rows < 0 || d < 8 || d % 8 || d > 16384 || !(eps > 0.f)) return SF_EINVAL;
  if (rows == 0) return SF_OK;
  if (!x || !g || !y || !rstd || !al16(x) || !al16(y) || (reinterpret_cast<uintptr_t>(g) & 7))
    return SF_EINVAL;
  sf::rmsnorm_fwd(x, reinterpret_cast<const bf16*>(g), reinterpret_cast<bf16*>(y), rstd, rows, d,
                  eps, S(stream));
  return launched();
}

int64_t sf_op_rmsnorm_bwd_scratch(int64_t rows, int32_t d) {
  return (int64_t)sf::rmsnorm_bwd_parts(rows, d) * d;
}

int sf_op_rmsnorm_bwd(const float* x, const uint16_t* g, const float* rstd, const float* dy,
                      const float* dres, float* dx, uint16_t* dxb, uint16_t* dg, float* scratch,
                      int64_t rows, int32_t d, void* stream) {
  if (rows < 1 || d < 8 || d % 8 || d > 16384) return SF_EINVAL;
  if (!x || !g || !rstd || !dy || !dx || !dxb || !dg || !scratch) return SF_EINVAL;
  if (!al16(x) || !al16(dy) || !al16(dx) || !al16(dxb) || !al16(scratch) ||
      (dres && !al16(dres)) || (reinterpret_cast<uintptr_t>(g) & 7))
    return SF_EINVAL;
  const int parts = sf::rmsnorm_bwd_parts(rows, d);
  sf::rmsnorm_bwd(x, reinterpret_cast<const bf16*>(g), rstd, dy, dres, dx,
                  reinterpret_cast<bf16*>(dxb), scratch, parts, rows, d, S(stream));
  sf::reduce_parts_bf16(scratch, parts, d, reinterpret_cast<bf16*>(dg), S(stream));
  return launched();
}

int sf_rope_table(int32_t seq, int32_t head_dim, float rope_base, float* out) {
  if (seq < 1 || head_dim < 2 || head_dim % 2 || !(rope_base > 1.f) || !out) return SF_EINVAL;
  const int half = head_dim / 2;
  for (int j = 0; j < half; ++j) {
    const double inv_freq = std::pow((double)rope_base, -2.0 * j / head_dim);
    for (int s = 0; s < seq; ++s) {
      const double ang = (double)s * inv_freq;
      out[((int64_t)s * half + j) * 2 + 0] = (float)std::cos(ang);
      out[((int64_t)s * half + j) * 2 + 1] = (float)std::sin(ang);
    }
  }
  return SF_OK;
}

int sf_op_rope(uint16_t* x, int64_t ld, int64_t tokens, int32_t seq, int32_t heads,
               int32_t head_dim, const float* table, int32_t inverse, void* stream) {
  if (tokens < 0 || seq < 1 || heads < 1 || head_dim < 16 || head_dim % 16 || ld % 8 ||
      ld < (int64_t)heads * head_dim)
    return SF_EINVAL;
  if (tokens == 0) return SF_OK;
  if (!x || !table || !al16(x) || (reinterpret_cast<uintptr_t>(table) & 7)) return SF_EINVAL;
  sf::rope_inplace(reinterpret_cast<bf16*>(x), ld, tokens, seq, heads, head_dim,
                   reinterpret_cast<const float2*>(table), inverse, S(stream));
  return launched();
}

int sf_op_attn_fwd(const uint16_t* qkv, uint16_t* o, float* lse, int32_t B, int32_t S_,
                   int32_t Hq, int32_t Hkv, int32_t hd, void* stream) {
  if (B < 0 || S_ < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || (hd != 64 && hd != 128)) return SF_EINVAL;
  if (B == 0 || S_ == 0) return SF_OK;
  if (!qkv || !o || !lse || !al16(qkv) || !al16(o)) return SF_EINVAL;
  int* err = dev_err_word();
  if (!err) return SF_ECUDA;
  if (sf::attn_fwd(reinterpret_cast<const bf16*>(qkv), reinterpret_cast<bf16*>(o), lse, B, S_,
                   Hq, Hkv, hd, err, S(stream)) != 0)
    return SF_ECUDA;
  return SF_OK;
}

int sf_op_attn_bwd(const uint16_t* qkv, const uint16_t* o, const uint16_t* dout,
                   const float* lse, float* delta, float* dq_acc, uint16_t* dqkv, int32_t B,
                   int32_t S_, int32_t Hq, int32_t Hkv, int32_t hd, const float* table,
                   int32_t deterministic, void* stream) {
  if (B < 0 || S_ < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || (hd != 64 && hd != 128)) return SF_EINVAL;
  if (B == 0 || S_ == 0) return SF_OK;
  if (!qkv || !o || !dout || !lse || !delta || !dq_acc || !dqkv) return SF_EINVAL;
  if (!al16(qkv) || !al16(o) || !al16(dout) || !al16(dq_acc) || !al16(dqkv)) return SF_EINVAL;
  int* err = dev_err_word();
  if (!err) return SF_ECUDA;
  if (sf::attn_bwd(reinterpret_cast<const bf16*>(qkv), reinterpret_cast<const bf16*>(o),
                   reinterpret_cast<const bf16*>(dout), lse, delta, dq_acc,
                   reinterpret_cast<bf16*>(dqkv), B, S_, Hq, Hkv, hd,
                   reinterpret_cast<const float2*>(table), deterministic != 0, err, S(stream)) != 0)
    return SF_ECUDA;
  return SF_OK;
}

int sf_op_swiglu_fwd(const uint16_t* ab, uint16_t* m, int64_t rows, int32_t ffn, void* stream) {
  if (rows < 0 || ffn < 8 || ffn % 8) return SF_EINVAL;
  if (rows == 0) return SF_OK;
  if (!ab || !m || !al16(ab) || !al16(m)) return SF_EINVAL;
  sf::swiglu_fwd(reinterpret_cast<const bf16*>(ab), reinterpret_cast<bf16*>(m), rows, ffn, S(stream));
  return launched();
}

int sf_op_swiglu_bwd(const uint16_t* dm, const uint16_t* ab, uint16_t* dab, int64_t rows,
                     int32_t ffn, void* stream) {
  if (rows < 0 || ffn < 8 || ffn % 8) return SF_EINVAL;
  if (rows == 0) return SF_OK;
  if (!dm || !ab || !dab || !al16(dm) || !al16(ab) || !al16(dab)) return SF_EINVAL;
  sf::swiglu_bwd(reinterpret_cast<const bf16*>(dm), reinterpret_cast<const bf16*>(ab),
                 reinterpret_cast<bf16*>(dab), rows, ffn, S(stream));
  return launched();
}

int64_t sf_op_lce_workspace_bytes(int64_t n, int32_t v, int64_t chunk_rows) {
  if (n < 1 || v < 8 || chunk_rows < 1) return -1;
  const int64_t c = chunk_rows < n ? chunk_rows : n;
  const int64_t logits = (c * v * 4 + 255) / 256 * 256;  // fp32 logits of a chunk
  const int64_t dz = (c * v * 2 + 255) / 256 * 256;      // their bf16 dZ
  const int64_t rows = (n * 4 + 255) / 256 * 256;
  return logits + dz + rows;
}

int sf_op_lce(const uint16_t* h, const uint16_t* w, const int32_t* labels, int64_t n, int32_t d,
              int32_t v, int64_t n_valid, int64_t chunk_rows, void* workspace, float* loss,
              float* dh, float* dw, void* stream) {
  if (n < 1 || d < 8 || d % 8 || v < 8 || v % 8 || chunk_rows < 1 || n_valid < 0 || n_valid > n)
    return SF_EINVAL;
  if (!h || !w || !labels || !workspace || !loss || !dh || !dw) return SF_EINVAL;
  if (!al16(h) || !al16(w) || !al16(dh) || !al16(dw) || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return SF_EINVAL;
  int* err = dev_err_word();
  if (!err) return SF_ECUDA;
  const int64_t c = chunk_rows < n ? chunk_rows : n;
  char* ws = reinterpret_cast<char*>(workspace);
  float* zf = reinterpret_cast<float*>(ws);
  ws += (c * v * 4 + 255) / 256 * 256;
  bf16* dz = reinterpret_cast<bf16*>(ws);
  ws += (c * v * 2 + 255) / 256 * 256;
  float* loss_rows = reinterpret_cast<float*>(ws);
  const bf16* H = reinterpret_cast<const bf16*>(h);
  const bf16* W = reinterpret_cast<const bf16*>(w);
  const float inv_n = n_valid > 0 ? 1.f / (float)n_valid : 0.f;
  char why[128];
  cudaStream_t st = S(stream);
  int count = 0;  // kernels launched, for sf_op_lce_launches
  lce_launches = 0;
  for (int64_t r0 = 0; r0 < n; r0 += c) {
    const int64_t rows = (c < n - r0) ? c : n - r0;
    sf::GemmArgs z;
    z.layout = sf::kNT; z.epi = sf::kEpiF32; z.M = rows; z.N = v; z.K = d;
    z.A = H + r0 * d; z.lda = d; z.B = W; z.ldb = d; z.C = zf; z.ldc = v; z.launched = &count;
    if (sf::gemm(z, err, st, why) != 0) return SF_ECUDA;
    if (sf::ce_rows_f32(zf, dz, labels + r0, rows, v, inv_n, loss_rows + r0, err, st) != 0)
      return SF_ECUDA;
    ++count;
    // dH over up to four vocabulary ranges when that fills the SMs better; the
    // partial sums go to the chunk's fp32 logits, which the row kernel has read
    sf::GemmArgs gx;
    gx.layout = sf::kNN; gx.epi = sf::kEpiF32; gx.M = rows; gx.N = d; gx.K = v;
    gx.A = dz; gx.lda = v; gx.B = W; gx.ldb = d; gx.C = dh + r0 * d; gx.ldc = d;
    gx.splitk_max = (int)std::min<int64_t>(4, 1 + (c * (int64_t)v) / (rows * (int64_t)d));
    gx.ws = zf; gx.launched = &count;
    if (sf::gemm(gx, err, st, why) != 0) return SF_ECUDA;
    sf::GemmArgs gw;
    gw.layout = sf::kTN; gw.epi = r0 == 0 ? sf::kEpiF32 : sf::kEpiF32Acc; gw.M = v; gw.N = d;
    gw.K = rows; gw.A = dz; gw.lda = v; gw.B = H + r0 * d; gw.ldb = d; gw.C = dw; gw.ldc = d;
    gw.launched = &count;
    if (sf::gemm(gw, err, st, why) != 0) return SF_ECUDA;
  }
  sf::sum_f32(loss_rows, n, inv_n, loss, st);
  lce_launches = count + 1;
  return launched();
}

int64_t sf_op_lce_launches(void) { return lce_launches; }

// The fused-epilogue projections: argument checks in sf::gemm_check.
static int run_gemm(const sf::GemmArgs& g, cudaStream_t st) {
  char why[128];
  if (sf::gemm_check(g, why) != 0) return SF_EINVAL;
  if (g.M == 0 || g.N == 0) return SF_OK;
  int* err = dev_err_word();
  if (!err) return SF_ECUDA;
  const int rc = sf::gemm(g, err, st, why);
  if (rc == -1) return SF_EINVAL;
  return rc == 0 ? SF_OK : SF_ECUDA;
}

int sf_op_gemm_qkv(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                   int64_t ldb, uint16_t* C, int64_t ldc, const uint16_t* bias, const float* table,
                   int32_t seq, int32_t rope_cols, int32_t head_dim, void* stream) {
  sf::GemmArgs g;
  g.layout = sf::kNT; g.epi = sf::kEpiQKV; g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = lda; g.B = B; g.ldb = ldb; g.C = C; g.ldc = ldc; g.bias = bias;
  g.cs = reinterpret_cast<const float2*>(table); g.seq = seq; g.rope_cols = rope_cols; g.hd = head_dim;
  return run_gemm(g, S(stream));
}

int sf_op_gemm_swiglu(int64_t M, int64_t F, int64_t K, const void* A, int64_t lda,
                      const void* B, int64_t ldb, uint16_t* m, int64_t ldm, float* ab,
                      int64_t ldab, void* stream) {
  sf::GemmArgs g;
  g.layout = sf::kNT; g.epi = sf::kEpiGLU; g.M = M; g.N = F; g.K = K;
  g.A = A; g.lda = lda; g.B = B; g.ldb = ldb; g.C = m; g.ldc = ldm; g.aux = ab; g.ldaux = ldab;
  return run_gemm(g, S(stream));
}

int sf_op_gemm_swiglu_bwd(int64_t M, int64_t F, int64_t K, const void* dy, int64_t lddy,
                          const void* wd, int64_t ldw, const float* ab, int64_t ldab,
                          uint16_t* dab, int64_t lddab, void* stream) {
  sf::GemmArgs g;
  g.layout = sf::kNN; g.epi = sf::kEpiGLUBwd; g.M = M; g.N = F; g.K = K;
  g.A = dy; g.lda = lddy; g.B = wd; g.ldb = ldw; g.C = dab; g.ldc = lddab; g.R = ab; g.ldr = ldab;
  return run_gemm(g, S(stream));
}

int sf_op_device_error(int32_t* out) {
  if (!out) return SF_EINVAL;
  int* e = dev_err_word();
  if (!e) return SF_ECUDA;
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return SF_ECUDA;
  if (cudaMemcpy(&v, e, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SF_ECUDA;
  if (cudaMemset(e, 0, sizeof(int)) != cudaSuccess) return SF_ECUDA;
  *out = v;
  return SF_OK;
}

}  // extern "C"
