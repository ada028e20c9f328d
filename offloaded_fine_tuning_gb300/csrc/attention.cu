// Causal grouped-query attention, forward and backward, with online softmax
// (Milakov & Gimelshein 2018; the tiling of Dao et al., FlashAttention 2022):
// the S x S score matrix never leaves the chip.
//
// Inputs come straight from the QKV projection's output row [T, (Hq+2Hkv)*hd]
// (token t = b*S + s): query head h at column h*hd, kv head g at (Hq+g)*hd
// (K) and (Hq+Hkv+g)*hd (V); query head h reads kv head h / (Hq/Hkv).
//
// (The forward runs on the tcgen05 tensor cores: attention_tc.cu.)
// Backward: one CTA per (64-key block, kv head, batch); it walks every query
// head of its group and every 32-query block at or after its keys, keeping
// dK and dV of its 64 keys in registers (so the group sum is free), and adds
// dQ into an fp32 buffer with vector atomics.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>
#include <cstdio>

#include "sf_internal.h"

namespace sf {

typedef __nv_bfloat16 bf16;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sz)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// rows x HD bf16 tile from global (row stride ld) into shared [rows][HD + 8];
// rows at or past `valid` are zero-filled.
template <int HD>
__device__ __forceinline__ void load_tile(bf16* sdst, const bf16* g, int64_t ld, int rows, int valid) {
  constexpr int CPR = HD / 8;
  const uint32_t base = su32(sdst);
  for (int c = threadIdx.x; c < rows * CPR; c += blockDim.x) {
    const int r = c / CPR, k = c % CPR;
    const bool v = r < valid;
    const bf16* src = g + (v ? (int64_t)r * ld : 0) + k * 8;
    cp_async16(base + (uint32_t)((r * (HD + 8) + k * 8) * 2), src, v);
  }
}

// A fragment (16 x 16) of a row-major shared tile at (r0, c0), ld in elements.
__device__ __forceinline__ void lds_a(const bf16* s, int ld, int r0, int c0, uint32_t (&a)[4]) {
  const int i = threadIdx.x & 31;
  const int r = r0 + (i & 7) + ((i >> 3) & 1) * 8, c = c0 + (i >> 4) * 8;
  ldsm_x4(su32(s + r * ld + c), a[0], a[1], a[2], a[3]);
}
// B fragments of two n8 tiles from a shared tile stored [n][k] (k contiguous).
__device__ __forceinline__ void lds_b_nk(const bf16* s, int ld, int n0, int k0, uint32_t& b0,
                                         uint32_t& b1, uint32_t& b2, uint32_t& b3) {
  const int i = threadIdx.x & 31;
  const int r = n0 + (i & 7) + (i >> 4) * 8, c = k0 + ((i >> 3) & 1) * 8;
  ldsm_x4(su32(s + r * ld + c), b0, b1, b2, b3);
}
// B fragments of two n8 tiles from a shared tile stored [k][n] (n contiguous).
__device__ __forceinline__ void lds_b_kn(const bf16* s, int ld, int k0, int n0, uint32_t& b0,
                                         uint32_t& b1, uint32_t& b2, uint32_t& b3) {
  const int i = threadIdx.x & 31;
  const int r = k0 + (i & 7) + ((i >> 3) & 1) * 8, c = n0 + (i >> 4) * 8;
  ldsm_x4_t(su32(s + r * ld + c), b0, b1, b2, b3);
}
// A fragment (16 x 16) at (m0, k0) of A = X^T where X is stored [k][m].
__device__ __forceinline__ void lds_a_t(const bf16* s, int ld, int m0, int k0, uint32_t (&a)[4]) {
  const int i = threadIdx.x & 31;
  const int r = k0 + (i & 7) + (i >> 4) * 8, c = m0 + ((i >> 3) & 1) * 8;
  ldsm_x4_t(su32(s + r * ld + c), a[0], a[1], a[2], a[3]);
}

// ------------------------------------------------------------------ backward
// delta[b, h, s] = sum_j dO[t, h*hd + j] * O[t, h*hd + j]   (one warp per row)
__global__ void attn_delta_kernel(const bf16* __restrict__ o, const bf16* __restrict__ dout,
                                  float* __restrict__ delta, int64_t rows, int S, int Hq, int hd) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= rows) return;
  const int64_t t = w / Hq;
  const int h = (int)(w % Hq);
  const bf16* orow = o + t * (int64_t)Hq * hd + (int64_t)h * hd;
  const bf16* drow = dout + t * (int64_t)Hq * hd + (int64_t)h * hd;
  float acc = 0.f;
  for (int j = lane * 2; j < hd; j += 64) {
    float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(orow + j));
    float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(drow + j));
    acc += a.x * c.x + a.y * c.y;
  }
#pragma unroll
  for (int k = 16; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
  if (lane == 0) {
    const int64_t b = t / S, s = t % S;
    delta[(b * Hq + h) * S + s] = acc;
  }
}

// dQ = scale * dq_acc, inverse RoPE, into the query columns of dqkv (8 pairs per thread)
__global__ void attn_dq_kernel(const float* __restrict__ dq_acc, bf16* __restrict__ dqkv,
                               int64_t tokens, int S, int Hq, int Hkv, int hd, float scale,
                               const float2* __restrict__ cs) {
  const int half = hd / 2, groups = half / 8;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= tokens * Hq * groups) return;
  const int gr = (int)(idx % groups);
  const int64_t th = idx / groups;
  const int h = (int)(th % Hq);
  const int64_t t = th / Hq;
  const int s = (int)(t % S);
  const float* src = dq_acc + t * (int64_t)Hq * hd + (int64_t)h * hd + gr * 8;
  bf16* dst = dqkv + t * (int64_t)(Hq + 2 * Hkv) * hd + (int64_t)h * hd + gr * 8;
  float x1[8], x2[8];
#pragma unroll
  for (int i = 0; i < 8; i += 4) {
    float4 a = *reinterpret_cast<const float4*>(src + i);
    float4 c = *reinterpret_cast<const float4*>(src + half + i);
    x1[i] = a.x; x1[i + 1] = a.y; x1[i + 2] = a.z; x1[i + 3] = a.w;
    x2[i] = c.x; x2[i + 1] = c.y; x2[i + 2] = c.z; x2[i + 3] = c.w;
  }
  uint32_t o1[4], o2[4];
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    float a1 = x1[i] * scale, b1 = x1[i + 1] * scale, a2 = x2[i] * scale, b2 = x2[i + 1] * scale;
    if (cs) {
      const float2 ca = cs[(int64_t)s * half + gr * 8 + i], cb = cs[(int64_t)s * half + gr * 8 + i + 1];
      const float y1a = a1 * ca.x + a2 * ca.y, y2a = a2 * ca.x - a1 * ca.y;
      const float y1b = b1 * cb.x + b2 * cb.y, y2b = b2 * cb.x - b1 * cb.y;
      a1 = y1a; a2 = y2a; b1 = y1b; b2 = y2b;
    }
    o1[i / 2] = pack2(a1, b1);
    o2[i / 2] = pack2(a2, b2);
  }
  *reinterpret_cast<uint4*>(dst) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
  *reinterpret_cast<uint4*>(dst + half) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
}

void attn_delta(const bf16* o, const bf16* dout, float* delta, int B, int S, int Hq, int hd,
                cudaStream_t st) {
  const int64_t rows = (int64_t)B * S * Hq;
  attn_delta_kernel<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(o, dout, delta, rows, S, Hq, hd);
}

void attn_dq_finalize(const float* dq_acc, bf16* dqkv, int B, int S, int Hq, int Hkv, int hd,
                      float scale, const float2* cs, cudaStream_t st) {
  const int64_t T = (int64_t)B * S;
  const int64_t n = T * Hq * (hd / 16);
  attn_dq_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(dq_acc, dqkv, T, S, Hq, Hkv, hd, scale, cs);
}

}  // namespace sf
