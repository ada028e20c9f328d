// Causal grouped-query attention: the small memory-bound kernels around the
// tcgen05 forward and backward (attention_tc.cu).
//
// Inputs come straight from the QKV projection's output row [T, (Hq+2Hkv)*hd]
// (token t = b*S + s): query head h at column h*hd, kv head g at (Hq+g)*hd
// (K) and (Hq+Hkv+g)*hd (V); query head h reads kv head h / (Hq/Hkv).
//
// attn_delta: D = rowsum(dO * O) per (token, head), the softmax-gradient term.
// attn_dq_finalize: dQ from the fp32 accumulation of the backward kernel
// (one buffer, or one slot per 128-key block summed in key order when the
// backward runs deterministically), scaled, inverse-rotated (RoPE) and
// written as bf16 into the query columns of dqkv.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sf_internal.h"

namespace sf {

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------ backward
// delta[b, h, s] = sum_j dO[t, h*hd + j] * O[t, h*hd + j]: TPR = hd / 8
// threads per (token, head) row, each reading 16 bytes of O and of dO, summed
// across the row's threads with shuffles.  Consecutive rows are consecutive
// heads of a token, so a warp reads contiguous memory.
template <int TPR>
__global__ void attn_delta_kernel(const bf16* __restrict__ o, const bf16* __restrict__ dout,
                                  float* __restrict__ delta, int64_t rows, int S, int Hq) {
  constexpr int HD = TPR * 8;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t w = g / TPR;
  const int sub = (int)(g % TPR);
  float acc = 0.f;
  if (w < rows) {  // no early return: every lane takes part in the shuffles
    const int64_t off = w * HD + sub * 8;  // row w = t * Hq + h starts at t*Hq*hd + h*hd
    const uint4 a = *reinterpret_cast<const uint4*>(o + off);
    const uint4 c = *reinterpret_cast<const uint4*>(dout + off);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(a2[i]), y = __bfloat1622float2(c2[i]);
      acc += x.x * y.x + x.y * y.y;
    }
  }
#pragma unroll
  for (int k = TPR / 2; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
  if (sub == 0 && w < rows) {
    const int64_t t = w / Hq;
    const int h = (int)(w % Hq);
    const int64_t b = t / S, s = t % S;
    delta[(b * Hq + h) * S + s] = acc;
  }
}

// dQ = scale * (sum of the fp32 partials), inverse RoPE, into the query
// columns of dqkv (8 pairs per thread).  slots == 0: one accumulated buffer
// [T, Hq*hd]; else slot j [T, Hq*hd] holds key block j's part, written for
// positions s >= 128 j, and the parts are added in the order j = 0, 1, ...
__global__ void attn_dq_kernel(const float* __restrict__ dq_acc, bf16* __restrict__ dqkv,
                               int64_t tokens, int S, int Hq, int Hkv, int hd, float scale,
                               const float2* __restrict__ cs, int slots) {
  const int half = hd / 2, groups = half / 8;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= tokens * Hq * groups) return;
  const int gr = (int)(idx % groups);
  const int64_t th = idx / groups;
  const int h = (int)(th % Hq);
  const int64_t t = th / Hq;
  const int s = (int)(t % S);
  const int64_t ld = (int64_t)Hq * hd;
  const float* src = dq_acc + t * ld + (int64_t)h * hd + gr * 8;
  bf16* dst = dqkv + t * (int64_t)(Hq + 2 * Hkv) * hd + (int64_t)h * hd + gr * 8;
  float x1[8], x2[8];
#pragma unroll
  for (int i = 0; i < 8; i += 4) {
    float4 a = *reinterpret_cast<const float4*>(src + i);
    float4 c = *reinterpret_cast<const float4*>(src + half + i);
    x1[i] = a.x; x1[i + 1] = a.y; x1[i + 2] = a.z; x1[i + 3] = a.w;
    x2[i] = c.x; x2[i + 1] = c.y; x2[i + 2] = c.z; x2[i + 3] = c.w;
  }
  const int last = slots > 0 ? s / 128 : 0;
  for (int j = 1; j <= last; ++j) {
    const float* p = src + (int64_t)j * tokens * ld;
#pragma unroll
    for (int i = 0; i < 8; i += 4) {
      float4 a = *reinterpret_cast<const float4*>(p + i);
      float4 c = *reinterpret_cast<const float4*>(p + half + i);
      x1[i] += a.x; x1[i + 1] += a.y; x1[i + 2] += a.z; x1[i + 3] += a.w;
      x2[i] += c.x; x2[i + 1] += c.y; x2[i + 2] += c.z; x2[i + 3] += c.w;
    }
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
  const int64_t threads = rows * (hd / 8);
  const unsigned grid = (unsigned)((threads + 255) / 256);
  if (hd == 128)
    attn_delta_kernel<16><<<grid, 256, 0, st>>>(o, dout, delta, rows, S, Hq);
  else
    attn_delta_kernel<8><<<grid, 256, 0, st>>>(o, dout, delta, rows, S, Hq);
}

void attn_dq_finalize(const float* dq_acc, bf16* dqkv, int B, int S, int Hq, int Hkv, int hd,
                      float scale, const float2* cs, int slots, cudaStream_t st) {
  const int64_t T = (int64_t)B * S;
  const int64_t n = T * Hq * (hd / 16);
  attn_dq_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(dq_acc, dqkv, T, S, Hq, Hkv, hd, scale,
                                                               cs, slots);
}

}  // namespace sf
