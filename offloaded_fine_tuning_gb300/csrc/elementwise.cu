// Memory-bound kernels of the decoder step: RMSNorm forward/backward, RoPE,
// SwiGLU forward/backward, the row softmax of the fused LM-head cross-entropy,
// reductions and casts.  All of them stream rows with 16-byte vector accesses
// and reduce with warp shuffles; none of them is a contraction.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"
#include "sf.h"
#include "sf_internal.h"

namespace sf {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Block-wide sum; every thread gets the result.  `sh` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* sh) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  float t = (lane < nw) ? sh[lane] : 0.f;
  return warp_sum(t);
}

__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

constexpr int kNormThreads = 256;

// ------------------------------------------------------------------ RMSNorm forward
// One CTA per row: y = bf16(g * x * rstd), rstd = 1/sqrt(mean(x^2) + eps).
// Thread t holds the float4 columns t, t+256, ... (CH of them) in registers
// between the sum of squares and the scaling, so x is read once.
template <int CH>
__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_fwd_kernel(const float* __restrict__ x, const __nv_bfloat16* __restrict__ g,
                       __nv_bfloat16* __restrict__ y, float* __restrict__ rstd_out, int d,
                       float eps) {
  __shared__ float sh[32];
  const int64_t row = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + row * d);
  const int n4 = d >> 2;
  float4 v[CH];
  float ss = 0.f;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int i = threadIdx.x + c * kNormThreads;
    v[c] = i < n4 ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += v[c].x * v[c].x + v[c].y * v[c].y + v[c].z * v[c].z + v[c].w * v[c].w;
  }
  ss = block_sum(ss, sh);
  const float rstd = rsqrtf(ss / d + eps);
  if (threadIdx.x == 0) rstd_out[row] = rstd;
  const uint2* gr = reinterpret_cast<const uint2*>(g);
  uint2* yr = reinterpret_cast<uint2*>(y + row * d);
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int i = threadIdx.x + c * kNormThreads;
    if (i < n4) {
      uint2 gu = gr[i];
      float2 g01 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&gu.x));
      float2 g23 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&gu.y));
      __nv_bfloat162 o01 = __floats2bfloat162_rn(v[c].x * rstd * g01.x, v[c].y * rstd * g01.y);
      __nv_bfloat162 o23 = __floats2bfloat162_rn(v[c].z * rstd * g23.x, v[c].w * rstd * g23.y);
      uint2 o;
      o.x = *reinterpret_cast<uint32_t*>(&o01);
      o.y = *reinterpret_cast<uint32_t*>(&o23);
      yr[i] = o;
    }
  }
}

template <int CH>
static void rmsnorm_fwd_ch(const float* x, const __nv_bfloat16* g, __nv_bfloat16* y, float* rstd,
                           int64_t rows, int d, float eps, cudaStream_t st) {
  rmsnorm_fwd_kernel<CH><<<(unsigned)rows, kNormThreads, 0, st>>>(x, g, y, rstd, d, eps);
}

void rmsnorm_fwd(const float* x, const __nv_bfloat16* g, __nv_bfloat16* y, float* rstd,
                 int64_t rows, int d, float eps, cudaStream_t st) {
  if (rows <= 0) return;
  const int ch = (d / 4 + kNormThreads - 1) / kNormThreads;  // d <= 16384: at most 16
  if (ch <= 1) rmsnorm_fwd_ch<1>(x, g, y, rstd, rows, d, eps, st);
  else if (ch <= 2) rmsnorm_fwd_ch<2>(x, g, y, rstd, rows, d, eps, st);
  else if (ch <= 4) rmsnorm_fwd_ch<4>(x, g, y, rstd, rows, d, eps, st);
  else if (ch <= 8) rmsnorm_fwd_ch<8>(x, g, y, rstd, rows, d, eps, st);
  else if (ch <= 12) rmsnorm_fwd_ch<12>(x, g, y, rstd, rows, d, eps, st);
  else rmsnorm_fwd_ch<16>(x, g, y, rstd, rows, d, eps, st);
}

// ------------------------------------------------------------------ RMSNorm backward
// CTAs stride over rows; thread t owns the float4 columns t, t+256, ... (CH of
// them) so the gain gradient sum over the CTA's rows stays in registers.  For
// d above 4096 the second pass over a row re-reads x and dy, which are still
// in L1/L2.

template <int CH>
__global__ void __launch_bounds__(kNormThreads, CH <= 4 ? 4 : (CH <= 8 ? 2 : 1))
    rmsnorm_bwd_kernel(const float* __restrict__ x, const __nv_bfloat16* __restrict__ g,
                       const float* __restrict__ rstd, const float* __restrict__ dy,
                       const float* __restrict__ dres, float* __restrict__ dx,
                       __nv_bfloat16* __restrict__ dxb, float* __restrict__ dg_part,
                       int64_t rows, int d) {
  __shared__ float sh[32];
  const int n4 = d >> 2;
  float4 gacc[CH], gg[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    gacc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    gg[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int i = threadIdx.x + c * kNormThreads;
    if (i < n4) {
      uint2 gu = reinterpret_cast<const uint2*>(g)[i];
      float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&gu.x));
      float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&gu.y));
      gg[c] = make_float4(a.x, a.y, b.x, b.y);
    }
  }
  const float inv_d = 1.f / d;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float r = rstd[row];
    const float4* xr = reinterpret_cast<const float4*>(x + row * d);
    const float4* dyr = reinterpret_cast<const float4*>(dy + row * d);
    float dot = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int i = threadIdx.x + c * kNormThreads;
      if (i < n4) {
        const float4 xv = xr[i], dv = dyr[i];
        const float4 xh = make_float4(xv.x * r, xv.y * r, xv.z * r, xv.w * r);
        dot += gg[c].x * dv.x * xh.x + gg[c].y * dv.y * xh.y + gg[c].z * dv.z * xh.z +
               gg[c].w * dv.w * xh.w;
        gacc[c].x += dv.x * xh.x; gacc[c].y += dv.y * xh.y;
        gacc[c].z += dv.z * xh.z; gacc[c].w += dv.w * xh.w;
      }
    }
    dot = block_sum(dot, sh) * inv_d;
    float4* dxr = reinterpret_cast<float4*>(dx + row * d);
    const float4* drr = dres ? reinterpret_cast<const float4*>(dres + row * d) : nullptr;
    uint2* dbr = reinterpret_cast<uint2*>(dxb + row * d);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int i = threadIdx.x + c * kNormThreads;
      if (i < n4) {
        const float4 xv = xr[i], dv = dyr[i];
        float4 o;
        o.x = r * (gg[c].x * dv.x - xv.x * r * dot);
        o.y = r * (gg[c].y * dv.y - xv.y * r * dot);
        o.z = r * (gg[c].z * dv.z - xv.z * r * dot);
        o.w = r * (gg[c].w * dv.w - xv.w * r * dot);
        if (drr) {
          const float4 q = drr[i];
          o.x += q.x; o.y += q.y; o.z += q.z; o.w += q.w;
        }
        dxr[i] = o;
        __nv_bfloat162 a = __floats2bfloat162_rn(o.x, o.y), b = __floats2bfloat162_rn(o.z, o.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&a);
        u.y = *reinterpret_cast<uint32_t*>(&b);
        dbr[i] = u;
      }
    }
  }
  float4* part = reinterpret_cast<float4*>(dg_part + (int64_t)blockIdx.x * d);
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int i = threadIdx.x + c * kNormThreads;
    if (i < n4) part[i] = gacc[c];
  }
}

// Up to d = 4096: 512-thread CTAs, two per SM, that load a row's x, dy and
// residual gradient into registers before the row's reduction (every load of
// the row in flight at once, and no second pass over x and dy).
constexpr int kNormBwdThreads = 512;

template <int CH>
__global__ void __launch_bounds__(kNormBwdThreads, 2)
    rmsnorm_bwd_hold_kernel(const float* __restrict__ x, const __nv_bfloat16* __restrict__ g,
                            const float* __restrict__ rstd, const float* __restrict__ dy,
                            const float* __restrict__ dres, float* __restrict__ dx,
                            __nv_bfloat16* __restrict__ dxb, float* __restrict__ dg_part,
                            int64_t rows, int d) {
  __shared__ float sh[32];
  const int n4 = d >> 2;
  float4 gacc[CH], gg[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    gacc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    gg[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int i = threadIdx.x + c * kNormBwdThreads;
    if (i < n4) {
      uint2 gu = reinterpret_cast<const uint2*>(g)[i];
      float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&gu.x));
      float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&gu.y));
      gg[c] = make_float4(a.x, a.y, b.x, b.y);
    }
  }
  const float inv_d = 1.f / d;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float r = rstd[row];
    const float4* xr = reinterpret_cast<const float4*>(x + row * d);
    const float4* dyr = reinterpret_cast<const float4*>(dy + row * d);
    const float4* drr = dres ? reinterpret_cast<const float4*>(dres + row * d) : nullptr;
    float4 xv[CH], dv[CH], qv[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int i = threadIdx.x + c * kNormBwdThreads;
      const bool in = i < n4;
      xv[c] = in ? xr[i] : zero;
      dv[c] = in ? dyr[i] : zero;
      qv[c] = (in && drr) ? drr[i] : zero;
    }
    float dot = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const float4 xh = make_float4(xv[c].x * r, xv[c].y * r, xv[c].z * r, xv[c].w * r);
      dot += gg[c].x * dv[c].x * xh.x + gg[c].y * dv[c].y * xh.y + gg[c].z * dv[c].z * xh.z +
             gg[c].w * dv[c].w * xh.w;
      gacc[c].x += dv[c].x * xh.x; gacc[c].y += dv[c].y * xh.y;
      gacc[c].z += dv[c].z * xh.z; gacc[c].w += dv[c].w * xh.w;
    }
    dot = block_sum(dot, sh) * inv_d;
    float4* dxr = reinterpret_cast<float4*>(dx + row * d);
    uint2* dbr = reinterpret_cast<uint2*>(dxb + row * d);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int i = threadIdx.x + c * kNormBwdThreads;
      if (i < n4) {
        float4 o;
        o.x = r * (gg[c].x * dv[c].x - xv[c].x * r * dot) + qv[c].x;
        o.y = r * (gg[c].y * dv[c].y - xv[c].y * r * dot) + qv[c].y;
        o.z = r * (gg[c].z * dv[c].z - xv[c].z * r * dot) + qv[c].z;
        o.w = r * (gg[c].w * dv[c].w - xv[c].w * r * dot) + qv[c].w;
        dxr[i] = o;
        __nv_bfloat162 a = __floats2bfloat162_rn(o.x, o.y), b = __floats2bfloat162_rn(o.z, o.w);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&a);
        u.y = *reinterpret_cast<uint32_t*>(&b);
        dbr[i] = u;
      }
    }
  }
  float4* part = reinterpret_cast<float4*>(dg_part + (int64_t)blockIdx.x * d);
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int i = threadIdx.x + c * kNormBwdThreads;
    if (i < n4) part[i] = gacc[c];
  }
}

// Row partition of the RMSNorm backward (and of the bias column sums): two
// CTAs per SM (two 512-thread CTAs up to d = 4096, two 256-thread CTAs up to
// d = 8192, one beyond), each summing the gain gradient of its rows.
int rmsnorm_bwd_parts(int64_t rows, int d) {
  (void)d;
  const int p = 2 * num_sms();
  return rows < p ? (int)(rows > 0 ? rows : 1) : p;
}

void rmsnorm_bwd(const float* x, const __nv_bfloat16* g, const float* rstd, const float* dy,
                 const float* dres, float* dx, __nv_bfloat16* dxb, float* dg_part, int parts,
                 int64_t rows, int d, cudaStream_t st) {
  if (d <= 2 * 4 * kNormBwdThreads) {
    if (d <= 4 * kNormBwdThreads)
      rmsnorm_bwd_hold_kernel<1><<<parts, kNormBwdThreads, 0, st>>>(x, g, rstd, dy, dres, dx, dxb,
                                                                     dg_part, rows, d);
    else
      rmsnorm_bwd_hold_kernel<2><<<parts, kNormBwdThreads, 0, st>>>(x, g, rstd, dy, dres, dx, dxb,
                                                                     dg_part, rows, d);
    return;
  }
  const int need = (d / 4 + kNormThreads - 1) / kNormThreads;  // float4 chunks per thread
#define SF_NORM_BWD(CH) \
  rmsnorm_bwd_kernel<CH><<<parts, kNormThreads, 0, st>>>(x, g, rstd, dy, dres, dx, dxb, dg_part, rows, d)
  if (need <= 8) SF_NORM_BWD(8);
  else if (need <= 12) SF_NORM_BWD(12);
  else SF_NORM_BWD(16);
#undef SF_NORM_BWD
}

// out[j] = sum_p part[p, j] over the partials [parts, d], in a fixed order
// (deterministic).  A CTA takes 32 columns with 8 warps: warp w sums the
// partials w, w + 8, w + 16, ... of its lane's column (each warp reads 128
// contiguous bytes per partial), then the eight sums are added in warp order.
constexpr int kRedWarps = 8;

template <typename OUT>
__global__ void __launch_bounds__(32 * kRedWarps)
    reduce_parts_kernel(const float* __restrict__ part, int parts, int d, OUT* __restrict__ out,
                        float scale) {
  __shared__ float sh[kRedWarps][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int j = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (j < d) {
    int p = w;
#pragma unroll 4
    for (; p < parts; p += kRedWarps) s += part[(int64_t)p * d + j];
  }
  sh[w][lane] = s;
  __syncthreads();
  if (w == 0 && j < d) {
    float t = sh[0][lane];
#pragma unroll
    for (int k = 1; k < kRedWarps; ++k) t += sh[k][lane];
    if constexpr (sizeof(OUT) == 2 && std::is_same<OUT, __half>::value)
      out[j] = __float2half_rn(t * scale);
    else
      out[j] = __float2bfloat16_rn(t);
  }
}

void reduce_parts_bf16(const float* part, int parts, int d, __nv_bfloat16* out, cudaStream_t st) {
  reduce_parts_kernel<__nv_bfloat16><<<(d + 31) / 32, 32 * kRedWarps, 0, st>>>(part, parts, d, out, 1.f);
}

void reduce_parts_f16(const float* part, int parts, int d, uint16_t* out, float scale,
                      cudaStream_t st) {
  reduce_parts_kernel<__half><<<(d + 31) / 32, 32 * kRedWarps, 0, st>>>(
      part, parts, d, reinterpret_cast<__half*>(out), scale);
}

// Column sums of x [rows, cols] bf16 (row stride ld) as fp32 partials:
// part[p][c] sums the rows [rows*p/parts, rows*(p+1)/parts).  Two columns per
// thread, so a warp reads 128 contiguous bytes of a row.
__global__ void colsum_parts_kernel(const __nv_bfloat16* __restrict__ x, int64_t ld, int64_t rows,
                                    int cols, float* __restrict__ part, int parts) {
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 2;
  const int p = blockIdx.y;
  if (c >= cols) return;
  const int64_t r0 = rows * p / parts, r1 = rows * (p + 1) / parts;
  float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
  for (int64_t r = r0; r < r1; ++r) {
    const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + r * ld + c));
    s0 += v.x;
    s1 += v.y;
  }
  part[(int64_t)p * cols + c] = s0;
  part[(int64_t)p * cols + c + 1] = s1;
}

void bias_grad(const __nv_bfloat16* x, int64_t ld, int64_t rows, int cols, float* part, int parts,
               __nv_bfloat16* out, cudaStream_t st) {
  dim3 grid((unsigned)((cols / 2 + 127) / 128), (unsigned)parts);
  colsum_parts_kernel<<<grid, 128, 0, st>>>(x, ld, rows, cols, part, parts);
  reduce_parts_bf16(part, parts, cols, out, st);
}

void bias_grad_f16(const __nv_bfloat16* x, int64_t ld, int64_t rows, int cols, float* part,
                   int parts, uint16_t* out, float scale, cudaStream_t st) {
  dim3 grid((unsigned)((cols / 2 + 127) / 128), (unsigned)parts);
  colsum_parts_kernel<<<grid, 128, 0, st>>>(x, ld, rows, cols, part, parts);
  reduce_parts_f16(part, parts, cols, out, scale, st);
}

// ------------------------------------------------------------------ RoPE
// In place on the first `heads` heads of each token row of qkv.  cs[s*hd/2 + j]
// = (cos, sin) of s * base^(-2j/hd).  inverse = 1 rotates by the opposite angle
// (the transpose, used on gradients).  One thread per (token, head, 8 pairs).
__global__ void rope_kernel(__nv_bfloat16* __restrict__ qkv, int64_t ld, int64_t tokens, int seq,
                            int heads, int hd, const float2* __restrict__ cs, int inverse) {
  const int half = hd >> 1;
  const int groups = half >> 3;  // 8 pairs per thread
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = tokens * heads * groups;
  if (idx >= total) return;
  const int grp = (int)(idx % groups);
  const int64_t th = idx / groups;
  const int h = (int)(th % heads);
  const int64_t t = th / heads;
  const int s = (int)(t % seq);
  __nv_bfloat16* base = qkv + t * ld + (int64_t)h * hd + grp * 8;
  float x1[8], x2[8];
  unpack8(*reinterpret_cast<const uint4*>(base), x1);
  unpack8(*reinterpret_cast<const uint4*>(base + half), x2);
  const float2* c = cs + (int64_t)s * half + grp * 8;
  float y1[8], y2[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float co = c[i].x, si = inverse ? -c[i].y : c[i].y;
    y1[i] = x1[i] * co - x2[i] * si;
    y2[i] = x2[i] * co + x1[i] * si;
  }
  *reinterpret_cast<uint4*>(base) = pack8(y1);
  *reinterpret_cast<uint4*>(base + half) = pack8(y2);
}

void rope_inplace(__nv_bfloat16* qkv, int64_t ld, int64_t tokens, int seq, int heads,
                  int head_dim, const float2* cs, int inverse, cudaStream_t st) {
  const int64_t total = tokens * heads * (head_dim / 16);
  if (total <= 0) return;
  rope_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(qkv, ld, tokens, seq, heads,
                                                                head_dim, cs, inverse);
}

// ------------------------------------------------------------------ SwiGLU
// ab row = [a (ffn) | b (ffn)];  m = silu(a) * b.
__global__ void swiglu_fwd_kernel(const __nv_bfloat16* __restrict__ ab, __nv_bfloat16* __restrict__ m,
                                  int64_t rows, int ffn) {
  const int per_row = ffn >> 3;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * per_row) return;
  const int64_t r = idx / per_row;
  const int c = (int)(idx % per_row) * 8;
  float a[8], b[8], o[8];
  unpack8(*reinterpret_cast<const uint4*>(ab + r * 2 * ffn + c), a);
  unpack8(*reinterpret_cast<const uint4*>(ab + r * 2 * ffn + ffn + c), b);
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = a[i] / (1.f + __expf(-a[i])) * b[i];
  *reinterpret_cast<uint4*>(m + r * ffn + c) = pack8(o);
}

void swiglu_fwd(const __nv_bfloat16* ab, __nv_bfloat16* m, int64_t rows, int ffn, cudaStream_t st) {
  const int64_t total = rows * (ffn / 8);
  if (total <= 0) return;
  swiglu_fwd_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(ab, m, rows, ffn);
}

// da = dm * b * s * (1 + a (1 - s)),  db = dm * a * s,  s = sigmoid(a)
__global__ void swiglu_bwd_kernel(const __nv_bfloat16* __restrict__ dm,
                                  const __nv_bfloat16* __restrict__ ab,
                                  __nv_bfloat16* __restrict__ dab, int64_t rows, int ffn) {
  const int per_row = ffn >> 3;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * per_row) return;
  const int64_t r = idx / per_row;
  const int c = (int)(idx % per_row) * 8;
  float a[8], b[8], g[8], da[8], db[8];
  unpack8(*reinterpret_cast<const uint4*>(ab + r * 2 * ffn + c), a);
  unpack8(*reinterpret_cast<const uint4*>(ab + r * 2 * ffn + ffn + c), b);
  unpack8(*reinterpret_cast<const uint4*>(dm + r * ffn + c), g);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float s = 1.f / (1.f + __expf(-a[i]));
    da[i] = g[i] * b[i] * s * (1.f + a[i] * (1.f - s));
    db[i] = g[i] * a[i] * s;
  }
  *reinterpret_cast<uint4*>(dab + r * 2 * ffn + c) = pack8(da);
  *reinterpret_cast<uint4*>(dab + r * 2 * ffn + ffn + c) = pack8(db);
}

void swiglu_bwd(const __nv_bfloat16* dm, const __nv_bfloat16* ab, __nv_bfloat16* dab, int64_t rows,
                int ffn, cudaStream_t st) {
  const int64_t total = rows * (ffn / 8);
  if (total <= 0) return;
  swiglu_bwd_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(dm, ab, dab, rows, ffn);
}

// ------------------------------------------------------------------ cross-entropy rows
// Per row of fp32 logits z: lse = log sum_v exp(z_v), loss = lse - z_label and
// dz = (exp(z - lse) - [v == label]) * inv_n as bf16 into its own buffer (the
// operand of the dH and dW products); rows whose label is negative (the
// ignore index -100 among them) get dz = 0 and loss 0, and so does a row
// whose label is at or beyond the vocabulary, which is also reported as
// kDevCeBadLabel (the kernel API takes labels in device memory, where the
// host cannot check them).
//
// Cluster form (rows of up to kCeMaxCluster slices of kCeSliceMax bytes):
// the CTAs of one cluster share a row, each holding a contiguous slice of it
// in shared memory, copied in by the bulk-copy unit in kCePieces pieces so
// that the max pass starts on the first piece while the rest lands.  Each
// CTA takes its slice's max m_r, overwrites its slice with exp(z - m_r)
// while summing it (s_r), and publishes (m_r, s_r); every CTA combines the
// cluster's pairs into lse through distributed shared memory and writes dz
// from its slice as exp(z - m_r) * exp(m_r - lse).  The row is read from HBM
// once (fp32) and dz written once (bf16): 6 bytes per logit.  (One online
// max / sum-exp pass with dz = exp(z - lse) recomputed measured 7% slower:
// two exponentials per logit instead of one.)
//
// One cluster per row, several CTAs per SM (slices up to kCeSliceShare bytes
// let three share an SM), so that one CTA's reductions, cluster barrier and
// stores overlap the others' copies.  Measured on 2,048 rows of 152,064
// logits: 256 threads a CTA beat 512 by 7% and 128 by 10%; clusters of 16
// (38 KB slices, five CTAs per SM) were 15% slower; a persistent form, one
// CTA per SM with two slice buffers and the next row's copy in flight, was
// 1.6x slower (each row's reductions and barriers then sit on the SM's
// critical path).  The published pair is ordered by its one writer's fence;
// every thread's cluster arrival is relaxed.

// (m, s) <- the pair of the union of two sets given as (max, sum of exp(x - max)).
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  s = s * __expf(m - M) + s2 * __expf(m2 - M);
  m = M;
}
// The pair of the whole warp, in every lane (lane 0's order of combination).
__device__ __forceinline__ void warp_lse_merge(float& m, float& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
  m = __shfl_sync(0xffffffffu, m, 0);
  s = __shfl_sync(0xffffffffu, s, 0);
}

constexpr int kCeThreads = 256;
constexpr int kCePieces = 4;
constexpr int kCeSliceMax = 200 * 1024;    // largest slice a CTA holds
constexpr int kCeSliceShare = 76 * 1024;   // three CTAs per SM up to this slice
constexpr int kCeMaxCluster = 8;

__global__ void __launch_bounds__(kCeThreads)
    ce_rows_cluster_kernel(const float* __restrict__ z, __nv_bfloat16* __restrict__ dz,
                           const int32_t* __restrict__ labels, int64_t vocab, float inv_n,
                           float* __restrict__ loss_rows, int* err) {
  extern __shared__ __align__(128) float4 slice[];
  __shared__ __align__(8) uint64_t bars[kCePieces];
  __shared__ __align__(8) float2 pub;  // (m_r, s_r), read by the cluster
  __shared__ float2 red[32];
  uint32_t ncl;
  asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(ncl));
  const uint32_t rank = cluster_ctarank();
  const int64_t row = blockIdx.x / ncl;
  const int64_t n4 = vocab >> 2;  // vocab % 8 == 0 (checked by the caller)
  const int64_t q = (n4 + ncl - 1) / ncl;
  const int64_t lo = rank * q < n4 ? rank * q : n4;
  const int len = (int)((lo + q < n4 ? lo + q : n4) - lo);  // float4 of this slice
  const int pq = (len + kCePieces - 1) / kCePieces;         // float4 per piece
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint2* dr = reinterpret_cast<uint2*>(dz + row * vocab) + lo;
  int label = labels[row];
  if (label >= vocab) {  // outside the vocabulary: reported, and the row ignored
    if (rank == 0 && threadIdx.x == 0) record_error(err, kDevCeBadLabel);
    label = -1;
  }
  if (label < 0) {  // uniform over the cluster: no cluster barrier is reached
    const uint2 zero = make_uint2(0, 0);
    for (int i = threadIdx.x; i < len; i += blockDim.x) dr[i] = zero;
    if (rank == 0 && threadIdx.x == 0) loss_rows[row] = 0.f;
    return;
  }
  if (threadIdx.x == 0) {
    const float4* src = reinterpret_cast<const float4*>(z + row * vocab) + lo;
    for (int k = 0; k < kCePieces; ++k) mbar_init(smem_u32(&bars[k]), 1);
    fence_mbar_init();
    for (int k = 0; k < kCePieces; ++k) {
      const int a = k * pq < len ? k * pq : len, b = a + pq < len ? a + pq : len;
      const uint32_t bytes = (uint32_t)(b - a) * 16u;
      mbar_arrive_expect_tx(smem_u32(&bars[k]), bytes);
      if (bytes > 0) bulk_load(smem_u32(slice + a), src + a, bytes, smem_u32(&bars[k]));
    }
  }
  __syncthreads();
  // the slice's max, piece by piece as the copies land
  bool ok = true;
  float m = -FLT_MAX;
  for (int k = 0; k < kCePieces; ++k) {
    if (ok && !mbar_wait(smem_u32(&bars[k]), 0, nullptr)) {
      record_error(err, kDevCeTimeout);
      ok = false;
    }
    const int a = k * pq < len ? k * pq : len, b = a + pq < len ? a + pq : len;
    if (ok)
      for (int i = a + threadIdx.x; i < b; i += blockDim.x) {
        const float4 f = slice[i];
        m = fmaxf(m, fmaxf(fmaxf(f.x, f.y), fmaxf(f.z, f.w)));
      }
  }
  m = warp_max(m);
  if (lane == 0) red[w].x = m;
  __syncthreads();
  float mr = -FLT_MAX;
  for (int i = 0; i < nw; ++i) mr = fmaxf(mr, red[i].x);
  // exp(z - m_r) over the slice, in place, and its sum
  float s = 0.f;
  if (ok)
    for (int i = threadIdx.x; i < len; i += blockDim.x) {
      float4 f = slice[i];
      f.x = __expf(f.x - mr); f.y = __expf(f.y - mr);
      f.z = __expf(f.z - mr); f.w = __expf(f.w - mr);
      slice[i] = f;
      s += (f.x + f.y) + (f.z + f.w);
    }
  s = warp_sum(s);
  if (lane == 0) red[w].y = s;
  __syncthreads();
  if (w == 0) {  // the CTA's pair, published for the cluster
    const float t = warp_sum(lane < nw ? red[lane].y : 0.f);
    if (lane == 0) {
      pub = make_float2(mr, t);
      fence_acq_rel_cluster();  // the pair before this thread's arrival
    }
  }
  cluster_arrive_relaxed();
  cluster_wait();  // every CTA's pair is published
  // lane r reads CTA r's pair (one remote round trip), the warp combines
  // them in lane 0's order: every thread of the cluster has the same lse
  float2 v = make_float2(-FLT_MAX, 0.f);
  if (lane < (int)ncl) v = ld_shared_cluster_f32x2(mapa_shared(smem_u32(&pub), lane));
  warp_lse_merge(v.x, v.y);
  cluster_arrive_relaxed();  // this CTA no longer reads its peers' shared memory
  const float lse = v.x + __logf(v.y);
  if (rank == 0 && threadIdx.x == 0) loss_rows[row] = lse - z[row * vocab + label];
  const float scale = __expf(mr - lse) * inv_n;
  const int64_t lab4 = (int64_t)label - lo * 4;  // label offset within the slice
  for (int i = threadIdx.x; i < len; i += blockDim.x) {
    const float4 f = slice[i];
    const int64_t k = lab4 - (int64_t)i * 4;
    __nv_bfloat162 lo2 = __floats2bfloat162_rn(f.x * scale - (k == 0 ? inv_n : 0.f),
                                               f.y * scale - (k == 1 ? inv_n : 0.f));
    __nv_bfloat162 hi2 = __floats2bfloat162_rn(f.z * scale - (k == 2 ? inv_n : 0.f),
                                               f.w * scale - (k == 3 ? inv_n : 0.f));
    dr[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo2), *reinterpret_cast<uint32_t*>(&hi2));
  }
  if (!ok && threadIdx.x == 0)  // let copies still in flight land before exit
    for (int k = 0; k < kCePieces; ++k) mbar_wait(smem_u32(&bars[k]), 0, nullptr);
  __syncwarp();
  cluster_wait();  // peers have read this CTA's pair
}

// Two-pass form, for rows longer than the clusters' shared memory holds: one
// CTA per row takes lse by an online max / sum-exp pass over the row in HBM,
// then reads the row again for dz (10 bytes per logit).
__global__ void __launch_bounds__(kCeThreads)
    ce_rows_f32_kernel(const float* __restrict__ z, __nv_bfloat16* __restrict__ dz,
                       const int32_t* __restrict__ labels, int64_t vocab, float inv_n,
                       float* __restrict__ loss_rows, int* err) {
  __shared__ float shm[32], shs[32];
  const int64_t row = blockIdx.x;
  const float4* zr = reinterpret_cast<const float4*>(z + row * vocab);
  uint2* dr = reinterpret_cast<uint2*>(dz + row * vocab);
  int label = labels[row];
  if (label >= vocab) {  // outside the vocabulary: reported, and the row ignored
    if (threadIdx.x == 0) record_error(err, kDevCeBadLabel);
    label = -1;
  }
  const int64_t n4 = vocab >> 2;  // vocab % 8 == 0 (checked by the caller)
  if (label < 0) {
    const uint2 zero = make_uint2(0, 0);
    for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) dr[i] = zero;
    if (threadIdx.x == 0) loss_rows[row] = 0.f;
    return;
  }
  float m = -FLT_MAX, s = 0.f;
  for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 f = zr[i];
    const float lm = fmaxf(fmaxf(f.x, f.y), fmaxf(f.z, f.w));
    if (lm > m) {
      s *= __expf(m - lm);
      m = lm;
    }
    s += __expf(f.x - m) + __expf(f.y - m) + __expf(f.z - m) + __expf(f.w - m);
  }
  // combine (m, s) across the block
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const float wm = warp_max(m);
  s = (m == -FLT_MAX) ? 0.f : s * __expf(m - wm);
  s = warp_sum(s);
  if (lane == 0) { shm[w] = wm; shs[w] = s; }
  __syncthreads();
  float bm = -FLT_MAX;
  for (int i = 0; i < nw; ++i) bm = fmaxf(bm, shm[i]);
  float bs = 0.f;
  for (int i = 0; i < nw; ++i) bs += shs[i] * __expf(shm[i] - bm);
  const float lse = bm + __logf(bs);
  if (threadIdx.x == 0) loss_rows[row] = lse - z[row * vocab + label];
  for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 f = zr[i];
    float p[4] = {__expf(f.x - lse), __expf(f.y - lse), __expf(f.z - lse), __expf(f.w - lse)};
    const int64_t k = label - i * 4;
    if (k >= 0 && k < 4) p[k] -= 1.f;
    __nv_bfloat162 lo = __floats2bfloat162_rn(p[0] * inv_n, p[1] * inv_n);
    __nv_bfloat162 hi = __floats2bfloat162_rn(p[2] * inv_n, p[3] * inv_n);
    dr[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
}

// CTAs per row of the cluster kernel for `vocab` logits: the smallest power
// of two up to kCeMaxCluster whose slices let three CTAs share an SM, else
// kCeMaxCluster while a slice fits kCeSliceMax; 0 (the two-pass kernel) for
// longer rows.
int ce_cluster_size(int64_t vocab) {
  const int64_t n4 = vocab / 4;
  for (int c = 1; c <= kCeMaxCluster; c *= 2)
    if ((n4 + c - 1) / c * 16 <= kCeSliceShare) return c;
  return (n4 + kCeMaxCluster - 1) / kCeMaxCluster * 16 <= kCeSliceMax ? kCeMaxCluster : 0;
}

int ce_rows_f32(const float* z, __nv_bfloat16* dz, const int32_t* labels, int64_t rows,
                int64_t vocab, float inv_n, float* loss_rows, int* err, cudaStream_t st) {
  if (rows <= 0) return 0;
  const int ncl = ce_cluster_size(vocab);
  if (ncl == 0) {
    ce_rows_f32_kernel<<<(unsigned)rows, kCeThreads, 0, st>>>(z, dz, labels, vocab, inv_n,
                                                              loss_rows, err);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
  }
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  if (!attr_set[dev]) {  // idempotent: racing threads set the same value
    if (cudaFuncSetAttribute(ce_rows_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kCeSliceMax) != cudaSuccess)
      return -1;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ncl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(rows * ncl));
  cfg.blockDim = dim3(kCeThreads);
  cfg.dynamicSmemBytes = (size_t)((vocab / 4 + ncl - 1) / ncl * 16);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, ce_rows_cluster_kernel, z, dz, labels, vocab, inv_n, loss_rows,
                         err) != cudaSuccess)
    return -1;
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

// ------------------------------------------------------------------ reductions / casts
// out[0] = scale * sum(x) in a fixed order (one CTA).
__global__ void sum_kernel(const float* __restrict__ x, int64_t n, float scale, float* out) {
  __shared__ float sh[32];
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) acc += x[i];
  float v = block_sum((float)acc, sh);
  if (threadIdx.x == 0) out[0] = v * scale;
}

void sum_f32(const float* x, int64_t n, float scale, float* out, cudaStream_t st) {
  sum_kernel<<<1, 1024, 0, st>>>(x, n, scale, out);
}

__global__ void cast_f32_bf16_kernel(const float* __restrict__ x, __nv_bfloat16* __restrict__ y, int64_t n) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i + 8 <= n) {
    float4 a = reinterpret_cast<const float4*>(x + i)[0], b = reinterpret_cast<const float4*>(x + i)[1];
    float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    *reinterpret_cast<uint4*>(y + i) = pack8(f);
  } else {
    for (int64_t j = i; j < n; ++j) y[j] = __float2bfloat16_rn(x[j]);
  }
}

__global__ void cast_f32_f16_kernel(const float* __restrict__ x, __half* __restrict__ y, int64_t n,
                                    float scale) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i + 8 <= n) {
    const float4 a = reinterpret_cast<const float4*>(x + i)[0], b = reinterpret_cast<const float4*>(x + i)[1];
    const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 h = __floats2half2_rn(f[2 * k] * scale, f[2 * k + 1] * scale);
      w[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(y + i) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    for (int64_t j = i; j < n; ++j) y[j] = __float2half_rn(x[j] * scale);
  }
}

void cast_f32_f16(const float* x, uint16_t* y, int64_t n, float scale, cudaStream_t st) {
  const int64_t threads = (n + 7) / 8;
  cast_f32_f16_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
      x, reinterpret_cast<__half*>(y), n, scale);
}

void cast_f32_bf16(const float* x, __nv_bfloat16* y, int64_t n, cudaStream_t st) {
  const int64_t threads = (n + 7) / 8;
  if (threads <= 0) return;
  cast_f32_bf16_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(x, y, n);
}

__global__ void cast_bf16_f32_kernel(const __nv_bfloat16* __restrict__ x, float* __restrict__ y, int64_t n) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i + 8 <= n) {
    float f[8];
    unpack8(*reinterpret_cast<const uint4*>(x + i), f);
    reinterpret_cast<float4*>(y + i)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(y + i)[1] = make_float4(f[4], f[5], f[6], f[7]);
  } else {
    for (int64_t j = i; j < n; ++j) y[j] = __bfloat162float(x[j]);
  }
}

void cast_bf16_f32(const __nv_bfloat16* x, float* y, int64_t n, cudaStream_t st) {
  const int64_t threads = (n + 7) / 8;
  if (threads <= 0) return;
  cast_bf16_f32_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(x, y, n);
}

}  // namespace sf
