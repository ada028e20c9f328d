// Causal grouped-query attention, forward and backward, with online softmax
// (Milakov & Gimelshein 2018; the tiling of Dao et al., FlashAttention 2022):
// the S x S score matrix never leaves the chip.
//
// Inputs come straight from the QKV projection's output row [T, (Hq+2Hkv)*hd]
// (token t = b*S + s): query head h at column h*hd, kv head g at (Hq+g)*hd
// (K) and (Hq+Hkv+g)*hd (V); query head h reads kv head h / (Hq/Hkv).
//
// Forward: one CTA per (64-query block, query head, batch), 4 warps x 16 rows;
// K/V tiles of 64 keys double-buffered in shared memory by cp.async; scores
// and P in registers (mma.sync m16n8k16 bf16, fp32 accumulate); writes O and
// the row log-sum-exp (natural log, scaled scores).
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

// ------------------------------------------------------------------ forward
template <int HD>
__global__ void __launch_bounds__(128)
    attn_fwd_kernel(const bf16* __restrict__ qkv, bf16* __restrict__ out, float* __restrict__ lse,
                    int S, int Hq, int Hkv, float scale_log2) {
  constexpr int BQ = 64, BKV = 64, LDS = HD + 8;
  extern __shared__ __align__(16) uint8_t smem[];
  bf16* sQ = reinterpret_cast<bf16*>(smem);
  bf16* sK = sQ + BQ * LDS;
  bf16* sV = sK + 2 * BKV * LDS;

  const int nqb = (S + BQ - 1) / BQ;
  const int qb = nqb - 1 - blockIdx.x;  // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (Hq / Hkv);
  const int64_t ld = (int64_t)(Hq + 2 * Hkv) * HD;
  const bf16* base = qkv + (int64_t)b * S * ld;
  const bf16* Qg = base + (int64_t)h * HD;
  const bf16* Kg = base + (int64_t)(Hq + g) * HD;
  const bf16* Vg = base + (int64_t)(Hq + Hkv + g) * HD;
  const int q0 = qb * BQ;
  const int nkv = qb + 1;

  load_tile<HD>(sQ, Qg + (int64_t)q0 * ld, ld, BQ, S - q0);
  load_tile<HD>(sK, Kg, ld, BKV, S);
  load_tile<HD>(sV, Vg, ld, BKV, S);
  cp_async_commit();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t qf[HD / 16][4];
  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-FLT_MAX, -FLT_MAX}, lrow[2] = {0.f, 0.f};

  for (int j = 0; j < nkv; ++j) {
    const int buf = j & 1;
    if (j + 1 < nkv) {
      const int k1 = (j + 1) * BKV;
      load_tile<HD>(sK + (buf ^ 1) * BKV * LDS, Kg + (int64_t)k1 * ld, ld, BKV, S - k1);
      load_tile<HD>(sV + (buf ^ 1) * BKV * LDS, Vg + (int64_t)k1 * ld, ld, BKV, S - k1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (j == 0) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) lds_a(sQ, LDS, warp * 16, kk * 16, qf[kk]);
    }
    const bf16* Kb = sK + buf * BKV * LDS;
    const bf16* Vb = sV + buf * BKV * LDS;
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int n2 = 0; n2 < 4; ++n2) {
        uint32_t b0, b1, b2, b3;
        lds_b_nk(Kb, LDS, n2 * 16, kk * 16, b0, b1, b2, b3);
        mma16816(s[2 * n2], qf[kk], b0, b1);
        mma16816(s[2 * n2 + 1], qf[kk], b2, b3);
      }
    }
    const bool diag = (j == qb);
    float mx[2] = {-FLT_MAX, -FLT_MAX};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = s[nt][e] * scale_log2;
        if (diag) {
          const int key = j * BKV + nt * 8 + 2 * tig + (e & 1);
          const int qr = q0 + warp * 16 + gid + (e >> 1) * 8;
          if (key > qr) v = -FLT_MAX;
        }
        s[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
    float corr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mnew = fmaxf(mrow[r], mx[r]);
      corr[r] = exp2f(mrow[r] - mnew);
      mrow[r] = mnew;
      lrow[r] *= corr[r];
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = exp2f(s[nt][e] - mrow[e >> 1]);
        s[nt][e] = p;
        lrow[e >> 1] += p;
      }
    }
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      o[i][0] *= corr[0]; o[i][1] *= corr[0];
      o[i][2] *= corr[1]; o[i][3] *= corr[1];
    }
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      uint32_t a[4];
      a[0] = pack2(s[2 * kc][0], s[2 * kc][1]);
      a[1] = pack2(s[2 * kc][2], s[2 * kc][3]);
      a[2] = pack2(s[2 * kc + 1][0], s[2 * kc + 1][1]);
      a[3] = pack2(s[2 * kc + 1][2], s[2 * kc + 1][3]);
#pragma unroll
      for (int n2 = 0; n2 < HD / 16; ++n2) {
        uint32_t b0, b1, b2, b3;
        lds_b_kn(Vb, LDS, kc * 16, n2 * 16, b0, b1, b2, b3);
        mma16816(o[2 * n2], a, b0, b1);
        mma16816(o[2 * n2 + 1], a, b2, b3);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
    lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
  }
  const int64_t ldo = (int64_t)Hq * HD;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int qr = q0 + warp * 16 + gid + r * 8;
    if (qr < S) {
      const float inv = 1.f / lrow[r];
      bf16* orow = out + ((int64_t)b * S + qr) * ldo + (int64_t)h * HD;
#pragma unroll
      for (int nt = 0; nt < HD / 8; ++nt)
        *reinterpret_cast<uint32_t*>(orow + nt * 8 + 2 * tig) =
            pack2(o[nt][2 * r] * inv, o[nt][2 * r + 1] * inv);
      if (tig == 0)
        lse[((int64_t)b * Hq + h) * S + qr] = (mrow[r] + log2f(lrow[r])) / kLog2e;
    }
  }
}

template <int HD>
static int fwd_t(const bf16* qkv, bf16* o, float* lse, int B, int S, int Hq, int Hkv,
                 cudaStream_t st) {
  constexpr int LDS = HD + 8;
  const int smem = (64 * LDS + 4 * 64 * LDS) * 2;
  static bool set = false;
  if (!set) {
    cudaFuncSetAttribute(attn_fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    set = true;
  }
  dim3 grid((S + 63) / 64, Hq, B);
  attn_fwd_kernel<HD><<<grid, 128, smem, st>>>(qkv, o, lse, S, Hq, Hkv,
                                               kLog2e / sqrtf((float)HD));
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int attn_fwd(const bf16* qkv, bf16* o, float* lse, int B, int S, int Hq, int Hkv, int hd,
             cudaStream_t st) {
  if (B <= 0 || S <= 0) return 0;
  if (Hkv <= 0 || Hq % Hkv) return -1;
  if (hd == 64) return fwd_t<64>(qkv, o, lse, B, S, Hq, Hkv, st);
  if (hd == 128) return fwd_t<128>(qkv, o, lse, B, S, Hq, Hkv, st);
  return -1;
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

template <int HD>
__global__ void __launch_bounds__(128)
    attn_bwd_kernel(const bf16* __restrict__ qkv, const bf16* __restrict__ dout,
                    const float* __restrict__ lse, const float* __restrict__ delta,
                    float* __restrict__ dq_acc, bf16* __restrict__ dqkv,
                    const float2* __restrict__ cs, int S, int Hq, int Hkv, float scale,
                    float scale_log2) {
  constexpr int BKV = 64, BQ = 32, LDS = HD + 8, LDP = BKV + 8;
  extern __shared__ __align__(16) uint8_t smem[];
  bf16* sK = reinterpret_cast<bf16*>(smem);
  bf16* sV = sK + BKV * LDS;
  bf16* sQ = sV + BKV * LDS;
  bf16* sdO = sQ + BQ * LDS;
  bf16* sdS = sdO + BQ * LDS;  // [BQ][LDP]: dS with queries as rows
  float* sL = reinterpret_cast<float*>(sdS + BQ * LDP);
  float* sD = sL + BQ;

  const int j = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int grp = Hq / Hkv;
  const int k0 = j * BKV;
  const int64_t ld = (int64_t)(Hq + 2 * Hkv) * HD;
  const int64_t ldo = (int64_t)Hq * HD;
  const bf16* base = qkv + (int64_t)b * S * ld;
  load_tile<HD>(sK, base + (int64_t)k0 * ld + (int64_t)(Hq + g) * HD, ld, BKV, S - k0);
  load_tile<HD>(sV, base + (int64_t)k0 * ld + (int64_t)(Hq + Hkv + g) * HD, ld, BKV, S - k0);
  cp_async_commit();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  float dk[HD / 8][4], dv[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;

  const int nqb = (S + BQ - 1) / BQ;
  const int first = k0 / BQ;
  for (int hh = 0; hh < grp; ++hh) {
    const int h = g * grp + hh;
    const float* lse_h = lse + ((int64_t)b * Hq + h) * S;
    const float* del_h = delta + ((int64_t)b * Hq + h) * S;
    for (int i = first; i < nqb; ++i) {
      const int q0 = i * BQ;
      __syncthreads();  // the previous block is done with sQ / sdO / sdS
      load_tile<HD>(sQ, base + (int64_t)q0 * ld + (int64_t)h * HD, ld, BQ, S - q0);
      load_tile<HD>(sdO, dout + ((int64_t)b * S + q0) * ldo + (int64_t)h * HD, ldo, BQ, S - q0);
      cp_async_commit();
      if (threadIdx.x < BQ) {
        const int q = q0 + threadIdx.x;
        sL[threadIdx.x] = (q < S) ? lse_h[q] * kLog2e : 0.f;
        sD[threadIdx.x] = (q < S) ? del_h[q] : 0.f;
      }
      cp_async_wait<0>();
      __syncthreads();

      // S^T = K_w Q^T  (16 keys x 32 queries per warp)
      float st[4][4], dp[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) st[n][e] = dp[n][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        uint32_t ak[4], av[4];
        lds_a(sK, LDS, warp * 16, kk * 16, ak);
        lds_a(sV, LDS, warp * 16, kk * 16, av);
#pragma unroll
        for (int n2 = 0; n2 < 2; ++n2) {
          uint32_t b0, b1, b2, b3;
          lds_b_nk(sQ, LDS, n2 * 16, kk * 16, b0, b1, b2, b3);
          mma16816(st[2 * n2], ak, b0, b1);
          mma16816(st[2 * n2 + 1], ak, b2, b3);
          lds_b_nk(sdO, LDS, n2 * 16, kk * 16, b0, b1, b2, b3);
          mma16816(dp[2 * n2], av, b0, b1);  // dP^T = V_w dO^T
          mma16816(dp[2 * n2 + 1], av, b2, b3);
        }
      }
      // P^T and dS^T
#pragma unroll
      for (int n = 0; n < 4; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = k0 + warp * 16 + gid + (e >> 1) * 8;
          const int ql = n * 8 + 2 * tig + (e & 1);
          const int q = q0 + ql;
          float p = 0.f;
          if (q < S && key <= q) p = exp2f(st[n][e] * scale_log2 - sL[ql]);
          st[n][e] = p;
          dp[n][e] = p * (dp[n][e] - sD[ql]);
        }
      }
      // dV += P^T dO ; dK += dS^T Q   (k = 32 queries = 2 k-steps)
#pragma unroll
      for (int kc = 0; kc < 2; ++kc) {
        uint32_t ap[4], ad[4];
        ap[0] = pack2(st[2 * kc][0], st[2 * kc][1]);
        ap[1] = pack2(st[2 * kc][2], st[2 * kc][3]);
        ap[2] = pack2(st[2 * kc + 1][0], st[2 * kc + 1][1]);
        ap[3] = pack2(st[2 * kc + 1][2], st[2 * kc + 1][3]);
        ad[0] = pack2(dp[2 * kc][0], dp[2 * kc][1]);
        ad[1] = pack2(dp[2 * kc][2], dp[2 * kc][3]);
        ad[2] = pack2(dp[2 * kc + 1][0], dp[2 * kc + 1][1]);
        ad[3] = pack2(dp[2 * kc + 1][2], dp[2 * kc + 1][3]);
#pragma unroll
        for (int n2 = 0; n2 < HD / 16; ++n2) {
          uint32_t b0, b1, b2, b3;
          lds_b_kn(sdO, LDS, kc * 16, n2 * 16, b0, b1, b2, b3);
          mma16816(dv[2 * n2], ap, b0, b1);
          mma16816(dv[2 * n2 + 1], ap, b2, b3);
          lds_b_kn(sQ, LDS, kc * 16, n2 * 16, b0, b1, b2, b3);
          mma16816(dk[2 * n2], ad, b0, b1);
          mma16816(dk[2 * n2 + 1], ad, b2, b3);
        }
        // stash dS (queries as rows) for the dQ product
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = 2 * kc + (e >> 1);
          (void)n;
        }
      }
#pragma unroll
      for (int n = 0; n < 4; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kl = warp * 16 + gid + (e >> 1) * 8;
          const int ql = n * 8 + 2 * tig + (e & 1);
          sdS[ql * LDP + kl] = __float2bfloat16_rn(dp[n][e]);
        }
      }
      __syncthreads();
      // dQ_i += dS K : warp w -> queries (w >> 1) * 16.., hd columns (w & 1) * HD/2..
      {
        const int m0 = (warp >> 1) * 16, c0 = (warp & 1) * (HD / 2);
        float dq[HD / 16][4];
#pragma unroll
        for (int n = 0; n < HD / 16; ++n) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;
#pragma unroll
        for (int kc = 0; kc < BKV / 16; ++kc) {
          uint32_t a[4];
          lds_a(sdS, LDP, m0, kc * 16, a);
#pragma unroll
          for (int n2 = 0; n2 < HD / 32; ++n2) {
            uint32_t b0, b1, b2, b3;
            lds_b_kn(sK, LDS, kc * 16, c0 + n2 * 16, b0, b1, b2, b3);
            mma16816(dq[2 * n2], a, b0, b1);
            mma16816(dq[2 * n2 + 1], a, b2, b3);
          }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int q = q0 + m0 + gid + r * 8;
          if (q < S) {
            float* row = dq_acc + ((int64_t)b * S + q) * ldo + (int64_t)h * HD + c0;
#pragma unroll
            for (int n = 0; n < HD / 16; ++n)
              atomicAdd(reinterpret_cast<float2*>(row + n * 8 + 2 * tig),
                        make_float2(dq[n][2 * r], dq[n][2 * r + 1]));
          }
        }
      }
    }
  }
  // dK (scaled, inverse RoPE) and dV of this block's keys
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int key = k0 + warp * 16 + gid + r * 8;
    if (key >= S) continue;
    bf16* row = dqkv + ((int64_t)b * S + key) * ld;
    bf16* krow = row + (int64_t)(Hq + g) * HD;
    bf16* vrow = row + (int64_t)(Hq + Hkv + g) * HD;
    const float2* c = cs ? cs + (int64_t)key * (HD / 2) : nullptr;
#pragma unroll
    for (int n = 0; n < HD / 16; ++n) {
      float x1a = dk[n][2 * r] * scale, x1b = dk[n][2 * r + 1] * scale;
      float x2a = dk[n + HD / 16][2 * r] * scale, x2b = dk[n + HD / 16][2 * r + 1] * scale;
      const int col = n * 8 + 2 * tig;
      if (c) {
        const float2 ca = c[col], cb = c[col + 1];
        const float y1a = x1a * ca.x + x2a * ca.y, y2a = x2a * ca.x - x1a * ca.y;
        const float y1b = x1b * cb.x + x2b * cb.y, y2b = x2b * cb.x - x1b * cb.y;
        x1a = y1a; x2a = y2a; x1b = y1b; x2b = y2b;
      }
      *reinterpret_cast<uint32_t*>(krow + col) = pack2(x1a, x1b);
      *reinterpret_cast<uint32_t*>(krow + col + HD / 2) = pack2(x2a, x2b);
    }
#pragma unroll
    for (int n = 0; n < HD / 8; ++n)
      *reinterpret_cast<uint32_t*>(vrow + n * 8 + 2 * tig) = pack2(dv[n][2 * r], dv[n][2 * r + 1]);
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

template <int HD>
static int bwd_t(const bf16* qkv, const bf16* o, const bf16* dout, const float* lse, float* delta,
                 float* dq_acc, bf16* dqkv, int B, int S, int Hq, int Hkv, const float2* cs,
                 cudaStream_t st) {
  constexpr int LDS = HD + 8, LDP = 64 + 8;
  const int smem = (2 * 64 * LDS + 2 * 32 * LDS + 32 * LDP) * 2 + 2 * 32 * 4;
  static bool set = false;
  if (!set) {
    cudaFuncSetAttribute(attn_bwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    set = true;
  }
  const int64_t T = (int64_t)B * S;
  const int64_t rows = T * Hq;
  if (cudaMemsetAsync(dq_acc, 0, (size_t)T * Hq * HD * sizeof(float), st) != cudaSuccess) return -3;
  attn_delta_kernel<<<(unsigned)((rows * 32 + 255) / 256), 256, 0, st>>>(o, dout, delta, rows, S, Hq, HD);
  const float scale = 1.f / sqrtf((float)HD);
  dim3 grid((S + 63) / 64, Hkv, B);
  attn_bwd_kernel<HD><<<grid, 128, smem, st>>>(qkv, dout, lse, delta, dq_acc, dqkv, cs, S, Hq, Hkv,
                                               scale, scale * kLog2e);
  const int64_t n = T * Hq * (HD / 16);
  attn_dq_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(dq_acc, dqkv, T, S, Hq, Hkv, HD, scale, cs);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int attn_bwd(const bf16* qkv, const bf16* o, const bf16* dout, const float* lse, float* delta,
             float* dq_acc, bf16* dqkv, int B, int S, int Hq, int Hkv, int hd, const float2* cs,
             cudaStream_t st) {
  if (B <= 0 || S <= 0) return 0;
  if (Hkv <= 0 || Hq % Hkv) return -1;
  if (hd == 64) return bwd_t<64>(qkv, o, dout, lse, delta, dq_acc, dqkv, B, S, Hq, Hkv, cs, st);
  if (hd == 128) return bwd_t<128>(qkv, o, dout, lse, delta, dq_acc, dqkv, B, S, Hq, Hkv, cs, st);
  return -1;
}

}  // namespace sf
