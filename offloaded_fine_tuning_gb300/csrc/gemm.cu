// Dense bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), operands
// staged by TMA.  Every dense contraction of the decoder step runs here: the
// QKV, O, gate/up and down projections forward, their dX and dW products
// backward, and the three LM-head products of the fused cross-entropy.
//
// Design (one persistent CTA per SM, 192 threads):
//   warp 0      TMA producer: A and B tiles of BK = 64 into a STAGES-deep ring
//   warp 1      MMA issuer: tcgen05.mma into a TMEM accumulator; also
//               allocates / frees TMEM (512 columns = 2 accumulators)
//   warps 2-5   epilogue: tcgen05.ld rows out of TMEM, convert, store
// Two TMEM accumulators let the epilogue of tile i overlap the mainloop of
// tile i+1.
//
// Work units are visited in groups along M or N (tile_coords, unit_order), so
// that the operand panels a group shares stay in L2.
//
// With BN = 256 the CTAs run in clusters of two that compute one 256 x 256
// tile with cta_group::2 MMAs (M = 256 across the pair): each CTA loads its
// own 128 rows of A and its half of B into its own shared memory (32 KB per
// k-block instead of the 48 KB a 128 x 256 tile needs), the leader's MMA
// warp issues for both SMs, whose tensor cores read A from their own shared
// memory and B from both, and each CTA's TMEM holds its 128 rows of D.  With
// half the operand bytes per SM in shared memory the ring has six stages, and
// the GEMMs went from 0.87-0.91 to 0.94-0.99 of the measured cuBLAS burst
// rate.  All operands use the 128-byte swizzle: a K-major tile is [rows][64]
// with 128-byte rows; an MN-major tile is a set of [64 K rows] x [64 MN]
// boxes placed 8 KB apart.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ptx.cuh"
#include "sf_internal.h"

namespace sf {

struct GemmParams {
  int M, N, K;
  void* C;
  int64_t ldc;
  const float* R;
  int64_t ldr;
  float alpha;
  int* err;
  const __nv_bfloat16* bias;  // kEpiBF16Bias, kEpiQKV: one value per output column (or null)
  const float2* cs;           // kEpiQKV: (cos, sin) [seq, hd/2]
  int seq, rope_cols, hd;
  float* aux;                 // kEpiGLU: fp32 a | b (or null)
  int64_t ldaux;
  int group;                  // work-unit order (tile_coords)
  int splitk;                 // K ranges (kEpiF32): split s > 0 writes ws + (s - 1) * ws_stride
  float* ws;
  int64_t ws_stride;
};

// Output columns of one work unit: the gated tile computes a and b for 128
// output columns in its 256 accumulator columns.
template <int BN, int EPI>
__host__ __device__ constexpr int unit_cols() { return EPI == kEpiGLU ? BN / 2 : BN; }

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;

// Shared memory of one CTA: STAGES x (A tile + B tile).  A pair of CTAs
// under one cta_group::2 MMA holds half of the B tile in each CTA.
template <int BN, bool PAIR = false>
struct GemmCfg {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * kBK * 2;
  static constexpr int STAGES = PAIR ? 6 : ((BN == 256) ? 4 : 6);
  static constexpr int BAR_OFF = STAGES * (A_BYTES + B_BYTES);
  // full[S], empty[S], tfull[2], tempty[2], drain; then tmem slot and abort flag
  static constexpr int SMEM = BAR_OFF + (2 * STAGES + 5) * 8 + 16 + 1024;
};

// Work-unit order.  Units are visited in groups: with group > 0, groups of
// `group` M-units crossed with every N-tile (the group's A panels stay in L2
// while the B panel streams through once per group); with group < 0, groups
// of -group N-tiles crossed with every M-unit (the group's B panels stay in
// L2 while A streams through once per group).  The host picks the side whose
// re-reads cost fewer bytes, with the resident panels within a share of L2.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group, int& tm,
                                            int& tn) {
  if (group > 0) {
    const int per_group = group * num_n;
    const int first_m = (tile / per_group) * group;
    const int gsize = min(num_m - first_m, group);
    const int r = tile % per_group;
    tm = first_m + r % gsize;
    tn = r / gsize;
  } else {
    const int g = -group;
    const int per_group = g * num_m;
    const int first_n = (tile / per_group) * g;
    const int gsize = min(num_n - first_n, g);
    const int r = tile % per_group;
    tn = first_n + r % gsize;
    tm = r / gsize;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 32 bf16 values to c[0..32): four 16-byte stores when the row has all of
// them and c is aligned, else one per column below n.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* c, const float (&y)[32], int n) {
  if (n >= 32 && ((reinterpret_cast<uintptr_t>(c) & 15) == 0)) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 v;
      v.x = pack_bf16x2(y[8 * q + 0], y[8 * q + 1]);
      v.y = pack_bf16x2(y[8 * q + 2], y[8 * q + 3]);
      v.z = pack_bf16x2(y[8 * q + 4], y[8 * q + 5]);
      v.w = pack_bf16x2(y[8 * q + 6], y[8 * q + 7]);
      reinterpret_cast<uint4*>(c)[q] = v;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n) c[j] = __float2bfloat16_rn(y[j]);
  }
}

__device__ __forceinline__ void store_f32x32(float* c, const float (&y)[32], int n) {
  if (n >= 32 && ((reinterpret_cast<uintptr_t>(c) & 15) == 0)) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      reinterpret_cast<float4*>(c)[q] = make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n) c[j] = y[j];
  }
}

__device__ __forceinline__ void load_f32x32(const float* c, float (&y)[32], int n) {
  if (n >= 32 && ((reinterpret_cast<uintptr_t>(c) & 15) == 0)) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 v = reinterpret_cast<const float4*>(c)[q];
      y[4 * q] = v.x; y[4 * q + 1] = v.y; y[4 * q + 2] = v.z; y[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = j < n ? c[j] : 0.f;
  }
}

// y[j] += bias[col + j] for the columns below n (bias 64-byte aligned, col % 32 == 0)
__device__ __forceinline__ void add_bias32(float (&y)[32], const __nv_bfloat16* bias, int n) {
  if (n >= 32) {
    const uint4* b4 = reinterpret_cast<const uint4*>(bias);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = b4[q];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        y[8 * q + 2 * k] += __uint_as_float(w[k] << 16);
        y[8 * q + 2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n) y[j] += __bfloat162float(bias[j]);
  }
}

// The Q/K/V projection's epilogue for 32 rotation pairs of one head: x1 holds
// the accumulator columns [col1, col1 + 32), x2 the columns 
// [col1 + hd/2, ...) of the same head; pair index jp = first pair's index j.
__device__ __forceinline__ void epi_qkv_pairs(const GemmParams& p, int row, int col1, int jp,
                                              const uint32_t (&r1)[32], const uint32_t (&r2)[32]) {
  const int half = p.hd >> 1;
  const int col2 = col1 + half;
  float x1[32], x2[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    x1[j] = __uint_as_float(r1[j]) * p.alpha;
    x2[j] = __uint_as_float(r2[j]) * p.alpha;
  }
  if (p.bias) {  // added before the rotation, in fp32
    add_bias32(x1, p.bias + col1, 32);
    add_bias32(x2, p.bias + col2, 32);
  }
  if (col1 < p.rope_cols) {
    const int s = row % p.seq;
    const float4* t = reinterpret_cast<const float4*>(p.cs + (int64_t)s * half + jp);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const float4 c = t[q];  // (cos, sin) of pairs jp + 2q and jp + 2q + 1
      const float a0 = x1[2 * q], b0 = x2[2 * q], a1 = x1[2 * q + 1], b1 = x2[2 * q + 1];
      x1[2 * q] = a0 * c.x - b0 * c.y;
      x2[2 * q] = b0 * c.x + a0 * c.y;
      x1[2 * q + 1] = a1 * c.z - b1 * c.w;
      x2[2 * q + 1] = b1 * c.z + a1 * c.w;
    }
  }
  __nv_bfloat16* c = reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc;
  store_bf16x32(c + col1, x1, 32);
  store_bf16x32(c + col2, x2, 32);
}

// The gate/up projection's SwiGLU epilogue for output columns [j, j + 32):
// ra holds a (gate), rb holds b (up).
__device__ __forceinline__ void epi_glu(const GemmParams& p, int row, int j,
                                        const uint32_t (&ra)[32], const uint32_t (&rb)[32]) {
  const int n = min(32, p.N - j);
  float a[32], b[32], m[32];
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    a[k] = __uint_as_float(ra[k]) * p.alpha;
    b[k] = __uint_as_float(rb[k]) * p.alpha;
    m[k] = a[k] / (1.f + __expf(-a[k])) * b[k];
  }
  store_bf16x32(reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc + j, m, n);
  if (p.aux) {
    float* x = p.aux + (int64_t)row * p.ldaux + j;
    store_f32x32(x, a, n);
    store_f32x32(x + p.N, b, n);
  }
}

// Store 32 accumulator columns [col, col+32) of one output row.
template <int EPI>
__device__ __forceinline__ void epi_store(const GemmParams& p, int row, int col,
                                          const uint32_t (&r)[32]) {
  const float a = p.alpha;
  const float a_ = a;
  const bool full = (col + 32 <= p.N);
  if constexpr (EPI == kEpiBF16 || EPI == kEpiBF16Bias) {
    __nv_bfloat16* c = reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc + col;
    float y[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(r[j]) * a;
    if constexpr (EPI == kEpiBF16Bias) {  // + bias[col], in fp32 before the rounding
      if (full) {
        const uint4* b4 = reinterpret_cast<const uint4*>(p.bias + col);  // 64-byte aligned: col % 32 == 0
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 u = b4[q];
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            y[8 * q + 2 * k] += __uint_as_float(w[k] << 16);
            y[8 * q + 2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col + j < p.N) y[j] += __bfloat162float(p.bias[col + j]);
      }
    }
    if (full && ((reinterpret_cast<uintptr_t>(c) & 15) == 0)) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 v;
        v.x = pack_bf16x2(y[8 * q + 0], y[8 * q + 1]);
        v.y = pack_bf16x2(y[8 * q + 2], y[8 * q + 3]);
        v.z = pack_bf16x2(y[8 * q + 4], y[8 * q + 5]);
        v.w = pack_bf16x2(y[8 * q + 6], y[8 * q + 7]);
        reinterpret_cast<uint4*>(c)[q] = v;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col + j < p.N) c[j] = __float2bfloat16_rn(y[j]);
    }
  } else if constexpr (EPI == kEpiGLUBwd) {
    // dm = alpha*acc; a, b from the forward (fp32); da | db as bf16
    const int n = min(32, p.N - col);
    const float* ar = p.R + (int64_t)row * p.ldr + col;
    float a[32], b[32], da[32], db[32];
    load_f32x32(ar, a, n);
    load_f32x32(ar + p.N, b, n);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float g = __uint_as_float(r[j]) * a_;
      const float sg = 1.f / (1.f + __expf(-a[j]));
      da[j] = g * b[j] * sg * (1.f + a[j] * (1.f - sg));
      db[j] = g * a[j] * sg;
    }
    __nv_bfloat16* c = reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc + col;
    store_bf16x32(c, da, n);
    store_bf16x32(c + p.N, db, n);
  } else if constexpr (EPI == kEpiBF16Acc) {
    const int n = min(32, p.N - col);
    float y[32];
    if (p.R) load_f32x32(p.R + (int64_t)row * p.ldr + col, y, n);
#pragma unroll
    for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(r[j]) * a_ + (p.R ? y[j] : 0.f);
    store_bf16x32(reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc + col, y, n);
  } else if constexpr (EPI == kEpiF16) {
    __half* c = reinterpret_cast<__half*>(p.C) + (int64_t)row * p.ldc + col;
    if (full && ((reinterpret_cast<uintptr_t>(c) & 15) == 0)) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          __half2 h = __floats2half2_rn(__uint_as_float(r[8 * q + 2 * k]) * a,
                                        __uint_as_float(r[8 * q + 2 * k + 1]) * a);
          w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        reinterpret_cast<uint4*>(c)[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col + j < p.N) c[j] = __float2half_rn(__uint_as_float(r[j]) * a);
    }
  } else {
    float* c = reinterpret_cast<float*>(p.C) + (int64_t)row * p.ldc + col;
    const float* rr = nullptr;
    if constexpr (EPI == kEpiF32Add) rr = p.R + (int64_t)row * p.ldr + col;
    if constexpr (EPI == kEpiF32Acc) rr = c;
    if (full && ((reinterpret_cast<uintptr_t>(c) & 15) == 0) &&
        (rr == nullptr || (reinterpret_cast<uintptr_t>(rr) & 15) == 0)) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 v = make_float4(__uint_as_float(r[4 * q + 0]) * a, __uint_as_float(r[4 * q + 1]) * a,
                               __uint_as_float(r[4 * q + 2]) * a, __uint_as_float(r[4 * q + 3]) * a);
        if constexpr (EPI == kEpiF32Add || EPI == kEpiF32Acc) {
          const float4 b = reinterpret_cast<const float4*>(rr)[q];
          v.x += b.x; v.y += b.y; v.z += b.z; v.w += b.w;
        }
        reinterpret_cast<float4*>(c)[q] = v;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (col + j < p.N) {
          float v = __uint_as_float(r[j]) * a;
          if constexpr (EPI == kEpiF32Add || EPI == kEpiF32Acc) v += rr[j];
          c[j] = v;
        }
      }
    }
  }
}

// CL == 2 (the 256-wide tiles): the two CTAs of a cluster run one
// cta_group::2 MMA of 256 x BN: each loads its own 128 rows of A and half of
// B into its own shared memory, both counted on the leader's (rank 0) full
// barrier; the leader's MMA warp issues for the pair and its commits reach
// both CTAs; each CTA's epilogue reads its own 128 rows from its own TMEM and
// reports to the leader that the buffer is free.  CL == 1 (narrow tiles):
// one CTA, one 128 x BN MMA.
template <bool A_MN, bool B_MN, int BN, int EPI, int CL>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmB2, const GemmParams p) {
  static_assert(CL == 1 || CL == 2, "clusters of one or two CTAs");
  constexpr bool PAIR = (CL == 2);
  static_assert(!PAIR || BN == 256, "pair MMAs: 256-wide tiles");
  // the gated tile: the cluster's two CTAs load the gate rows (tmB) and the
  // up rows (tmB2) of the same 128 output columns
  constexpr bool GATED = (EPI == kEpiGLU);
  static_assert(!GATED || (CL == 2 && BN == 256 && !B_MN), "gated tiles: 2-CTA clusters, K-major B");
  constexpr int UC = unit_cols<BN, EPI>();
  using Cfg = GemmCfg<BN, PAIR>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int A_BYTES = Cfg::A_BYTES, B_BYTES = Cfg::B_BYTES;
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t IDESC = umma_idesc_bf16(PAIR ? 2 * kBM : kBM, BN, A_MN, B_MN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // CTA rank in the cluster: which M-tile of the pair, and which half of B it loads
  const int crank = CL == 2 ? (int)cluster_ctarank() : 0;
  constexpr uint16_t kPair = 0x3;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);  // by the commit of the (pair's) MMA warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      // pair: one arrival per epilogue warp of both CTAs, on the leader's barrier
      mbar_init(tempty_bar(b), PAIR ? 8 : 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (GATED) tma_prefetch_desc(&tmB2);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (CL == 2) cluster_sync_all();  // the peer's barriers exist before its first remote arrival
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // work units: CL M-tiles of one N-tile, one per CTA of the cluster, times
  // the K ranges (all tiles of range 0 first)
  const int num_m = (p.M + kBM - 1) / kBM;
  const int num_mu = (num_m + CL - 1) / CL;
  const int num_n = (p.N + UC - 1) / UC;
  const int num_mn = num_mu * num_n;
  const int splitk = p.splitk > 1 ? p.splitk : 1;
  const int num_units = num_mn * splitk;
  const int unit0 = (int)blockIdx.x / CL, unit_step = (int)gridDim.x / CL;
  const int nk = (p.K + kBK - 1) / kBK;
  const int kps = (nk + splitk - 1) / splitk;  // k-blocks per range (the host keeps every range non-empty)
  auto krange = [&](int unit, int& umn, int& kb0, int& kb1) {
    const int ks = unit / num_mn;
    umn = unit - ks * num_mn;
    kb0 = ks * kps;
    kb1 = kb0 + kps < nk ? kb0 + kps : nk;
  };

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- producer
    int stage = 0;
    uint32_t phase = 0;
    long issued = 0;
    bool ok = true;
    for (int unit = unit0; unit < num_units && ok; unit += unit_step) {
      int tmu, tn, umn, kb0, kb1;
      krange(unit, umn, kb0, kb1);
      tile_coords(umn, num_mu, num_n, p.group, tmu, tn);
      const int m0 = (tmu * CL + crank) * kBM, n0 = tn * BN;
      for (int kb = kb0; kb < kb1; ++kb) {
        // the stage is free once the MMAs that read it (the pair's, for a pair) completed
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) { ok = false; break; }
        const int k0 = kb * kBK;
        const uint32_t a_dst = sA + stage * A_BYTES, b_dst = sB + stage * B_BYTES;
        if constexpr (PAIR) {
          // both CTAs' tiles count on the leader's full barrier
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          if (crank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * (A_BYTES + B_BYTES));
          if constexpr (A_MN) {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j) tma_load_2d_pair(a_dst + j * 8192, &tmA, fb, m0 + 64 * j, k0);
          } else {
            tma_load_2d_pair(a_dst, &tmA, fb, k0, m0);
          }
          constexpr int HB = BN / 2;  // this CTA's half of B
          if constexpr (B_MN) {
#pragma unroll
            for (int j = 0; j < HB / 64; ++j)
              tma_load_2d_pair(b_dst + j * 8192, &tmB, fb, n0 + crank * HB + 64 * j, k0);
          } else if constexpr (GATED) {
            tma_load_2d_pair(b_dst, crank ? &tmB2 : &tmB, fb, k0, tn * UC);
          } else {
            tma_load_2d_pair(b_dst, &tmB, fb, k0, n0 + crank * HB);
          }
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          continue;
        }
        mbar_arrive_expect_tx(full_bar(stage), A_BYTES + B_BYTES);
        if constexpr (A_MN) {
#pragma unroll
          for (int j = 0; j < kBM / 64; ++j) tma_load_2d(a_dst + j * 8192, &tmA, full_bar(stage), m0 + 64 * j, k0);
        } else {
          tma_load_2d(a_dst, &tmA, full_bar(stage), k0, m0);
        }
        if constexpr (B_MN) {
#pragma unroll
          for (int j = 0; j < BN / 64; ++j) tma_load_2d(b_dst + j * 8192, &tmB, full_bar(stage), n0 + 64 * j, k0);
        } else {
          tma_load_2d(b_dst, &tmB, full_bar(stage), k0, n0);
        }
        ++issued;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (ok) {
      // every stage this CTA loaded has been released by the MMAs, so no
      // arrival is still on its way to the barriers and no MMA reads the tiles
      const long n = issued < STAGES ? issued : STAGES;
      int st = stage;
      uint32_t ph = phase;
      for (long i = 0; i < n && ok; ++i) {
        if (st == 0) { st = STAGES - 1; ph ^= 1u; } else { --st; }
        ok = mbar_wait(empty_bar(st), ph, abort_flag);
      }
      if (!ok) { record_error(p.err, kDevGemmTimeout); *abort_flag = 1; }
    }
    if (!ok) {
      record_error(p.err, kDevGemmTimeout);
      *abort_flag = 1;
      // let the copies already issued land before the CTA's shared memory goes
      // away (a pair's loads count on the leader's barriers: the leader waits)
      const long n = issued < STAGES ? issued : STAGES;
      if (!PAIR || crank == 0) {
        for (long i = 0; i < n; ++i) {
          if (stage == 0) { stage = STAGES - 1; phase ^= 1u; } else { --stage; }
          mbar_wait(full_bar(stage), phase, nullptr);
        }
      }
    }
  } else if (warp == 1 && lane == 0 && (!PAIR || crank == 0)) {
    // ---------------------------------------------------------------- MMA issuer
    int stage = 0;
    uint32_t phase = 0;
    int iter = 0;
    bool ok = true;
    for (int unit = unit0; unit < num_units && ok; unit += unit_step, ++iter) {
      const int acc = iter & 1;
      const uint32_t acc_phase = (iter >> 1) & 1;
      if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      int umn, kb0, kb1;
      krange(unit, umn, kb0, kb1);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_base = sA + stage * A_BYTES, b_base = sB + stage * B_BYTES;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          uint64_t ad, bd;
          if constexpr (A_MN) ad = smem_desc_sw128(a_base + k * 2048, 8192, 1024);
          else ad = smem_desc_sw128(a_base + k * 32, 16, 1024);
          if constexpr (B_MN) bd = smem_desc_sw128(b_base + k * 2048, 8192, 1024);
          else bd = smem_desc_sw128(b_base + k * 32, 16, 1024);
          const uint32_t accum = (kb != kb0 || k != 0) ? 1u : 0u;
          if constexpr (PAIR) umma_bf16_pair(d_tmem, ad, bd, IDESC, accum);
          else umma_bf16(d_tmem, ad, bd, IDESC, accum);
        }
        if constexpr (PAIR) umma_commit_pair(empty_bar(stage), kPair);
        else umma_commit(empty_bar(stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if constexpr (PAIR) umma_commit_pair(tfull_bar(acc), kPair);
      else umma_commit(tfull_bar(acc));
    }
    if (!ok) {
      record_error(p.err, kDevGemmTimeout);
      *abort_flag = 1;
      if constexpr (PAIR) umma_commit_pair(drain_bar, 0x1);
      else umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, nullptr);
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    int iter = 0;
    for (int unit = unit0; unit < num_units; unit += unit_step, ++iter) {
      int tmu, tn, umn, kb0, kb1;
      krange(unit, umn, kb0, kb1);
      tile_coords(umn, num_mu, num_n, p.group, tmu, tn);
      const int tm = tmu * CL + crank;
      const int acc = iter & 1;
      const uint32_t acc_phase = (iter >> 1) & 1;
      bool ok = mbar_wait(tfull_bar(acc), acc_phase, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        if (lane == 0) { record_error(p.err, kDevGemmTimeout); *abort_flag = 1; }
        break;
      }
      tc_fence_after();
      const int row = tm * kBM + quarter * 32 + lane;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if constexpr (EPI == kEpiQKV) {
        // head by head: the pair (j, j + hd/2) meets in one thread
        const int half = p.hd >> 1;
        for (int h0 = 0; h0 < BN; h0 += p.hd) {
          const int col0 = tn * BN + h0;
          if (col0 >= p.N) break;  // uniform across the warp
          for (int j = 0; j < half; j += 32) {
            uint32_t r1[32], r2[32];
            tmem_ld_32x32b_x32(taddr + h0 + j, r1);
            tmem_ld_32x32b_x32(taddr + h0 + half + j, r2);
            tmem_ld_wait();
            if (row < p.M) epi_qkv_pairs(p, row, col0 + j, j, r1, r2);
          }
        }
      } else if constexpr (GATED) {
        // accumulator columns [0, 128): a; [128, 256): b, for the same outputs
        for (int c = 0; c < UC; c += 32) {
          const int col = tn * UC + c;
          if (col >= p.N) break;
          uint32_t ra[32], rb[32];
          tmem_ld_32x32b_x32(taddr + c, ra);
          tmem_ld_32x32b_x32(taddr + UC + c, rb);
          tmem_ld_wait();
          if (row < p.M) epi_glu(p, row, col, ra, rb);
        }
      } else {
        // a K range after the first (kEpiF32) writes into its workspace slice
        GemmParams q = p;
        if constexpr (EPI == kEpiF32) {
          if (unit >= num_mn) q.C = p.ws + (int64_t)(unit / num_mn - 1) * p.ws_stride;
        }
        for (int c = 0; c < BN; c += 32) {
          const int col = tn * BN + c;
          if (col >= p.N) break;  // uniform across the warp
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c, r);
          tmem_ld_wait();
          if (row < p.M) epi_store<EPI>(q, row, col, r);
        }
      }
      tc_fence_before();
      if constexpr (PAIR) {
        // the leader's MMA warp reuses the buffer once both CTAs' warps are done
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(tempty_bar(acc), 0));
      } else {
        mbar_arrive(tempty_bar(acc));
      }
    }
  }
  tc_fence_before();
  if constexpr (PAIR) {
    // the pair's MMAs read both CTAs' shared memory and write both TMEMs:
    // neither CTA frees them before the other is done
    cluster_sync_all();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, cols] matrix with row stride ld
// (elements), box [box_rows, 64] with the 128-byte swizzle.
static bool make_map(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t ld,
                     int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// CTAs per cluster: the wide tiles run as cta_group::2 pair MMAs.
constexpr int gemm_cluster(int BN) { return BN == 256 ? 2 : 1; }

constexpr int kMaxDevices = 64;

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return -1;
  }
  return dev;
}

// SM count of the current device, looked up once per device.
int num_sms() {
  static int n[kMaxDevices] = {0};
  const int dev = current_device();
  if (dev < 0) return 1;
  if (n[dev] == 0) {  // idempotent: racing threads store the same value
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
      cudaGetLastError();
      v = 1;
    }
    n[dev] = v;
  }
  return n[dev];
}

template <bool A_MN, bool B_MN, int BN, int EPI>
static int launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tb2,
                    const GemmParams& p, cudaStream_t st, char* why) {
  constexpr int CL = gemm_cluster(BN);
  using Cfg = GemmCfg<BN, CL == 2>;
  constexpr int UC = unit_cols<BN, EPI>();
  auto kern = gemm_tcgen05_kernel<A_MN, B_MN, BN, EPI, CL>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // per instantiation and device: the shared-memory attribute is set and the
  // number of CTAs that can be resident at once is found on first use there
  static int max_ctas[kMaxDevices] = {0};
  static std::mutex mu;
  const int dev = current_device();
  if (dev < 0) {
    snprintf(why, 64, "gemm: no current device");
    return -3;
  }
  int ctas;
  {
    std::lock_guard<std::mutex> l(mu);
    if (max_ctas[dev] == 0) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) !=
          cudaSuccess) {
        cudaGetLastError();
        snprintf(why, 64, "gemm: cannot reserve %d B shared memory", Cfg::SMEM);
        return -3;
      }
      int clusters = 0;
      cfg.gridDim = dim3(CL * num_sms());
      if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) {
        cudaGetLastError();
        snprintf(why, 64, "gemm: no resident cluster of %d CTAs", CL);
        return -3;
      }
      max_ctas[dev] = clusters * CL < num_sms() ? clusters * CL : num_sms() / CL * CL;
    }
    ctas = max_ctas[dev];
  }
  const int units = ((p.M + kBM * CL - 1) / (kBM * CL)) * ((p.N + UC - 1) / UC) * (p.splitk > 1 ? p.splitk : 1);
  cfg.gridDim = dim3(units * CL < ctas ? units * CL : ctas);
  cudaLaunchKernelEx(&cfg, kern, ta, tb, tb2, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(why, 64, "gemm launch: %s", cudaGetErrorString(e));
    return -3;
  }
  return 0;
}

template <bool A_MN, bool B_MN, int BN>
static int launch_epi(int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                      const CUtensorMap& tb2, const GemmParams& p, cudaStream_t st, char* why) {
  switch (epi) {
    case kEpiBF16: return launch_t<A_MN, B_MN, BN, kEpiBF16>(ta, tb, tb2, p, st, why);
    case kEpiF32: return launch_t<A_MN, B_MN, BN, kEpiF32>(ta, tb, tb2, p, st, why);
    case kEpiF32Add: return launch_t<A_MN, B_MN, BN, kEpiF32Add>(ta, tb, tb2, p, st, why);
    case kEpiF32Acc: return launch_t<A_MN, B_MN, BN, kEpiF32Acc>(ta, tb, tb2, p, st, why);
    case kEpiBF16Bias:  // forward projections only (Y = X W^T + b)
      if constexpr (!A_MN && !B_MN) return launch_t<A_MN, B_MN, BN, kEpiBF16Bias>(ta, tb, tb2, p, st, why);
      break;
    case kEpiQKV:  // the Q/K/V projection with its rotation
      if constexpr (!A_MN && !B_MN) return launch_t<A_MN, B_MN, BN, kEpiQKV>(ta, tb, tb2, p, st, why);
      break;
    case kEpiGLU:  // the gate/up projection with SwiGLU: 256-column gated tiles only
      if constexpr (!A_MN && !B_MN && BN == 256) return launch_t<A_MN, B_MN, BN, kEpiGLU>(ta, tb, tb2, p, st, why);
      break;
    case kEpiGLUBwd:  // the down projection's input gradient through SwiGLU
      if constexpr (!A_MN && B_MN) return launch_t<A_MN, B_MN, BN, kEpiGLUBwd>(ta, tb, tb2, p, st, why);
      break;
    case kEpiF16:  // weight gradients only (dW = dY^T X)
      if constexpr (A_MN && B_MN) return launch_t<A_MN, B_MN, BN, kEpiF16>(ta, tb, tb2, p, st, why);
      break;
    case kEpiBF16Acc:  // the last chunk of a summed weight gradient
      if constexpr (A_MN && B_MN) return launch_t<A_MN, B_MN, BN, kEpiBF16Acc>(ta, tb, tb2, p, st, why);
      break;
  }
  snprintf(why, 64, "gemm: bad epilogue %d", epi);
  return -1;
}

static bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int gemm_check(const GemmArgs& a, char* why) {
  if (a.M == 0 || a.N == 0) return 0;
  if (a.M < 0 || a.N < 0 || a.K <= 0 || a.M > INT32_MAX || a.N > INT32_MAX || a.K > INT32_MAX) {
    snprintf(why, 64, "gemm: bad sizes");
    return -1;
  }
  const int need_layout[] = {-1, -1, -1, -1, kNT, kTN, kNT, kNT, kNN, kTN};
  if (a.layout < kNT || a.layout > kTN || a.epi < kEpiBF16 || a.epi > kEpiBF16Acc ||
      (need_layout[a.epi] >= 0 && a.layout != need_layout[a.epi])) {
    snprintf(why, 64, "gemm: bad layout %d or epilogue %d", a.layout, a.epi);
    return -1;
  }
  if (!a.A || !a.B || !a.C || (a.epi == kEpiF32Add && !a.R) || (a.epi == kEpiBF16Bias && !a.bias) ||
      (a.epi == kEpiGLUBwd && !a.R) || (a.epi == kEpiQKV && !a.cs)) {
    snprintf(why, 64, "gemm: null operand");
    return -1;
  }
  if ((a.epi == kEpiBF16Bias || a.epi == kEpiQKV) && a.bias && !al(a.bias, 64)) {
    snprintf(why, 64, "gemm: bias must be 64-byte aligned");
    return -1;
  }
  // TMA: 16-byte aligned bases and row strides.
  if (!al(a.A, 16) || !al(a.B, 16) || (a.lda % 8) || (a.ldb % 8)) {
    snprintf(why, 64, "gemm: operands must be 16-byte aligned");
    return -1;
  }
  const bool a_mn = (a.layout == kTN);
  const bool b_mn = (a.layout == kNN || a.layout == kTN);
  // row extents of the stored matrices must fit their leading dimensions
  const int64_t a_cols = a_mn ? a.M : a.K, b_cols = b_mn ? a.N : a.K;
  const bool reads_r = a.epi == kEpiF32Add || a.epi == kEpiGLUBwd || (a.epi == kEpiBF16Acc && a.R);
  const int64_t r_cols = a.epi == kEpiGLUBwd ? 2 * a.N : a.N;
  const int64_t c_cols = a.epi == kEpiGLUBwd ? 2 * a.N : a.N;
  if (a.lda < a_cols || a.ldb < b_cols || a.ldc < c_cols || (reads_r && a.ldr < r_cols)) {
    snprintf(why, 64, "gemm: leading dimension too small");
    return -1;
  }
  if (a.epi == kEpiQKV) {
    if ((a.hd != 64 && a.hd != 128) || a.seq < 1 || a.N % a.hd || a.rope_cols < 0 ||
        a.rope_cols % a.hd || a.rope_cols > a.N || a.ldc % 8 || !al(a.C, 16) || !al(a.cs, 16)) {
      snprintf(why, 64, "gemm: bad rotation arguments");
      return -1;
    }
  }
  if (a.epi == kEpiGLU || a.epi == kEpiGLUBwd) {
    // the gated tile holds 2 x 128 columns; SwiGLU halves sit N apart
    if (a.N % 8 || (a.epi == kEpiGLU && a.aux && (a.ldaux < 2 * a.N || a.ldaux % 4 || !al(a.aux, 16))) ||
        (a.epi == kEpiGLUBwd && (a.ldr % 4 || !al(a.R, 16)))) {
      snprintf(why, 64, "gemm: bad SwiGLU arguments");
      return -1;
    }
  }
  return 0;
}

// The unit order of tile_coords.  By default groups of 8 M-units: the ~76
// clusters that run at once then cover about 8 M-units x 9 N-tiles, a near
// square window whose panels the L2 serves without hot spots.  Two cases do
// better with a whole side resident in L2 (each of its panels then leaves
// DRAM once), as measured at the step's shapes: all M-units in one group when
// their A panels fit in 40 MB (the LM head's logits: -2%), and all N-tiles in
// one group when there are at most 16 and their B panels fit (the output
// projection and its dX product: -4 to -5%; the LM head's dW: -2%).  The Q/K/V
// projection's 24 N-tiles make an all-N window of 3 x 24 that ran 3% slower
// than groups of 8, and 16 panels of 50 MB in all (the Q/K/V dX product) 2%.
static int unit_order(int64_t M, int64_t N, int64_t K, int BN, bool gated) {
  const int64_t CL = gemm_cluster(BN);
  const int64_t uc = gated ? BN / 2 : BN;
  const int64_t num_mu = (M + kBM * CL - 1) / (kBM * CL), num_n = (N + uc - 1) / uc;
  const int64_t a_unit = kBM * CL * K * 2, b_unit = (int64_t)BN * K * 2;  // bytes per unit panel
  const int64_t budget = (int64_t)40 << 20;
  if (num_mu > 8 && num_mu * a_unit <= budget) return (int)num_mu;
  if (num_n <= 16 && num_n * b_unit <= budget && num_mu > 8) return -(int)num_n;
  return 8;
}

// C[r, c] += sum over s of ws[s][r, c], s in order: the partial sums of the
// K ranges after the first, so the result does not depend on timing.
__global__ void splitk_sum_kernel(float* __restrict__ C, int64_t ldc, const float* __restrict__ ws,
                                  int64_t stride, int64_t M, int64_t N, int parts) {
  const int64_t n4 = N / 4;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < M * n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / n4, c = (i - r * n4) * 4;
    float4 v = *reinterpret_cast<const float4*>(C + r * ldc + c);
    for (int s = 0; s < parts; ++s) {
      const float4 w = *reinterpret_cast<const float4*>(ws + s * stride + r * ldc + c);
      v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
    }
    *reinterpret_cast<float4*>(C + r * ldc + c) = v;
  }
}

// Number of K ranges for a plain fp32 GEMM: the one of 1..max whose work
// units fill the waves of pairs (or CTAs) best, each range keeping at least
// 16 k-blocks; ties go to fewer ranges.
static int choose_splitk(int64_t M, int64_t N, int64_t K, int BN, int max_split) {
  const int64_t CL = gemm_cluster(BN);
  const int64_t mn = ((M + kBM * CL - 1) / (kBM * CL)) * ((N + BN - 1) / BN);
  const int64_t slots = std::max<int64_t>(1, num_sms() / CL);
  const int64_t nk = (K + kBK - 1) / kBK;
  int best = 1;
  double best_eff = 0;
  for (int s = 1; s <= max_split; ++s) {
    const int64_t kps = (nk + s - 1) / s;
    if (s > 1 && (kps < 16 || (s - 1) * kps >= nk)) break;
    const int64_t units = mn * s;
    const double eff = (double)units / (double)(((units + slots - 1) / slots) * slots);
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

int gemm(const GemmArgs& a, int* dev_err, cudaStream_t st, char* why) {
  if (a.M == 0 || a.N == 0) return 0;
  if (int c = gemm_check(a, why)) return c;
  const bool a_mn = (a.layout == kTN);
  const bool b_mn = (a.layout == kNN || a.layout == kTN);
  const bool gated = (a.epi == kEpiGLU);
  const int BN = (gated || a.N > 128) ? 256 : 128;
  CUtensorMap ta, tb, tb2;
  bool ok = a_mn ? make_map(&ta, a.A, a.M, a.K, a.lda, 64, 64)
                 : make_map(&ta, a.A, a.K, a.M, a.lda, 64, kBM);
  // with clusters each CTA loads half of a K-major B tile; the gated tile's
  // halves are the gate rows [0, N) and the up rows [N, 2N) of B
  ok = ok && (b_mn ? make_map(&tb, a.B, a.N, a.K, a.ldb, 64, 64)
                   : make_map(&tb, a.B, a.K, a.N, a.ldb, 64, BN / gemm_cluster(BN)));
  if (gated)
    ok = ok && make_map(&tb2, static_cast<const __nv_bfloat16*>(a.B) + a.N * a.ldb, a.K, a.N,
                        a.ldb, 64, BN / gemm_cluster(BN));
  else
    tb2 = tb;
  if (!ok) {
    snprintf(why, 64, "gemm: tensor map encode failed");
    return -3;
  }
  const bool can_split = a.epi == kEpiF32 && a.ws != nullptr && a.splitk_max > 1 && a.N % 4 == 0 &&
                         a.ldc % 4 == 0 && (reinterpret_cast<uintptr_t>(a.C) & 15) == 0 &&
                         (reinterpret_cast<uintptr_t>(a.ws) & 15) == 0;
  const int splitk = can_split ? choose_splitk(a.M, a.N, a.K, BN, a.splitk_max) : 1;
  GemmParams p{(int)a.M, (int)a.N, (int)a.K, a.C, a.ldc, a.R, a.ldr, a.alpha, dev_err,
               reinterpret_cast<const __nv_bfloat16*>(a.bias), a.cs, a.seq, a.rope_cols, a.hd,
               a.aux, a.ldaux, unit_order(a.M, a.N, a.K, BN, gated), splitk, a.ws, a.M * a.ldc};
  int rc;
  if (BN == 256) {
    if (a.layout == kNT) rc = launch_epi<false, false, 256>(a.epi, ta, tb, tb2, p, st, why);
    else if (a.layout == kNN) rc = launch_epi<false, true, 256>(a.epi, ta, tb, tb2, p, st, why);
    else rc = launch_epi<true, true, 256>(a.epi, ta, tb, tb2, p, st, why);
  } else if (a.layout == kNT) {
    rc = launch_epi<false, false, 128>(a.epi, ta, tb, tb2, p, st, why);
  } else if (a.layout == kNN) {
    rc = launch_epi<false, true, 128>(a.epi, ta, tb, tb2, p, st, why);
  } else {
    rc = launch_epi<true, true, 128>(a.epi, ta, tb, tb2, p, st, why);
  }
  if (rc == 0 && a.launched) *a.launched += 1;
  if (rc == 0 && splitk > 1) {
    const int64_t n = a.M * (a.N / 4);
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, (int64_t)num_sms() * 8);
    splitk_sum_kernel<<<blocks, 256, 0, st>>>(static_cast<float*>(a.C), a.ldc, a.ws, a.M * a.ldc, a.M,
                                              a.N, splitk - 1);
    if (cudaGetLastError() != cudaSuccess) {
      snprintf(why, 64, "gemm: split-K sum launch failed");
      return -3;
    }
    if (a.launched) *a.launched += 1;
  }
  return rc;
}

}  // namespace sf
