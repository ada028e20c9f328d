// Causal grouped-query attention, forward and backward, on the tcgen05
// tensor cores.
//
// Forward: online softmax over key blocks (Milakov & Gimelshein 2018; the
// blocking of Dao et al., FlashAttention 2022), laid out for sm_103a.  The
// kernel is persistent: one CTA per SM walks items of two 128-query tiles in
// longest-first order.  Both tiles of an item read the same K and V blocks,
// and they take turns on the tensor core: while one tile's softmax warps turn
// S into P, the tensor core runs the other tile's O += P V and next S = Q K^T.
// Four softmax warps per tile give one thread per query row, so the row max
// and row sum need no shuffles.  P goes back into TMEM over its S columns, as
// the tensor-memory A operand of P V.
//
// Two measurements on GB300 set the shape of the softmax code.
//   - One thread issues every MMA, and each 128 x 128 x 16 MMA runs only
//     about 64 cycles.
//   - Scalar fp32 max instructions in the softmax warps slow that issuing
//     warp more than twice over.
// So the row max uses three-input maxima, the exponent arguments and row
// sums use paired fp32 instructions, and the causal mask is compiled only
// into the diagonal block's code.
//
// Operands: Q and K tiles are K-major [128 rows][hd] (128-byte swizzle, 64
// columns per box); V is the MN-major operand of P V ([128 keys][64 hd]
// boxes).  The qkv rows are read through a 3-D tensor map (column, position,
// batch), so rows past the sequence end arrive as zeros.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include "ptx.cuh"
#include "sf_internal.h"

namespace sf {

namespace {

constexpr int kAttThreads = 192;
// Grid position in longest-first order: the CTAs are dispatched roughly in
// linear block order, so every CTA of rank 0 (the most work) is placed before
// any CTA of rank 1, and so on, whatever the other two coordinates.
__device__ __forceinline__ void grid_rank_first(int& rank, int& y, int& z) {
  const int lin = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  const int per = (int)(gridDim.y * gridDim.z);
  rank = lin / per;
  const int rem = lin - rank * per;
  y = rem % (int)gridDim.y;
  z = rem / (int)gridDim.y;
}

// 2^x on the special-function unit (relative error ~2^-22, flushes denormals).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// (x, y) * c + (d, d) as one paired fp32 FMA (round to nearest)
__device__ __forceinline__ void fma2_scalar(float& x, float& y, float c, float d) {
  asm("{\n\t.reg .b64 t, u, w;\n\t"
      "mov.b64 t, {%0, %1};\n\t"
      "mov.b64 u, {%2, %2};\n\t"
      "mov.b64 w, {%3, %3};\n\t"
      "fma.rn.f32x2 t, t, u, w;\n\t"
      "mov.b64 {%0, %1}, t;\n\t}"
      : "+f"(x), "+f"(y)
      : "f"(c), "f"(d));
}

// (x, y) * c + (d0, d1) as one paired fp32 FMA (round to nearest)
__device__ __forceinline__ void fma2(float& x, float& y, float c, float d0, float d1) {
  asm("{\n\t.reg .b64 t, u, w;\n\t"
      "mov.b64 t, {%0, %1};\n\t"
      "mov.b64 u, {%2, %2};\n\t"
      "mov.b64 w, {%3, %4};\n\t"
      "fma.rn.f32x2 t, t, u, w;\n\t"
      "mov.b64 {%0, %1}, t;\n\t}"
      : "+f"(x), "+f"(y)
      : "f"(c), "f"(d0), "f"(d1));
}

// (x, y) *= (a, b) as one paired fp32 multiply
__device__ __forceinline__ void mul2(float& x, float& y, float a, float b) {
  asm("{\n\t.reg .b64 t, u;\n\t"
      "mov.b64 t, {%0, %1};\n\t"
      "mov.b64 u, {%2, %3};\n\t"
      "mul.rn.f32x2 t, t, u;\n\t"
      "mov.b64 {%0, %1}, t;\n\t}"
      : "+f"(x), "+f"(y)
      : "f"(a), "f"(b));
}

// (x, y) += (a, b) as one paired fp32 add
__device__ __forceinline__ void add2(float& x, float& y, float a, float b) {
  asm("{\n\t.reg .b64 t, u;\n\t"
      "mov.b64 t, {%0, %1};\n\t"
      "mov.b64 u, {%2, %3};\n\t"
      "add.rn.f32x2 t, t, u;\n\t"
      "mov.b64 {%0, %1}, t;\n\t}"
      : "+f"(x), "+f"(y)
      : "f"(a), "f"(b));
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace

// ------------------------------------------------------------------ forward, two query tiles per CTA
// The same online softmax with two 128-query tiles per CTA that share every
// K and V tile: two query heads of one kv group at the same query block when
// the group size is even, else query blocks 2p and 2p + 1 of one head (block
// 2p + 1 is then fully masked for the first tile).  Sharing halves the K/V
// bytes each tensor-core FLOP pulls from L2, and the two tiles ping-pong: the
// tensor core runs one tile's P V and next Q K^T while the other tile's
// softmax warps work, so each tile's TMEM holds one S (P written over it as
// bf16) and one O.
//
//   warp 0      TMA: one ring of K/V entries (2 at head dim 128, 4 at 64;
//               entry G + 1 carries V(G) and K(G + 1), what the MMA step of
//               block G reads), both Q tiles at an item's first block
//   warp 1      MMA issuer; TMEM owner (S0 | S1 | O0 | O1)
//   warp 2      TMA store of each staged O tile
//   warps 3-6   softmax of tile 0, one thread per query row
//   warps 7-10  softmax of tile 1
//
// Per block G the MMA thread waits once for its K/V entry, issues O0 += P0
// V, S0' = Q0 K'^T, O1 += P1 V, S1' = Q1 K'^T, and releases the entry once.
// S' overwrites the columns that held P: the tensor core
// executes one thread's MMAs in issue order, so P is read before it is
// overwritten.  A commit after S' also covers every earlier P V of the CTA,
// so once a softmax thread sees S' it may rescale its O row: no P V of its
// tile is in flight until it publishes the next P.
namespace {
constexpr int kAttFwd2Threads = 352;

template <int HD>
struct AttFwd2Cfg {
  static constexpr int TILE = HD / 64 * 16384;  // 128 rows x HD bf16
  static constexpr int NE = HD == 128 ? 2 : 4;  // stages of the K/V ring (K and V tiles each)
  static constexpr int OFF_Q = 0;  // Q of tile 0, then of tile 1
  static constexpr int OFF_K = 2 * TILE;
  static constexpr int OFF_V = OFF_K + NE * TILE;
  static constexpr int OFF_O = OFF_V + NE * TILE;  // staging of an O tile for its TMA store
  static constexpr int OFF_BAR = OFF_O + TILE;
  static constexpr int NBAR = 13 + 2 * NE;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
};
static_assert(AttFwd2Cfg<128>::SMEM <= 232448, "forward shared memory");
}  // namespace

template <int HD>
__global__ void __launch_bounds__(kAttFwd2Threads, 1)
    attn_fwd_pp_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tm_o,
                       float* __restrict__ lse, int S, int Hq, int Hkv, int B, float scale_log2,
                       int pair_heads, int* err) {
  using C = AttFwd2Cfg<HD>;
  constexpr int NB = HD / 64;  // 64-column boxes per tile
  constexpr uint32_t ID_S = umma_idesc_bf16(128, 128, false, false);
  constexpr uint32_t ID_O = umma_idesc_bf16(128, HD, false, true);
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t O_COL = 256;  // O of tile t at O_COL + t * HD; S (and P) of tile t at t * 128

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sQ = s0 + C::OFF_Q, sK = s0 + C::OFF_K, sV = s0 + C::OFF_V, sO = s0 + C::OFF_O;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const uint32_t b0 = smem_u32(bars);
  auto q_full = [&](int t) { return b0 + 8u * t; };
  auto q_empty = [&](int t) { return b0 + 8u * (2 + t); };
  auto s_full = [&](int t) { return b0 + 8u * (4 + t); };
  auto p_full = [&](int t) { return b0 + 8u * (6 + t); };
  auto o_done = [&](int t) { return b0 + 8u * (8 + t); };
  const uint32_t st_ready = b0 + 8u * 10;  // an O tile's rows are in the staging buffer
  const uint32_t st_free = b0 + 8u * 11;   // the staging buffer has been read by the TMA store
  const uint32_t drain = b0 + 8u * 12;
  // Entry e of the K/V ring holds K(e) in K stage e % NE and V(e - 1) in V
  // stage (e - 1) % NE, G counting key blocks over all items of the CTA: the
  // MMA step of block G reads V(G) and K(G + 1), i.e. entry G + 1, and frees
  // it at the step's end.
  auto kv_full = [&](int s) { return b0 + 8u * (13 + s); };
  auto kv_empty = [&](int s) { return b0 + 8u * (13 + C::NE + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = (S + 127) / 128;
  const int grp = Hq / Hkv;
  // Items in longest-first order (every item of the most keys comes first);
  // CTA c takes items c, c + gridDim.x, ...
  const int npb = pair_heads ? nqb : (nqb + 1) / 2;  // query positions of an item
  const int per_rank = pair_heads ? (Hq / 2) * B : Hq * B;
  const int num_items = npb * per_rank;
  struct Item { int h0, h1, qb0, qb1, b, g, nkv; };
  auto item_of = [&](int t) -> Item {
    const int rank = t / per_rank, rem = t - rank * per_rank;
    Item x;
    if (pair_heads) {
      const int hp = rem % (Hq / 2);
      x.b = rem / (Hq / 2);
      x.h0 = 2 * hp;
      x.h1 = 2 * hp + 1;
      x.qb0 = x.qb1 = nqb - 1 - rank;
    } else {
      x.h0 = x.h1 = rem % Hq;
      x.b = rem / Hq;
      x.qb0 = 2 * (npb - 1 - rank);
      x.qb1 = x.qb0 + 1;
    }
    x.g = x.h0 / grp;
    x.nkv = x.qb1 + 1 < nqb ? x.qb1 + 1 : nqb;
    return x;
  };

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(q_full(t), 1);
      mbar_init(q_empty(t), 1);
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), 128);
      mbar_init(o_done(t), 1);
    }
    for (int s = 0; s < C::NE; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    mbar_init(st_ready, 128);
    mbar_init(st_free, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm);
    tma_prefetch_desc(&tm_o);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    // Entries in order: entry e carries K(e) and V(e - 1); both Q tiles of an
    // item follow the entry with the item's first K (each once the previous
    // item's last S of that tile has read the buffer); a last entry carries
    // the last V alone.
    bool ok = true;
    long e = 0;  // entries issued
    int it = 0, q_issued[2] = {-1, -1};
    int pv_col = 0, pv_row = 0, pv_b = 0;  // where the previous block's V comes from
    auto entry = [&](bool with_k, int colK, int krow, int kb) -> bool {
      const int st = (int)(e % C::NE);
      if (!mbar_wait(kv_empty(st), (uint32_t)((e / C::NE) & 1) ^ 1u, abort_flag)) return false;
      mbar_arrive_expect_tx(kv_full(st), (uint32_t)((with_k ? C::TILE : 0) + (e > 0 ? C::TILE : 0)));
      if (with_k) {
#pragma unroll
        for (int c = 0; c < NB; ++c)
          tma_load_3d(sK + st * C::TILE + c * 16384, &tm, kv_full(st), colK + 64 * c, krow, kb);
      }
      if (e > 0) {
        const int vs = (int)((e - 1) % C::NE);
#pragma unroll
        for (int c = 0; c < NB; ++c)
          tma_load_3d(sV + vs * C::TILE + c * 16384, &tm, kv_full(st), pv_col + 64 * c, pv_row, pv_b);
      }
      ++e;
      return true;
    };
    for (int t = blockIdx.x; ok && t < num_items; t += gridDim.x, ++it) {
      const Item x = item_of(t);
      const int colK = (Hq + x.g) * HD, colV = (Hq + Hkv + x.g) * HD;
      for (int j = 0; j < x.nkv; ++j) {
        if (!entry(true, colK, j * 128, x.b)) { ok = false; break; }
        pv_col = colV;
        pv_row = j * 128;
        pv_b = x.b;
        if (j == 0) {
          for (int tt = 0; tt < 2; ++tt) {
            if (it > 0 && !mbar_wait(q_empty(tt), (uint32_t)((it - 1) & 1), abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(q_full(tt), C::TILE);
            const int h = tt ? x.h1 : x.h0, qb = tt ? x.qb1 : x.qb0;
#pragma unroll
            for (int c = 0; c < NB; ++c)
              tma_load_3d(sQ + tt * C::TILE + c * 16384, &tm, q_full(tt), h * HD + 64 * c, qb * 128, x.b);
            q_issued[tt] = it;
          }
          if (!ok) break;
        }
      }
    }
    if (ok && e > 0 && !entry(false, 0, 0, 0)) ok = false;  // the last V
    if (!ok) {
      record_error(err, kDevAttnTimeout);
      *abort_flag = 1;
      // let the copies already issued land before the CTA's shared memory goes away
      for (int tt = 0; tt < 2; ++tt)
        if (q_issued[tt] >= 0) mbar_wait(q_full(tt), (uint32_t)(q_issued[tt] & 1), nullptr);
      for (long k = e - 1; k >= 0 && k >= e - C::NE; --k)
        mbar_wait(kv_full((int)(k % C::NE)), (uint32_t)((k / C::NE) & 1), nullptr);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    bool ok = true;
    // Descriptors of the buffers' first rows; an operand at byte offset o
    // within a buffer is the base descriptor plus o / 16 (the address field
    // cannot carry: shared addresses stay below 2^18).
    const uint64_t dQ = smem_desc_sw128(sQ, 16, 1024), dK = smem_desc_sw128(sK, 16, 1024);
    const uint64_t dV = smem_desc_sw128(sV, 16384, 1024);
    // S_t = Q_t K(G)^T into the S columns of tile t
    auto issue_s = [&](int tt, long G) {
      const uint32_t ks = (uint32_t)(G % C::NE);
      const uint64_t a0 = dQ + (uint32_t)(tt * C::TILE / 16), b0 = dK + ks * (uint32_t)(C::TILE / 16);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) / 16;
        umma_bf16(tmem_base + tt * 128, a0 + off, b0 + off, ID_S, kk > 0 ? 1u : 0u);
      }
      umma_commit(s_full(tt));
    };
    long G = 0;  // global index of the current key block over the CTA's items
    int it = 0;
    int t = blockIdx.x;
    if (t < num_items) {  // the first item's S of both tiles
      const Item x = item_of(t);
      for (int tt = 0; ok && tt < 2; ++tt) {
        if ((tt == 0 && !mbar_wait(kv_full(0), 0, abort_flag)) || !mbar_wait(q_full(tt), 0, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(tt, 0);
        if (x.nkv == 1) umma_commit(q_empty(tt));
      }
      if (ok) umma_commit(kv_empty(0));  // entry 0: K(0) alone
    }
    for (; ok && t < num_items; t += gridDim.x, ++it) {
      const Item x = item_of(t);
      const bool has_next_item = t + (int)gridDim.x < num_items;
      const int nkv_next = has_next_item ? item_of(t + gridDim.x).nkv : 0;
      for (int j = 0; ok && j < x.nkv; ++j, ++G) {
        const bool last = j + 1 == x.nkv;
        const bool has_next = !last || has_next_item;
        const long Gn = G + 1;
        // the next block's S: the last of its item releases that item's Q tile
        const bool next_is_last = last ? nkv_next == 1 : j + 2 == x.nkv;
        const int vs = (int)(G % C::NE);
        const int es = (int)(Gn % C::NE);  // entry G + 1: V(G) and K(G + 1)
        if (!mbar_wait(kv_full(es), (uint32_t)((Gn / C::NE) & 1), abort_flag)) {
          ok = false;
          break;
        }
        for (int tt = 0; tt < 2; ++tt) {
          if (!mbar_wait(p_full(tt), (uint32_t)(G & 1), abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bv = dV + (uint32_t)vs * (uint32_t)(C::TILE / 16);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // O_t += P_t V: P as the tensor-memory A operand
            umma_bf16_ts(tmem_base + O_COL + tt * HD, tmem_base + tt * 128 + kk * 8, bv + kk * (2048 / 16),
                         ID_O, (j > 0 || kk > 0) ? 1u : 0u);
          if (last) umma_commit(o_done(tt));
          if (has_next) {
            if (last && !mbar_wait(q_full(tt), (uint32_t)((it + 1) & 1), abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(tt, Gn);
            if (next_is_last) umma_commit(q_empty(tt));
          }
        }
        if (!ok) break;
        umma_commit(kv_empty(es));  // V(G) and K(G + 1) have been read
      }
    }
    if (!ok) {
      record_error(err, kDevAttnTimeout);
      *abort_flag = 1;
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp == 2 && lane == 0) {
    // ---------------------------------------------------------------- O store
    bool ok = true;
    int c = 0;  // O tiles stored so far: tile 0 then tile 1 of each item
    for (int t = blockIdx.x; ok && t < num_items; t += gridDim.x) {
      const Item x = item_of(t);
      for (int tt = 0; tt < 2; ++tt, ++c) {
        if (!mbar_wait(st_ready, (uint32_t)(c & 1), abort_flag)) { ok = false; break; }
        const int h = tt ? x.h1 : x.h0, qb = tt ? x.qb1 : x.qb0;
        if (qb * 128 < S) {  // rows past the sequence end are outside the tensor map and not written
#pragma unroll
          for (int cc = 0; cc < NB; ++cc) tma_store_3d(&tm_o, sO + cc * 16384, h * HD + 64 * cc, qb * 128, x.b);
          bulk_commit_group();
          bulk_wait_group_read0();
        }
        mbar_arrive(st_free);
      }
    }
    bulk_wait_group0();
    if (!ok) {
      record_error(err, kDevAttnTimeout);
      *abort_flag = 1;
    }
  } else if (warp >= 3) {
    // ---------------------------------------------------------------- softmax
    const int tt = (warp - 3) >> 2;
    const int quarter = warp & 3;  // TMEM lanes a warp may access: 32 x (warp % 4)
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_col = (uint32_t)tt * 128u, o_col = O_COL + (uint32_t)tt * HD;
    bool ok = true;
    long G = 0;
    int it = 0;
    for (int t = blockIdx.x; ok && t < num_items; t += gridDim.x, ++it) {
      const Item x = item_of(t);
      const int qb = tt ? x.qb1 : x.qb0, h = tt ? x.h1 : x.h0;
      const int q = qb * 128 + row;
      // m: the row max in log2 units that the exponentials are taken against;
      // it only moves when a block's max exceeds it by more than 8, so O in
      // TMEM is rarely rescaled (O / l does not depend on the choice of m).
      float m = -INFINITY, l = 0.f;
      // One key block: S from TMEM, P back over it.  Compiled twice, with the
      // causal mask (the diagonal block and any block past it) and without.
      auto block = [&](int j, long G, auto diag) -> bool {
        constexpr bool DIAG = decltype(diag)::value;
        if (!__all_sync(0xffffffffu, mbar_wait(s_full(tt), (uint32_t)(G & 1), abort_flag))) return false;
        tc_fence_after();
        float s[128];
        {
          uint32_t r[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(lane_base + s_col + 32 * c, r[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) s[32 * c + i] = __uint_as_float(r[c][i]);
        }
        if (DIAG) {  // keys after the query are masked (every key of a block past the diagonal)
          const int lim = q - j * 128;
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i > lim) s[i] = -INFINITY;
        }
        // row max: eight chains of three-input maxima over columns 16..127
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = fmaxf(s[a], s[a + 8]);
#pragma unroll
        for (int i = 16; i < 128; i += 16)
#pragma unroll
          for (int a = 0; a < 8; ++a) mx8[a] = max3f(mx8[a], s[i + a], s[i + 8 + a]);
        float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        mx *= scale_log2;  // the scale is positive: the max commutes with it
        const bool grow = mx > m + 8.f;
        const float m_new = grow ? mx : m;
        const float corr = ex2_approx(m - m_new);  // 1 without growth, 0 on the first block
        // p = 2^(s * scale - m): the arguments and the partial row sums as
        // paired fp32 operations, the exponentials on the special-function unit
        float ps8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 128; i += 2) {
          fma2_scalar(s[i], s[i + 1], scale_log2, -m_new);
          s[i] = ex2_approx(s[i]);
          s[i + 1] = ex2_approx(s[i + 1]);
          add2(ps8[i & 7], ps8[(i & 7) + 1], s[i], s[i + 1]);
        }
        const float ps = ((ps8[0] + ps8[1]) + (ps8[2] + ps8[3])) + ((ps8[4] + ps8[5]) + (ps8[6] + ps8[7]));
        l = l * corr + ps;
        m = m_new;
        // the row of P, bf16 pairs, over the first 64 columns of S
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack2_bf16(s[64 * hh + 2 * i], s[64 * hh + 2 * i + 1]);
          tmem_st_32x32b_x32(lane_base + s_col + 32 * hh, pk);
        }
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          // every P V of this tile so far has completed (the S commit covers
          // them), and the next waits for this thread's P arrival below
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(lane_base + o_col + 32 * c, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
            tmem_st_32x32b_x32(lane_base + o_col + 32 * c, r);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full(tt));
        return true;
      };
      for (int j = 0; j < x.nkv; ++j, ++G) {
        ok = j >= qb ? block(j, G, std::true_type{}) : block(j, G, std::false_type{});
        if (!ok) break;
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(o_done(tt), (uint32_t)(it & 1), abort_flag));
      // the staging buffer is free once the previous O tile's store has read it
      const int c = 2 * it + tt;
      if (ok && c > 0) ok = __all_sync(0xffffffffu, mbar_wait(st_free, (uint32_t)((c - 1) & 1), abort_flag));
      if (!ok) break;
      tc_fence_after();
      const float inv = 1.f / l;
      // the O row, bf16, into the staging buffer in the tensor map's swizzled
      // layout: box c / 2 holds columns [64 (c / 2), 64 (c / 2) + 64)
      const uint32_t orow = sO + (uint32_t)row * 128u;
#pragma unroll
      for (int cc = 0; cc < HD / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(lane_base + o_col + 32 * cc, r);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int chunk = (cc & 1) * 4 + k;  // 16-byte chunk within the 128-byte row
          const uint32_t addr = orow + (cc >> 1) * 16384 + (uint32_t)((chunk ^ (row & 7)) * 16);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                       "r"(pack2_bf16(__uint_as_float(r[8 * k + 0]) * inv, __uint_as_float(r[8 * k + 1]) * inv)),
                       "r"(pack2_bf16(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv)),
                       "r"(pack2_bf16(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv)),
                       "r"(pack2_bf16(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv))
                       : "memory");
        }
      }
      // O has left TMEM: the next item's first P V of this tile (issued after
      // this thread's next P arrival) may overwrite it
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(st_ready);
      if (q < S) lse[((int64_t)x.b * Hq + h) * S + q] = (m + log2f(l)) * 0.69314718055994531f;
    }
    if (!ok && lane == 0) {
      record_error(err, kDevAttnTimeout);
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ backward
// One CTA per (128-key block j, kv head g, batch b).  It walks every query
// head of the group and every 128-query block i >= j.  Per (head, block):
//   MMA:     S^T = K Q^T -> TMEM[0,128),  dP^T = V dO^T -> TMEM[128,256)
//   threads: one per key row: P^T = exp2(S^T*scale*log2e - lse*log2e) (causal),
//            dS^T = P^T * (dP^T - D), both to shared memory (bf16, swizzled)
//   MMA:     dV += P^T dO, dK += dS^T Q (TMEM, kept over the whole walk);
//            dQ = dS K -> TMEM[0,hd) (the S^T columns, already consumed)
//   threads: one per query row: dQ added into the fp32 dq_acc (vector atomics)
// dS^T is stored once and read both as the K-major A of dK and as the
// MN-major A (dS) of dQ.  At the end the threads write dK (scaled, inverse
// RoPE) and dV of their key rows.
namespace {
template <int HD>
struct AttBwdCfg {
  static constexpr int TILE = HD / 64 * 16384;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE;
  static constexpr int OFF_Q = 2 * TILE;
  static constexpr int OFF_DO = 3 * TILE;
  static constexpr int OFF_PT = 4 * TILE;
  static constexpr int OFF_DST = OFF_PT + 32768;
  static constexpr int OFF_LD = OFF_DST + 32768;  // lse*log2e and D, 2 buffers x 128 each
  static constexpr int OFF_BAR = OFF_LD + 4 * 128 * 4;
  static constexpr int NBAR = 11;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
};
}  // namespace

template <int HD, bool DET>
__global__ void __launch_bounds__(kAttThreads, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                       const __grid_constant__ CUtensorMap tm_do, const float* __restrict__ lse,
                       const float* __restrict__ delta, float* __restrict__ dq_acc,
                       __nv_bfloat16* __restrict__ dqkv, const float2* __restrict__ cs, int S,
                       int Hq, int Hkv, float scale, float scale_log2, int* err) {
  using C = AttBwdCfg<HD>;
  constexpr int NB = HD / 64;
  constexpr uint32_t ID_SQ = umma_idesc_bf16(128, 128, false, false);  // S^T, dP^T
  constexpr uint32_t ID_KV = umma_idesc_bf16(128, HD, false, true);    // dV, dK
  constexpr uint32_t ID_Q = umma_idesc_bf16(128, HD, true, true);      // dQ
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t COL_DP = 128, COL_DV = 256, COL_DK = 256 + HD;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + C::OFF_K, sV = s0 + C::OFF_V, sQ = s0 + C::OFF_Q, sDO = s0 + C::OFF_DO;
  const uint32_t sPt = s0 + C::OFF_PT, sDSt = s0 + C::OFF_DST;
  float* sLD = reinterpret_cast<float*>(smem + C::OFF_LD);  // [2][lse 128 | D 128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const uint32_t b0 = smem_u32(bars);
  const uint32_t kv_full = b0, qdo_full = b0 + 8, qdo_empty = b0 + 16, sp_full = b0 + 24,
                 ps_full = b0 + 32, dq_full = b0 + 40, dq_free = b0 + 48, acc_done = b0 + 56,
                 drain = b0 + 64;
  auto ld_full = [&](int i) { return b0 + 72u + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int j, g, b;
  grid_rank_first(j, g, b);  // key block 0 sees the most query blocks
  const int grp = Hq / Hkv;
  const int k0 = j * 128;
  const int nqb = (S + 127) / 128;
  const int n_it = grp * (nqb - j);  // (head, query block) pairs

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(qdo_full, 1);
    mbar_init(qdo_empty, 1);
    mbar_init(sp_full, 1);
    mbar_init(ps_full, 128);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 128);
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    mbar_init(ld_full(0), 128);
    mbar_init(ld_full(1), 128);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    mbar_arrive_expect_tx(kv_full, 2 * C::TILE);
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      tma_load_3d(sK + c * 16384, &tm_qkv, kv_full, (Hq + g) * HD + 64 * c, k0, b);
      tma_load_3d(sV + c * 16384, &tm_qkv, kv_full, (Hq + Hkv + g) * HD + 64 * c, k0, b);
    }
    bool ok = true;
    int issued = 0;
    for (int it = 0; it < n_it; ++it) {
      const int h = g * grp + it / (nqb - j);
      const int q0 = (j + it % (nqb - j)) * 128;
      if (!mbar_wait(qdo_empty, (it & 1) ^ 1, abort_flag)) { ok = false; break; }
      mbar_arrive_expect_tx(qdo_full, 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < NB; ++c) {
        tma_load_3d(sQ + c * 16384, &tm_qkv, qdo_full, h * HD + 64 * c, q0, b);
        tma_load_3d(sDO + c * 16384, &tm_do, qdo_full, h * HD + 64 * c, q0, b);
      }
      issued = it + 1;
    }
    if (!ok) {
      record_error(err, kDevAttnTimeout);
      *abort_flag = 1;
      mbar_wait(kv_full, 0, nullptr);
      if (issued > 0) mbar_wait(qdo_full, (issued - 1) & 1, nullptr);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    bool ok = mbar_wait(kv_full, 0, abort_flag);
    for (int it = 0; ok && it < n_it; ++it) {
      const uint32_t ph = it & 1;
      if (!mbar_wait(qdo_full, ph, abort_flag) || !mbar_wait(dq_free, ph ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        umma_bf16(tmem_base, smem_desc_sw128(sK + off, 16, 1024), smem_desc_sw128(sQ + off, 16, 1024),
                  ID_SQ, kk > 0 ? 1u : 0u);
        umma_bf16(tmem_base + COL_DP, smem_desc_sw128(sV + off, 16, 1024),
                  smem_desc_sw128(sDO + off, 16, 1024), ID_SQ, kk > 0 ? 1u : 0u);
      }
      umma_commit(sp_full);
      if (!mbar_wait(ps_full, ph, abort_flag)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {  // contraction over the 128 queries
        const uint32_t a_off = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
        umma_bf16(tmem_base + COL_DV, smem_desc_sw128(sPt + a_off, 16, 1024),
                  smem_desc_sw128(sDO + kk * 2048, 16384, 1024), ID_KV, acc);
        umma_bf16(tmem_base + COL_DK, smem_desc_sw128(sDSt + a_off, 16, 1024),
                  smem_desc_sw128(sQ + kk * 2048, 16384, 1024), ID_KV, acc);
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // contraction over the 128 keys
        umma_bf16(tmem_base, smem_desc_sw128(sDSt + kk * 2048, 16384, 1024),
                  smem_desc_sw128(sK + kk * 2048, 16384, 1024), ID_Q, kk > 0 ? 1u : 0u);
      umma_commit(dq_full);
      umma_commit(qdo_empty);
    }
    if (ok) {
      umma_commit(acc_done);
    } else {
      record_error(err, kDevAttnTimeout);
      *abort_flag = 1;
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- softmax-gradient threads
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row for S^T / dP^T, query row for dQ
    const int key = k0 + r;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const int tid = threadIdx.x - 64;  // 0..127
    const int64_t ldo = (int64_t)Hq * HD;
    bool ok = true;
    // lse (log2 units) and D of the query block, one value per thread, loaded
    // one block ahead so the global latency is off the critical path
    auto fetch = [&](int it_, float& lv, float& dv) {
      lv = 0.f;
      dv = 0.f;
      if (it_ >= n_it) return;
      const int h_ = g * grp + it_ / (nqb - j);
      const int q_ = (j + it_ % (nqb - j)) * 128 + tid;
      if (q_ < S) {
        const int64_t o = ((int64_t)b * Hq + h_) * S + q_;
        lv = lse[o] * 1.4426950408889634f;
        dv = delta[o];
      }
    };
    float next_l, next_d;
    fetch(0, next_l, next_d);
    for (int it = 0; it < n_it; ++it) {
      const int h = g * grp + it / (nqb - j);
      const int q0 = (j + it % (nqb - j)) * 128;
      const uint32_t ph = it & 1;
      float* bL = sLD + (it & 1) * 256;
      float* bD = bL + 128;
      // The buffer written here was last read for block it - 2, and every
      // thread finished that before the MMA warp could issue block it - 1,
      // whose S^T this thread has already waited for.
      bL[tid] = next_l;
      bD[tid] = next_d;
      mbar_arrive(ld_full(it & 1));
      fetch(it + 1, next_l, next_d);
      ok = __all_sync(0xffffffffu, mbar_wait(ld_full(it & 1), (it >> 1) & 1, abort_flag));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(sp_full, ph, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t rowoff = (uint32_t)r * 128u;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t sr[32], dr[32];
        tmem_ld_32x32b_x32(lane_base + 32 * c, sr);
        tmem_ld_32x32b_x32(lane_base + COL_DP + 32 * c, dr);
        tmem_ld_wait();
        float p[32], ds[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int qq = 32 * c + e;
          const int q = q0 + qq;
          float pv = 0.f;
          if (q < S && key <= q) pv = ex2_approx(fmaf(__uint_as_float(sr[e]), scale_log2, -bL[qq]));
          p[e] = pv;
          ds[e] = pv * (__uint_as_float(dr[e]) - bD[qq]);
        }
        const uint32_t box = (uint32_t)(c >> 1) * 16384u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int jj = (c & 1) * 4 + k;
          const uint32_t off = box + rowoff + (uint32_t)((jj ^ (r & 7)) * 16);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sPt + off),
                       "r"(pack2_bf16(p[8 * k], p[8 * k + 1])), "r"(pack2_bf16(p[8 * k + 2], p[8 * k + 3])),
                       "r"(pack2_bf16(p[8 * k + 4], p[8 * k + 5])), "r"(pack2_bf16(p[8 * k + 6], p[8 * k + 7]))
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sDSt + off),
                       "r"(pack2_bf16(ds[8 * k], ds[8 * k + 1])), "r"(pack2_bf16(ds[8 * k + 2], ds[8 * k + 3])),
                       "r"(pack2_bf16(ds[8 * k + 4], ds[8 * k + 5])), "r"(pack2_bf16(ds[8 * k + 6], ds[8 * k + 7]))
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ps_full);
      // dQ rows of this query block (thread = query row)
      ok = __all_sync(0xffffffffu, mbar_wait(dq_full, ph, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const int q = q0 + r;
      // deterministic: this key block's own slot, plain stores
      const int64_t row = DET ? ((int64_t)j * gridDim.z + b) * S + q : (int64_t)b * S + q;
      float* dst = dq_acc + row * ldo + (int64_t)h * HD;
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(lane_base + 32 * c, v);
        tmem_ld_wait();
        if (q < S) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 x = make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                         __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
            if (DET)
              *reinterpret_cast<float4*>(dst + 32 * c + 4 * k) = x;
            else
              atomicAdd(reinterpret_cast<float4*>(dst + 32 * c + 4 * k), x);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(dq_free);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag));
    if (ok) {
      tc_fence_after();
      // dK: pairs (d, d + HD/2) get the inverse rotation of the key's position
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t x1[32], x2[32];
        tmem_ld_32x32b_x32(lane_base + COL_DK + 32 * c, x1);
        tmem_ld_32x32b_x32(lane_base + COL_DK + HD / 2 + 32 * c, x2);
        tmem_ld_wait();
        if (key < S) {
          const int64_t ld = (int64_t)(Hq + 2 * Hkv) * HD;
          __nv_bfloat16* krow = dqkv + ((int64_t)b * S + key) * ld + (int64_t)(Hq + g) * HD;
          uint32_t o1[16], o2[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float a1 = __uint_as_float(x1[e]) * scale, b1 = __uint_as_float(x1[e + 1]) * scale;
            float a2 = __uint_as_float(x2[e]) * scale, b2 = __uint_as_float(x2[e + 1]) * scale;
            if (cs) {
              const float2 ca = cs[(int64_t)key * (HD / 2) + 32 * c + e];
              const float2 cb = cs[(int64_t)key * (HD / 2) + 32 * c + e + 1];
              const float y1a = a1 * ca.x + a2 * ca.y, y2a = a2 * ca.x - a1 * ca.y;
              const float y1b = b1 * cb.x + b2 * cb.y, y2b = b2 * cb.x - b1 * cb.y;
              a1 = y1a; a2 = y2a; b1 = y1b; b2 = y2b;
            }
            o1[e / 2] = pack2_bf16(a1, b1);
            o2[e / 2] = pack2_bf16(a2, b2);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            *reinterpret_cast<uint4*>(krow + 32 * c + 8 * k) = make_uint4(o1[4 * k], o1[4 * k + 1], o1[4 * k + 2], o1[4 * k + 3]);
            *reinterpret_cast<uint4*>(krow + HD / 2 + 32 * c + 8 * k) = make_uint4(o2[4 * k], o2[4 * k + 1], o2[4 * k + 2], o2[4 * k + 3]);
          }
        }
      }
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(lane_base + COL_DV + 32 * c, v);
        tmem_ld_wait();
        if (key < S) {
          const int64_t ld = (int64_t)(Hq + 2 * Hkv) * HD;
          __nv_bfloat16* vrow = dqkv + ((int64_t)b * S + key) * ld + (int64_t)(Hq + Hkv + g) * HD;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 u;
            u.x = pack2_bf16(__uint_as_float(v[8 * k + 0]), __uint_as_float(v[8 * k + 1]));
            u.y = pack2_bf16(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3]));
            u.z = pack2_bf16(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5]));
            u.w = pack2_bf16(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7]));
            *reinterpret_cast<uint4*>(vrow + 32 * c + 8 * k) = u;
          }
        }
      }
    } else if (lane == 0) {
      record_error(err, kDevAttnTimeout);
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Backward for head_dim 128 with 64-query blocks.  The Q and dO tiles have
// three stages, so loads run two blocks ahead.  dQ is formed transposed,
// dQ^T = K^T dS^T (M = head_dim = 128), one thread per head-dim lane; each
// warp stages its 32 x 32 piece in shared memory and the TMA unit adds it
// into the fp32 dQ buffer (cp.reduce.async.bulk), so no thread issues atomics;
// in the deterministic variant it stores the piece into this key block's own
// slot instead, and the slots are summed in key order afterwards.  The threads copy S^T and dP^T into
// registers and release those TMEM columns at once, so the MMA warp computes
// the next block's S^T and dP^T, and this block's dV, dK and dQ^T, while
// they work.  TMEM columns: S^T [0,64), dP^T [64,128), dQ^T two buffers
// [128,256), dV [256,384), dK [384,512).  Every mbarrier below completes at
// most once before its waiter has seen the previous completion (each has a
// dependency chain through its waiter), so parity waits are unambiguous.
namespace {
constexpr int kAttBwd2Threads = 320;  // TMA warp, MMA warp, 8 softmax-gradient warps
struct AttBwd2Cfg {
  static constexpr int KV = 32768;  // 128 keys x 128 hd
  static constexpr int QT = 16384;  // 64 queries x 128 hd
  static constexpr int NQ = 3;      // Q / dO stages
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KV;
  static constexpr int OFF_Q = 2 * KV;
  static constexpr int OFF_DO = OFF_Q + NQ * QT;
  static constexpr int OFF_PT = OFF_DO + NQ * QT;  // 128 keys x 64 queries
  static constexpr int OFF_DST = OFF_PT + 16384;
  static constexpr int OFF_DQS = OFF_DST + 16384;  // dQ staging: 8 warps x [32 q][32 d] fp32
  static constexpr int OFF_LD = OFF_DQS + 8 * 4096;  // [2][lse 64 | D 64]
  static constexpr int OFF_BAR = OFF_LD + 2 * 128 * 4;
  static constexpr int NBAR = 19;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16 + 1024;
};
}  // namespace

template <bool DET>
__global__ void __launch_bounds__(kAttBwd2Threads, 1)
    attn_bwd_tc2_kernel(const __grid_constant__ CUtensorMap tm_kv,
                        const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_do,
                        const __grid_constant__ CUtensorMap tm_dq,
                        const __grid_constant__ CUtensorMap tm_dkv, const float* __restrict__ lse,
                        const float* __restrict__ delta, const float2* __restrict__ cs, int S,
                        int Hq, int Hkv, float scale, float scale_log2, int* err) {
  using C = AttBwd2Cfg;
  constexpr int HD = 128;
  constexpr uint32_t ID_SP = umma_idesc_bf16(128, 64, false, false);  // S^T, dP^T
  constexpr uint32_t ID_KV = umma_idesc_bf16(128, HD, false, true);   // dV, dK
  constexpr uint32_t ID_Q = umma_idesc_bf16(128, 64, true, true);     // dQ^T
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t COL_DP = 64, COL_DQ = 128, COL_DV = 256, COL_DK = 384;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0 + C::OFF_K, sV = s0 + C::OFF_V, sQ = s0 + C::OFF_Q, sDO = s0 + C::OFF_DO;
  const uint32_t sPt = s0 + C::OFF_PT, sDSt = s0 + C::OFF_DST, sDQS = s0 + C::OFF_DQS;
  float* sLD = reinterpret_cast<float*>(smem + C::OFF_LD);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const uint32_t b0 = smem_u32(bars);
  const uint32_t kv_full = b0;
  auto qdo_full = [&](int i) { return b0 + 8u * (1 + i); };
  auto qdo_empty = [&](int i) { return b0 + 8u * (4 + i); };
  const uint32_t sp_full = b0 + 56, s_free = b0 + 64, ps_full = b0 + 72, pds_free = b0 + 80;
  auto dq_full = [&](int i) { return b0 + 88u + 8u * i; };
  auto dq_free = [&](int i) { return b0 + 104u + 8u * i; };
  const uint32_t acc_done = b0 + 120, drain = b0 + 128;
  auto ld_full = [&](int i) { return b0 + 136u + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int j, g, b;
  grid_rank_first(j, g, b);  // key block 0 sees the most query blocks
  const int grp = Hq / Hkv;
  const int k0 = j * 128;
  const int nqb = (S + 63) / 64;
  const int first = 2 * j;  // first 64-query block that can see these keys
  const int per_head = nqb - first;
  const int n_it = grp * per_head;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < C::NQ; ++i) {
      mbar_init(qdo_full(i), 1);
      mbar_init(qdo_empty(i), 1);
    }
    mbar_init(sp_full, 1);
    mbar_init(s_free, 256);
    mbar_init(ps_full, 256);
    mbar_init(pds_free, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(dq_full(i), 1);
      mbar_init(dq_free(i), 256);
      mbar_init(ld_full(i), 64);
    }
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_kv);
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    mbar_arrive_expect_tx(kv_full, 2 * C::KV);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      tma_load_3d(sK + c * 16384, &tm_kv, kv_full, (Hq + g) * HD + 64 * c, k0, b);
      tma_load_3d(sV + c * 16384, &tm_kv, kv_full, (Hq + Hkv + g) * HD + 64 * c, k0, b);
    }
    bool ok = true;
    int issued = 0;
    for (int it = 0; it < n_it; ++it) {
      const int bq = it % C::NQ;
      const int h = g * grp + it / per_head;
      const int q0 = (first + it % per_head) * 64;
      if (!mbar_wait(qdo_empty(bq), ((it / C::NQ) & 1) ^ 1, abort_flag)) { ok = false; break; }
      mbar_arrive_expect_tx(qdo_full(bq), 2 * C::QT);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(sQ + bq * C::QT + c * 8192, &tm_q, qdo_full(bq), h * HD + 64 * c, q0, b);
        tma_load_3d(sDO + bq * C::QT + c * 8192, &tm_do, qdo_full(bq), h * HD + 64 * c, q0, b);
      }
      issued = it + 1;
    }
    if (!ok) {
      record_error(err, kDevAttnTimeout);
      *abort_flag = 1;
      mbar_wait(kv_full, 0, nullptr);
      for (int it = issued - 1; it >= 0 && it >= issued - C::NQ; --it)
        mbar_wait(qdo_full(it % C::NQ), (it / C::NQ) & 1, nullptr);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    bool ok = mbar_wait(kv_full, 0, abort_flag);
    // Descriptors of each operand's first row (K-major views, then the
    // MN-major views of the P V-style products); an operand at byte offset o
    // is the base plus o / 16 (shared addresses stay below 2^18, so the
    // 14-bit address field cannot carry).
    const uint64_t dK = smem_desc_sw128(sK, 16, 1024), dV = smem_desc_sw128(sV, 16, 1024);
    const uint64_t dQk = smem_desc_sw128(sQ, 16, 1024), dDOk = smem_desc_sw128(sDO, 16, 1024);
    const uint64_t dPt = smem_desc_sw128(sPt, 16, 1024), dDSt = smem_desc_sw128(sDSt, 16, 1024);
    const uint64_t dQm = smem_desc_sw128(sQ, 8192, 1024), dDOm = smem_desc_sw128(sDO, 8192, 1024);
    const uint64_t dKm = smem_desc_sw128(sK, 16384, 1024), dDStm = smem_desc_sw128(sDSt, 16384, 1024);
    for (int it = 0; ok && it <= n_it; ++it) {
      if (it < n_it) {  // S^T and dP^T of block it, once the threads hold block it - 1's
        const int bq = it % C::NQ;
        if (!mbar_wait(qdo_full(bq), (it / C::NQ) & 1, abort_flag)) { ok = false; break; }
        if (it >= 1 && !mbar_wait(s_free, (it - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qo = (uint32_t)bq * (uint32_t)(C::QT / 16);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t ka = ((kk >> 2) * 16384 + (kk & 3) * 32) / 16;  // K / V: 128-row boxes
          const uint32_t qa = ((kk >> 2) * 8192 + (kk & 3) * 32) / 16;    // Q / dO: 64-row boxes
          umma_bf16(tmem_base, dK + ka, dQk + qo + qa, ID_SP, kk > 0 ? 1u : 0u);
          umma_bf16(tmem_base + COL_DP, dV + ka, dDOk + qo + qa, ID_SP, kk > 0 ? 1u : 0u);
        }
        umma_commit(sp_full);
      }
      if (it >= 1) {  // dV, dK, dQ^T of block it - 1, once its P^T and dS^T are in shared memory
        const int ip = it - 1, bq = ip % C::NQ, bd = ip & 1;
        if (!mbar_wait(ps_full, ip & 1, abort_flag)) { ok = false; break; }
        if (ip >= 2 && !mbar_wait(dq_free(bd), ((ip >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qo = (uint32_t)bq * (uint32_t)(C::QT / 16);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // over the 64 queries
          const uint32_t acc = (ip > 0 || kk > 0) ? 1u : 0u;
          umma_bf16(tmem_base + COL_DV, dPt + kk * 2, dDOm + qo + kk * 128, ID_KV, acc);
          umma_bf16(tmem_base + COL_DK, dDSt + kk * 2, dQm + qo + kk * 128, ID_KV, acc);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // over the 128 keys
          umma_bf16(tmem_base + COL_DQ + 64 * bd, dKm + kk * 128, dDStm + kk * 128, ID_Q, kk > 0 ? 1u : 0u);
        umma_commit(dq_full(bd));
        umma_commit(qdo_empty(bq));
        umma_commit(pds_free);
      }
    }
    if (ok) {
      umma_commit(acc_done);
    } else {
      record_error(err, kDevAttnTimeout);
      *abort_flag = 1;
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr);
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- threads
    // Eight warps: two per TMEM lane quarter, each taking one half (32) of the
    // block's 64 query columns, so every scheduler has two warps to switch
    // between and each thread handles 32 elements of a block.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;  // key row of S^T / dP^T; head-dim lane of dQ^T
    const int key = k0 + r;
    const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const int tid = threadIdx.x - 64;
    bool ok = true;
    auto fetch = [&](int it_, float& lv, float& dv) {
      lv = 0.f;
      dv = 0.f;
      if (it_ >= n_it || tid >= 64) return;
      const int h_ = g * grp + it_ / per_head;
      const int q_ = (first + it_ % per_head) * 64 + tid;
      if (q_ < S) {
        const int64_t o = ((int64_t)b * Hq + h_) * S + q_;
        lv = lse[o] * 1.4426950408889634f;
        dv = delta[o];
      }
    };
    // dQ^T of block it_ (this warp's 32 queries, head-dim lanes of its
    // quarter) from registers into the warp's staging tile, then one TMA
    // reduce-add into the fp32 dQ buffer.  The tile is rewritten only after
    // the previous reduce has finished reading it.
    const uint32_t stage = sDQS + (uint32_t)(warp - 2) * 4096u;
    auto stage_dq = [&](int it_, const uint32_t (&v)[32]) {
      if (lane == 0) bulk_wait_group_read0();
      __syncwarp();
#pragma unroll
      for (int e = 0; e < 32; ++e)
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(stage + (uint32_t)e * 128u + (uint32_t)lane * 4u),
                     "r"(v[e])
                     : "memory");
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int h_ = g * grp + it_ / per_head;
        const int qb_ = (first + it_ % per_head) * 64 + 32 * half;
        if (DET)  // this key block's own slot of the dQ buffer
          tma_store_3d(&tm_dq, stage, h_ * HD + 32 * quarter, qb_, j * (int)gridDim.z + b);
        else
          tma_reduce_add_3d(&tm_dq, stage, h_ * HD + 32 * quarter, qb_, b);
        bulk_commit_group();
      }
    };
    auto emit_dq = [&](int it_) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(dq_full(it_ & 1), (it_ >> 1) & 1, abort_flag))) return false;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld_32x32b_x32(lane_base + COL_DQ + 64 * (it_ & 1) + 32 * half, v);
      tmem_ld_wait();
      stage_dq(it_, v);
      return true;
    };
    float next_l, next_d;
    fetch(0, next_l, next_d);
    const uint32_t rowoff = (uint32_t)r * 128u;
    for (int it = 0; it < n_it; ++it) {
      const int q0 = (first + it % per_head) * 64;
      const int qb = q0 + 32 * half;  // first query of this thread's columns
      float* bL = sLD + (it & 1) * 128;
      float* bD = bL + 64;
      // The buffer written here was last read for block it - 2; this thread
      // has since waited for that block's P^T / dS^T to be consumed, which
      // needed every thread to have finished computing it.
      if (tid < 64) {
        bL[tid] = next_l;
        bD[tid] = next_d;
        mbar_arrive(ld_full(it & 1));
      }
      fetch(it + 1, next_l, next_d);
      ok = __all_sync(0xffffffffu, mbar_wait(ld_full(it & 1), (it >> 1) & 1, abort_flag));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(sp_full, it & 1, abort_flag));
      // dQ^T of block it - 2 (its buffer is the one block it will use) is
      // read together with this block's S^T and dP^T
      if (ok && it >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait(dq_full(it & 1), ((it - 2) >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[32], dr[32], qv[32];
      tmem_ld_32x32b_x32(lane_base + 32 * half, sr);
      tmem_ld_32x32b_x32(lane_base + COL_DP + 32 * half, dr);
      if (it >= 2) tmem_ld_32x32b_x32(lane_base + COL_DQ + 64 * (it & 1) + 32 * half, qv);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(s_free);  // S^T / dP^T are in registers: the next block may overwrite them
      if (it >= 2) {
        mbar_arrive(dq_free(it & 1));
        stage_dq(it - 2, qv);
      }
      const float4* L4 = reinterpret_cast<const float4*>(bL + 32 * half);
      const float4* D4 = reinterpret_cast<const float4*>(bD + 32 * half);
      uint32_t pp[16], dd[16];
      auto grad_tile = [&](auto mask_tag) {
        constexpr bool kMask = decltype(mask_tag)::value;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 l4 = L4[k], d4 = D4[k];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
          const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
          float pv[4], sv[4];
#pragma unroll
          for (int i = 0; i < 4; i += 2) {
            const int e = 4 * k + i;
            // (x0, x1) = s * scale_log2 - lse * log2(e), one paired FMA
            float x0 = __uint_as_float(sr[e]), x1 = __uint_as_float(sr[e + 1]);
            fma2(x0, x1, scale_log2, -lv[i], -lv[i + 1]);
            x0 = ex2_approx(x0);
            x1 = ex2_approx(x1);
            if (kMask && !(qb + e < S && key <= qb + e)) x0 = 0.f;
            if (kMask && !(qb + e + 1 < S && key <= qb + e + 1)) x1 = 0.f;
            pv[i] = x0;
            pv[i + 1] = x1;
            // dS = P (dP - D): a paired subtract and a paired multiply
            float d0 = __uint_as_float(dr[e]), d1 = __uint_as_float(dr[e + 1]);
            add2(d0, d1, -dv[i], -dv[i + 1]);
            mul2(d0, d1, x0, x1);
            sv[i] = d0;
            sv[i + 1] = d1;
          }
          pp[2 * k] = pack2_bf16(pv[0], pv[1]);
          pp[2 * k + 1] = pack2_bf16(pv[2], pv[3]);
          dd[2 * k] = pack2_bf16(sv[0], sv[1]);
          dd[2 * k + 1] = pack2_bf16(sv[2], sv[3]);
        }
      };
      // Only blocks that touch the diagonal or the sequence end need the mask.
      if (qb < k0 + 128 || qb + 32 > S)
        grad_tile(std::true_type{});
      else
        grad_tile(std::false_type{});
      if (it >= 1) {  // P^T, dS^T of the previous block consumed
        ok = __all_sync(0xffffffffu, mbar_wait(pds_free, (it - 1) & 1, abort_flag));
        if (!ok) break;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int jj = half * 4 + k;  // 16-byte chunk of the 128-byte row
        const uint32_t off = rowoff + (uint32_t)((jj ^ (r & 7)) * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sPt + off), "r"(pp[4 * k]),
                     "r"(pp[4 * k + 1]), "r"(pp[4 * k + 2]), "r"(pp[4 * k + 3])
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sDSt + off), "r"(dd[4 * k]),
                     "r"(dd[4 * k + 1]), "r"(dd[4 * k + 2]), "r"(dd[4 * k + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(ps_full);
    }
    // the last two blocks' dQ
    for (int ip = n_it >= 2 ? n_it - 2 : 0; ok && ip < n_it; ++ip) ok = emit_dq(ip);
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag));
    if (ok) {
      tc_fence_after();
      // dK and dV rows go into the K and V tiles' shared memory (every MMA
      // that read them has completed), in the tensor map's swizzled layout;
      // one thread then stores both tiles with the TMA unit.
      auto put = [&](uint32_t tile, int col, uint32_t a, uint32_t b_, uint32_t c_, uint32_t d_) {
        const int chunk = (col & 63) >> 3;  // 16-byte chunk of the 128-byte row
        const uint32_t addr = tile + (uint32_t)(col >> 6) * 16384u + (uint32_t)r * 128u +
                              (uint32_t)((chunk ^ (r & 7)) * 16);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b_),
                     "r"(c_), "r"(d_)
                     : "memory");
      };
      // dK: pairs (d, d + HD/2) get the inverse rotation of the key's position;
      // this warp takes d in [32 half, 32 half + 32) and its partners
      {
        const int c = half;
        uint32_t x1[32], x2[32];
        tmem_ld_32x32b_x32(lane_base + COL_DK + 32 * c, x1);
        tmem_ld_32x32b_x32(lane_base + COL_DK + HD / 2 + 32 * c, x2);
        tmem_ld_wait();
        {
          const int kp = key < S ? key : S - 1;  // rows past the end are computed, not stored
          uint32_t o1[16], o2[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float a1 = __uint_as_float(x1[e]) * scale, b1 = __uint_as_float(x1[e + 1]) * scale;
            float a2 = __uint_as_float(x2[e]) * scale, b2 = __uint_as_float(x2[e + 1]) * scale;
            if (cs) {
              const float2 ca = cs[(int64_t)kp * (HD / 2) + 32 * c + e];
              const float2 cb = cs[(int64_t)kp * (HD / 2) + 32 * c + e + 1];
              const float y1a = a1 * ca.x + a2 * ca.y, y2a = a2 * ca.x - a1 * ca.y;
              const float y1b = b1 * cb.x + b2 * cb.y, y2b = b2 * cb.x - b1 * cb.y;
              a1 = y1a; a2 = y2a; b1 = y1b; b2 = y2b;
            }
            o1[e / 2] = pack2_bf16(a1, b1);
            o2[e / 2] = pack2_bf16(a2, b2);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            put(sK, 32 * c + 8 * k, o1[4 * k], o1[4 * k + 1], o1[4 * k + 2], o1[4 * k + 3]);
            put(sK, HD / 2 + 32 * c + 8 * k, o2[4 * k], o2[4 * k + 1], o2[4 * k + 2], o2[4 * k + 3]);
          }
        }
      }
      // dV: this warp takes columns [64 half, 64 half + 64)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * half + cc;
        uint32_t v[32];
        tmem_ld_32x32b_x32(lane_base + COL_DV + 32 * c, v);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          put(sV, 32 * c + 8 * k, pack2_bf16(__uint_as_float(v[8 * k + 0]), __uint_as_float(v[8 * k + 1])),
              pack2_bf16(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
              pack2_bf16(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
              pack2_bf16(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
      }
      fence_proxy_async_smem();
    } else if (lane == 0) {
      record_error(err, kDevAttnTimeout);
      *abort_flag = 1;
    }
    if (lane == 0) bulk_wait_group0();  // this warp's dQ reduces are complete
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  } else if (threadIdx.x == 64 && !*abort_flag) {
    // dK and dV tiles; key rows past the sequence end are outside the map
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      tma_store_3d(&tm_dkv, sK + c * 16384, (Hq + g) * HD + 64 * c, k0, b);
      tma_store_3d(&tm_dkv, sV + c * 16384, (Hq + Hkv + g) * HD + 64 * c, k0, b);
    }
    bulk_commit_group();
    bulk_wait_group0();
  }
}

// ------------------------------------------------------------------ host side
namespace {

// Reserve `bytes` of dynamic shared memory for `kern` on the current device,
// once per kernel and device (the attribute is per device).
bool smem_attr_set(const void* kern, int bytes) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;  // (kernel, device)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> l(mu);
  for (const auto& e : done)
    if (e.first == kern && e.second == dev) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  done.emplace_back(kern, dev);
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_att() {
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

template <int HD>
int fwd_pp(const __nv_bfloat16* qkv, __nv_bfloat16* o, float* lse, int B, int S, int Hq, int Hkv,
           int* err, cudaStream_t st) {
  using C = AttFwd2Cfg<HD>;
  auto fn = encode_fn_att();
  if (!fn) return -3;
  const int64_t W = (int64_t)(Hq + 2 * Hkv) * HD, WO = (int64_t)Hq * HD;
  CUtensorMap tm, tm_o;
  cuuint64_t dims[3] = {(cuuint64_t)W, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)(W * 2), (cuuint64_t)(S * W * 2)};
  cuuint64_t dims_o[3] = {(cuuint64_t)WO, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides_o[2] = {(cuuint64_t)(WO * 2), (cuuint64_t)(S * WO * 2)};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(qkv), dims, strides,
         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      fn(&tm_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o, dims_o, strides_o, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return -3;
  if (!smem_attr_set(reinterpret_cast<const void*>(attn_fwd_pp_kernel<HD>), C::SMEM)) return -3;
  // two query heads of a group per item when the group size is even, else
  // two consecutive query blocks of one head
  const int pair_heads = (Hq / Hkv) % 2 == 0 ? 1 : 0;
  const int nqb = (S + 127) / 128;
  const int items = pair_heads ? nqb * (Hq / 2) * B : ((nqb + 1) / 2) * Hq * B;
  const int grid = items < num_sms() ? items : num_sms();
  attn_fwd_pp_kernel<HD><<<grid, kAttFwd2Threads, C::SMEM, st>>>(
      tm, tm_o, lse, S, Hq, Hkv, B, 1.4426950408889634f / sqrtf((float)HD), pair_heads, err);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

template <int HD, bool DET>
int bwd_tc(const __nv_bfloat16* qkv, const __nv_bfloat16* o, const __nv_bfloat16* dout,
           const float* lse, float* delta, float* dq_acc, __nv_bfloat16* dqkv, int B, int S, int Hq,
           int Hkv, const float2* cs, int* err, cudaStream_t st) {
  using C = AttBwdCfg<HD>;
  auto fn = encode_fn_att();
  if (!fn) return -3;
  const int64_t W = (int64_t)(Hq + 2 * Hkv) * HD, WO = (int64_t)Hq * HD;
  CUtensorMap tq, td;
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  cuuint64_t dq[3] = {(cuuint64_t)W, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t sq[2] = {(cuuint64_t)(W * 2), (cuuint64_t)(S * W * 2)};
  cuuint64_t dd[3] = {(cuuint64_t)WO, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t sd[2] = {(cuuint64_t)(WO * 2), (cuuint64_t)(S * WO * 2)};
  if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(qkv), dq, sq, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      fn(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(dout), dd, sd, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return -3;
  if (!smem_attr_set(reinterpret_cast<const void*>(attn_bwd_tc_kernel<HD, DET>), C::SMEM)) return -3;
  const int64_t T = (int64_t)B * S;
  if (!DET && cudaMemsetAsync(dq_acc, 0, (size_t)T * WO * sizeof(float), st) != cudaSuccess)
    return -3;
  attn_delta(o, dout, delta, B, S, Hq, HD, st);
  const float scale = 1.f / sqrtf((float)HD);
  dim3 grid((S + 127) / 128, Hkv, B);
  attn_bwd_tc_kernel<HD, DET><<<grid, kAttThreads, C::SMEM, st>>>(
      tq, td, lse, delta, dq_acc, dqkv, cs, S, Hq, Hkv, scale, scale * 1.4426950408889634f, err);
  attn_dq_finalize(dq_acc, dqkv, B, S, Hq, Hkv, HD, scale, cs, DET ? (S + 127) / 128 : 0, st);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

template <bool DET>
int bwd_tc2(const __nv_bfloat16* qkv, const __nv_bfloat16* o, const __nv_bfloat16* dout,
            const float* lse, float* delta, float* dq_acc, __nv_bfloat16* dqkv, int B, int S, int Hq,
            int Hkv, const float2* cs, int* err, cudaStream_t st) {
  using C = AttBwd2Cfg;
  constexpr int HD = 128;
  auto fn = encode_fn_att();
  if (!fn) return -3;
  const int64_t W = (int64_t)(Hq + 2 * Hkv) * HD, WO = (int64_t)Hq * HD;
  CUtensorMap tkv, tq, td, tdq, tdkv;
  cuuint32_t box_kv[3] = {64, 128, 1}, box_q[3] = {64, 64, 1}, box_dq[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  cuuint64_t dq[3] = {(cuuint64_t)W, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t sq[2] = {(cuuint64_t)(W * 2), (cuuint64_t)(S * W * 2)};
  cuuint64_t dd[3] = {(cuuint64_t)WO, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t sd[2] = {(cuuint64_t)(WO * 2), (cuuint64_t)(S * WO * 2)};
  auto enc = [&](CUtensorMap* m, const void* base, cuuint64_t* dims, cuuint64_t* strides,
                 cuuint32_t* box) {
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  cuuint64_t sdq[2] = {(cuuint64_t)(WO * 4), (cuuint64_t)(S * WO * 4)};
  const int nkb = (S + 127) / 128;
  cuuint64_t ddq[3] = {(cuuint64_t)WO, (cuuint64_t)S, (cuuint64_t)(DET ? B * nkb : B)};
  if (!enc(&tkv, qkv, dq, sq, box_kv) || !enc(&tq, qkv, dq, sq, box_q) ||
      !enc(&td, dout, dd, sd, box_q) || !enc(&tdkv, dqkv, dq, sq, box_kv) ||
      fn(&tdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dq_acc, ddq, sdq, box_dq, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return -3;
  if (!smem_attr_set(reinterpret_cast<const void*>(attn_bwd_tc2_kernel<DET>), C::SMEM)) return -3;
  const int64_t T = (int64_t)B * S;
  if (!DET && cudaMemsetAsync(dq_acc, 0, (size_t)T * WO * sizeof(float), st) != cudaSuccess)
    return -3;
  attn_delta(o, dout, delta, B, S, Hq, HD, st);
  const float scale = 1.f / sqrtf((float)HD);
  dim3 grid((S + 127) / 128, Hkv, B);
  attn_bwd_tc2_kernel<DET><<<grid, kAttBwd2Threads, C::SMEM, st>>>(
      tkv, tq, td, tdq, tdkv, lse, delta, cs, S, Hq, Hkv, scale, scale * 1.4426950408889634f, err);
  attn_dq_finalize(dq_acc, dqkv, B, S, Hq, Hkv, HD, scale, cs, DET ? nkb : 0, st);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace

int attn_bwd(const __nv_bfloat16* qkv, const __nv_bfloat16* o, const __nv_bfloat16* dout,
             const float* lse, float* delta, float* dq_acc, __nv_bfloat16* dqkv, int B, int S,
             int Hq, int Hkv, int hd, const float2* cs, bool deterministic, int* err,
             cudaStream_t st) {
  if (B <= 0 || S <= 0) return 0;
  if (Hkv <= 0 || Hq % Hkv) return -1;
  if (hd == 64)
    return deterministic
               ? bwd_tc<64, true>(qkv, o, dout, lse, delta, dq_acc, dqkv, B, S, Hq, Hkv, cs, err, st)
               : bwd_tc<64, false>(qkv, o, dout, lse, delta, dq_acc, dqkv, B, S, Hq, Hkv, cs, err, st);
  if (hd == 128)
    return deterministic
               ? bwd_tc2<true>(qkv, o, dout, lse, delta, dq_acc, dqkv, B, S, Hq, Hkv, cs, err, st)
               : bwd_tc2<false>(qkv, o, dout, lse, delta, dq_acc, dqkv, B, S, Hq, Hkv, cs, err, st);
  return -1;
}

int attn_fwd(const __nv_bfloat16* qkv, __nv_bfloat16* o, float* lse, int B, int S, int Hq, int Hkv,
             int hd, int* err, cudaStream_t st) {
  if (B <= 0 || S <= 0) return 0;
  if (Hkv <= 0 || Hq % Hkv) return -1;
  if ((reinterpret_cast<uintptr_t>(qkv) & 15) != 0) return -1;
  if (hd == 64) return fwd_pp<64>(qkv, o, lse, B, S, Hq, Hkv, err, st);
  if (hd == 128) return fwd_pp<128>(qkv, o, lse, B, S, Hq, Hkv, err, st);
  return -1;
}

}  // namespace sf
