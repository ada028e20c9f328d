// RMSNorm backward for callers that cannot allocate device memory.
//
// sf_op_rmsnorm_bwd needs a scratch buffer for the per-block partial sums of
// the gain gradient, which its caller allocates.  Some callers cannot: code
// that runs inside a host application whose memory manager owns the device's
// whole budget, or a latency-critical loop in which a cudaMalloc (which can
// synchronise the device and can fail at any time) is not acceptable.  This
// variant keeps that scratch in a fixed array of this library's own device
// memory instead, so a call allocates nothing.
//
// The array below is reserved on every GPU that loads this part of the
// library and stays reserved until the process exits.  All calls share it:
// two calls whose kernels overlap on the GPU (different streams, or different
// host threads) race on it and must not be issued.  Each call writes every
// partial it later reads, so the contents left by an earlier call never need
// clearing.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sf.h"
#include "sf_internal.h"

namespace {

static __device__ __align__(256) float g_norm_bwd_scratch[SF_STATIC_SCRATCH_FLOATS];

// Device address of the array, looked up once per device with that device
// current.  In host code the array's name is only a host-side stand-in, never
// a device address, so kernels are given this looked-up pointer.
constexpr int kMaxDevices = 64;
float* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_m;

float* scratch_on_current_device(int dev) {
  std::lock_guard<std::mutex> l(g_scratch_m);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_norm_bwd_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  return g_scratch_addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int sf_op_rmsnorm_bwd_noalloc(const float* x, const uint16_t* g, const float* rstd,
                                         const float* dy, const float* dres, float* dx,
                                         uint16_t* dxb, uint16_t* dg, int64_t rows, int32_t d,
                                         void* stream) {
  if (rows < 1 || d < 8 || d % 8 || d > 16384) return SF_EINVAL;
  if (!x || !g || !rstd || !dy || !dx || !dxb || !dg) return SF_EINVAL;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dx) || !aligned16(dxb) ||
      (dres && !aligned16(dres)) || (reinterpret_cast<uintptr_t>(g) & 7))
    return SF_EINVAL;
  // same partition of rows as the scratch-taking entry point: identical sums
  const int parts = sf::rmsnorm_bwd_parts(rows, d);
  if ((int64_t)parts * d > (int64_t)SF_STATIC_SCRATCH_FLOATS) return SF_EINVAL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SF_ECUDA;
  float* scratch = scratch_on_current_device(dev);
  if (scratch == nullptr) return SF_ECUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  sf::rmsnorm_bwd(x, reinterpret_cast<const __nv_bfloat16*>(g), rstd, dy, dres, dx,
                  reinterpret_cast<__nv_bfloat16*>(dxb), scratch, parts, rows, d, st);
  sf::reduce_parts_bf16(scratch, parts, d, reinterpret_cast<__nv_bfloat16*>(dg), st);
  return cudaGetLastError() == cudaSuccess ? SF_OK : SF_ECUDA;
}
