// Layer-sliding training engine: the model API of sf.h.
//
// SlideFormer ("An Efficient Heterogeneous Co-Design for Fine-Tuning on a
// Single GPU", gist.science technical summary):
//   2.A  layers slide through the GPU; one host thread drives separate CUDA
//        streams for transfers and compute; after layer i's backward its
//        gradients go to the host while the GPU runs layer i-1's backward and
//        prefetches layer i-2; the CPU updates layer i meanwhile.
//   2.B  a pre-allocated queue of identical GPU buffers holds the active
//        layers; gradients and the fp32->bf16 conversions share fixed host
//        buffers; Adam state lives in host memory and is updated per layer.
//   2.C  fused LinearCrossEntropy keeps the logits out of memory.
//
// This engine: R ring slots (weights + gradients of one layer each) on the
// device; streams C (compute), U (host->device) and D (device->host) fenced
// by events; one pinned bf16 pack per layer that first carries the weights to
// the GPU and then receives that layer's gradients, which the host Adam
// workers turn back into the next step's bf16 weights in place.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <functional>
#include <memory>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "sf.h"
#include "sf_internal.h"

namespace {

using bf16 = __nv_bfloat16;
using Clock = std::chrono::steady_clock;

thread_local std::string g_init_error;

inline uint16_t f2bf(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}
// IEEE binary16 bits to float (the host's native half type)
inline float h2f(uint16_t h) {
  _Float16 x;
  std::memcpy(&x, &h, 2);
  return (float)x;
}
// A gradient element from a pack: bf16, or fp16 scaled by the step's loss scale
template <bool F16>
inline float grd(uint16_t x, float inv) {
  if constexpr (F16) {
    return h2f(x) * inv;
  } else {
    (void)inv;
    uint32_t u = (uint32_t)x << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
  }
}

inline float bf2f(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}
inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ thread pool
// parallel_for over [0, n) in chunks; the calling thread takes part.  One
// parallel_for runs at a time (callers are serialised).
class Pool {
 public:
  explicit Pool(int threads) {
    for (int i = 1; i < threads; ++i) workers_.emplace_back([this] { work(); });
  }
  ~Pool() {
    {
      std::lock_guard<std::mutex> l(m_);
      stop_ = true;
    }
    cv_.notify_all();
    for (auto& t : workers_) t.join();
  }
  int size() const { return (int)workers_.size() + 1; }
  void parallel_for(int64_t n, int64_t chunk, const std::function<void(int64_t, int64_t)>& fn) {
    if (n <= 0) return;
    std::lock_guard<std::mutex> run(run_m_);
    {
      std::lock_guard<std::mutex> l(m_);
      fn_ = &fn;
      n_ = n;
      chunk_ = std::max<int64_t>(1, chunk);
      next_.store(0);
      active_ = (int)workers_.size();
      ++gen_;
    }
    cv_.notify_all();
    run_chunks();
    std::unique_lock<std::mutex> l(m_);
    done_cv_.wait(l, [&] { return active_ == 0; });
    fn_ = nullptr;
  }

 private:
  void run_chunks() {
    while (true) {
      const int64_t b = next_.fetch_add(chunk_);
      if (b >= n_) break;
      (*fn_)(b, std::min(b + chunk_, n_));
    }
  }
  void work() {
    uint64_t seen = 0;
    std::unique_lock<std::mutex> l(m_);
    while (true) {
      cv_.wait(l, [&] { return stop_ || gen_ != seen; });
      if (stop_) return;
      seen = gen_;
      l.unlock();
      run_chunks();
      l.lock();
      if (--active_ == 0) done_cv_.notify_all();
    }
  }
  std::vector<std::thread> workers_;
  std::mutex m_, run_m_;
  std::condition_variable cv_, done_cv_;
  const std::function<void(int64_t, int64_t)>* fn_ = nullptr;
  int64_t n_ = 0, chunk_ = 1;
  std::atomic<int64_t> next_{0};
  int active_ = 0;
  uint64_t gen_ = 0;
  bool stop_ = false;
};

// One host copy of a unit's state.  pack = bf16 weights to stream in, then
// (after the unit's backward) its bf16 gradients, then the updated weights.
struct HostUnit {
  int64_t elems = 0;          // padded pack length
  uint16_t* pack = nullptr;   // pinned
  std::unique_ptr<float[]> master, m, v;
  std::unique_ptr<uint16_t[]> m16, v16;  // the moments as bf16 (compressed optimizer state)
  std::vector<uint16_t> retained;  // last step's gradients (retain_grads)
  std::unique_ptr<float[]> acc;    // gradient sum over the micro-batches of a step
  bool acc_bad = false;            // a micro-batch's fp16 gradients overflowed
  std::vector<float> retained_acc; // last accumulated step's summed gradients
  float retained_inv = 0.f;        // 1/scale of retained fp16 gradients (0: bf16)
};

// Steps without an overflow before the fp16 gradient scale doubles.
constexpr int64_t kScaleWindow = 1000;

// Where a micro-batch stands in a step: the only one, or the first, a middle
// or the last of several whose gradients are summed before the update.
enum Phase : int { kOnly = 0, kFirst = 1, kMid = 2, kLast = 3 };

// Adam constants of one step (bias corrections folded in by adam_consts).
// Adam constants of one step, with the bias corrections folded in:
// lr (m/bc1) / (sqrt(v/bc2) + eps) = alpha m / (sqrt(v) + eps2) with
// alpha = lr sqrt(bc2) / bc1 and eps2 = eps sqrt(bc2): one square root and
// one division per element (the divider is the bottleneck of a host core).
struct AdamK {
  float b1, b2, lrwd, alpha, eps2;
};

// (offset in the caller's unpadded order, offset in the padded pack, count)
struct Seg {
  int64_t src, dst, n;
};

}  // namespace

struct sf_ctx {
  sf_config cfg{};
  std::string err;
  bool poisoned = false;
  int L = 0, R = 0;
  int64_t d = 0, qdim = 0, kvdim = 0, qkvdim = 0, F = 0, V = 0, Tmax = 0, Smax = 0;
  int64_t off_g1 = 0, off_qkv = 0, off_bqkv = 0, off_o = 0, off_g2 = 0, off_gu = 0, off_d = 0,
          pack_elems = 0;
  bool bias = false, tied = false;  // Q/K/V projection biases; LM head = embedding
  std::vector<Seg> segs;
  int64_t chunk_rows = 0;
  int dg_parts = 0;

  // device
  std::vector<void*> dev_allocs;
  std::vector<bf16*> ring;  // R slots of 2 * pack_elems (weights, then grads)
  float* X = nullptr;       // checkpoints of the residual stream: L+1 slots, or 4 when they slide
  bool xoff = false;        // sliding activations: checkpoints live in pinned host memory
  float* x_pin = nullptr;   // [L][Tmax * d] host copies of the checkpoints
  cudaEvent_t ev_xused[4] = {}, ev_xfree[4] = {}, ev_xready[4] = {};
  bf16 *u = nullptr, *qkv = nullptr, *o = nullptr, *w2 = nullptr, *mb = nullptr;
  float* ab32 = nullptr;  // gate and up outputs [T, 2F] fp32, kept for the SwiGLU backward
  float *rstd1 = nullptr, *rstd2 = nullptr, *rstdf = nullptr, *lse = nullptr, *h = nullptr;
  float *dX = nullptr, *dw2 = nullptr, *dh = nullptr, *du = nullptr, *dq_acc = nullptr,
        *delta = nullptr, *dg_part = nullptr;
  bf16 *dXb = nullptr, *dab = nullptr, *dhb = nullptr, *dob = nullptr, *dqkv = nullptr;
  bf16 *hf = nullptr, *Wlm = nullptr, *gf = nullptr, *dWlm16 = nullptr, *dgf = nullptr,
       *dz = nullptr, *x0b = nullptr;
  // one chunk of fp32 logits, and its bf16 dZ
  float *zf = nullptr, *dhf = nullptr, *dWlm32 = nullptr, *loss_rows = nullptr, *loss_dev = nullptr;
  float2* rope_cs = nullptr;
  int32_t* labels_dev = nullptr;
  int* dev_err = nullptr;

  // host
  std::vector<HostUnit> layers;
  HostUnit lm, fn;  // LM head [V*d], final norm [d]
  std::unique_ptr<float[]> E, Em, Ev, dE;
  std::unique_ptr<uint16_t[]> Em16, Ev16;  // compressed embedding moments
  bool cstate = false;                     // bf16 Adam moments, stochastically rounded
  // fp16 gradients: weight gradients leave the GPU as fp16 times lscale; the
  // scale halves after a step whose gradients overflowed and doubles after
  // kScaleWindow steps without one
  bool f16g = false;
  float lscale = 1.f;
  int64_t lgood = 0;
  std::atomic<int64_t> skipped{0};  // unit updates skipped for overflow (total)
  int64_t skipped_seen = 0;
  float cur_inv = 0.f;              // 1/scale of the running step's gradients (0: bf16)
  int gepi() const { return f16g ? sf::kEpiF16 : sf::kEpiBF16; }
  float gscale() const { return f16g ? lscale : 1.f; }
  uint32_t e_key = 0;                      // their random stream for a pending embedding update
  bool e_bad = false;                      // the tied head's fp16 gradient overflowed this step
  uint16_t* x0_pin = nullptr;    // gathered embeddings, later the input gradient dX0
  int32_t* lab_pin = nullptr;
  float* loss_pin = nullptr;
  int* err_pin = nullptr;
  std::vector<void*> pinned;

  // streams and events
  cudaStream_t sC = nullptr, sU = nullptr, sD = nullptr;
  std::vector<cudaEvent_t> ev_loaded, ev_free, ev_grads, ev_d2h;  // per slot x3, per layer
  cudaEvent_t ev_x0 = nullptr, ev_lm = nullptr, ev_head = nullptr, ev_head_d2h = nullptr,
              ev_dx0 = nullptr, ev_start = nullptr, ev_end = nullptr, ev_end_d = nullptr;
  std::vector<cudaEvent_t> all_events;

  // timing
  bool timing = false;
  std::vector<cudaEvent_t> t_ev;  // pairs
  size_t t_used = 0;
  std::vector<int> t_kind;        // 0 gemm, 1 attention
  std::vector<double> t_flops;
  sf_stats stats{};
  int64_t launches = 0;

  // host workers
  std::unique_ptr<Pool> pool;
  std::thread adam_thread;
  std::mutex aq_m;
  std::condition_variable aq_cv, aq_done_cv;
  struct Task {
    int unit;
    cudaEvent_t ev;
    int prio;  // the order the next step needs the unit in: embedding, layers, LM head
    Clock::time_point deadline;
    bool adam_on;   // the step's optimizer settings, fixed when the task is posted
    sf_adam adam;
    int64_t t;
    int arg;        // row range of a deferred embedding-update task
    int phase;      // micro-batch phase (Phase)
    float ginv;     // 1/scale of the benchmark's fp16 gradients (0: bf16)
  };
  std::deque<Task> aq;
  int aq_pending = 0;
  // pending tasks per unit slot [L + 3]: layers, LM head + final norm (L),
  // embedding gradient (L + 1), deferred embedding-row updates (L + 2)
  std::vector<int> unit_pending;
  // A deferred embedding update: e_state[row] is 0 (to update), 1 (being
  // updated) or 2 (done), so every row is updated exactly once whether the
  // next step's gather or a background task reaches it first.
  std::unique_ptr<std::atomic<uint8_t>[]> e_state;
  bool e_pending = false;
  AdamK e_k{};
  std::vector<int32_t> e_rows;  // rows of dE that hold the last step's gradient
  std::vector<int32_t> tok_copy;   // tokens of the step whose embedding update is pending
  bool async = false;
  int aq_status = SF_OK;
  std::string aq_err;
  bool aq_stop = false;
  const sf_adam* cur_adam = nullptr;
  int phase = kOnly;          // of the micro-batch being run; copied into its tasks
  bool last_accum = false;    // the last step summed several micro-batches
  double upd_layer_ms = 0.0;  // host Adam time of layer tasks since the last stats
  int64_t upd_layer_n = 0;
  sf_adam adam_copy{};
  bool adam_on = false;
  int64_t adam_t = 0;
  double adam_ms = 0.0;
  std::atomic<int> inject_fail_unit{-1000};
  std::atomic<int> inject_sleep_ms{0};

  // host timeline (sf_get_trace)
  std::mutex tr_m;
  std::vector<sf_trace_event> trace;
  size_t tr_head = 0;
  Clock::time_point t0 = Clock::now();

  bool have_loss = false;
  float loss = 0.f;
  int64_t wait_ms = 300000;

  void set_err(const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    err = buf;
  }
};

namespace {

void trace(sf_ctx* ctx, int kind, int unit) {
  const double t = std::chrono::duration<double, std::milli>(Clock::now() - ctx->t0).count();
  std::lock_guard<std::mutex> l(ctx->tr_m);
  constexpr size_t kCap = 8192;
  if (ctx->trace.size() < kCap) {
    ctx->trace.push_back({t, kind, unit});
  } else {
    ctx->trace[ctx->tr_head] = {t, kind, unit};
    ctx->tr_head = (ctx->tr_head + 1) % kCap;
  }
}

#define CK(call)                                                                     \
  do {                                                                               \
    cudaError_t e_ = (call);                                                         \
    if (e_ != cudaSuccess) {                                                         \
      ctx->set_err("%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, \
                   __LINE__);                                                        \
      ctx->poisoned = true;                                                          \
      return SF_ECUDA;                                                               \
    }                                                                                \
  } while (0)

bool dev_alloc(sf_ctx* ctx, void** p, size_t bytes) {
  if (bytes == 0) bytes = 256;
  if (cudaMalloc(p, bytes) != cudaSuccess) {
    cudaGetLastError();
    ctx->set_err("cudaMalloc of %zu bytes failed", bytes);
    return false;
  }
  ctx->dev_allocs.push_back(*p);
  return true;
}
template <class T>
bool dalloc(sf_ctx* ctx, T** p, int64_t n) {
  return dev_alloc(ctx, reinterpret_cast<void**>(p), (size_t)n * sizeof(T));
}
template <class T>
bool halloc(sf_ctx* ctx, T** p, int64_t n) {
  void* q = nullptr;
  size_t bytes = std::max<size_t>(256, (size_t)n * sizeof(T));
  if (cudaHostAlloc(&q, bytes, cudaHostAllocPortable) != cudaSuccess) {
    cudaGetLastError();
    ctx->set_err("cudaHostAlloc of %zu bytes failed", bytes);
    return false;
  }
  ctx->pinned.push_back(q);
  *p = reinterpret_cast<T*>(q);
  return true;
}
bool new_floats(sf_ctx* ctx, std::unique_ptr<float[]>& p, int64_t n) {
  p.reset(new (std::nothrow) float[std::max<int64_t>(n, 1)]);
  if (!p) ctx->set_err("host allocation of %lld floats failed", (long long)n);
  return (bool)p;
}
bool new_halves(sf_ctx* ctx, std::unique_ptr<uint16_t[]>& p, int64_t n) {
  p.reset(new (std::nothrow) uint16_t[std::max<int64_t>(n, 1)]);
  if (!p) ctx->set_err("host allocation of %lld 16-bit values failed", (long long)n);
  return (bool)p;
}
// Zero elements [b, e) of a unit's moments, whichever storage it uses.
void zero_moments(sf_ctx* ctx, float* m, float* v, uint16_t* m16, uint16_t* v16, int64_t b,
                  int64_t e) {
  ctx->pool->parallel_for(e - b, 1 << 18, [=](int64_t x, int64_t y) {
    if (m) std::memset(m + b + x, 0, (size_t)(y - x) * 4);
    if (v) std::memset(v + b + x, 0, (size_t)(y - x) * 4);
    if (m16) std::memset(m16 + b + x, 0, (size_t)(y - x) * 2);
    if (v16) std::memset(v16 + b + x, 0, (size_t)(y - x) * 2);
  });
}

// Bounded host wait on an event.
int wait_event(sf_ctx* ctx, cudaEvent_t ev, const char* what) {
  const auto deadline = Clock::now() + std::chrono::milliseconds(ctx->wait_ms);
  while (true) {
    cudaError_t r = cudaEventQuery(ev);
    if (r == cudaSuccess) return SF_OK;
    if (r != cudaErrorNotReady) {
      ctx->set_err("waiting for %s: %s", what, cudaGetErrorString(r));
      ctx->poisoned = true;
      return SF_ECUDA;
    }
    if (Clock::now() > deadline) {
      ctx->set_err("timed out after %lld ms waiting for %s", (long long)ctx->wait_ms, what);
      return SF_ETIMEOUT;
    }
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

// ------------------------------------------------------------------ Adam on host
// The element loops take restrict-qualified pointers so that the compiler
// vectorises them (the update is bound by host memory bandwidth).

template <bool F16>
void adam_bf16_span(uint16_t* __restrict p, float* __restrict w, float* __restrict m,
                    float* __restrict v, int64_t b, int64_t e, const AdamK k, float inv) {
  for (int64_t i = b; i < e; ++i) {
    const float g = grd<F16>(p[i], inv);
    const float mi = k.b1 * m[i] + (1.f - k.b1) * g;
    const float vi = k.b2 * v[i] + (1.f - k.b2) * g * g;
    float th = w[i];
    th = th - k.lrwd * th - k.alpha * mi / (std::sqrt(vi) + k.eps2);
    m[i] = mi;
    v[i] = vi;
    w[i] = th;
    p[i] = f2bf(th);
  }
}

void adam_f32_span(const float* __restrict g, float* __restrict w, float* __restrict m,
                   float* __restrict v, int64_t b, int64_t e, const AdamK k) {
  for (int64_t i = b; i < e; ++i) {
    const float gi = g[i];
    const float mi = k.b1 * m[i] + (1.f - k.b1) * gi;
    const float vi = k.b2 * v[i] + (1.f - k.b2) * gi * gi;
    float th = w[i];
    th = th - k.lrwd * th - k.alpha * mi / (std::sqrt(vi) + k.eps2);
    m[i] = mi;
    v[i] = vi;
    w[i] = th;
  }
}

void refresh_bf16_span(uint16_t* __restrict p, const float* __restrict w, int64_t b, int64_t e) {
  for (int64_t i = b; i < e; ++i) p[i] = f2bf(w[i]);
}

// A micro-batch's gradient (in the pack) into the fp32 sum, then the
// unchanged weights back into the pack for the next micro-batch's copy.
template <bool F16>
void accum_span(uint16_t* __restrict p, float* __restrict acc, const float* __restrict w,
                int64_t b, int64_t e, bool first, float inv) {
  for (int64_t i = b; i < e; ++i) {
    const float g = grd<F16>(p[i], inv);
    acc[i] = first ? g : acc[i] + g;
    p[i] = f2bf(w[i]);
  }
}

// Adam on the summed gradient (fp32 sum + the last micro-batch's part).
template <bool F16>
void adam_acc_span(uint16_t* __restrict p, const float* __restrict acc, float* __restrict w,
                   float* __restrict m, float* __restrict v, int64_t b, int64_t e, const AdamK k,
                   float inv) {
  for (int64_t i = b; i < e; ++i) {
    const float g = acc[i] + grd<F16>(p[i], inv);
    const float mi = k.b1 * m[i] + (1.f - k.b1) * g;
    const float vi = k.b2 * v[i] + (1.f - k.b2) * g * g;
    float th = w[i];
    th = th - k.lrwd * th - k.alpha * mi / (std::sqrt(vi) + k.eps2);
    m[i] = mi;
    v[i] = vi;
    w[i] = th;
    p[i] = f2bf(th);
  }
}

AdamK adam_consts(const sf_adam& a, int64_t step_t) {
  const double bc1 = 1.0 - std::pow((double)a.beta1, (double)step_t);
  const double sbc2 = std::sqrt(1.0 - std::pow((double)a.beta2, (double)step_t));
  return {a.beta1, a.beta2, a.lr * a.weight_decay, (float)(a.lr * sbc2 / bc1),
          (float)(a.eps * sbc2)};
}

// ---- compressed optimizer state: bf16 moments, rounded stochastically.
// Random bits: a counter-based hash (lowbias32, C. Wellons' xorshift-multiply
// hash) of the element's index in its unit, keyed by step and unit; its low
// half-word rounds the first moment, its high half-word the second.
inline uint32_t lowbias32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352dU;
  x ^= x >> 15;
  x *= 0x846ca68bU;
  x ^= x >> 16;
  return x;
}
inline uint32_t sr_key(int64_t t, int unit) {
  return lowbias32(lowbias32((uint32_t)t) ^ ((uint32_t)(unit + 3) * 0x9E3779B9U));
}
// x to bf16, rounded up in magnitude with probability (low 16 bits of x) / 2^16
inline uint16_t bf16_sr(float x, uint32_t r) {
  uint32_t u;
  std::memcpy(&u, &x, 4);
  return (uint16_t)((u + (r & 0xFFFFu)) >> 16);
}

// Adam on [b, e) with bf16 moments.  G: 0 = bf16 gradient in the pack, 1 =
// fp32 sum acc + the pack's bf16 part, 2 = fp32 gradient acc (the pack, if
// any, only receives the new bf16 weights).  idx_off: the caller's index of
// element 0 (selects the random words).
template <int G, bool F16 = false>
void adam_c_span(uint16_t* __restrict p, const float* __restrict acc, float* __restrict w,
                 uint16_t* __restrict m, uint16_t* __restrict v, int64_t b, int64_t e,
                 const AdamK k, uint32_t key, int64_t idx_off, float inv = 1.f) {
  for (int64_t i = b; i < e; ++i) {
    const float g = G == 0 ? grd<F16>(p[i], inv) : G == 1 ? acc[i] + grd<F16>(p[i], inv) : acc[i];
    const float mi = k.b1 * bf2f(m[i]) + (1.f - k.b1) * g;
    const float vi = k.b2 * bf2f(v[i]) + (1.f - k.b2) * g * g;
    float th = w[i];
    th = th - k.lrwd * th - k.alpha * mi / (std::sqrt(vi) + k.eps2);
    w[i] = th;
    if (G != 2 || p) p[i] = f2bf(th);
    const uint32_t r = lowbias32((uint32_t)(i + idx_off) ^ key);
    m[i] = bf16_sr(mi, r);
    v[i] = bf16_sr(vi, r >> 16);
  }
}

// The compressed-state update of a packed unit, segment by segment so that
// every element draws the random words of its index in the caller's order.
void adam_compressed(sf_ctx* ctx, HostUnit& hu, int unit, const AdamK k, int64_t step_t,
                     bool with_acc, float inv) {
  const uint32_t key = sr_key(step_t, unit);
  std::vector<Seg> one;
  const std::vector<Seg>* segs = &ctx->segs;
  if (unit < 0) {  // LM head or final norm: one unpadded range
    one.push_back({0, 0, unit == SF_UNIT_FINAL_NORM ? ctx->d : ctx->V * ctx->d});
    segs = &one;
  }
  for (const Seg& s : *segs) {
    uint16_t* p = hu.pack + s.dst;
    const float* acc = with_acc ? hu.acc.get() + s.dst : nullptr;
    float* w = hu.master.get() + s.dst;
    uint16_t* m = hu.m16.get() + s.dst;
    uint16_t* v = hu.v16.get() + s.dst;
    const int64_t off = s.src;
    ctx->pool->parallel_for(s.n, 1 << 16, [=](int64_t b, int64_t e) {
      if (inv != 0.f) {
        if (with_acc)
          adam_c_span<1, true>(p, acc, w, m, v, b, e, k, key, off, inv);
        else
          adam_c_span<0, true>(p, nullptr, w, m, v, b, e, k, key, off, inv);
      } else {
        if (with_acc)
          adam_c_span<1>(p, acc, w, m, v, b, e, k, key, off);
        else
          adam_c_span<0>(p, nullptr, w, m, v, b, e, k, key, off);
      }
    });
  }
}

// Does a pack of scaled fp16 gradients hold an overflow (an infinity or NaN)?
bool f16_overflow(sf_ctx* ctx, const uint16_t* p, int64_t n) {
  std::atomic<bool> bad{false};
  ctx->pool->parallel_for(n, 1 << 18, [&](int64_t b, int64_t e) {
    uint16_t any = 0;
    for (int64_t i = b; i < e; ++i) any |= (uint16_t)((p[i] & 0x7C00u) == 0x7C00u);
    if (any) bad.store(true, std::memory_order_relaxed);
  });
  return bad.load();
}

// One unit: optional copy of the gradients, then either the Adam update of the
// fp32 master (refreshing the bf16 pack in place) or, without an optimizer, a
// refresh of the pack from the unchanged master.  Micro-batches before the
// last only add their gradient into the unit's fp32 sum; the last one updates
// with the whole sum.  inv != 0: the pack holds fp16 gradients scaled by
// 1/inv; a unit whose gradients overflowed skips its update (its weights and
// moments stay as they are) and counts one skipped update.
void host_update(sf_ctx* ctx, HostUnit& hu, int unit, bool retain, bool adam_on,
                 const sf_adam& a, int64_t step_t, int phase, float inv) {
  uint16_t* p = hu.pack;
  float* w = hu.master.get();
  float* acc = hu.acc.get();
  const bool f16 = inv != 0.f;
  const bool bad = f16 && f16_overflow(ctx, p, hu.elems);
  if (phase == kFirst || phase == kMid) {
    const bool first = phase == kFirst;
    if (first) hu.acc_bad = false;
    hu.acc_bad = hu.acc_bad || bad;
    ctx->pool->parallel_for(hu.elems, 1 << 16, [p, acc, w, first, inv, f16](int64_t b, int64_t e) {
      if (f16)
        accum_span<true>(p, acc, w, b, e, first, inv);
      else
        accum_span<false>(p, acc, w, b, e, first, inv);
    });
    return;
  }
  const bool skip = bad || (phase == kLast && hu.acc_bad);
  if (retain) {
    hu.retained_inv = inv;
    if (phase == kLast) {
      hu.retained_acc.resize((size_t)hu.elems);
      float* dst = hu.retained_acc.data();
      ctx->pool->parallel_for(hu.elems, 1 << 16, [dst, p, acc, inv, f16](int64_t b, int64_t e) {
        for (int64_t i = b; i < e; ++i)
          dst[i] = acc[i] + (f16 ? grd<true>(p[i], inv) : grd<false>(p[i], inv));
      });
    } else {
      hu.retained.resize((size_t)hu.elems);
      uint16_t* dst = hu.retained.data();
      ctx->pool->parallel_for(hu.elems, 1 << 18, [&](int64_t b, int64_t e) {
        std::memcpy(dst + b, p + b, (size_t)(e - b) * 2);
      });
    }
  }
  if (skip) ctx->skipped.fetch_add(1, std::memory_order_relaxed);
  if (!adam_on || skip) {
    ctx->pool->parallel_for(hu.elems, 1 << 16,
                            [p, w](int64_t b, int64_t e) { refresh_bf16_span(p, w, b, e); });
    return;
  }
  const AdamK k = adam_consts(a, step_t);
  const bool with_acc = phase == kLast;
  if (ctx->cstate) {
    adam_compressed(ctx, hu, unit, k, step_t, with_acc, inv);
    return;
  }
  float* m = hu.m.get();
  float* v = hu.v.get();
  ctx->pool->parallel_for(hu.elems, 1 << 16, [=](int64_t b, int64_t e) {
    if (with_acc) {
      if (f16) adam_acc_span<true>(p, acc, w, m, v, b, e, k, inv);
      else adam_acc_span<false>(p, acc, w, m, v, b, e, k, inv);
    } else {
      if (f16) adam_bf16_span<true>(p, w, m, v, b, e, k, inv);
      else adam_bf16_span<false>(p, w, m, v, b, e, k, inv);
    }
  });
}

constexpr int kUnitEmbedRest = -10;  // internal: background embedding-row updates
constexpr int kEmbedRestTasks = 16;

int unit_slot(const sf_ctx* ctx, int unit) {
  if (unit >= 0) return unit;
  if (unit == SF_UNIT_EMBED) return ctx->L + 1;
  if (unit == kUnitEmbedRest) return ctx->L + 2;
  return ctx->L;  // LM head and final norm share a task
}

// Adam update of embedding row r, exactly once per pending update.
void e_update_row(sf_ctx* ctx, int64_t r) {
  std::atomic<uint8_t>& st = ctx->e_state[r];
  uint8_t expect = 0;
  if (st.compare_exchange_strong(expect, 1, std::memory_order_acq_rel)) {
    const int64_t d = ctx->d, o = r * d;
    if (ctx->cstate) {  // the tied head's bf16 row is written by the update itself
      adam_c_span<2>(ctx->tied ? ctx->lm.pack + o : nullptr, ctx->dE.get() + o, ctx->E.get() + o,
                     ctx->Em16.get() + o, ctx->Ev16.get() + o, 0, d, ctx->e_k, ctx->e_key, o);
    } else {
      adam_f32_span(ctx->dE.get() + o, ctx->E.get() + o, ctx->Em.get() + o, ctx->Ev.get() + o, 0,
                    d, ctx->e_k);
      if (ctx->tied) refresh_bf16_span(ctx->lm.pack + o, ctx->E.get() + o, 0, d);  // the head's copy
    }
    st.store(2, std::memory_order_release);
  } else {
    while (st.load(std::memory_order_acquire) != 2) std::this_thread::yield();
  }
}

void e_update_rows(sf_ctx* ctx, int64_t r0, int64_t r1) {
  ctx->pool->parallel_for(r1 - r0, 64, [ctx, r0](int64_t b, int64_t e) {
    for (int64_t r = r0 + b; r < r0 + e; ++r) e_update_row(ctx, r);
  });
}

void post_task(sf_ctx* ctx, int unit, cudaEvent_t ev, int arg = 0);

// Embedding gradient: zero the rows of dE the previous gradient touched,
// scatter-add the bf16 input gradient (by column ranges: no races).  The Adam
// update of the embedding is then deferred: the next step's gather updates the
// rows its tokens need, and background tasks of the lowest priority update
// the rest while the update thread would otherwise wait for gradients.
// A tied LM head adds its (dense) gradient, which the head's pack holds, to
// every row, and each row's update refreshes that row of the head's pack.
// Micro-batches before the last only add into dE (and put the unchanged
// embedding back into the head's pack for the next micro-batch).
void embed_grad(sf_ctx* ctx, bool adam_on, const sf_adam& a, int64_t step_t, int phase,
                float inv) {
  const int64_t d = ctx->d, V = ctx->V, T = (int64_t)ctx->tok_copy.size();
  if (ctx->e_pending) e_update_rows(ctx, 0, V);  // finish a previous update first
  ctx->e_pending = false;
  float* dE = ctx->dE.get();
  const bool first = phase == kOnly || phase == kFirst;
  if (ctx->tied) {
    const uint16_t* gh = ctx->lm.pack;
    const bool f16 = inv != 0.f;
    const bool bad = f16 && f16_overflow(ctx, gh, V * d);
    ctx->e_bad = (first ? false : ctx->e_bad) || bad;
    ctx->pool->parallel_for(V * d, 1 << 16, [dE, gh, first, f16, inv](int64_t b, int64_t e) {
      for (int64_t i = b; i < e; ++i)
        dE[i] = (first ? 0.f : dE[i]) + (f16 ? grd<true>(gh[i], inv) : grd<false>(gh[i], inv));
    });
  } else if (first) {
    const int32_t* rows = ctx->e_rows.data();
    ctx->pool->parallel_for((int64_t)ctx->e_rows.size(), 64, [rows, dE, d](int64_t b, int64_t e) {
      for (int64_t i = b; i < e; ++i) std::memset(dE + (int64_t)rows[i] * d, 0, (size_t)d * 4);
    });
    ctx->e_rows.clear();
  }
  const int32_t* tokens = ctx->tok_copy.data();
  const uint16_t* g = ctx->x0_pin;
  ctx->pool->parallel_for(d, 64, [tokens, dE, g, T, d](int64_t c0, int64_t c1) {
    for (int64_t t = 0; t < T; ++t) {
      float* __restrict row = dE + (int64_t)tokens[t] * d;
      const uint16_t* __restrict gr = g + t * d;
      for (int64_t j = c0; j < c1; ++j) row[j] += bf2f(gr[j]);
    }
  });
  if (!ctx->tied) {  // rows holding gradient, zeroed before the next step's scatter
    ctx->e_rows.insert(ctx->e_rows.end(), ctx->tok_copy.begin(), ctx->tok_copy.end());
    std::sort(ctx->e_rows.begin(), ctx->e_rows.end());
    ctx->e_rows.erase(std::unique(ctx->e_rows.begin(), ctx->e_rows.end()), ctx->e_rows.end());
  }
  const bool last = phase == kOnly || phase == kLast;
  const bool skip = last && ctx->tied && ctx->e_bad;  // the tied head's fp16 gradient overflowed
  if (skip) ctx->skipped.fetch_add(1, std::memory_order_relaxed);
  if (!last || !adam_on || skip) {
    if (ctx->tied) {  // the head's pack holds gradients: put the weights back
      uint16_t* p = ctx->lm.pack;
      const float* E = ctx->E.get();
      ctx->pool->parallel_for(V * d, 1 << 16, [p, E](int64_t b, int64_t e) { refresh_bf16_span(p, E, b, e); });
    }
    return;
  }
  ctx->e_k = adam_consts(a, step_t);
  ctx->e_key = sr_key(step_t, SF_UNIT_EMBED);
  for (int64_t r = 0; r < V; ++r) ctx->e_state[r].store(0, std::memory_order_relaxed);
  std::atomic_thread_fence(std::memory_order_release);
  ctx->e_pending = true;
  for (int i = 0; i < kEmbedRestTasks; ++i) post_task(ctx, kUnitEmbedRest, nullptr, i);
}

void finish_task(sf_ctx* ctx, const sf_ctx::Task& t, int st, const std::string& why) {
  {
    std::lock_guard<std::mutex> l(ctx->aq_m);
    if (st != SF_OK && ctx->aq_status == SF_OK) {
      ctx->aq_status = st;
      ctx->aq_err = why;
    }
    --ctx->unit_pending[unit_slot(ctx, t.unit)];
    --ctx->aq_pending;
  }
  ctx->aq_done_cv.notify_all();
}

void run_task(sf_ctx* ctx, const sf_ctx::Task& t) {
  if (ctx->inject_sleep_ms.load() > 0)
    std::this_thread::sleep_for(std::chrono::milliseconds(ctx->inject_sleep_ms.load()));
  if (ctx->inject_fail_unit.load() == t.unit && t.unit != SF_UNIT_EMBED && t.unit != kUnitEmbedRest) {
    // the gradients are dropped: put the unchanged weights back into the pack
    if (t.unit >= 0) {
      host_update(ctx, ctx->layers[t.unit], t.unit, false, false, t.adam, t.t, kOnly, 0.f);
    } else {
      if (!ctx->tied) host_update(ctx, ctx->lm, SF_UNIT_LM_HEAD, false, false, t.adam, t.t, kOnly, 0.f);
      host_update(ctx, ctx->fn, SF_UNIT_FINAL_NORM, false, false, t.adam, t.t, kOnly, 0.f);
    }
    finish_task(ctx, t, SF_ESTATE, "injected Adam worker failure on unit " + std::to_string(t.unit));
    return;
  }
  const auto t0 = Clock::now();
  trace(ctx, 5, t.unit);
  const bool retain = ctx->cfg.retain_grads != 0;
  if (t.unit >= 0) {
    host_update(ctx, ctx->layers[t.unit], t.unit, retain, t.adam_on, t.adam, t.t, t.phase, t.ginv);
  } else if (t.unit == SF_UNIT_EMBED) {
    embed_grad(ctx, t.adam_on, t.adam, t.t, t.phase, t.ginv);
  } else if (t.unit == kUnitEmbedRest) {
    const int64_t V = ctx->V;
    e_update_rows(ctx, V * t.arg / kEmbedRestTasks, V * (t.arg + 1) / kEmbedRestTasks);
  } else {  // LM head (unless tied: the embedding task takes its gradient) and final norm
    if (!ctx->tied)
      host_update(ctx, ctx->lm, SF_UNIT_LM_HEAD, retain, t.adam_on, t.adam, t.t, t.phase, t.ginv);
    host_update(ctx, ctx->fn, SF_UNIT_FINAL_NORM, retain, t.adam_on, t.adam, t.t, t.phase, t.ginv);
  }
  const double ms = std::chrono::duration<double, std::milli>(Clock::now() - t0).count();
  ctx->adam_ms += ms;
  if (t.unit >= 0) {
    std::lock_guard<std::mutex> l(ctx->aq_m);
    ctx->upd_layer_ms += ms;
    ++ctx->upd_layer_n;
  }
  trace(ctx, 6, t.unit);
  finish_task(ctx, t, SF_OK, std::string());
}

// The update coordinator: of the units whose gradient copy has landed, update
// the one the next step needs first (embedding, then layers 0 .. L-1, then the
// LM head), so that the next step's forward can start before every update is
// done.  A copy that fails, or does not land within the bound, fails its task.
void adam_loop(sf_ctx* ctx) {
  std::vector<sf_ctx::Task> mine;
  while (true) {
    {
      std::unique_lock<std::mutex> l(ctx->aq_m);
      if (mine.empty()) ctx->aq_cv.wait(l, [&] { return ctx->aq_stop || !ctx->aq.empty(); });
      while (!ctx->aq.empty()) {
        mine.push_back(ctx->aq.front());
        ctx->aq.pop_front();
      }
      if (mine.empty() && ctx->aq_stop) return;
    }
    int best = -1;
    for (size_t i = 0; i < mine.size();) {
      const cudaError_t r = mine[i].ev ? cudaEventQuery(mine[i].ev) : cudaSuccess;  // null: no copy to wait for
      if (r == cudaSuccess) {
        if (best < 0 || mine[i].prio < mine[best].prio) best = (int)i;
        ++i;
        continue;
      }
      if (r != cudaErrorNotReady || Clock::now() > mine[i].deadline) {
        const bool to = (r == cudaErrorNotReady);
        ctx->poisoned = true;  // the pack is in an unknown state
        finish_task(ctx, mine[i], to ? SF_ETIMEOUT : SF_ECUDA,
                    to ? std::string("timed out waiting for a gradient copy")
                       : std::string("gradient copy failed: ") + cudaGetErrorString(r));
        mine.erase(mine.begin() + i);
        if (best > (int)i) --best;
        continue;
      }
      ++i;
    }
    if (best < 0) {
      std::this_thread::sleep_for(std::chrono::microseconds(20));
      continue;
    }
    const sf_ctx::Task t = mine[best];
    mine.erase(mine.begin() + best);
    run_task(ctx, t);
  }
}

void post_task(sf_ctx* ctx, int unit, cudaEvent_t ev, int arg) {
  {
    std::lock_guard<std::mutex> l(ctx->aq_m);
    const int prio = unit == SF_UNIT_EMBED ? -1
                     : unit == kUnitEmbedRest ? ctx->L + 1
                     : (unit >= 0 ? unit : ctx->L);
    ctx->aq.push_back({unit, ev, prio, Clock::now() + std::chrono::milliseconds(ctx->wait_ms),
                       ctx->adam_on, ctx->adam_copy, ctx->adam_t, arg, ctx->phase, ctx->cur_inv});
    ++ctx->unit_pending[unit_slot(ctx, unit)];
    ++ctx->aq_pending;
  }
  ctx->aq_cv.notify_one();
}

// Bounded wait until the host update of one unit (posted by an earlier step) is done.
int wait_unit(sf_ctx* ctx, int unit) {
  trace(ctx, 3, unit);
  struct End {
    sf_ctx* c;
    int u;
    ~End() { trace(c, 4, u); }
  } end{ctx, unit};
  std::unique_lock<std::mutex> l(ctx->aq_m);
  const int u = unit_slot(ctx, unit);
  const bool ok = ctx->aq_done_cv.wait_for(l, std::chrono::milliseconds(ctx->wait_ms),
                                           [&] { return ctx->unit_pending[u] == 0; });
  if (!ok) {
    ctx->set_err("timed out waiting for the host update of unit %d", unit);
    return SF_ETIMEOUT;
  }
  if (ctx->aq_status != SF_OK) {
    ctx->set_err("%s", ctx->aq_err.c_str());
    const int st = ctx->aq_status;
    ctx->aq_status = SF_OK;
    return st;
  }
  return SF_OK;
}

int wait_tasks(sf_ctx* ctx) {
  std::unique_lock<std::mutex> l(ctx->aq_m);
  const bool ok = ctx->aq_done_cv.wait_for(l, std::chrono::milliseconds(ctx->wait_ms),
                                           [&] { return ctx->aq_pending == 0; });
  if (!ok) {
    ctx->set_err("timed out waiting for the host Adam workers");
    return SF_ETIMEOUT;
  }
  if (ctx->aq_status != SF_OK) {
    ctx->set_err("%s", ctx->aq_err.c_str());
    int st = ctx->aq_status;
    ctx->aq_status = SF_OK;
    return st;
  }
  return SF_OK;
}

// ------------------------------------------------------------------ timing helpers
struct Timed {
  sf_ctx* ctx;
  int kind;
  double flops;
  cudaEvent_t b = nullptr, e = nullptr;
  cudaStream_t st;
  // kind: 0 GEMM, 1 attention, 2 layer forward, 3 layer backward, 4 gradient D2H, 5 head
  Timed(sf_ctx* c, int k, double f, cudaStream_t s = nullptr)
      : ctx(c), kind(k), flops(f), st(s ? s : c->sC) {
    if (!ctx->timing) return;
    while (ctx->t_ev.size() < 2 * (ctx->t_used + 1)) {
      cudaEvent_t x;
      if (cudaEventCreate(&x) != cudaSuccess) return;
      ctx->t_ev.push_back(x);
    }
    b = ctx->t_ev[2 * ctx->t_used];
    e = ctx->t_ev[2 * ctx->t_used + 1];
    ++ctx->t_used;
    ctx->t_kind.push_back(kind);
    ctx->t_flops.push_back(flops);
    cudaEventRecord(b, st);
  }
  ~Timed() {
    if (e) cudaEventRecord(e, st);
  }
};

// A GEMM with the fused epilogues' extra arguments (flops: the algorithmic
// count when it is not 2*M*N*K, e.g. the gated tile's two products).
// Vocabulary ranges of the LM head's dH product (split-K, fixed-order sum).
constexpr int kHeadSplitK = 4;

int gemm_args(sf_ctx* ctx, const sf::GemmArgs& g, double flops = 0.0) {
  int st;
  char why[128] = {0};
  int launched = 0;
  sf::GemmArgs a = g;
  a.launched = &launched;
  {
    Timed t(ctx, 0, flops > 0.0 ? flops : 2.0 * g.M * g.N * g.K);
    st = sf::gemm(a, ctx->dev_err, ctx->sC, why);
  }
  ctx->launches += launched;  // the GEMM and, for a split K, its fixed-order sum
  ctx->stats.gemm_launches += 1;
  if (st != 0) {
    ctx->set_err("%s", why);
    if (st == -3) ctx->poisoned = true;
    return st == -3 ? SF_ECUDA : SF_EINVAL;
  }
  return SF_OK;
}

int gemm(sf_ctx* ctx, int layout, int epi, int64_t M, int64_t N, int64_t K, const void* A,
         int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc, const float* R = nullptr,
         int64_t ldr = 0, float alpha = 1.f, const void* bias = nullptr) {
  sf::GemmArgs g;
  g.layout = layout; g.epi = epi; g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = lda; g.B = B; g.ldb = ldb; g.C = C; g.ldc = ldc; g.R = R; g.ldr = ldr;
  g.alpha = alpha;
  g.bias = bias;
  return gemm_args(ctx, g);
}

double attn_fwd_flops(int64_t B, int64_t S, int64_t Hq, int64_t hd) {
  // QK^T and PV over the causal half (diagonal included): 2 * 2 * hd * S(S+1)/2 per head
  return 2.0 * B * Hq * hd * (double)S * (double)(S + 1);
}

#define RET(x)                    \
  do {                            \
    int r_ = (x);                 \
    if (r_ != SF_OK) return r_;   \
  } while (0)

// Device address of checkpoint l (the input of layer l; l = L is the final
// hidden state).  Resident: one slot per checkpoint.  Sliding: a window of
// four slots, the others in pinned host memory.
float* xck(sf_ctx* c, int l, int64_t T) {
  if (c->xoff) return c->X + (int64_t)(l % 4) * c->Tmax * c->d;
  return c->X + (int64_t)l * T * c->d;
}

// ------------------------------------------------------------------ layer compute
struct LayerW {
  const bf16 *g1, *wqkv, *bqkv, *wo, *g2, *wgu, *wd;  // bqkv null without projection biases
};
struct LayerG {
  bf16 *g1, *wqkv, *bqkv, *wo, *g2, *wgu, *wd;
};
LayerW slot_w(sf_ctx* c, int s) {
  const bf16* b = c->ring[s];
  return {b + c->off_g1, b + c->off_qkv, c->bias ? b + c->off_bqkv : nullptr, b + c->off_o,
          b + c->off_g2, b + c->off_gu, b + c->off_d};
}
LayerG slot_g(sf_ctx* c, int s) {
  bf16* b = c->ring[s] + c->pack_elems;
  return {b + c->off_g1, b + c->off_qkv, c->bias ? b + c->off_bqkv : nullptr, b + c->off_o,
          b + c->off_g2, b + c->off_gu, b + c->off_d};
}

// A gain gradient from the per-block partials: bf16, or fp16 times the loss scale.
void grad_parts(sf_ctx* c, int d, bf16* out) {
  if (c->f16g)
    sf::reduce_parts_f16(c->dg_part, c->dg_parts, d, reinterpret_cast<uint16_t*>(out), c->lscale, c->sC);
  else
    sf::reduce_parts_bf16(c->dg_part, c->dg_parts, d, out, c->sC);
}

// Forward of one layer from X_l (fp32) to X_{l+1}; with `full == false` the
// final down projection is skipped (recompute for the backward needs only the
// intermediates).  keep_ab stores the gate and up outputs in fp32 for the
// SwiGLU backward (the recompute, and the last layer, whose backward follows
// the head without a recompute).
int layer_forward(sf_ctx* c, const LayerW& w, const float* Xin, float* Xout, int B, int S,
                  bool full, bool keep_ab) {
  sf_ctx* ctx = c;
  const int64_t T = (int64_t)B * S, d = c->d, F = c->F;
  const int Hq = c->cfg.n_heads, Hkv = c->cfg.n_kv_heads, hd = c->cfg.head_dim;
  sf::rmsnorm_fwd(Xin, w.g1, c->u, c->rstd1, T, (int)d, c->cfg.rms_eps, c->sC);
  {
    // Q/K/V projection; its epilogue adds the biases (if any) to the fp32
    // accumulator, rotates the Q and K heads and rounds to bf16 once
    sf::GemmArgs g;
    g.layout = sf::kNT; g.epi = sf::kEpiQKV; g.M = T; g.N = c->qkvdim; g.K = d;
    g.A = c->u; g.lda = d; g.B = w.wqkv; g.ldb = d; g.C = c->qkv; g.ldc = c->qkvdim;
    g.bias = w.bqkv; g.cs = c->rope_cs; g.seq = S; g.rope_cols = (int)((Hq + Hkv) * hd); g.hd = hd;
    RET(gemm_args(c, g));
  }
  {
    Timed t(c, 1, attn_fwd_flops(B, S, Hq, hd));
    if (sf::attn_fwd(c->qkv, c->o, c->lse, B, S, Hq, Hkv, hd, c->dev_err, c->sC) != 0) {
      ctx->set_err("attention forward launch failed");
      return SF_ECUDA;
    }
  }
  RET(gemm(c, sf::kNT, sf::kEpiF32Add, T, d, c->qdim, c->o, c->qdim, w.wo, c->qdim, c->h, d,
           Xin, d));
  sf::rmsnorm_fwd(c->h, w.g2, c->w2, c->rstd2, T, (int)d, c->cfg.rms_eps, c->sC);
  {
    // gate/up projection; its epilogue forms m = silu(a) * b from the fp32
    // accumulator (and keeps a, b in fp32 when the backward needs them)
    sf::GemmArgs g;
    g.layout = sf::kNT; g.epi = sf::kEpiGLU; g.M = T; g.N = F; g.K = d;
    g.A = c->w2; g.lda = d; g.B = w.wgu; g.ldb = d; g.C = c->mb; g.ldc = F;
    if (keep_ab) { g.aux = c->ab32; g.ldaux = 2 * F; }
    RET(gemm_args(c, g, 2.0 * T * 2 * F * d));
  }
  c->launches += 3;
  if (full)
    RET(gemm(c, sf::kNT, sf::kEpiF32Add, T, d, F, c->mb, F, w.wd, F, Xout, d, c->h, d));
  return SF_OK;
}

// Backward of one layer.  On entry dX / dXb hold dLoss/dX_{l+1}; on exit they
// hold dLoss/dX_l.  Weight gradients go into the slot's gradient area (bf16).
int layer_backward(sf_ctx* c, const LayerW& w, const LayerG& g, const float* Xin, int B, int S) {
  sf_ctx* ctx = c;
  const int64_t T = (int64_t)B * S, d = c->d, F = c->F;
  const int Hq = c->cfg.n_heads, Hkv = c->cfg.n_kv_heads, hd = c->cfg.head_dim;
  // down projection: X_{l+1} = h + m Wd^T.  dm = dX Wd stays in the fp32
  // accumulator: the epilogue takes it through SwiGLU into [da | db]
  RET(gemm(c, sf::kNN, sf::kEpiGLUBwd, T, F, d, c->dXb, d, w.wd, F, c->dab, 2 * F, c->ab32, 2 * F));
  RET(gemm(c, sf::kTN, c->gepi(), d, F, T, c->dXb, d, c->mb, F, g.wd, F, nullptr, 0, c->gscale()));
  // gate/up projection from w2 = RMSNorm(h; g2)
  RET(gemm(c, sf::kNN, sf::kEpiF32, T, d, 2 * F, c->dab, 2 * F, w.wgu, d, c->dw2, d));
  RET(gemm(c, sf::kTN, c->gepi(), 2 * F, d, T, c->dab, 2 * F, c->w2, d, g.wgu, d, nullptr, 0,
           c->gscale()));
  sf::rmsnorm_bwd(c->h, w.g2, c->rstd2, c->dw2, c->dX, c->dh, c->dhb, c->dg_part, c->dg_parts,
                  T, (int)d, c->sC);
  grad_parts(c, (int)d, g.g2);
  // output projection: h = X_l + o Wo^T
  RET(gemm(c, sf::kNN, sf::kEpiBF16, T, c->qdim, d, c->dhb, d, w.wo, c->qdim, c->dob, c->qdim));
  RET(gemm(c, sf::kTN, c->gepi(), d, c->qdim, T, c->dhb, d, c->o, c->qdim, g.wo, c->qdim, nullptr,
           0, c->gscale()));
  {
    Timed t(c, 1, 2.5 * attn_fwd_flops(B, S, Hq, hd));
    if (sf::attn_bwd(c->qkv, c->o, c->dob, c->lse, c->delta, c->dq_acc, c->dqkv, B, S, Hq, Hkv,
                     hd, c->rope_cs, c->cfg.deterministic != 0, c->dev_err, c->sC) != 0) {
      ctx->set_err("attention backward launch failed");
      return SF_ECUDA;
    }
  }
  // the biases' gradient: column sums of the pre-rotation dQ, dK, dV
  if (g.bqkv) {
    if (c->f16g)
      sf::bias_grad_f16(c->dqkv, c->qkvdim, T, (int)c->qkvdim, c->dg_part, c->dg_parts,
                        reinterpret_cast<uint16_t*>(g.bqkv), c->lscale, c->sC);
    else
      sf::bias_grad(c->dqkv, c->qkvdim, T, (int)c->qkvdim, c->dg_part, c->dg_parts, g.bqkv, c->sC);
    c->launches += 2;
  }
  // QKV projection from u = RMSNorm(X_l; g1)
  RET(gemm(c, sf::kNN, sf::kEpiF32, T, d, c->qkvdim, c->dqkv, c->qkvdim, w.wqkv, d, c->du, d));
  RET(gemm(c, sf::kTN, c->gepi(), c->qkvdim, d, T, c->dqkv, c->qkvdim, c->u, d, g.wqkv, d, nullptr,
           0, c->gscale()));
  sf::rmsnorm_bwd(Xin, w.g1, c->rstd1, c->du, c->dh, c->dX, c->dXb, c->dg_part, c->dg_parts, T,
                  (int)d, c->sC);
  grad_parts(c, (int)d, g.g1);
  c->launches += 7;  // 2 norm, 2 reduce, 3 attention (GEMMs are counted in gemm())
  return SF_OK;
}

// Final norm + fused chunked LM head / cross-entropy + final norm backward.
int head_fwd_bwd(sf_ctx* c, int64_t T, int64_t n_valid) {
  sf_ctx* ctx = c;
  const int64_t d = c->d, V = c->V;
  const float* XL = xck(c, c->L, T);
  sf::rmsnorm_fwd(XL, c->gf, c->hf, c->rstdf, T, (int)d, c->cfg.rms_eps, c->sC);
  const float inv_n = n_valid > 0 ? 1.f / (float)n_valid : 0.f;
  for (int64_t r0 = 0; r0 < T; r0 += c->chunk_rows) {
    const int64_t n = std::min(c->chunk_rows, T - r0);
    const bool first = r0 == 0, last = r0 + n >= T;
    // fp32 logits of the chunk; the row softmax writes dZ (bf16) beside them
    RET(gemm(c, sf::kNT, sf::kEpiF32, n, V, d, c->hf + r0 * d, d, c->Wlm, d, c->zf, V));
    if (sf::ce_rows_f32(c->zf, c->dz, c->labels_dev + r0, n, V, inv_n, c->loss_rows + r0,
                        c->dev_err, c->sC) != 0) {
      ctx->set_err("cross-entropy launch failed");
      return SF_ECUDA;
    }
    {  // dH = dZ W_lm, over up to kHeadSplitK vocabulary ranges when that fills
       // the SMs better; the partial sums go to the chunk's fp32 logits, which
       // the cross-entropy kernel has already read
      sf::GemmArgs g;
      g.layout = sf::kNN; g.epi = sf::kEpiF32; g.M = n; g.N = d; g.K = V;
      g.A = c->dz; g.lda = V; g.B = c->Wlm; g.ldb = d; g.C = c->dhf + r0 * d; g.ldc = d;
      g.splitk_max = (int)std::min<int64_t>(kHeadSplitK, 1 + (c->chunk_rows * V) / (n * d));
      g.ws = c->zf;
      RET(gemm_args(c, g));
    }
    // dW_lm: fp32 sums over the chunks; the last chunk's product adds the sum
    // and rounds the bf16 gradient in its epilogue
    if (last && !c->f16g)
      RET(gemm(c, sf::kTN, sf::kEpiBF16Acc, V, d, n, c->dz, V, c->hf + r0 * d, d, c->dWlm16, d,
               first ? nullptr : c->dWlm32, d));
    else
      RET(gemm(c, sf::kTN, first ? sf::kEpiF32 : sf::kEpiF32Acc, V, d, n, c->dz, V,
               c->hf + r0 * d, d, c->dWlm32, d));
    c->launches += 1;
  }
  sf::sum_f32(c->loss_rows, T, inv_n, c->loss_dev, c->sC);
  sf::rmsnorm_bwd(XL, c->gf, c->rstdf, c->dhf, nullptr, c->dX, c->dXb, c->dg_part, c->dg_parts,
                  T, (int)d, c->sC);
  grad_parts(c, (int)d, c->dgf);
  c->launches += 4;
  if (c->f16g) {
    sf::cast_f32_f16(c->dWlm32, reinterpret_cast<uint16_t*>(c->dWlm16), V * d, c->lscale, c->sC);
    c->launches += 1;
  }
  return SF_OK;
}

// Rows of one chunk of the fused LM head: a chunk holds fp32 logits and their
// bf16 dZ (6 bytes per logit) within 2 GiB, in equal chunks of a multiple of
// 128 rows (at the 8B shape: 6 chunks of 2816 rows, 2.2 GB).
int64_t lce_chunk_rows(int64_t T, int64_t V) {
  const int64_t cap = std::max<int64_t>(128, (((int64_t)2 << 30) / (6 * V)) / 128 * 128);
  const int64_t chunks = (T + cap - 1) / cap;
  const int64_t rows = ((T + chunks - 1) / chunks + 127) / 128 * 128;
  return std::min<int64_t>(rows, T);
}

size_t unit_numel_cfg(const sf_config* c, int32_t unit) {
  if (!c) return 0;
  const int64_t d = c->hidden, q = (int64_t)c->n_heads * c->head_dim,
                kv = (int64_t)c->n_kv_heads * c->head_dim, F = c->ffn;
  if (unit >= 0) {
    if (unit >= c->n_layers) return 0;
    return (size_t)(2 * d + q * d + 2 * kv * d + d * q + 3 * F * d + (c->qkv_bias ? q + 2 * kv : 0));
  }
  if (unit == SF_UNIT_LM_HEAD && c->tie_embeddings) return 0;  // the head is the embedding
  if (unit == SF_UNIT_EMBED || unit == SF_UNIT_LM_HEAD) return (size_t)c->vocab * (size_t)d;
  if (unit == SF_UNIT_FINAL_NORM) return (size_t)d;
  return 0;
}

const char* validate(const sf_config* c) {
  if (!c) return "null config";
  if (c->n_layers < 1) return "n_layers must be >= 1";
  if (c->hidden < 8 || c->hidden % 8 || c->hidden > 16384) return "hidden must be a multiple of 8 in [8, 16384]";
  if (c->head_dim != 64 && c->head_dim != 128) return "head_dim must be 64 or 128";
  if (c->n_heads < 1 || c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads) return "n_heads must be a positive multiple of n_kv_heads";
  if (c->ffn < 8 || c->ffn % 8) return "ffn must be a positive multiple of 8";
  if (c->vocab < 8 || c->vocab % 8) return "vocab must be a positive multiple of 8";
  if (c->max_batch < 1 || c->max_seq < 1) return "max_batch and max_seq must be >= 1";
  if ((int64_t)c->max_batch * c->max_seq > (int64_t)1 << 26) return "max_batch * max_seq too large";
  if (c->ring_slots < 2 || c->ring_slots > std::max(2, c->n_layers)) return "ring_slots must be in [2, max(2, n_layers)]";
  if (c->lce_chunk_rows < 0) return "lce_chunk_rows must be >= 0";
  if (!(c->rms_eps > 0.f) || !(c->rope_base > 1.f)) return "rms_eps must be > 0 and rope_base > 1";
  if (c->qkv_bias < 0 || c->qkv_bias > 1 || c->tie_embeddings < 0 || c->tie_embeddings > 1 ||
      c->deterministic < 0 || c->deterministic > 1 || c->bf16_adam_state < 0 ||
      c->bf16_adam_state > 1 || c->fp16_grads < 0 || c->fp16_grads > 1)
    return "qkv_bias, tie_embeddings, deterministic, bf16_adam_state and fp16_grads must be 0 or 1";
  if (!(c->loss_scale >= 0.f) || c->loss_scale > 16777216.f) return "loss_scale must be in [0, 2^24]";
  return nullptr;
}

int init(sf_ctx* ctx) {
  const sf_config& cf = ctx->cfg;
  ctx->L = cf.n_layers;
  ctx->R = std::min(cf.ring_slots, cf.n_layers);
  ctx->d = cf.hidden;
  ctx->qdim = (int64_t)cf.n_heads * cf.head_dim;
  ctx->kvdim = (int64_t)cf.n_kv_heads * cf.head_dim;
  ctx->qkvdim = ctx->qdim + 2 * ctx->kvdim;
  ctx->F = cf.ffn;
  ctx->V = cf.vocab;
  ctx->Smax = cf.max_seq;
  ctx->Tmax = (int64_t)cf.max_batch * cf.max_seq;
  ctx->wait_ms = cf.wait_timeout_ms > 0 ? cf.wait_timeout_ms : 300000;
  const int64_t d = ctx->d, T = ctx->Tmax, F = ctx->F, V = ctx->V, L = ctx->L;
  // padded pack: each group starts on a 256-byte boundary
  constexpr int64_t A = 128;
  ctx->bias = cf.qkv_bias != 0;
  ctx->tied = cf.tie_embeddings != 0;
  ctx->cstate = cf.bf16_adam_state != 0;
  ctx->f16g = cf.fp16_grads != 0;
  ctx->lscale = cf.loss_scale > 0.f ? cf.loss_scale : 65536.f;
  ctx->off_g1 = 0;
  ctx->off_qkv = round_up(d, A);
  ctx->off_bqkv = round_up(ctx->off_qkv + ctx->qkvdim * d, A);  // only when biased
  ctx->off_o = ctx->bias ? round_up(ctx->off_bqkv + ctx->qkvdim, A) : ctx->off_bqkv;
  ctx->off_g2 = round_up(ctx->off_o + d * ctx->qdim, A);
  ctx->off_gu = round_up(ctx->off_g2 + d, A);
  ctx->off_d = round_up(ctx->off_gu + 2 * F * d, A);
  ctx->pack_elems = round_up(ctx->off_d + d * F, A);
  int64_t src = 0;
  auto seg = [&](int64_t dst, int64_t n) {
    ctx->segs.push_back({src, dst, n});
    src += n;
  };
  seg(ctx->off_g1, d);
  seg(ctx->off_qkv, ctx->qkvdim * d);
  if (ctx->bias) seg(ctx->off_bqkv, ctx->qkvdim);
  seg(ctx->off_o, d * ctx->qdim);
  seg(ctx->off_g2, d);
  seg(ctx->off_gu, 2 * F * d);
  seg(ctx->off_d, d * F);
  if (cf.lce_chunk_rows > 0) {
    ctx->chunk_rows = std::min<int64_t>(cf.lce_chunk_rows, T);
  } else {
    ctx->chunk_rows = lce_chunk_rows(T, V);
  }
  ctx->dg_parts = sf::rmsnorm_bwd_parts(T, (int)d);

  if (cudaSetDevice(cf.device) != cudaSuccess) {
    cudaGetLastError();
    ctx->set_err("cudaSetDevice(%d) failed", cf.device);
    return SF_ECUDA;
  }
  int threads = cf.adam_threads > 0 ? cf.adam_threads : (int)std::thread::hardware_concurrency();
  ctx->pool.reset(new Pool(std::max(1, threads)));

  // ---- device buffers
  bool ok = true;
  ctx->ring.resize(ctx->R);
  for (int s = 0; s < ctx->R && ok; ++s) ok = dalloc(ctx, &ctx->ring[s], 2 * ctx->pack_elems);
  ctx->xoff = cf.offload_activations != 0;
  ok = ok && dalloc(ctx, &ctx->X, (ctx->xoff ? 4 : L + 1) * T * d);
  ok = ok && dalloc(ctx, &ctx->u, T * d) && dalloc(ctx, &ctx->qkv, T * ctx->qkvdim) &&
       dalloc(ctx, &ctx->o, T * ctx->qdim) && dalloc(ctx, &ctx->w2, T * d) &&
       dalloc(ctx, &ctx->ab32, T * 2 * F) && dalloc(ctx, &ctx->mb, T * F) &&
       dalloc(ctx, &ctx->rstd1, T) && dalloc(ctx, &ctx->rstd2, T) && dalloc(ctx, &ctx->rstdf, T) &&
       dalloc(ctx, &ctx->lse, T * cf.n_heads) && dalloc(ctx, &ctx->h, T * d);
  ok = ok && dalloc(ctx, &ctx->dX, T * d) && dalloc(ctx, &ctx->dw2, T * d) &&
       dalloc(ctx, &ctx->dh, T * d) && dalloc(ctx, &ctx->du, T * d) &&
       dalloc(ctx, &ctx->dq_acc, (cf.deterministic ? (ctx->Smax + 127) / 128 : 1) * T * ctx->qdim) &&
       dalloc(ctx, &ctx->delta, T * cf.n_heads) &&
       dalloc(ctx, &ctx->dg_part, (int64_t)ctx->dg_parts * std::max(d, ctx->qkvdim)) &&
       dalloc(ctx, &ctx->dXb, T * d) &&
       dalloc(ctx, &ctx->dab, T * 2 * F) &&
       dalloc(ctx, &ctx->dhb, T * d) && dalloc(ctx, &ctx->dob, T * ctx->qdim) &&
       dalloc(ctx, &ctx->dqkv, T * ctx->qkvdim);
  ok = ok && dalloc(ctx, &ctx->hf, T * d) && dalloc(ctx, &ctx->Wlm, V * d) &&
       dalloc(ctx, &ctx->gf, round_up(d, A)) && dalloc(ctx, &ctx->dWlm16, V * d) &&
       dalloc(ctx, &ctx->dgf, round_up(d, A)) && dalloc(ctx, &ctx->zf, ctx->chunk_rows * V) &&
       dalloc(ctx, &ctx->dz, ctx->chunk_rows * V) &&
       dalloc(ctx, &ctx->x0b, T * d) && dalloc(ctx, &ctx->dhf, T * d) &&
       dalloc(ctx, &ctx->dWlm32, V * d) && dalloc(ctx, &ctx->loss_rows, T) &&
       dalloc(ctx, &ctx->loss_dev, 1) && dalloc(ctx, &ctx->labels_dev, T) &&
       dalloc(ctx, &ctx->rope_cs, ctx->Smax * cf.head_dim / 2) && dalloc(ctx, &ctx->dev_err, 1);
  if (!ok) return SF_ENOMEM;
  // gradient areas: padding stays zero forever
  for (int s = 0; s < ctx->R; ++s)
    CK(cudaMemset(ctx->ring[s], 0, (size_t)2 * ctx->pack_elems * sizeof(bf16)));
  CK(cudaMemset(ctx->dev_err, 0, sizeof(int)));
  {
    std::vector<float> tab((size_t)ctx->Smax * cf.head_dim);
    sf_rope_table((int32_t)ctx->Smax, cf.head_dim, cf.rope_base, tab.data());
    CK(cudaMemcpy(ctx->rope_cs, tab.data(), tab.size() * sizeof(float), cudaMemcpyHostToDevice));
  }

  // ---- host buffers
  ctx->layers.resize(L);
  // pack_only: the tied LM head, whose weights and state are the embedding's
  auto host_unit = [&](HostUnit& hu, int64_t elems, bool pack_only = false) -> bool {
    hu.elems = elems;
    if (!halloc(ctx, &hu.pack, elems)) return false;
    uint16_t* p = hu.pack;
    if (pack_only) {
      ctx->pool->parallel_for(elems, 1 << 18, [&](int64_t s, int64_t e) {
        std::memset(p + s, 0, (size_t)(e - s) * 2);
      });
      return true;
    }
    if (!new_floats(ctx, hu.master, elems)) return false;
    if (ctx->cstate ? !new_halves(ctx, hu.m16, elems) || !new_halves(ctx, hu.v16, elems)
                    : !new_floats(ctx, hu.m, elems) || !new_floats(ctx, hu.v, elems))
      return false;
    float* a = hu.master.get();
    ctx->pool->parallel_for(elems, 1 << 18, [&](int64_t s, int64_t e) {
      std::memset(a + s, 0, (size_t)(e - s) * 4);
      std::memset(p + s, 0, (size_t)(e - s) * 2);
    });
    zero_moments(ctx, hu.m.get(), hu.v.get(), hu.m16.get(), hu.v16.get(), 0, elems);
    return true;
  };
  for (int l = 0; l < L && ok; ++l) ok = host_unit(ctx->layers[l], ctx->pack_elems);
  ok = ok && host_unit(ctx->lm, V * d, ctx->tied) && host_unit(ctx->fn, round_up(d, A));
  ok = ok && new_floats(ctx, ctx->E, V * d) && new_floats(ctx, ctx->dE, V * d) &&
       (ctx->cstate ? new_halves(ctx, ctx->Em16, V * d) && new_halves(ctx, ctx->Ev16, V * d)
                    : new_floats(ctx, ctx->Em, V * d) && new_floats(ctx, ctx->Ev, V * d));
  if (ok && ctx->xoff) ok = halloc(ctx, &ctx->x_pin, L * T * d);
  ok = ok && halloc(ctx, &ctx->x0_pin, T * d) && halloc(ctx, &ctx->lab_pin, T) &&
       halloc(ctx, &ctx->loss_pin, 1) && halloc(ctx, &ctx->err_pin, 1);
  if (!ok) return SF_ENOMEM;
  {
    float* a = ctx->E.get();
    float* e2 = ctx->dE.get();
    ctx->pool->parallel_for(V * d, 1 << 18, [&](int64_t s, int64_t e) {
      std::memset(a + s, 0, (size_t)(e - s) * 4);
      std::memset(e2 + s, 0, (size_t)(e - s) * 4);
    });
    zero_moments(ctx, ctx->Em.get(), ctx->Ev.get(), ctx->Em16.get(), ctx->Ev16.get(), 0, V * d);
  }

  // ---- streams and events
  CK(cudaStreamCreateWithFlags(&ctx->sC, cudaStreamNonBlocking));
  CK(cudaStreamCreateWithFlags(&ctx->sU, cudaStreamNonBlocking));
  CK(cudaStreamCreateWithFlags(&ctx->sD, cudaStreamNonBlocking));
  auto mk = [&](cudaEvent_t* e, bool timed) -> int {
    CK(cudaEventCreateWithFlags(e, timed ? cudaEventDefault : cudaEventDisableTiming));
    ctx->all_events.push_back(*e);
    return SF_OK;
  };
  ctx->ev_loaded.resize(ctx->R);
  ctx->ev_free.resize(ctx->R);
  ctx->ev_grads.resize(ctx->R);
  ctx->ev_d2h.resize(L);
  for (int s = 0; s < ctx->R; ++s) {
    RET(mk(&ctx->ev_loaded[s], false));
    RET(mk(&ctx->ev_free[s], false));
    RET(mk(&ctx->ev_grads[s], false));
  }
  for (int l = 0; l < L; ++l) RET(mk(&ctx->ev_d2h[l], false));
  for (int i = 0; i < 4; ++i) {
    RET(mk(&ctx->ev_xused[i], false));
    RET(mk(&ctx->ev_xfree[i], false));
    RET(mk(&ctx->ev_xready[i], false));
  }
  RET(mk(&ctx->ev_x0, false));
  RET(mk(&ctx->ev_lm, false));
  RET(mk(&ctx->ev_head, false));
  RET(mk(&ctx->ev_head_d2h, false));
  RET(mk(&ctx->ev_dx0, false));
  RET(mk(&ctx->ev_start, true));
  RET(mk(&ctx->ev_end, true));
  RET(mk(&ctx->ev_end_d, false));
  ctx->unit_pending.assign(L + 3, 0);
  ctx->e_state.reset(new (std::nothrow) std::atomic<uint8_t>[(size_t)V]);
  if (!ctx->e_state) return SF_ENOMEM;
  for (int64_t r = 0; r < V; ++r) ctx->e_state[r].store(2, std::memory_order_relaxed);
  ctx->async = cf.async_update != 0;
  ctx->adam_thread = std::thread(adam_loop, ctx);
  return SF_OK;
}

void destroy(sf_ctx* ctx) {
  if (ctx->adam_thread.joinable()) {
    {
      std::lock_guard<std::mutex> l(ctx->aq_m);
      ctx->aq_stop = true;
    }
    ctx->aq_cv.notify_all();
    ctx->adam_thread.join();
  }
  if (ctx->sC) cudaStreamSynchronize(ctx->sC);
  if (ctx->sU) cudaStreamSynchronize(ctx->sU);
  if (ctx->sD) cudaStreamSynchronize(ctx->sD);
  for (auto e : ctx->all_events) cudaEventDestroy(e);
  for (auto e : ctx->t_ev) cudaEventDestroy(e);
  for (auto s : {ctx->sC, ctx->sU, ctx->sD})
    if (s) cudaStreamDestroy(s);
  for (void* p : ctx->dev_allocs) cudaFree(p);
  for (void* p : ctx->pinned) cudaFreeHost(p);
  ctx->pool.reset();
}

// Copy `unit`'s fp32 values between the caller's order and the padded pack.
void scatter_unit(sf_ctx* ctx, const float* in, float* master) {
  for (const Seg& s : ctx->segs) {
    const float* a = in + s.src;
    float* b = master + s.dst;
    ctx->pool->parallel_for(s.n, 1 << 18, [&](int64_t x, int64_t y) {
      std::memcpy(b + x, a + x, (size_t)(y - x) * 4);
    });
  }
}

// Host-side check of a step's tokens and labels; counts the valid labels.
int check_batch(sf_ctx* ctx, const int32_t* tokens, const int32_t* labels, int64_t T,
                int64_t* n_valid) {
  const int64_t V = ctx->V;
  int64_t n = 0;
  for (int64_t t = 0; t < T; ++t) {
    if (tokens[t] < 0 || tokens[t] >= V) {
      ctx->set_err("token %d at position %lld outside [0, %lld)", tokens[t], (long long)t, (long long)V);
      return SF_EINVAL;
    }
    const int32_t y = labels[t];
    if (y == SF_IGNORE_INDEX) continue;
    if (y < 0 || y >= V) {
      ctx->set_err("label %d at position %lld outside [0, %lld) and not ignore_index", y, (long long)t, (long long)V);
      return SF_EINVAL;
    }
    ++n;
  }
  *n_valid = n;
  return SF_OK;
}

// One micro-batch through the whole stack (its tokens and labels already
// checked).  n_valid_total: valid labels of the whole step (all its
// micro-batches), which normalises the loss; phase: where this micro-batch
// stands (the host tasks it posts sum or update).
int step(sf_ctx* ctx, const int32_t* tokens, const int32_t* labels, int B, int S,
         const sf_adam* adam, int phase, int64_t n_valid_total) {
  const int64_t T = (int64_t)B * S, d = ctx->d, V = ctx->V;
  const int L = ctx->L, R = ctx->R;
  const auto t_host0 = Clock::now();
  trace(ctx, 1, -9);
  // The embedding update of the previous step reads its tokens and the pinned
  // input-gradient buffer, which this step is about to overwrite.  Without
  // async_update every update of the previous step is finished here (also the
  // ones left over by a step that timed out, which still own the pinned packs).
  if (ctx->async) RET(wait_unit(ctx, SF_UNIT_EMBED));
  else RET(wait_tasks(ctx));
  ctx->tok_copy.assign(tokens, tokens + T);
  ctx->phase = phase;
  ctx->cur_inv = ctx->f16g ? 1.f / ctx->lscale : 0.f;
  const bool updates = phase == kOnly || phase == kLast;  // this micro-batch's tasks update
  ctx->adam_on = adam != nullptr && updates;
  if (ctx->adam_on) {
    ctx->adam_copy = *adam;
    ++ctx->adam_t;
  }
  ctx->stats = sf_stats{};
  ctx->stats.timing_enabled = ctx->timing ? 1 : 0;
  ctx->t_used = 0;
  ctx->t_kind.clear();
  ctx->t_flops.clear();
  ctx->launches = 0;
  ctx->adam_ms = 0.0;
  double h2d = 0, d2h = 0;

  // ---- A0: gather bf16 embedding rows into the pinned input buffer
  {
    const float* E = ctx->E.get();
    uint16_t* x0 = ctx->x0_pin;
    const bool upd = ctx->e_pending;  // rows still owed the previous step's update
    ctx->pool->parallel_for(T, 64, [&](int64_t b, int64_t e) {
      for (int64_t t = b; t < e; ++t) {
        if (upd) e_update_row(ctx, tokens[t]);
        const float* src = E + (int64_t)tokens[t] * d;
        uint16_t* dst = x0 + t * d;
        for (int64_t j = 0; j < d; ++j) dst[j] = f2bf(src[j]);
      }
    });
    std::memcpy(ctx->lab_pin, labels, (size_t)T * 4);
  }
  trace(ctx, 2, -9);
  CK(cudaEventRecord(ctx->ev_start, ctx->sC));
  CK(cudaStreamWaitEvent(ctx->sU, ctx->ev_start, 0));
  CK(cudaMemcpyAsync(ctx->x0b, ctx->x0_pin, (size_t)T * d * 2, cudaMemcpyHostToDevice, ctx->sU));
  CK(cudaMemcpyAsync(ctx->labels_dev, ctx->lab_pin, (size_t)T * 4, cudaMemcpyHostToDevice, ctx->sU));
  CK(cudaEventRecord(ctx->ev_x0, ctx->sU));
  h2d += (double)T * d * 2 + (double)T * 4;
  CK(cudaStreamWaitEvent(ctx->sC, ctx->ev_x0, 0));
  if (ctx->xoff) CK(cudaStreamWaitEvent(ctx->sC, ctx->ev_xused[0], 0));  // previous step's X_0
  sf::cast_bf16_f32(ctx->x0b, xck(ctx, 0, T), T * d, ctx->sC);
  ctx->launches += 1;

  const size_t pack_bytes = (size_t)ctx->pack_elems * 2;
  auto h2d_layer = [&](int l) -> int {
    const int s = l % R;
    CK(cudaStreamWaitEvent(ctx->sU, ctx->ev_free[s], 0));
    CK(cudaMemcpyAsync(ctx->ring[s], ctx->layers[l].pack, pack_bytes, cudaMemcpyHostToDevice, ctx->sU));
    CK(cudaEventRecord(ctx->ev_loaded[s], ctx->sU));
    h2d += (double)pack_bytes;
    return SF_OK;
  };
  // slots start free
  for (int s = 0; s < R; ++s) CK(cudaEventRecord(ctx->ev_free[s], ctx->sC));

  // ---- forward through the ring (A1-A9)
  for (int l = 0; l < L; ++l) {
    const int s = l % R;
    if (ctx->async) RET(wait_unit(ctx, l));  // the previous step's update of this layer
    RET(h2d_layer(l));
    if (l == L - 1) {  // the LM head and final norm follow the last layer on the copy stream
      if (ctx->async) RET(wait_unit(ctx, SF_UNIT_LM_HEAD));
      if (ctx->async && ctx->tied) RET(wait_unit(ctx, kUnitEmbedRest));  // every row refreshed
      CK(cudaMemcpyAsync(ctx->Wlm, ctx->lm.pack, (size_t)V * d * 2, cudaMemcpyHostToDevice, ctx->sU));
      CK(cudaMemcpyAsync(ctx->gf, ctx->fn.pack, (size_t)ctx->fn.elems * 2, cudaMemcpyHostToDevice, ctx->sU));
      CK(cudaEventRecord(ctx->ev_lm, ctx->sU));
      h2d += (double)V * d * 2 + (double)ctx->fn.elems * 2;
    }
    CK(cudaStreamWaitEvent(ctx->sC, ctx->ev_loaded[s], 0));
    const float* Xin = xck(ctx, l, T);
    float* Xout = xck(ctx, l + 1, T);
    // sliding: X_{l+1}'s slot held X_{l-3}, whose copy to the host must be done
    if (ctx->xoff && l + 1 >= 4) CK(cudaStreamWaitEvent(ctx->sC, ctx->ev_xfree[(l + 1) % 4], 0));
    {
      Timed tl(ctx, 2, 0.0);
      RET(layer_forward(ctx, slot_w(ctx, s), Xin, Xout, B, S, true, l == L - 1));
    }
    CK(cudaEventRecord(ctx->ev_free[s], ctx->sC));
    if (ctx->xoff) {  // the checkpoint slides to the host while the next layers compute
      CK(cudaEventRecord(ctx->ev_xused[l % 4], ctx->sC));
      CK(cudaStreamWaitEvent(ctx->sD, ctx->ev_xused[l % 4], 0));
      CK(cudaMemcpyAsync(ctx->x_pin + (int64_t)l * T * d, Xin, (size_t)T * d * 4,
                         cudaMemcpyDeviceToHost, ctx->sD));
      CK(cudaEventRecord(ctx->ev_xfree[l % 4], ctx->sD));
      d2h += (double)T * d * 4;
    }
  }

  // ---- A10: fused LM head + cross-entropy, forward and backward
  CK(cudaStreamWaitEvent(ctx->sC, ctx->ev_lm, 0));
  {
    Timed th(ctx, 5, 0.0);
    RET(head_fwd_bwd(ctx, T, n_valid_total));
  }
  CK(cudaEventRecord(ctx->ev_head, ctx->sC));
  // sliding: bring checkpoint l back into slot l % 4 once that slot's last user
  // is done (the head for the slot of X_L, else the backward of layer l + 4)
  auto h2d_ck = [&](int l, cudaEvent_t after) -> int {
    CK(cudaStreamWaitEvent(ctx->sU, after, 0));
    CK(cudaStreamWaitEvent(ctx->sU, ctx->ev_xfree[l % 4], 0));
    CK(cudaMemcpyAsync(xck(ctx, l, T), ctx->x_pin + (int64_t)l * T * d, (size_t)T * d * 4,
                       cudaMemcpyHostToDevice, ctx->sU));
    CK(cudaEventRecord(ctx->ev_xready[l % 4], ctx->sU));
    h2d += (double)T * d * 4;
    return SF_OK;
  };
  if (ctx->xoff && L - 4 >= 0) RET(h2d_ck(L - 4, ctx->ev_head));
  CK(cudaStreamWaitEvent(ctx->sD, ctx->ev_head, 0));
  CK(cudaMemcpyAsync(ctx->lm.pack, ctx->dWlm16, (size_t)V * d * 2, cudaMemcpyDeviceToHost, ctx->sD));
  CK(cudaMemcpyAsync(ctx->fn.pack, ctx->dgf, (size_t)ctx->fn.elems * 2, cudaMemcpyDeviceToHost, ctx->sD));
  CK(cudaEventRecord(ctx->ev_head_d2h, ctx->sD));
  d2h += (double)V * d * 2 + (double)ctx->fn.elems * 2;
  post_task(ctx, SF_UNIT_LM_HEAD, ctx->ev_head_d2h);

  // ---- A11-A15: recompute + backward, gradients out, prefetch the next layers in
  for (int l = L - 1; l >= 0; --l) {
    const int s = l % R;
    const bool resident = l >= L - R;  // still in its slot from the forward
    if (!resident) CK(cudaStreamWaitEvent(ctx->sC, ctx->ev_loaded[s], 0));
    const LayerW w = slot_w(ctx, s);
    const float* Xin = xck(ctx, l, T);
    if (ctx->xoff && l <= L - 4) CK(cudaStreamWaitEvent(ctx->sC, ctx->ev_xready[l % 4], 0));
    // the last layer's intermediates are still in the workspace from the forward
    {
      Timed tl(ctx, 3, 0.0);
      if (l != L - 1) RET(layer_forward(ctx, w, Xin, nullptr, B, S, false, true));
      RET(layer_backward(ctx, w, slot_g(ctx, s), Xin, B, S));
    }
    CK(cudaEventRecord(ctx->ev_grads[s], ctx->sC));
    if (ctx->xoff) {
      CK(cudaEventRecord(ctx->ev_xused[l % 4], ctx->sC));
      if (l - 4 >= 0) RET(h2d_ck(l - 4, ctx->ev_xused[l % 4]));
    }
    CK(cudaStreamWaitEvent(ctx->sD, ctx->ev_grads[s], 0));
    {
      Timed tl(ctx, 4, 0.0, ctx->sD);
      CK(cudaMemcpyAsync(ctx->layers[l].pack, ctx->ring[s] + ctx->pack_elems, pack_bytes,
                         cudaMemcpyDeviceToHost, ctx->sD));
    }
    CK(cudaEventRecord(ctx->ev_d2h[l], ctx->sD));
    CK(cudaEventRecord(ctx->ev_free[s], ctx->sD));
    d2h += (double)pack_bytes;
    post_task(ctx, l, ctx->ev_d2h[l]);
    const int nl = l - R;  // the next layer that is not resident goes into this slot
    if (nl >= 0) RET(h2d_layer(nl));
  }

  // ---- A16: input gradient to the host, loss
  sf::cast_f32_bf16(ctx->dX, ctx->x0b, T * d, ctx->sC);
  ctx->launches += 1;
  CK(cudaMemcpyAsync(ctx->err_pin, ctx->dev_err, sizeof(int), cudaMemcpyDeviceToHost, ctx->sC));
  CK(cudaEventRecord(ctx->ev_end, ctx->sC));
  CK(cudaStreamWaitEvent(ctx->sD, ctx->ev_end, 0));
  CK(cudaMemcpyAsync(ctx->x0_pin, ctx->x0b, (size_t)T * d * 2, cudaMemcpyDeviceToHost, ctx->sD));
  CK(cudaMemcpyAsync(ctx->loss_pin, ctx->loss_dev, sizeof(float), cudaMemcpyDeviceToHost, ctx->sD));
  CK(cudaEventRecord(ctx->ev_dx0, ctx->sD));
  d2h += (double)T * d * 2 + 4;

  int st = wait_event(ctx, ctx->ev_dx0, "the input gradient copy");
  if (st != SF_OK) {
    wait_tasks(ctx);
    return st;
  }
  const auto t_gpu_done = Clock::now();
  trace(ctx, 7, -9);
  if (*ctx->err_pin != 0) {
    ctx->set_err(*ctx->err_pin == sf::kDevCeBadLabel
                     ? "a label outside the vocabulary reached the cross-entropy kernel (code %d)"
                     : "device wait limit reached in a kernel (code %d)",
                 *ctx->err_pin);
    ctx->poisoned = true;
    wait_tasks(ctx);
    return SF_EDEVICE;
  }
  // embedding gradient and update: a host task like the others
  post_task(ctx, SF_UNIT_EMBED, ctx->ev_dx0);
  if (!ctx->async) {
    st = wait_tasks(ctx);
    if (st != SF_OK) return st;
  }
  ctx->loss = *ctx->loss_pin;
  ctx->have_loss = true;

  // ---- counters
  float ms = 0.f;
  if (cudaEventElapsedTime(&ms, ctx->ev_start, ctx->ev_end) == cudaSuccess) ctx->stats.step_ms = ms;
  for (size_t i = 0; i < ctx->t_used; ++i) {
    float x = 0.f;
    if (cudaEventElapsedTime(&x, ctx->t_ev[2 * i], ctx->t_ev[2 * i + 1]) != cudaSuccess) continue;
    if (ctx->t_kind[i] == 0) {
      ctx->stats.gemm_ms += x;
      ctx->stats.gemm_flops += ctx->t_flops[i];
    } else if (ctx->t_kind[i] == 1) {
      ctx->stats.attn_ms += x;
      ctx->stats.attn_flops += ctx->t_flops[i];
    } else if (ctx->t_kind[i] == 2) {
      ctx->stats.fwd_layer_ms += x / L;
    } else if (ctx->t_kind[i] == 3) {
      ctx->stats.bwd_layer_ms += x / L;
    } else if (ctx->t_kind[i] == 5) {
      ctx->stats.head_ms += x;
    } else {
      ctx->stats.d2h_layer_ms += x / L;
    }
  }
  if (ctx->timing) {
    ctx->stats.compute_ms = L * (ctx->stats.fwd_layer_ms + ctx->stats.bwd_layer_ms) + ctx->stats.head_ms;
    ctx->stats.exposed_ms = std::max(0.0, ctx->stats.step_ms - ctx->stats.compute_ms);
  }
  {
    std::lock_guard<std::mutex> l(ctx->aq_m);
    ctx->stats.update_layer_ms = ctx->upd_layer_n ? ctx->upd_layer_ms / ctx->upd_layer_n : 0.0;
    ctx->upd_layer_ms = 0.0;
    ctx->upd_layer_n = 0;
  }
  cudaGetLastError();
  ctx->stats.h2d_bytes = h2d;
  ctx->stats.d2h_bytes = d2h;
  ctx->stats.host_adam_ms = ctx->adam_ms;
  ctx->stats.host_wait_ms = std::chrono::duration<double, std::milli>(Clock::now() - t_gpu_done).count();
  ctx->stats.kernel_launches = ctx->launches;
  ctx->stats.loss_scale = ctx->f16g ? ctx->lscale : 0.0;
  ctx->stats.skipped_updates = ctx->skipped.load();
  (void)t_host0;
  trace(ctx, 8, -9);
  return SF_OK;
}

}  // namespace

// ==================================================================== C ABI
extern "C" {

size_t sf_unit_numel(const sf_config* cfg, int32_t unit) { return unit_numel_cfg(cfg, unit); }

int sf_init_model(const sf_config* cfg, sf_ctx** out) {
  if (!out) {
    g_init_error = "null output pointer";
    return SF_EINVAL;
  }
  *out = nullptr;
  if (const char* why = validate(cfg)) {
    g_init_error = why;
    return SF_EINVAL;
  }
  sf_ctx* ctx = new (std::nothrow) sf_ctx();
  if (!ctx) {
    g_init_error = "out of host memory";
    return SF_ENOMEM;
  }
  ctx->cfg = *cfg;
  int st;
  try {
    st = init(ctx);
  } catch (...) {
    ctx->set_err("host allocation failed during init");
    st = SF_ENOMEM;
  }
  if (st != SF_OK) {
    g_init_error = ctx->err;
    destroy(ctx);
    delete ctx;
    return st;
  }
  g_init_error.clear();
  *out = ctx;
  return SF_OK;
}

void sf_free(sf_ctx* ctx) {
  if (!ctx) return;
  destroy(ctx);
  delete ctx;
}

const char* sf_last_error(const sf_ctx* ctx) { return ctx ? ctx->err.c_str() : g_init_error.c_str(); }

int sf_load_layer_weights(sf_ctx* ctx, int32_t unit, const float* w, size_t numel) {
  if (!ctx) return SF_EINVAL;
  if (ctx->poisoned) return SF_ESTATE;
  if (int st = wait_tasks(ctx)) return st;
  if (!w || unit_numel_cfg(&ctx->cfg, unit) == 0 || numel != unit_numel_cfg(&ctx->cfg, unit)) {
    ctx->set_err("sf_load_layer_weights: bad unit %d or numel %zu", unit, numel);
    return SF_EINVAL;
  }
  const int64_t n = (int64_t)numel;
  if (unit == SF_UNIT_EMBED) {
    float* master = ctx->E.get();
    ctx->pool->parallel_for(n, 1 << 18, [&](int64_t b, int64_t e) {
      std::memcpy(master + b, w + b, (size_t)(e - b) * 4);
    });
    if (ctx->tied) {  // the LM head streams the embedding's bf16 copy
      uint16_t* p = ctx->lm.pack;
      const float* E = master;
      ctx->pool->parallel_for(n, 1 << 16, [p, E](int64_t b, int64_t e) { refresh_bf16_span(p, E, b, e); });
    }
    zero_moments(ctx, ctx->Em.get(), ctx->Ev.get(), ctx->Em16.get(), ctx->Ev16.get(), 0, n);
    return SF_OK;
  }
  HostUnit* hu = unit >= 0 ? &ctx->layers[unit] : unit == SF_UNIT_LM_HEAD ? &ctx->lm : &ctx->fn;
  float* master = hu->master.get();
  if (unit >= 0) {
    scatter_unit(ctx, w, master);
  } else {
    ctx->pool->parallel_for(n, 1 << 18, [&](int64_t b, int64_t e) {
      std::memcpy(master + b, w + b, (size_t)(e - b) * 4);
    });
  }
  uint16_t* p = hu->pack;
  ctx->pool->parallel_for(hu->elems, 1 << 16, [p, master](int64_t b, int64_t e) {
    refresh_bf16_span(p, master, b, e);
  });
  zero_moments(ctx, hu->m.get(), hu->v.get(), hu->m16.get(), hu->v16.get(), 0, hu->elems);
  return SF_OK;
}

// The Adam moments of a unit, as fp32 in the caller's order (checkpointing).
int sf_get_adam_state(sf_ctx* ctx, int32_t unit, float* m, float* v, size_t numel) {
  if (!ctx || !m || !v || unit_numel_cfg(&ctx->cfg, unit) == 0 || numel != unit_numel_cfg(&ctx->cfg, unit)) {
    if (ctx) ctx->set_err("sf_get_adam_state: bad unit %d or numel %zu", unit, numel);
    return SF_EINVAL;
  }
  if (int st = wait_tasks(ctx)) return st;
  const float *fm, *fv;
  const uint16_t *hm, *hv;
  if (unit == SF_UNIT_EMBED) {
    fm = ctx->Em.get(); fv = ctx->Ev.get(); hm = ctx->Em16.get(); hv = ctx->Ev16.get();
  } else {
    const HostUnit& hu = unit >= 0 ? ctx->layers[unit] : unit == SF_UNIT_LM_HEAD ? ctx->lm : ctx->fn;
    fm = hu.m.get(); fv = hu.v.get(); hm = hu.m16.get(); hv = hu.v16.get();
  }
  auto copy = [&](int64_t src, int64_t dst, int64_t cnt) {
    for (int64_t i = 0; i < cnt; ++i) {
      m[src + i] = fm ? fm[dst + i] : bf2f(hm[dst + i]);
      v[src + i] = fv ? fv[dst + i] : bf2f(hv[dst + i]);
    }
  };
  if (unit >= 0) {
    for (const Seg& s : ctx->segs) copy(s.src, s.dst, s.n);
  } else {
    copy(0, 0, (int64_t)numel);
  }
  return SF_OK;
}

// Restore a unit's Adam moments (bf16 storage rounds them to nearest).
int sf_set_adam_state(sf_ctx* ctx, int32_t unit, const float* m, const float* v, size_t numel) {
  if (!ctx || !m || !v || unit_numel_cfg(&ctx->cfg, unit) == 0 || numel != unit_numel_cfg(&ctx->cfg, unit)) {
    if (ctx) ctx->set_err("sf_set_adam_state: bad unit %d or numel %zu", unit, numel);
    return SF_EINVAL;
  }
  if (ctx->poisoned) return SF_ESTATE;
  if (int st = wait_tasks(ctx)) return st;
  float *fm, *fv;
  uint16_t *hm, *hv;
  if (unit == SF_UNIT_EMBED) {
    fm = ctx->Em.get(); fv = ctx->Ev.get(); hm = ctx->Em16.get(); hv = ctx->Ev16.get();
  } else {
    HostUnit& hu = unit >= 0 ? ctx->layers[unit] : unit == SF_UNIT_LM_HEAD ? ctx->lm : ctx->fn;
    fm = hu.m.get(); fv = hu.v.get(); hm = hu.m16.get(); hv = hu.v16.get();
  }
  auto copy = [&](int64_t src, int64_t dst, int64_t cnt) {
    for (int64_t i = 0; i < cnt; ++i) {
      if (fm) { fm[dst + i] = m[src + i]; fv[dst + i] = v[src + i]; }
      else { hm[dst + i] = f2bf(m[src + i]); hv[dst + i] = f2bf(v[src + i]); }
    }
  };
  if (unit >= 0) {
    for (const Seg& s : ctx->segs) copy(s.src, s.dst, s.n);
  } else {
    copy(0, 0, (int64_t)numel);
  }
  return SF_OK;
}

int sf_get_adam_step(sf_ctx* ctx, int64_t* t) {
  if (!ctx || !t) return SF_EINVAL;
  if (int st = wait_tasks(ctx)) return st;
  *t = ctx->adam_t;
  return SF_OK;
}

int sf_set_adam_step(sf_ctx* ctx, int64_t t) {
  if (!ctx || t < 0) return SF_EINVAL;
  if (int st = wait_tasks(ctx)) return st;
  ctx->adam_t = t;
  return SF_OK;
}

}  // extern "C"

namespace {

// One optimizer step over n_micro micro-batches of batch x seq tokens each:
// the micro-batches run one after another through the ring, their gradients
// are summed on the host, and the update uses the sum (the loss is the mean
// over every valid label of the step).
int train(sf_ctx* ctx, const int32_t* tokens, const int32_t* labels, int32_t n_micro,
          int32_t batch, int32_t seq, const sf_adam* adam, const char* fn) {
  if (!ctx) return SF_EINVAL;
  if (ctx->poisoned) {
    ctx->set_err("context is poisoned by an earlier CUDA error");
    return SF_ESTATE;
  }
  if (!tokens || !labels || n_micro < 1 || batch < 1 || seq < 1 || seq > ctx->Smax ||
      (int64_t)batch * seq > ctx->Tmax) {
    ctx->set_err("%s: bad arguments (micro-batches %d, batch %d, seq %d)", fn, n_micro, batch, seq);
    return SF_EINVAL;
  }
  if (adam && !(adam->lr >= 0.f && adam->beta1 >= 0.f && adam->beta1 < 1.f &&
                adam->beta2 >= 0.f && adam->beta2 < 1.f && adam->eps > 0.f)) {
    ctx->set_err("%s: bad Adam hyper-parameters", fn);
    return SF_EINVAL;
  }
  const int64_t T = (int64_t)batch * seq;
  int64_t n_valid_total = 0;
  for (int i = 0; i < n_micro; ++i) {
    int64_t n = 0;
    RET(check_batch(ctx, tokens + i * T, labels + i * T, T, &n));
    n_valid_total += n;
  }
  if (cudaSetDevice(ctx->cfg.device) != cudaSuccess) {
    ctx->set_err("cudaSetDevice failed");
    return SF_ECUDA;
  }
  if (n_micro > 1) {  // fp32 gradient sums, allocated once
    auto need = [&](HostUnit& hu) { return hu.master && !hu.acc && !new_floats(ctx, hu.acc, hu.elems); };
    bool fail = false;
    for (HostUnit& hu : ctx->layers) fail = fail || need(hu);
    fail = fail || need(ctx->lm) || need(ctx->fn);
    if (fail) return SF_ENOMEM;
  }
  if (ctx->f16g) {  // dynamic loss scale, from the updates skipped so far
    const int64_t sk = ctx->skipped.load();
    if (sk != ctx->skipped_seen) {
      ctx->skipped_seen = sk;
      ctx->lscale = std::max(1.f, ctx->lscale * 0.5f);
      ctx->lgood = 0;
    } else if (ctx->have_loss && ++ctx->lgood >= kScaleWindow) {
      ctx->lscale = std::min(ctx->lscale * 2.f, 16777216.f);
      ctx->lgood = 0;
    }
  }
  int st = SF_OK;
  double loss = 0.0;
  try {
    for (int i = 0; i < n_micro && st == SF_OK; ++i) {
      const int phase = n_micro == 1 ? kOnly : i == 0 ? kFirst : i == n_micro - 1 ? kLast : kMid;
      st = step(ctx, tokens + i * T, labels + i * T, batch, seq, adam, phase, n_valid_total);
      loss += ctx->loss;
    }
  } catch (...) {
    ctx->set_err("host exception in the step");
    ctx->poisoned = true;
    st = SF_ESTATE;
  }
  if (st == SF_OK) {
    ctx->loss = (float)loss;
    ctx->last_accum = n_micro > 1;
  } else if (st != SF_EINVAL) {
    // leave no copy, kernel or host update of this step in flight
    const std::string why = ctx->err;
    cudaStreamSynchronize(ctx->sC);
    cudaStreamSynchronize(ctx->sU);
    cudaStreamSynchronize(ctx->sD);
    wait_tasks(ctx);
    ctx->err = why;
    if (st == SF_ECUDA || st == SF_EDEVICE) ctx->poisoned = true;
  }
  return st;
}

}  // namespace

extern "C" {

int sf_train_step(sf_ctx* ctx, const int32_t* tokens, const int32_t* labels, int32_t batch,
                  int32_t seq, const sf_adam* adam) {
  return train(ctx, tokens, labels, 1, batch, seq, adam, "sf_train_step");
}

int sf_train_step_accum(sf_ctx* ctx, const int32_t* tokens, const int32_t* labels,
                        int32_t n_micro, int32_t batch, int32_t seq, const sf_adam* adam) {
  return train(ctx, tokens, labels, n_micro, batch, seq, adam, "sf_train_step_accum");
}

int sf_get_grads(sf_ctx* ctx, int32_t unit, float* out, size_t numel) {
  if (!ctx || !out || unit_numel_cfg(&ctx->cfg, unit) == 0 || numel != unit_numel_cfg(&ctx->cfg, unit)) {
    if (ctx) ctx->set_err("sf_get_grads: bad unit %d or numel %zu", unit, numel);
    return SF_EINVAL;
  }
  if (int st = wait_tasks(ctx)) return st;
  if (!ctx->cfg.retain_grads || !ctx->have_loss) {
    ctx->set_err("sf_get_grads needs retain_grads = 1 and a finished step");
    return SF_ESTATE;
  }
  if (unit == SF_UNIT_EMBED) {
    std::memcpy(out, ctx->dE.get(), numel * 4);
    return SF_OK;
  }
  const HostUnit& hu = unit >= 0 ? ctx->layers[unit] : (unit == SF_UNIT_LM_HEAD ? ctx->lm : ctx->fn);
  if (ctx->last_accum) {  // the fp32 sum over the step's micro-batches
    const float* g = hu.retained_acc.data();
    if (unit >= 0) {
      for (const Seg& s : ctx->segs) std::memcpy(out + s.src, g + s.dst, (size_t)s.n * 4);
    } else {
      std::memcpy(out, g, numel * 4);
    }
    return SF_OK;
  }
  const uint16_t* g = hu.retained.data();
  const float inv = hu.retained_inv;  // fp16 gradients carry the step's loss scale
  auto cvt = [inv](uint16_t x) { return inv != 0.f ? grd<true>(x, inv) : grd<false>(x, inv); };
  if (unit >= 0) {
    for (const Seg& s : ctx->segs)
      for (int64_t i = 0; i < s.n; ++i) out[s.src + i] = cvt(g[s.dst + i]);
  } else {
    for (size_t i = 0; i < numel; ++i) out[i] = cvt(g[i]);
  }
  return SF_OK;
}

int sf_get_weights(sf_ctx* ctx, int32_t unit, float* out, size_t numel) {
  if (!ctx || !out || unit_numel_cfg(&ctx->cfg, unit) == 0 || numel != unit_numel_cfg(&ctx->cfg, unit)) {
    if (ctx) ctx->set_err("sf_get_weights: bad unit %d or numel %zu", unit, numel);
    return SF_EINVAL;
  }
  if (int st = wait_tasks(ctx)) return st;
  if (unit == SF_UNIT_EMBED) {
    std::memcpy(out, ctx->E.get(), numel * 4);
    return SF_OK;
  }
  const HostUnit& hu = unit >= 0 ? ctx->layers[unit] : (unit == SF_UNIT_LM_HEAD ? ctx->lm : ctx->fn);
  if (unit >= 0) {
    for (const Seg& s : ctx->segs) std::memcpy(out + s.src, hu.master.get() + s.dst, (size_t)s.n * 4);
  } else {
    std::memcpy(out, hu.master.get(), numel * 4);
  }
  return SF_OK;
}

// Host-pointer LM head + cross-entropy for a standalone workload (no model):
// stages the inputs on the device, runs sf_op_lce, returns loss, dh (bf16)
// and dw (fp32).
int sf_lce_step(sf_ctx* ctx, const uint16_t* h, const uint16_t* w, const int32_t* labels,
                int64_t n, int32_t d, int32_t v, int32_t ignore_index, float* loss, uint16_t* dh,
                float* dw) {
  if (!h || !w || !labels || !loss || !dh || !dw || n < 1 || d < 8 || d % 8 || d > 16384 ||
      v < 8 || v % 8)
    return SF_EINVAL;
  std::vector<int32_t> lab((size_t)n);
  int64_t n_valid = 0;
  for (int64_t t = 0; t < n; ++t) {
    const int32_t y = labels[t];
    if (y == ignore_index) {
      lab[t] = SF_IGNORE_INDEX;
    } else if (y < 0 || y >= v) {
      if (ctx) ctx->set_err("sf_lce_step: label %d at row %lld outside [0, %d)", y, (long long)t, v);
      return SF_EINVAL;
    } else {
      lab[t] = y;
      ++n_valid;
    }
  }
  if (ctx && cudaSetDevice(ctx->cfg.device) != cudaSuccess) return SF_ECUDA;
  const int64_t chunk = lce_chunk_rows(n, v);
  const int64_t ws = sf_op_lce_workspace_bytes(n, v, chunk);
  void *dH = nullptr, *dW = nullptr, *dLab = nullptr, *dLoss = nullptr, *dDh = nullptr,
       *dDw = nullptr, *dWs = nullptr, *dDh16 = nullptr;
  cudaStream_t st = nullptr;
  int rc = SF_OK;
  auto alloc = [&](void** ptr, size_t bytes) {
    if (rc == SF_OK && cudaMalloc(ptr, bytes) != cudaSuccess) {
      cudaGetLastError();
      rc = SF_ENOMEM;
    }
  };
  alloc(&dH, (size_t)n * d * 2);
  alloc(&dW, (size_t)v * d * 2);
  alloc(&dLab, (size_t)n * 4);
  alloc(&dLoss, 256);
  alloc(&dDh, (size_t)n * d * 4);
  alloc(&dDw, (size_t)v * d * 4);
  alloc(&dWs, (size_t)ws);
  alloc(&dDh16, (size_t)n * d * 2);
  if (rc == SF_OK && cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) rc = SF_ECUDA;
  if (rc == SF_OK) {
    bool ok = cudaMemcpyAsync(dH, h, (size_t)n * d * 2, cudaMemcpyHostToDevice, st) == cudaSuccess &&
              cudaMemcpyAsync(dW, w, (size_t)v * d * 2, cudaMemcpyHostToDevice, st) == cudaSuccess &&
              cudaMemcpyAsync(dLab, lab.data(), (size_t)n * 4, cudaMemcpyHostToDevice, st) == cudaSuccess;
    if (ok) {
      rc = sf_op_lce(static_cast<const uint16_t*>(dH), static_cast<const uint16_t*>(dW),
                     static_cast<const int32_t*>(dLab), n, d, v, n_valid, chunk, dWs,
                     static_cast<float*>(dLoss), static_cast<float*>(dDh), static_cast<float*>(dDw), st);
    } else {
      rc = SF_ECUDA;
    }
    if (rc == SF_OK) {
      sf::cast_f32_bf16(static_cast<const float*>(dDh), static_cast<bf16*>(dDh16), n * d, st);
      ok = cudaMemcpyAsync(loss, dLoss, 4, cudaMemcpyDeviceToHost, st) == cudaSuccess &&
           cudaMemcpyAsync(dh, dDh16, (size_t)n * d * 2, cudaMemcpyDeviceToHost, st) == cudaSuccess &&
           cudaMemcpyAsync(dw, dDw, (size_t)v * d * 4, cudaMemcpyDeviceToHost, st) == cudaSuccess &&
           cudaStreamSynchronize(st) == cudaSuccess;
      if (!ok) rc = SF_ECUDA;
    }
    if (rc == SF_OK) {
      int32_t e = 0;
      if (sf_op_device_error(&e) != SF_OK) rc = SF_ECUDA;
      else if (e != 0) rc = SF_EDEVICE;
    }
  }
  if (st) {
    cudaStreamSynchronize(st);
    cudaStreamDestroy(st);
  }
  for (void* q : {dH, dW, dLab, dLoss, dDh, dDw, dWs, dDh16})
    if (q) cudaFree(q);
  if (rc != SF_OK && ctx) ctx->set_err("sf_lce_step failed with status %d", rc);
  return rc;
}

int sf_sync(sf_ctx* ctx) {
  if (!ctx) return SF_EINVAL;
  return wait_tasks(ctx);
}

int sf_loss(sf_ctx* ctx, float* out) {
  if (!ctx || !out) return SF_EINVAL;
  if (!ctx->have_loss) {
    ctx->set_err("no step has finished yet");
    return SF_ESTATE;
  }
  *out = ctx->loss;
  return SF_OK;
}

int sf_set_timing(sf_ctx* ctx, int32_t enabled) {
  if (!ctx) return SF_EINVAL;
  ctx->timing = enabled != 0;
  return SF_OK;
}

int sf_get_stats(const sf_ctx* ctx, sf_stats* out) {
  if (!ctx || !out) return SF_EINVAL;
  *out = ctx->stats;
  return SF_OK;
}

int sf_probe_host_bandwidth(int32_t threads, int64_t bytes, double* gbs) {
  if (!gbs || bytes < (1 << 20) || threads < 0) return SF_EINVAL;
  const int nt = threads > 0 ? threads : (int)std::max(1u, std::thread::hardware_concurrency());
  const int64_t n = bytes / 28;
  std::unique_ptr<uint16_t[]> p(new (std::nothrow) uint16_t[n]);
  std::unique_ptr<float[]> w(new (std::nothrow) float[n]), m(new (std::nothrow) float[n]),
      v(new (std::nothrow) float[n]);
  if (!p || !w || !m || !v) return SF_ENOMEM;
  Pool pool(nt);
  uint16_t* pp = p.get();
  float *ww = w.get(), *mm = m.get(), *vv = v.get();
  pool.parallel_for(n, 1 << 16, [pp, ww, mm, vv](int64_t b, int64_t e) {
    for (int64_t i = b; i < e; ++i) {
      pp[i] = 0x3c00;
      ww[i] = 1.f;
      mm[i] = 0.f;
      vv[i] = 0.f;
    }
  });
  double best = 1e30;
  for (int rep = 0; rep < 3; ++rep) {
    const auto t0 = Clock::now();
    pool.parallel_for(n, 1 << 16, [pp, ww, mm, vv](int64_t b, int64_t e) {
      uint16_t* __restrict P = pp;
      float* __restrict W = ww;
      float* __restrict M = mm;
      float* __restrict Vv = vv;
      for (int64_t i = b; i < e; ++i) {
        const float g = bf2f(P[i]);
        M[i] += g;
        Vv[i] += g;
        W[i] += g;
        P[i] = f2bf(W[i]);
      }
    });
    best = std::min(best, std::chrono::duration<double>(Clock::now() - t0).count());
  }
  *gbs = 28.0 * (double)n / best / 1e9;
  return SF_OK;
}

int sf_get_trace(sf_ctx* ctx, sf_trace_event* out, int32_t cap, int32_t* n) {
  if (!ctx || !n || cap < 0 || (cap > 0 && !out)) return SF_EINVAL;
  std::lock_guard<std::mutex> l(ctx->tr_m);
  const size_t sz = ctx->trace.size();
  const size_t take = std::min<size_t>(sz, (size_t)cap);
  for (size_t i = 0; i < take; ++i) out[i] = ctx->trace[(ctx->tr_head + sz - take + i) % sz];
  *n = (int32_t)take;
  ctx->trace.clear();
  ctx->tr_head = 0;
  return SF_OK;
}

int sf_debug_inject(sf_ctx* ctx, int32_t what, int32_t arg) {
  if (!ctx) return SF_EINVAL;
  if (what == 0) {
    ctx->inject_fail_unit = -1000;
    ctx->inject_sleep_ms = 0;
  } else if (what == 1) {
    ctx->inject_fail_unit = arg;
  } else if (what == 2) {
    ctx->inject_sleep_ms = std::max(0, arg);
  } else {
    return SF_EINVAL;
  }
  return SF_OK;
}

}  // extern "C"
