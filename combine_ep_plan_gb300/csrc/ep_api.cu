// ep_api.cu — the C ABI: argument checks, the plan handle, its device
// memory layout and the launch sequences.  Host code only.
//
// A handle owns one stream-ordered device allocation carved by a cursor into
// regions (the symmetric-workspace idea of "Ascend DeepEP MoE Dispatch
// Optimization", section "Workspace 不是一个 Tensor，而是一块地址空间", here a
// single-device window).  Only the control words are cleared, once, when
// the handle is made; every other array is fully written by each plan
// before it is read.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "ep_plan.h"
#include "ep_internal.cuh"

namespace {

constexpr int kAbiVersion = 4;
constexpr long long kDefaultPollLimit = 1ll << 20;

long long g_poll_limit = kDefaultPollLimit;
int g_suppress_tile = -1;

struct Layout {
  size_t off = 0;
  size_t take(size_t bytes) {
    off = (off + 255) & ~static_cast<size_t>(255);
    size_t at = off;
    off += bytes;
    return at;
  }
};

}  // namespace

// Pinned host slots for the counts an asynchronous dispatch reads back.
constexpr int kCountSlots = 8;
constexpr int kCountWords = 4;  // N_recv, N_exp, N_pad, status word

struct ep_handle_s {
  ep::PlanDev dev;
  void* base = nullptr;
  size_t bytes = 0;
  size_t zero_bytes = 0;
  int64_t cap_recv = 0, cap_exp = 0, cap_pad = 0;
  int device = 0;
  // SM budget of the dispatch, combine and backward launches (0 = all)
  int sm_budget = 0;
  // asynchronous calls: communication stream, pinned count slots in use,
  // pending objects not yet waited on
  cudaStream_t comm = nullptr;
  unsigned* counts_host = nullptr;  // [kCountSlots][kCountWords], pinned
  unsigned slots_used = 0;
  int outstanding = 0;
  // per-CTA profile records
  unsigned long long* prof_rec = nullptr;
  long long prof_cap = 0, prof_next = 0;
  unsigned prof_seq = 0;
};

struct ep_pending_s {
  ep_handle_s* h = nullptr;
  cudaStream_t compute = nullptr;
  cudaEvent_t counted = nullptr;  // dispatch: the counts are in the pinned slot
  cudaEvent_t done = nullptr;     // all issued work
  int slot = -1;                  // pinned count slot (dispatch), else -1
  bool have_counts = false;
  unsigned counts[kCountWords] = {0, 0, 0, 0};
};

namespace ep {

int num_sms() {
  static std::atomic<int> cached[64];  // zero-initialised (static storage)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace ep

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ep_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return EP_OK;
  if (e == cudaErrorMemoryAllocation) return EP_ERR_OOM;
  return EP_ERR_CUDA;
}

// Keep freed handle memory in the device's default pool, so that planning
// every step does not return memory to the driver and re-map it.
void keep_pool_memory(int dev) {
  static std::once_flag once[64];
  if (dev < 0 || dev >= 64) return;
  std::call_once(once[dev], [dev] {
    cudaMemPool_t pool;
    if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
      uint64_t thr = UINT64_MAX;
      cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
    }
  });
}

// The launch shape for a handle's kernel: its SM budget, and the next
// profile records when profiling is on.  finish_launch advances the record
// cursor by the CTAs the launch used.
struct Launch {
  ep::LaunchCfg cfg;
  long long ctas = 0;
  unsigned long long* prof_rec = nullptr;
  long long prof_meta = 0;
  explicit Launch(const ep_handle_s* h) {
    cfg.sm_budget = h->sm_budget;
    cfg.ctas = &ctas;
    if (h->prof_rec) {
      const long long at = h->prof_next < h->prof_cap ? h->prof_next : h->prof_cap;
      prof_rec = h->prof_rec + at * ep::kProfWords;
      prof_meta = (static_cast<long long>(h->prof_seq & 0xffffffu) << ep::kProfAvailBits) | (h->prof_cap - at);
    }
  }
  template <class Dev>
  void target(Dev& d) const {
    d.prof_rec = prof_rec;
    d.prof_meta = prof_meta;
  }
};

cudaError_t finish_launch(ep_handle_s* h, const Launch& L, cudaError_t e) {
  if (e == cudaSuccess && h->prof_rec) {
    h->prof_next += L.ctas;
    h->prof_seq = (h->prof_seq + 1u) & 0xffffffu;
  }
  return e;
}

ep_status_t check_shape(int64_t S, int P, int K, int E, int A, int* C) {
  if (S < 1 || P < 1 || P > EP_MAX_RANKS || E < 1 || E > EP_MAX_EXPERTS || K < 1 ||
      K > EP_MAX_TOPK || K > E || A < 1)
    return EP_ERR_INVALID;
  if (E % P != 0) return EP_ERR_INVALID;
  if (*C == 0) *C = static_cast<int>(S < EP_DEFAULT_CHANNELS ? S : EP_DEFAULT_CHANNELS);
  if (*C < 1 || *C > S) return EP_ERR_INVALID;
  const int64_t T = static_cast<int64_t>(P) * S;
  if (T > INT32_MAX / 2) return EP_ERR_INVALID;
  const int64_t worst = T * K + static_cast<int64_t>(E) * (A - 1);
  if (worst >= INT32_MAX) return EP_ERR_INVALID;
  return EP_OK;
}

// Sizes every region and records device pointers relative to `base`.
size_t layout_handle(ep_handle_s* h, char* base) {
  ep::PlanDev& p = h->dev;
  const int64_t T = p.T, P = p.P, E = p.E, K = p.K, C = p.C, A = p.A;
  Layout L;
  // control words (cleared once per handle), then scratch
  const size_t o_ctr = L.take(sizeof(unsigned) * ep::kCtrWords);
  h->zero_bytes = L.off;
  const size_t o_agg = L.take(sizeof(int) * p.num_tiles * (P + E));
  const size_t o_tpre = L.take(sizeof(int) * p.num_tiles * (P + E));
  const size_t o_bits = L.take(sizeof(uint32_t) * p.num_tiles * ep::kTileWords * (P + E));
  const size_t o_wpre = L.take(sizeof(int) * p.num_tiles * ep::kTileWords * (P + E));
  const size_t o_sizes = L.take(sizeof(int) * ep::kSizeWords);
  const size_t o_totals = L.take(sizeof(int) * (P + E));
  const size_t o_trep = L.take(sizeof(int) * ep::kTotRep * (P + E));
  const size_t o_ntpe = L.take(sizeof(int) * P * E);
  // outputs
  const size_t o_ntpr = L.take(sizeof(int) * P * P);
  const size_t o_rpm = L.take(sizeof(int) * P * P);
  const size_t o_cpm = L.take(sizeof(int) * P * P * C);
  const size_t o_rcpm = L.take(sizeof(int) * P * P * C);
  const size_t o_roff = L.take(sizeof(int) * (P + 1));
  const size_t o_eoff = L.take(sizeof(int) * (E + 1));
  const size_t o_poff = L.take(sizeof(int) * (E + 1));
  const size_t o_slot = L.take(sizeof(int) * T * K);
  const size_t o_head = L.take(sizeof(int) * T * P);
  h->cap_recv = T * (K < P ? K : P);
  const size_t o_rsrc = L.take(sizeof(int) * h->cap_recv);
  h->cap_exp = T * K + E * (A - 1);
  const size_t o_esrc = L.take(sizeof(int) * h->cap_exp);
  h->cap_pad = E * (A - 1);
  const size_t o_pads = L.take(sizeof(int) * (h->cap_pad > 0 ? h->cap_pad : 1));
  p.cap_recv = h->cap_recv;
  p.cap_exp = h->cap_exp;
  p.cap_pad = h->cap_pad;
  const size_t o_inr = L.take(sizeof(unsigned char) * T * P);
  const size_t total = L.take(0);
  if (base) {
    p.ctr = reinterpret_cast<unsigned*>(base + o_ctr);
    p.tile_bits = reinterpret_cast<uint32_t*>(base + o_bits);
    p.tile_wpre = reinterpret_cast<int*>(base + o_wpre);
    p.sizes = reinterpret_cast<int*>(base + o_sizes);
    p.totals = reinterpret_cast<int*>(base + o_totals);
    p.totals_rep = reinterpret_cast<int*>(base + o_trep);
    p.ntpe = reinterpret_cast<int*>(base + o_ntpe);
    p.agg = reinterpret_cast<int*>(base + o_agg);
    p.tile_pre = reinterpret_cast<int*>(base + o_tpre);
    p.ntpr = reinterpret_cast<int*>(base + o_ntpr);
    p.rpm = reinterpret_cast<int*>(base + o_rpm);
    p.cpm = reinterpret_cast<int*>(base + o_cpm);
    p.rcpm = reinterpret_cast<int*>(base + o_rcpm);
    p.recv_off = reinterpret_cast<int*>(base + o_roff);
    p.exp_off = reinterpret_cast<int*>(base + o_eoff);
    p.pad_off = reinterpret_cast<int*>(base + o_poff);
    p.slot = reinterpret_cast<int*>(base + o_slot);
    p.send_head = reinterpret_cast<int*>(base + o_head);
    p.recv_src_idx = reinterpret_cast<int*>(base + o_rsrc);
    p.exp_src = reinterpret_cast<int*>(base + o_esrc);
    p.pad_rows = reinterpret_cast<int*>(base + o_pads);
    p.in_rank = reinterpret_cast<unsigned char*>(base + o_inr);
  }
  return total;
}

ep_status_t enqueue_plan(ep_handle_s* h, const int64_t* topk_idx, cudaStream_t stream) {
  h->dev.topk_idx = topk_idx;
  h->dev.poll_limit = g_poll_limit;
  h->dev.suppress_tile = g_suppress_tile;
  Launch L(h);
  L.target(h->dev);
  const cudaError_t e = ep::launch_plan(h->dev, stream, L.cfg);
  return cuda_status(finish_launch(h, L, e));
}

ep_status_t read_status_word(ep_handle_s* h, cudaStream_t stream, bool clear, int sizes[3]) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_status(e);
  unsigned st = 0;
  e = cudaMemcpy(&st, h->dev.ctr + ep::kCtrStatus, sizeof st, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  if (sizes) {
    e = cudaMemcpy(sizes, h->dev.sizes, sizeof(int) * 3, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (clear && st) {
    // after a timed-out wait the barrier counts may be off: reset them too
    const unsigned zeros[ep::kCtrWords] = {};
    if (st & ep::kStTimeout) {
      e = cudaMemcpy(h->dev.ctr, zeros, sizeof zeros, cudaMemcpyHostToDevice);
    } else {
      e = cudaMemcpy(h->dev.ctr + ep::kCtrStatus, zeros, sizeof(unsigned), cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (st & (ep::kStInvalidId | ep::kStDuplicate)) return EP_ERR_INVALID;
  if (st & ep::kStTimeout) return EP_ERR_TIMEOUT;
  if (st & ep::kStCapacity) return EP_ERR_CAPACITY;
  return EP_OK;
}

ep_status_t check_dispatch_args(ep_handle_s* h, const void* x, ep_dtype_t x_dtype, const float* x_scales,
                                int64_t H, ep_dtype_t out_dtype, int flags, void* recv_x, float* recv_scales,
                                int64_t capacity) {
  if (!h || !x || !recv_x || capacity < 0 || H < 8 || H % 8 != 0) return EP_ERR_INVALID;
  if ((flags & ~(EP_DISPATCH_ZERO_PAD | EP_DISPATCH_SCALES_COL_MAJOR)) != 0) return EP_ERR_INVALID;
  if (!aligned(x, 16) || !aligned(recv_x, 16)) return EP_ERR_INVALID;
  if (x_dtype == EP_DTYPE_BF16) {
    if (x_scales) return EP_ERR_INVALID;
    if (out_dtype == EP_DTYPE_BF16) {
      if (recv_scales || (flags & EP_DISPATCH_SCALES_COL_MAJOR)) return EP_ERR_INVALID;
    } else if (out_dtype == EP_DTYPE_FP8_E4M3) {
      if (H % 128 != 0 || !recv_scales || !aligned(recv_scales, 16)) return EP_ERR_INVALID;
    } else {
      return EP_ERR_INVALID;
    }
  } else if (x_dtype == EP_DTYPE_FP8_E4M3) {
    // pre-quantised input is passed through: codes and scales
    if (out_dtype != EP_DTYPE_FP8_E4M3 || H % 128 != 0 || !x_scales || !aligned(x_scales, 4) ||
        !recv_scales || !aligned(recv_scales, 4))
      return EP_ERR_INVALID;
  } else {
    return EP_ERR_INVALID;
  }
  return EP_OK;
}

}  // namespace

extern "C" {

int ep_abi_version(void) { return kAbiVersion; }

const char* ep_status_string(ep_status_t s) {
  switch (s) {
    case EP_OK: return "EP_OK";
    case EP_ERR_INVALID: return "EP_ERR_INVALID: invalid argument or routing data";
    case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY: output capacity below the exact need";
    case EP_ERR_TIMEOUT: return "EP_ERR_TIMEOUT: a bounded device wait gave up";
    case EP_ERR_CUDA: return "EP_ERR_CUDA: CUDA runtime error";
    case EP_ERR_MISMATCH: return "EP_ERR_MISMATCH: cached handle shape mismatch";
    case EP_ERR_OOM: return "EP_ERR_OOM: allocation failed";
  }
  return "EP_ERR_UNKNOWN";
}

ep_status_t ep_plan(const int64_t* topk_idx, int64_t S, int P, int K, int E, int A, int C,
                    ep_stream_t stream_, ep_handle_t* out) {
  if (!out) return EP_ERR_INVALID;
  *out = nullptr;
  if (!topk_idx || !aligned(topk_idx, 8)) return EP_ERR_INVALID;
  ep_status_t st = check_shape(S, P, K, E, A, &C);
  if (st != EP_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  ep_handle_s* h = new (std::nothrow) ep_handle_s();
  if (!h) return EP_ERR_OOM;
  ep::PlanDev& p = h->dev;
  p.S = S;
  p.T = static_cast<int64_t>(P) * S;
  p.P = P;
  p.E = E;
  p.K = K;
  p.A = A;
  p.C = C;
  p.El = E / P;
  p.chunk = (S + C - 1) / C;
  p.num_tiles = static_cast<int>((p.T + ep::kTile - 1) / ep::kTile);
  p.ncols = P + E;
  cudaGetDevice(&h->device);
  keep_pool_memory(h->device);
  h->bytes = layout_handle(h, nullptr);
  cudaError_t e = cudaMallocAsync(&h->base, h->bytes, stream);
  if (e != cudaSuccess) {
    delete h;
    return cuda_status(e);
  }
  layout_handle(h, static_cast<char*>(h->base));
  e = cudaMemsetAsync(h->base, 0, h->zero_bytes, stream);
  st = e == cudaSuccess ? enqueue_plan(h, topk_idx, stream) : cuda_status(e);
  if (st != EP_OK) {
    cudaFreeAsync(h->base, stream);
    delete h;
    return st;
  }
  *out = h;
  return EP_OK;
}

ep_status_t ep_replan(ep_handle_t h, const int64_t* topk_idx, ep_stream_t stream) {
  if (!h || !topk_idx || !aligned(topk_idx, 8)) return EP_ERR_INVALID;
  return enqueue_plan(h, topk_idx, reinterpret_cast<cudaStream_t>(stream));
}

ep_status_t ep_plan_sizes(ep_handle_t h, ep_stream_t stream, int64_t* n_exp, int64_t* n_recv) {
  if (!h) return EP_ERR_INVALID;
  int sizes[3] = {0, 0, 0};
  ep_status_t st = read_status_word(h, reinterpret_cast<cudaStream_t>(stream), false, sizes);
  if (st == EP_ERR_CUDA || st == EP_ERR_OOM) return st;
  if (n_exp) *n_exp = sizes[ep::kSizeExp];
  if (n_recv) *n_recv = sizes[ep::kSizeRecv];
  return st;
}

int64_t ep_worst_expanded_rows(int64_t T, int K, int E, int A) {
  if (T < 0 || K < 1 || E < 1 || A < 1) return -1;
  return T * K + static_cast<int64_t>(E) * (A - 1);
}

ep_status_t ep_dispatch(ep_handle_t h, const void* x, ep_dtype_t x_dtype, const float* x_scales, int64_t H,
                        ep_dtype_t out_dtype, int flags, void* recv_x, float* recv_scales, int64_t capacity,
                        ep_stream_t stream_) {
  ep_status_t st = check_dispatch_args(h, x, x_dtype, x_scales, H, out_dtype, flags, recv_x, recv_scales, capacity);
  if (st != EP_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const bool zero_pad = (flags & EP_DISPATCH_ZERO_PAD) != 0;
  ep::DispatchDev d;
  d.x = x;
  d.x_scales = x_scales;
  d.slot = h->dev.slot;
  d.pad_rows = h->dev.pad_rows;
  d.sizes = h->dev.sizes;
  d.status = h->dev.ctr + ep::kCtrStatus;
  d.out = recv_x;
  d.scales = recv_scales;
  d.T = h->dev.T;
  d.K = h->dev.K;
  d.H = H;
  d.capacity = capacity;
  d.max_pad = zero_pad ? h->cap_pad : 0;
  d.zero_pad = zero_pad ? 1 : 0;
  d.scales_col_major = (flags & EP_DISPATCH_SCALES_COL_MAJOR) ? 1 : 0;
  Launch L(h);
  L.target(d);
  cudaError_t e;
  if (x_dtype == EP_DTYPE_FP8_E4M3)
    e = ep::launch_dispatch_fp8_input(d, stream, L.cfg);
  else if (out_dtype == EP_DTYPE_BF16)
    e = ep::launch_dispatch_bf16(d, stream, L.cfg);
  else
    e = ep::launch_dispatch_fp8(d, stream, L.cfg);
  return cuda_status(finish_launch(h, L, e));
}

ep_status_t ep_dispatch_cached(ep_handle_t h, int E, int A, int64_t S, const void* x, ep_dtype_t x_dtype,
                               const float* x_scales, int64_t H, ep_dtype_t out_dtype, int flags, void* recv_x,
                               float* recv_scales, int64_t capacity, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID;
  if (h->dev.E != E || h->dev.A != A || h->dev.S != S) return EP_ERR_MISMATCH;
  return ep_dispatch(h, x, x_dtype, x_scales, H, out_dtype, flags, recv_x, recv_scales, capacity, stream);
}

ep_status_t ep_dispatch_fresh(const int64_t* topk_idx, int64_t S, int P, int K, int E, int A, int C,
                              const void* x, ep_dtype_t x_dtype, const float* x_scales, int64_t H,
                              ep_dtype_t out_dtype, int flags, void* recv_x, float* recv_scales,
                              int64_t capacity, ep_stream_t stream, ep_handle_t* out) {
  if (!out) return EP_ERR_INVALID;
  *out = nullptr;
  // Check the dispatch arguments before planning so that nothing is enqueued
  // for a call that cannot run (a dummy handle pointer stands in for the plan).
  ep_handle_s probe;
  ep_status_t st = check_dispatch_args(&probe, x, x_dtype, x_scales, H, out_dtype, flags, recv_x, recv_scales,
                                       capacity);
  if (st != EP_OK) return st;
  ep_handle_t h = nullptr;
  st = ep_plan(topk_idx, S, P, K, E, A, C, stream, &h);
  if (st != EP_OK) return st;
  st = ep_dispatch(h, x, x_dtype, x_scales, H, out_dtype, flags, recv_x, recv_scales, capacity, stream);
  if (st != EP_OK) {
    ep_handle_destroy(h, stream);
    return st;
  }
  *out = h;
  return EP_OK;
}

ep_status_t ep_dispatch_metadata(ep_handle_t h, const float* w, float* recv_weights, int32_t* recv_meta,
                                 int64_t capacity, int zero_pad, ep_stream_t stream) {
  if (!h || !w || !recv_weights || !recv_meta || capacity < 0) return EP_ERR_INVALID;
  if (!aligned(w, 4) || !aligned(recv_weights, 4) || !aligned(recv_meta, 4)) return EP_ERR_INVALID;
  ep::MetaDev m;
  m.slot = h->dev.slot;
  m.weights = w;
  m.pad_rows = h->dev.pad_rows;
  m.sizes = h->dev.sizes;
  m.status = h->dev.ctr + ep::kCtrStatus;
  m.recv_weights = recv_weights;
  m.recv_meta = recv_meta;
  m.T = h->dev.T;
  m.K = h->dev.K;
  m.capacity = capacity;
  m.max_pad = zero_pad ? h->cap_pad : 0;
  return cuda_status(ep::launch_dispatch_metadata(m, reinterpret_cast<cudaStream_t>(stream)));
}

ep_status_t ep_combine(ep_handle_t h, const void* y, int64_t y_rows, const float* w, const void* bias,
                       int64_t H, void* out, ep_stream_t stream) {
  if (!h || !y || !w || !out || y_rows < 0 || H < 8 || H % 8 != 0) return EP_ERR_INVALID;
  if (!aligned(y, 16) || !aligned(out, 16) || !aligned(w, 4) || (bias && !aligned(bias, 16)))
    return EP_ERR_INVALID;
  ep::CombineDev c;
  c.y = y;
  c.bias = bias;
  c.slot = h->dev.slot;
  c.weights = w;
  c.status = h->dev.ctr + ep::kCtrStatus;
  c.out = out;
  c.T = h->dev.T;
  c.K = h->dev.K;
  c.H = H;
  c.y_rows = y_rows;
  Launch L(h);
  L.target(c);
  return cuda_status(finish_launch(h, L, ep::launch_combine(c, reinterpret_cast<cudaStream_t>(stream), L.cfg)));
}

ep_status_t ep_dispatch_backward(ep_handle_t h, const void* grad_recv, int64_t grad_rows, int64_t H,
                                 void* grad_x, ep_stream_t stream) {
  if (!h || !grad_recv || !grad_x || grad_rows < 0 || H < 8 || H % 8 != 0) return EP_ERR_INVALID;
  if (!aligned(grad_recv, 16) || !aligned(grad_x, 16)) return EP_ERR_INVALID;
  ep::CombineDev c;
  c.y = grad_recv;
  c.bias = nullptr;
  c.slot = h->dev.slot;
  c.weights = nullptr;  // unit weights: the sum over the token's expanded rows
  c.status = h->dev.ctr + ep::kCtrStatus;
  c.out = grad_x;
  c.T = h->dev.T;
  c.K = h->dev.K;
  c.H = H;
  c.y_rows = grad_rows;
  Launch L(h);
  L.target(c);
  return cuda_status(finish_launch(h, L, ep::launch_combine(c, reinterpret_cast<cudaStream_t>(stream), L.cfg)));
}

ep_status_t ep_combine_backward(ep_handle_t h, const void* grad_out, const void* y, int64_t y_rows,
                                const float* w, int64_t H, int zero_pad, void* grad_y, int64_t grad_y_rows,
                                float* grad_w, ep_stream_t stream) {
  if (!h || !grad_out || !y || !w || !grad_y || !grad_w || y_rows < 0 || grad_y_rows < 0 || H < 8 ||
      H % 8 != 0)
    return EP_ERR_INVALID;
  if (!aligned(grad_out, 16) || !aligned(y, 16) || !aligned(grad_y, 16) || !aligned(w, 4) ||
      !aligned(grad_w, 4))
    return EP_ERR_INVALID;
  ep::CombineBwdDev c;
  c.grad_out = grad_out;
  c.y = y;
  c.slot = h->dev.slot;
  c.weights = w;
  c.pad_rows = h->dev.pad_rows;
  c.sizes = h->dev.sizes;
  c.status = h->dev.ctr + ep::kCtrStatus;
  c.grad_y = grad_y;
  c.grad_w = grad_w;
  c.T = h->dev.T;
  c.K = h->dev.K;
  c.H = H;
  c.y_rows = y_rows;
  c.grad_y_rows = grad_y_rows;
  c.max_pad = zero_pad ? h->cap_pad : 0;
  Launch L(h);  // not profiled: the combine backward has no record variant
  return cuda_status(ep::launch_combine_backward(c, reinterpret_cast<cudaStream_t>(stream), L.cfg));
}

ep_status_t ep_sync_status(ep_handle_t h, ep_stream_t stream) {
  if (!h) return EP_ERR_INVALID;
  return read_status_word(h, reinterpret_cast<cudaStream_t>(stream), true, nullptr);
}

ep_status_t ep_handle_get(ep_handle_t h, ep_field_t f, const void** ptr, int64_t shape[3], int* ndim) {
  if (!h || !ptr || !shape || !ndim) return EP_ERR_INVALID;
  const ep::PlanDev& p = h->dev;
  const int64_t T = p.T, P = p.P, E = p.E, K = p.K, C = p.C;
  shape[0] = shape[1] = shape[2] = 1;
  switch (f) {
    case EP_FIELD_IS_TOKEN_IN_RANK: *ptr = p.in_rank; shape[0] = T; shape[1] = P; *ndim = 2; break;
    case EP_FIELD_SEND_HEAD: *ptr = p.send_head; shape[0] = T; shape[1] = P; *ndim = 2; break;
    case EP_FIELD_NUM_TOKENS_PER_RANK: *ptr = p.ntpr; shape[0] = P; shape[1] = P; *ndim = 2; break;
    case EP_FIELD_NUM_TOKENS_PER_EXPERT: *ptr = p.ntpe; shape[0] = P; shape[1] = E; *ndim = 2; break;
    case EP_FIELD_EXPERT_COUNTS: *ptr = p.totals + P; shape[0] = E; *ndim = 1; break;
    case EP_FIELD_NUM_RECV: *ptr = p.totals; shape[0] = P; *ndim = 1; break;
    case EP_FIELD_RANK_PREFIX: *ptr = p.rpm; shape[0] = P; shape[1] = P; *ndim = 2; break;
    case EP_FIELD_CHANNEL_PREFIX: *ptr = p.cpm; shape[0] = P; shape[1] = P; shape[2] = C; *ndim = 3; break;
    case EP_FIELD_RECV_CHANNEL_PREFIX: *ptr = p.rcpm; shape[0] = P; shape[1] = P; shape[2] = C; *ndim = 3; break;
    case EP_FIELD_RECV_OFFSETS: *ptr = p.recv_off; shape[0] = P + 1; *ndim = 1; break;
    case EP_FIELD_RECV_SRC_IDX: *ptr = p.recv_src_idx; shape[0] = h->cap_recv; *ndim = 1; break;
    case EP_FIELD_EXPERT_OFFSETS: *ptr = p.exp_off; shape[0] = E + 1; *ndim = 1; break;
    case EP_FIELD_SLOT: *ptr = p.slot; shape[0] = T; shape[1] = K; *ndim = 2; break;
    case EP_FIELD_EXP_SRC: *ptr = p.exp_src; shape[0] = h->cap_exp; *ndim = 1; break;
    case EP_FIELD_PAD_ROWS: *ptr = p.pad_rows; shape[0] = h->cap_pad; *ndim = 1; break;
    default: return EP_ERR_INVALID;
  }
  return EP_OK;
}

ep_status_t ep_handle_info(ep_handle_t h, int64_t* S, int* P, int* K, int* E, int* A, int* C) {
  if (!h) return EP_ERR_INVALID;
  if (S) *S = h->dev.S;
  if (P) *P = h->dev.P;
  if (K) *K = h->dev.K;
  if (E) *E = h->dev.E;
  if (A) *A = h->dev.A;
  if (C) *C = h->dev.C;
  return EP_OK;
}

ep_status_t ep_handle_destroy(ep_handle_t h, ep_stream_t stream_) {
  if (!h) return EP_ERR_INVALID;
  if (h->outstanding > 0) return EP_ERR_INVALID;  // wait on its pending calls first
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaError_t e = cudaSuccess;
  if (h->comm) {
    // the communication stream's work ends before the memory is released
    e = cudaStreamSynchronize(h->comm);
    cudaStreamDestroy(h->comm);
    if (h->counts_host) cudaFreeHost(h->counts_host);
  }
  if (h->base) {
    const cudaError_t e2 = cudaFreeAsync(h->base, stream);
    if (e == cudaSuccess) e = e2;
  }
  delete h;
  return cuda_status(e);
}

ep_status_t ep_set_num_sms(ep_handle_t h, int num_sms) {
  if (!h || num_sms < 0) return EP_ERR_INVALID;
  h->sm_budget = num_sms >= ep::num_sms() ? 0 : num_sms;
  return EP_OK;
}

ep_status_t ep_profile_begin(ep_handle_t h, uint64_t* records, int64_t capacity) {
  if (!h || !records || capacity < 1 || capacity >= (1ll << ep::kProfAvailBits) || !aligned(records, 8))
    return EP_ERR_INVALID;
  h->prof_rec = reinterpret_cast<unsigned long long*>(records);
  h->prof_cap = capacity;
  h->prof_next = 0;
  h->prof_seq = 0;
  return EP_OK;
}

ep_status_t ep_profile_end(ep_handle_t h, int64_t* written, int64_t* dropped) {
  if (!h || !h->prof_rec) return EP_ERR_INVALID;
  const long long n = h->prof_next;
  if (written) *written = n < h->prof_cap ? n : h->prof_cap;
  if (dropped) *dropped = n > h->prof_cap ? n - h->prof_cap : 0;
  h->prof_rec = nullptr;
  h->prof_cap = h->prof_next = 0;
  return EP_OK;
}

}  // extern "C"

namespace {

// The communication stream and the pinned count slots, made on first use.
ep_status_t ensure_comm(ep_handle_s* h) {
  if (h->comm) return EP_OK;
  int cur = 0;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_status(e);
  if (cur != h->device) return EP_ERR_INVALID;
  e = cudaHostAlloc(reinterpret_cast<void**>(&h->counts_host), sizeof(unsigned) * kCountSlots * kCountWords,
                    cudaHostAllocDefault);
  if (e != cudaSuccess) return cuda_status(e);
  std::memset(h->counts_host, 0, sizeof(unsigned) * kCountSlots * kCountWords);
  e = cudaStreamCreateWithFlags(&h->comm, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    cudaFreeHost(h->counts_host);
    h->counts_host = nullptr;
    h->comm = nullptr;
    return cuda_status(e);
  }
  return EP_OK;
}

// A pending object with its events; the communication stream is ordered
// after `previous`, or after everything enqueued on `compute` so far.
ep_status_t begin_async(ep_handle_s* h, cudaStream_t compute, cudaEvent_t previous, bool counts,
                        ep_pending_s** out) {
  ep_status_t st = ensure_comm(h);
  if (st != EP_OK) return st;
  int slot = -1;
  if (counts) {
    for (int i = 0; i < kCountSlots; ++i)
      if (!(h->slots_used & (1u << i))) {
        slot = i;
        break;
      }
    if (slot < 0) return EP_ERR_CAPACITY;  // too many dispatches in flight
  }
  ep_pending_s* p = new (std::nothrow) ep_pending_s();
  if (!p) return EP_ERR_OOM;
  p->h = h;
  p->compute = compute;
  p->slot = slot;
  cudaError_t e = cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming);
  if (e == cudaSuccess && counts) e = cudaEventCreateWithFlags(&p->counted, cudaEventDisableTiming);
  cudaEvent_t ready = previous;
  if (e == cudaSuccess && !ready) {
    e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
    if (e == cudaSuccess) {
      e = cudaEventRecord(ready, compute);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(h->comm, ready, 0);
      cudaEventDestroy(ready);  // released once the wait no longer needs it
    }
  } else if (e == cudaSuccess) {
    e = cudaStreamWaitEvent(h->comm, ready, 0);
  }
  if (e != cudaSuccess) {
    if (p->done) cudaEventDestroy(p->done);
    if (p->counted) cudaEventDestroy(p->counted);
    delete p;
    return cuda_status(e);
  }
  if (slot >= 0) h->slots_used |= 1u << slot;
  ++h->outstanding;
  *out = p;
  return EP_OK;
}

// Copies the sizes and the status word to the pending object's pinned slot,
// on the communication stream, and marks it.
cudaError_t enqueue_counts(ep_pending_s* p) {
  ep_handle_s* h = p->h;
  unsigned* dst = h->counts_host + p->slot * kCountWords;
  cudaError_t e = cudaMemcpyAsync(dst, h->dev.sizes, sizeof(unsigned) * 3, cudaMemcpyDeviceToHost, h->comm);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(dst + 3, h->dev.ctr + ep::kCtrStatus, sizeof(unsigned), cudaMemcpyDeviceToHost, h->comm);
  if (e == cudaSuccess) e = cudaEventRecord(p->counted, h->comm);
  return e;
}

// The host side of the epilogue: wait for the counts, keep them.
ep_status_t read_counts(ep_pending_s* p) {
  if (p->have_counts || p->slot < 0) return EP_OK;
  cudaError_t e = cudaEventSynchronize(p->counted);
  if (e != cudaSuccess) return cuda_status(e);
  std::memcpy(p->counts, p->h->counts_host + p->slot * kCountWords, sizeof p->counts);
  p->have_counts = true;
  return EP_OK;
}

ep_status_t status_of(unsigned st) {
  if (st & (ep::kStInvalidId | ep::kStDuplicate)) return EP_ERR_INVALID;
  if (st & ep::kStTimeout) return EP_ERR_TIMEOUT;
  if (st & ep::kStCapacity) return EP_ERR_CAPACITY;
  return EP_OK;
}

void release_pending(ep_pending_s* p) {
  ep_handle_s* h = p->h;
  if (p->slot >= 0) h->slots_used &= ~(1u << p->slot);
  --h->outstanding;
  if (p->counted) cudaEventDestroy(p->counted);
  if (p->done) cudaEventDestroy(p->done);
  delete p;
}

}  // namespace

extern "C" {

ep_status_t ep_dispatch_async(ep_handle_t h, const int64_t* topk_idx, const void* x, ep_dtype_t x_dtype,
                              const float* x_scales, int64_t H, ep_dtype_t out_dtype, int flags, void* recv_x,
                              float* recv_scales, int64_t capacity, ep_stream_t compute_, ep_event_t previous,
                              int defer_epilogue, ep_pending_t* out) {
  if (!out) return EP_ERR_INVALID;
  *out = nullptr;
  ep_status_t st = check_dispatch_args(h, x, x_dtype, x_scales, H, out_dtype, flags, recv_x, recv_scales, capacity);
  if (st != EP_OK) return st;
  if (topk_idx && !aligned(topk_idx, 8)) return EP_ERR_INVALID;
  ep_pending_s* p = nullptr;
  st = begin_async(h, reinterpret_cast<cudaStream_t>(compute_), reinterpret_cast<cudaEvent_t>(previous), true, &p);
  if (st != EP_OK) return st;
  ep_stream_t comm = reinterpret_cast<ep_stream_t>(h->comm);
  if (topk_idx) st = enqueue_plan(h, topk_idx, h->comm);
  if (st == EP_OK) st = cuda_status(enqueue_counts(p));
  if (st == EP_OK) st = ep_dispatch(h, x, x_dtype, x_scales, H, out_dtype, flags, recv_x, recv_scales, capacity, comm);
  if (st == EP_OK) st = cuda_status(cudaEventRecord(p->done, h->comm));
  if (st == EP_OK && !defer_epilogue) st = read_counts(p);
  if (st != EP_OK) {
    cudaStreamSynchronize(h->comm);
    release_pending(p);
    return st;
  }
  *out = p;
  return EP_OK;
}

ep_status_t ep_combine_async(ep_handle_t h, const void* y, int64_t y_rows, const float* w, const void* bias,
                             int64_t H, void* out_dev, ep_stream_t compute_, ep_event_t previous,
                             int defer_epilogue, ep_pending_t* out) {
  (void)defer_epilogue;  // a combine has no host-side epilogue: both forms return at once
  if (!out) return EP_ERR_INVALID;
  *out = nullptr;
  if (!h || !y || !w || !out_dev || y_rows < 0 || H < 8 || H % 8 != 0) return EP_ERR_INVALID;
  if (!aligned(y, 16) || !aligned(out_dev, 16) || !aligned(w, 4) || (bias && !aligned(bias, 16)))
    return EP_ERR_INVALID;
  ep_pending_s* p = nullptr;
  ep_status_t st =
      begin_async(h, reinterpret_cast<cudaStream_t>(compute_), reinterpret_cast<cudaEvent_t>(previous), false, &p);
  if (st != EP_OK) return st;
  st = ep_combine(h, y, y_rows, w, bias, H, out_dev, reinterpret_cast<ep_stream_t>(h->comm));
  if (st == EP_OK) st = cuda_status(cudaEventRecord(p->done, h->comm));
  if (st != EP_OK) {
    cudaStreamSynchronize(h->comm);
    release_pending(p);
    return st;
  }
  *out = p;
  return EP_OK;
}

ep_status_t ep_pending_wait(ep_pending_t p, int64_t* n_exp, int64_t* n_recv) {
  if (!p) return EP_ERR_INVALID;
  ep_status_t st = EP_OK;
  if ((n_exp || n_recv) && p->slot >= 0) st = read_counts(p);
  const cudaError_t e = cudaStreamWaitEvent(p->compute, p->done, 0);
  if (st == EP_OK) st = cuda_status(e);
  if (st == EP_OK && p->have_counts) {
    if (n_exp) *n_exp = static_cast<int>(p->counts[ep::kSizeExp]);
    if (n_recv) *n_recv = static_cast<int>(p->counts[ep::kSizeRecv]);
    st = status_of(p->counts[3]);
  } else {
    if (n_exp) *n_exp = 0;
    if (n_recv) *n_recv = 0;
  }
  release_pending(p);
  return st;
}

void ep_debug_set_plan_wait(int64_t poll_limit, int suppress_tile) {
  g_poll_limit = poll_limit > 0 ? poll_limit : kDefaultPollLimit;
  g_suppress_tile = suppress_tile;
}

}  // extern "C"
