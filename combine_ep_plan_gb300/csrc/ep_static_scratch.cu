// ep_static_scratch.cu — ep_plan_static_scratch: the routing plan for callers
// that cannot allocate device memory.
//
// ep_plan keeps its plan arrays and its scratch (per-tile counts and
// prefixes, tile bit matrices, barrier counts, status word, column totals) in
// one allocation that it makes per handle.  Some callers cannot allocate at that point: a serving
// runtime that reserved all device memory for its own arena at start-up, or a
// latency-critical loop where an allocation may block on the device or fail
// under fragmentation.  This entry point runs the same plan kernels, writes
// the plan into arrays the caller owns, and keeps its scratch in a fixed
// file-scope device array instead.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "ep_plan.h"
#include "ep_internal.cuh"

namespace {

// The scratch of every call on a device.  Each device that loads the library
// holds these EP_STATIC_SCRATCH_BYTES until the process exits.
__device__ __align__(256) unsigned char g_plan_scratch[EP_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct DeviceScratch {
  std::mutex mu;
  std::atomic<void*> ptr{nullptr};
};
DeviceScratch g_scratch[kMaxDevices];

// Device address of g_plan_scratch on the current device.  In host code the
// array's name only stands in for the symbol; the address a kernel may use
// comes from cudaGetSymbolAddress, looked up with that device current on the
// first successful call of the entry point on it and kept from then on.  A
// failed lookup is not kept: the next call tries again (and the runtime's
// last-error slot is cleared, so that it does not surface in a later,
// unrelated launch check).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceScratch& s = g_scratch[dev];
  void* p = s.ptr.load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(s.mu);
    p = s.ptr.load(std::memory_order_relaxed);
    if (p == nullptr) {
      e = cudaGetSymbolAddress(&p, g_plan_scratch);
      if (e != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
      }
      s.ptr.store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

bool aligned4(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) % 4) == 0; }

ep_status_t to_status(cudaError_t e) {
  if (e == cudaSuccess) return EP_OK;
  return e == cudaErrorMemoryAllocation ? EP_ERR_OOM : EP_ERR_CUDA;
}

}  // namespace

extern "C" ep_status_t ep_plan_static_scratch(const int64_t* topk_idx, int64_t S, int P, int K, int E,
                                              int A, int C, const ep_plan_buffers_t* out,
                                              ep_stream_t stream_) {
  // Shape checks: the same limits as ep_plan.
  if (!topk_idx || (reinterpret_cast<uintptr_t>(topk_idx) % 8) != 0 || !out) return EP_ERR_INVALID;
  if (S < 1 || P < 1 || P > EP_MAX_RANKS || E < 1 || E > EP_MAX_EXPERTS || K < 1 || K > EP_MAX_TOPK ||
      K > E || A < 1 || E % P != 0)
    return EP_ERR_INVALID;
  if (C == 0) C = static_cast<int>(S < EP_DEFAULT_CHANNELS ? S : EP_DEFAULT_CHANNELS);
  if (C < 1 || C > S) return EP_ERR_INVALID;
  const int64_t T = static_cast<int64_t>(P) * S;
  if (T > INT32_MAX / 2 || T * K + static_cast<int64_t>(E) * (A - 1) >= INT32_MAX) return EP_ERR_INVALID;
  if (!out->is_token_in_rank || !aligned4(out->send_head) || !aligned4(out->num_tokens_per_rank) ||
      !aligned4(out->num_tokens_per_expert) || !aligned4(out->expert_counts) || !aligned4(out->num_recv) ||
      !aligned4(out->rank_prefix) || !aligned4(out->channel_prefix) || !aligned4(out->recv_channel_prefix) ||
      !aligned4(out->recv_offsets) || !aligned4(out->recv_src_idx) || !aligned4(out->expert_offsets) ||
      !aligned4(out->slot) || !aligned4(out->exp_src) || !aligned4(out->pad_rows) || !aligned4(out->info))
    return EP_ERR_INVALID;

  // Scratch layout: control words, per-tile counts and prefixes, tile bit matrices
  // and word prefixes, sizes, column totals, padding offsets.
  const int ncols = P + E;
  const int num_tiles = static_cast<int>((T + ep::kTile - 1) / ep::kTile);
  const size_t tile_words = static_cast<size_t>(num_tiles) * ep::kTileWords * ncols;
  const size_t o_ctr = 0;
  const size_t cleared = sizeof(unsigned) * ep::kCtrWords;
  const size_t o_agg = round256(cleared);
  const size_t o_tpre = round256(o_agg + sizeof(int) * static_cast<size_t>(num_tiles) * ncols);
  const size_t o_bits = round256(o_tpre + sizeof(int) * static_cast<size_t>(num_tiles) * ncols);
  const size_t o_wpre = round256(o_bits + sizeof(uint32_t) * tile_words);
  const size_t o_sizes = round256(o_wpre + sizeof(int) * tile_words);
  const size_t o_totals = round256(o_sizes + sizeof(int) * ep::kSizeWords);
  const size_t o_trep = round256(o_totals + sizeof(int) * ncols);
  const size_t o_padoff = round256(o_trep + sizeof(int) * ep::kTotRep * ncols);
  if (o_padoff + sizeof(int) * (E + 1) > EP_STATIC_SCRATCH_BYTES) return EP_ERR_CAPACITY;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  void* base_v = nullptr;
  cudaError_t e = scratch_address(&base_v);
  if (e != cudaSuccess) return to_status(e);
  char* base = static_cast<char*>(base_v);

  // Every call shares the scratch and finds the last call's contents in it:
  // clear the control words; the rest is written before it is read.
  e = cudaMemsetAsync(base, 0, cleared, stream);
  if (e != cudaSuccess) return to_status(e);

  ep::PlanDev p{};
  p.S = S;
  p.T = T;
  p.P = P;
  p.E = E;
  p.K = K;
  p.A = A;
  p.C = C;
  p.El = E / P;
  p.chunk = (S + C - 1) / C;
  p.num_tiles = num_tiles;
  p.ncols = ncols;
  p.topk_idx = topk_idx;
  p.ctr = reinterpret_cast<unsigned*>(base + o_ctr);
  p.agg = reinterpret_cast<int*>(base + o_agg);
  p.tile_pre = reinterpret_cast<int*>(base + o_tpre);
  p.tile_bits = reinterpret_cast<uint32_t*>(base + o_bits);
  p.tile_wpre = reinterpret_cast<int*>(base + o_wpre);
  p.sizes = reinterpret_cast<int*>(base + o_sizes);
  p.totals = reinterpret_cast<int*>(base + o_totals);
  p.totals_rep = reinterpret_cast<int*>(base + o_trep);
  p.ntpe = out->num_tokens_per_expert;
  p.ntpr = out->num_tokens_per_rank;
  p.rpm = out->rank_prefix;
  p.cpm = out->channel_prefix;
  p.rcpm = out->recv_channel_prefix;
  p.recv_off = out->recv_offsets;
  p.exp_off = out->expert_offsets;
  p.pad_off = reinterpret_cast<int*>(base + o_padoff);
  p.slot = out->slot;
  p.send_head = out->send_head;
  p.recv_src_idx = out->recv_src_idx;
  p.exp_src = out->exp_src;
  p.pad_rows = out->pad_rows;
  p.in_rank = out->is_token_in_rank;
  p.cap_recv = T * (K < P ? K : P);
  p.cap_exp = T * K + static_cast<int64_t>(E) * (A - 1);
  p.cap_pad = static_cast<int64_t>(E) * (A - 1);
  p.poll_limit = 1ll << 20;
  p.suppress_tile = -1;

  e = ep::launch_plan(p, stream, ep::LaunchCfg{});
  if (e != cudaSuccess) return to_status(e);

  // Totals, sizes and the status word leave the scratch for the caller.
  e = cudaMemcpyAsync(out->num_recv, p.totals, sizeof(int) * P, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(out->expert_counts, p.totals + P, sizeof(int) * E, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(out->info, p.sizes, sizeof(int) * 3, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(out->info + 3, p.ctr + ep::kCtrStatus, sizeof(int), cudaMemcpyDeviceToDevice, stream);
  return to_status(e);
}
