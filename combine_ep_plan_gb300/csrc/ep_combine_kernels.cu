// ep_combine_kernels.cu — the weighted combine on sm_103a.
//
// One warp per token, grid-stride.  Each lane owns 16-byte vectors (8 bf16)
// of the hidden dimension; for a chunk of kUnroll vectors it issues the loads
// of all K expert rows first (K*kUnroll independent 16-byte loads in flight),
// then accumulates in fp32 in fixed slot order k = 0..K-1 with fmaf and
// rounds once to bf16 (TileLang tutorial ch. 38, §4.5: widen to fp32,
// accumulate, round to nearest even).  Rows of unused slots are not read.
#include <cuda_bf16.h>

#include "ep_internal.cuh"

namespace ep {
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
  return *reinterpret_cast<unsigned*>(&h);
}

// Work item = (token, column chunk of 32*U vectors), so that every warp gets
// many small items and the kernel has no long tail.  PROF: the same kernel,
// plus a per-CTA record (items, payload bytes, start and end).
template <int KMAX, int U, int MINB, bool PROF>
__global__ void __launch_bounds__(256, MINB) ep_combine_kernel(CombineDev c) {
  pdl_wait();
  unsigned long long t0 = 0, units = 0, bytes = 0;
  if (PROF && threadIdx.x == 0) t0 = prof_now();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t hv = c.H / 8;
  constexpr int kChunk = 32 * U;
  const int64_t chunks = (hv + kChunk - 1) / kChunk;
  const int64_t n_items = c.T * chunks;
  const uint4* y = static_cast<const uint4*>(c.y);
  uint4* out = static_cast<uint4*>(c.out);

  for (int64_t item = warp; item < n_items; item += nwarps) {
    const int64_t g = item / chunks;
    const int64_t v0 = (item - g * chunks) * kChunk;
    int my_row = -1;
    float my_w = 0.0f;
    if (lane < c.K) {
      my_row = c.slot[g * c.K + lane];
      my_w = c.weights ? c.weights[g * c.K + lane] : 1.0f;
      if (my_row >= c.y_rows) {
        atomicOr(c.status, kStCapacity);
        my_row = -1;
      }
    }
    int row[KMAX];
    float wk[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      row[k] = __shfl_sync(0xffffffffu, my_row, k);
      wk[k] = __shfl_sync(0xffffffffu, my_w, k);
      if (k >= c.K) row[k] = -1;
    }
    if (PROF) {  // rows read, the bias row, the output row
      const int64_t item_bytes = 16 * (hv - v0 < kChunk ? hv - v0 : kChunk);
      int n = 1 + (c.bias ? 1 : 0);
#pragma unroll
      for (int k = 0; k < KMAX; ++k) n += row[k] >= 0;
      ++units;
      bytes += n * item_bytes;
    }
    uint4 buf[KMAX][U];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const uint4* src = y + static_cast<int64_t>(row[k] < 0 ? 0 : row[k]) * hv;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t v = v0 + u * 32 + lane;
        if (row[k] >= 0 && v < hv) buf[k][u] = ld_stream(src + v);
      }
    }
    uint4 bv[U];
    if (c.bias) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t v = v0 + u * 32 + lane;
        if (v < hv) bv[u] = ld_stream(static_cast<const uint4*>(c.bias) + g * hv + v);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + u * 32 + lane;
      if (v >= hv) continue;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (row[k] < 0) continue;
        const unsigned wv[4] = {buf[k][u].x, buf[k][u].y, buf[k][u].z, buf[k][u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(wk[k], __uint_as_float(wv[i] << 16), acc[2 * i]);
          acc[2 * i + 1] = fmaf(wk[k], __uint_as_float(wv[i] & 0xffff0000u), acc[2 * i + 1]);
        }
      }
      if (c.bias) {  // the fused residual / shared-expert row, added once in fp32
        const unsigned bw[4] = {bv[u].x, bv[u].y, bv[u].z, bv[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(bw[i] << 16));
          acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(bw[i] & 0xffff0000u));
        }
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      out[g * hv + v] = o;
    }
  }
  if (PROF) prof_cta_end(c, c.weights ? kProfCombine : kProfDispatchBackward, t0, 0, 0, 0, units, bytes);
}

// One full wave of resident CTAs (grid-stride inside); under an SM budget,
// that many SMs' worth.
template <typename Kernel>
int resident_grid(Kernel kernel, int threads) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return per_sm * num_sms();
}

// 0: one resident wave; otherwise this many CTAs per SM.
#ifndef EP_COMBINE_CTAS_PER_SM
#define EP_COMBINE_CTAS_PER_SM 0
#endif

template <int KMAX, int U, int MINB, bool PROF>
cudaError_t launch_kp(const CombineDev& c, cudaStream_t stream, const LaunchCfg& cfg) {
  // one resident wave, cached per host thread for the last device it was
  // asked for
  thread_local int full = 0, full_dev = -1;
  auto kernel = ep_combine_kernel<KMAX, U, MINB, PROF>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  if (full == 0 || dev != full_dev) {
    full = EP_COMBINE_CTAS_PER_SM > 0 ? EP_COMBINE_CTAS_PER_SM * num_sms() : resident_grid(kernel, 256);
    full_dev = dev;
  }
  long long grid = full;
  const long long cap = budget_cap(kernel, 256, 0, cfg.sm_budget);
  if (cap > 0 && grid > cap) grid = cap;
  const cudaError_t e = launch_pdl(kernel, static_cast<unsigned>(grid), 256, stream, c);
  if (cfg.ctas) *cfg.ctas = grid;
  return e;
}

template <int KMAX, int U, int MINB>
cudaError_t launch_k(const CombineDev& c, cudaStream_t stream, const LaunchCfg& cfg) {
  return c.prof_rec ? launch_kp<KMAX, U, MINB, true>(c, stream, cfg) : launch_kp<KMAX, U, MINB, false>(c, stream, cfg);
}

// Combine backward, one CTA of 128 threads per token: grad_out[g] is read
// once; for each slot k the row y[slot] is read for the dot product grad_w =
// <grad_out[g], y[slot]> and grad_y[slot] = bf16(w * grad_out[g]) is written.
// The dot products are summed per thread over its vectors, then by a fixed
// shuffle tree per warp and over the four warps in order: deterministic.
// Items beyond T zero the padding rows of grad_y.  One CTA per token, and at
// most kBwdPadCtas more for the padding rows (the grid covers T plus at most
// that many of the E*(A-1) possible ones); CTAs loop over the items beyond
// their first, and an SM budget caps the grid the same way.
// CTAs of the combine backward beyond one per token: they take the padding
// rows in turn (a grid of T + E*(A-1) left most of those CTAs without a row).
constexpr long long kBwdPadCtas = 1024;

template <int KMAX>
__device__ __forceinline__ void combine_backward_item(const CombineBwdDev& c, int64_t item) {
  constexpr int kWarps = 4;
  __shared__ int s_row[KMAX];
  __shared__ float s_w[KMAX];
  __shared__ float s_dot[kWarps][KMAX];
  const int64_t hv = c.H / 8;
  uint4* gy = static_cast<uint4*>(c.grad_y);
  const unsigned long long pol = l2_evict_first_policy();  // the grad_y rows
  if (item >= c.T) {
    const int64_t pi = item - c.T;
    if (pi >= c.sizes[kSizePad] || pi >= c.max_pad) return;
    const int r = c.pad_rows[pi];
    if (r < 0 || r >= c.grad_y_rows) {
      if (threadIdx.x == 0) atomicOr(c.status, kStCapacity);
      return;
    }
    for (int64_t v = threadIdx.x; v < hv; v += blockDim.x)
      st_evict_first(gy + static_cast<int64_t>(r) * hv + v, make_uint4(0u, 0u, 0u, 0u), pol);
    return;
  }
  const int64_t g = item;
  if (threadIdx.x < KMAX) {
    const int k = threadIdx.x;
    int r = -1;
    float wk = 0.0f;
    if (k < c.K) {
      r = c.slot[g * c.K + k];
      wk = c.weights[g * c.K + k];
      if (r >= c.y_rows || r >= c.grad_y_rows) {
        atomicOr(c.status, kStCapacity);
        r = -1;
      }
    }
    s_row[k] = r;
    s_w[k] = wk;
  }
  __syncthreads();
  int row[KMAX];
  float wk[KMAX], dot[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    row[k] = s_row[k];
    wk[k] = s_w[k];
    dot[k] = 0.0f;
  }
  const uint4* go_row = static_cast<const uint4*>(c.grad_out) + g * hv;
  const uint4* y = static_cast<const uint4*>(c.y);
  for (int64_t v = threadIdx.x; v < hv; v += blockDim.x) {
    const uint4 go = ld_stream(go_row + v);
    uint4 yv[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (row[k] >= 0) yv[k] = ld_stream(y + static_cast<int64_t>(row[k]) * hv + v);
    const unsigned gw[4] = {go.x, go.y, go.z, go.w};
    float gof[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      gof[2 * i] = __uint_as_float(gw[i] << 16);
      gof[2 * i + 1] = __uint_as_float(gw[i] & 0xffff0000u);
    }
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (row[k] < 0) continue;
      const unsigned yw[4] = {yv[k].x, yv[k].y, yv[k].z, yv[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dot[k] = fmaf(gof[2 * i], __uint_as_float(yw[i] << 16), dot[k]);
        dot[k] = fmaf(gof[2 * i + 1], __uint_as_float(yw[i] & 0xffff0000u), dot[k]);
      }
      uint4 o;
      o.x = pack_bf16x2(__fmul_rn(wk[k], gof[0]), __fmul_rn(wk[k], gof[1]));
      o.y = pack_bf16x2(__fmul_rn(wk[k], gof[2]), __fmul_rn(wk[k], gof[3]));
      o.z = pack_bf16x2(__fmul_rn(wk[k], gof[4]), __fmul_rn(wk[k], gof[5]));
      o.w = pack_bf16x2(__fmul_rn(wk[k], gof[6]), __fmul_rn(wk[k], gof[7]));
      st_evict_first(gy + static_cast<int64_t>(row[k]) * hv + v, o, pol);
    }
  }
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    float d = dot[k];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if (lane == 0) s_dot[warp][k] = d;
  }
  __syncthreads();
  if (threadIdx.x < c.K) {
    const int k = threadIdx.x;
    float d = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) d += s_dot[w][k];
    c.grad_w[g * c.K + k] = row[k] >= 0 ? d : 0.0f;
  }
}

// At least six CTAs of 128 threads per SM (80 registers) for K <= 8: fp8
// workload 504.7 -> 495.4 us, the others unchanged.  The K <= 16 variant
// is held to three CTAs per SM, where it keeps its registers (it would
// spill at 80).
template <int KMAX>
__global__ void __launch_bounds__(128, KMAX <= 8 ? 6 : 3) ep_combine_backward_kernel(CombineBwdDev c) {
  const int64_t n_items = c.T + c.max_pad;
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    combine_backward_item<KMAX>(c, item);
    __syncthreads();  // the next item reuses the shared slots
  }
}

template <int KMAX>
cudaError_t launch_bwd(const CombineBwdDev& c, cudaStream_t stream, const LaunchCfg& cfg) {
  long long blocks = c.T + (c.max_pad < kBwdPadCtas ? c.max_pad : kBwdPadCtas);
  const long long cap = budget_cap(ep_combine_backward_kernel<KMAX>, 128, 0, cfg.sm_budget);
  if (cap > 0 && blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  ep_combine_backward_kernel<KMAX><<<static_cast<unsigned>(blocks), 128, 0, stream>>>(c);
  if (cfg.ctas) *cfg.ctas = blocks;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine_backward(const CombineBwdDev& c, cudaStream_t stream, const LaunchCfg& cfg) {
  if (c.K <= 2) return launch_bwd<2>(c, stream, cfg);
  if (c.K <= 4) return launch_bwd<4>(c, stream, cfg);
  if (c.K <= 6) return launch_bwd<6>(c, stream, cfg);
  if (c.K <= 8) return launch_bwd<8>(c, stream, cfg);
  return launch_bwd<16>(c, stream, cfg);
}

cudaError_t launch_combine(const CombineDev& c, cudaStream_t stream, const LaunchCfg& cfg) {
  switch (c.K) {
    case 1: return launch_k<1, 4, 4>(c, stream, cfg);
    case 2: return launch_k<2, 2, 4>(c, stream, cfg);
    case 3: return launch_k<3, 2, 4>(c, stream, cfg);
    case 4: return launch_k<4, 1, 4>(c, stream, cfg);
    case 5: return launch_k<5, 1, 4>(c, stream, cfg);
    case 6: return launch_k<6, 1, 4>(c, stream, cfg);
    case 7: return launch_k<7, 1, 3>(c, stream, cfg);
    case 8: return launch_k<8, 1, 3>(c, stream, cfg);
    default: return launch_k<16, 1, 1>(c, stream, cfg);
  }
}

}  // namespace ep
