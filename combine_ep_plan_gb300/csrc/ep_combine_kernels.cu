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
// many small items and the kernel has no long tail.
template <int KMAX, int U, int MINB>
__global__ void __launch_bounds__(256, MINB) ep_combine_kernel(CombineDev c) {
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
      my_w = c.weights[g * c.K + lane];
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
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      out[g * hv + v] = o;
    }
  }
}

// One full wave of resident CTAs (grid-stride inside).
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

template <int KMAX, int U, int MINB>
cudaError_t launch_k(const CombineDev& c, cudaStream_t stream) {
  static int grid = 0;  // per process; one device type
  if (grid == 0)
    grid = EP_COMBINE_CTAS_PER_SM > 0 ? EP_COMBINE_CTAS_PER_SM * num_sms()
                                      : resident_grid(ep_combine_kernel<KMAX, U, MINB>, 256);
  ep_combine_kernel<KMAX, U, MINB><<<grid, 256, 0, stream>>>(c);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const CombineDev& c, cudaStream_t stream) {
  switch (c.K) {
    case 1: return launch_k<1, 4, 4>(c, stream);
    case 2: return launch_k<2, 2, 4>(c, stream);
    case 3: return launch_k<3, 2, 4>(c, stream);
    case 4: return launch_k<4, 1, 4>(c, stream);
    case 5: return launch_k<5, 1, 4>(c, stream);
    case 6: return launch_k<6, 1, 4>(c, stream);
    case 7: return launch_k<7, 1, 3>(c, stream);
    case 8: return launch_k<8, 1, 3>(c, stream);
    default: return launch_k<16, 1, 1>(c, stream);
  }
}

}  // namespace ep
