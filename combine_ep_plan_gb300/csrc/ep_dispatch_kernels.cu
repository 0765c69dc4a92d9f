// ep_dispatch_kernels.cu — the dispatch row scatter on sm_103a.
//
// One warp per work item, grid-stride over T source tokens followed by the
// N_pad padding rows.  A token's hidden row is read from HBM exactly once
// (16-byte non-allocating loads) and stored to each of its expanded rows
// (the per-destination dedup of TileLang tutorial ch. 38 §1.3 becomes "one
// read, K writes" on a single device).  Padding rows are zero-filled when
// requested (§2.2).  FP8: per 128-element group, amax over the group, scale =
// amax/448 by IEEE division, codes by IEEE division and the hardware E4M3
// conversion with round-to-nearest-even and satfinite (§3.6).
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

__device__ __forceinline__ void st_row(uint4* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Unroll factor: 16-byte vectors per lane loaded before the K stores.
constexpr int kUnroll = 4;

// N_pad as the plan wrote it, at most max_pad (the entries the handle holds).
__device__ __forceinline__ int64_t pad_count(const DispatchDev& a) {
  const int64_t n = a.sizes[kSizePad];
  return n < a.max_pad ? n : a.max_pad;
}

// Work item = (row item, column chunk of 32*kUnroll vectors): T token rows
// then N_pad padding rows, each cut into chunks, so that every warp gets many
// small items and the kernel has no long tail.
// Scale index of group j of expanded row r, in the requested layout.
__device__ __forceinline__ int64_t scale_at(const DispatchDev& a, int64_t r, int64_t j, int64_t groups) {
  return a.scales_col_major ? j * a.capacity + r : r * groups + j;
}

// Copies whole rows: BF16 hidden rows (row_vec = H/8 vectors), or E4M3 codes
// of pre-quantised input (row_vec = H/16) together with their H/128 fp32
// scales, which the warp owning chunk 0 of a row copies.  PROF: the same
// kernel, plus a per-CTA record (items, payload bytes, start and end).
// The pre-quantised variant is held to five CTAs per SM (48 registers),
// where its scales load once per row without spills (fp8 workload 149.7 ->
// 146.5 us, bf16 129.5 -> 128.3, rt unchanged; loading them once at 58
// registers and four CTAs, or four CTAs alone, gained half as much).
constexpr int kScaleRegs = 4;

template <int ROW_DIV, bool WITH_SCALES, bool PROF>
__global__ void __launch_bounds__(256, ROW_DIV == 16 ? 5 : 0) ep_dispatch_copy_kernel(DispatchDev a) {
  // Before anything else, even before the wait for the previous kernel: one
  // bulk L2 prefetch of the warp's first source chunk (token items only; x
  // is an input, never written by the plan), so that the row is on its way
  // while the plan outputs are read.  Measured 2.8 us faster per bf16 step.
  {
    const int64_t hv = a.H / ROW_DIV;
    constexpr int kChunk = 32 * kUnroll;
    const int64_t chunks = (hv + kChunk - 1) / kChunk;
    const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if ((threadIdx.x & 31) == 0 && w < a.T * chunks) {
      const int64_t ri = w / chunks;
      const int64_t v0 = (w - ri * chunks) * kChunk;
      const unsigned n = static_cast<unsigned>((hv - v0 < kChunk ? hv - v0 : kChunk) * 16);
      const uint4* src = static_cast<const uint4*>(a.x) + ri * hv + v0;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(n) : "memory");
    }
  }
  pdl_wait();
  unsigned long long t0 = 0, units = 0, bytes = 0;
  if (PROF && threadIdx.x == 0) t0 = prof_now();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t hv = a.H / ROW_DIV;  // 16-byte vectors per row
  const int64_t groups = a.H / 128;
  constexpr int kChunk = 32 * kUnroll;
  const int64_t chunks = (hv + kChunk - 1) / kChunk;
  const int64_t n_pad = a.zero_pad ? pad_count(a) : 0;
  const int64_t n_items = (a.T + n_pad) * chunks;
  const uint4* x = static_cast<const uint4*>(a.x);
  uint4* out = static_cast<uint4*>(a.out);
  const unsigned long long pol = l2_evict_first_policy();  // the written rows

  for (int64_t item = warp; item < n_items; item += nwarps) {
    const int64_t ri = item / chunks;
    const int64_t v0 = (item - ri * chunks) * kChunk;
    // payload bytes of this item's part of one row (codes or bf16), and of
    // its scales (chunk 0 only)
    const int64_t item_bytes = 16 * (hv - v0 < kChunk ? hv - v0 : kChunk);
    const int64_t scale_bytes = (WITH_SCALES && v0 == 0) ? 4 * groups : 0;
    if (PROF) ++units;
    if (ri < a.T) {
      const int64_t g = ri;
      int my_row = -1;
      if (lane < a.K) my_row = a.slot[g * a.K + lane];
      if (my_row >= a.capacity) {
        atomicOr(a.status, kStCapacity);
        my_row = -1;
      }
      const uint4* src = x + g * hv;
      uint4 buf[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t v = v0 + u * 32 + lane;
        if (v < hv) buf[u] = ld_stream(src + v);
      }
      const bool copy_scales = WITH_SCALES && v0 == 0;
      if (PROF) bytes += item_bytes + scale_bytes;
      // the row's scales, loaded once before the K stores: up to 128 groups
      // in registers, any beyond that read again per destination
      float sreg[kScaleRegs];
      if (copy_scales) {
#pragma unroll
        for (int q = 0; q < kScaleRegs; ++q) {
          const int64_t j = lane + 32 * q;
          sreg[q] = j < groups ? a.x_scales[g * groups + j] : 0.0f;
        }
      }
      for (int k = 0; k < a.K; ++k) {
        const int r = __shfl_sync(0xffffffffu, my_row, k);
        if (r < 0) continue;
        if (PROF) bytes += item_bytes + scale_bytes;
        uint4* dst = out + static_cast<int64_t>(r) * hv;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t v = v0 + u * 32 + lane;
          if (v < hv) st_evict_first(dst + v, buf[u], pol);
        }
        if (copy_scales) {
#pragma unroll
          for (int q = 0; q < kScaleRegs; ++q) {
            const int64_t j = lane + 32 * q;
            if (j < groups) a.scales[scale_at(a, r, j, groups)] = sreg[q];
          }
          for (int64_t j = lane + 32 * kScaleRegs; j < groups; j += 32)
            a.scales[scale_at(a, r, j, groups)] = a.x_scales[g * groups + j];
        }
      }
    } else {
      const int r = a.pad_rows[ri - a.T];
      if (r < 0 || r >= a.capacity) {
        if (lane == 0) atomicOr(a.status, kStCapacity);
        continue;
      }
      if (PROF) bytes += item_bytes + scale_bytes;
      uint4* dst = out + static_cast<int64_t>(r) * hv;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t v = v0 + u * 32 + lane;
        if (v < hv) st_evict_first(dst + v, z, pol);
      }
      if (WITH_SCALES && v0 == 0)
        for (int64_t j = lane; j < groups; j += 32) a.scales[scale_at(a, r, j, groups)] = 0.0f;
    }
  }
  if (PROF)
    prof_cta_end(a, ROW_DIV == 8 ? kProfDispatchBf16 : kProfDispatchFp8Input, t0, 0, 0, 0, units, bytes);
}

// Two fp32 values -> two E4M3 codes (lo in the low byte), RNE, satfinite.
__device__ __forceinline__ unsigned short cvt_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// x / s rounded to nearest (IEEE binary32), given y = RN(1/s): Markstein's
// correction (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990; the division
// theorem in Muller et al., "Handbook of Floating-Point Arithmetic"): with
// q0 = RN(x*y) within one ulp of x/s, the remainder r = x - q0*s is exact
// under FMA and RN(q0 + r*y) = RN(x/s), provided nothing underflows.  The
// caller guarantees that (see kFastQuotientMinAmax).  The quotient takes the
// sign of x: a no-op for x != 0 (s > 0), and for x = -0 it restores the
// sign the IEEE quotient has (the remainder step turns -0 into +0).
__device__ __forceinline__ float quotient_rn(float x, float s, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = __fmaf_rn(-q0, s, x);
  return copysignf(__fmaf_rn(r, y, q0), x);
}

// RN(1/448) in binary32.  quotient_rn(amax, 448, kRcp448) equals the IEEE
// quotient amax/448 for every finite bf16 amax >= 0, subnormals included
// (checked exhaustively); non-finite amax takes the IEEE division.
constexpr float kRcp448 = 0.002232142857142857f;

// Groups whose amax is at least this use quotient_rn: then scale >= 2^-69 and
// every remainder of a quotient that can round to a non-zero E4M3 code
// (|x/s| >= 2^-10) stays a normal number; quotients below 2^-10 round to a
// signed zero whatever their last bits.  Checked exhaustively, code for
// code, over every bf16 x and every bf16 amax >= 2^-60 with |x| <= amax.
// Smaller groups use __fdiv_rn.
constexpr float kFastQuotientMinAmax = 8.673617379884035e-19f;  // 2^-60

__device__ __forceinline__ float bf16_lo(unsigned w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(unsigned w) { return __uint_as_float(w & 0xffff0000u); }

// FP8 work item = (row item, chunk of kFp8Units*512 elements).  In each unit
// a lane owns 16 consecutive elements (two 16-byte loads, one 16-byte store
// of codes) and eight lanes form one 128-element scale group; the chunk's
// 4*kFp8Units scales are stored by as many lanes in one contiguous store.
#ifndef EP_FP8_UNITS
#define EP_FP8_UNITS 4
#endif
constexpr int kFp8Units = EP_FP8_UNITS;
// Threads per CTA, and work items per warp at the full grid (tuning knobs).
#ifndef EP_FP8_CTA
#define EP_FP8_CTA 256
#endif
#ifndef EP_FP8_WARP_ITEMS
#define EP_FP8_WARP_ITEMS 2
#endif
#ifndef EP_FP8_PREFETCH_NEXT
#define EP_FP8_PREFETCH_NEXT 1
#endif
constexpr int kFp8Cta = EP_FP8_CTA;

// Four CTAs of 256 threads per SM (64 registers): measured faster than three
// at 80.  The profiling variant keeps three, so that its counters do not
// spill.  The grid gives each warp two items; after loading one, a warp
// sends its next item's source chunk to L2 with a bulk prefetch, so that the
// next load is short (fp8 workload: 169.6 us with one item per warp, 163.8
// with two, 160.4 with two and the prefetch).
template <bool PROF>
__global__ void __launch_bounds__(kFp8Cta, PROF ? 768 / kFp8Cta : 1024 / kFp8Cta)
    ep_dispatch_fp8_kernel(DispatchDev a) {
  pdl_wait();
  unsigned long long t0 = 0, units = 0, bytes = 0;
  if (PROF && threadIdx.x == 0) t0 = prof_now();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t hv = a.H / 8;     // 16-byte vectors of bf16 per source row
  const int64_t qv = a.H / 16;    // 16-byte vectors of codes per expanded row
  const int64_t groups = a.H / 128;
  constexpr int kUnitVec = 32;                 // 16-element units per warp per unit step
  constexpr int kChunkVec = kUnitVec * kFp8Units;
  const int64_t chunks = (qv + kChunkVec - 1) / kChunkVec;
  const int64_t n_pad = a.zero_pad ? pad_count(a) : 0;
  const int64_t n_items = (a.T + n_pad) * chunks;
  const uint4* x = static_cast<const uint4*>(a.x);
  uint4* out = static_cast<uint4*>(a.out);

  for (int64_t item = warp; item < n_items; item += nwarps) {
    const int64_t ri = item / chunks;
    const int64_t q_base = (item - ri * chunks) * kChunkVec;  // first 16-element unit of the chunk
    const int64_t g_base = q_base / 8;                          // first scale group of the chunk
    // lanes 0 .. 4*kFp8Units-1 own the chunk's scales, in order
    const int sc_lane = lane < 4 * kFp8Units ? lane : 0;
    const bool sc_active = lane < 4 * kFp8Units && g_base + lane < groups;
    // payload of the item: 32 bytes of bf16 in, 16 bytes of codes out per
    // 16-element unit, and 4 bytes per scale written
    const int64_t n_q = qv - q_base < kChunkVec ? qv - q_base : kChunkVec;
    const int64_t n_g = groups - g_base < 4 * kFp8Units ? groups - g_base : 4 * kFp8Units;
    if (PROF) ++units;
    if (ri < a.T) {
      const int64_t g = ri;
      int my_row = -1;
      if (lane < a.K) my_row = a.slot[g * a.K + lane];
      if (my_row >= a.capacity) {
        atomicOr(a.status, kStCapacity);
        my_row = -1;
      }
      const uint4* src = x + g * hv;
      uint4 lo[kFp8Units], hi[kFp8Units];
#pragma unroll
      for (int u = 0; u < kFp8Units; ++u) {
        const int64_t qi = q_base + u * kUnitVec + lane;
        lo[u] = make_uint4(0u, 0u, 0u, 0u);
        hi[u] = lo[u];
        if (qi < qv) {
          lo[u] = ld_stream(src + 2 * qi);
          hi[u] = ld_stream(src + 2 * qi + 1);
        }
      }
#if EP_FP8_PREFETCH_NEXT
      {
        // the warp's next token item: its source chunk on its way to L2
        // while this one is converted and stored
        const int64_t nx = item + nwarps;
        if (lane == 0 && nx < a.T * chunks) {
          const int64_t nr = nx / chunks;
          const int64_t nq = (nx - nr * chunks) * kChunkVec;
          const unsigned nbytes = static_cast<unsigned>((qv - nq < kChunkVec ? qv - nq : kChunkVec) * 32);
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(x + nr * hv + 2 * nq), "r"(nbytes)
                       : "memory");
        }
      }
#endif
      uint4 q[kFp8Units];
      float scale_u[kFp8Units];
#pragma unroll
      for (int u = 0; u < kFp8Units; ++u) {
        float f[16];
        const unsigned w[8] = {lo[u].x, lo[u].y, lo[u].z, lo[u].w, hi[u].x, hi[u].y, hi[u].z, hi[u].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          f[2 * i] = bf16_lo(w[i]);
          f[2 * i + 1] = bf16_hi(w[i]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        const float scale =
            amax <= 3.402823466e38f ? quotient_rn(amax, 448.0f, kRcp448) : __fdiv_rn(amax, 448.0f);
        scale_u[u] = scale;
        q[u] = make_uint4(0u, 0u, 0u, 0u);
        if (amax != 0.0f) {
          unsigned short c[8];
          if (amax >= kFastQuotientMinAmax && amax <= 3.402823466e38f) {
            const float y = __frcp_rn(scale);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              c[i] = cvt_e4m3x2(quotient_rn(f[2 * i], scale, y), quotient_rn(f[2 * i + 1], scale, y));
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              c[i] = cvt_e4m3x2(__fdiv_rn(f[2 * i], scale), __fdiv_rn(f[2 * i + 1], scale));
          }
          q[u].x = c[0] | (static_cast<unsigned>(c[1]) << 16);
          q[u].y = c[2] | (static_cast<unsigned>(c[3]) << 16);
          q[u].z = c[4] | (static_cast<unsigned>(c[5]) << 16);
          q[u].w = c[6] | (static_cast<unsigned>(c[7]) << 16);
        }
      }
      // gather the chunk's scales: scale of group j (j = u*4 + m) lives in lane 8*m of unit u
      float my_scale = 0.0f;
#pragma unroll
      for (int u = 0; u < kFp8Units; ++u) {
        const float v = __shfl_sync(0xffffffffu, scale_u[u], (sc_lane & 3) * 8);
        if ((sc_lane >> 2) == u) my_scale = v;
      }
      if (PROF) bytes += 32 * n_q;
      for (int k = 0; k < a.K; ++k) {
        const int r = __shfl_sync(0xffffffffu, my_row, k);
        if (r < 0) continue;
        if (PROF) bytes += 16 * n_q + 4 * n_g;
        uint4* dst = out + static_cast<int64_t>(r) * qv;
#pragma unroll
        for (int u = 0; u < kFp8Units; ++u) {
          const int64_t qi = q_base + u * kUnitVec + lane;
          if (qi < qv) st_row(dst + qi, q[u]);
        }
        if (sc_active) a.scales[scale_at(a, r, g_base + lane, groups)] = my_scale;
      }
    } else {
      const int r = a.pad_rows[ri - a.T];
      if (r < 0 || r >= a.capacity) {
        if (lane == 0) atomicOr(a.status, kStCapacity);
        continue;
      }
      if (PROF) bytes += 16 * n_q + 4 * n_g;
      uint4* dst = out + static_cast<int64_t>(r) * qv;
#pragma unroll
      for (int u = 0; u < kFp8Units; ++u) {
        const int64_t qi = q_base + u * kUnitVec + lane;
        if (qi < qv) st_row(dst + qi, make_uint4(0u, 0u, 0u, 0u));
      }
      if (sc_active) a.scales[scale_at(a, r, g_base + lane, groups)] = 0.0f;
    }
  }
  if (PROF) prof_cta_end(a, kProfDispatchFp8, t0, 0, 0, 0, units, bytes);
}

// One warp per work item (FP8: per two): the grid covers the worst-case item
// count (T rows plus E*(A-1) padding rows, in chunks); warps without an item
// exit at once.
// Many short-lived CTAs, balanced by the hardware block scheduler, keep more
// stores in flight than a resident grid looping over the items.  Under an
// SM budget the grid is capped at that many SMs' worth of resident CTAs,
// which then loop over the items.
long long item_grid(int64_t rows, int64_t chunks, int threads = 256, int warp_items = 1) {
  const int64_t warps = (rows * chunks + warp_items - 1) / warp_items;
  const int64_t per_cta = threads / 32;
  const int64_t blocks = (warps + per_cta - 1) / per_cta;
  return blocks < 1 ? 1 : (blocks > 0x7fffffff ? 0x7fffffff : blocks);
}

template <typename Kernel>
cudaError_t launch_items(Kernel kernel, const DispatchDev& d, int64_t chunks, cudaStream_t stream,
                         const LaunchCfg& cfg, int threads = 256, int warp_items = 1) {
  long long grid = item_grid(d.T + d.max_pad, chunks, threads, warp_items);
  const long long cap = budget_cap(kernel, threads, 0, cfg.sm_budget);
  if (cap > 0 && grid > cap) grid = cap;
  const cudaError_t e = launch_pdl(kernel, static_cast<unsigned>(grid), threads, stream, d);
  if (cfg.ctas) *cfg.ctas = grid;
  return e;
}

}  // namespace

cudaError_t launch_dispatch_bf16(const DispatchDev& d, cudaStream_t stream, const LaunchCfg& cfg) {
  const int64_t chunks = (d.H / 8 + 32 * kUnroll - 1) / (32 * kUnroll);
  if (d.prof_rec) return launch_items(ep_dispatch_copy_kernel<8, false, true>, d, chunks, stream, cfg);
  return launch_items(ep_dispatch_copy_kernel<8, false, false>, d, chunks, stream, cfg);
}

cudaError_t launch_dispatch_fp8_input(const DispatchDev& d, cudaStream_t stream, const LaunchCfg& cfg) {
  const int64_t chunks = (d.H / 16 + 32 * kUnroll - 1) / (32 * kUnroll);
  if (d.prof_rec) return launch_items(ep_dispatch_copy_kernel<16, true, true>, d, chunks, stream, cfg);
  return launch_items(ep_dispatch_copy_kernel<16, true, false>, d, chunks, stream, cfg);
}

namespace {

// Per expanded row: the routing weight and {source token, slot k}; one
// thread per (token, slot), then one per padding row.
__global__ void __launch_bounds__(256) ep_dispatch_metadata_kernel(MetaDev m) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t pairs = m.T * m.K;
  if (i < pairs) {
    const int r = m.slot[i];
    if (r < 0) return;
    if (r >= m.capacity) {
      atomicOr(m.status, kStCapacity);
      return;
    }
    m.recv_weights[r] = m.weights[i];
    m.recv_meta[2 * static_cast<int64_t>(r)] = static_cast<int>(i / m.K);
    m.recv_meta[2 * static_cast<int64_t>(r) + 1] = static_cast<int>(i % m.K);
    return;
  }
  const int64_t pi = i - pairs;
  if (pi >= m.sizes[kSizePad] || pi >= m.max_pad) return;
  const int r = m.pad_rows[pi];
  if (r < 0 || r >= m.capacity) {
    atomicOr(m.status, kStCapacity);
    return;
  }
  m.recv_weights[r] = 0.0f;
  m.recv_meta[2 * static_cast<int64_t>(r)] = -1;
  m.recv_meta[2 * static_cast<int64_t>(r) + 1] = -1;
}

}  // namespace

cudaError_t launch_dispatch_metadata(const MetaDev& m, cudaStream_t stream) {
  const int64_t n = m.T * m.K + m.max_pad;
  ep_dispatch_metadata_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(m);
  return cudaGetLastError();
}

cudaError_t launch_dispatch_fp8(const DispatchDev& d, cudaStream_t stream, const LaunchCfg& cfg) {
  const int64_t chunks = (d.H / 16 + 32 * kFp8Units - 1) / (32 * kFp8Units);
  if (d.prof_rec)
    return launch_items(ep_dispatch_fp8_kernel<true>, d, chunks, stream, cfg, kFp8Cta, EP_FP8_WARP_ITEMS);
  return launch_items(ep_dispatch_fp8_kernel<false>, d, chunks, stream, cfg, kFp8Cta, EP_FP8_WARP_ITEMS);
}

}  // namespace ep
