// ep_internal.cuh — device-side layout of a plan and helpers shared by the
// plan, dispatch and combine kernels.  Internal to the library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ep {

// Tokens handled by one CTA of the plan kernels (one thread per token).
#ifndef EP_TILE
#define EP_TILE 256
#endif
constexpr int kTile = EP_TILE;
constexpr int kTileWords = kTile / 32;

// Bits of the device status word.
constexpr unsigned kStInvalidId = 1u;   // expert id outside [-1, E)
constexpr unsigned kStDuplicate = 2u;   // same expert twice in one token row
constexpr unsigned kStCapacity = 4u;    // an output row at or beyond capacity
constexpr unsigned kStTimeout = 8u;     // a bounded grid-barrier wait gave up

// Control words (zeroed when a handle is created), each in its own 128-byte
// line.  The grid barriers use one of two arrival counts, picked by the
// parity of a generation word every CTA reads when the plan starts; after
// the second barrier CTA 0 zeroes the other count and bumps the generation,
// so each launch (and each replay of a captured launch) finds a zeroed count
// and leaves one for the next.  A launch whose barrier wait gave up leaves
// its count as it was and sets kStTimeout; until the host clears the control
// words (when it reads the status), later launches that find kStTimeout set
// do not arrive at a barrier at all, so that no launch can pass a barrier on
// a timed-out launch's arrivals.
constexpr int kCtrBarCount = 0;   // grid barriers: CTAs arrived, generation 0, 2, ...
constexpr int kCtrBarCount1 = 32; // ... generation 1, 3, ...
constexpr int kCtrBarGen = 64;    // generation
constexpr int kCtrStatus = 96;    // device status word
constexpr int kCtrWords = 128;

// Copies of the column totals: every CTA reads the totals right after the
// second grid barrier; spreading the reads over 16 copies (CTA b reads copy
// b % 16) keeps them from queuing on the same few L2 lines (fp8 plan, 256
// experts: 17.7 -> 16.5 us).
constexpr int kTotRep = 16;

// Size slots.
constexpr int kSizeRecv = 0;  // N_recv
constexpr int kSizeExp = 1;   // N_exp
constexpr int kSizePad = 2;   // N_pad
constexpr int kSizeWords = 4;

// Per-CTA profile records, a compile-time switch: only the PROF
// instantiations of the plan, dispatch and combine kernels write one, so the
// default kernels carry no profiling code at all.  Each CTA owns one record
// of kProfWords words (no atomics); the host reads the buffer once.
//   [0] kernel id << 56 | launch sequence << 32 | CTA index
//   [1] start  [2..4] stage marks (kernel specific, 0 if unused)  [5] end
//       (global timer, ns)
//   [6] work units  [7] payload bytes read + written
constexpr int kProfWords = 8;
enum : unsigned {
  kProfPlan = 1,
  kProfDispatchBf16 = 2,
  kProfDispatchFp8 = 3,
  kProfDispatchFp8Input = 4,
  kProfCombine = 5,
  kProfDispatchBackward = 6,
};
// The record target travels in each kernel's parameter struct as two plain
// fields (the copy kernel's parameters stay within 128 bytes; beyond that it
// needed more registers):
//   prof_rec   this launch's first record, NULL when profiling is off
//   prof_meta  launch sequence (24 bits) << 40 | records available
#define EP_PROF_FIELDS          \
  unsigned long long* prof_rec; \
  long long prof_meta
constexpr int kProfAvailBits = 40;

__device__ __forceinline__ unsigned long long prof_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Written by thread 0 of the CTA; records past the buffer are dropped.
template <class Dev>
__device__ __forceinline__ void prof_write(const Dev& d, unsigned kind, unsigned long long t0,
                                           unsigned long long ta, unsigned long long tb, unsigned long long tc,
                                           unsigned long long t_end, unsigned long long units,
                                           unsigned long long bytes) {
  const long long avail = d.prof_meta & ((1ll << kProfAvailBits) - 1);
  const unsigned long long seq = static_cast<unsigned long long>(d.prof_meta) >> kProfAvailBits;
  if (d.prof_rec == nullptr || static_cast<long long>(blockIdx.x) >= avail) return;
  unsigned long long* r = d.prof_rec + static_cast<long long>(blockIdx.x) * kProfWords;
  r[0] = (static_cast<unsigned long long>(kind) << 56) | ((seq & 0xffffffu) << 32) | blockIdx.x;
  r[1] = t0;
  r[2] = ta;
  r[3] = tb;
  r[4] = tc;
  r[5] = t_end;
  r[6] = units;
  r[7] = bytes;
}

// End of a profiled CTA, called by all its threads: sums the warp-uniform
// counters over the CTA's warps; thread 0 writes the record.
template <class Dev>
__device__ __forceinline__ void prof_cta_end(const Dev& d, unsigned kind, unsigned long long t0,
                                             unsigned long long ta, unsigned long long tb, unsigned long long tc,
                                             unsigned long long units, unsigned long long bytes) {
  __shared__ unsigned long long s_units[32], s_bytes[32];
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    s_units[warp] = units;
    s_bytes[warp] = bytes;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long u = 0, b = 0;
    for (int w = 0; w < static_cast<int>((blockDim.x + 31) >> 5); ++w) {
      u += s_units[w];
      b += s_bytes[w];
    }
    prof_write(d, kind, t0, ta, tb, tc, prof_now(), u, b);
  }
}

// Programmatic dependent launch.  The dispatch and combine kernels are
// launched with programmatic stream serialization, so that the launch of a
// grid overlaps the end of the kernel before it in the stream: pdl_wait
// blocks until that kernel has completed and its memory is visible, and
// comes before every global memory access of the kernel.  None of the
// kernels triggers its dependents early: early-launched CTAs that sit
// waiting took SM slots from the tail of the running grid (measured slower).
// The wait is a no-op in a kernel launched without the attribute.
// EP_USE_PDL=0 builds plain launches.
#ifndef EP_USE_PDL
#define EP_USE_PDL 1
#endif
__device__ __forceinline__ void pdl_wait() {
  if (EP_USE_PDL) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// An L2 cache policy that marks the lines it touches evict-first, and a
// 16-byte store through it.  The scatters that write every expanded row once
// and do not read it back (the BF16 / pre-quantised dispatch copy, the
// combine backward's grad_y rows) store this way, so that L2 gives up their
// dirty lines before the source rows still to be read.  Measured, kernels
// alone: dispatch copy 246.7 -> 243.8 us (bf16 workload), 715.8 -> 696.6 us
// (rt); combine backward 469.3 -> 460.0 us (bf16), 494.8 -> 485.4 us (fp8),
// 1360.5 -> 1339.8 us (rt).  Not kept: the same policy on the FP8 dispatch's
// code stores, on the combine's output stores, and on the loads of the
// dispatch, the combine or its backward (each unchanged or slower).
__device__ __forceinline__ unsigned long long l2_evict_first_policy() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void st_evict_first(uint4* p, const uint4& v, unsigned long long pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}

template <typename Dev>
cudaError_t launch_pdl(void (*kernel)(Dev), unsigned grid, unsigned block, cudaStream_t stream, const Dev& arg) {
  if (!EP_USE_PDL) {
    kernel<<<grid, block, 0, stream>>>(arg);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, arg);
}

// How a launch is shaped: an SM budget (0 = the whole device), and where
// the launcher reports the CTAs it launched (the profile record cursor).
struct LaunchCfg {
  int sm_budget = 0;
  long long* ctas = nullptr;
};

// Everything the plan kernels need, passed by value.
struct PlanDev {
  // shape
  int64_t S, T;
  int P, E, K, A, C, El;
  int64_t chunk;  // tokens per channel, ceil(S/C)
  int num_tiles;
  int ncols;  // P + E: ranks first, then experts
  // input (read during the plan only)
  const int64_t* topk_idx;
  // scratch
  unsigned* ctr;       // [kCtrWords], zeroed once per handle
  uint32_t* tile_bits; // [num_tiles, kTileWords, P+E] tile bit matrices
  int* tile_wpre;      // [num_tiles, kTileWords, P+E] exclusive prefix per word inside the tile
  int* agg;            // [P+E, num_tiles] bits per tile and column
  int* tile_pre;       // [P+E, num_tiles] exclusive prefix of each tile over the tiles before it
  // outputs
  int* sizes;          // [kSizeWords]
  int* totals;         // [P+E]: num_recv[d], then expert_counts[e]
  int* totals_rep;     // [kTotRep][P+E]: copies of the totals, read by the CTAs in turn
  int* ntpe;           // [P,E]  num_tokens_per_expert
  int* ntpr;           // [P,P]
  int* rpm;            // [P,P]
  int* cpm;            // [P,P,C] [s][d][c]
  int* rcpm;           // [P,P,C] [d][s][c]
  int* recv_off;       // [P+1]
  int* exp_off;        // [E+1]
  int* pad_off;        // [E+1]
  int* slot;           // [T,K]
  int* send_head;      // [T,P]
  int* recv_src_idx;   // [T*min(K,P)]
  int* exp_src;        // [T*K + E*(A-1)]
  int* pad_rows;       // [E*(A-1)]
  unsigned char* in_rank;  // [T,P]
  // entries allocated in recv_src_idx, exp_src and pad_rows: every store the
  // plan makes at an index derived from other CTAs' counts is checked
  // against them (an index beyond records kStCapacity and is not written)
  int64_t cap_recv, cap_exp, cap_pad;
  // bounded wait of the grid barriers, and a test hook (a tile whose CTA
  // returns before the first barrier)
  long long poll_limit;
  int suppress_tile;
  EP_PROF_FIELDS;
};

// Host-side launchers (defined in the .cu files, called by the C ABI layer).
cudaError_t launch_plan(const PlanDev& p, cudaStream_t stream, const LaunchCfg& cfg);
size_t plan_smem_bytes(int P, int E, int K);

struct DispatchDev {
  const void* x;          // [T,H] bf16, or [T,H] E4M3 codes (pre-quantised input)
  const float* x_scales;  // [T,H/128] scales of pre-quantised input, else NULL
  const int* slot;        // [T,K]
  const int* pad_rows;    // [N_pad]
  const int* sizes;       // device sizes (N_pad read on device)
  unsigned* status;
  void* out;              // [cap,H] bf16 or e4m3
  float* scales;          // [cap,H/128] for FP8
  int64_t T;
  int K;
  int64_t H;
  int64_t capacity;
  int64_t max_pad;        // upper bound of N_pad: E*(A-1) (sizes the grid)
  int zero_pad;
  int scales_col_major;   // scales stored [H/128][capacity] instead of [capacity][H/128]
  EP_PROF_FIELDS;
};
cudaError_t launch_dispatch_bf16(const DispatchDev& d, cudaStream_t stream, const LaunchCfg& cfg);
cudaError_t launch_dispatch_fp8(const DispatchDev& d, cudaStream_t stream, const LaunchCfg& cfg);
cudaError_t launch_dispatch_fp8_input(const DispatchDev& d, cudaStream_t stream, const LaunchCfg& cfg);

struct MetaDev {
  const int* slot;        // [T,K]
  const float* weights;   // [T,K]
  const int* pad_rows;    // [N_pad]
  const int* sizes;
  unsigned* status;
  float* recv_weights;    // [capacity]
  int* recv_meta;         // [capacity,2]
  int64_t T;
  int K;
  int64_t capacity;
  int64_t max_pad;
};
cudaError_t launch_dispatch_metadata(const MetaDev& m, cudaStream_t stream);

struct CombineDev {
  const void* y;          // [y_rows,H] bf16
  const void* bias;       // [T,H] bf16 added after the weighted sum, or NULL
  const int* slot;        // [T,K]
  const float* weights;   // [T,K]; NULL: unit weights (the dispatch backward)
  unsigned* status;
  void* out;              // [T,H] bf16
  int64_t T;
  int K;
  int64_t H;
  int64_t y_rows;
  EP_PROF_FIELDS;
};
cudaError_t launch_combine(const CombineDev& c, cudaStream_t stream, const LaunchCfg& cfg);

struct CombineBwdDev {
  const void* grad_out;   // [T,H] bf16
  const void* y;          // [y_rows,H] bf16
  const int* slot;        // [T,K]
  const float* weights;   // [T,K]
  const int* pad_rows;    // [N_pad]
  const int* sizes;       // device sizes (N_pad)
  unsigned* status;
  void* grad_y;           // [grad_y_rows,H] bf16
  float* grad_w;          // [T,K]
  int64_t T;
  int K;
  int64_t H;
  int64_t y_rows;
  int64_t grad_y_rows;
  int64_t max_pad;        // upper bound of N_pad, 0 without zero padding
};
cudaError_t launch_combine_backward(const CombineBwdDev& c, cudaStream_t stream, const LaunchCfg& cfg);

int num_sms();

// At most `budget` SMs' worth of resident CTAs (budget 0: no cap).
template <typename Kernel>
long long budget_cap(Kernel kernel, int threads, size_t smem, int budget) {
  if (budget <= 0) return -1;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  return static_cast<long long>(per_sm) * budget;
}

}  // namespace ep
