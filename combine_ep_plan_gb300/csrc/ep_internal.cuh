// ep_internal.cuh — device-side layout of a plan and helpers shared by the
// plan, dispatch and combine kernels.  Internal to the library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ep {

// Tokens handled by one CTA of the plan kernels (one thread per token).
constexpr int kTile = 256;
constexpr int kTileWords = kTile / 32;

// Bits of the device status word.
constexpr unsigned kStInvalidId = 1u;   // expert id outside [-1, E)
constexpr unsigned kStDuplicate = 2u;   // same expert twice in one token row
constexpr unsigned kStCapacity = 4u;    // an output row at or beyond capacity
constexpr unsigned kStTimeout = 8u;     // bounded look-back wait gave up

// Control words (zeroed when a handle is created), each in its own 128-byte
// line: the barrier's waiters poll the generation word while arrivals
// update the count.
constexpr int kCtrBarCount = 0;   // grid barrier: CTAs arrived
constexpr int kCtrBarGen = 32;    // grid barrier: generation
constexpr int kCtrStatus = 64;    // device status word
constexpr int kCtrWords = 96;

// Size slots.
constexpr int kSizeRecv = 0;  // N_recv
constexpr int kSizeExp = 1;   // N_exp
constexpr int kSizePad = 2;   // N_pad
constexpr int kSizeWords = 4;

// Look-back descriptor: high 32 bits = (plan epoch << 2) | state, low 32
// bits = value.
constexpr unsigned long long kDescAggregate = 1ull;
constexpr unsigned long long kDescInclusive = 2ull;

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
  unsigned epoch;      // this plan's epoch (>= 1), tags the descriptors
  unsigned long long* desc;  // [num_tiles, P+E] look-back descriptors
  uint32_t* tile_bits; // [num_tiles, kTileWords, P+E] tile bit matrices
  int* tile_wpre;      // [num_tiles, kTileWords, P+E] exclusive prefix per word
  // outputs
  int* sizes;          // [kSizeWords]
  int* totals;         // [P+E]: num_recv[d], then expert_counts[e]
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
  // bounded wait of the look-back, and a test hook
  long long poll_limit;
  int suppress_tile;
};

// Host-side launchers (defined in the .cu files, called by the C ABI layer).
cudaError_t launch_plan(const PlanDev& p, cudaStream_t stream);
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
};
cudaError_t launch_dispatch_bf16(const DispatchDev& d, cudaStream_t stream);
cudaError_t launch_dispatch_fp8(const DispatchDev& d, cudaStream_t stream);
cudaError_t launch_dispatch_fp8_input(const DispatchDev& d, cudaStream_t stream);

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
};
cudaError_t launch_combine(const CombineDev& c, cudaStream_t stream);

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
cudaError_t launch_combine_backward(const CombineBwdDev& c, cudaStream_t stream);

int num_sms();

}  // namespace ep
