// ep_plan_kernels.cu — the routing plan on sm_103a, in one cooperative kernel.
//
// Phase 1, one CTA per tile of 256 tokens (CTAs loop if there are more tiles
// than co-resident CTAs):
//   - a bit matrix in shared memory, one 32-bit word per (column, warp):
//     column d < P = "token routed to rank d" (the OR deduplicates the token's
//     slots that land on one rank), column P+e = "token picked expert e";
//     per-lane shared-memory atomicOr; invalid and duplicate ids are
//     reported;
//   - the tile's bit matrix, its per-word prefixes inside the tile and its
//     count per column go to global memory.
// Grid barrier 1.  Column scans: one warp per column turns the tiles' counts
// into each tile's exclusive prefix and the column total.  Grid barrier 2
// (both barriers bounded).  (A single-pass decoupled look-back over the
// tiles, with one barrier, measured slower: every tile reached its
// predecessors while they were still publishing.)
// Phase 2, all CTAs: with X_col(g) = #{g' < g with the bit set in column col}
// available for any g from three loads (or, for the tokens of the tile a CTA
// scanned, from the bit matrix still in its shared memory), every plan
// array is computed directly:
//   send_head[g][d] = X_d(g) (if routed), recv_src_idx, slot[g][k] =
//   expert_offset[e] + X_e(g), exp_src, padding rows,
//   recv_channel_prefix[d][s][c] = X_d(start of channel c of source s),
//   channel_prefix[s][d][c] = X_d(end of channel c) - X_d(s*S),
//   rank_prefix[s][d] = X_d((s+1)*S), num_tokens_per_rank, and
//   num_tokens_per_expert[s][e] = X_e((s+1)*S) - X_e(s*S).
//
// Definitions followed: "Ascend DeepEP MoE Dispatch Optimization", the
// dispatch handle table, the notify stage and the per-channel cursor bases;
// TileLang tutorial ch. 38 "DeepEP-Ascend", §1.3 dedup, §2.2 expanded layout
// and padding, §3.5 deterministic order.
#include "ep_plan.h"
#include "ep_internal.cuh"

namespace ep {
namespace {

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Plan threads resident per SM at most (a small grid keeps the grid
// barriers cheap).
constexpr int kPlanThreadsPerSm = 512;

// Lanes below l within a word.
__device__ __forceinline__ uint32_t lanes_below(int l) { return l ? (0xffffffffu >> (32 - l)) : 0u; }

// Loads this tile's expert ids into shared memory (coalesced), checking them.
// All of a thread's loads are issued before any is used.
template <int KMAX>
__device__ __forceinline__ void load_tile_ids(const PlanDev& p, int64_t t0, int* ids) {
  const int64_t base = t0 * p.K;
  const int64_t end = p.T * p.K;
  const int n = kTile * p.K;  // <= kTile * KMAX
  long long v[KMAX];
#pragma unroll
  for (int u = 0; u < KMAX; ++u) {
    const int i = threadIdx.x + u * kTile;
    v[u] = (i < n && base + i < end) ? p.topk_idx[base + i] : -1ll;
  }
#pragma unroll
  for (int u = 0; u < KMAX; ++u) {
    const int i = threadIdx.x + u * kTile;
    if (i < n) {
      int e = -1;
      if (v[u] >= 0 && v[u] < p.E)
        e = static_cast<int>(v[u]);
      else if (v[u] != -1)
        atomicOr(&p.ctr[kCtrStatus], kStInvalidId);
      ids[i] = e;
    }
  }
}

// Builds the tile bit matrix (layout bits[w * ncols + col], zeroed before):
// each lane ORs its own bit into the word of its expert and of the expert's
// rank (shared-memory atomics; the OR deduplicates a token's slots on one
// rank).  A duplicate expert in one row shows up as its bit already set.
// (Aggregating lanes with __match_any_sync first measured slower on sm_103a
// with ~25 distinct experts per warp.)
__device__ __forceinline__ void build_tile_bits(const PlanDev& p, const int* ids, uint32_t* bits) {
  const unsigned me = 1u << (threadIdx.x & 31);
  uint32_t* row = bits + (threadIdx.x >> 5) * p.ncols;
  for (int k = 0; k < p.K; ++k) {
    const int e = ids[threadIdx.x * p.K + k];
    if (e < 0) continue;
    const unsigned old = atomicOr(&row[p.P + e], me);
    if (old & me) atomicOr(&p.ctr[kCtrStatus], kStDuplicate);
    atomicOr(&row[e / p.El], me);
  }
}

// Bounded grid-wide barrier for a cooperative launch.  Each CTA adds one
// arrival to this launch's count (a release reduction: nothing to wait for)
// and polls it until it reaches `round` times the grid: the release of the
// last CTA is the one reduction, seen by each poller one load later.
// `count` and `refuse` are meaningful in thread 0 only; a CTA that refuses
// (the launch found a timed-out predecessor's mark) neither arrives nor
// waits, and fails the barrier.
__device__ bool grid_sync(const PlanDev& p, unsigned* count, unsigned round, bool refuse) {
  __shared__ int s_ok;
  if (gridDim.x == 1) {  // a one-CTA plan: the CTA barrier orders everything
    __syncthreads();
    return true;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 0;
    if (!refuse) {
      const unsigned target = round * gridDim.x;
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(count) : "memory");
      ok = 1;
      long long polls = 0;
      unsigned ns = 32;
      while (static_cast<int>(ld_acquire(count) - target) < 0) {
        if (++polls > p.poll_limit) {
          ok = 0;
          break;
        }
        __nanosleep(ns);
        if (ns < 128) ns <<= 1;
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// i < n for a signed index and a capacity, as one unsigned comparison.
__device__ __forceinline__ bool in_cap(int64_t i, int64_t n) {
  return static_cast<uint64_t>(i) < static_cast<uint64_t>(n);
}

// Column scans, one warp per column: the tiles' counts in order, 32 at a
// time, to each tile's exclusive prefix (tile_pre) and the column total.
__device__ void column_scans(const PlanDev& p) {
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t col = gwarp; col < p.ncols; col += nwarps) {
    const int* agg = p.agg + col * p.num_tiles;
    int* pre = p.tile_pre + col * p.num_tiles;
    int carry = 0;
    constexpr int kBatch = 8;  // chunks of 32 tiles loaded before any is scanned
    for (int b0 = 0; b0 < p.num_tiles; b0 += 32 * kBatch) {
      int v[kBatch];
#pragma unroll
      for (int c = 0; c < kBatch; ++c) {
        const int t = b0 + 32 * c + lane;
        v[c] = t < p.num_tiles ? __ldcg(&agg[t]) : 0;
      }
#pragma unroll
      for (int c = 0; c < kBatch; ++c) {
        const int t = b0 + 32 * c + lane;
        int inc = v[c];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += n;
        }
        if (t < p.num_tiles) pre[t] = carry + inc - v[c];
        carry += __shfl_sync(0xffffffffu, inc, 31);
      }
    }
    if (lane == 0) p.totals[col] = carry;
    if (lane < kTotRep) p.totals_rep[static_cast<int64_t>(lane) * p.ncols + col] = carry;
  }
}

// Position of token i of the CTA's own tile in column col: the tile's
// exclusive prefix plus the bits set before i in the shared bit matrix.
__device__ __forceinline__ int tile_pos(const uint32_t* bits, const int* s_run, int ncols, int col, int i) {
  const int w = i >> 5;
  int pos = s_run[col];
  for (int v = 0; v < w; ++v) pos += __popc(bits[v * ncols + col]);
  return pos + __popc(bits[w * ncols + col] & lanes_below(i & 31));
}

// X_col(g): bits set in column col for tokens before g (g in [0, T]).
__device__ __forceinline__ int x_at(const PlanDev& p, int col, int64_t g) {
  if (g >= p.T) return __ldcg(&p.totals_rep[static_cast<int64_t>(blockIdx.x % kTotRep) * p.ncols + col]);
  const int64_t t = g / kTile;
  const int gl = static_cast<int>(g - t * kTile);
  const int64_t at = (t * kTileWords + (gl >> 5)) * p.ncols + col;
  return __ldcg(&p.tile_pre[static_cast<int64_t>(col) * p.num_tiles + t]) + __ldcg(&p.tile_wpre[at]) +
         __popc(__ldcg(&p.tile_bits[at]) & lanes_below(gl & 31));
}

// Column total col, from global memory (written by other CTAs) or from the
// CTA's own shared memory.
template <bool SMEM>
__device__ __forceinline__ int load_total(const int* tot, int col) {
  if (SMEM) return tot[col];
  return __ldcg(&tot[col]);
}

// One warp turns the column totals tot[P+E] (ranks, then experts) into the
// offsets, in shared memory: expert segments padded to A (exp_off), padding
// rows per expert (pad_off) and receive windows (recv_off), each an
// exclusive scan with its total at the end; sizes[] gets {N_recv, N_exp,
// N_pad}.  Each lane scans a contiguous run of each array, one shuffle scan
// joins the lanes.  The first batch of rank totals is loaded together with
// the first batch of expert totals (one round trip up to 256 experts and
// 256 ranks).
template <bool SMEM>
__device__ void offsets_warp_scan(const PlanDev& p, const int* tot, int* exp_off, int* pad_off, int* recv_off,
                                  int* sizes) {
  const int lane = threadIdx.x & 31;
  const int per_e = (p.E + 31) / 32;
  const int per_d = (p.P + 31) / 32;
  const int lo_e = lane * per_e;
  const int lo_d = lane * per_d;
  int sum_exp = 0, sum_pad = 0, sum_recv = 0;
  constexpr int kBatch = 8;  // loads issued before any is used
  int nd[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int d = lo_d + u;
    nd[u] = (u < per_d && d < p.P) ? load_total<SMEM>(tot, d) : 0;
  }
  for (int i0 = 0; i0 < per_e; i0 += kBatch) {
    int n[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int e = lo_e + i0 + u;
      n[u] = (i0 + u < per_e && e < p.E) ? load_total<SMEM>(tot, p.P + e) : 0;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int e = lo_e + i0 + u;
      if (i0 + u < per_e && e < p.E) {
        const int v = (n[u] + p.A - 1) / p.A * p.A;
        exp_off[e] = v;
        pad_off[e] = v - n[u];
        sum_exp += v;
        sum_pad += v - n[u];
      }
    }
  }
  for (int i0 = 0; i0 < per_d; i0 += kBatch) {
    int n[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int d = lo_d + i0 + u;
      n[u] = i0 == 0 ? nd[u] : ((i0 + u < per_d && d < p.P) ? load_total<SMEM>(tot, d) : 0);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int d = lo_d + i0 + u;
      if (i0 + u < per_d && d < p.P) {
        recv_off[d] = n[u];
        sum_recv += n[u];
      }
    }
  }
  int inc_exp = sum_exp, inc_pad = sum_pad, inc_recv = sum_recv;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, inc_exp, off);
    const int b = __shfl_up_sync(0xffffffffu, inc_pad, off);
    const int c = __shfl_up_sync(0xffffffffu, inc_recv, off);
    if (lane >= off) {
      inc_exp += a;
      inc_pad += b;
      inc_recv += c;
    }
  }
  int run_exp = inc_exp - sum_exp, run_pad = inc_pad - sum_pad, run_recv = inc_recv - sum_recv;
  for (int i = 0; i < per_e; ++i) {
    const int e = lo_e + i;
    if (e < p.E) {
      const int ve = exp_off[e], vp = pad_off[e];
      exp_off[e] = run_exp;
      pad_off[e] = run_pad;
      run_exp += ve;
      run_pad += vp;
    }
  }
  for (int i = 0; i < per_d; ++i) {
    const int d = lo_d + i;
    if (d < p.P) {
      const int v = recv_off[d];
      recv_off[d] = run_recv;
      run_recv += v;
    }
  }
  if (lane == 31) {
    exp_off[p.E] = inc_exp;
    pad_off[p.E] = inc_pad;
    recv_off[p.P] = inc_recv;
    sizes[kSizeRecv] = inc_recv;
    sizes[kSizeExp] = inc_exp;
    sizes[kSizePad] = inc_pad;
  }
}

// PROF: the same kernel, plus a per-CTA record: marks after the route scan
// of its last tile and past each grid barrier; the tokens it scanned.
template <bool PROF, int KMAX>
__global__ void __launch_bounds__(kTile, kPlanThreadsPerSm / kTile) ep_plan_kernel(PlanDev p) {
  extern __shared__ __align__(16) uint32_t smem[];
  unsigned long long t_start = 0, t_scan = 0, t_bar1 = 0, t_bar2 = 0, scanned = 0;
  if (PROF && threadIdx.x == 0) t_start = prof_now();
  // this launch's barrier count, and whether a launch before it timed out
  // (thread 0; both reads are first used at barrier 1)
  const unsigned gen = threadIdx.x == 0 ? __ldcg(&p.ctr[kCtrBarGen]) : 0u;
  const unsigned status0 = threadIdx.x == 0 ? __ldcg(&p.ctr[kCtrStatus]) : 0u;
  unsigned* bar_count = p.ctr + ((gen & 1u) ? kCtrBarCount1 : kCtrBarCount);

  // ---------------- phase 1: tiles ----------------
  uint32_t* bits = smem;                                           // [kTileWords * ncols]
  int* ids = reinterpret_cast<int*>(bits + kTileWords * p.ncols);  // [kTile * K]
  int* s_run = ids + kTile * p.K;                                  // [ncols] tile's exclusive prefix
  for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
    // test hook: a tile that never arrives at the first barrier
    if (tile == p.suppress_tile) return;
    const int64_t t0 = static_cast<int64_t>(tile) * kTile;
    for (int i = threadIdx.x; i < kTileWords * p.ncols; i += blockDim.x) bits[i] = 0u;
    load_tile_ids<KMAX>(p, t0, ids);
    __syncthreads();
    build_tile_bits(p, ids, bits);
    __syncthreads();
    if (PROF && threadIdx.x == 0) {
      t_scan = prof_now();
      scanned += static_cast<unsigned long long>(min64(kTile, p.T - t0));
    }
    uint32_t* g_bits = p.tile_bits + static_cast<int64_t>(tile) * kTileWords * p.ncols;
    int* g_wpre = p.tile_wpre + static_cast<int64_t>(tile) * kTileWords * p.ncols;
    for (int i = threadIdx.x; i < kTileWords * p.ncols; i += blockDim.x) g_bits[i] = bits[i];
    // per column: word prefixes inside the tile, and the tile's count
    for (int col = threadIdx.x; col < p.ncols; col += blockDim.x) {
      int n = 0;
#pragma unroll
      for (int j = 0; j < kTileWords; ++j) {
        g_wpre[j * p.ncols + col] = n;
        n += __popc(bits[j * p.ncols + col]);
      }
      p.agg[static_cast<int64_t>(col) * p.num_tiles + tile] = n;
    }
    __syncthreads();  // before the next tile reuses shared memory (and for phase 2)
  }

  if (!grid_sync(p, bar_count, 1, (status0 & kStTimeout) != 0)) {
    if (threadIdx.x == 0) atomicOr(&p.ctr[kCtrStatus], kStTimeout);
    return;
  }
  if (PROF && threadIdx.x == 0) t_bar1 = prof_now();
  column_scans(p);
  if (!grid_sync(p, bar_count, 2, false)) {
    if (threadIdx.x == 0) atomicOr(&p.ctr[kCtrStatus], kStTimeout);
    return;
  }
  if (PROF && threadIdx.x == 0) t_bar2 = prof_now();
  if (blockIdx.x == 0 && threadIdx.x == 0 && gridDim.x > 1) {
    // nobody uses the other count in this launch: zero it for the next one
    p.ctr[(gen & 1u) ? kCtrBarCount : kCtrBarCount1] = 0u;
    p.ctr[kCtrBarGen] = gen + 1u;
  }

  // ---------------- phase 2: every plan array, all CTAs ----------------
  int* exp_off = s_run + p.ncols;               // [E+1]
  int* pad_off = exp_off + (p.E + 1);           // [E+1]
  int* recv_off = pad_off + (p.E + 1);          // [P+1]
  int* s_slot = recv_off + (p.P + 1);           // [kTile * K] own tile's slots
  __shared__ int s_sizes[3];
  const bool own_tile = gridDim.x >= static_cast<unsigned>(p.num_tiles);
  const bool has_tile = own_tile && blockIdx.x < static_cast<unsigned>(p.num_tiles);
  if (threadIdx.x < 32) {
    offsets_warp_scan<false>(p, p.totals_rep + static_cast<int64_t>(blockIdx.x % kTotRep) * p.ncols, exp_off, pad_off,
                             recv_off, s_sizes);
  } else if (has_tile) {
    // the own tile's exclusive prefix per column
    for (int col = threadIdx.x - 32; col < p.ncols; col += blockDim.x - 32)
      s_run[col] = __ldcg(&p.tile_pre[static_cast<int64_t>(col) * p.num_tiles + blockIdx.x]);
  }
  __syncthreads();
  const int n_recv = s_sizes[kSizeRecv];
  const int n_exp = s_sizes[kSizeExp];
  const int n_pad = s_sizes[kSizePad];
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
      p.exp_off[i] = exp_off[i];
      p.pad_off[i] = pad_off[i];
    }
    for (int i = threadIdx.x; i <= p.P; i += blockDim.x) p.recv_off[i] = recv_off[i];
    if (threadIdx.x == 0) {
      p.sizes[kSizeRecv] = n_recv;
      p.sizes[kSizeExp] = n_exp;
      p.sizes[kSizePad] = n_pad;
    }
  }

  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // With at least one CTA per tile, every CTA still holds its own tile in
  // shared memory (ids, bit matrix, exclusive prefix): its tokens' slots
  // need no global loads.  CTAs without a tile take the small passes.  (The
  // tile's [T,P] rows from shared memory too measured slower: the rows are
  // better spread over all CTAs.)
  const int64_t extra = own_tile ? static_cast<int64_t>(gridDim.x - p.num_tiles) * blockDim.x : 0;
  // thread range of the small passes (negative: this thread takes none)
  const int64_t stid = extra > 0 ? gtid - static_cast<int64_t>(p.num_tiles) * blockDim.x : gtid;
  const int64_t snthr = extra > 0 ? extra : nthr;
  const bool small_passes = stid >= 0;

  if (own_tile) {
    if (has_tile) {
      // one token per thread; the slots are staged in shared memory and
      // leave as one contiguous block
      const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTile;
      const int n_tok = static_cast<int>(min64(kTile, p.T - t0));
      const int i = threadIdx.x;
      if (i < n_tok) {
        for (int k = 0; k < p.K; ++k) {
          const int e = ids[i * p.K + k];
          int r = -1;
          if (e >= 0) {
            r = exp_off[e] + tile_pos(bits, s_run, p.ncols, p.P + e, i);
            if (in_cap(r, p.cap_exp)) {
              p.exp_src[r] = static_cast<int>(t0 + i);
            } else {
              atomicOr(&p.ctr[kCtrStatus], kStCapacity);
              r = -1;
            }
          }
          s_slot[i * p.K + k] = r;
        }
      }
      __syncthreads();
      for (int j = threadIdx.x; j < n_tok * p.K; j += blockDim.x) p.slot[t0 * p.K + j] = s_slot[j];
    }
  } else {
    // slot and exp_src, one token per thread: the token's K ids, then all
    // their window positions, are loaded before any is used.
    for (int64_t g = gtid; g < p.T; g += nthr) {
      int e[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        const long long v = k < p.K ? p.topk_idx[g * p.K + k] : -1ll;
        e[k] = (v >= 0 && v < p.E) ? static_cast<int>(v) : -1;
      }
      const int64_t t = g / kTile;
      const int gl = static_cast<int>(g - t * kTile);
      const int64_t word = (t * kTileWords + (gl >> 5)) * p.ncols + p.P;
      int pre[KMAX];
      uint32_t bw[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        pre[k] = 0;
        bw[k] = 0u;
        if (e[k] >= 0) {
          pre[k] = __ldcg(&p.tile_pre[static_cast<int64_t>(p.P + e[k]) * p.num_tiles + t]) +
                   __ldcg(&p.tile_wpre[word + e[k]]);
          bw[k] = __ldcg(&p.tile_bits[word + e[k]]);
        }
      }
      const uint32_t below = lanes_below(gl & 31);
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k >= p.K) break;
        int r = -1;
        if (e[k] >= 0) {
          r = exp_off[e[k]] + pre[k] + __popc(bw[k] & below);
          if (in_cap(r, p.cap_exp)) {
            p.exp_src[r] = static_cast<int>(g);
          } else {
            atomicOr(&p.ctr[kCtrStatus], kStCapacity);
            r = -1;
          }
        }
        p.slot[g * p.K + k] = r;
      }
    }
  }

  // dense [T,P]: is_token_in_rank, send_head, and recv_src_idx.  One thread
  // per (32-token word, sub-group of the word, rank d): one bit word and its
  // prefix, then the sub-group's tokens with a running count.  Threads keep
  // a fixed d (the stride is a multiple of P), lanes hold consecutive d, so
  // each store of a token row is coalesced.  The word is split into `sub`
  // groups so that there are about as many units as threads.
  {
    const int64_t words = (p.T + 31) / 32;
    const int64_t lanes_d = (nthr / p.P) * p.P;  // threads used: a multiple of P
    // the largest split that still gives every thread at most one unit
    int sub = 1;
    while (sub < 32 && words * (2 * sub) * p.P <= lanes_d) sub <<= 1;
    const int per = 32 / sub;
    const int log_sub = __ffs(sub) - 1;
    // units go to the CTAs without a tile first: the others have slots to write
    const int64_t dtid = own_tile ? (gtid + nthr - static_cast<int64_t>(p.num_tiles) * blockDim.x) % nthr : gtid;
    if (dtid < lanes_d) {
      const int d = static_cast<int>(dtid % p.P);
      const int base = recv_off[d];
      const int64_t step = lanes_d / p.P;
      for (int64_t wq = dtid / p.P; wq < words * sub; wq += step) {
        const int64_t tw = wq >> log_sub;  // word index: tile * kTileWords + warp
        const int l0 = static_cast<int>(wq & (sub - 1)) * per;
        const int64_t at = tw * p.ncols + d;
        const uint32_t word = __ldcg(&p.tile_bits[at]);
        int pos = __ldcg(&p.tile_pre[static_cast<int64_t>(d) * p.num_tiles + (tw / kTileWords)]) +
                  __ldcg(&p.tile_wpre[at]) + __popc(word & lanes_below(l0));
        const int64_t g0 = tw * 32 + l0;
        const int n_tok = static_cast<int>(min64(per, p.T - g0));
        int t_local = static_cast<int>(static_cast<uint32_t>(g0) % static_cast<uint32_t>(p.S));
        for (int l = 0; l < n_tok; ++l) {
          const int64_t g = g0 + l;
          const int bit = (word >> (l0 + l)) & 1;
          p.in_rank[g * p.P + d] = static_cast<unsigned char>(bit);
          p.send_head[g * p.P + d] = bit ? pos : -1;
          if (bit) {
            const int64_t at_r = static_cast<int64_t>(base) + pos++;
            if (in_cap(at_r, p.cap_recv))
              p.recv_src_idx[at_r] = t_local;
            else
              atomicOr(&p.ctr[kCtrStatus], kStCapacity);
          }
          if (++t_local == p.S) t_local = 0;
        }
      }
    }
  }

  // prefix matrices, one (s, d, c) per thread; layout of i is [s][d][c]
#pragma unroll 2
  // The small passes below start at different points of the thread range,
  // so that they do not all land on the first CTAs after the slot pass.
  for (int64_t i = small_passes ? (stid + snthr / 2) % snthr : INT64_MAX; i < static_cast<int64_t>(p.P) * p.P * p.C;
       i += snthr) {
    const int c = static_cast<int>(i % p.C);
    const int64_t sd = i / p.C;
    const int d = static_cast<int>(sd % p.P);
    const int64_t s = sd / p.P;
    const int64_t src0 = s * p.S;
    const int64_t lo = src0 + min64(p.S, static_cast<int64_t>(c) * p.chunk);
    const int64_t hi = src0 + min64(p.S, static_cast<int64_t>(c + 1) * p.chunk);
    const int x0 = x_at(p, d, src0);
    p.rcpm[(static_cast<int64_t>(d) * p.P + s) * p.C + c] = x_at(p, d, lo);
    p.cpm[i] = x_at(p, d, hi) - x0;
    if (c == 0) {
      const int x1 = x_at(p, d, src0 + p.S);
      p.rpm[s * p.P + d] = x1;
      p.ntpr[s * p.P + d] = x1 - x0;
    }
  }

  // per-source expert counts
  for (int i = small_passes ? static_cast<int>((stid + 3 * snthr / 4) % snthr) : INT32_MAX; i < p.P * p.E;
       i += static_cast<int>(snthr)) {
    const int s = i / p.E;
    const int e = i - s * p.E;
    p.ntpe[i] = x_at(p, p.P + e, (s + 1) * p.S) - x_at(p, p.P + e, static_cast<int64_t>(s) * p.S);
  }

  // padding rows of the expanded layout
  const int64_t n_pad_w = n_pad < p.cap_pad ? n_pad : p.cap_pad;
  if (small_passes && stid == 0 && n_pad > p.cap_pad) atomicOr(&p.ctr[kCtrStatus], kStCapacity);
  for (int64_t i = small_passes ? (stid + snthr / 4) % snthr : INT64_MAX; i < n_pad_w; i += snthr) {
    int lo = 0, hi = p.E;  // e with pad_off[e] <= i < pad_off[e+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pad_off[mid] <= i) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int n_e = (exp_off[e + 1] - exp_off[e]) - (pad_off[e + 1] - pad_off[e]);
    const int row = exp_off[e] + n_e + static_cast<int>(i - pad_off[e]);
    p.pad_rows[i] = row;
    if (in_cap(row, p.cap_exp))
      p.exp_src[row] = -1;
    else
      atomicOr(&p.ctr[kCtrStatus], kStCapacity);
  }
  if (PROF) prof_cta_end(p, kProfPlan, t_start, t_scan, t_bar1, t_bar2, scanned, 0);
}

// X_col(g) of a one-tile plan, all in shared memory: the word prefix of g's
// word plus the bits before g in it; g == T gives the column total.
__device__ __forceinline__ int x_one(const uint32_t* bits, const int* wpre, const int* tot, int ncols, int col,
                                     int g, int T) {
  if (g >= T) return tot[col];
  const int at = (g >> 5) * ncols + col;
  return wpre[at] + __popc(bits[at] & lanes_below(g & 31));
}

// The whole plan of at most one tile (T <= 256 tokens) in one CTA, with every
// intermediate in shared memory: the bit matrix, each word's prefix inside
// the column, the column totals and the offsets.  The only global loads are
// the routing ids; every output is a store.  (The general kernel with one
// CTA computes the same through global scratch: a chain of L2 round trips.)
// PROF marks: [2] route scan done, [3] column counts done, [4] offsets done.
template <bool PROF, int KMAX>
__global__ void __launch_bounds__(kTile, 1) ep_plan_one_tile_kernel(PlanDev p) {
  extern __shared__ __align__(16) uint32_t smem[];
  unsigned long long t_start = 0, t_scan = 0, t_count = 0, t_off = 0;
  if (PROF && threadIdx.x == 0) t_start = prof_now();
  const int nc = p.ncols;
  const int T = static_cast<int>(p.T);
  uint32_t* bits = smem;                                      // [kTileWords][ncols]
  int* wpre = reinterpret_cast<int*>(bits + kTileWords * nc);  // [kTileWords][ncols]
  int* tot = wpre + kTileWords * nc;                           // [ncols]
  int* ids = tot + nc;                                         // [kTile * K], then the slots
  int* exp_off = ids + kTile * p.K;                            // [E+1]
  int* pad_off = exp_off + (p.E + 1);                          // [E+1]
  int* recv_off = pad_off + (p.E + 1);                         // [P+1]
  __shared__ int s_sizes[3];

  for (int i = threadIdx.x; i < kTileWords * nc; i += blockDim.x) bits[i] = 0u;
  load_tile_ids<KMAX>(p, 0, ids);
  __syncthreads();
  build_tile_bits(p, ids, bits);
  __syncthreads();
  if (PROF && threadIdx.x == 0) t_scan = prof_now();
  for (int col = threadIdx.x; col < nc; col += blockDim.x) {
    int n = 0;
#pragma unroll
    for (int j = 0; j < kTileWords; ++j) {
      wpre[j * nc + col] = n;
      n += __popc(bits[j * nc + col]);
    }
    tot[col] = n;
    p.totals[col] = n;
  }
  __syncthreads();
  if (PROF && threadIdx.x == 0) t_count = prof_now();
  if (threadIdx.x < 32) {
    offsets_warp_scan<true>(p, tot, exp_off, pad_off, recv_off, s_sizes);
  } else {
    // the outputs that need no offsets, while warp 0 scans: the prefix
    // matrices and per-source expert counts
    const int tid = threadIdx.x - 32, nthr = blockDim.x - 32;
    const int S = static_cast<int>(p.S);
    for (int i = tid; i < p.P * p.P * p.C; i += nthr) {
      const int c = i % p.C;
      const int sd = i / p.C;
      const int d = sd % p.P;
      const int s = sd / p.P;
      const int src0 = s * S;
      const int lo = src0 + static_cast<int>(min64(p.S, static_cast<int64_t>(c) * p.chunk));
      const int hi = src0 + static_cast<int>(min64(p.S, static_cast<int64_t>(c + 1) * p.chunk));
      const int x0 = x_one(bits, wpre, tot, nc, d, src0, T);
      p.rcpm[(d * p.P + s) * p.C + c] = x_one(bits, wpre, tot, nc, d, lo, T);
      p.cpm[i] = x_one(bits, wpre, tot, nc, d, hi, T) - x0;
      if (c == 0) {
        const int x1 = x_one(bits, wpre, tot, nc, d, src0 + S, T);
        p.rpm[s * p.P + d] = x1;
        p.ntpr[s * p.P + d] = x1 - x0;
      }
    }
    for (int i = tid; i < p.P * p.E; i += nthr) {
      const int s = i / p.E;
      const int e = i - s * p.E;
      p.ntpe[i] = x_one(bits, wpre, tot, nc, p.P + e, (s + 1) * S, T) - x_one(bits, wpre, tot, nc, p.P + e, s * S, T);
    }
  }
  __syncthreads();
  if (PROF && threadIdx.x == 0) t_off = prof_now();
  const int n_pad = s_sizes[kSizePad];
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
    p.exp_off[i] = exp_off[i];
    p.pad_off[i] = pad_off[i];
  }
  for (int i = threadIdx.x; i <= p.P; i += blockDim.x) p.recv_off[i] = recv_off[i];
  if (threadIdx.x == 0) {
    p.sizes[kSizeRecv] = s_sizes[kSizeRecv];
    p.sizes[kSizeExp] = s_sizes[kSizeExp];
    p.sizes[kSizePad] = n_pad;
  }
  // slots and exp_src, one token per thread; each slot replaces its id in
  // shared memory and the block leaves as one contiguous store
  if (threadIdx.x < T) {
    const int i = threadIdx.x;
    for (int k = 0; k < p.K; ++k) {
      const int e = ids[i * p.K + k];
      int r = -1;
      if (e >= 0) {
        r = exp_off[e] + x_one(bits, wpre, tot, nc, p.P + e, i, T);
        if (in_cap(r, p.cap_exp)) {
          p.exp_src[r] = i;
        } else {
          atomicOr(&p.ctr[kCtrStatus], kStCapacity);
          r = -1;
        }
      }
      ids[i * p.K + k] = r;
    }
  }
  // dense [T,P]: is_token_in_rank, send_head, recv_src_idx; one token per
  // thread, its ranks in turn (no division per entry: the CTA span of the
  // tiny plan 4.83 -> 4.13 us against one (token, rank) per thread)
  if (threadIdx.x < T) {
    const int g = threadIdx.x;
    const int t_local = g % static_cast<int>(p.S);
    const uint32_t below = lanes_below(g & 31);
    for (int d = 0; d < p.P; ++d) {
      const int at = (g >> 5) * nc + d;
      const uint32_t word = bits[at];
      const int bit = (word >> (g & 31)) & 1;
      const int pos = wpre[at] + __popc(word & below);
      p.in_rank[g * p.P + d] = static_cast<unsigned char>(bit);
      p.send_head[g * p.P + d] = bit ? pos : -1;
      if (bit) {
        const int64_t at_r = static_cast<int64_t>(recv_off[d]) + pos;
        if (in_cap(at_r, p.cap_recv))
          p.recv_src_idx[at_r] = t_local;
        else
          atomicOr(&p.ctr[kCtrStatus], kStCapacity);
      }
    }
  }
  // padding rows of the expanded layout
  const int n_pad_w = n_pad < p.cap_pad ? n_pad : static_cast<int>(p.cap_pad);
  if (threadIdx.x == 0 && n_pad > p.cap_pad) atomicOr(&p.ctr[kCtrStatus], kStCapacity);
  for (int i = threadIdx.x; i < n_pad_w; i += blockDim.x) {
    int lo = 0, hi = p.E;  // e with pad_off[e] <= i < pad_off[e+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pad_off[mid] <= i) lo = mid; else hi = mid;
    }
    const int n_e = (exp_off[lo + 1] - exp_off[lo]) - (pad_off[lo + 1] - pad_off[lo]);
    const int row = exp_off[lo] + n_e + (i - pad_off[lo]);
    p.pad_rows[i] = row;
    if (in_cap(row, p.cap_exp))
      p.exp_src[row] = -1;
    else
      atomicOr(&p.ctr[kCtrStatus], kStCapacity);
  }
  __syncthreads();
  for (int j = threadIdx.x; j < T * p.K; j += blockDim.x) p.slot[j] = ids[j];
  if (PROF)  // units: the tokens scanned, counted once (prof_cta_end sums over the warps)
    prof_cta_end(p, kProfPlan, t_start, t_scan, t_count, t_off,
                 threadIdx.x == 0 ? static_cast<unsigned long long>(T) : 0ull, 0);
}

}  // namespace

size_t plan_smem_bytes(int P, int E, int K) {
  // phase 1: bit matrix, ids, exclusive prefix per column (kept for phase 2);
  // phase 2: the offsets and the own tile's slots
  return sizeof(uint32_t) * kTileWords * (P + E) + sizeof(int) * (kTile * K + (P + E)) +
         sizeof(int) * (2 * (E + 1) + (P + 1) + kTile * K);
}

// Shared memory of the one-tile kernel: bit matrix, word prefixes, totals,
// ids (then slots) and the offsets.
size_t plan_one_tile_smem_bytes(int P, int E, int K) {
  return sizeof(uint32_t) * kTileWords * (P + E) * 2 + sizeof(int) * (P + E) + sizeof(int) * kTile * K +
         sizeof(int) * (2 * (E + 1) + (P + 1));
}

// Phase-2 outputs per CTA that size the grid (tuning knob).
#ifndef EP_PLAN_WORK_PER_CTA
#define EP_PLAN_WORK_PER_CTA 1024
#endif

namespace {

// Co-resident CTAs (at most two per SM, which keeps the grid barrier cheap;
// under an SM budget, two per budgeted SM), and no more than the plan's work
// needs: one CTA per tile at least, and about one CTA per
// EP_PLAN_WORK_PER_CTA phase-2 outputs.  Phase 1 loops over the tiles when the grid is smaller.
template <bool PROF, int KMAX>
int plan_grid(const PlanDev& p, int sm_budget) {
  const size_t smem = plan_smem_bytes(p.P, p.E, p.K);
  // occupancy, cached per host thread for the last (device, shared memory)
  // it was asked for
  thread_local int cached_dev = -1;
  thread_local size_t cached_smem = ~static_cast<size_t>(0);
  thread_local int cached_per_sm = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (smem != cached_smem || dev != cached_dev) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ep_plan_kernel<PROF, KMAX>, kTile, smem) != cudaSuccess ||
        per_sm < 1)
      return 0;
    cached_per_sm = per_sm > kPlanThreadsPerSm / kTile ? kPlanThreadsPerSm / kTile : per_sm;
    cached_smem = smem;
    cached_dev = dev;
  }
  const int sms = sm_budget > 0 && sm_budget < num_sms() ? sm_budget : num_sms();
  const int64_t cap = static_cast<int64_t>(cached_per_sm) * sms;
  if (p.num_tiles == 1) return 1;  // one tile: one CTA, no grid barrier, no cooperative launch
  const int64_t work = p.T * (p.K + p.P) + static_cast<int64_t>(p.P) * p.P * p.C + static_cast<int64_t>(p.P) * p.E;
  int64_t grid = (work + EP_PLAN_WORK_PER_CTA - 1) / EP_PLAN_WORK_PER_CTA;
  if (grid < p.num_tiles) grid = p.num_tiles;
  if (grid > cap) grid = cap;
  // the dense [T,P] pass keeps one rank per thread: at least P threads, even
  // under a tight SM budget (the whole device co-hosts far more)
  const int64_t min_grid = (p.P + kTile - 1) / kTile;
  const int64_t full = static_cast<int64_t>(cached_per_sm) * num_sms();
  if (grid < min_grid) grid = min_grid < full ? min_grid : full;
  return static_cast<int>(grid);
}

// The largest dynamic shared memory a CTA may ask for on this device.
size_t max_dyn_smem() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return 48 * 1024;
  return static_cast<size_t>(v);
}

template <bool PROF, int KMAX>
cudaError_t launch_plan_t(const PlanDev& p, cudaStream_t stream, const LaunchCfg& cfg) {
  if (p.num_tiles == 1) {
    const size_t smem1 = plan_one_tile_smem_bytes(p.P, p.E, p.K);
    if (smem1 <= max_dyn_smem()) {
      if (smem1 > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(ep_plan_one_tile_kernel<PROF, KMAX>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem1));
        if (err != cudaSuccess) return err;
      }
      if (cfg.ctas) *cfg.ctas = 1;
      ep_plan_one_tile_kernel<PROF, KMAX><<<1, kTile, smem1, stream>>>(p);
      return cudaGetLastError();
    }
  }
  const size_t smem = plan_smem_bytes(p.P, p.E, p.K);
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(ep_plan_kernel<PROF, KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
  }
  const int grid = plan_grid<PROF, KMAX>(p, cfg.sm_budget);
  if (grid < 1) return cudaErrorInvalidConfiguration;
  if (grid == 1) {
    if (cfg.ctas) *cfg.ctas = 1;
    ep_plan_kernel<PROF, KMAX><<<1, kTile, smem, stream>>>(p);
    return cudaGetLastError();
  }
  PlanDev arg = p;
  void* args[] = {&arg};
  if (cfg.ctas) *cfg.ctas = grid;
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(ep_plan_kernel<PROF, KMAX>), dim3(grid), dim3(kTile),
                                     args, smem, stream);
}

}  // namespace

cudaError_t launch_plan(const PlanDev& p, cudaStream_t stream, const LaunchCfg& cfg) {
  // top-k arrays sized for K <= 8 or K <= 16: less unrolled code for the
  // common small K (the kernel runs once per plan, its code cold in the
  // instruction cache)
  if (p.K <= 8)
    return p.prof_rec ? launch_plan_t<true, 8>(p, stream, cfg) : launch_plan_t<false, 8>(p, stream, cfg);
  return p.prof_rec ? launch_plan_t<true, EP_MAX_TOPK>(p, stream, cfg)
                    : launch_plan_t<false, EP_MAX_TOPK>(p, stream, cfg);
}

}  // namespace ep
