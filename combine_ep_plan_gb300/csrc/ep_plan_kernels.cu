// ep_plan_kernels.cu — the routing plan on sm_103a.
//
// Three kernels, in stream order:
//   1. ep_count_kernel: per tile of 256 tokens, a bit matrix in shared memory
//      with one 32-bit word per (column, warp): column = destination rank d
//      (deduplicated by the OR) or expert e.  Warp-aggregated updates
//      (__match_any_sync, one shared atomicOr per distinct key per warp).
//      Column totals and per-source expert counts go to global memory with one
//      atomic per non-zero (tile, column).  The last CTA to finish turns the
//      totals into padded expert offsets, receive-window offsets and padding
//      offsets.
//   2. ep_emit_kernel: the same bit matrix, then a single-pass decoupled
//      look-back scan over tiles, column by column (each descriptor packs its
//      state and value in one 64-bit word, so no fence pairs are needed), with
//      a bounded wait.  With the exclusive prefix X of every column it writes
//      is_token_in_rank, send_head, recv_src_idx, slot, exp_src, the padding
//      rows, and X at every channel start (the recv_channel_prefix_matrix).
//   3. ep_prefix_kernel: rank_prefix_matrix, channel_prefix_matrix and
//      num_tokens_per_rank as differences of X at channel and source starts.
//
// Definitions followed ("Ascend DeepEP MoE Dispatch Optimization", the
// dispatch handle table and the notify stage; TileLang tutorial ch. 38
// "DeepEP-Ascend", §1.3 dedup, §2.2 expanded layout and padding, §3.5
// deterministic order):
//   X[g][d]  = #{g' < g : d in dests(g')}             (window row of (g,d))
//   slot     = expert_offset[e] + #{g' < g : e in idx[g']}
//   rcpm[d][s][c] = X[s*S + c*chunk][d]                (segment start)
#include "ep_internal.cuh"

namespace ep {
namespace {

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ unsigned long long ld_desc(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_desc(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Bits set in word-columns [0, i) of one column of the tile bit matrix
// (layout bits[w * ncols + col]).
__device__ __forceinline__ int prefix_in_tile(const uint32_t* bits, int ncols, int col, int i) {
  int w = i >> 5;
  int n = 0;
#pragma unroll
  for (int j = 0; j < kTileWords; ++j)
    if (j < w) n += __popc(bits[j * ncols + col]);
  uint32_t lt = (i & 31) ? (0xffffffffu >> (32 - (i & 31))) : 0u;
  if (w < kTileWords) n += __popc(bits[w * ncols + col] & lt);
  return n;
}

// Bits set in tokens [lo, hi) of one column.
__device__ __forceinline__ int count_range(const uint32_t* bits, int ncols, int col, int lo, int hi) {
  return prefix_in_tile(bits, ncols, col, hi) - prefix_in_tile(bits, ncols, col, lo);
}

// Loads this tile's expert ids into shared memory (coalesced), checking them.
__device__ __forceinline__ void load_tile_ids(const PlanDev& p, int64_t t0, int* ids, bool report) {
  const int64_t base = t0 * p.K;
  const int64_t end = p.T * p.K;
  for (int i = threadIdx.x; i < kTile * p.K; i += blockDim.x) {
    int e = -1;
    if (base + i < end) {
      long long v = p.topk_idx[base + i];
      if (v >= 0 && v < p.E) {
        e = static_cast<int>(v);
      } else if (v != -1 && report) {
        atomicOr(&p.ctr[kCtrStatus], kStInvalidId);
      }
    }
    ids[i] = e;
  }
}

// Builds the tile bit matrix from the ids (shared memory must be zeroed).
// Column d < P: token routed to rank d (OR deduplicates); column P+e: token
// picked expert e.  A duplicate expert in one row shows up as a bit that is
// already set when the leader ORs its lane mask.
__device__ __forceinline__ void build_tile_bits(const PlanDev& p, const int* ids, uint32_t* bits,
                                                bool report) {
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  for (int k = 0; k < p.K; ++k) {
    const int e = ids[threadIdx.x * p.K + k];
    const unsigned me = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(me) - 1) {
      unsigned old = atomicOr(&bits[w * p.ncols + p.P + e], me);
      if ((old & me) && report) atomicOr(&p.ctr[kCtrStatus], kStDuplicate);
    }
    const int d = e >= 0 ? e / p.El : -1;
    const unsigned md = __match_any_sync(0xffffffffu, d);
    if (d >= 0 && lane == __ffs(md) - 1) atomicOr(&bits[w * p.ncols + d], md);
  }
}

// Inclusive-to-exclusive scan of n ints in place, one CTA; returns the total.
__device__ int block_exclusive_scan(int* a, int n, int* scratch /* blockDim.x */) {
  const int nt = blockDim.x;
  const int per = (n + nt - 1) / nt;
  const int lo = threadIdx.x * per;
  int sum = 0;
  for (int i = 0; i < per; ++i)
    if (lo + i < n) sum += a[lo + i];
  scratch[threadIdx.x] = sum;
  __syncthreads();
  for (int off = 1; off < nt; off <<= 1) {
    int v = threadIdx.x >= off ? scratch[threadIdx.x - off] : 0;
    __syncthreads();
    scratch[threadIdx.x] += v;
    __syncthreads();
  }
  int run = scratch[threadIdx.x] - sum;
  for (int i = 0; i < per; ++i)
    if (lo + i < n) {
      int v = a[lo + i];
      a[lo + i] = run;
      run += v;
    }
  const int total = scratch[nt - 1];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kTile) ep_count_kernel(PlanDev p) {
  extern __shared__ __align__(16) uint32_t smem[];
  uint32_t* bits = smem;                                       // [kTileWords * ncols]
  int* ids = reinterpret_cast<int*>(bits + kTileWords * p.ncols);  // [kTile * K]
  __shared__ int scan_scratch[kTile];
  __shared__ bool is_last;

  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTile;
  const int rows = static_cast<int>(min64(kTile, p.T - t0));
  for (int i = threadIdx.x; i < kTileWords * p.ncols; i += blockDim.x) bits[i] = 0u;
  load_tile_ids(p, t0, ids, true);
  __syncthreads();
  build_tile_bits(p, ids, bits, true);
  __syncthreads();

  // Column totals and per-source expert counts (one atomic per non-zero pair).
  const int64_t s_first = t0 / p.S;
  const int64_t s_last = (t0 + rows - 1) / p.S;
  for (int col = threadIdx.x; col < p.ncols; col += blockDim.x) {
    int n = 0;
#pragma unroll
    for (int j = 0; j < kTileWords; ++j) n += __popc(bits[j * p.ncols + col]);
    if (n == 0) continue;
    atomicAdd(&p.totals[col], n);
    if (col >= p.P) {
      const int e = col - p.P;
      if (s_first == s_last) {
        atomicAdd(&p.ntpe[s_first * p.E + e], n);
      } else {
        for (int64_t s = s_first; s <= s_last; ++s) {
          int lo = static_cast<int>(max64(s * p.S, t0) - t0);
          int hi = static_cast<int>(min64((s + 1) * p.S, t0 + rows) - t0);
          int m = count_range(bits, p.ncols, col, lo, hi);
          if (m) atomicAdd(&p.ntpe[s * p.E + e], m);
        }
      }
    }
  }

  // The last CTA derives the offsets from the totals.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(&p.ctr[kCtrCountDone], 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  // Reuse the bit-matrix space: [E+1] padded sizes, [E+1] pads, [P+1] receives.
  int* padded = reinterpret_cast<int*>(smem);
  int* pads = padded + (p.E + 1);
  int* recv = pads + (p.E + 1);
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    const int n = __ldcg(&p.totals[p.P + e]);
    const int v = (n + p.A - 1) / p.A * p.A;
    padded[e] = v;
    pads[e] = v - n;
  }
  for (int d = threadIdx.x; d < p.P; d += blockDim.x) recv[d] = __ldcg(&p.totals[d]);
  __syncthreads();
  const int n_exp = block_exclusive_scan(padded, p.E, scan_scratch);
  const int n_pad = block_exclusive_scan(pads, p.E, scan_scratch);
  const int n_recv = block_exclusive_scan(recv, p.P, scan_scratch);
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
    p.exp_off[e] = padded[e];
    p.pad_off[e] = pads[e];
  }
  for (int d = threadIdx.x; d < p.P; d += blockDim.x) p.recv_off[d] = recv[d];
  if (threadIdx.x == 0) {
    p.exp_off[p.E] = n_exp;
    p.pad_off[p.E] = n_pad;
    p.recv_off[p.P] = n_recv;
    p.sizes[kSizeRecv] = n_recv;
    p.sizes[kSizeExp] = n_exp;
    p.sizes[kSizePad] = n_pad;
  }
}

// Exclusive prefix of one column over all earlier tiles, by decoupled
// look-back: walk back through predecessors eight at a time, adding
// aggregates until an inclusive prefix is found.  Every poll is bounded.
__device__ int lookback(const PlanDev& p, int tile, int col, bool* timed_out) {
  constexpr int kWindow = 8;
  int sum = 0;
  int j = tile - 1;
  long long polls = 0;
  while (j >= 0) {
    unsigned long long v[kWindow];
#pragma unroll
    for (int u = 0; u < kWindow; ++u)
      v[u] = (j - u >= 0) ? ld_desc(&p.desc[static_cast<int64_t>(j - u) * p.ncols + col]) : 0ull;
#pragma unroll
    for (int u = 0; u < kWindow; ++u) {
      if (j - u < 0) break;
      unsigned long long d = v[u];
      unsigned ns = 32;
      while ((d >> 32) == 0ull) {
        if (++polls > p.poll_limit) {
          *timed_out = true;
          return sum;  // give up; the result is flagged invalid
        }
        __nanosleep(ns);
        if (ns < 1024) ns <<= 1;
        d = ld_desc(&p.desc[static_cast<int64_t>(j - u) * p.ncols + col]);
      }
      sum += static_cast<int>(static_cast<unsigned>(d));
      if ((d >> 32) == kDescInclusive) return sum;
    }
    j -= kWindow;
  }
  return sum;
}

__global__ void __launch_bounds__(kTile) ep_emit_kernel(PlanDev p) {
  extern __shared__ __align__(16) uint32_t smem[];
  uint32_t* bits = smem;                                           // [kTileWords * ncols]
  int* excl = reinterpret_cast<int*>(bits + kTileWords * p.ncols);  // [ncols]
  int* ids = excl + p.ncols;                                       // [kTile * K]
  int* recv_off = ids + kTile * p.K;                               // [P+1]
  int* exp_off = recv_off + (p.P + 1);                             // [E+1]
  __shared__ int s_tile;
  __shared__ int s_timeout;

  if (threadIdx.x == 0) {
    s_tile = static_cast<int>(atomicAdd(&p.ctr[kCtrTicket], 1u));
    s_timeout = 0;
  }
  for (int i = threadIdx.x; i < kTileWords * p.ncols; i += blockDim.x) bits[i] = 0u;
  for (int i = threadIdx.x; i <= p.P; i += blockDim.x) recv_off[i] = p.recv_off[i];
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) exp_off[i] = p.exp_off[i];
  __syncthreads();
  const int tile = s_tile;
  const int64_t t0 = static_cast<int64_t>(tile) * kTile;
  const int rows = static_cast<int>(min64(kTile, p.T - t0));
  load_tile_ids(p, t0, ids, false);
  __syncthreads();
  build_tile_bits(p, ids, bits, false);
  __syncthreads();

  // Publish this tile's aggregate (tile 0: its inclusive prefix) per column.
  const bool publish = tile != p.suppress_tile;
  unsigned long long* my_desc = p.desc + static_cast<int64_t>(tile) * p.ncols;
  for (int col = threadIdx.x; col < p.ncols; col += blockDim.x) {
    int n = 0;
#pragma unroll
    for (int j = 0; j < kTileWords; ++j) n += __popc(bits[j * p.ncols + col]);
    excl[col] = n;
    if (publish)
      st_desc(&my_desc[col], ((tile == 0 ? kDescInclusive : kDescAggregate) << 32) |
                                 static_cast<unsigned>(n));
  }
  // Look back, then publish the inclusive prefix.
  if (tile > 0) {
    bool timed_out = false;
    for (int col = threadIdx.x; col < p.ncols; col += blockDim.x) {
      const int n = excl[col];
      const int pre = lookback(p, tile, col, &timed_out);
      excl[col] = pre;
      if (publish) st_desc(&my_desc[col], (kDescInclusive << 32) | static_cast<unsigned>(pre + n));
    }
    if (timed_out) s_timeout = 1;
  } else {
    for (int col = threadIdx.x; col < p.ncols; col += blockDim.x) excl[col] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0 && s_timeout) atomicOr(&p.ctr[kCtrStatus], kStTimeout);

  // slot and exp_src, one thread per token.
  if (threadIdx.x < rows) {
    const int64_t g = t0 + threadIdx.x;
    for (int k = 0; k < p.K; ++k) {
      const int e = ids[threadIdx.x * p.K + k];
      int r = -1;
      if (e >= 0) {
        const int col = p.P + e;
        r = exp_off[e] + excl[col] + prefix_in_tile(bits, p.ncols, col, threadIdx.x);
        p.exp_src[r] = static_cast<int>(g);
      }
      p.slot[g * p.K + k] = r;
    }
  }

  // Dense [rows, P] outputs: is_token_in_rank, send_head, and recv_src_idx.
  const int dense = rows * p.P;
  for (int i = threadIdx.x; i < dense; i += blockDim.x) {
    const int gl = i / p.P;
    const int d = i - gl * p.P;
    const uint32_t word = bits[(gl >> 5) * p.ncols + d];
    const int bit = (word >> (gl & 31)) & 1;
    const int64_t g = t0 + gl;
    int pos = -1;
    if (bit) {
      pos = excl[d] + prefix_in_tile(bits, p.ncols, d, gl);
      p.recv_src_idx[recv_off[d] + pos] = static_cast<int>(g % p.S);
    }
    p.in_rank[t0 * p.P + i] = static_cast<unsigned char>(bit);
    p.send_head[t0 * p.P + i] = pos;
  }

  // X at every channel start inside this tile: the segment starts of the
  // recv_channel_prefix_matrix.
  const int64_t s_first = t0 / p.S;
  const int64_t s_last = (t0 + rows - 1) / p.S;
  for (int64_t s = s_first; s <= s_last; ++s) {
    const int64_t src0 = s * p.S;
    // channels c with start src0 + c*chunk in [t0, t0 + rows) and c*chunk < S
    int64_t c_lo = t0 > src0 ? (t0 - src0 + p.chunk - 1) / p.chunk : 0;
    int64_t c_hi = (t0 + rows - 1 - src0) / p.chunk;  // inclusive
    c_hi = min64(c_hi, p.C - 1);
    c_hi = min64(c_hi, (p.S - 1) / p.chunk);
    if (c_hi < c_lo) continue;
    const int nstart = static_cast<int>(c_hi - c_lo + 1);
    for (int i = threadIdx.x; i < nstart * p.P; i += blockDim.x) {
      const int ci = i / p.P;
      const int d = i - ci * p.P;
      const int64_t c = c_lo + ci;
      const int gl = static_cast<int>(src0 + c * p.chunk - t0);
      p.rcpm[(static_cast<int64_t>(d) * p.P + s) * p.C + c] =
          excl[d] + prefix_in_tile(bits, p.ncols, d, gl);
    }
  }

  // Padding rows of the expanded layout, spread over the tiles.
  const int n_pad = p.sizes[kSizePad];
  for (int64_t i = static_cast<int64_t>(tile) * kTile + threadIdx.x; i < n_pad;
       i += static_cast<int64_t>(p.num_tiles) * kTile) {
    int lo = 0, hi = p.E;  // find e with pad_off[e] <= i < pad_off[e+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.pad_off[mid] <= i) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int row = exp_off[e] + p.totals[p.P + e] + static_cast<int>(i - p.pad_off[e]);
    p.pad_rows[i] = row;
    p.exp_src[row] = -1;
  }
}

__global__ void ep_prefix_kernel(PlanDev p) {
  const int64_t total = static_cast<int64_t>(p.P) * p.P * p.C;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int c = static_cast<int>(i % p.C);
  const int64_t sd = i / p.C;
  const int d = static_cast<int>(sd % p.P);
  const int s = static_cast<int>(sd / p.P);
  // X at the start of source s2 (s2 == P: the end of the last source).
  auto x_src = [&](int s2) -> int {
    return s2 < p.P ? p.rcpm[(static_cast<int64_t>(d) * p.P + s2) * p.C] : p.totals[d];
  };
  auto channel_live = [&](int c2) { return c2 < p.C && static_cast<int64_t>(c2) * p.chunk < p.S; };
  const int x0 = x_src(s);
  const int x_end = x_src(s + 1);
  const int x_next = channel_live(c + 1) ? p.rcpm[(static_cast<int64_t>(d) * p.P + s) * p.C + c + 1] : x_end;
  p.cpm[i] = x_next - x0;
  if (!channel_live(c)) p.rcpm[(static_cast<int64_t>(d) * p.P + s) * p.C + c] = x_end;
  if (c == 0) {
    p.rpm[static_cast<int64_t>(s) * p.P + d] = x_end;
    p.ntpr[static_cast<int64_t>(s) * p.P + d] = x_end - x0;
  }
}

size_t count_smem_bytes(const PlanDev& p) {
  size_t a = sizeof(uint32_t) * kTileWords * p.ncols + sizeof(int) * kTile * p.K;
  size_t b = sizeof(int) * (2 * (p.E + 1) + (p.P + 1));  // finalize reuse
  return a > b ? a : b;
}

}  // namespace

size_t plan_emit_smem_bytes(int P, int E, int K) {
  const int ncols = P + E;
  return sizeof(uint32_t) * kTileWords * ncols + sizeof(int) * ncols + sizeof(int) * kTile * K +
         sizeof(int) * (P + 1 + E + 1);
}

cudaError_t launch_plan(const PlanDev& p, cudaStream_t stream) {
  const size_t count_smem = count_smem_bytes(p);
  const size_t emit_smem = plan_emit_smem_bytes(p.P, p.E, p.K);
  cudaError_t err;
  if (count_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(ep_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(count_smem));
    if (err != cudaSuccess) return err;
  }
  if (emit_smem > 48 * 1024) {
    err = cudaFuncSetAttribute(ep_emit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(emit_smem));
    if (err != cudaSuccess) return err;
  }
  ep_count_kernel<<<p.num_tiles, kTile, count_smem, stream>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  ep_emit_kernel<<<p.num_tiles, kTile, emit_smem, stream>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const int64_t total = static_cast<int64_t>(p.P) * p.P * p.C;
  const int threads = 256;
  ep_prefix_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ep
