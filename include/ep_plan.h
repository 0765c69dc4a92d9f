/*
 * ep_plan.h — C ABI of the GB300 (sm_103a) MoE expert-parallel routing plan,
 * dispatch row scatter and weighted combine.
 *
 * One GPU holds all P logical ranks.  Source rank s owns the global tokens
 * g = s*S + t (t < S); expert e lives on rank e / (E/P).  Every "transfer" of
 * the method is an HBM-to-HBM copy inside one device allocation.
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are device pointers; *_host are host pointers.
 *     The caller owns every input and output buffer it passes.  A handle owns
 *     the plan arrays it allocates (one device allocation, stream-ordered).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on that stream unless the comment says "synchronises".
 *   - Host-checkable argument errors return EP_ERR_INVALID (or
 *     EP_ERR_MISMATCH / EP_ERR_CAPACITY) before anything is enqueued.
 *     Errors that only the device can see (an expert id out of range, a
 *     duplicate expert in one token row, an output row beyond the caller's
 *     capacity, a bounded wait that gave up) are recorded in the handle's
 *     device status word; no out-of-range row is ever written.  They are
 *     returned by the next synchronising call (ep_plan_sizes, ep_sync_status).
 *   - A plan whose bounded wait gave up (EP_ERR_TIMEOUT) leaves the handle's
 *     plan arrays unfinished.  Until ep_sync_status reads and clears that
 *     status, later plans on the handle do no work (they could otherwise
 *     pass a grid barrier on the timed-out plan's arrivals), and dispatch,
 *     combine and backward calls on the handle keep every access inside the
 *     caller's buffers and the handle's arrays but produce unspecified rows.
 *     ep_plan_sizes and ep_pending_wait report the status without clearing it.
 *   - A handle is not thread-safe; calls that use one handle on different
 *     streams must be ordered by the caller.
 *   - ep_replan, ep_dispatch, ep_dispatch_cached, ep_dispatch_metadata,
 *     ep_combine and the backward calls may be captured in a CUDA graph and
 *     replayed (the plan's grid barriers leave a zeroed count for the next
 *     launch); the asynchronous calls and ep_plan_sizes may not.
 *     Profile records of captured launches land at the capture-time
 *     positions on every replay.
 *
 * Sources are cited by page title and section:
 *   [DO] "Ascend DeepEP MoE Dispatch Optimization"
 *   [TT] TileLang tutorial, chapter 38 "DeepEP-Ascend"
 */
#ifndef EP_PLAN_GB300_H
#define EP_PLAN_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *ep_stream_t;

typedef struct ep_handle_s *ep_handle_t;

/* Same underlying type as cudaEvent_t. */
struct CUevent_st;
typedef struct CUevent_st *ep_event_t;

/* An issued asynchronous dispatch or combine (see ep_dispatch_async). */
typedef struct ep_pending_s *ep_pending_t;

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID = 1,  /* bad argument, or routing data the method rejects */
    EP_ERR_CAPACITY = 2, /* an output buffer is smaller than the exact need */
    EP_ERR_TIMEOUT = 3,  /* a bounded device wait gave up; results are invalid */
    EP_ERR_CUDA = 4,     /* a CUDA runtime call or kernel launch failed */
    EP_ERR_MISMATCH = 5, /* cached handle used with different shape parameters */
    EP_ERR_OOM = 6       /* device or host allocation failed */
} ep_status_t;

typedef enum {
    EP_DTYPE_BF16 = 0,     /* bfloat16, 2 bytes */
    EP_DTYPE_FP8_E4M3 = 1  /* OCP E4M3 ("fn"), 1 byte, with fp32 scales per 128 */
} ep_dtype_t;

/* Flags of the dispatch entry points. */
#define EP_DISPATCH_ZERO_PAD 1          /* zero the padding rows (codes and scales) */
#define EP_DISPATCH_SCALES_COL_MAJOR 2  /* FP8 scales stored [H/128][capacity_rows] */

/* Limits of this implementation (checked; EP_ERR_INVALID beyond them). */
#define EP_MAX_RANKS 1024
#define EP_MAX_EXPERTS 2048
#define EP_MAX_TOPK 16
#define EP_DEFAULT_CHANNELS 16

/* Plan arrays readable through ep_handle_get.  Shapes use T = P*S. */
typedef enum {
    EP_FIELD_IS_TOKEN_IN_RANK = 0,  /* [T,P]   uint8: 1 if some expert of g lives on d */
    EP_FIELD_SEND_HEAD = 1,         /* [T,P]   int32: row of g in d's compact window, -1 if not sent */
    EP_FIELD_NUM_TOKENS_PER_RANK = 2,   /* [P,P] int32 [s][d]: tokens of s sent to d (dedup) */
    EP_FIELD_NUM_TOKENS_PER_EXPERT = 3, /* [P,E] int32 [s][e]: (token,slot) pairs of s picking e */
    EP_FIELD_EXPERT_COUNTS = 4,     /* [E]     int32: n_e, all sources */
    EP_FIELD_NUM_RECV = 5,          /* [P]     int32: distinct tokens received by d */
    EP_FIELD_RANK_PREFIX = 6,       /* [P,P]   int32 [s][d]: inclusive sum over sources <= s */
    EP_FIELD_CHANNEL_PREFIX = 7,    /* [P,P,C] int32 [s][d][c]: inclusive sum over channels <= c */
    EP_FIELD_RECV_CHANNEL_PREFIX = 8, /* [P,P,C] int32 [d][s][c]: start of segment (s,c) in d's window */
    EP_FIELD_RECV_OFFSETS = 9,      /* [P+1]   int32: start of d's window in RECV_SRC_IDX */
    EP_FIELD_RECV_SRC_IDX = 10,     /* [N_recv] int32: source-local token t of each window row */
    EP_FIELD_EXPERT_OFFSETS = 11,   /* [E+1]   int32: padded start of expert e's rows */
    EP_FIELD_SLOT = 12,             /* [T,K]   int32: expanded row of (g,k), -1 for an unused slot */
    EP_FIELD_EXP_SRC = 13,          /* [N_exp] int32: source token g of each expanded row, -1 on padding */
    EP_FIELD_PAD_ROWS = 14,         /* [N_pad] int32: the padding rows of the expanded layout */
    EP_FIELD_COUNT = 15
} ep_field_t;

/* Version of this ABI (bumped on any incompatible change). */
int ep_abi_version(void);

/* Human-readable name of a status code (static storage). */
const char *ep_status_string(ep_status_t status);

/*
 * ep_plan — build the routing plan of one MoE layer.
 *
 * Defines: the six-tensor dispatch handle ([DO] "从 Python 接口进入真实调用链",
 * the handle table: rank_prefix_matrix, channel_prefix_matrix,
 * recv_channel_prefix_matrix, recv_src_idx, is_token_in_rank, send_head);
 * the counts and prefixes the notify stage produces ([DO] "Notify 先交换数量和
 * 前缀"); per-destination dedup ([TT] §1.3); the expanded layout padded to
 * expert_alignment ([TT] §2.2) in the deterministic order of [TT] §3.5.
 *
 * topk_idx_dev        [T,K] int64, row-major, 8-byte aligned.  Entry -1 marks
 *                     an unused slot; other entries must be distinct experts
 *                     in [0,E) (device-checked, EP_ERR_INVALID on sync).
 *                     Read by the plan's kernel on `stream`: keep it unchanged
 *                     until the stream has passed the plan.  The handle keeps
 *                     no reference to it (later calls use the plan arrays).
 * num_tokens_per_rank S >= 1; T = P*S.
 * num_ranks           P, 1..EP_MAX_RANKS, E % P == 0.
 * num_topk            K, 1..min(E, EP_MAX_TOPK).
 * num_experts         E, 1..EP_MAX_EXPERTS.
 * expert_alignment    A >= 1: each expert segment is padded to a multiple of A.
 * num_channels        C in 1..S, or 0 for min(EP_DEFAULT_CHANNELS, S).  Channel c
 *                     of a source covers tokens [c*ceil(S/C), min(S,(c+1)*ceil(S/C))).
 * out_handle_host     receives the new handle (NULL on error).
 * The expanded-row count N_exp must fit int32 (checked on the worst case).
 */
ep_status_t ep_plan(const int64_t *topk_idx_dev, int64_t num_tokens_per_rank,
                    int num_ranks, int num_topk, int num_experts,
                    int expert_alignment, int num_channels, ep_stream_t stream,
                    ep_handle_t *out_handle_host);

/*
 * ep_replan — rebuild the plan of an existing handle for new routing with the
 * same shape (S, P, K, E, A, C), reusing its device memory: a fresh plan with
 * no allocation.  Same inputs and checks as ep_plan.
 */
ep_status_t ep_replan(ep_handle_t handle, const int64_t *topk_idx_dev, ep_stream_t stream);

/*
 * ep_plan_sizes — synchronises `stream`, then returns the exact expanded-row
 * count N_exp (sum over e of ceil(n_e/A)*A) and compact receive-row count
 * N_recv (sum over d of num_recv[d]); the do_cpu_sync path of the pages
 * ([DO] "输出长度有动态和固定两种模式").  Returns the device status too.
 * Either output pointer may be NULL.
 */
ep_status_t ep_plan_sizes(ep_handle_t handle, ep_stream_t stream,
                          int64_t *num_expanded_host, int64_t *num_recv_host);

/*
 * ep_worst_expanded_rows — an upper bound of N_exp without any device read:
 * T*K + E*(A-1), the fixed-output-length (num_worst_tokens) path of the pages
 * ([DO] "输出长度有动态和固定两种模式").  Returns -1 on invalid arguments.
 */
int64_t ep_worst_expanded_rows(int64_t num_tokens, int num_topk, int num_experts,
                               int expert_alignment);

/*
 * ep_dispatch — the row scatter: each token's hidden row is read once and
 * written to every expanded row of its (token, slot) pairs, which groups rows
 * by expert and pads each segment to A rows ([TT] §2.2, §4.3 local copy).
 *
 * x_dev          [T,H], 16-byte aligned, H % 8 == 0: bfloat16 (x_dtype
 *                EP_DTYPE_BF16), or E4M3 codes already quantised with fp32
 *                scales per 128 elements (x_dtype EP_DTYPE_FP8_E4M3, [TT]
 *                §3.6: x arrives as (codes, scales)).
 * x_scales_dev   [T,H/128] fp32 row-major scales of pre-quantised input;
 *                NULL for bfloat16 input.
 * hidden         H.
 * out_dtype      EP_DTYPE_BF16 (bfloat16 input only): recv_x is
 *                [capacity_rows,H] bfloat16, a bit copy.
 *                EP_DTYPE_FP8_E4M3: recv_x is [capacity_rows,H] E4M3 codes and
 *                recv_scales_dev holds H/128 fp32 scales per row.  From
 *                bfloat16 input the rows are quantised inside dispatch ([TT]
 *                §3.6): per row and per 128 elements, scale = amax/448 (IEEE
 *                fp32 division), code = E4M3(x/scale) rounded to nearest even
 *                with saturation; amax == 0 gives scale 0 and zero codes.  From
 *                pre-quantised input codes and scales are copied.  Needs
 *                H % 128 == 0.
 * flags          EP_DISPATCH_ZERO_PAD: padding rows are zero (codes and
 *                scales), otherwise untouched ([TT] §2.2, do_zero_padding).
 *                EP_DISPATCH_SCALES_COL_MAJOR: scale j of row r is stored at
 *                recv_scales[j*capacity_rows + r] (the column-major layout of
 *                [TT] §3.6, stride (1, rows) for a [rows, H/128] view) instead
 *                of recv_scales[r*(H/128) + j].
 * recv_x_dev     output, 16-byte aligned.  Rows >= N_exp are never written.
 * recv_scales_dev output for FP8; must be NULL for BF16 output.
 * capacity_rows  rows available in recv_x (and recv_scales).  A capacity below
 *                N_exp records EP_ERR_CAPACITY and writes no row at or beyond it.
 * Reusing a handle on new x is the cached dispatch of [TT] §2.4: no plan work.
 */
ep_status_t ep_dispatch(ep_handle_t handle, const void *x_dev, ep_dtype_t x_dtype,
                        const float *x_scales_dev, int64_t hidden, ep_dtype_t out_dtype, int flags,
                        void *recv_x_dev, float *recv_scales_dev, int64_t capacity_rows,
                        ep_stream_t stream);

/*
 * ep_dispatch_cached — ep_dispatch on an existing handle after checking that
 * (num_experts, expert_alignment, num_tokens_per_rank) are the ones the
 * handle was planned with, as the cached-handle path of [TT] §2.4 asserts.
 * A difference returns EP_ERR_MISMATCH and enqueues nothing.
 */
ep_status_t ep_dispatch_cached(ep_handle_t handle, int num_experts, int expert_alignment,
                               int64_t num_tokens_per_rank, const void *x_dev, ep_dtype_t x_dtype,
                               const float *x_scales_dev, int64_t hidden, ep_dtype_t out_dtype,
                               int flags, void *recv_x_dev, float *recv_scales_dev,
                               int64_t capacity_rows, ep_stream_t stream);

/*
 * ep_dispatch_fresh — ep_plan followed by ep_dispatch in one call (a fresh
 * dispatch that re-plans the routing, [DO] "Fresh dispatch 是什么意思").  On
 * success *out_handle_host holds the new plan for later cached dispatches and
 * combines.  Arguments as for ep_plan and ep_dispatch; invalid dispatch
 * arguments are rejected before the plan is enqueued.
 */
ep_status_t ep_dispatch_fresh(const int64_t *topk_idx_dev, int64_t num_tokens_per_rank,
                              int num_ranks, int num_topk, int num_experts,
                              int expert_alignment, int num_channels, const void *x_dev,
                              ep_dtype_t x_dtype, const float *x_scales_dev, int64_t hidden,
                              ep_dtype_t out_dtype, int flags, void *recv_x_dev,
                              float *recv_scales_dev, int64_t capacity_rows, ep_stream_t stream,
                              ep_handle_t *out_handle_host);

/*
 * ep_dispatch_metadata — the metadata that travels with each dispatched row
 * ([TT] §2.1 and §4.2: the routing weight and the source token): for every
 * expanded row r = slot[g,k], recv_weights[r] = topk_weights[g,k] and
 * recv_meta[r] = {g, k}.  With zero_pad, padding rows get weight 0 and
 * {-1, -1}; otherwise they are untouched.
 * topk_weights_dev [T,K] float32; recv_weights_dev [capacity_rows] float32;
 * recv_meta_dev [capacity_rows,2] int32.  A row at or beyond capacity_rows
 * records EP_ERR_CAPACITY and is not written.
 */
ep_status_t ep_dispatch_metadata(ep_handle_t handle, const float *topk_weights_dev,
                                 float *recv_weights_dev, int32_t *recv_meta_dev,
                                 int64_t capacity_rows, int zero_pad, ep_stream_t stream);

/*
 * ep_combine — the inverse of dispatch ([TT] §2.3): gather each token's
 * expert outputs back to token order and reduce them with the top-k weights.
 * out[g,:] = bf16_RNE( sum over k = 0..K-1 with slot[g,k] >= 0, in that
 * order, of fmaf(w[g,k], float(y[slot[g,k],:]), acc) ), acc starting at 0;
 * fp32 accumulation, rounded once ([TT] §4.5).  A token with no valid slot
 * gives zeros.  Padding rows of y are never read.  With a bias row (the
 * fused residual or shared-expert output of [TT] §3.3) the sum is
 * acc + float(bias[g,:]) before the rounding.
 *
 * y_dev          [y_rows,H] bfloat16 expert outputs in the expanded layout,
 *                16-byte aligned, H % 8 == 0.  y_rows < N_exp records
 *                EP_ERR_CAPACITY (rows beyond y_rows are not read).
 * topk_weights_dev [T,K] float32.
 * bias_dev       [T,H] bfloat16, 16-byte aligned, or NULL.
 * out_dev        [T,H] bfloat16, 16-byte aligned.
 */
ep_status_t ep_combine(ep_handle_t handle, const void *y_dev, int64_t y_rows,
                       const float *topk_weights_dev, const void *bias_dev, int64_t hidden,
                       void *out_dev, ep_stream_t stream);

/*
 * ep_dispatch_backward — the backward of dispatch, which is a combine on the
 * same handle ([TT] §2.3): every forward row recv[slot[g,k]] is a copy of
 * x[g], so grad_x[g] = bf16_RNE( sum over k = 0..K-1 with slot[g,k] >= 0, in
 * that order, of float(grad_recv[slot[g,k]]) ), accumulated in fp32.
 *
 * grad_recv_dev  [grad_rows,H] bfloat16 gradient of the expanded rows, 16-byte
 *                aligned, H % 8 == 0; padding rows are never read; a slot at or
 *                beyond grad_rows records EP_ERR_CAPACITY and is skipped.
 * grad_x_dev     [T,H] bfloat16 output, 16-byte aligned.
 */
ep_status_t ep_dispatch_backward(ep_handle_t handle, const void *grad_recv_dev, int64_t grad_rows,
                                 int64_t hidden, void *grad_x_dev, ep_stream_t stream);

/*
 * ep_combine_backward — the backward of combine, which is a dispatch on the
 * same handle ([TT] §2.3).  With out[g] = sum_k w[g,k] * y[slot[g,k]]:
 *   grad_y[slot[g,k]] = bf16_RNE(w[g,k] * float(grad_out[g]))  (fp32 product),
 *   grad_w[g,k]       = <grad_out[g], y[slot[g,k]]>, fp32, summed in a fixed
 *                       order (deterministic; 0 for an unused slot).
 * grad_out_dev   [T,H] bfloat16, 16-byte aligned, H % 8 == 0.
 * y_dev          [y_rows,H] bfloat16 forward expert outputs, 16-byte aligned.
 * topk_weights_dev [T,K] float32.
 * zero_pad       nonzero: padding rows of grad_y are zeroed; 0: untouched.
 * grad_y_dev     [grad_y_rows,H] bfloat16 output, 16-byte aligned.
 * grad_weights_dev [T,K] float32 output.
 * A slot at or beyond y_rows or grad_y_rows records EP_ERR_CAPACITY and is
 * skipped.
 */
ep_status_t ep_combine_backward(ep_handle_t handle, const void *grad_out_dev, const void *y_dev,
                                int64_t y_rows, const float *topk_weights_dev, int64_t hidden,
                                int zero_pad, void *grad_y_dev, int64_t grad_y_rows,
                                float *grad_weights_dev, ep_stream_t stream);

/*
 * ep_sync_status — synchronises `stream`, returns the first error recorded in
 * the handle's device status word (EP_OK if none) and clears it; after
 * EP_ERR_TIMEOUT it also resets the plan's grid-barrier words, so that the
 * next plan runs normally.
 */
ep_status_t ep_sync_status(ep_handle_t handle, ep_stream_t stream);

/*
 * ep_handle_get — device pointer and shape of one plan array (see ep_field_t).
 * The pointer stays valid until the handle is destroyed or re-planned; the
 * arrays are written by kernels on the plan's stream.  shape_host receives up
 * to 3 extents (unused ones are 1) and *ndim_host the rank of the array; for
 * RECV_SRC_IDX, EXP_SRC and PAD_ROWS the extent is the allocated capacity and
 * the valid prefix is given by ep_plan_sizes / expert and pad counts.
 */
ep_status_t ep_handle_get(ep_handle_t handle, ep_field_t field, const void **dev_ptr_host,
                          int64_t shape_host[3], int *ndim_host);

/*
 * ep_handle_info — the plan's shape: S, P, K, E, A, C (any pointer may be NULL).
 */
ep_status_t ep_handle_info(ep_handle_t handle, int64_t *num_tokens_per_rank, int *num_ranks,
                           int *num_topk, int *num_experts, int *expert_alignment,
                           int *num_channels);

/*
 * ep_handle_destroy — release the handle.  Its device memory is freed in
 * stream order on `stream` (after work already enqueued there).  If the
 * handle issued asynchronous calls, this synchronises its communication
 * stream first.  EP_ERR_INVALID, and nothing released, while a pending
 * object of the handle has not been waited on.
 */
ep_status_t ep_handle_destroy(ep_handle_t handle, ep_stream_t stream);

/*
 * ep_plan_static_scratch — the routing plan without any device allocation.
 * The source pages have no counterpart: this entry exists for callers that
 * cannot allocate device memory when they plan, such as a serving runtime
 * that hands all device memory to its own arena at start-up, or a
 * latency-critical loop where an allocation may block on the device or fail
 * under fragmentation.  It computes exactly what ep_plan computes, with the
 * same kernels, but writes every plan array into buffers the caller owns
 * (ep_plan_buffers_t) and keeps its scratch (per-tile counts and prefixes, counters,
 * column totals) in one fixed array in the library's device memory,
 * EP_STATIC_SCRATCH_BYTES large, which every GPU that loads the library holds
 * until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine; it enqueues memsets, the plan kernels and small
 * device-to-device copies on `stream`.
 *
 * - The first call on a device looks up the scratch array's device address
 *   (cudaGetSymbolAddress, with that device current).  Under CUDA's lazy
 *   module loading (the default) that lookup is also where the library's
 *   device code, and with it the scratch array, is loaded onto the device:
 *   "allocates nothing" holds from the first successful call on.  Make that
 *   first call before any stream capture.  A failed lookup is not kept: the
 *   next call tries again.
 * - All calls on a device share the one scratch array, and it keeps the last
 *   call's contents; each call clears what it needs.  Calls whose work
 *   overlaps on the GPU (other streams, other threads) race on the scratch:
 *   order them.
 * - Scratch need: about 0.28*T*(P+E) + 4*(17P+18E) + 2 KB bytes (per-tile
 *   counts and prefixes, tile bit matrices and their word prefixes, column
 *   totals and their copies); a plan that
 *   would need more than EP_STATIC_SCRATCH_BYTES returns EP_ERR_CAPACITY
 *   before anything is enqueued (16384 tokens with P+E = 384 need about
 *   1.8 MB; 65536 tokens fit with P+E up to about 220).
 * - Arguments and shape limits are those of ep_plan; out and all its pointers
 *   must be non-NULL device pointers, 4-byte aligned except the uint8 array.
 *   out->info receives {N_recv, N_exp, N_pad, device status bits}; status
 *   bit 1 = expert id out of range, 2 = duplicate expert in a row, 4 = an
 *   index beyond the buffers' sizes (not written; only after a failed wait),
 *   8 = a bounded wait gave up (the plan is then invalid).
 */
#define EP_STATIC_SCRATCH_BYTES (4u << 20)

typedef struct {
    uint8_t *is_token_in_rank;      /* [T,P] */
    int32_t *send_head;             /* [T,P] */
    int32_t *num_tokens_per_rank;   /* [P,P] */
    int32_t *num_tokens_per_expert; /* [P,E] */
    int32_t *expert_counts;         /* [E] */
    int32_t *num_recv;              /* [P] */
    int32_t *rank_prefix;           /* [P,P] */
    int32_t *channel_prefix;        /* [P,P,C] */
    int32_t *recv_channel_prefix;   /* [P,P,C] */
    int32_t *recv_offsets;          /* [P+1] */
    int32_t *recv_src_idx;          /* [T*min(K,P)] (valid prefix N_recv) */
    int32_t *expert_offsets;        /* [E+1] */
    int32_t *slot;                  /* [T,K] */
    int32_t *exp_src;               /* [T*K + E*(A-1)] (valid prefix N_exp) */
    int32_t *pad_rows;              /* [max(1, E*(A-1))] (valid prefix N_pad) */
    int32_t *info;                  /* [4]: N_recv, N_exp, N_pad, status bits */
} ep_plan_buffers_t;

ep_status_t ep_plan_static_scratch(const int64_t *topk_idx_dev, int64_t num_tokens_per_rank,
                                   int num_ranks, int num_topk, int num_experts,
                                   int expert_alignment, int num_channels,
                                   const ep_plan_buffers_t *out_dev_buffers, ep_stream_t stream);

/*
 * ep_set_num_sms — SM budget of the handle's kernels ([TT] §3.3: num_sms,
 * which cached dispatch and combine take from the handle).  num_sms = 0 (the
 * default) or at least the device's SM count: every launch may use the whole
 * device.  Otherwise the plan, dispatch, combine and backward launches made
 * with this handle use grids of at most num_sms SMs' worth of resident CTAs,
 * which loop over the work, so that other kernels running at the same time
 * (an overlapped shared expert) keep the remaining SMs.  Results do not
 * depend on the budget.  EP_ERR_INVALID for num_sms < 0.
 */
ep_status_t ep_set_num_sms(ep_handle_t handle, int num_sms);

/*
 * ep_dispatch_async / ep_combine_async / ep_pending_wait — issue now, finish
 * later ([TT] §3.4 defer_epilogue + async_with_compute_stream, §4.4 why the
 * dispatch epilogue can be deferred).
 *
 * The work is enqueued on the handle's communication stream (a non-blocking
 * stream the handle creates on first use, on the handle's device, which must
 * be current) and the call returns a pending object.  That stream first
 * waits for `previous` (an event the caller recorded on its compute stream
 * once the inputs were ready), or, with previous = NULL, for all work
 * enqueued on compute_stream before the call.  Meanwhile the compute stream
 * is free for independent work; ep_set_num_sms leaves it SMs to run on.
 *
 * Dispatch: topk_idx_dev non-NULL re-plans the handle first (ep_replan on the
 * communication stream: a fresh dispatch); NULL dispatches with the
 * handle's current plan (a cached dispatch).  The other arguments are those
 * of ep_dispatch.  On one device the rows land in recv_x_dev during the
 * issue; what the method's epilogue adds is the exact receive counts the
 * caller sizes its tensors by.  The device copies the counts (and the status
 * word) to pinned host memory right after the plan, before the row scatter.
 *   defer_epilogue = 0: the call waits on the host for those counts (the plan
 *                       only; the scatter keeps running) before it returns.
 *   defer_epilogue = 1: the call returns at once; the counts are read when
 *                       ep_pending_wait asks for them.
 * At most 8 dispatches of one handle may be pending: the 9th returns
 * EP_ERR_CAPACITY before enqueuing anything.
 *
 * Combine: the arguments are those of ep_combine.  A combine has no host-side
 * epilogue: both values of defer_epilogue return at once.
 *
 * ep_pending_wait — makes compute_stream wait (on the device, no host
 * block) for all the issued work, then frees the pending object; results are
 * usable in compute-stream order afterwards.  num_expanded_host /
 * num_recv_host (may be NULL) receive N_exp and N_recv of a dispatch (0 for a
 * combine); asking for them makes a deferred dispatch wait on the host for
 * the plan.  Returns the status the device recorded up to the plan (an
 * invalid expert id, a grid-barrier timeout) when the counts were read, else
 * EP_OK; later device errors (a capacity overflow in the scatter) are
 * returned by the next ep_sync_status.  Every pending object must be waited
 * on exactly once, before its handle is destroyed, and the buffers it uses
 * must stay allocated until then.
 */
ep_status_t ep_dispatch_async(ep_handle_t handle, const int64_t *topk_idx_dev, const void *x_dev,
                              ep_dtype_t x_dtype, const float *x_scales_dev, int64_t hidden,
                              ep_dtype_t out_dtype, int flags, void *recv_x_dev,
                              float *recv_scales_dev, int64_t capacity_rows,
                              ep_stream_t compute_stream, ep_event_t previous,
                              int defer_epilogue, ep_pending_t *pending_host);

ep_status_t ep_combine_async(ep_handle_t handle, const void *y_dev, int64_t y_rows,
                             const float *topk_weights_dev, const void *bias_dev, int64_t hidden,
                             void *out_dev, ep_stream_t compute_stream, ep_event_t previous,
                             int defer_epilogue, ep_pending_t *pending_host);

ep_status_t ep_pending_wait(ep_pending_t pending, int64_t *num_expanded_host,
                            int64_t *num_recv_host);

/*
 * ep_profile_begin / ep_profile_end — per-CTA profile records ([DO] "Device
 * 侧计时": stage times and bytes per core, each core writing its own slot,
 * no atomics, read by the host once).  The records come from separate
 * instantiations of the kernels that the library launches only while
 * profiling is on, so the default kernels carry no profiling code.
 *
 * Between begin and end, every plan, dispatch, combine and dispatch-backward
 * launch of this handle writes one record per CTA into records_dev (device,
 * 8-byte aligned, capacity_records records of 8 uint64 each), in launch order;
 * records that do not fit are dropped.  Outputs are identical to unprofiled
 * launches.  The combine backward writes none.  Record layout:
 *   [0] kernel << 56 | launch sequence (24 bits) << 32 | CTA index; kernel
 *       1 plan, 2 BF16 dispatch, 3 FP8 dispatch (quantising), 4 dispatch of
 *       pre-quantised FP8, 5 combine, 6 dispatch backward
 *   [1] start, [5] end: device global timer, ns
 *   [2] [3] [4] stage marks (plan: route scan of the CTA's last tile done,
 *       first grid barrier passed, second grid barrier passed; a plan of at
 *       most 256 tokens runs as one CTA without grid barriers and marks the
 *       route scan, the column counts and the offsets instead; 0 for the
 *       other kernels)
 *   [6] work units: plan, tokens scanned; others, (row, column chunk) items
 *   [7] payload bytes read and written by the CTA (hidden rows, codes, scales,
 *       bias; 0 for the plan)
 * ep_profile_end stops recording and returns how many records were written
 * and dropped (either pointer may be NULL); read the records after
 * synchronising the streams the launches ran on.
 */
ep_status_t ep_profile_begin(ep_handle_t handle, uint64_t *records_dev, int64_t capacity_records);
ep_status_t ep_profile_end(ep_handle_t handle, int64_t *records_written_host,
                           int64_t *records_dropped_host);

/*
 * ep_debug_set_plan_wait — test hook for the bounded waits of the plan's two
 * grid barriers.  poll_limit > 0 sets how many times a CTA polls the
 * barrier before it gives up and records EP_ERR_TIMEOUT (0 restores the
 * default); suppress_tile >= 0 makes the CTA of that tile return before the
 * first barrier, so that the others' wait runs out (-1 disables).
 * Process-wide; affects plans enqueued afterwards.
 */
void ep_debug_set_plan_wait(int64_t poll_limit, int suppress_tile);

#ifdef __cplusplus
}
#endif

#endif /* EP_PLAN_GB300_H */
