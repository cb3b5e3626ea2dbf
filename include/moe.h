/*
 * moe.h - C ABI of libmoe: the single-GPU hot path of one Mixture-of-Experts layer's expert
 * computation (GB300 / sm_103a), forward and backward.
 *
 * Source of the method: "Scalable Pretraining of Large MoE LMs on Aurora" (arXiv 2604.00785).
 * Its FastSparseMoE module (brief, section 核心方法) counts tokens per expert and generates their
 * indices with GPU kernels, then merges every expert's FFN into one grouped GEMM; the summary page
 * (section 关键设计) adds optimised matmul and activation kernels, and both pages report the module
 * on the forward and backward pass (brief, sections 为什么值得记录 / 关键结果). The pages fix
 * neither the router nor the activation; this library implements softmax top-k routing with
 * renormalised weights (ties to the lower expert id) and SwiGLU experts.
 *
 * Layer, per token t with input x_t [d], router logits L[t, :] [E], grad_out g_t [d]:
 *   S_t      = the k experts with largest L[t,e], ordered by (L desc, e asc)
 *   w_{t,e}  = softmax of L[t, S_t]                       (topk_idx / topk_w, slot j = t*k + j)
 *   out_t    = sum_{e in S_t} w_{t,e} * Wd[e] (silu(Wg[e] x_t) * (Wu[e] x_t))
 *
 * Conventions for every call:
 *   - Returns MOE_OK (0) or a negative moe_status. Argument errors are detected on the host before
 *     anything is enqueued. Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *     never synchronise, except moe_read_status.
 *   - Every pointer named like a tensor is DEVICE memory owned by the caller, contiguous, row-major,
 *     16-byte aligned. The library allocates nothing and keeps no per-call state between calls.
 *   - dtype: MOE_F32 or MOE_BF16 for x, weights, grad_out and every grouped activation buffer.
 *     Logits, routing weights and their gradients are always fp32; indices are int32.
 *   - Calls that can detect an error on the device (a bad expert id, a wait that ran out) write a
 *     status word at the start of their workspace `ws`; read it with moe_read_status(ws, stream).
 *
 * Grouped layout. The permuted ("grouped") buffers hold the routed rows expert by expert. Expert
 * e's rows start at row tile_offsets[e] * MOE_GROUP_ROWS and follow increasing slot index (so
 * increasing token index); the rows after the last token of an expert up to the next multiple of
 * MOE_GROUP_ROWS are padding and are kept at zero. Every grouped buffer has
 * rows_max = moe_grouped_rows_max(T, k, E) rows; rows from tile_offsets[E] * MOE_GROUP_ROWS on are
 * never touched. With this layout every grouped-GEMM tile belongs to one expert and is full: no
 * TMA box straddles two experts, no tile needs row masks, and the weight-gradient GEMMs may sum
 * over an expert's padded rows because the padding is zero. This is why moe_permute and
 * moe_combine_bwd take counts and tile_offsets (they write the padding zeros), why the grouped
 * FFN calls take tile_offsets and rows_max, and why token_of_row has rows_max entries.
 */
#ifndef MOE_LAYER_H_
#define MOE_LAYER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *moe_stream_t;

#define MOE_VERSION 100         /* 1.0.0 */
#define MOE_GROUP_ROWS 128      /* rows per grouped-GEMM tile; each expert's row group is aligned to it */
#define MOE_MAX_EXPERTS 256
#define MOE_MAX_TOPK 16

enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 };

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,     /* null pointer, bad size, misalignment, workspace too small */
  MOE_ERR_UNSUPPORTED = -2,     /* shape or dtype outside what a kernel supports (see each call) */
  MOE_ERR_CUDA = -3,            /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = -4,  /* a bounded device-side wait ran out (device status word) */
  MOE_ERR_BAD_INDEX = -5,       /* an expert id outside [0, E) was seen (device status word) */
  MOE_ERR_CHECK_FAILED = -6     /* a consistency check of the debug build failed (device status word):
                                   see "Debug build" below */
};

/* Debug build. Compiled with -DMOE_CHECKS=1 (mixture_experts_layer_histogram_gb300/build.py:
 * build(checks=True) writes libmoe_checks.so), the grouped-GEMM kernels check on the device that
 * every tile's rows lie inside its expert's row group (offsets and tile_offsets agree: an expert's
 * routed rows fit its padded group) and inside rows_max, that every row a tile stores, zero-fills or
 * reads as a weight-gradient operand lies below rows_max, and that tile_offsets is non-decreasing.
 * A failed check records MOE_ERR_CHECK_FAILED in the workspace status word and the tile is skipped:
 * nothing is written outside the buffers and no kernel traps. The release build compiles the
 * checks out. */

/* ---------------------------------------------------------------------------------------------
 * Routing (brief, section 核心方法: expert selection feeding the token counting step).
 * logits [T, E] fp32 -> topk_idx [T, k] int32 (ordered by logit desc, lower id on ties; -0 == +0),
 *                       topk_w [T, k] fp32 = softmax over the k selected logits.
 * Requires 1 <= E <= MOE_MAX_EXPERTS, 1 <= k <= min(E, MOE_MAX_TOPK), T >= 0. Logits must be
 * finite (non-finite input gives unspecified selections). No workspace, no device status.
 */
int moe_route_topk(const float *logits, int T, int E, int k, int32_t *topk_idx, float *topk_w,
                   moe_stream_t stream);

/* Rows of every grouped buffer: round_up(T*k + E*(MOE_GROUP_ROWS-1), MOE_GROUP_ROWS). */
int64_t moe_grouped_rows_max(int T, int k, int E);

/* ---------------------------------------------------------------------------------------------
 * Token counting and index generation (brief, section 核心方法: "GPU kernels for token counting and
 * index generation"). A stable counting sort of the T*k slots by expert id, in two kernels:
 * a warp-aggregated histogram, then a per-expert decoupled look-back scan over blocks and a
 * stable scatter.
 *   topk_idx     [T*k] int32 in [0, E)
 *   counts       [E]   rows routed to each expert
 *   offsets      [E+1] exclusive scan of counts (offsets[E] = T*k)
 *   tile_offsets [E+1] exclusive scan of ceil(counts[e] / MOE_GROUP_ROWS)
 *   row_of_slot  [T*k] grouped row of slot t*k+j: tile_offsets[e]*MOE_GROUP_ROWS + (number of
 *                      earlier slots routed to the same expert)
 *   token_of_row [rows_max] token of each grouped row, -1 on padding rows
 * ws: moe_count_index_workspace_size(T, k, E) bytes of device memory, any content (the call
 * resets what it needs). Device errors: MOE_ERR_BAD_INDEX (such slots get row_of_slot = -1 and
 * are not counted), MOE_ERR_DEVICE_TIMEOUT (the look-back wait is bounded to about 0.2 s).
 * Fault-injection hook (for tests of the bounded wait): the int32 at byte offset
 * moe_count_index_hook_offset(E) of ws is read on the device by the call. If it holds b + 1
 * (b >= 0), scan block b withholds its published prefix, so its successor's bounded wait runs out
 * and the call reports MOE_ERR_DEVICE_TIMEOUT. The call clears the hook; leave it 0 otherwise.
 */
size_t moe_count_index_workspace_size(int T, int k, int E);
size_t moe_count_index_hook_offset(int E);
int moe_count_index(const int32_t *topk_idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                    int32_t *tile_offsets, int32_t *row_of_slot, int32_t *token_of_row, void *ws,
                    size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Routing, token counting and index generation in one launch (brief, section 核心方法: expert
 * selection feeding the GPU kernels for token counting and index generation): the results of
 * moe_route_topk followed by moe_count_index, bit for bit (topk_idx, topk_w, counts, offsets,
 * tile_offsets, row_of_slot, token_of_row), from one kernel whose blocks route their tokens, rank
 * their slots and publish their per-expert counts; once every block has published (a bounded wait
 * of about 0.2 s), each block scans the totals, sums its predecessors' counts and scatters.
 * Arguments, shapes, workspace size and device errors are those of the two
 * calls (the selection cannot produce an expert id outside [0, E)); the look-back fault hook is not
 * read and is cleared. The blocks wait for one another, so the kernel runs only when all of them
 * fit on the GPU at once (T*k up to about 300K slots on a GB300); above that the call makes the
 * two separate calls itself.
 */
int moe_route_count_index(const float *logits, int T, int E, int k, int32_t *topk_idx, float *topk_w,
                          int32_t *counts, int32_t *offsets, int32_t *tile_offsets, int32_t *row_of_slot,
                          int32_t *token_of_row, void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * moe_count_index without a workspace. The paper has no counterpart: this entry point exists for
 * callers that cannot allocate device memory (for example a plugin inside a host framework that
 * owns all device allocations and passes only input and output buffers, or a service that forbids
 * allocation after start-up). Arguments, outputs and results are those of moe_count_index; the
 * scratch lives in a fixed device array of MOE_STATIC_SCRATCH_BYTES inside the library, present on
 * every GPU that loads the library until the process exits.
 *   - Size limit: calls whose moe_count_index_workspace_size(T, k, E) exceeds
 *     MOE_STATIC_SCRATCH_BYTES return MOE_ERR_UNSUPPORTED (1 MiB covers T*k up to 2,095,104 slots at
 *     E = 64, or up to 523,264 slots at E = 256).
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) and
 *     caches it for the life of the process; make that first call before any stream capture on
 *     that device. The cache does not survive a reset of the device's primary context
 *     (cudaDeviceReset): after one, the library reloads in a new context and the cached address is
 *     stale, so do not call this entry point again in that process.
 *   - Every call on a device shares the one array: calls that overlap on the GPU (different streams
 *     without ordering between them) race and give wrong results. Each call clears what must start
 *     at zero, so consecutive calls are independent.
 *   - Device-detected errors (a bad expert id, a look-back wait that ran out) are not reported to
 *     the caller; slots with a bad id still get row_of_slot = -1. Use moe_count_index with a
 *     workspace where the device status is needed.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define MOE_STATIC_SCRATCH_BYTES (1 << 20)
int moe_count_index_static(const int32_t *topk_idx, int T, int k, int E, int32_t *counts, int32_t *offsets,
                           int32_t *tile_offsets, int32_t *row_of_slot, int32_t *token_of_row,
                           moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Token permutation into the grouped layout (the consumer of the generated indices; brief,
 * section 核心方法). x [T, d] -> x_perm [rows_max, d]: x_perm[row_of_slot[t*k+j]] = x[t]; padding
 * rows of every expert are written with zeros. Each x row is read once and written k times.
 * Requires d*sizeof(dtype) % 16 == 0. Slots whose row is outside [0, rows_max) are skipped.
 */
int moe_permute(const void *x, int dtype, int T, int d, int k, int E, const int32_t *row_of_slot,
                const int32_t *counts, const int32_t *tile_offsets, int64_t rows_max, void *x_perm,
                moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Grouped expert FFN, forward (brief, section 核心方法: "Grouped GEMM merges the experts'
 * computation"; summary page, section 关键设计: optimised matmul and activation).
 *   x_perm    [rows_max, d]   grouped tokens
 *   w_gate_up [E, 2f, d]      rows 0..f-1: gate projection Wg[e]; rows f..2f-1: up projection Wu[e]
 *   w_down    [E, d, f]       Wd[e]
 *   ab        [rows_max, 2f]  saved for backward: columns 0..f-1 a = x Wg^T, f..2f-1 b = x Wu^T;
 *                             may be NULL, and a, b are then not stored: a forward that no
 *                             moe_grouped_ffn_bwd on these activations follows (inference, or a
 *                             layer whose backward recomputes them, moe_grouped_ffn_bwd_recompute)
 *   h         [rows_max, f]   saved: silu(a) * b
 *   y_perm    [rows_max, d]   h Wd^T
 * GEMM1 fuses the SwiGLU gate into its epilogue; GEMM2 is a plain grouped GEMM. bf16: tcgen05
 * tensor cores, fp32 accumulation, outputs rounded to bf16; requires d % 256 == 0 and
 * f % 256 == 0. fp32: SIMT fp32 FMA, any d, f >= 1. tile_offsets and offsets come from
 * moe_count_index: tile_offsets places each expert's rows, offsets gives how many are real (the
 * bf16 kernels compute an expert's rows only up to the next multiple of 32 past its last token and
 * write the rest of its padding as zeros). ws: moe_grouped_ffn_workspace_size(...) bytes (device
 * status word). Padding rows come out as zeros.
 */
size_t moe_grouped_ffn_workspace_size(int E, int d, int f, int64_t rows_max, int dtype, int backward);
int moe_grouped_ffn_fwd(const void *x_perm, const void *w_gate_up, const void *w_down,
                        const int32_t *tile_offsets, const int32_t *offsets, int E, int d, int f, int64_t rows_max,
                        int dtype, void *ab, void *h, void *y_perm, void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Grouped expert FFN, backward (brief, sections 为什么值得记录 / 关键结果: the module is measured
 * on the forward-backward pass). With dy = dy_perm (from moe_combine_bwd):
 *   dab      [rows_max, 2f]  da = dh * b * s(a)(1 + a(1 - s(a))), db = dh * silu(a), dh = dy Wd[e]
 *   dx_perm  [rows_max, d]   dab Wgu[e]
 *   dw_down  [E, d, f]       sum over expert e's rows of dy^T h      (overwritten, not accumulated)
 *   dw_gate_up [E, 2f, d]    sum over expert e's rows of dab^T x_perm (overwritten)
 * Padding rows of dy_perm must be zero (moe_combine_bwd writes them so). Same dtype rules as the
 * forward; gradients are written in the parameter dtype, accumulated in fp32.
 */
int moe_grouped_ffn_bwd(const void *dy_perm, const void *x_perm, const void *ab, const void *h,
                        const void *w_gate_up, const void *w_down, const int32_t *tile_offsets,
                        const int32_t *offsets, int E, int d, int f, int64_t rows_max, int dtype, void *dab,
                        void *dx_perm, void *dw_gate_up, void *dw_down, void *ws, size_t ws_bytes,
                        moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Backward with recomputation (brief, section 核心方法: selective activation checkpointing, which
 * may recompute the SparseMoE module in the backward pass to save memory). Same arguments and
 * results as moe_grouped_ffn_bwd, but `ab` and `h` are outputs here: they are first recomputed
 * from x_perm by the forward's GEMM1 (with its SwiGLU epilogue), then the backward runs on them.
 * The forward may therefore write ab and h into scratch that other layers reuse before this
 * layer's backward; the cost is one more GEMM1 (4 M d f FLOP).
 */
int moe_grouped_ffn_bwd_recompute(const void *dy_perm, const void *x_perm, void *ab, void *h, const void *w_gate_up,
                                  const void *w_down, const int32_t *tile_offsets, const int32_t *offsets, int E,
                                  int d, int f, int64_t rows_max, int dtype, void *dab, void *dx_perm,
                                  void *dw_gate_up, void *dw_down, void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * The grouped FFN with the permutation fused into the GEMMs' token loads (brief, section 核心方法:
 * the generated indices feed the grouped GEMM directly). Same results, bit for bit, as
 * moe_permute followed by the calls above, but x_perm is never formed: the tokens are passed in
 * token order, x [T, d], with token_of_row [rows_max] from moe_count_index (-1 on padding rows,
 * which read as zeros), and GEMM1 (forward and recompute) and the gate/up weight gradient
 * (backward) gather their token rows through it. Every other argument, rule and result is that of
 * the call without _gather. The bf16 kernels copy the rows with cp.async by two loader warps per
 * CTA; entries of token_of_row outside [-1, T) read as padding rows.
 */
int moe_grouped_ffn_fwd_gather(const void *x, const int32_t *token_of_row, int T, const void *w_gate_up,
                               const void *w_down, const int32_t *tile_offsets, const int32_t *offsets, int E, int d,
                               int f, int64_t rows_max, int dtype, void *ab, void *h, void *y_perm, void *ws,
                               size_t ws_bytes, moe_stream_t stream);
int moe_grouped_ffn_bwd_gather(const void *dy_perm, const void *x, const int32_t *token_of_row, int T, const void *ab,
                               const void *h, const void *w_gate_up, const void *w_down, const int32_t *tile_offsets,
                               const int32_t *offsets, int E, int d, int f, int64_t rows_max, int dtype, void *dab,
                               void *dx_perm, void *dw_gate_up, void *dw_down, void *ws, size_t ws_bytes,
                               moe_stream_t stream);
int moe_grouped_ffn_bwd_recompute_gather(const void *dy_perm, const void *x, const int32_t *token_of_row, int T,
                                         void *ab, void *h, const void *w_gate_up, const void *w_down,
                                         const int32_t *tile_offsets, const int32_t *offsets, int E, int d, int f,
                                         int64_t rows_max, int dtype, void *dab, void *dx_perm, void *dw_gate_up,
                                         void *dw_down, void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Weighted un-permute (combine) back to token order:
 *   out[t] = sum_j topk_w[t,j] * y_perm[row_of_slot[t*k+j]]   (fp32 accumulation in slot order)
 * With topk_w == NULL the rows are summed unweighted: the backward of moe_permute
 * (dx[t] = sum_j dx_perm[row_of_slot[t*k+j]]). out [T, d] in dtype. Same size rules as permute.
 */
int moe_combine_fwd(const void *y_perm, const float *topk_w, const int32_t *row_of_slot, int T, int d,
                    int k, int64_t rows_max, int dtype, void *out, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Backward of the combine and of the routing weights, per token t with g = grad_out[t]:
 *   dy_perm[row_of_slot[t*k+j]] = topk_w[t,j] * g                       (dtype; padding rows zeroed)
 *   d_topk_w[t,j]  = <g, y_perm[row_of_slot[t*k+j]]>                     [T, k] fp32
 *   d_logits[t,e]  = w_e (d_topk_w_e - sum_j w_j d_topk_w_j) for e in S_t, else 0    [T, E] fp32
 * (the softmax-over-selected-logits backward; the selection itself is held fixed).
 */
int moe_combine_bwd(const void *grad_out, const void *y_perm, const float *topk_w, const int32_t *topk_idx,
                    const int32_t *row_of_slot, const int32_t *counts, const int32_t *tile_offsets, int T,
                    int d, int k, int E, int64_t rows_max, int dtype, void *dy_perm, float *d_topk_w,
                    float *d_logits, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Router, the step before the selection (summary page, section 关键设计: expert selection). The
 * logits are a linear map of the token, L[t,e] = sum_c x[t,c] w_router[e,c] (fp32 accumulation),
 * followed in the same kernel by the selection and weights of moe_route_topk:
 *   x          [T, d]  dtype
 *   w_router   [E, d]  dtype; row e scores expert e
 *   logits     [T, E]  fp32 output, or NULL when the caller does not need the logits
 *   topk_idx   [T, k]  int32: the k largest logits, ordered by (logit desc, id asc), -0 == +0
 *   topk_w     [T, k]  fp32: softmax over the selected logits. The selection is the one
 *                      moe_route_topk makes on the same fp32 logits; the weights may differ from
 *                      moe_route_topk's in the last bit (here the selected exponentials are summed
 *                      in slot order).
 * bf16: one tcgen05 kernel (TMA-fed tiles of 128 tokens x all E experts, the fp32 accumulator in
 * TMEM, the top-k and softmax in the epilogue, one thread per token); requires d % 8 == 0.
 * fp32: SIMT fp32 FMA, then the moe_route_topk kernel on the logits; any d >= 1.
 * Requires 1 <= E <= MOE_MAX_EXPERTS, 1 <= k <= min(E, MOE_MAX_TOPK), T >= 0, and
 * ws: moe_router_workspace_size(T, d, E, dtype) bytes of device memory, 256-byte aligned, any
 * content (device status word; scratch of the fp32 path and of the backward). Device errors:
 * MOE_ERR_DEVICE_TIMEOUT (every pipeline wait of the bf16 kernels is bounded to about 0.2 s).
 */
size_t moe_router_workspace_size(int T, int d, int E, int dtype);
int moe_router_fwd(const void *x, const void *w_router, int T, int d, int E, int k, int dtype, float *logits,
                   int32_t *topk_idx, float *topk_w, void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Router backward, for d_logits [T, E] fp32 (from moe_combine_bwd):
 *   dx         [T, d]  dtype   accumulate_dx = 0:  dx  = d_logits w_router
 *                              accumulate_dx = 1:  dx += d_logits w_router  (adds the router's
 *                              share to the experts' dx; read and written in place)
 *   dw_router  [E, d]  dtype   d_logits^T x  (overwritten, not accumulated)
 * bf16: d_logits is rounded to bf16 once (the tensor-core operand); both products run on tcgen05
 * with fp32 accumulation; dw_router is the sum, in a fixed order, of fp32 partial products over
 * token ranges (deterministic). fp32: SIMT fp32 FMA. Same shape rules and workspace as the
 * forward (the same ws may serve both calls when they are ordered on one stream).
 */
int moe_router_bwd(const void *x, const void *w_router, const float *d_logits, int T, int d, int E, int dtype,
                   int accumulate_dx, void *dx, void *dw_router, void *ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------------------------
 * Synchronises `stream`, then returns the device status word at the start of a workspace used by
 * moe_count_index, moe_grouped_ffn_* or moe_router_*: MOE_OK or a negative moe_status. Not for
 * the hot path.
 */
int moe_read_status(const void *ws, moe_stream_t stream);
const char *moe_status_string(int status);
int moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_LAYER_H_ */
