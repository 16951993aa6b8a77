/*
 * colibri_moe.h -- C ABI of a GB300 (sm_103a) Mixture-of-Experts layer forward.
 *
 * One call of colibri_moe_forward runs, on the caller's CUDA stream:
 *   1. router: logits L = x W_r^T (+ b_r), top-k experts per token (k = 1..4), gates
 *      (zskr.cn/news/2272131 "Colibri: a lightweight C MoE inference engine for
 *      edge devices" 3.2; hnwysp.cn/news/30485 3.1);
 *   2. dispatch: per-expert counts, offsets, tokens gathered into
 *      expert-contiguous rows (zskr.cn 2.1 "Dispatch", 3.2 "expert_counts");
 *   3. expert FFN as grouped GEMMs with the activation fused
 *      (zskr.cn 2.1 "Compute: grouped GEMM"; m.nxbn.cn/news/48047 2.1, 3.1);
 *   4. gate-weighted combine in fp32 (m.nxbn.cn 3.3 "output aggregation";
 *      hnwysp.cn 2.2).
 *
 * Math of the layer (all row-major, nn.Linear [out, in] weight layout):
 *   L[t,e]   = sum_j x[t,j] W_r[e,j] (+ b_r[e])
 *   e_1..e_k = the k experts ranked first by (L descending, expert index ascending)
 *   gates    = softmax of L over e_1..e_k (default; k = 2: g_1 = 1/(1+exp(L_e2 - L_e1)), g_2 = 1 - g_1),
 *              or the softmax over all E experts evaluated at e_1..e_k (COLIBRI_GATE_SOFTMAX_ALL)
 *   SwiGLU:  y_e(x) = W2_e (silu(W1_e x) * (W3_e x))      W1 = W_gate, W3 = W_up, W2 = W_down
 *   ReLU:    y_e(x) = W2_e max(W1_e x + b1_e, 0) + b2_e
 *   out[t]   = sum_j g_j y_{e_j}(x_t) (+ y_shared(x_t))   (fp32 sum in slot order; no residual add)
 * (the two gate modes: news.rkmt.cn/news/2271114 5.2 "linear top-2" (Mixtral) vs "softmax top-2"
 * (DeepSeek), the latter being the weights hnwysp.cn 3.1's code returns; top_k: hnwysp.cn 3.1;
 * shared expert: news.rkmt.cn 5.2, Qwen2-MoE's always-on expert.)
 *
 * Conventions (m.nxbn.cn 3.3 and 5.1: int status codes, 0 = success;
 * zskr.cn 5.3: one context per thread; hnwysp.cn 2.1: no allocation on the
 * forward path; m.nxbn.cn 3.1: maximum batch fixed at initialisation):
 *   - Every function returns 0 or a negative COLIBRI_ERR_* code; none aborts.
 *   - A context owns all device memory it allocates; the caller owns x, out,
 *     the stream and any buffer it passes in.
 *   - A context is not thread-safe: use one per host thread.
 *   - `stream` arguments are cudaStream_t values passed as void* (NULL = the
 *     legacy default stream).  Kernel faults are asynchronous and surface at
 *     the caller's next synchronisation.
 */
#ifndef COLIBRI_MOE_H
#define COLIBRI_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define COLIBRI_API __attribute__((visibility("default")))
#else
#define COLIBRI_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (m.nxbn.cn 5.1: -1 size exceeded, -2 out of memory, -3 corrupt weights) ---- */
#define COLIBRI_OK 0
#define COLIBRI_ERR_INVALID_ARG (-1)  /* NULL pointer, T < 0 or T > max_tokens, host pointer where a
                                         device pointer is required, aliasing x/out, top_k outside
                                         1..4 or above num_experts, num_experts outside 2..16, bad
                                         enum value */
#define COLIBRI_ERR_OOM (-2)          /* a device allocation failed */
#define COLIBRI_ERR_BAD_WEIGHTS (-3)  /* a required weight or bias pointer is NULL, or one is given
                                         that the activation does not use */
#define COLIBRI_ERR_CUDA (-4)         /* a CUDA runtime / driver call failed (includes: no device) */
#define COLIBRI_ERR_STATE (-5)        /* forward before load_weights, or no forward yet */
#define COLIBRI_ERR_UNSUPPORTED (-6)  /* shape/dtype combination this build does not run */
#define COLIBRI_ERR_DEVICE (-7)       /* a kernel reported a failure through the device status word */

/* ---- enums (stored as int32_t in the structs) ---- */
#define COLIBRI_DTYPE_F32 0   /* fp32 activations and weights: SIMT fp32 path           */
#define COLIBRI_DTYPE_BF16 1  /* bf16 activations and weights: tcgen05 tensor-core path  */
#define COLIBRI_ACT_RELU_BIAS 0 /* y = W2 max(W1 x + b1, 0) + b2 (b1, b2 required)       */
#define COLIBRI_ACT_SWIGLU 1    /* y = W2 (silu(W1 x) * (W3 x)), no biases                 */

#define COLIBRI_GATE_SOFTMAX_SELECTED 0 /* softmax over the k selected logits (sums to 1)          */
#define COLIBRI_GATE_SOFTMAX_ALL 1      /* softmax over all experts, at the selected ones (sum < 1) */

/* Grouped-GEMM form of the most recent call (colibri_moe_last_gemm) */
#define COLIBRI_GEMM_NONE 0                /* no forward yet, T = 0, or a call without GEMMs        */
#define COLIBRI_GEMM_DECODE_FUSED 1        /* decode batch: the cooperative weight-streaming kernel  */
#define COLIBRI_GEMM_DECODE_SPLIT 2        /* decode batch: separate weight-streaming kernels        */
#define COLIBRI_GEMM_PAIR 3                /* CTA-pair GEMMs, token rows on M, one launch each       */
#define COLIBRI_GEMM_SINGLE_CTA 4          /* single-CTA tcgen05 GEMMs                               */
#define COLIBRI_GEMM_SIMT 5                /* fp32 SIMT GEMMs                                        */
#define COLIBRI_GEMM_WEIGHT_MAJOR 6        /* CTA-pair GEMMs, weight rows on M, one launch each      */
#define COLIBRI_GEMM_WEIGHT_MAJOR_FUSED 7  /* the same, both projections in one launch               */

#define COLIBRI_MAX_EXPERTS 16
#define COLIBRI_MAX_TOP_K 4

typedef struct colibri_moe colibri_moe_t; /* opaque */

typedef struct {
  int32_t d_model;         /* d: hidden size.  Multiple of 8; bf16 also needs d % 256 == 0        */
  int32_t d_ff;            /* f: expert inner size.  bf16 SwiGLU: f % 128 == 0; bf16 ReLU: f % 256 */
  int32_t num_experts;     /* E, 2..16 routed experts                                               */
  int32_t top_k;           /* k, 1..4 and <= E                                                      */
  int32_t max_tokens;      /* largest T any forward will be given (> 0); sizes the workspace        */
  int32_t dtype;           /* COLIBRI_DTYPE_*: dtype of x and of all weights                         */
  int32_t act;             /* COLIBRI_ACT_*                                                          */
  int32_t has_router_bias; /* 0/1: b_r present                                                       */
  int32_t out_dtype;       /* COLIBRI_DTYPE_*: dtype of out (the combine itself is fp32)             */
  int32_t gate_mode;       /* COLIBRI_GATE_*                                                         */
  int32_t has_shared_expert; /* 0/1: an always-on expert of the same shape, added with weight 1      */
} colibri_moe_config_t;

/* Per-tensor pointers, nn.Linear [out, in] row-major, dtype = config.dtype for weights and fp32 for
 * biases.  Each pointer may be a host or a device pointer; load_weights copies (it never keeps
 * them).  Arrays of E pointers are host arrays. */
typedef struct {
  const void* w_router;      /* [E, d]                                             */
  const float* b_router;     /* [E] fp32, required iff has_router_bias, else NULL  */
  const void* const* w1;     /* E x [f, d]: ReLU W1, SwiGLU W_gate                 */
  const void* const* w3;     /* E x [f, d]: SwiGLU W_up; NULL for ReLU             */
  const void* const* w2;     /* E x [d, f]: W2 / W_down                            */
  const float* const* b1;    /* E x [f] fp32: ReLU only (required), else NULL      */
  const float* const* b2;    /* E x [d] fp32: ReLU only (required), else NULL      */
  const void* ws1;           /* shared expert [f, d] (W1 / W_gate); NULL without one */
  const void* ws3;           /* shared expert [f, d] W_up (SwiGLU)                    */
  const void* ws2;           /* shared expert [d, f] (W2 / W_down)                    */
  const float* bs1;          /* shared expert [f] fp32 (ReLU)                         */
  const float* bs2;          /* shared expert [d] fp32 (ReLU)                         */
} colibri_moe_weights_t;

/* Validates the config, selects `device`, and allocates the workspace for max_tokens tokens
 * (expert-contiguous activation rows, routing arrays, per-chunk histograms, staging for
 * forward_host).  On success *out receives the context; on failure *out is NULL. */
COLIBRI_API int colibri_moe_create(const colibri_moe_config_t* cfg, int device, colibri_moe_t** out);

/* Copies all weights into one device arena (each expert's block 256-byte aligned, experts
 * contiguous; zskr.cn 2.2) in the layout the kernels read, builds the TMA descriptors, then
 * synchronises `stream`.  May be called again to replace the weights. */
COLIBRI_API int colibri_moe_load_weights(colibri_moe_t* ctx, const colibri_moe_weights_t* w, void* stream);

/* out[T, d] = MoE layer applied to x[T, d].  x (config.dtype) and out (config.out_dtype) are device
 * pointers, row-major and contiguous, and must not overlap.  Asynchronous on `stream`: no host
 * synchronisation and no allocation, so a call can be captured into a CUDA graph and replayed (the
 * replay reads x and writes out at the captured addresses).  T == 0 is a no-op.  Calls on one context
 * must be ordered (same stream, or synchronised): the workspace is shared.  With two routed slots and
 * an fp32 output, out is written by accumulation (cleared first, then both expert outputs added). */
COLIBRI_API int colibri_moe_forward(colibri_moe_t* ctx, const void* x, void* out, int32_t T, void* stream);

/* Same as forward with HOST buffers: copies x host->device into the context's staging buffer,
 * runs forward, copies out device->host, then synchronises `stream`.  Pinned host memory gives
 * asynchronous copies; pageable memory works but copies synchronously. */
COLIBRI_API int colibri_moe_forward_host(colibri_moe_t* ctx, const void* x_host, void* out_host, int32_t T, void* stream);

/* Pipelined form of forward_host for serving loops (no counterpart in the articles, which run one
 * synchronous batch at a time): returns without waiting.  The context keeps three device staging
 * slots used in turn and two internal copy streams, so the host->device copy of one call and the
 * device->host copies of earlier ones overlap the forwards on `stream` (a call's input copy waits
 * only for the result copy of the call three back).  The forward is enqueued
 * on `stream` after this call's input copy; the result copy is ordered after it on an internal
 * stream.  out_host holds the result, and x_host may be reused, once colibri_moe_host_sync returns
 * (until then the copies may still be reading or writing them).  Host buffers should be pinned:
 * pageable memory makes the copies synchronous.  Calls on one context must use one `stream` (or be
 * ordered by the caller).  Errors as forward; -4 if a copy or event call fails. */
COLIBRI_API int colibri_moe_forward_host_async(colibri_moe_t* ctx, const void* x_host, void* out_host, int32_t T,
                                               void* stream);

/* Waits until every copy of earlier forward_host_async calls has completed. */
COLIBRI_API int colibri_moe_host_sync(colibri_moe_t* ctx);

/* Routing of the most recent forward -- the routing dump the articles' engine offers as a debug
 * function to call after a forward (zskr.cn 5.2, colibri_dump_routing) -- copied into caller
 * DEVICE buffers on `stream` (any may be NULL): idx[T,k] int32 (slot 0 = highest logit), gate[T,k] fp32, counts[E] int32 (routed
 * experts), offsets[E+1] int32 (row where each routed expert's segment starts; segments padded to
 * 128 rows; offsets[E] is where the shared expert's rows start when there is one), row_of[T,k]
 * int32 (row of token t's slot s; row_of - offsets[e] is t's rank among e's tokens). */
COLIBRI_API int colibri_moe_get_routing(colibri_moe_t* ctx, int32_t* idx, float* gate, int32_t* counts, int32_t* offsets,
                            int32_t* row_of, void* stream);

/* Debug view of internal device buffers (read-only use; valid until destroy or the next forward):
 *   which = 0: Xp, gathered token rows [rows, d] (config.dtype);
 *           1: H, expert hidden activations [rows, f] (bf16 on the bf16 path, fp32 on the fp32 path);
 *           2: Y, expert outputs before the combine [rows, d] (fp32);
 *           3: token_of_row [rows] (int32).
 * Only rows inside an expert's segment [offsets[e], offsets[e] + counts[e]) of the last forward
 * hold defined values; padding rows hold stale data.  Xp is not written by the cooperative decode
 * kernel or with COLIBRI_MOE_GATHER=fused (the GEMM reads x in place), Y not when the combine is
 * fused into the down GEMM.  *ptr receives the device address and *rows the allocated row count
 * (may be NULL). */
COLIBRI_API int colibri_moe_debug_buffer(colibri_moe_t* ctx, int32_t which, void** ptr, int64_t* rows);

/* Number of timed pipeline stages of forward (router, dispatch, up GEMM, down GEMM, combine), for
 * set_stage_events.  A stage holds one kernel, two (the decode path's GEMM + reduction) or none
 * (the combine, when fused into the down GEMM). */
COLIBRI_API int colibri_moe_num_stages(const colibri_moe_t* ctx, int32_t* n_stages);

/* *n = the number of kernels the most recent forward (or forward_host) enqueued: 4 on the grouped
 * GEMM path (bf16 prefill or fp32) with the combine fused into the down GEMM (two slots, fp32
 * output), 5 with a separate combine, one fewer for bf16 prefill batches of 9..1024 tokens (the
 * router writes the dispatch itself), 2 on the
 * decode path (by default T <= 32 for experts of at least 2^25 weights per matrix, else T <= 16;
 * 128 / 64 when the build runs single-CTA GEMMs: the router and one cooperative kernel), one fewer
 * than the grouped-GEMM counts where the weight-major GEMM runs both projections in one launch
 * (colibri_moe_last_gemm tells which), 6 on the separate
 * decode kernels (COLIBRI_MOE_DECODE_FUSED=0, T <= 64); 0 before the first forward and after a
 * forward with T = 0; after an expert-parallel call, the kernels that call enqueued. */
COLIBRI_API int colibri_moe_last_kernel_count(const colibri_moe_t* ctx, int32_t* n);

/* *kind = the grouped-GEMM form (COLIBRI_GEMM_*) the most recent forward, forward_host or
 * ep_experts call ran: which of the Compute-stage implementations (zskr.cn/news/2272131, "Colibri:
 * a lightweight C MoE inference engine for edge devices", 2.1: one GEMM per expert over its rows)
 * served the batch, chosen from its size and the build's switches.  A debugging and benchmarking
 * aid; results are the same whichever form runs (bit for bit between the bf16 prefill forms).
 * Errors: COLIBRI_ERR_INVALID_ARG for a NULL argument. */
COLIBRI_API int colibri_moe_last_gemm(const colibri_moe_t* ctx, int32_t* kind);

/* Stage timing: with n == num_stages + 1 cudaEvent_t values (passed as void*), every later forward
 * records events[i] just before stage i and events[n-1] after the last stage, on its stream; NULL
 * entries are skipped (record only the boundaries you need: each record sits between two kernels).
 * events == NULL (n == 0) turns it off.  The caller owns the events. */
COLIBRI_API int colibri_moe_set_stage_events(colibri_moe_t* ctx, void* const* events, int32_t n);

/* Reads (synchronously) and clears the device status word that kernels set when a bounded wait
 * gives up or an index check fails: *status = 0 means none did. */
COLIBRI_API int colibri_moe_device_status(colibri_moe_t* ctx, int32_t* status);

/* Failure-detection probe (a diagnostic with no counterpart in the articles).  Every wait inside
 * the layer's kernels is bounded: when one gives up, the kernel sets a bit of the device status
 * word, stops, drains its own copies and returns, and colibri_moe_device_status reports the bit.
 * This call enqueues on `stream` (a cudaStream_t, NULL = legacy default stream) one small kernel
 * that runs the same bounded wait on a barrier nothing arrives on, for timeout_us microseconds
 * (1 .. 1000000), then sets COLIBRI_STATUS_WAIT_PROBE.  No fault, no hang: the context stays usable.
 * Returns COLIBRI_ERR_INVALID_ARG for a NULL ctx or a limit out of range, COLIBRI_ERR_CUDA if the
 * launch fails.  Asynchronous: read the bit with colibri_moe_device_status. */
#define COLIBRI_STATUS_WAIT_PROBE (1 << 6)
COLIBRI_API int colibri_moe_probe_wait_timeout(colibri_moe_t* ctx, int32_t timeout_us, void* stream);

/* Routing without any allocation (no counterpart in the articles: an addition for callers that
 * cannot allocate device memory -- code that runs inside a host framework whose memory pool owns
 * the whole GPU, real-time loops where cudaMalloc's implicit synchronisation is not allowed, or
 * deployments with a fixed device-memory budget set at start-up).  It computes, from device
 * buffers on the CURRENT device, the routing colibri_moe_get_routing reports after a forward of
 * the same x and router weights (top-2, gates summing to 1): idx[T,2], gate[T,2], counts[E],
 * offsets[E+1], row_of[T,2].  Its router kernel may sum the logits in another order than the one
 * forward picks for the same T, so the two agree on every token whose fp64 logit gaps (first to
 * second and second to third expert) are at least 1e-5, with gates within 1e-5; a token closer to
 * a tie may be routed either way (and counts, offsets and rows follow its choice).
 *   x [T, d_model] and w_router [E, d_model] in `dtype` (16-byte aligned), b_router [E] fp32 or NULL.
 * It needs no context.  Its scratch (per-chunk histograms and the routing summary) is a fixed
 * __device__ array of about 137 KB inside the library, present on every GPU that loads the library
 * until the process exits; hence T <= 65536 (larger T returns COLIBRI_ERR_INVALID_ARG).  The first
 * call on a device looks up the array's device address and sets kernel attributes (host-side
 * set-up, no allocation); make that first call before any stream capture.  Every call on a device
 * shares the one array, and each call clears the part that must start at zero: calls that overlap
 * on the GPU (different streams, or concurrent host threads) race and give wrong results.
 * Asynchronous on `stream`; it calls no cudaMalloc, cudaFree or allocating library routine.  It
 * has no context and so no device status word: a bounded wait that gives up inside its router
 * kernel is not reported (the routing it returns is then undefined). */
COLIBRI_API int colibri_moe_route_noalloc(const void* x, const void* w_router, const float* b_router, int32_t T,
                                          int32_t d_model, int32_t num_experts, int32_t dtype, int32_t* idx,
                                          float* gate, int32_t* counts, int32_t* offsets, int32_t* row_of,
                                          void* stream);

/* ---- expert parallelism: the experts of one layer split over ep_size GPUs ----
 * The articles run the whole layer on one device; these calls split its Dispatch and Compute stages
 * (zskr.cn 2.1) across GPUs, one process (and one context) per GPU, with the caller's communicator
 * moving rows between them.  Rank r owns experts [r*El, (r+1)*El), El = E / ep_size; it routes its
 * own tokens over all E experts and runs the expert FFN for every token routed to its experts:
 *
 *   ep_dispatch(x, T) -> send_rows [T*k, d], send_counts [E]     rows grouped by expert, so rank q's
 *                                                                rows are one contiguous block
 *   all-to-all of send_counts (El per peer) -> recv_counts [ep_size, El]   (host copy for the call below)
 *   all-to-all of the rows (split sizes = per-peer sums of the counts) -> recv_rows
 *   ep_experts(recv_rows, recv_counts) -> y_rows [R, d] fp32     same order as recv_rows
 *   all-to-all of y_rows back (the split sizes swapped) -> y_back [T*k, d] fp32
 *   ep_combine(y_back) -> out [T, d]                              gate-weighted sum in slot order
 *
 * Every call is asynchronous on `stream`, allocates nothing and synchronises nothing; the caller
 * orders them with its exchanges.  The result equals colibri_moe_forward's for the same weights,
 * bit for bit wherever forward runs the grouped GEMMs (batches above its decode-path limit). */

/* Context of rank ep_rank of an expert-parallel layer.  cfg describes the whole layer (num_experts =
 * E across all ranks, max_tokens = most tokens one rank routes per step); E must be a multiple of
 * ep_size (1..E); no shared expert.  max_recv_rows bounds the rows one ep_experts call may receive
 * (at most ep_size * max_tokens * top_k; the workspace holds that many expert rows).  The context
 * holds the router weights and its own experts' weights only: load_weights reads entries
 * [ep_rank*El, (ep_rank+1)*El) of the per-expert arrays and ignores (may be NULL) the others.
 * colibri_moe_forward / forward_host / forward_host_async return COLIBRI_ERR_UNSUPPORTED on it.
 * Errors: COLIBRI_ERR_INVALID_ARG (bad rank, size, or E not divisible), COLIBRI_ERR_UNSUPPORTED
 * (shared expert), and those of colibri_moe_create. */
COLIBRI_API int colibri_moe_ep_create(const colibri_moe_config_t* cfg, int32_t ep_rank, int32_t ep_size,
                                      int32_t max_recv_rows, int device, colibri_moe_t** out);

/* Source side, before the exchange: routes x [T, d] (device, config.dtype, T <= max_tokens) over all
 * E experts and writes send_rows [T*k, d] (device, config.dtype): row i holds a token routed to the
 * expert whose block contains i, experts in ascending order, each expert's tokens in ascending token
 * order (the dispatch order of zskr.cn 3.2, without padding).  send_counts [E] (device int32) gets
 * the rows per expert.  The routing is kept for ep_combine (and get_routing, whose row_of then gives
 * each (token, slot)'s row of send_rows).  x, send_rows and send_counts must not overlap; x and
 * send_rows 16-byte aligned.  T == 0 zeroes send_counts. */
COLIBRI_API int colibri_moe_ep_dispatch(colibri_moe_t* ctx, const void* x, int32_t T, void* send_rows,
                                        int32_t* send_counts, void* stream);

/* Expert side: recv_counts is a HOST int32 array [ep_size, El]: the rows source p sent for local
 * expert j.  recv_rows [R, d] (device, config.dtype, R = the sum of recv_counts <= max_recv_rows) are
 * the received rows in source order, each source's rows grouped by local expert.  Writes y_rows
 * [R, d] (device fp32): each row's expert output y_e(x) (no gate), in the order of recv_rows.
 * Runs the grouped up GEMM (activation fused) and down GEMM over the local experts. */
COLIBRI_API int colibri_moe_ep_experts(colibri_moe_t* ctx, const void* recv_rows, const int32_t* recv_counts,
                                       void* y_rows, void* stream);

/* Source side, after the exchange back: y_back [T*k, d] (device fp32) holds the expert outputs of
 * send_rows' rows in the same order; out [T, d] (device, config.out_dtype) = sum over the token's
 * slots of gate * y_back[row], in slot order in fp32 (m.nxbn.cn 3.3), T from the last ep_dispatch. */
COLIBRI_API int colibri_moe_ep_combine(colibri_moe_t* ctx, const float* y_back, void* out, void* stream);

/* Frees everything the context owns (the articles' colibri_free, the release call every program
 * must make once it is done: zskr.cn 4.3, m.nxbn.cn 4.3).  NULL-safe. */
COLIBRI_API void colibri_moe_destroy(colibri_moe_t* ctx);

/* Static text for one of the status codes above (the int codes of m.nxbn.cn 3.3 and 5.1); unknown
 * codes get a generic string.  Never NULL. */
COLIBRI_API const char* colibri_moe_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif
