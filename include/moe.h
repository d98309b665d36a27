/*
 * moe.h — C ABI of libmoe.so, the GB300 (sm_103a) sparse-MoE feed-forward layer.
 *
 * The layer is the MoE FFN sublayer described in "Step3.5 Flash 大模型技术深度
 * 解析：稀疏 MoE、混合注意力与 MTP 的高效推理革命" (jsqmd.com):
 *   §3.2.1  each MoE layer holds E routed experts (288) and one always-on
 *           shared expert, each an independent FFN;
 *   §3.2.2  a linear router followed by a softmax scores every routed expert,
 *           the k most probable (top-8) plus the shared expert run, and their
 *           outputs are summed with weights.
 * Readings where that page is silent: the expert FFN is SiLU-gated,
 *   y_e(x) = W_d[e] · (silu(W_g[e]·x) ⊙ (W_u[e]·x));
 * a routed expert's weight is its softmax probability over all E experts (not
 * renormalised over the top-k); the shared expert's weight is 1; equal
 * probabilities rank the lower expert index first.  The layer maps the
 * sublayer input x to the FFN output (no norm, no residual add).
 *
 * Conventions shared by every entry point:
 *   - All tensors are dense row-major.  bf16 is IEEE bfloat16 bit patterns.
 *   - Device pointers must point to memory of the device that was current at
 *     moe_init, 16-byte aligned.  The caller owns every buffer it passes.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     is asynchronous on it and never synchronises the device, except
 *     moe_check and moe_forward_host, which say so.
 *   - A handle holds one workspace: calls on one handle must be ordered (one
 *     stream, or ordered by the caller).  Different handles are independent.
 *   - Any host thread may call: each call on a handle makes the handle's device
 *     current for its duration (binding the device's primary context in a
 *     thread that has not used CUDA yet) and restores the caller's device.
 *   - MOE_TRACE_ERRORS=1 in the environment prints every failing CUDA call
 *     (source line and error name) on stderr.
 *   - Return value: MOE_OK (0) or one of the MOE_ERR_* codes below.  Argument
 *     errors are found on the host before anything is enqueued; nothing traps
 *     on the device.  Device-side failures (a pipeline wait that exceeded its
 *     time limit) set an error word that moe_check reports.
 */
#ifndef MOE_H_
#define MOE_H_

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1     /* null / misaligned pointer, bad size, bad handle      */
#define MOE_ERR_TOO_MANY_TOKENS 2 /* T > max_tokens of the handle                         */
#define MOE_ERR_UNSUPPORTED 3     /* shape outside the supported set (see moe_config)     */
#define MOE_ERR_CUDA 4            /* a CUDA runtime/driver call failed                    */
#define MOE_ERR_DEVICE 5          /* a kernel reported a failure (moe_check)              */
#define MOE_ERR_NO_DEVICE 6       /* no sm_100-family (Blackwell) device current          */

/*
 * Layer shape.  Supported set: d_model % 128 == 0, ffn_width % 128 == 0,
 * 1 <= n_experts <= 512, 1 <= top_k <= min(n_experts, 32), has_shared in {0,1},
 * 1 <= max_tokens <= 1<<20 with (top_k+1)*max_tokens < 2^31.
 */
typedef struct moe_config {
  int d_model;    /* d: hidden size (4096 for Step 3.5 Flash)                    */
  int n_experts;  /* E: routed experts (288)                                      */
  int top_k;      /* k: routed experts per token (8)                              */
  int ffn_width;  /* F: expert FFN width (1280)                                   */
  int has_shared; /* 1: add the always-on shared expert (group index E)           */
  int max_tokens; /* largest T any later call may pass; sizes the workspace       */
  int out_fp32;   /* 0: y is bf16 [T][d]; 1: y is fp32 [T][d]                     */
} moe_config;

/*
 * Weights, all device pointers, borrowed (not copied): they must stay alive
 * and unchanged until moe_free.  G = n_experts + has_shared groups; group E is
 * the shared expert.
 *   w_router   fp32 [E][d]
 *   w_gate_up  bf16 [G][2F][d]   rows 0..F-1 are the gate projection W_g,
 *                                rows F..2F-1 the up projection W_u
 *   w_down     bf16 [G][d][F]
 */
typedef struct moe_weights {
  const float* w_router;
  const void* w_gate_up;
  const void* w_down;
} moe_weights;

typedef struct moe_handle moe_handle;

/*
 * Validates cfg and w, allocates the workspace for cfg->max_tokens on the
 * current device, builds the TMA descriptors of the weights and writes a new
 * handle to *out.  Synchronous.  On failure *out is set to NULL and nothing
 * stays allocated.
 */
int moe_init(const moe_config* cfg, const moe_weights* w, moe_handle** out);

/*
 * FP8 expert weights ("Step3.5 Flash 大模型技术深度解析" §8.1: FP8/FP16 mixed-
 * precision inference; format, scales and the activations' form are this
 * library's reading of that line).  Device pointers, borrowed like moe_weights:
 *   w_router   fp32 [E][d]
 *   w_gate_up  [G][2F][d] bytes: OCP FP8 E4M3 codes, same row order as bf16
 *   s_gate_up  fp32 [G][2F]   the scale of each row of w_gate_up
 *   w_down     [G][d][F] bytes: E4M3 codes
 *   s_down     fp32 [G][d]    the scale of each row of w_down
 * Weight value = E4M3 value of the code * the row's scale (moe_quantize_fp8
 * produces such codes and scales from bf16 rows).
 */
typedef struct moe_weights_fp8 {
  const float* w_router;
  const void* w_gate_up;
  const float* s_gate_up;
  const void* w_down;
  const float* s_down;
} moe_weights_fp8;

/*
 * moe_init for FP8 expert weights.  The handle then runs the same calls (route,
 * forward, forward_host, route_stats, ...).  Inside moe_forward the E4M3 codes
 * meet E4M3 activations on the tensor cores: every token row x (and every row
 * of the gate output H, kept as fp16 in between) is carried as two E4M3 rows,
 * hi = e4m3(s*v) and lo = e4m3(s*v - hi), with one power-of-two scale s per row
 * (the largest with s*max|v| <= 448); hi + lo reproduces a bf16 x exactly
 * except for entries below about 1/1000 of the row's largest (there to within
 * 2^-18 of it), and H to 8 significant bits.  Products accumulate in fp32 and
 * the weight row scales and 1/s are applied to the sums.  x and H must lie
 * within the fp16 range (|v| < 65504).  MOE_FP8_X2=0 in the environment (and
 * ffn_width > 8192) widens the codes to fp16 on chip instead and keeps x and H
 * as fp16.  Token tiles are
 * at most 128 rows (no CTA-pair tiles).  Same errors as moe_init.
 */
int moe_init_fp8(const moe_config* cfg, const moe_weights_fp8* w, moe_handle** out);

/*
 * Expert parallelism (page 2 §3.2.3 and §8.1: EP = 8, the 288 routed experts
 * spread as 36 per GPU).  Rank r of ep_size owns the routed experts
 * [r * E_loc, (r + 1) * E_loc), E_loc = n_experts / ep_size, and the shared
 * expert.  One layer call on a rank is three library phases around two
 * exchanges that the caller performs (any all-to-all, e.g. NCCL):
 *   1. moe_ep_dispatch: route this rank's T tokens over all E experts and
 *      lay the routed rows out expert by expert (rank q's rows are one block);
 *   -> exchange the counts and the rows (+ their gate weights) to the owners;
 *   2. moe_ep_experts: run the local experts over the rows received from
 *      every source (blocks in source order, inside a block expert by expert);
 *   -> exchange the output rows and their exponent chunks back, per source;
 *   3. moe_ep_combine: this rank's shared expert and the fixed-order combine.
 * The rows a rank gets back, concatenated in rank order, line up with its own
 * dispatch order, and so do their exponent chunks (a (source, expert) block is
 * cut into 16-row chunks exactly as the source cuts that expert's rows).
 * Not part of the pages' text: the phase split is this library's; bf16 weights
 * only.
 */
typedef struct moe_ep_config {
  moe_config layer;   /* the whole layer (n_experts = all routed experts), this rank's max_tokens */
  int ep_size;        /* ranks, >= 1, divides n_experts                                    */
  int ep_rank;        /* this rank, 0 <= ep_rank < ep_size                                 */
  int max_recv_rows;  /* most routed rows moe_ep_experts may be given in one call          */
} moe_ep_config;

/* w_router fp32 [E][d] (all experts); w_gate_up bf16 [E_loc + has_shared][2F][d]
 * and w_down bf16 [E_loc + has_shared][d][F]: this rank's experts in order, then
 * the shared expert.  Device pointers, borrowed until moe_free. */
typedef struct moe_ep_weights {
  const float* w_router;
  const void* w_gate_up;
  const void* w_down;
} moe_ep_weights;

/* A handle for phases 1-3 (moe_route also works; moe_forward and
 * moe_forward_host return MOE_ERR_INVALID_ARG on it).  Same errors as
 * moe_init, plus MOE_ERR_UNSUPPORTED when ep_size does not divide n_experts. */
int moe_ep_init(const moe_ep_config* cfg, const moe_ep_weights* w, moe_handle** out);

/*
 * Phase 1.  x bf16 [T][d] (device, T <= max_tokens).  Writes (device, caller-
 * owned): send_rows bf16 [T*k][d] (the routed rows in dispatch order: rank 0's
 * block, then rank 1's, ...), send_w fp32 [T*k] (each row's gate weight),
 * send_counts int [E] (rows per expert; rank q's part is [q*E_loc, (q+1)*E_loc)),
 * and rows_per_rank (HOST int [ep_size]).  Synchronises `stream` (the exchange
 * sizes are needed on the host).  Keeps this call's routing for phase 3.
 */
int moe_ep_dispatch(moe_handle* h, const void* x, int T, void* send_rows, float* send_w, int* send_counts,
                    int* rows_per_rank, void* stream);

/*
 * Phase 2.  recv_rows bf16 [n_recv][d], recv_w fp32 [n_recv], recv_counts int
 * [ep_size][E_loc] (device): what every source sent, in source order.
 * n_recv <= max_recv_rows and must equal the sum of recv_counts
 * (MOE_ERR_INVALID_ARG otherwise).  Writes out_rows fp16 [n_recv][d] and
 * out_exp int8 [chunks][d] (device, caller-owned; chunks <= n_recv/16 +
 * ep_size*E_loc), the outputs w * FFN(row) in the library's scaled fp16
 * (value = out_rows * 2^out_exp, one exponent per feature and 16-row chunk),
 * and chunks_per_source (HOST int [ep_size]): the exponent chunks of each
 * source's block, which follow one another in source order.  Synchronises
 * `stream` before the GEMMs (to check the counts).
 */
int moe_ep_experts(moe_handle* h, const void* recv_rows, const int* recv_counts, const float* recv_w, int n_recv,
                   void* out_rows, void* out_exp, int* chunks_per_source, void* stream);

/*
 * Phase 3.  ret_rows fp16 [T*k][d] and ret_exp int8 [chunks][d] (device): the
 * rows and exponent chunks the owners sent back, concatenated in rank order.
 * Runs the shared expert on this rank's tokens of the last moe_ep_dispatch and
 * writes y [T][d] (bf16, or fp32 with out_fp32) with the same fixed-order
 * combine as moe_forward.  Asynchronous.
 */
int moe_ep_combine(moe_handle* h, const void* ret_rows, const void* ret_exp, void* y, void* stream);

/*
 * Per-row E4M3 quantisation of a bf16 matrix w [rows][cols] (device):
 *   s[r] = max_i |w[r][i]| / 448 (fp32),   q[r][i] = E4M3 nearest to w[r][i] / s[r]
 * (fp32 quotient, ties to even, magnitudes above 448 saturated); a row of
 * zeros gets s = 0 and codes 0.  q: [rows][cols] bytes, s: fp32 [rows], both
 * device, caller-owned.  Asynchronous on `stream`.  Needs no handle.
 * Returns MOE_ERR_INVALID_ARG for null / host pointers or sizes out of range.
 */
int moe_quantize_fp8(const void* w, long long rows, int cols, void* q, float* s, void* stream);

/*
 * Routing only (§3.2.2 router + softmax + top-k, and the dispatch order):
 *   x        bf16 [T][d]   layer input, device
 *   idx      int  [T][k]   chosen experts, by descending probability (ties:
 *                          lower index first), device
 *   prob     fp32 [T][k]   their softmax probabilities (over all E), device
 *   perm     int  [T*k]    assignment ids a = t*k + j listed expert by expert,
 *                          inside one expert by increasing t, device
 *   offsets  int  [E+2]    offsets[e] = rows of experts < e; offsets[E+1] =
 *                          offsets[E] + T (the shared expert's rows, token
 *                          order, implicit in perm), device
 *   gap      fp32 [T] or NULL: p(k-th) - p((k+1)-th) per token (+inf if k == E),
 *                          device
 * 0 <= T <= max_tokens.  Results are deterministic run to run.
 */
int moe_route(moe_handle* h, const void* x, int T, int* idx, float* prob, int* perm, int* offsets,
              float* gap, void* stream);

/*
 * The whole layer: routing, dispatch, the grouped expert FFNs (the shared
 * expert as one more group), and the gate-weighted combine
 *   y[t] = sum_{j<k} prob[t][j] * y_{idx[t][j]}(x_t)  +  y_shared(x_t),
 * summed in slot order then the shared expert, in fp32, without atomics
 * (bit-identical run to run).  With few tokens the bf16 expert GEMMs may cut
 * K into parts (MOE_GEMM_KSPLIT in the environment: 1 = never, 2..4 = that
 * many per work item, b = equal contiguous ranges of K steps per CTA); the
 * parts are summed in a fixed order, so this holds there too.
 *   x  bf16 [T][d], device;  y  [T][d] bf16 or fp32 (cfg.out_fp32), device.
 * 0 <= T <= max_tokens; T == 0 enqueues nothing.
 */
int moe_forward(moe_handle* h, const void* x, int T, void* y, void* stream);

/*
 * Per-call routing choices, after "Step3.5 Flash 大模型技术深度解析" (jsqmd.com)
 * §8.2, which varies the number of experts per token at inference time
 * (top-4 for simple inputs, top-8 for complex ones).
 *   top_k        0: the handle's top_k; otherwise 1..cfg.top_k experts per token
 *   renormalize  0: weights are the softmax probabilities over all E experts;
 *                1: the k weights are divided by their sum (summed in slot order)
 */
typedef struct moe_call_options {
  int top_k;
  int renormalize;
} moe_call_options;

/*
 * moe_route / moe_forward with per-call options (opt may be NULL = defaults).
 * With top_k = k' the route outputs are idx/prob [T][k'], perm [T*k'];
 * prob holds the weights actually used (renormalised if asked).  The gap is
 * always p(k'-th) - p((k'+1)-th) of the raw probabilities.
 */
int moe_route_ex(moe_handle* h, const void* x, int T, const moe_call_options* opt, int* idx, float* prob,
                 int* perm, int* offsets, float* gap, void* stream);
int moe_forward_ex(moe_handle* h, const void* x, int T, const moe_call_options* opt, void* y, void* stream);

/*
 * Routing statistics of a batch (router, softmax and top-k with the handle's
 * top_k; no expert FFNs), after §3.2.3 of the same page: the E experts form
 * n_groups equal groups of consecutive indices (8 groups of 36 for EP = 8).
 *   counts   int   [E]         rows routed to each expert, device
 *   group_f  fp32  [n_groups]  share of the T*k rows that go to group g, device
 *   group_p  fp32  [n_groups]  mean over tokens of the group's probability mass, device
 *   summary  fp32  [4]         device: [0] L_EP = n_groups * sum_g f_g p_g (1 when
 *                              balanced), [1] max/mean rows per expert, [2] mean
 *                              router entropy -sum_e p_e ln p_e (nats), [3] experts
 *                              with no row
 * 1 <= n_groups <= 64 and n_groups divides E.  Deterministic run to run.
 */
int moe_route_stats(moe_handle* h, const void* x, int T, int n_groups, int* counts, float* group_f,
                    float* group_p, float* summary, void* stream);

/*
 * moe_forward on host buffers: copies x (host, bf16 [T][d]) to the handle's
 * staging buffer, runs the layer and copies y back to host memory (bf16 or
 * fp32 per cfg.out_fp32), all on `stream`, then synchronises that stream.
 * Host buffers should be page-locked for the copies to be asynchronous.
 */
int moe_forward_host(moe_handle* h, const void* x_host, int T, void* y_host, void* stream);

/*
 * Synchronises `stream`, then reads and clears the handle's device error word.
 * Returns MOE_OK, MOE_ERR_DEVICE if a kernel since the last check gave up on a
 * pipeline wait, or MOE_ERR_CUDA if the stream reports an error.  After
 * MOE_ERR_DEVICE the outputs of the calls since the last check are undefined;
 * the check also clears the handle's K split part counts, so the handle is
 * usable again.
 */
int moe_check(moe_handle* h, void* stream);

/*
 * Number of kernels the last moe_forward / moe_forward_ex / moe_forward_host
 * on this handle enqueued (0 after a call with T = 0; otherwise 7: the router
 * GEMM, top-k, dispatch, row gather, gate/up, down and combine kernels, and
 * from 1024 tokens on 9: two more that count each expert's rows per 256-token
 * chunk and scan those counts, in place of counters in the top-k kernel; from
 * 2048 tokens on 11 with bf16 weights: the shared expert's gate/up and down on
 * a second stream; from 1 to 4 tokens with bf16 weights 4: one launch for the
 * router's logits and copies of the token rows (the gate/up launch finishing
 * the top-k and the dispatch), gate/up, down and combine; with FP8 weights 5:
 * the routing launch also does the top-k and dispatch, and the row gather
 * follows it; one more on a handle with two-term E4M3 rows: the
 * requantisation of H).
 * Host-only, never synchronises.  Returns -1 for an invalid handle.  No
 * counterpart in the pages: instrumentation for launch accounting.
 */
int moe_last_kernel_count(const moe_handle* h);

/*
 * Upper bound, in nanoseconds, on every pipeline wait inside the kernels of
 * this handle (default 2e9).  A wait that exceeds it makes the kernel record
 * MOE_ERR_DEVICE, drain the copies it started, release its tensor memory and
 * return.  0 restores the default.
 */
int moe_set_wait_limit(moe_handle* h, unsigned long long ns);

/*
 * Per-stage timing.  enable != 0: every later moe_forward / moe_forward_host on
 * this handle also records CUDA events on its stream at the boundaries of its
 * six stages (0 routing, 1 dispatch, 2 row gather, 3 gate/up GEMM, 4 down GEMM,
 * 5 combine); up to 4096 calls are kept, later calls are not recorded.
 * enable == 0 stops recording and discards the record.
 */
int moe_profile_enable(moe_handle* h, int enable);

/*
 * Waits for the recorded events, writes the total milliseconds of each stage
 * over the recorded calls to ms[0..5] and the number of calls to *n_calls,
 * then clears the record (recording stays as it was).
 */
int moe_profile_read(moe_handle* h, float* ms, int* n_calls);

/*
 * moe_dispatch_noalloc — the dispatch step alone (offsets and perm, exactly as
 * moe_route writes them) from routing the caller already has, without a handle
 * and without allocating any device memory.  The paper has no counterpart for
 * this entry point; it exists for callers that cannot call cudaMalloc: code
 * whose device memory is owned by another allocator or memory pool that must
 * not be bypassed, and latency-critical loops that cannot afford cudaMalloc's
 * implicit device synchronisation.
 *   idx      int [T][k] device: expert ids in [0, n_experts), distinct within
 *            a row (ids outside the range are ignored: their perm slots are
 *            left unwritten)
 *   offsets  int [n_experts+2] device (output, as in moe_route)
 *   perm     int [T*k] device (output, as in moe_route)
 * Its scratch (per-expert row counts) is a fixed array of 512 ints in the
 * library's own device memory, present on every GPU that loads the library
 * until the process exits.  Limits: n_experts <= 512 and top_k <= 32 (beyond
 * them: MOE_ERR_UNSUPPORTED); 4-byte aligned pointers.  The array is cleared at
 * the start of every call, but it is shared: calls whose work overlaps on the
 * GPU (different streams, or different host threads on one device) race and
 * give wrong results; order them.  The first call on each device looks the
 * array's address up (with that device current), so make that first call
 * before any stream capture.  The looked-up address is kept for the life of
 * the process: after cudaDeviceReset (or anything else that replaces the
 * device's primary context) it no longer points at the array, so the entry
 * point must not be called on that device again.  Asynchronous on `stream`.
 */
int moe_dispatch_noalloc(const int* idx, int T, int n_experts, int top_k, int has_shared, int* offsets, int* perm,
                         void* stream);

/* Frees the handle and its workspace (synchronises the device first). */
int moe_free(moe_handle* h);

/* Static description of a status code; never NULL. */
const char* moe_status_string(int status);

/*
 * Launches one kernel that waits on a barrier nothing ever arrives at, with a
 * limit of `limit_ns`, on `stream`, then synchronises it.  Returns
 * MOE_ERR_DEVICE when the wait gave up as designed (the expected result),
 * MOE_OK if it did not.  Exercises the bounded-wait path without a fault.
 */
int moe_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
