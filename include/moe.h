/*
 * moe.h -- C ABI of the single-GPU mixture-of-experts FFN layer forward (sm_103a).
 *
 * The layer, as the expert-parallelism pages state it ("Expert Parallelism (MoE)",
 * section "MoE Layer Structure"; "Expert Parallelism (EP)", section "Key math / How
 * it works"):
 *
 *   1. router: logits = X . W_r^T (+ b_r), softmax over the E experts, top-K per token;
 *   2. dispatch: every token goes to each of its K experts; on one GPU this is a
 *      permutation that packs each expert's rows contiguously (the all-to-all of
 *      "The All-to-All Communication"), after a per-expert capacity
 *      C = floor((T / E) * capacity_factor) drops the assignments that arrive when their
 *      expert is full ("Top-K Routing and Capacity Factor");
 *   3. experts: Linear(d -> F) -> GELU -> Linear(F -> d) on each expert's rows;
 *   4. combine: Y[t] = sum over t's kept assignments of routing_weight * expert_output;
 *   5. aux statistics f_i, P_i and L_aux = alpha * sum_i f_i P_i ("Load Balancing: The
 *      Auxiliary Loss"), reported and never added to Y.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor pointers are DEVICE pointers, row-major, 16-byte aligned, owned by the
 *   caller.  The library never allocates or frees device memory.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).  Every
 *   call only enqueues work on it and returns without synchronising the host.
 * - The returned status covers argument validation and kernel-launch errors.  Errors
 *   that arise on the device (an expert id out of range, a bounded wait that gave up,
 *   packed rows exceeding the buffer, an fp16 overflow) are recorded in a status word inside `ws`;
 *   moe_sync_status() synchronises the stream, returns and clears it.
 * - Activations and weights have the config's dtype (fp32 or bf16); logits, routing
 *   weights, biases and statistics are fp32; the intermediate activation h and the
 *   expert outputs (y_perm, y_shared) are fp16 for bf16 layers and fp32 for fp32
 *   layers; indices are int32.
 * - Weights use the Linear layout [out, in]: W_r [E, d], W1 [G, F, d], W2 [G, d, F].
 * - Flat assignment index a = t*K + k.  Routing ties: logits compare as fp32, higher
 *   first, equal values -> lower expert id.  Routing weights are the softmax
 *   probabilities (cfg.renormalize = 1 divides them by their sum over the K picks).
 * - Drop order: an assignment is dropped iff its expert already holds C assignments
 *   that arrived before it, in flat order unless cfg.drop_order says otherwise.  Rows
 *   inside an expert's packed block are in arrival order.  Routing, counts, offsets,
 *   slot and src are deterministic.
 * - Limits: 1 <= K <= min(E, 32), E <= 256, T >= 0 with T*K < 2^31; d and F multiples
 *   of 8 (bf16) or 4 (fp32).  Violations return MOE_ERR_INVALID / MOE_ERR_UNSUPPORTED.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,      /* bad argument: null / misaligned pointer, bad sizes */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement */
  MOE_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_TIMEOUT = 4,      /* (device) a bounded spin-wait gave up */
  MOE_ERR_DEVICE = 5        /* (device) bad expert id, packed-row or fp16 overflow */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_F16 = 2 /* moe_quantize_e4m3 input only */ } moe_dtype_t;

typedef struct {
  int32_t T;            /* tokens */
  int32_t d;            /* hidden size */
  int32_t E;            /* routed experts */
  int32_t K;            /* experts per token */
  int32_t F;            /* expert width (the "4d" of the FFN) */
  int32_t dtype;        /* moe_dtype_t of activations and weights */
  int32_t capacity;     /* C per expert; < 0 means no dropping */
  int32_t renormalize;  /* 0: w = softmax prob (default); 1: w / sum_k w */
  float alpha;          /* aux-loss weight */
  int32_t drop_order;   /* moe_drop_order_t: the order assignments arrive at experts */
} moe_config;

/* Arrival order that decides which assignments a full expert drops and the row order
 * inside an expert's packed block.  TOKEN_MAJOR (default): flat order a = t*K + k.
 * SLOT_MAJOR: every token's k-th choice arrives before any token's (k+1)-th choice
 * (order k*T + t), so first choices are dropped last. */
typedef enum { MOE_DROP_TOKEN_MAJOR = 0, MOE_DROP_SLOT_MAJOR = 1 } moe_drop_order_t;

/* Bytes of device workspace `ws` the calls below need for this config.  The caller
 * allocates it and ZERO-FILLS it once before first use; the library keeps it
 * consistent afterwards.  One workspace must not be used by two calls that can run
 * concurrently, with one exception: moe_aux_stats reads only the probability sums that
 * moe_route left and writes only its own region (per-expert f_i*P_i and its completion
 * counter), so it may run concurrently with the expert-GEMM calls (moe_expert_up,
 * _gather, _down, their E4M3 forms, moe_grouped_ffn) and moe_combine on the same
 * workspace -- those touch only the status word, by atomic OR.  It must not overlap
 * moe_route, moe_route_select_bias or moe_dispatch on that workspace. */
size_t moe_workspace_size(const moe_config* cfg);

/* Clock telemetry in the workspace: bytes [64, 80) of `ws` hold two uint64 counters to
 * which every CTA of the tensor-core kernels (the router of bf16 layers and the expert
 * GEMMs) adds the SM clock cycles and the nanoseconds it ran.  A caller may zero them,
 * run calls, and read cycles / nanoseconds: the mean SM clock (GHz) those kernels ran at. */
#define MOE_WS_CLOCK_CYCLES_OFFSET 64
#define MOE_WS_CLOCK_NS_OFFSET 72

/* Rows the packed buffers (src, x_perm, h, y_perm) must hold:
 * min(T*K, E*C) with dropping, T*K without. */
int64_t moe_rows_capacity(const moe_config* cfg);

/* Step 1 -- router Linear, softmax over E, top-K ("MoE Layer Structure").
 *   x        [T, d]  dtype, or NULL: then `logits` is an INPUT holding fp32 logits
 *   w_r      [E, d]  dtype (ignored when x == NULL)
 *   b_r      [E]     fp32, nullable (added to the logits before softmax)
 *   logits   [T, E]  fp32, written (or read when x == NULL)
 *   topk_ids [T, K]  int32 out, sorted by logit descending
 *   topk_w   [T, K]  fp32 out, routing weights
 *   ws       workspace; receives per-block partial sums of the softmax probabilities
 *            that moe_aux_stats reduces. */
moe_status_t moe_route(const moe_config* cfg, const void* x, const void* w_r, const float* b_r,
                       float* logits, int32_t* topk_ids, float* topk_w, void* ws, void* stream);

/* Step 1 with a selection-only expert bias: the auxiliary-loss-free balancing that
 * "Expert Parallelism (EP)", "Load balancing" names for DeepSeek-V3 (a per-expert bias
 * adjusted to balance the load instead of an auxiliary loss).  Same as moe_route, except
 * that the top-K choice compares fl32(logit + sel_bias[e]) (ties -> lower id) while the
 * routing weights and the probability sums for P_i stay those of the unbiased softmax.
 *   sel_bias [E] fp32 device pointer, required (4-byte aligned). */
moe_status_t moe_route_select_bias(const moe_config* cfg, const void* x, const void* w_r,
                                   const float* b_r, const float* sel_bias, float* logits,
                                   int32_t* topk_ids, float* topk_w, void* ws, void* stream);

/* Steps 1 and 2's plan in one pass, for token-major arrival order (cfg.drop_order =
 * MOE_DROP_TOKEN_MAJOR, else MOE_ERR_UNSUPPORTED): moe_route -- or, with sel_bias given,
 * moe_route_select_bias -- followed in the same kernel by the histogram, capacity and
 * positions of moe_dispatch ("Top-K Routing and Capacity Factor"): each block of the
 * routing kernel ranks its tokens' assignments per expert and records its count per
 * expert, and a second kernel (one block per expert) turns the counts into each block's
 * count in the blocks before it and writes counts and offsets.  No kernel of this call
 * waits for another block.
 *   x, w_r, b_r, sel_bias (nullable), logits, topk_ids, topk_w: as moe_route /
 *     moe_route_select_bias;
 *   counts [E], offsets [E+1]: as moe_dispatch;
 *   ws: receives the ranks and per-block bases, read by moe_dispatch_planned (and the
 *     probability sums moe_aux_stats reduces).
 * Results are those of moe_route (or moe_route_select_bias) followed by moe_dispatch. */
moe_status_t moe_route_plan(const moe_config* cfg, const void* x, const void* w_r, const float* b_r,
                            const float* sel_bias, float* logits, int32_t* topk_ids, float* topk_w,
                            int32_t* counts, int32_t* offsets, void* ws, void* stream);

/* Step 2's permutation after moe_route_plan on the same ws and topk_ids: slot, src and
 * (x and x_perm given) the row copy x_perm[r] = x[src[r] / K]; an assignment's position
 * in its expert is its rank plus its routing block's base, both left in ws by
 * moe_route_plan.  Arguments and results as moe_dispatch; offsets is an input
 * here (as moe_route_plan wrote it).  Token-major arrival order only. */
moe_status_t moe_dispatch_planned(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                                  const int32_t* offsets, int32_t* slot, int32_t* src,
                                  void* x_perm, void* ws, void* stream);

/* Nudge the selection bias toward balance after a step (the bias-adjustment scheme of
 * the same section; the pages name it without a formula, and this rule is the reading
 * taken here): sel_bias[i] += gamma * sign(T*K/E - counts[i]) -- lowered for experts
 * above the mean load, raised below it, unchanged at it (the comparison is exact, in
 * integers), each sum rounded once to fp32.
 *   counts [E] int32 (pre-drop counts from moe_dispatch), sel_bias [E] fp32 in/out,
 *   gamma >= 0 and finite, else MOE_ERR_INVALID. */
moe_status_t moe_adjust_select_bias(const moe_config* cfg, const int32_t* counts, float* sel_bias,
                                    float gamma, void* stream);

/* Step 2 -- histogram, capacity, drop mask and dispatch permutation
 * ("The All-to-All Communication", "Top-K Routing and Capacity Factor").
 *   x        [T, d] dtype (nullable together with x_perm: routing only, no row copy)
 *   topk_ids [T, K] int32 in
 *   counts   [E]    int32 out: assignments per expert before dropping
 *   offsets  [E+1]  int32 out: exclusive scan of kept counts; offsets[E] = R rows kept
 *   slot     [T, K] int32 out: packed row of assignment (t,k), or -1 if dropped
 *   src      [moe_rows_capacity] int32 out: packed row -> flat assignment t*K+k
 *   x_perm   [moe_rows_capacity, d] dtype out: x_perm[r] = x[src[r] / K]
 * Rows at and beyond offsets[E] are left untouched. */
moe_status_t moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                          int32_t* counts, int32_t* offsets, int32_t* slot, int32_t* src,
                          void* x_perm, void* ws, void* stream);

/* moe_dispatch without a workspace argument.  The pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory when they run the
 * layer (code inside a custom allocator or memory pool, plugins barred from cudaMalloc,
 * runtimes that reserve all memory up front).  Same arguments, outputs, results and
 * argument checks as moe_dispatch minus `ws`: its scratch (status word, scan
 * descriptors, ticket, positions) lives in a static 4 MiB device array inside the
 * library, which every GPU that loads the library holds until the process exits.  It
 * allocates nothing and calls no allocating routine.
 * - Limit: the scratch must hold 256 + ceil(T*K/4096)*E*8 + T*K*4 bytes (each part
 *   rounded up to 256 bytes), i.e. T*K up to about 930,000 assignments at E = 256 and
 *   1,040,000 at E = 8; larger configs return MOE_ERR_UNSUPPORTED with a message on
 *   stderr before any CUDA call.
 * - The first call on each device looks up the array's device address (with that device
 *   current); make that first call before any stream capture.
 * - All calls share the array: calls that can overlap on the GPU (other streams, other
 *   host threads) race and must be serialised by the caller.
 * - Device-side errors (an out-of-range expert id, which gets slot -1 and is left out of
 *   counts; a look-back wait that gave up, which leaves that call's results invalid) are
 *   recorded in the array's status word, which keeps them across calls until
 *   moe_dispatch_noalloc_status reads it.
 * - The test hook moe_test_arm_scan_timeout applies to this call as to moe_dispatch. */
moe_status_t moe_dispatch_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_ids,
                                  int32_t* counts, int32_t* offsets, int32_t* slot, int32_t* src,
                                  void* x_perm, void* stream);

/* Status of the moe_dispatch_noalloc calls on the current device: synchronises `stream`,
 * then returns and clears the status word of the static scratch (MOE_OK, MOE_ERR_TIMEOUT
 * or MOE_ERR_DEVICE), or MOE_ERR_CUDA if a CUDA call failed.  Like the dispatch itself it
 * allocates nothing. */
moe_status_t moe_dispatch_noalloc_status(void* stream);

/* Step 3a -- grouped first expert Linear with GELU fused in its epilogue
 * ("Each expert applies: Linear(d -> 4d) -> GELU -> Linear(4d -> d)").
 *   x_perm   [rows_cap, d] dtype in; group g owns rows [offsets[g], offsets[g+1])
 *   offsets  [n_groups+1] int32 DEVICE pointer (read on the device; no host sync)
 *   w1       [n_groups, F, d] dtype
 *   h        [rows_cap, F] out: h = GELU(x_perm . W1[g]^T), exact erf form, fp32
 *            accumulation, rounded once -- to fp32 for MOE_F32 layers and to FP16 for
 *            MOE_BF16 layers (11 significant bits instead of bf16's 8, which keeps the
 *            layer output within its error bound; |h| > 65504 is reported as
 *            MOE_ERR_DEVICE by moe_sync_status).
 * MOE_BF16 runs on the tcgen05 tensor cores (TMA-fed, TMEM accumulators); MOE_F32 on
 * the CUDA cores (fp32 products).
 * n_groups = E for the routed experts; n_groups = 1 with offsets {0, T} and x in place
 * of x_perm runs a shared (always-on) expert over all tokens. */
moe_status_t moe_expert_up(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                           int32_t n_groups, int64_t rows_cap, const void* w1, void* h,
                           void* ws, void* stream);

/* Step 3a with the dispatch fused into the expert GEMM's operand load: the packed rows
 * are gathered from the token matrix while each tile is loaded (TMA row gathers), so
 * no x_perm is written or read.  Same result as moe_dispatch's row copy followed by
 * moe_expert_up:
 *   h[r] = GELU(x[src[r] / K] . W1[g]^T)   for r in [offsets[g], offsets[g+1])
 *   x    [T, d] dtype (the layer's input rows; cfg.T rows)
 *   src  [rows_cap] int32 device pointer (4-byte aligned): packed row -> flat assignment
 *        t*K + k, as written by moe_dispatch (which can then run with x = x_perm = NULL)
 *   the other arguments as moe_expert_up.  A src entry naming a token outside [0, T) is
 *   reported as MOE_ERR_DEVICE and gathers row 0 instead. */
moe_status_t moe_expert_up_gather(const moe_config* cfg, const void* x, const int32_t* src,
                                  const int32_t* offsets, int32_t n_groups, int64_t rows_cap,
                                  const void* w1, void* h, void* ws, void* stream);

/* Step 3b -- grouped second expert Linear: y_perm = h . W2[g]^T.
 *   h [rows_cap, F] as written by moe_expert_up (fp32, or fp16 for MOE_BF16 layers);
 *   w2 [n_groups, d, F]: fp32 for MOE_F32 layers; FP16 for MOE_BF16 layers (convert the
 *   bf16 weights once with moe_bf16_to_f16);
 *   y_perm [rows_cap, d] out: fp32 for MOE_F32 layers; FP16 for MOE_BF16 layers (11
 *   significant bits, rounded once from the fp32 accumulator; the combine then sums in
 *   fp32 and rounds the layer output once; |y| > 65504 is reported as MOE_ERR_DEVICE). */
moe_status_t moe_expert_down(const moe_config* cfg, const void* h, const int32_t* offsets,
                             int32_t n_groups, int64_t rows_cap, const void* w2, void* y_perm,
                             void* ws, void* stream);

/* FP8 variant of step 3 for MOE_BF16 layers.  The pages fix no FP8 recipe (they only
 * note that MoE is the most FP8-sensitive architecture); this is the plainest one:
 * E4M3 operands (round to nearest even, saturating at +-448) with one fp32 scale per
 * row of each operand -- per token row of x, per row of h, per output channel of each
 * weight -- and fp32 accumulation on the tensor cores (tcgen05 kind::f8f6f4).  Results
 * differ from the bf16 path by the E4M3 rounding of every operand (about 2^-4 relative
 * per element); the outputs keep the bf16 path's types.
 *
 * moe_quantize_e4m3: codes[r, c] = E4M3(src[r, c] * (448 / amax_r)) and
 *   scales[r] = amax_r / 448 (amax_r = max_c |src[r, c]|; a zero row gives zero codes and
 *   scale 0), each step one correctly rounded fp32 operation.
 *   src [rows, cols] of dtype MOE_F32, MOE_BF16 or MOE_F16 (16-byte aligned), cols a
 *   multiple of 16; codes [rows, cols] bytes (16-byte aligned); scales [rows] fp32.
 *   rows_dev: nullable device int32; when given, only the first min(rows, *rows_dev)
 *   rows are converted (e.g. offsets + E: the packed rows actually kept).
 *   Use it once for the stacked weights (W1 as [E*F, d] rows, W2 as [E*d, F]), and per
 *   step for x ([T, d]) and for h ([rows_cap, F], fp16).
 *
 * moe_expert_up_e4m3: h[r] = GELU(x_scale[a] * w1_scale[g*F + n] * sum_k xq[a,k] w1q[g*F+n,k])
 *   with a = src[r] / K (rows gathered from the quantised token matrix xq [T, d], as in
 *   moe_expert_up_gather) or a = r when src is NULL (xq then holds the packed rows);
 *   h [rows_cap, F] fp16 out.
 * moe_expert_down_e4m3: y_perm[r] = h_scale[r] * w2_scale[g*d + n] * sum_k hq[r,k] w2q[g*d+n,k];
 *   y_perm [rows_cap, d] fp16 out (as moe_expert_down for bf16 layers).
 * Other arguments as moe_expert_up / moe_expert_down.  d and F must be multiples of 16
 * (else MOE_ERR_UNSUPPORTED); MOE_F32 layers return MOE_ERR_UNSUPPORTED. */
moe_status_t moe_quantize_e4m3(const void* src, int32_t dtype, int64_t rows, int32_t cols,
                               const int32_t* rows_dev, void* codes, float* scales, void* stream);
moe_status_t moe_expert_up_e4m3(const moe_config* cfg, const void* xq, const float* x_scale,
                                const int32_t* src, const int32_t* offsets, int32_t n_groups,
                                int64_t rows_cap, const void* w1q, const float* w1_scale, void* h,
                                void* ws, void* stream);
moe_status_t moe_expert_down_e4m3(const moe_config* cfg, const void* hq, const float* h_scale,
                                  const int32_t* offsets, int32_t n_groups, int64_t rows_cap,
                                  const void* w2q, const float* w2_scale, void* y_perm, void* ws,
                                  void* stream);

/* Step 3 -- both expert Linears (moe_expert_up then moe_expert_down). */
moe_status_t moe_grouped_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                             int32_t n_groups, int64_t rows_cap, const void* w1, const void* w2,
                             void* h, void* y_perm, void* ws, void* stream);

/* Step 4 -- combine back to token order ("Y = sum over selected experts of
 * expert_output[token] * routing_weight[token]").  Gather-side, no atomics:
 *   Y[t] = sum_{k ascending, slot[t,k] >= 0} topk_w[t,k] * y_perm[slot[t,k]]
 *          (+ y_shared[t]), accumulated in fp32 and rounded once.
 *   y_perm [rows_cap, d] and y_shared [T, d] (nullable): fp16 for MOE_BF16 layers, fp32
 *   for MOE_F32 layers, as moe_expert_down writes them; slot [T, K], topk_w [T, K];
 *   y [T, d] dtype out.  A dropped assignment contributes exactly 0. */
moe_status_t moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* slot,
                         const float* topk_w, const void* y_shared, void* y, void* stream);

/* Step 5 -- auxiliary load-balancing statistics ("Load Balancing: The Auxiliary Loss"):
 *   f[i] = counts[i] / (T*K)          (pre-drop assignment fraction)
 *   P[i] = mean_t softmax(logits)[t,i] (from the partial sums moe_route left in ws)
 *   l_aux[0] = alpha * sum_i f[i] * P[i]
 * All outputs fp32 device pointers; with T = 0 all are 0.  Must follow the moe_route
 * call that used the same ws. */
moe_status_t moe_aux_stats(const moe_config* cfg, const int32_t* counts, const void* ws,
                           float* f, float* P, float* l_aux, void* stream);

/* Backward of the auxiliary loss (the pages: it "is added to the main task loss and
 * backpropagated"; it does not affect inference).  Writes the gradient of
 * L_aux = alpha * sum_i f_i P_i with respect to the router logits:
 *   grad_logits[t,j] = (alpha / T) * p[t,j] * (f_j - sum_i f_i p[t,i]),
 * p = softmax(logits[t]) recomputed in fp32.  f_i is a count of top-K choices, a step
 * function of the logits whose derivative is zero away from ties, so only P_i carries
 * gradient.  logits [T, E] fp32 (as moe_route wrote them), f [E] fp32 (from
 * moe_aux_stats), grad_logits [T, E] fp32 out; all 4-byte aligned device pointers. */
moe_status_t moe_aux_loss_grad(const moe_config* cfg, const float* logits, const float* f,
                               float* grad_logits, void* stream);

/* Convert n bf16 values to fp16 (n a multiple of 8), e.g. the second expert Linear's
 * weights of a MOE_BF16 layer.  Magnitudes in [2^-17, 65504] convert exactly, smaller
 * ones round at 2^-25; larger ones are reported as MOE_ERR_DEVICE in the status word
 * of `ws` (any workspace of this library). */
moe_status_t moe_bf16_to_f16(const void* src, void* dst, int64_t n, void* ws, void* stream);

/* Synchronise `stream`, then return and clear the device status word in `ws`
 * (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE), or MOE_ERR_CUDA if a kernel failed. */
moe_status_t moe_sync_status(void* ws, void* stream);

/* Which tensor-core kernels run the expert GEMMs of MOE_BF16 layers (moe_expert_up /
 * moe_expert_down).  Not a step of the layer: a process-wide performance setting.
 *   MOE_GEMM_SINGLE one CTA per 128-row tile (tcgen05 cta_group::1);
 *   MOE_GEMM_PAIR   two CTAs per 256-row tile (tcgen05 cta_group::2: one MMA over two
 *                   SMs, each SM loading half of the operands), which pads each group
 *                   to a multiple of 256 rows;
 *   MOE_GEMM_SPLIT  pairs for each group's whole 256-row tiles and, at the same time on
 *                   the other SMs, one CTA per 128-row tile for the remaining rows (the
 *                   second kernel runs on a library-owned stream per device, forked from
 *                   and joined back into the caller's stream with events, which also
 *                   works under stream capture; calls on different streams that use this
 *                   plan share that side stream);
 *   MOE_GEMM_PAIR_T two CTAs per tile computing the transpose: 256 weight rows (output
 *                   columns) on the MMA's M side and up to 256 of a group's rows on its
 *                   N side, sized to the group (rounded up to 32), so no group is padded
 *                   to 256 rows (row-gathered calls take MOE_GEMM_PAIR instead);
 *   MOE_GEMM_MIXED  CTA pairs only, in one launch: each group's whole 256-row tiles as
 *                   for MOE_GEMM_PAIR and its remaining rows (fewer than 256) as one
 *                   transposed tile per 256-wide slab of output columns, as for
 *                   MOE_GEMM_PAIR_T, so no group is padded to 256 rows and every weight
 *                   slab is walked by one kernel (16-bit operands; E4M3 and row-gathered
 *                   calls take MOE_GEMM_SPLIT instead);
 *   MOE_GEMM_AUTO   (default) pairs when the 256-row padding is at most 5% of the rows
 *                   (judged from the capacity), the split when the capacity reaches 256
 *                   rows, transposed pairs when the groups have no capacity bound, one
 *                   CTA otherwise (all pair plans need the output width to be a
 *                   multiple of 256).  The E4M3 calls take the same plans with E4M3
 *                   operands, except that AUTO keeps them on one CTA where it would pick
 *                   pairs for groups under 512 rows or transposed pairs.
 * Every choice sums the same products in the same order, so results are identical.
 * Returns MOE_ERR_INVALID for any other value.  Calls already enqueued are unaffected. */
typedef enum {
  MOE_GEMM_AUTO = 0,
  MOE_GEMM_SINGLE = 1,
  MOE_GEMM_PAIR = 2,
  MOE_GEMM_SPLIT = 3,
  MOE_GEMM_PAIR_T = 4,
  MOE_GEMM_MIXED = 5
} moe_gemm_pairing_t;
moe_status_t moe_set_gemm_pairing(int32_t mode);

/* SM budget of the persistent tensor-core expert GEMMs (moe_expert_up, _gather, _down and
 * their E4M3 forms), process-wide: n = 0 (default) all SMs; n >= 2 at most n SMs (capped
 * at the device's count), so that a GEMM on another stream can run beside them on the
 * rest -- e.g. a shared expert on a few SMs next to the routed experts, which are bound by
 * their weight stream from HBM.  The setting is read when a call is made; calls already
 * enqueued keep theirs.  Results do not depend on it.  Returns MOE_ERR_INVALID for n < 0
 * or n = 1. */
moe_status_t moe_set_gemm_sms(int32_t n);

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status_t status);

/* Number of kernels this library has launched in this process (host-side counter). */
uint64_t moe_launch_count(void);

/* Test hook for the bounded wait of the dispatch scan.  When skip_block >= 0, the next
 * moe_dispatch or moe_dispatch_noalloc call makes block `skip_block` of
 * its look-back withhold its published counts, so its
 * successor's wait runs out after `spin_limit` polls and records MOE_ERR_TIMEOUT in
 * the device status word; every block still terminates.  Results of that call are
 * invalid.  The hook disarms itself after one call; skip_block < 0 disarms it. */
void moe_test_arm_scan_timeout(int32_t skip_block, int32_t spin_limit);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
