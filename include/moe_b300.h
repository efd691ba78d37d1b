/*
 * moe_b300.h -- C ABI of the B300 (sm_103a) sparse Mixture-of-Experts layer
 * forward pass.
 *
 * The layer, step by step (pages cited by title and section):
 *   1. router logits      H = x W_g + b_g + eps * softplus(x W_noise)
 *                         ("LLM part 09: Sparse Mixture-of-Experts (MoE)",
 *                         s2 noisy top-k gating; "Mixture-of-Experts Sparse
 *                         Model Scaling", Mathematical Formulation)
 *   2. top-k + gates      idx = k largest H (ties -> lower expert index),
 *                         w = softmax over the k selected logits
 *                         (same s2; "Mixture-of-experts Models", Level 2
 *                         "Router scores become a sparse dispatch decision")
 *   3. dispatch           capacity C = ceil(cf*T*k/E) ("3D mixture-of-experts
 *                         routing lab", Capacity card); first-come slots in
 *                         rank-major priority order (every token's first
 *                         choice before any second choice, tokens in order);
 *                         over-capacity assignments dropped
 *                         ("Mixture-of-Experts Sparse Model Scaling", Lab 3
 *                         and Advanced Theory; "Mixture-of-experts Models",
 *                         "Capacity limits make dispatch observable")
 *   4. experts            GELU:   y = gelu(x W1^T + b1) W2^T + b2
 *                         SwiGLU: y = (silu(x W1^T) * (x W3^T)) W2^T + b2
 *   5. combine            out[t] = residual[t] + sum_{kept r} w[t,r] y_{t,r}
 *                         ("LLM part 09", s1 y = sum_i G(x)_i E_i(x); s3:
 *                         a dropped assignment bypasses its expert and the
 *                         residual carries the token)
 *                         (+ the shared experts' output on every token, when
 *                         the layer has shared experts; see moe_shared_t)
 *
 * Conventions for every entry point
 *   - All tensor arguments are DEVICE pointers of the current CUDA device,
 *     row-major, densely packed, owned by the caller.  The library never
 *     allocates, frees, or synchronises (except moe_get_device_error) and
 *     keeps no per-call state outside the caller's workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *     All work is enqueued on it; every call returns before the GPU is done.
 *   - Argument errors are detected on the host, before anything is enqueued,
 *     and returned as MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *     MOE_ERR_WORKSPACE.  A CUDA runtime failure returns MOE_ERR_CUDA.
 *     Errors found on the device (a bounded wait that gave up, an index out
 *     of range) are recorded in the workspace's error word and read back
 *     with moe_get_device_error(); kernels never trap or abort.
 *   - dtype MOE_F32: x, expert weights, out are fp32 (CUDA-core path,
 *     intended for small layers).  MOE_BF16: x, W1, W3, W2, out are bf16,
 *     expert GEMMs run on the tcgen05 tensor cores with fp32 accumulation;
 *     needs d and d_ff multiples of 64.  Router tensors (W_g, b_g, W_noise,
 *     eps), gates, expert biases and the per-assignment expert outputs are
 *     fp32 for both dtypes.
 *   - Limits: 1 <= E <= 128, 1 <= k <= min(E, 16), 1 <= d, d_ff,
 *     0 <= T < 2^31 / k.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null pointer, bad size, k > E, ...          */
  MOE_ERR_UNSUPPORTED = 2,    /* valid but outside the supported set         */
  MOE_ERR_WORKSPACE = 3,      /* workspace null, misaligned or too small     */
  MOE_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed           */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait gave up          */
  MOE_ERR_BOUNDS = 6          /* a device-side index check failed            */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;
typedef enum { MOE_ACT_GELU = 0, MOE_ACT_SWIGLU = 1 } moe_act_t;
/* Token choice: each token takes its top-k experts (steps 2-3 above).
 * Expert choice: each expert takes its min(C, T) highest-scoring tokens
 * ("Mixture-of-Experts Sparse Model Scaling", Advanced Theory &
 * Extensions); see moe_route_expert_choice. */
typedef enum { MOE_ROUTE_TOKEN_CHOICE = 0, MOE_ROUTE_EXPERT_CHOICE = 1 } moe_routing_t;
/* Gates of the selected experts (token choice): renormalised over the k
 * selected (the default), or the raw routing probabilities p_i, the full
 * softmax over all E ("Mixture-of-Experts Sparse Model Scaling",
 * Mathematical Formulation, the displayed top-k output). */
typedef enum { MOE_GATES_RENORM = 0, MOE_GATES_RAW = 1 } moe_gates_t;
/* An assignment over capacity (token choice): dropped (the default), or
 * re-routed to the token's backup expert, its (k+1)-th ranked one, when that
 * expert has room ("Mixture-of-experts Models", Level 2, "Capacity limits
 * make dispatch observable" and "Overflow handling defines an output
 * contract").  Only the token's first dropped assignment asks for the
 * backup; requests are served after the capacity dispatch, first-come in the
 * same priority order (rank, then token); a re-routed assignment keeps its
 * gate.  Available through moe_forward. */
typedef enum { MOE_OVERFLOW_DROP = 0, MOE_OVERFLOW_REROUTE = 1 } moe_overflow_t;

/* Shape of one layer call.  T tokens of width d, E experts of hidden width
 * d_ff, top-k routing.  dtype is a moe_dtype_t, act a moe_act_t.
 * d_ff_shared is the hidden width of the shared experts (0 = none; bf16
 * needs a multiple of 64).  routing is a moe_routing_t; with expert choice
 * k is the average number of experts per token (it sets the capacity) and
 * T*E < 2^31.  gates (moe_gates_t) and overflow (moe_overflow_t) apply to
 * token choice; with expert choice both must be 0 (its gates are the
 * routing probabilities by definition and nothing overflows). */
typedef struct {
  int64_t T;
  int32_t d;
  int32_t E;
  int32_t k;
  int32_t d_ff;
  int32_t dtype;
  int32_t act;
  int32_t d_ff_shared;
  int32_t routing;
  int32_t gates;
  int32_t overflow;
} moe_shape_t;

/* Shared experts ("Mixture-of-Experts Sparse Model Scaling", Advanced Theory
 * & Extensions: dedicated shared experts that every token passes through
 * unconditionally, next to the fine-grained routed ones; Real-World
 * Applications: DeepSeek-MoE).  They have the routed experts' form (act of
 * the shape) and enter the combine with weight 1.  S shared experts of width
 * F_s are given as ONE FFN of width d_ff_shared = S*F_s: W1s and W3s stack
 * the experts' rows, W2s stacks their columns, b1s concatenates, b2s is the
 * sum of the experts' b2 (the same function, evaluated as one GEMM pair).
 *   W1s [d_ff_shared,d] dtype           gate (SwiGLU) / up (GELU) projection
 *   W3s [d_ff_shared,d] dtype | NULL    SwiGLU up projection (NULL for GELU)
 *   W2s [d,d_ff_shared] dtype           down projection
 *   b1s [d_ff_shared] fp32 | NULL       GELU only
 *   b2s [d] fp32 | NULL */
typedef struct {
  const void* W1s;
  const void* W3s;
  const void* W2s;
  const float* b1s;
  const float* b2s;
} moe_shared_t;

/* Expert capacity C = ceil(capacity_factor * T * k / E), evaluated in double
 * in that order ("3D mixture-of-experts routing lab", Capacity card; the
 * k = 1 form is "LLM part 09", s3).  Returns -1 for T < 0, k < 1, E < 1 or a
 * capacity factor that is not finite and positive, or a result that does
 * not fit in int32. */
MOE_API int32_t moe_capacity(int64_t T, int32_t k, int32_t E, double capacity_factor);

/* Rows of the expert-grouped buffers for capacity C: min(T*k, E*C) with
 * token choice, E*min(C, T) with expert choice. */
MOE_API int64_t moe_max_rows(const moe_shape_t* shape, int32_t C);

/* Workspace bytes that moe_forward needs for this shape and capacity (it
 * also covers moe_dispatch and moe_expert_ffn).  The workspace is a device
 * buffer of at least this many bytes, 256-byte aligned, ZERO-FILLED ONCE
 * after allocation; the library keeps its control words consistent after
 * that.  Returns MOE_ERR_INVALID_ARG for a bad shape or C < 0. */
MOE_API moe_status_t moe_workspace_size(const moe_shape_t* shape, int32_t C, size_t* bytes);

/* Step 1+2: router logits, top-k and gates, for every token.
 *   x        [T,d]  dtype        tokens
 *   W_g      [d,E]  fp32         router weight
 *   b_g      [E]    fp32 | NULL  router bias (NULL = none)
 *   W_noise  [d,E]  fp32 | NULL  noise projection; with eps, adds
 *   eps      [T,E]  fp32 | NULL  eps * softplus(x W_noise) to the logits
 *   idx      [T,k]  int32 out    selected experts, largest logit first
 *   w        [T,k]  fp32  out    gates (softmax over the selected logits;
 *                                 with shape->gates = MOE_GATES_RAW the
 *                                 full-softmax probabilities p_i)
 *   logits   [T,E]  fp32 | NULL  out: the (noisy) logits, computed in fp32
 *   stats    [2]    int64 | NULL out, ADDED to: [0] tokens whose selection
 *                   was settled by the fp64 re-evaluation, [1] tokens whose
 *                   k-th and (k+1)-th fp32 logits differ by < 1e-4
 * Selection is exact: logits are computed in fp32 together with a rigorous
 * error bound; a token whose order is not settled by the bound has its
 * candidate logits re-evaluated in fp64, so idx equals the top-k of the
 * exactly computed logits (up to fp64 rounding).  W_noise and eps must be
 * both NULL or both set. */
MOE_API moe_status_t moe_route(const moe_shape_t* shape, const void* x, const float* W_g,
                       const float* b_g, const float* W_noise, const float* eps,
                       int32_t* idx, float* w, float* logits, int64_t* stats,
                       void* stream);

/* Expert-choice routing (shape->routing == MOE_ROUTE_EXPERT_CHOICE), in
 * place of steps 2-3: expert e takes the C' = min(C, T) tokens with the
 * largest router score H[t,e] (ties -> lower token index); the gate of a
 * chosen (t, e) is the router probability p[t,e] = softmax over all E of
 * H[t] (not renormalised).  A token may be chosen by no expert (the residual
 * carries it) or by several ("Mixture-of-Experts Sparse Model Scaling",
 * Advanced Theory & Extensions).
 *   C          capacity (moe_capacity with the shape's k, or any C >= 0)
 *   x, W_g, b_g, W_noise, eps   as in moe_route
 *   sel      [E,C'] int32 out   chosen tokens of each expert, ascending
 *   gates    [E,C'] fp32 out    p[t,e] of those pairs
 *   logits   [T,E] fp32 | NULL  out: the router logits
 *   dropped  [1] int64 | NULL   out: tokens no expert chose
 *   ws, ws_bytes  workspace of moe_workspace_size(shape, C)
 * Selection is exact: the router bounds every fp32 logit's rounding error;
 * tokens whose order against the C'-th score is not settled by the bounds
 * are re-scored in fp64, so sel equals the top-C' sets of the exactly
 * computed scores (up to fp64 rounding). */
MOE_API moe_status_t moe_route_expert_choice(const moe_shape_t* shape, int32_t C, const void* x,
                                             const float* W_g, const float* b_g, const float* W_noise,
                                             const float* eps, int32_t* sel, float* gates, float* logits,
                                             int64_t* dropped, void* ws, size_t ws_bytes, void* stream);

/* Step 3: capacity-limited dispatch and the gather into expert order.
 *   C         capacity (moe_capacity, or any C >= 0)
 *   idx       [T,k]  int32        from moe_route (values in [0,E))
 *   x         [T,d]  dtype        tokens
 *   pos       [T,k]  int32 out    slot of (t,r) inside expert idx[t,r]'s
 *                                 segment, -1 if the assignment was dropped
 *   counts    [E]    int32 out    kept assignments per expert, min(load, C)
 *   offsets   [E+1]  int32 out    exclusive prefix sum of counts
 *   dropped   [1]    int64 out    sum_e max(0, load_e - C)
 *   x_perm    [moe_max_rows,d] dtype out   row offsets[e]+pos[t,r] = x[t]
 *   row_token [moe_max_rows] int32 | NULL  out: token of each row
 *   ws, ws_bytes  workspace (moe_workspace_size)
 * x and x_perm must be 16-byte aligned (else MOE_ERR_UNSUPPORTED).
 * Results are deterministic (no atomics decide any slot).  An expert id
 * outside [0,E) sets MOE_ERR_BOUNDS in the error word; that assignment gets
 * pos = -1 and is counted in no load. */
MOE_API moe_status_t moe_dispatch(const moe_shape_t* shape, int32_t C, const int32_t* idx,
                          const void* x, int32_t* pos, int32_t* counts, int32_t* offsets,
                          int64_t* dropped, void* x_perm, int32_t* row_token,
                          void* ws, size_t ws_bytes, void* stream);

/* moe_dispatch for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a library-integration entry point, not a step
 * of the method.  Some callers cannot allocate a workspace: a plug-in whose
 * host framework owns all device memory and passes it only the operation's
 * inputs and outputs, or a serving loop whose device memory plan is fixed up
 * front and where cudaMalloc (which may synchronise the device) is not
 * allowed.  This call computes exactly what moe_dispatch computes (same
 * arguments and outputs, minus the workspace) and keeps its scan state in
 * a fixed array in the library's own device global memory instead.
 *   error_out  [1] int32 | NULL  device output: set to 0 at the start of the
 *                                call, then to the first device-side error of
 *                                the call (MOE_ERR_BOUNDS / _DEVICE_TIMEOUT)
 * Limits: T*k <= 1048576 assignments (and E <= 128); larger sizes return
 * MOE_ERR_UNSUPPORTED before anything is enqueued.  The array (about
 * 257 KiB) stays resident on every GPU that loads the library until the
 * process exits.  It allocates nothing: no cudaMalloc, cudaFree or
 * allocating library call.  It accepts exactly the shapes moe_dispatch
 * accepts, and like moe_dispatch returns MOE_ERR_UNSUPPORTED for an x or
 * x_perm that is not 16-byte aligned.  The first call in each CUDA context,
 * with that context current, looks up the array's device address
 * (cudaGetSymbolAddress) and caches it under the context's process-unique
 * id, so a context that is destroyed and recreated (cudaDeviceReset) gets a
 * fresh lookup; make that first call before any stream capture.  All calls
 * share the one array and each call clears the parts that must start at
 * zero: calls whose kernels may overlap on the GPU (unordered streams,
 * several host threads) race on it and must be serialised by the caller. */
MOE_API moe_status_t moe_dispatch_noalloc(const moe_shape_t* shape, int32_t C, const int32_t* idx,
                                          const void* x, int32_t* pos, int32_t* counts, int32_t* offsets,
                                          int64_t* dropped, void* x_perm, int32_t* row_token,
                                          int32_t* error_out, void* stream);

/* Step 4: every expert's FFN over its segment of the expert-grouped rows.
 *   x_perm   [moe_max_rows,d]  dtype   grouped rows (moe_dispatch)
 *   offsets  [E+1] int32               segment starts (moe_dispatch)
 *   W1       [E,d_ff,d] dtype          up projection (GELU) / gate (SwiGLU)
 *   W3       [E,d_ff,d] dtype | NULL   SwiGLU up projection (NULL for GELU)
 *   W2       [E,d,d_ff] dtype          down projection
 *   b1       [E,d_ff] fp32 | NULL      GELU only (must be NULL for SwiGLU)
 *   b2       [E,d]    fp32 | NULL
 *   y_perm   [moe_max_rows,d] fp32 out expert output of each grouped row;
 *                                      rows past offsets[E] are untouched
 *   ws, ws_bytes  workspace (holds the [moe_max_rows,d_ff] hidden activations)
 * bf16: the hidden activation is rounded to bf16 between the two GEMMs. */
MOE_API moe_status_t moe_expert_ffn(const moe_shape_t* shape, int32_t C, const void* x_perm,
                            const int32_t* offsets, const void* W1, const void* W3,
                            const void* W2, const float* b1, const float* b2,
                            float* y_perm, void* ws, size_t ws_bytes, void* stream);

/* The shared experts (see moe_shared_t) on every token: one dense FFN.
 *   x         [T,d] dtype        tokens
 *   shared    weights; required when shape->d_ff_shared > 0
 *   y_shared  [T,d] fp32 out     the shared experts' summed output
 *   ws, ws_bytes  a workspace of moe_workspace_size(shape, C) for any C
 *                 (holds the [T,d_ff_shared] hidden activation)
 * bf16: tcgen05 GEMMs with fp32 accumulation, the hidden activation rounded
 * to bf16 between them, as for the routed experts.  shape->d_ff_shared == 0
 * returns MOE_ERR_INVALID_ARG. */
MOE_API moe_status_t moe_shared_ffn(const moe_shape_t* shape, const void* x, const moe_shared_t* shared,
                                    float* y_shared, void* ws, size_t ws_bytes, void* stream);

/* Step 5: weighted combine into the residual, one token at a time, ranks
 * summed in order 0..k-1 (deterministic), then the shared experts' output.
 *   y_perm   [moe_max_rows,d] fp32   expert outputs (moe_expert_ffn)
 *   idx, w, pos [T,k], offsets [E+1]  as produced above
 *   residual [T,d] dtype | NULL       NULL = zero residual
 *   y_shared [T,d] fp32 | NULL        shared experts' output (moe_shared_ffn),
 *                                     added with weight 1; NULL = none
 *   out      [T,d] dtype out          residual + moe
 *   moe_out  [T,d] fp32 | NULL out    everything the experts add (routed
 *                                     sum + shared output), alone */
MOE_API moe_status_t moe_combine(const moe_shape_t* shape, int32_t C, const float* y_perm,
                         const int32_t* idx, const float* w, const int32_t* pos,
                         const int32_t* offsets, const void* residual, const float* y_shared,
                         void* out, float* moe_out, void* stream);

/* The whole layer: steps 1-5 on one stream, residual = x.
 *   capacity_factor  used when C_override < 0; else C = C_override
 *   x, W_g, b_g, W_noise, eps, W1, W3, W2, b1, b2   as above
 *   shared  moe_shared_t* | NULL: the shared experts' weights, required iff
 *           shape->d_ff_shared > 0; their FFN runs first (on every token)
 *           and its output is added in the combine
 * Routing is as in moe_route.  For long bf16 batches (T >= 16384) whose
 * logit table has 32..256 columns (E, or 2E with noise), when no logits
 * output is asked for and the gates are renormalised, the router first
 * filters the experts with a tensor-core pass (weights split into two bf16
 * parts, fp32 accumulation) and a margin of 2^-10 ||x|| ||w_col||, then
 * ranks the remaining candidates exactly as moe_route does; the margin
 * assumes the tensor core's fp32 accumulation of exact bf16 products loses
 * fewer than about ten of fp32's 24 bits per step.
 * Decode-sized bf16 batches (T <= 128 with T*k >= 4E, d and d_ff multiples
 * of 64) run both expert GEMMs and the combine in one kernel.
 * - Self-routing: when the overflow policy is drop and the logit table has a
 *   power-of-two number of columns from 4 to 256, that kernel also routes
 *   and dispatches the batch, so the whole layer is one launch.
 * - Same results: its top-k, slots and drops are exactly moe_route's and
 *   moe_dispatch's.
 * - Rounding: its fp32 logits are summed in another order, so logits and w
 *   may differ from moe_route's in the last bits (within the same rigorous
 *   bound).
 * With overflow re-routing (shape->overflow) idx holds, for each
 * assignment, the expert it was finally sent to (the backup for a re-routed
 * one), pos its slot there, dropped the assignments left without an expert.
 * With expert-choice routing (shape->routing) the token-choice tables idx,
 * w, pos must be NULL and stats is untouched; counts (= C' each), offsets
 * (e*C') and dropped (tokens no expert chose) are written when given, and
 * out[t] = x[t] + sum over the experts e that chose t, in order e = 0..E-1,
 * of p[t,e] * E_e(x_t) (+ the shared experts).
 *   out [T,d] dtype out; moe_out [T,d] fp32 | NULL out
 *   idx, w, pos [T,k], counts [E], offsets [E+1], dropped [1], stats [2]:
 *     optional outputs (NULL = keep them in the workspace only; stats as
 *     in moe_route, added to)
 *   logits [T,E] fp32 | NULL  optional output: the router's (noisy) logits,
 *     as in moe_route; with idx, counts and dropped it feeds
 *     moe_routing_stats
 *   ws, ws_bytes  workspace of moe_workspace_size(shape, C) bytes */
MOE_API moe_status_t moe_forward(const moe_shape_t* shape, double capacity_factor, int32_t C_override,
                         const void* x, const float* W_g, const float* b_g,
                         const float* W_noise, const float* eps, const void* W1,
                         const void* W3, const void* W2, const float* b1, const float* b2,
                         const moe_shared_t* shared, void* out, float* moe_out, int32_t* idx,
                         float* w, int32_t* pos, int32_t* counts, int32_t* offsets, int64_t* dropped,
                         int64_t* stats, float* logits, void* ws, size_t ws_bytes, void* stream);

/* moe_forward, recording up to six CUDA events (cudaEvent_t, created by the
 * caller) on `stream` at the stage boundaries, so each stage can be timed
 * with cudaEventElapsedTime:
 *   stage_events[0] before the layer's first kernel (the shared experts'
 *   FFN when there is one, else the router)  [1] after the router
 *   [2] after dispatch + gather              [3] after the first expert GEMM
 *   [4] after the second expert GEMM         [5] after the combine
 * A NULL entry records nothing at that boundary.  The layer's kernels are
 * launched with programmatic dependent launch, so a kernel may start its
 * prologue while its predecessor finishes; an event between two kernels
 * orders them fully.  While `stream` is being captured into a CUDA graph the
 * events are recorded as external event nodes (they time every launch of
 * the graph).  MOE_ERR_INVALID_ARG if stage_events is NULL. */
MOE_API moe_status_t moe_forward_timed(const moe_shape_t* shape, double capacity_factor, int32_t C_override,
                                       const void* x, const float* W_g, const float* b_g,
                                       const float* W_noise, const float* eps, const void* W1,
                                       const void* W3, const void* W2, const float* b1, const float* b2,
                                       const moe_shared_t* shared, void* out, float* moe_out, int32_t* idx,
                                       float* w, int32_t* pos, int32_t* counts, int32_t* offsets,
                                       int64_t* dropped, int64_t* stats, float* logits, void* ws,
                                       size_t ws_bytes, void* stream,
                                       void* const* stage_events);

/* Routing diagnostics of one batch and the auxiliary load-balancing loss
 * ("Mixture-of-Experts Sparse Model Scaling", Mathematical Formulation and
 * Lab 2: L_aux = E * sum_e f_e P_e, uniform routing gives 1; "LLM part 09",
 * s4; "Mixture-of-experts Models", Level 3 wants the probability mass,
 * the realised loads, overflow and utilisation side by side).
 *   logits   [T,E] fp32       router logits (moe_route / moe_forward output)
 *   idx      [T,k] int32      selected experts
 *   counts   [E]   int32      kept assignments per expert (after capacity)
 *   dropped  [1]   int64      assignments over capacity
 *   f        [E]   fp64 out   routed (pre-capacity) load of e over T*k
 *   P        [E]   fp64 out   mean over tokens of softmax(logits[t])[e]
 *   summary  [6]   fp64 out   [0] aux loss E * sum_e f_e P_e
 *                             [1] mean router entropy -sum_e p ln p (nats)
 *                             [2] routed-load imbalance: population std /
 *                                 mean of the pre-capacity loads
 *                             [3] the same for the kept counts
 *                             [4] utilisation: fraction of experts with a
 *                                 kept assignment
 *                             [5] overflow: dropped / (T*k)
 *   ws, ws_bytes  the workspace of moe_workspace_size(shape, C) for any C
 * T = 0 gives all zeros.  One kernel; the softmax is taken in fp32 and the
 * sums are exact fixed-point integer sums (each probability rounded to a
 * multiple of 2^-(62 - bits(T))), so results are deterministic.  An expert id
 * outside [0,E) is counted nowhere and sets MOE_ERR_BOUNDS in the error
 * word.  Calls that share a workspace must be ordered on one stream. */
MOE_API moe_status_t moe_routing_stats(const moe_shape_t* shape, const float* logits, const int32_t* idx,
                                       const int32_t* counts, const int64_t* dropped, double* f, double* P,
                                       double* summary, void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, reads the workspace's device error word, clears it,
 * and returns it as a status (MOE_OK when no device-side error was recorded
 * since the last read).  `ws` is the workspace passed to the calls. */
MOE_API moe_status_t moe_get_device_error(void* ws, void* stream);

/* Number of kernels the library has enqueued since it was loaded (every
 * entry point, all threads).  Work that a CUDA graph replays is not
 * enqueued again: count one captured call to know a graph's kernels. */
MOE_API unsigned long long moe_kernel_launches(void);

/* Static, human-readable name of a status code. */
MOE_API const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
