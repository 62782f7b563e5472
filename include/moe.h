/*
 * moe.h — C ABI of the B300 (sm_103a) DeepSeekMoE layer forward and backward.
 *
 * The layer computed here (page "02 · 细粒度 MoE：从 Mixtral 到 DeepSeekMoE",
 * llm-infra-atlas, §3.1 Eq. 9–11; DeepSeek-V3 form Eq. 12–15):
 *
 *   h_t = Σ_{j<Ks} FFN_j^shared(u_t) + Σ_{i routed} g_{i,t} · FFN_i(u_t) + u_t
 *
 * with fine-grained segmentation (§2.1: mN experts of width M/m, mK active)
 * and shared-expert isolation (§3.1: Ks always-on experts, routed top-k is
 * mK − Ks).  Two gates are supported:
 *   MOE_GATE_SOFTMAX       s = softmax over the routed logits, g = s for the
 *                          chosen experts, not renormalised (§2.1 Eq. 6–8);
 *   MOE_GATE_SIGMOID_BIAS  s = sigmoid(logit); the choice is taken on s + b_i
 *                          (b_i used for the choice only, page "MoE 的分水岭",
 *                          ibossgateway ch. 7 §7.4); g = s / Σ_chosen s
 *                          (§3.1 Eq. 12–15).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, except the
 *    host token buffers of moe_layer_forward_host and
 *    moe_layer_forward_host_stream.  The library allocates
 *    nothing: scratch comes from the caller through `ws`/`ws_bytes`, sized by
 *    the matching *_workspace_size function, 256-byte aligned.
 *  - Layouts are dense row-major.  Weights follow the nn.Linear convention
 *    (output rows, contracted dimension contiguous):
 *      centroids [E, H];  w1, w3 [E, I, H];  w2 [E, H, I];
 *      sw1, sw3 [Ks, I, H];  sw2 [Ks, H, I];  w3 / sw3 are NULL for ReLU.
 *    Tokens u and outputs h are [T, H].  Element type of u, weights,
 *    centroids, permuted rows and h is shape->dtype (fp32 or bf16); logits,
 *    gate weights, biases and offsets are always fp32; indices are int32.
 *  - Every call enqueues work on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and returns without synchronising.  Arguments are
 *    checked on the host before anything is launched; a failed check
 *    launches nothing.  Errors are returned, never thrown.  The device-side
 *    calls (all but the two host-buffer forwards and moe_device_status) can be
 *    captured into a CUDA graph on a capturing stream once each has run
 *    outside a capture (the first call on a device sets the kernels'
 *    shared-memory limits); a replay repeats the call on the same buffers.
 *  - The expert routing never drops a token (no capacity factor; the
 *    page's §4 states that DeepSeekMoE drops none).
 *
 * Limits: 1 ≤ n_routed + n_shared ≤ 1024; 0 ≤ top_k ≤ min(32, n_routed);
 * H % 8 == 0 and inter % 8 == 0.  bf16 additionally needs H % 128 == 0 and
 * inter % 64 (SwiGLU) or inter % 128 (ReLU) == 0, and for SwiGLU the gate
 * and up stacks (w1 and w3, sw1 and sw3) must start at different addresses
 * less than 2^40 bytes apart (the kernel reads them through one tensor map
 * that steps from one to the other); otherwise MOE_ERR_UNSUPPORTED.
 * Group-limited routing needs 1 <= n_groups <= 32, n_routed % n_groups == 0,
 * 1 <= topk_groups <= n_groups and topk_groups * (n_routed / n_groups) >=
 * top_k (else MOE_ERR_INVALID_ARG; n_groups > 32: MOE_ERR_UNSUPPORTED).
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_API __attribute__((visibility("default")))

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* NULL where a pointer is required, bad sizes/enums, misalignment */
  MOE_ERR_UNSUPPORTED = 2, /* valid layer, but outside this build's kernel limits (see above) */
  MOE_ERR_WORKSPACE = 3,   /* ws NULL or ws_bytes below the *_workspace_size value */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call failed; see moe_last_cuda_error() */
  MOE_ERR_TIMEOUT = 5      /* a kernel's bounded wait expired (reported by moe_device_status) */
} moe_status;

typedef enum { MOE_GATE_SOFTMAX = 0, MOE_GATE_SIGMOID_BIAS = 1 } moe_gate;
typedef enum { MOE_ACT_RELU = 0, MOE_ACT_SWIGLU = 1 } moe_act;
typedef enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 } moe_dtype;

/* One layer's shape.  T tokens of hidden size H; n_routed routed experts of
 * which top_k are chosen per token; n_shared always-on experts; every expert
 * has intermediate width `inter` (M/m in the segmentation notation).
 * n_groups > 0 makes the routing group-limited (page "02 · 细粒度 MoE", §4,
 * node-limited routing): the routed experts form n_groups groups of
 * n_routed / n_groups consecutive experts, each token keeps the topk_groups
 * groups with the largest sum of its experts' scores (softmax scores, or
 * s + b with MOE_GATE_SIGMOID_BIAS), ties to the lower group index, and
 * chooses its top_k experts among those groups only.  n_groups = 0 (and
 * topk_groups = 0): no limit. */
typedef struct {
  int32_t T, H, n_routed, n_shared, top_k, inter;
  int32_t gate;  /* moe_gate */
  int32_t act;   /* moe_act */
  int32_t dtype; /* moe_dtype */
  int32_t n_groups, topk_groups;
} moe_shape;

/* Layer parameters (device pointers).  logit_offset [E] (may be NULL) is
 * added to the logit before scoring and so changes choice and weight alike;
 * select_bias [E] (may be NULL; ignored by the softmax gate) changes only the
 * choice. */
typedef struct {
  const void* centroids;
  const float* logit_offset;
  const float* select_bias;
  const void *w1, *w3, *w2;
  const void *sw1, *sw3, *sw2;
} moe_weights;

/* Optional routing outputs of moe_layer_forward (each may be NULL). */
typedef struct {
  float* logits;           /* [T, E] */
  int32_t* topk_idx;       /* [T, top_k] */
  float* topk_w;           /* [T, top_k] */
  int32_t* expert_offsets; /* [E + 1] */
} moe_route_outputs;

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(int status);

/* cudaError_t of the most recent MOE_ERR_CUDA returned on this host thread
 * (0 if none). */
MOE_API int moe_last_cuda_error(void);

/* Synchronises `stream`, then reads and clears this device's error word,
 * which kernels set instead of trapping or hanging: bit 1, 2 or 4 when a
 * bounded wait of the grouped GEMM's producer, MMA or epilogue role
 * expires, 8 for an expert index out of range, 16 for a grouped-GEMM launch
 * with less dynamic shared memory than its layout (it then does nothing).
 * *code receives the raw word (0 = clean).  Returns MOE_ERR_TIMEOUT if the
 * word was set, MOE_ERR_CUDA if the synchronisation failed, else MOE_OK. */
MOE_API moe_status moe_device_status(moe_stream_t stream, int32_t* code);

/* Self-test of failure detection: launches one thread that waits, with the
 * same bounded barrier wait the grouped GEMM's roles use but a limit of
 * limit_us microseconds (1..1000000), on a barrier phase that nothing
 * completes.  The wait expires, the kernel sets the timeout bit of this
 * device's error word and returns, so the next moe_device_status reports
 * MOE_ERR_TIMEOUT and the context stays usable.  No GPU fault, trap or hang
 * is involved. */
MOE_API moe_status moe_check_bounded_wait(uint32_t limit_us, moe_stream_t stream);

/* Scratch sizes in bytes (0 is a valid answer; an invalid shape returns 0). */
MOE_API size_t moe_dispatch_workspace_size(const moe_shape* shape);
MOE_API size_t moe_expert_ffn_workspace_size(const moe_shape* shape);
MOE_API size_t moe_layer_workspace_size(const moe_shape* shape);
MOE_API size_t moe_router_logits_workspace_size(const moe_shape* shape);

/* Router logits z[t, i] = u_tᵀ e_i (+ logit_offset[i]), fp32 accumulation
 * (page "02 · 细粒度 MoE", §2.1 Eq. 8: the score is a function of u_tᵀ e_i).
 * u [T, H], centroids [E, H] in shape->dtype; logits [T, E] fp32 out.
 * ws: NULL, or moe_router_logits_workspace_size(shape) bytes (16-byte
 * aligned; fewer give MOE_ERR_WORKSPACE).  With it, a bf16 batch with few
 * 128-expert x 64-token tiles (decode-sized) has its contraction over H cut
 * into ranges whose partial logits land in ws and are added in range order,
 * then the offset; without it (or when the size is 0) the contraction runs
 * whole.  Each way gives the same logits on every run; the two differ only
 * by fp32 rounding. */
MOE_API moe_status moe_router_logits(const moe_shape* shape, const void* u,
                                     const void* centroids,
                                     const float* logit_offset, float* logits, void* ws,
                                     size_t ws_bytes, moe_stream_t stream);

/* Scores, top-k choice and gate weights per token from fp32 logits
 * (§2.1 Eq. 6–8 for softmax; §3.1 Eq. 12–15 and ch. 7 §7.4 for sigmoid+bias).
 * The choice is ordered by descending key, ties to the lower expert index;
 * the softmax key is the logit itself (softmax is increasing in it), the
 * sigmoid key is fp32(sigmoid(z)) + b_i.  topk_idx [T, top_k] int32 and
 * topk_w [T, top_k] fp32 out; kth_gap [T] (may be NULL) receives the k-th
 * minus the (k+1)-th largest score (softmax) or key (sigmoid+bias), +inf if
 * top_k == E.  select_bias may be NULL. */
MOE_API moe_status moe_route(const moe_shape* shape, const float* logits,
                             const float* select_bias, int32_t* topk_idx,
                             float* topk_w, float* kth_gap,
                             moe_stream_t stream);

/* Groups token rows by expert (no dropping).  expert_offsets [E + 1] out
 * (exclusive prefix sum of per-expert counts); permuted rows are sorted by
 * expert, then token; row_token [T·k] out (token of each permuted row);
 * slot_row [T·k] out (row of token t's slot s at t·k + s); u_perm [T·k, H]
 * out, u_perm[r] = u[row_token[r]].  Deterministic (no order-dependent
 * atomics).  An expert index outside [0, E) sets the device error word and
 * that entry is skipped.  ws: moe_dispatch_workspace_size bytes. */
MOE_API moe_status moe_dispatch(const moe_shape* shape, const int32_t* topk_idx,
                                const void* u, int32_t* expert_offsets,
                                int32_t* row_token, int32_t* slot_row,
                                void* u_perm, void* ws, size_t ws_bytes,
                                moe_stream_t stream);

/* Expert FFNs over routed and shared experts (page "19-deepseek-moe",
 * ai.tomabc.com: an expert is ReLU(x W1ᵀ) W2ᵀ without biases; SwiGLU form
 * (SiLU(x W1ᵀ) ⊙ x W3ᵀ) W2ᵀ).  Routed expert e runs on permuted rows
 * [expert_offsets[e], expert_offsets[e+1]) of u_perm and writes the same rows
 * of y_perm [T·k, H]; shared expert j runs on all rows of u and writes
 * y_shared [Ks, T, H].  Only the w1/w3/w2/sw1/sw3/sw2 members of `weights`
 * are read.  fp32 accumulation; bf16 layers round the intermediate
 * activation and the outputs to bf16.  ws: moe_expert_ffn_workspace_size. */
MOE_API moe_status moe_expert_ffn(const moe_shape* shape,
                                  const moe_weights* weights, const void* u,
                                  const void* u_perm,
                                  const int32_t* expert_offsets, void* y_perm,
                                  void* y_shared, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* h_t = u_t + Σ_{j<Ks} y_shared[j, t] + Σ_{s<k} topk_w[t, s] · y_perm[slot_row[t, s]]
 * (§3.1 Eq. 9–11), accumulated in fp32 in exactly this order and rounded
 * once to shape->dtype.  h [T, H] out; h may not alias any input. */
MOE_API moe_status moe_combine(const moe_shape* shape, const void* u,
                               const void* y_perm, const void* y_shared,
                               const float* topk_w, const int32_t* slot_row,
                               void* h, moe_stream_t stream);

/* Selection-bias controller of the aux-loss-free load balancing (page "MoE
 * 的分水岭", ibossgateway ch. 7 §7.4): for every routed expert e, its load
 * L_e = expert_offsets[e+1] - expert_offsets[e] (the rows moe_dispatch gave
 * it) is compared with the mean load T·k / E (exactly, in integers);
 * select_bias[e] -= gamma if L_e is above the mean, += gamma if below, and
 * stays if equal (one fp32 rounding).  select_bias [E] fp32 is updated in
 * place; loads [E] int32 (may be NULL) receives L_e.  gamma >= 0 and finite
 * (the pages give no value; it is the caller's step).  The bias is the one
 * MOE_GATE_SIGMOID_BIAS adds for the choice only. */
MOE_API moe_status moe_update_select_bias(const moe_shape* shape,
                                          const int32_t* expert_offsets,
                                          float* select_bias, float gamma,
                                          int32_t* loads, moe_stream_t stream);

/* Statistics of the expert-level balance loss (page "19-deepseek-moe",
 * ai.tomabc.com, load-balance section: the loss is proportional to
 * Σ_i f_i P_i).  That formula did not survive on the page; the reading:
 *   f[i] = E · L_i / (k · T), L_i = expert_offsets[i+1] - expert_offsets[i],
 *          the routing distribution counted over all E routed experts (an
 *          even routing gives 1); one fp64 division, rounded to fp32; 0 when
 *          k · T = 0;
 *   p[i] = (1/T) Σ_t q_{i,t}, q_t the token's gate distribution over the E
 *          routed experts computed from logits [T, E] (fp32, as
 *          moe_router_logits writes them): softmax scores, or for
 *          MOE_GATE_SIGMOID_BIAS the sigmoid scores divided by their sum over
 *          all E (select_bias plays no part); 0 when T = 0.
 * f, p [E] fp32 out.  The sums run in a fixed order (fp32 within 256-token
 * chunks, fp64 across chunks), so results are reproducible.  Group limits
 * in the shape are ignored.  ws: moe_balance_stats_workspace_size bytes. */
MOE_API size_t moe_balance_stats_workspace_size(const moe_shape* shape);
MOE_API moe_status moe_balance_stats(const moe_shape* shape, const float* logits,
                                     const int32_t* expert_offsets, float* f,
                                     float* p, void* ws, size_t ws_bytes,
                                     moe_stream_t stream);

/* Whole layer: router logits, route, dispatch, expert FFNs, combine, all on
 * `stream`.  route_out (may be NULL) receives copies of the routing
 * intermediates.  ws: moe_layer_workspace_size bytes. */
MOE_API moe_status moe_layer_forward(const moe_shape* shape,
                                     const moe_weights* weights, const void* u,
                                     void* h, const moe_route_outputs* route_out,
                                     void* ws, size_t ws_bytes,
                                     moe_stream_t stream);

/* The same layer with HOST token buffers: copies u_host [T, H] into u_dev,
 * runs moe_layer_forward, copies h_dev into h_host [T, H], and returns
 * without synchronising; once `stream` has completed, h_host holds the
 * result (synchronise `stream` before reading it).  Host buffers should be
 * pinned for the copies to be asynchronous.
 * Large batches are pipelined: the tokens are cut into up to 8 chunks (each
 * at least 4096 tokens and, on average, at least 512 rows per routed expert)
 * and the copy of one chunk to the device, the layer on the previous chunk
 * and the copy back of the one before run at the same time.  The copies run
 * on two non-blocking streams that the library creates on the first such
 * call on a device and keeps; they wait for the work queued on `stream`
 * before the call, and `stream` waits for the last copy back.  The result is
 * bitwise the same as one moe_layer_forward over all tokens (tokens are
 * independent).  ws: moe_layer_workspace_size(shape) bytes. */
MOE_API moe_status moe_layer_forward_host(const moe_shape* shape,
                                          const moe_weights* weights,
                                          const void* u_host, void* h_host,
                                          void* u_dev, void* h_dev, void* ws,
                                          size_t ws_bytes,
                                          moe_stream_t stream);

/* The layer on a sequence of n_batches token batches in HOST memory, each
 * [T, H] (shape->T tokens): u_host[b] in, h_host[b] out (host pointers,
 * pinned for the copies to be asynchronous; arrays of n_batches pointers).
 * Batch b + 1's copy to the device and batch b - 1's copy back overlap the
 * layer on batch b, so a long sequence runs at the rate of the slower of the
 * layer and the host link.  u_dev and h_dev are device buffers of two slots
 * of [T, H] each (2·T·H elements), used alternately; ws:
 * moe_layer_workspace_size(shape) bytes, reused batch after batch on
 * `stream`.  The copies run on the library's two copy streams (as for
 * moe_layer_forward_host); they wait for the work queued on `stream` before
 * the call, and `stream` waits for the last copies back, so h_host[b] is
 * complete once `stream` has completed.  Each h_host[b] is bitwise
 * moe_layer_forward of u_host[b].  Returns MOE_ERR_INVALID_ARG for
 * n_batches < 0 or a NULL pointer; n_batches = 0 or T = 0 does nothing. */
MOE_API moe_status moe_layer_forward_host_stream(const moe_shape* shape,
                                                 const moe_weights* weights,
                                                 int n_batches,
                                                 const void* const* u_host,
                                                 void* const* h_host, void* u_dev,
                                                 void* h_dev, void* ws,
                                                 size_t ws_bytes,
                                                 moe_stream_t stream);

/* Weight gradients of moe_layer_backward (device pointers, fp32, written, not
 * accumulated): d_centroids [E, H]; dw1, dw3 [E, I, H]; dw2 [E, H, I]; the
 * shared experts' dsw1, dsw3 [Ks, I, H] and dsw2 [Ks, H, I] (NULL when
 * n_shared = 0); dw3 and dsw3 are NULL for ReLU. */
typedef struct {
  float* d_centroids;
  float *dw1, *dw3, *dw2;
  float *dsw1, *dsw3, *dsw2;
} moe_weight_grads;

/* Backward of moe_layer_forward for the upstream gradient dh = dL/dh [T, H]
 * (bf16): du = dL/du [T, H] (bf16 out) and the weight gradients `grads`.
 * The forward is h_t = u_t + Σ_j FFN_j^shared(u_t) + Σ_s g_{t,s}
 * FFN_{idx[t,s]}(u_t) (page "02 · 细粒度 MoE", §3.1 Eq. 9–15; expert FFN as on
 * page "19-deepseek-moe"), differentiated with the chosen experts held fixed:
 * the top-k choice is piecewise constant in the logits, so gradients reach
 * the router only through the gate weights g, and select_bias (which only
 * changes the choice) gets none.  logit_offset is read like the forward
 * reads it (no gradient is returned for it).
 *   du_t = dh_t + Σ_j J_j^T dh_t + Σ_s g_{t,s} J_{idx}^T dh_t + Σ_i dz_{t,i} e_i,
 *   dg_{t,s} = <dh_t, FFN_{idx[t,s]}(u_t)>, dz = dL/dlogits through softmax
 *   (no renormalisation) or the normalised sigmoid, d e_i = Σ_t dz_{t,i} u_t.
 * With saved == NULL the call recomputes the forward's routing and the
 * experts' pre-activations from u, so it needs only the forward's inputs;
 * with the `saved` buffer that moe_layer_forward_train filled for the same
 * u and weights it reuses them instead (saved_bytes >= moe_layer_saved_size).
 * fp32 accumulation; the intermediates (pre-activations, per-row gradients,
 * transposed operands) are bf16, as in the forward.  bf16 layers only, with
 * inter % 128 == 0 and (n_routed + n_shared) x (2 for SwiGLU, else 1) <= 1024
 * (otherwise MOE_ERR_UNSUPPORTED).  T = 0 writes zero gradients.
 * ws: moe_layer_backward_workspace_size bytes. */
MOE_API size_t moe_layer_backward_workspace_size(const moe_shape* shape);
MOE_API moe_status moe_layer_backward(const moe_shape* shape,
                                      const moe_weights* weights, const void* u,
                                      const void* dh, void* du,
                                      const moe_weight_grads* grads,
                                      const void* saved, size_t saved_bytes,
                                      void* ws, size_t ws_bytes,
                                      moe_stream_t stream);

/* Training forward: moe_layer_forward (same result h, bitwise) that also
 * keeps, in the caller's `saved` buffer (device, 16-byte aligned,
 * moe_layer_saved_size bytes), what moe_layer_backward would otherwise
 * recompute: the router logits, the choice and gate weights, the dispatch
 * (offsets and permutation), the permuted token rows and the experts'
 * pre-activations x W1ᵀ (and x W3ᵀ for SwiGLU) in bf16, written by the
 * gate/up GEMM's epilogue next to the activation.  The buffer's layout is
 * private to the library; it stays valid while u and the weights do.  bf16
 * layers only (0 / MOE_ERR_UNSUPPORTED otherwise).  ws:
 * moe_layer_workspace_size bytes. */
MOE_API size_t moe_layer_saved_size(const moe_shape* shape);
MOE_API moe_status moe_layer_forward_train(const moe_shape* shape,
                                           const moe_weights* weights,
                                           const void* u, void* h, void* saved,
                                           size_t saved_bytes, void* ws,
                                           size_t ws_bytes, moe_stream_t stream);

/* ---- Expert parallelism (page "02 · 细粒度 MoE：从 Mixtral 到 DeepSeekMoE",
 * llm-infra-atlas, §3.2: the routed experts are spread over devices and token
 * rows reach them through all-to-all exchanges; the shared experts are
 * replicated on every device and need no exchange).  With D ranks, rank d
 * holds routed experts [d·E_loc, (d+1)·E_loc), E_loc = E / D.  A rank's
 * moe_dispatch output is already grouped by destination (rows sorted by
 * expert); the caller exchanges the per-expert counts and the rows (NCCL or
 * any all-to-all), and these two calls do the local part: */

/* Expert FFNs on rows given explicitly (the rows an expert-parallel rank
 * received), same arithmetic as moe_expert_ffn.  shape: this rank's layer —
 * T local tokens (the shared experts run on u [T, H]), n_routed = E_loc
 * local experts, top_k ignored (0 is valid).  Routed expert e runs on rows
 * [expert_offsets[e], expert_offsets[e+1]) of x_rows [n_rows, H] and writes
 * the same rows of y_rows [n_rows, H]; expert_offsets [E_loc + 1] (device)
 * must end at n_rows.  n_rows = 0 with zero offsets runs the shared experts
 * only; shape->n_shared = 0 runs the routed experts only.  weights: w1/w3/w2
 * hold this rank's E_loc experts ([E_loc, I, H] and [E_loc, H, I]).  ws:
 * moe_expert_ffn_rows_workspace_size(shape, m) bytes for any n_rows <= m. */
MOE_API size_t moe_expert_ffn_rows_workspace_size(const moe_shape* shape, int64_t max_rows);
MOE_API moe_status moe_expert_ffn_rows(const moe_shape* shape, const moe_weights* weights,
                                       int64_t n_rows, const void* u, const void* x_rows,
                                       const int32_t* expert_offsets, void* y_rows,
                                       void* y_shared, void* ws, size_t ws_bytes,
                                       moe_stream_t stream);

/* Moves the n_rows rows a rank received between the order the exchange
 * delivers (source-major: for each source rank s, for each local expert e,
 * the rows s sent to e) and the order the expert GEMMs read (expert-major:
 * for each local expert e, for each source s).  counts [n_ranks · E_loc]
 * (device, int32): counts[s · E_loc + e] rows from source s for local expert
 * e, summing to n_rows; shape->n_routed = E_loc, shape->H and ->dtype give
 * the row size.  to_expert_major != 0: src is source-major, dst
 * expert-major; 0: the inverse.  expert_offsets (device, may be NULL) [E_loc
 * + 1] out: the expert-major offsets.  n_ranks · E_loc <= 1024.  src and dst
 * [n_rows, H] may not alias.  No scratch, no host synchronisation. */
MOE_API moe_status moe_ep_regroup(const moe_shape* shape, int32_t n_ranks,
                                  const int32_t* counts, int64_t n_rows, const void* src,
                                  void* dst, int32_t* expert_offsets,
                                  int32_t to_expert_major, moe_stream_t stream);

/* moe_dispatch without a workspace argument, for callers that cannot
 * allocate device memory: a runtime whose allocator already owns all of the
 * GPU's memory and has no scratch to lend, or a latency-critical path that
 * must not call cudaMalloc (it can synchronise the device).  The source pages
 * have no counterpart; this is a deployment convenience.
 *
 * Same arguments and results as moe_dispatch minus ws/ws_bytes.  Its scratch
 * is a fixed 1 MiB array inside the library, held by every GPU that loads the
 * library until the process exits; it fits ceil(T / 256) * n_routed <= 131072
 * (for example T <= 32768 tokens with 1024 experts, or T <= 131072 with 256).
 * Larger shapes return MOE_ERR_UNSUPPORTED and launch nothing.  The library
 * looks up the array's device address on the first call made on each device
 * (with that device current), so make that first call before any stream
 * capture; it looks the address up again when the device's current context
 * has changed since (after cudaDeviceReset, the module may be loaded at
 * another address).  All calls share the one array, and every call overwrites what it
 * uses before reading it: calls that may overlap on the GPU (different
 * streams, or concurrent host threads) race and must be serialised by the
 * caller.  Allocates nothing. */
MOE_API moe_status moe_dispatch_static(const moe_shape* shape,
                                       const int32_t* topk_idx, const void* u,
                                       int32_t* expert_offsets,
                                       int32_t* row_token, int32_t* slot_row,
                                       void* u_perm, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
