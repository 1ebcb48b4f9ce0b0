/*
 * moe.h -- C ABI of libmoe.so: the forward pass of one mixture-of-experts
 * (MoE) feed-forward layer on one NVIDIA B300 (sm_103a).
 *
 * The layer (page titles cited; section or equation after each):
 *   s   = x W_r^T (+ b_r)                  router scores
 *         ("Mixture of Experts: More Parameters, Same FLOPs", 'The router';
 *          "Mixture of experts" (frontiers track), 'Where the experts live')
 *   idx = top-k of s, largest first, lower expert index first on equal scores
 *   w   = gate weights, by gating mode (see moe_gating_mode)
 *   C   = ceil(capacity_factor * T * k / E)   expert capacity
 *         ("Mixture of Experts" (module 17), 17.5 equation); assignments
 *         beyond C, in token order, are dropped by that expert only
 *   y_t = FFN_shared(x_t) + sum_{j<k, kept} w_tj FFN_{idx_tj}(x_t)
 *         (module 17, 17.2 equation), FFN(v) = W_down (silu(W_gate v) * (W_up v))
 *   aux = alpha * E * sum_e f_e P_e, f_e = n_e / (T k), P_e = mean_t p_te
 *         (module 17, 17.4 equation; "Mixture of experts" (frontiers track),
 *          'Keeping the load balanced'); n_e counts assignments before capacity.
 * The residual connection is not added: y excludes x.
 *
 * Conventions (all entry points):
 *   - Every tensor pointer is DEVICE memory allocated and owned by the caller;
 *     the library allocates nothing and keeps no pointer after a call returns.
 *   - Work is enqueued on `stream` and the call returns without waiting; no
 *     entry point except moe_read_device_status synchronises.
 *   - Errors the host can detect return a non-zero moe_status before anything
 *     is launched and leave every output untouched.
 *   - Entry points may be called from several host threads at once; calls
 *     that run concurrently on the GPU need their own outputs and workspace
 *     (moe_forward_no_alloc shares one static scratch: see there).
 *   - Row-major, dense, contiguous tensors.  "K-major" weights: each output
 *     row is contiguous over the reduction dimension.
 *   - dtype applies to x, the expert weights, W_r and y; router scores, gate
 *     weights and statistics are fp32 in every dtype.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

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
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad enum, ... */
    MOE_ERR_UNSUPPORTED = 2,   /* a shape outside the supported set below */
    MOE_ERR_WORKSPACE = 3,     /* workspace too small or not 256-byte aligned */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
    MOE_ERR_DEVICE_STATUS = 5  /* a kernel reported an error (see below) */
} moe_status;

/* Gate weights for the k selected experts of a token.
 *   MOE_GATE_SOFTMAX_SELECTED: w_j = e^{s_j} / sum_{j' in top-k} e^{s_j'}
 *     (Mixtral; module 17, 17.2; frontiers track, gate equation); sums to 1.
 *   MOE_GATE_SOFTMAX_ALL: p = softmax(s) over all E, w_j = p_{idx_j}, no
 *     renormalisation (Switch Transformer / Qwen2; module 17, 17.2); with
 *     k = 1 this is the raw top-1 probability ('The router', last remark).
 *   MOE_GATE_SOFTMAX_ALL_RENORM: w_j = p_{idx_j} / sum_{j'} p_{idx_j'}
 *     ('The router', equation MoE(x)); w = 1 when k = 1.
 *   MOE_GATE_SIGMOID_SELECTED: a = sigmoid(s), w_j = a_{idx_j} / sum_{j'}
 *     a_{idx_j'} ('The router', closing remark: DeepSeek-V3 scores experts
 *     with a sigmoid, normalised over the chosen ones); the selection is by s
 *     (sigmoid is monotone); for the balance loss p = a / sum over all E. */
typedef enum {
    MOE_GATE_SOFTMAX_SELECTED = 0,
    MOE_GATE_SOFTMAX_ALL = 1,
    MOE_GATE_SOFTMAX_ALL_RENORM = 2,
    MOE_GATE_SIGMOID_SELECTED = 3
} moe_gating_mode;

typedef enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_FP32 = 1 } moe_dtype;

/* Layer shape and options.  Supported:
 *   T >= 0 tokens, T * top_k < 2^31;
 *   1 <= n_experts <= 256; 1 <= top_k <= min(8, n_experts);
 *   1 <= d_model, d_expert <= 2^20; 0 <= d_shared <= 2^20 (0 = no shared
 *   expert);
 *   bf16: d_model, d_expert and d_shared multiples of 64;
 *   fp32: any sizes (SIMT path, for small layers and exact checks).
 * capacity_factor <= 0 means dropless.  aux_alpha scales aux_loss.
 * bias_selection_only: 0 = router_bias is part of the scores (selection and
 * weights); 1 = router_bias only shifts the top-k selection keys, fp32(s + b),
 * and the scores and weights exclude it ("Mixture of Experts: More
 * Parameters, Same FLOPs", 'Keeping the load even', bias balancing: the bias
 * is added to the scores only when choosing the top k). */
typedef struct {
    int32_t T;
    int32_t d_model;
    int32_t n_experts;
    int32_t d_expert;
    int32_t top_k;
    int32_t d_shared;
    int32_t dtype;          /* moe_dtype */
    int32_t gating_mode;    /* moe_gating_mode */
    float capacity_factor;
    float aux_alpha;
    int32_t bias_selection_only;
} moe_config;

/* Device status codes written by kernels (read with moe_read_device_status). */
#define MOE_DEVICE_OK 0
#define MOE_DEVICE_NONFINITE_SCORE 1   /* a router score was NaN/Inf */
#define MOE_DEVICE_PIPELINE_TIMEOUT 2  /* a bounded in-kernel wait ran out */
#define MOE_DEVICE_LAUNCH_MISMATCH 3   /* a kernel got less shared memory than its layout needs */
#define MOE_DEVICE_SHARD_MISMATCH 4    /* split batch: the exchanged counts do not hold
                                          this rank's own or do not add up to T_global*k */
#define MOE_DEVICE_INDEX_OUT_OF_RANGE 5 /* an expert index outside [0, E), or a row that
                                          falls outside its expert's segment: checked on
                                          the topk_idx a caller hands to moe_sharded_finish,
                                          and on every index the routing and combine
                                          kernels use in a build with MOE_DEBUG_BOUNDS */

/* Bytes of scratch moe_forward needs for `cfg` (x gathered by expert, the
 * SwiGLU hidden rows, per-expert scan tables, ...).  Returns
 * MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for an invalid config. */
MOE_API moe_status moe_workspace_size(const moe_config *cfg, size_t *bytes);

/* Expert capacity the library uses for `cfg`: ceil(capacity_factor * T *
 * top_k / n_experts) computed in double, or -1 when dropless
 * (module 17, 17.5 equation); a value of 9.2e18 or more (larger than any
 * demand, so nothing is dropped) saturates at INT64_MAX.  Host only; no GPU
 * needed. */
MOE_API int64_t moe_capacity(const moe_config *cfg);

/* The forward pass (one call = the whole layer, enqueued on `stream`).
 *
 * Inputs (device, dtype = cfg->dtype unless stated):
 *   x            [T, d_model]
 *   W_r          [E, d_model]               router, K-major
 *   router_bias  [E] fp32, or NULL          added to the scores before
 *                                           selection and weighting, or to
 *                                           the selection keys only
 *                                           (cfg->bias_selection_only)
 *   W_gate, W_up [E, d_expert, d_model]     K-major
 *   W_down       [E, d_model, d_expert]     K-major
 *   Ws_gate, Ws_up [d_shared, d_model]; Ws_down [d_model, d_shared];
 *                                           all NULL when d_shared == 0
 * Outputs (device):
 *   y             [T, d_model] dtype
 *   router_logits [T, E] fp32   the scores s (bias included unless it is
 *                               selection-only)
 *   topk_idx      [T, k] int32  selected experts, largest score first
 *   topk_w        [T, k] fp32   gate weights (not renormalised after drops)
 *   dropped_mask  [T, k] uint8  1 = dropped by capacity
 *   expert_counts [E] int32     assignments per expert before capacity
 *   kept_counts   [E] int32     assignments per expert after capacity
 *   aux_loss      [1] fp32      balance loss (0 when T == 0)
 * workspace: device, 256-byte aligned, >= moe_workspace_size(cfg) bytes;
 *   its contents on entry are ignored.
 * When T == 0 only expert_counts, kept_counts, aux_loss and workspace must
 * be non-NULL; they are zeroed and nothing else is touched.
 * Inputs must be finite; a non-finite score sets MOE_DEVICE_NONFINITE_SCORE
 * (outputs then stay in bounds but are unspecified).
 * Returns MOE_OK once everything is enqueued. */
MOE_API moe_status moe_forward(const moe_config *cfg,
                       const void *x, const void *W_r, const float *router_bias,
                       const void *W_gate, const void *W_up, const void *W_down,
                       const void *Ws_gate, const void *Ws_up, const void *Ws_down,
                       void *y, float *router_logits, int32_t *topk_idx,
                       float *topk_w, uint8_t *dropped_mask,
                       int32_t *expert_counts, int32_t *kept_counts,
                       float *aux_loss, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Per-unit timeline of the routed CTA-pair GEMMs and per-block timeline of
 * the dispatch kernel, for profiling (a measurement aid, not an operation of
 * the layer the pages define).  Only the library built with
 * MOE_TIMELINE (libmoe_timeline.so; python -m
 * mixture_experts_layer_capacity_b300.build --timeline) records them; other
 * builds return MOE_ERR_UNSUPPORTED.  All words are globaltimer
 * nanoseconds.  CTA 0 of each routed pair launch writes, for its i-th unit,
 * 8 words at [region * 32768 + i * 8], region 0 for the gate/up GEMM and 1
 * for the down projection, i < 4096:
 *   [0] the MMA thread starts waiting for a free accumulator, [1] it has one,
 *   [2] the unit's first ring stage is full, [3] its last MMA is issued,
 *   [7] the epilogue starts the unit (E4M3 tiles first copy their column
 *   scales) and waits for the accumulator, [4] it is full, [5] the epilogue
 *   is done; [6] is 1 for a swap unit, 0 for a pair tile.
 * Dispatch block b < 4096 writes 8 words at [65536 + b * 8]: [0] its start,
 * [1] its rows staged, [2] its router scores done, [3] its tokens gated
 * (these three for its first chunk of tokens; equal to [0] for a block
 * without tokens), [4] its gating done, [5] past the grid barrier, [6] the
 * segment tables done, [7] its last row copy done.
 * Unwritten words stay 0; a later launch of the same kernel overwrites the
 * records, so read them after the forward pass of interest.
 * moe_timeline_clear zeroes all 98304 words; moe_timeline_read copies the
 * first n_words (<= 98304) into host_words, caller-owned host memory of at
 * least n_words words.  Both synchronise with the device.  Errors: a null
 * host_words or n_words outside [0, 98304] -> MOE_ERR_INVALID_ARG (checked
 * after MOE_ERR_UNSUPPORTED); a failed copy -> MOE_ERR_CUDA. */
#define MOE_TIMELINE_WORDS 98304
MOE_API moe_status moe_timeline_clear(void);
MOE_API moe_status moe_timeline_read(uint64_t *host_words, int64_t n_words);

/* Which kernels moe_forward launches for `cfg` (for profiling and launch
 * counts; host only, no GPU needed).  *flags is a bit set of: */
#define MOE_PLAN_ROUTER_FUSED 1   /* router GEMM inside the gating kernel */
#define MOE_PLAN_DIRECT_Y 2       /* down projection writes y; no combine kernel */
#define MOE_PLAN_PAIR_ROUTED 4    /* routed GEMMs on CTA pairs (256-row tiles) */
#define MOE_PLAN_PAIR_SHARED 8    /* shared-expert GEMMs on CTA pairs */
#define MOE_PLAN_SHARED_FUSED 16  /* shared-expert tiles run inside the routed GEMM
                                     launches (no separate shared launches) */
#define MOE_PLAN_PAIR_TAILS 32    /* with CTA pairs, the small experts (fewer rows
                                     than one swap chunk: 128 in the gate/up GEMM,
                                     64 or 128 in the down projection) run as
                                     "swap" units in the same launch: their
                                     weights are the MMA's 256-row operand and
                                     their token rows (rounded up to 32) the
                                     other, so they are not padded to 256 rows;
                                     larger experts keep 256-row tiles */
#define MOE_PLAN_W8A8_SWAP 64     /* moe_forward_w8a8 only: at most 64 rows per
                                     expert on average (T * k <= 64 * E), so its
                                     expert GEMMs take the weights as the 128-row
                                     MMA operand and up to 32 token rows of an
                                     expert as the other; else 128-row token tiles */
MOE_API moe_status moe_launch_plan(const moe_config *cfg, int32_t *flags);

/* Workspace bytes moe_latent_forward needs for `cfg` (whose d_model is the
 * latent width L) and outer width d_outer; MOE_ERR_UNSUPPORTED when d_outer
 * is not a multiple of 64 for bf16. */
MOE_API moe_status moe_latent_workspace_size(const moe_config *cfg, int32_t d_outer,
                                             size_t *bytes);

/* A latent MoE ("Mixture of Experts: Sparse FFNs, Routers, and Shared
 * Experts", the Nemotron 3 Super variant that closes the page after 'The 2026
 * configuration table': the whole MoE layer runs at a narrower width L, e.g.
 * L = 1024 inside a 4096-wide model, between a projection down to L and one
 * back up):
 *   x_lat = x W_in^T,  y_lat = the layer of moe_forward on x_lat,
 *   y     = y_lat W_out^T.
 * cfg describes the layer at the latent width (cfg->d_model = L); the router,
 * experts and shared expert all work at width L.
 *   x     [T, d_outer]; W_in [L, d_outer]; W_out [d_outer, L]  (dtype, K-major)
 *   y     [T, d_outer]
 * The other arguments, outputs and conventions are those of moe_forward
 * (router_logits are the latent router's scores).  workspace >=
 * moe_latent_workspace_size(cfg, d_outer); x_lat and y_lat live in it. */
MOE_API moe_status moe_latent_forward(const moe_config *cfg, int32_t d_outer,
                       const void *x, const void *W_in, const void *W_out,
                       const void *W_r, const float *router_bias,
                       const void *W_gate, const void *W_up, const void *W_down,
                       const void *Ws_gate, const void *Ws_up, const void *Ws_down,
                       void *y, float *router_logits, int32_t *topk_idx,
                       float *topk_w, uint8_t *dropped_mask,
                       int32_t *expert_counts, int32_t *kept_counts,
                       float *aux_loss, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Where moe_latent_forward keeps the latent activations inside its
 * workspace (same cfg and d_outer): x_lat = x W_in^T at byte offset
 * *x_lat_offset and y_lat (the layer's output at width L) at *y_lat_offset,
 * each [T][L] row-major in the config's dtype.  Both stay there after the
 * call until the workspace is used again, so a caller can read them, e.g. to
 * check the router scores against the exact latent rows the router saw.
 * MOE_ERR_INVALID_ARG for null pointers or d_outer < 1; MOE_ERR_UNSUPPORTED
 * as moe_latent_workspace_size.  Host only; launches nothing. */
MOE_API moe_status moe_latent_offsets(const moe_config *cfg, int32_t d_outer,
                                      size_t *x_lat_offset, size_t *y_lat_offset);

/* ---- e4m3 (FP8) expert weights for decode-sized batches.
 *
 * At small T the expert GEMMs are bound by the bytes of the touched expert
 * weights ("Mixture of Experts: More Parameters, Same FLOPs", 'What experts
 * cost at serving time': decoding reads each weight for ~2 FLOPs, and serving
 * memory is sized at 8 bits per weight).  These entry points store every
 * routed and shared expert weight matrix as e4m3 codes with one fp32 scale
 * per weight row (output feature): W[r][c] = decode(q[r][c]) * scale[r].
 * In moe_forward_w8 the activations, the router and all accumulation stay as
 * in moe_forward (bf16 inputs, fp32 accumulation); the e4m3 values enter the
 * tensor cores exactly (every e4m3 value is a bf16 value).  moe_forward_w8a8
 * quantizes the expert GEMMs' activation rows to e4m3 as well. */

/* Row-wise quantization of a bf16 matrix W [rows, cols] (device, row-major):
 *   scale[r] = max_c |W[r][c]| / 448 in fp32 (1 when the row is all zero),
 *   q[r][c]  = e4m3(W[r][c] / scale[r]): fp32 division, round to nearest
 *              even, saturating to +-448 (OCP FP8 E4M3, no infinities).
 * q [rows, cols] uint8 and scale [rows] fp32 are device outputs.  W and q
 * 16-byte aligned, cols a multiple of 16 (MOE_ERR_INVALID_ARG otherwise).
 * Stacked expert weights [E, n, m] are rows = E*n, cols = m. */
MOE_API moe_status moe_quantize_e4m3_rows(int64_t rows, int64_t cols, const void *W,
                                          uint8_t *q, float *scale, cudaStream_t stream);

/* The forward pass of moe_forward with e4m3 expert weights (cfg->dtype must
 * be MOE_DTYPE_BF16, else MOE_ERR_UNSUPPORTED):
 *   W_gate_q, W_up_q [E, d_expert, d_model], W_down_q [E, d_model, d_expert]
 *   uint8 (16-byte aligned); W_gate_scale, W_up_scale [E * d_expert],
 *   W_down_scale [E * d_model] fp32; likewise Ws_*_q / Ws_*_scale for the
 *   shared expert ([d_shared, d_model] / [d_model, d_shared], scales
 *   [d_shared] / [d_model]; all NULL when d_shared == 0).
 * Every other argument, output and convention is that of moe_forward, with
 * the same workspace size (moe_workspace_size).  The expert GEMMs run one
 * tensor-core kernel per projection with the weights as the operand held in
 * tensor memory, sized for batches of up to a few hundred tokens; larger
 * batches are correct but stream each weight tile once per 32 rows of an
 * expert. */
MOE_API moe_status moe_forward_w8(const moe_config *cfg,
                       const void *x, const void *W_r, const float *router_bias,
                       const uint8_t *W_gate_q, const float *W_gate_scale,
                       const uint8_t *W_up_q, const float *W_up_scale,
                       const uint8_t *W_down_q, const float *W_down_scale,
                       const uint8_t *Ws_gate_q, const float *Ws_gate_scale,
                       const uint8_t *Ws_up_q, const float *Ws_up_scale,
                       const uint8_t *Ws_down_q, const float *Ws_down_scale,
                       void *y, float *router_logits, int32_t *topk_idx,
                       float *topk_w, uint8_t *dropped_mask,
                       int32_t *expert_counts, int32_t *kept_counts,
                       float *aux_loss, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* The forward pass of moe_forward_w8 with E4M3 activations too ("Mixture of
 * Experts: More Parameters, Same FLOPs", 'What experts cost at serving
 * time' and its arithmetic of published configurations: DeepSeek-V3 sends
 * the dispatched token rows in FP8).  The permuted token rows, the
 * shared expert's token rows and the hidden rows h between the two expert
 * GEMMs are quantized row by row with moe_quantize_e4m3_rows's rule (fp32
 * scale = max|row| / 448, codes round to nearest even of v / scale,
 * saturating; h is quantized from its fp32 value), and each expert GEMM
 * multiplies E4M3 codes by E4M3 codes on the tensor cores with an fp32
 * accumulator, scaled by the token row's and the weight row's scales.
 * Arguments, outputs and conventions are those of moe_forward_w8, except the
 * workspace: >= moe_w8a8_workspace_size(cfg) bytes, 256-byte aligned
 * (MOE_ERR_WORKSPACE otherwise).  A layer with a shared expert and
 * d_expert < 128 is MOE_ERR_UNSUPPORTED.  Batches of any size run the
 * 128-row tile GEMMs with the weights as the wide operand. */
MOE_API moe_status moe_w8a8_workspace_size(const moe_config *cfg, size_t *bytes);
MOE_API moe_status moe_forward_w8a8(const moe_config *cfg,
                       const void *x, const void *W_r, const float *router_bias,
                       const uint8_t *W_gate_q, const float *W_gate_scale,
                       const uint8_t *W_up_q, const float *W_up_scale,
                       const uint8_t *W_down_q, const float *W_down_scale,
                       const uint8_t *Ws_gate_q, const float *Ws_gate_scale,
                       const uint8_t *Ws_up_q, const float *Ws_up_scale,
                       const uint8_t *Ws_down_q, const float *Ws_down_scale,
                       void *y, float *router_logits, int32_t *topk_idx,
                       float *topk_w, uint8_t *dropped_mask,
                       int32_t *expert_counts, int32_t *kept_counts,
                       float *aux_loss, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Where moe_forward_w8a8 keeps its quantized activations inside its
 * workspace (same cfg), as byte offsets: the permuted token rows' codes
 * (uint8 [R][d_model]) and scales (fp32 [R]), the hidden rows before
 * quantization (fp32 [R][d_expert]), their codes (uint8 [R][d_expert]) and
 * scales (fp32 [R]).  Row r is the r-th kept (token, expert) assignment in
 * expert order, tokens ascending within an expert; R = the sum of
 * kept_counts.  They stay there after the call until the workspace is used
 * again.  MOE_ERR_INVALID_ARG for a null pointer; other errors as
 * moe_w8a8_workspace_size.  Host only; launches nothing. */
MOE_API moe_status moe_w8a8_offsets(const moe_config *cfg, size_t *x_codes, size_t *x_scales,
                                    size_t *h_values, size_t *h_codes, size_t *h_scales);

/* ---- One batch split over several ranks (data parallel), same results as
 * one moe_forward over the whole batch.
 *
 * The layer's tokens are independent except for two couplings: capacity is
 * applied in token order over the WHOLE batch ("Mixture of Experts" (module
 * 17), 17.5: C = ceil(capacity_factor * T * k / E) with T the batch, tokens
 * past C dropped), and the balance loss uses f_e and P_e over the whole batch
 * (17.4 equation).  Rank r holds tokens [start_r, start_r + T_r) of the batch,
 * ranks in token order, sum of T_r = T_global.  Per rank:
 *   1. moe_sharded_route: gating of the rank's tokens; writes its per-expert
 *      demand counts and probability sums;
 *   2. the caller exchanges them (an all-gather in rank order) into
 *      all_expert_counts [n_ranks][E] and all_prob_sums [n_ranks][E];
 *   3. moe_sharded_finish: an assignment's global position is the count of
 *      earlier ranks' assignments to its expert plus its position here; it is
 *      kept iff that is below C (T = T_global); then the experts, combine and
 *      the balance loss over all ranks (probability sums added in rank order).
 * cfg->T is this rank's token count T_r (0 allowed); T_global >= cfg->T.
 * Both calls take the same workspace (>= moe_sharded_workspace_size bytes),
 * whose contents must survive between them, on streams ordered route ->
 * finish.  The outputs match moe_forward's for the rank's tokens, except
 * that expert_counts (from the route call) are this rank's demand counts
 * while kept_counts are this rank's kept assignments, and aux_loss is the
 * loss of the whole batch (the same on every rank). */
MOE_API moe_status moe_sharded_workspace_size(const moe_config *cfg, int64_t T_global,
                                              size_t *bytes);

/* Step 1.  x, W_r, router_bias, router_logits, topk_idx, topk_w as for
 * moe_forward (this rank's T rows).  Outputs: expert_counts [E] int32 and
 * prob_sums [E] fp64 (sum over this rank's tokens of the router
 * probabilities, for the balance loss).  When T == 0 they are zeroed and
 * nothing else is touched. */
MOE_API moe_status moe_sharded_route(const moe_config *cfg, int64_t T_global,
                       const void *x, const void *W_r, const float *router_bias,
                       float *router_logits, int32_t *topk_idx, float *topk_w,
                       int32_t *expert_counts, double *prob_sums,
                       void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Step 3.  all_expert_counts [n_ranks][E] int32 and all_prob_sums
 * [n_ranks][E] fp64 (device, rank order, row `rank` = this rank's step-1
 * outputs); topk_idx and topk_w are step 1's outputs (read only).  Writes y,
 * dropped_mask, kept_counts and aux_loss as moe_forward does.  A device check
 * that row `rank` equals this rank's counts and that all counts add up to
 * T_global * k sets MOE_DEVICE_SHARD_MISMATCH otherwise (later kernels then
 * skip their work).  0 <= rank < n_ranks. */
MOE_API moe_status moe_sharded_finish(const moe_config *cfg, int64_t T_global,
                       int32_t n_ranks, int32_t rank,
                       const int32_t *all_expert_counts, const double *all_prob_sums,
                       const void *x, const void *W_gate, const void *W_up,
                       const void *W_down, const void *Ws_gate, const void *Ws_up,
                       const void *Ws_down, const int32_t *topk_idx, const float *topk_w,
                       void *y, uint8_t *dropped_mask, int32_t *kept_counts,
                       float *aux_loss, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Size of the library's static device scratch used by moe_forward_no_alloc. */
#define MOE_STATIC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* The forward pass without a caller workspace, for callers that cannot
 * allocate device memory: for example a host program that links only this C
 * library and has no device allocator of its own, or a serving loop that must
 * not call cudaMalloc in its steady state (cudaMalloc can synchronise the
 * device).  (The pages have no counterpart to this entry point; it is a
 * property of this library, not of the layer.)
 *
 * Same arguments and results as moe_forward, minus the workspace: the
 * scratch is a 64 MiB array (MOE_STATIC_SCRATCH_BYTES) that the library holds
 * in device memory on every GPU that loads it, until the process exits.  The
 * function allocates nothing and calls no allocating routine.
 *   - Layers whose moe_workspace_size exceeds MOE_STATIC_SCRATCH_BYTES are
 *     rejected with MOE_ERR_WORKSPACE before anything is launched (for bf16:
 *     roughly decode-sized batches of the large layers, and batches of a few
 *     thousand tokens of small layers, fit).
 *   - Every call made outside stream capture looks up the array's device
 *     address on the current device (cudaGetSymbolAddress); a call made
 *     while its stream is capturing uses the address found by the last call
 *     outside capture on that device.  So make the first call on a device
 *     before any stream capture, and after a cudaDeviceReset make one call
 *     outside capture before capturing again (a reset may move the array).
 *   - All calls share the one array and it keeps the last call's contents;
 *     each call clears what must start at zero on its own stream.  Calls whose
 *     work overlaps on the GPU (other streams, other host threads) race on
 *     the array: serialise them.
 *   - The device status word lives in the shared array, so
 *     moe_read_device_status does not apply to this entry point. */
MOE_API moe_status moe_forward_no_alloc(const moe_config *cfg,
                       const void *x, const void *W_r, const float *router_bias,
                       const void *W_gate, const void *W_up, const void *W_down,
                       const void *Ws_gate, const void *Ws_up, const void *Ws_down,
                       void *y, float *router_logits, int32_t *topk_idx,
                       float *topk_w, uint8_t *dropped_mask,
                       int32_t *expert_counts, int32_t *kept_counts,
                       float *aux_loss, cudaStream_t stream);

/* Waits for `stream`, then reads the device status word the last
 * moe_forward on this workspace wrote: *code = MOE_DEVICE_OK or one of the
 * MOE_DEVICE_* codes.  Returns MOE_ERR_DEVICE_STATUS when *code != 0,
 * MOE_ERR_CUDA if the stream reported an error. */
MOE_API moe_status moe_read_device_status(const moe_config *cfg, const void *workspace,
                                  cudaStream_t stream, int32_t *code);

/* Test hook for the bounded waits (not for production use).  With
 * extra_arrivals = 1 every later moe_forward (and latent / split-batch
 * forward) makes the routing kernel's grid-wide barrier wait for one block
 * more than the grid has, so the barrier cannot complete: each block gives up
 * after limit_ns (0 = the default of 2 s; else 1 us ... 2 s), records
 * MOE_DEVICE_PIPELINE_TIMEOUT in the status word and returns, and the later
 * kernels of that forward pass see the status and do no work.  No copy or
 * other asynchronous work is in flight at that barrier, and the next call
 * clears the status word, so the context stays usable.
 * moe_debug_barrier_fault(0, 0) restores normal operation.  The setting is
 * process-wide and read when a forward pass is launched (a captured graph
 * keeps the setting it was captured with).  MOE_ERR_INVALID_ARG for other
 * values.  Host only; launches nothing. */
MOE_API moe_status moe_debug_barrier_fault(int32_t extra_arrivals, uint64_t limit_ns);

/* Stage timing (optional; for benchmarks and profiling).  While `events`
 * is non-NULL, every moe_forward call records events[i] on its stream at the
 * stage boundaries below, so that cudaEventElapsedTime(events[i],
 * events[i+1]) is the device time of stage i:
 *   0 start | 1 router scores | 2 dispatch (gating, counts, capacity,
 *   gather) | 3 routed gate/up GEMM | 4 routed down GEMM | 5 shared gate/up
 *   GEMM | 6 shared down GEMM | 7 combine (end)
 * (stage 1 is empty when the router runs inside the dispatch kernel, stages
 * 5-6 without a shared expert, and stage 7 when k = 1 without a shared expert
 * in bf16, where the down projection writes y).  Recorded during stream
 * capture they become event nodes of the graph.  n_events must be
 * MOE_NUM_STAGE_EVENTS.  The events are the caller's; the setting is
 * process-wide and not thread-safe.  Pass NULL to stop. */
#define MOE_NUM_STAGE_EVENTS 8
MOE_API moe_status moe_set_stage_events(cudaEvent_t *events, int n_events);

/* Static, human-readable name of a status. */
MOE_API const char *moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
