// moe_internal.h -- host-side internals of libmoe.so: workspace layout and
// the kernel launchers the C ABI sequences.  Not part of the public ABI.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kChunk = 32;       // most tokens per routing chunk (one bit each in a 32-bit mask)
constexpr int kMaxDispatchBlocks = 256;  // most blocks of the dispatch kernel
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;
constexpr int kMaxWidth = 1 << 20;  // largest d_model, d_expert, d_shared, d_outer
constexpr int kTileM = 128;      // rows per tensor-core tile (UMMA M)

// Byte offsets of the scratch regions inside the caller's workspace.  Every
// region starts on a 1024-byte boundary.
struct WorkspaceLayout {
    size_t status;   // int32[16] device status word, then the scan's block counter
    size_t bcount;   // int32[E][blocks]  per-block expert counts of the dispatch kernel
    size_t ppart;    // float[E][nchunk]  per-chunk sums of softmax probabilities
    size_t rank;     // int32[T*k]        rank of an assignment among its block's tokens
    size_t psum;     // double[E]         sum over tokens of the softmax probabilities
    size_t gcount;   // int32[E]          demand counts over all ranks (split batch)
    size_t seg_off;  // int32[E+1]        first x_perm row of each expert's segment
    size_t mtile;    // int32[E+1]        prefix sum of 128-row tiles per segment
    size_t row_of;   // int32[T*k]        x_perm row of an assignment, -1 if dropped
    size_t row_tok;  // int32[R_max]      token of each x_perm row (direct-y mode)
    size_t row_w;    // float[R_max]      gate weight of each x_perm row (direct-y mode)
    size_t x_perm;   // dtype[R_max, D]   token rows gathered in expert order
    size_t h;        // dtype[R_max, F]   SwiGLU hidden rows of the routed experts
    size_t z;        // dtype[R_max, D]   routed expert outputs (unweighted)
    size_t hs;       // dtype[T, S]       shared-expert hidden rows
    size_t zs;       // dtype[T, D]       shared-expert outputs (fp32 split partials at decode)
    size_t lpart;    // float[splits][T][E] router partial scores (split router only)
    size_t total;
    int64_t R_max;   // rows of x_perm: T*k dropless, else min(T*k, E*C)
    int64_t C;       // capacity, -1 dropless
    int nchunk;      // the most routing chunks: max(min(T, kMaxDispatchBlocks), ceil(T / kChunk))
};

// Inputs of the balance loss aux = alpha * E * sum_e f_e P_e, with
// f_e = n_e / (T k) and P_e = psum_e / T ("Mixture of Experts" (module 17),
// 17.4 equation; "Mixture of experts" (frontiers track), balance equation of
// 'Keeping the load balanced').  psum and counts are written by the dispatch
// kernel; the first expert kernel, which starts after it has completed,
// evaluates the loss.
struct AuxArgs {
    const double *psum;      // [E] sum over tokens of the softmax probabilities
    const int32_t *counts;   // [E] demand counts n_e
    float *out;              // [1], or null: nothing to compute
    int E, T, k;
    float alpha;
};

// Which kernels a forward pass on `c` launches (bf16 tensor-core path).
struct LaunchPlan {
    bool router_fused;  // router GEMM inside the dispatch kernel
    bool direct_y;      // the down projection writes y (no combine kernel)
    bool pair_routed;   // routed GEMMs on CTA pairs (256-row tiles)
    bool pair_shared;   // shared-expert GEMMs on CTA pairs
    bool shared_fused;  // shared-expert tiles inside the routed single-CTA launches
    bool pair_tails;    // pairs run each segment's full 256-row tiles, and its
                        // remaining rows as swap units in the same launch
    int router_splits;  // K-splits of the tensor-core router (1 = none)
};
// CTA pairs for large problems whose segments average at least 512 rows;
// decode-sized and small batches keep single-CTA tiles (few rows would
// leave most of a 256-row tile empty, and small GEMMs are bound by latency,
// not by shared-memory traffic).
constexpr long long kPairMinRows = 16384;  // fewest routed GEMM rows for pairs
LaunchPlan plan_of(const moe_config &c);

// K-splits of the shared expert's down projection when its tiles run inside
// the routed launch: a tile reduces over S while a routed tile reduces over
// F, so S is cut into ceil(S / F) pieces (at most 8) to give every work unit
// about the same length.  The pieces write fp32 partial sums [splits][T][D]
// that the combine kernel adds in split order.  1 = no split (bf16 [T][D]).
int shared_down_splits(const moe_config &c);
constexpr int kMaxSharedSplits = 8;

// K-splits of the tensor-core router GEMM.  Batches below 512 tokens give
// it one to four 128-row tiles, so its reduction over d_model is split
// (about one work unit per SM); the splits write fp32 partial scores
// [splits][T][E], which the dispatch kernel adds in split order.  1 = no
// split (scores written directly).  Only for bf16 routers not fused into the
// dispatch kernel.
int router_splits(const moe_config &c);
constexpr int kMaxRouterSplits = 8;

moe_status validate_config(const moe_config *cfg);
// Capacity and workspace layout.  T_cap: the tokens that set the capacity
// (all ranks' tokens for a split batch); -1 = cfg->T.
int64_t capacity_of(const moe_config *cfg, int64_t T_cap = -1);
WorkspaceLayout layout_of(const moe_config *cfg, int64_t T_cap = -1);

// One rank's share of a batch split over several ranks (see moe_dispatch.cu).
struct ShardArgs {
    int phases;                // 1: gate and statistics only; 2: placement only
    const int32_t *all_counts; // [n_ranks][E] every rank's demand counts (phase 2)
    const double *all_psum;    // [n_ranks][E] every rank's probability sums (phase 2)
    int n_ranks, rank;
    long long T_global;        // tokens over all ranks
    double *psum_out;          // [E] this rank's probability sums (phase 1)
};

// Launchers (all enqueue on `stream`; return the launch's error).
cudaError_t launch_router_simt(const moe_config &c, const void *x, const void *W_r,
                               float *logits, cudaStream_t stream);
// True when the router GEMM runs inside the dispatch kernel (W_r staged in
// shared memory: E <= 16 and E * d_model * elem_size <= 64 KiB).
bool router_fused(const moe_config &c);
// True when the down projection writes y itself (k = 1, no shared expert, bf16):
// each kept row goes straight to its token, scaled by its gate weight.
bool direct_y(const moe_config &c);
// Routing, capacity and dispatch in one cooperative kernel (see moe_dispatch.cu).
// `lpart`/`lsplit`: the split router's partial scores (null/1: scores are
// already in `logits`, or the router is fused).
// What the dispatch copies into expert order when it is not the x rows:
// E4M3 token rows src [T][row_bytes] into dst [R_max][row_bytes], and each
// token's scale scale[t] into scale_dst[row].  src and scale are written
// first, in the same forward pass, by the row quantizer (route_step).
struct GatherArgs {
    uint8_t *src;
    size_t row_bytes;
    float *scale;
    uint8_t *dst;
    float *scale_dst;
};
cudaError_t launch_dispatch(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                            const void *x, const void *W_r, bool fused, float *logits,
                            const float *lpart, int lsplit, const float *bias,
                            int32_t *topk_idx, float *topk_w, uint8_t *dropped_mask,
                            int32_t *expert_counts, int32_t *kept_counts, void *y,
                            cudaStream_t stream, const ShardArgs *shard = nullptr,
                            const GatherArgs *gather = nullptr);
// Split batch, rank without tokens: counts and sums over all ranks into
// gcount/gpsum, then the balance loss of `aux` (which points at them).
// The dispatch kernel's per-block phase stamps (MOE_TIMELINE builds):
// copy the first `words` words to host memory, or zero them.
cudaError_t dispatch_timeline_copy(uint64_t *host, size_t words);
cudaError_t dispatch_timeline_clear();
cudaError_t launch_shard_stats(const int32_t *all_counts, const double *all_psum, int n_ranks,
                               int rank, long long TK_global, int32_t *gcount, double *gpsum,
                               const AuxArgs &aux, int32_t *status, cudaStream_t stream);
cudaError_t launch_combine(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                           const float *topk_w, void *y, cudaStream_t stream);
// `aux`: the balance loss, evaluated by the first expert kernel.
cudaError_t launch_experts_simt(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                                const void *x, const void *W_gate, const void *W_up,
                                const void *W_down, const void *Ws_gate, const void *Ws_up,
                                const void *Ws_down, const AuxArgs &aux, cudaStream_t stream,
                                cudaEvent_t *ev = nullptr);

// Records ev[i] on `stream` when ev is not null.  Under stream capture the
// record becomes an external event node of the graph, so that replays
// timestamp it (a plain record would only order the capture).
inline cudaError_t record_stage(cudaEvent_t *ev, int i, cudaStream_t stream)
{
    if (!ev)
        return cudaSuccess;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t err = cudaStreamIsCapturing(stream, &cap);
    if (err != cudaSuccess)
        return err;
    if (cap == cudaStreamCaptureStatusActive)
        return cudaEventRecordWithFlags(ev[i], stream, cudaEventRecordExternal);
    return cudaEventRecord(ev[i], stream);
}

// Tensor-core (tcgen05 + TMA) paths, bf16 only.  Return cudaErrorInvalidValue
// if a tensor map cannot be encoded.  The router writes scores [T][E] to
// `out` when splits == 1, else fp32 partials [splits][T][E].
cudaError_t launch_router_tc(const moe_config &c, const void *x, const void *W_r, float *out,
                             int splits, int32_t *status, cudaStream_t stream);
// `ev` (nullable): stage events 3..6 are recorded after each GEMM.  `aux`:
// the balance loss, evaluated by the first expert kernel.
cudaError_t launch_experts_tc(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                              const void *x, const void *W_gate, const void *W_up,
                              const void *W_down, const void *Ws_gate, const void *Ws_up,
                              const void *Ws_down, void *y, const AuxArgs &aux,
                              cudaStream_t stream, cudaEvent_t *ev = nullptr);

// Dense GEMM out[rows][N] = A[rows][K] . B[N][K]^T (the latent MoE's
// projections): bf16 on the tensor cores, fp32 on CUDA cores.  Kernels
// check the status word and do nothing after an earlier failure.
cudaError_t launch_dense_tc(int rows, int N, int K, const void *A, const void *B, void *out,
                            int32_t *status, cudaStream_t stream);
cudaError_t launch_dense_simt(int rows, int N, int K, const float *A, const float *B, float *out,
                              const int32_t *status, cudaStream_t stream);

// Tensor maps for TMA (moe_gemm_tc.cu): a bf16 [rows, k] tensor in boxes of
// 64 x box_rows with 128-byte swizzle, and a byte (e4m3) [rows, k] tensor in
// boxes of 128 x box_rows with 128-byte swizzle.  false: cannot be encoded.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t k, uint32_t box_rows);
bool make_map_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t k, uint32_t box_rows);

// e4m3 expert weights with one fp32 scale per weight row (output feature):
// W[r][c] = decode(q[r][c]) * scale[r].  Shared-expert fields null when
// d_shared == 0.
struct ExpertW8 {
    const uint8_t *gate, *up, *down;        // [E,F,D], [E,F,D], [E,D,F]
    const float *gate_s, *up_s, *down_s;    // [E*F], [E*F], [E*D]
    const uint8_t *sgate, *sup, *sdown;     // [S,D], [S,D], [D,S]
    const float *sgate_s, *sup_s, *sdown_s; // [S], [S], [D]
    bool a8;                                // activations in E4M3 too (launch_experts_w8a8)
};
// The routed and shared SwiGLU experts with e4m3 weights (moe_gemm_w8.cu);
// `ev`: stage events 3..6 as in launch_experts_tc.
cudaError_t launch_experts_w8(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                              const void *x, const ExpertW8 &w, void *y, const AuxArgs &aux,
                              cudaStream_t stream, cudaEvent_t *ev = nullptr);
// Extra workspace of the E4M3-activation path (after WorkspaceLayout::total):
// E4M3 codes and fp32 row scales of the token rows, of the hidden rows (kept
// in fp32 before they are quantized), and of the shared expert's x and
// hidden rows.
struct A8Layout {
    size_t xq, xs;     // uint8[R_max][D], float[R_max]
    size_t hf;         // float[R_max][F]
    size_t hq, hsc;    // uint8[R_max][F], float[R_max]
    size_t sxq, sxs;   // uint8[T][D], float[T]         (shared expert)
    size_t shf;        // float[T][S]
    size_t shq, shs;   // uint8[T][S], float[T]
    size_t total;
};
A8Layout a8_layout_of(const moe_config &c, const WorkspaceLayout &L);
// The routed and shared SwiGLU experts with E4M3 weights and E4M3
// activations (moe_gemm_tc.cu): the token rows, and the hidden rows between
// the two GEMMs, are quantized row-wise; the tensor-core GEMMs take both
// operands in E4M3 (kind::f8f6f4) and scale the accumulator by the row's and
// the weight row's scales.  `ev`: stage events 3..6 as in launch_experts_tc.
cudaError_t launch_experts_w8a8(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                                const void *x, const ExpertW8 &w, void *y, const AuxArgs &aux,
                                cudaStream_t stream, cudaEvent_t *ev = nullptr);
// The same with the E4M3-weight kernel's unit layout (moe_gemm_w8.cu): the
// weights are the MMA's 128-row operand and up to 32 token rows of a segment
// the other, for layers with few rows per expert (w8a8_swap).
cudaError_t launch_experts_w8a8_swap(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                                     const ExpertW8 &w, void *y, const AuxArgs &aux,
                                     cudaStream_t stream, cudaEvent_t *ev = nullptr);
// True when moe_forward_w8a8 runs launch_experts_w8a8_swap: at most 64 rows
// per expert on average (T * k <= 64 * E).
bool w8a8_swap(const moe_config &c);
// q[r][c] = e4m3(W[r][c] / scale[r]), scale[r] = max_c |W[r][c]| / 448
// (moe_gemm_w8.cu).
cudaError_t launch_quantize_e4m3(long long rows, long long cols, const void *W, uint8_t *q,
                                 float *scale, cudaStream_t stream);
// Row-wise E4M3 quantization of activation rows X [rows, cols] (bf16, or
// fp32 when fp32), launched with programmatic serialization; rows_dev non-null:
// only the first min(rows, *rows_dev) rows.
cudaError_t launch_quantize_e4m3_act(long long rows, long long cols, const void *X, bool fp32,
                                     uint8_t *q, float *scale, const int32_t *rows_dev,
                                     cudaStream_t stream);

// The layer on a validated config and workspace (moe_api.cu).
moe_status forward_body(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                        const void *x, const void *W_r, const float *router_bias,
                        const void *W_gate, const void *W_up, const void *W_down,
                        const void *Ws_gate, const void *Ws_up, const void *Ws_down, void *y,
                        float *router_logits, int32_t *topk_idx, float *topk_w,
                        uint8_t *dropped_mask, int32_t *expert_counts, int32_t *kept_counts,
                        float *aux_loss, bool clear_status, cudaStream_t stream,
                        const ExpertW8 *w8 = nullptr);

int sm_count();

// One-time launch setup per device (function attributes, occupancy
// queries), safe to use from several host threads: pending(dev) is true
// until done(dev) has been called for that device.  Devices from 64 up are
// set up on every call.
class DeviceOnce {
public:
    bool pending(int dev) const
    {
        return dev < 0 || dev >= 64 || !(bits_.load(std::memory_order_acquire) & (1ull << dev));
    }
    void done(int dev)
    {
        if (dev >= 0 && dev < 64)
            bits_.fetch_or(1ull << dev, std::memory_order_release);
    }

private:
    std::atomic<uint64_t> bits_{0};
};

// Launches `kern` on `stream` with programmatic stream serialization, so
// that it may be scheduled while the previous kernel drains.  Every kernel
// launched this way calls griddep_wait() before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Asks for the largest shared-memory carveout for `kern`.  Every kernel of
// the layer runs with the same L1/shared split, so consecutive kernels do not
// wait for the SMs to be reconfigured (the GEMMs need ~200 KB per CTA).
template <typename Kern>
cudaError_t prefer_max_shared_carveout(Kern kern)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared);
}

// Stage events set by moe_set_stage_events (null = not recording).
extern std::atomic<cudaEvent_t *> g_stage_events;

}  // namespace moe
