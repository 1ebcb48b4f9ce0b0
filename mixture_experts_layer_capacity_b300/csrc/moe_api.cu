// moe_api.cu -- the C ABI of libmoe.so (declared in include/moe.h):
// argument validation, capacity, workspace layout, and the launch sequence
//   router -> gate -> scan/finalize -> scatter -> experts -> combine
// on the caller's stream, with no host synchronisation.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "moe_internal.h"

namespace moe {

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

moe_status validate_config(const moe_config *c)
{
    if (!c)
        return MOE_ERR_INVALID_ARG;
    if (c->T < 0 || c->d_model < 1 || c->d_expert < 1 || c->d_shared < 0 || c->n_experts < 1 ||
        c->top_k < 1 || c->top_k > c->n_experts)
        return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_DTYPE_BF16 && c->dtype != MOE_DTYPE_FP32)
        return MOE_ERR_INVALID_ARG;
    if (c->gating_mode < MOE_GATE_SOFTMAX_SELECTED || c->gating_mode > MOE_GATE_SIGMOID_SELECTED)
        return MOE_ERR_INVALID_ARG;
    if (c->bias_selection_only != 0 && c->bias_selection_only != 1)
        return MOE_ERR_INVALID_ARG;
    if (std::isnan(c->capacity_factor) || std::isinf(c->capacity_factor) ||
        !std::isfinite(c->aux_alpha))
        return MOE_ERR_INVALID_ARG;
    if (c->n_experts > kMaxExperts || c->top_k > kMaxTopK)
        return MOE_ERR_UNSUPPORTED;
    // widths up to 2^20 keep every workspace term (at most 4 bytes x 2^31
    // rows x 2^20) and their sum far inside size_t
    if (c->d_model > kMaxWidth || c->d_expert > kMaxWidth || c->d_shared > kMaxWidth)
        return MOE_ERR_UNSUPPORTED;
    if ((long long)c->T * c->top_k >= (1ll << 31))
        return MOE_ERR_UNSUPPORTED;
    if (c->dtype == MOE_DTYPE_BF16) {
        if (c->d_model % 64 || c->d_expert % 64 || c->d_shared % 64)
            return MOE_ERR_UNSUPPORTED;
    } else {
        // the SIMT path launches one grid row per 8 output rows
        if ((long long)c->T * c->top_k > 500000)
            return MOE_ERR_UNSUPPORTED;
    }
    return MOE_OK;
}

// C = ceil(capacity_factor * T * k / E) in double; -1 when dropless.
int64_t capacity_of(const moe_config *c, int64_t T_cap)
{
    if (!(c->capacity_factor > 0.0f))
        return -1;
    const int64_t T = T_cap < 0 ? c->T : T_cap;
    const double cap = std::ceil((double)c->capacity_factor * (double)(T * c->top_k) /
                                 (double)c->n_experts);
    // a capacity beyond int64 exceeds every expert's demand (at most T*k),
    // so it keeps every assignment, as INT64_MAX does
    return cap >= 9.2e18 ? INT64_MAX : (int64_t)cap;
}

WorkspaceLayout layout_of(const moe_config *c, int64_t T_cap)
{
    WorkspaceLayout L{};
    const int64_t T = c->T, E = c->n_experts, k = c->top_k;
    const int64_t D = c->d_model, F = c->d_expert, S = c->d_shared;
    const size_t esz = c->dtype == MOE_DTYPE_BF16 ? 2 : 4;
    L.nchunk = (int)std::max<int64_t>(std::min<int64_t>(T, kMaxDispatchBlocks),
                                     (T + kChunk - 1) / kChunk);
    L.C = capacity_of(c, T_cap);
    const int64_t TK = T * k;
    L.R_max = (L.C < 0 || L.C >= TK) ? TK : std::min<int64_t>(TK, E * L.C);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 1024);
        return o;
    };
    L.status = take(64);
    L.bcount = take(sizeof(int32_t) * E * L.nchunk);
    L.ppart = take(sizeof(float) * E * L.nchunk);
    L.rank = take(sizeof(int32_t) * TK);
    L.psum = take(sizeof(double) * E);
    L.gcount = take(sizeof(int32_t) * E);
    L.seg_off = take(sizeof(int32_t) * (E + 1));
    L.mtile = take(sizeof(int32_t) * (E + 1));
    L.row_of = take(sizeof(int32_t) * TK);
    L.row_tok = take(sizeof(int32_t) * L.R_max);
    L.row_w = take(sizeof(float) * L.R_max);
    L.x_perm = take(esz * L.R_max * D);
    L.h = take(esz * L.R_max * F);
    L.z = take(esz * L.R_max * D);
    L.hs = take(S > 0 ? esz * T * S : 0);
    const int zsplit = S > 0 ? shared_down_splits(*c) : 1;
    L.zs = take(S > 0 ? (zsplit > 1 ? sizeof(float) * zsplit * T * D : esz * T * D) : 0);
    const int lsplit = router_splits(*c);
    L.lpart = take(lsplit > 1 ? sizeof(float) * lsplit * T * E : 0);
    L.total = off;
    return L;
}

A8Layout a8_layout_of(const moe_config &c, const WorkspaceLayout &L)
{
    A8Layout A{};
    const int64_t T = c.T, D = c.d_model, F = c.d_expert, S = c.d_shared, R = L.R_max;
    size_t off = L.total;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 1024);
        return o;
    };
    A.xq = take((size_t)R * D);
    A.xs = take(sizeof(float) * R);
    A.hf = take(sizeof(float) * R * F);
    A.hq = take((size_t)R * F);
    A.hsc = take(sizeof(float) * R);
    A.sxq = take((size_t)T * D);
    A.sxs = take(sizeof(float) * T);
    A.shf = take(S > 0 ? sizeof(float) * T * S : 0);
    A.shq = take(S > 0 ? (size_t)T * S : 0);
    A.shs = take(S > 0 ? sizeof(float) * T : 0);
    A.total = off;
    return A;
}

bool w8a8_swap(const moe_config &c)
{
    return (long long)c.T * c.top_k <= 64LL * c.n_experts;
}

int shared_down_splits(const moe_config &c)
{
    if (!plan_of(c).shared_fused)
        return 1;
    const int s = (c.d_shared + c.d_expert - 1) / c.d_expert;
    return std::max(1, std::min(s, kMaxSharedSplits));
}

LaunchPlan plan_of(const moe_config &c)
{
    LaunchPlan pl{};
    const bool bf16 = c.dtype == MOE_DTYPE_BF16;
    pl.router_fused = router_fused(c);
    pl.direct_y = bf16 && direct_y(c);
    const long long routed_rows = (long long)c.T * c.top_k;
    pl.pair_routed = bf16 && routed_rows >= kPairMinRows &&
                     routed_rows >= 2LL * 2 * kTileM * c.n_experts;
    pl.pair_shared = bf16 && c.d_shared > 0 && c.T >= kPairMinRows / 4;
    pl.shared_fused = bf16 && c.d_shared > 0 && !pl.pair_routed && !pl.pair_shared;
    // 256-row pair tiles over whole segments would pad about E * 128 rows;
    // each segment's remainder runs instead as swap units (weights as the
    // 256-row operand, the remaining token rows rounded up to 32 as the
    // other) interleaved with the full tiles of the same launch
    pl.pair_tails = pl.pair_routed;
    pl.router_splits = router_splits(c);
    return pl;
}

int router_splits(const moe_config &c)
{
    if (c.dtype != MOE_DTYPE_BF16 || c.T <= 0 || c.T >= 512 || router_fused(c))
        return 1;
    const long long E = c.n_experts;
    const long long bn = E <= 16 ? 16 : E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256;
    const long long tiles = ((c.T + kTileM - 1) / kTileM) * ((E + bn - 1) / bn);
    const long long nk = c.d_model / 64;
    constexpr long long kNominalSms = 148;
    long long s = std::min<long long>(kNominalSms / tiles, nk / 4);  // >= 4 k-steps per split
    return (int)std::max<long long>(1, std::min<long long>(s, kMaxRouterSplits));
}

std::atomic<cudaEvent_t *> g_stage_events{nullptr};

int sm_count()
{
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 1;
    const bool slot = dev >= 0 && dev < 64;
    if (slot) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0)
            return c;
    }
    int n = 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 1;
    if (slot)
        cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_workspace_size(const moe_config *cfg, size_t *bytes)
{
    if (!bytes)
        return MOE_ERR_INVALID_ARG;
    const moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    *bytes = layout_of(cfg).total;
    return MOE_OK;
}

int64_t moe_capacity(const moe_config *cfg)
{
    if (validate_config(cfg) != MOE_OK)
        return -1;
    return capacity_of(cfg);
}

moe_status moe_launch_plan(const moe_config *cfg, int32_t *flags)
{
    if (!flags)
        return MOE_ERR_INVALID_ARG;
    const moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    const LaunchPlan pl = plan_of(*cfg);
    *flags = (pl.router_fused ? MOE_PLAN_ROUTER_FUSED : 0) | (pl.direct_y ? MOE_PLAN_DIRECT_Y : 0) |
             (pl.pair_routed ? MOE_PLAN_PAIR_ROUTED : 0) |
             (pl.pair_shared ? MOE_PLAN_PAIR_SHARED : 0) |
             (pl.shared_fused ? MOE_PLAN_SHARED_FUSED : 0) |
             (pl.pair_tails ? MOE_PLAN_PAIR_TAILS : 0) |
             (w8a8_swap(*cfg) ? MOE_PLAN_W8A8_SWAP : 0);
    return MOE_OK;
}

}  // extern "C"

namespace moe {

namespace {

bool cuda_ok(cudaError_t e) { return e == cudaSuccess; }

// Router scores (small routers run inside the dispatch kernel instead), then
// the dispatch kernel: gating, demand counts, capacity, segments and the
// gather of x into expert order -- or, for one rank of a split batch, the
// part of it that `shard->phases` names.
moe_status route_step(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws, const void *x,
                      const void *W_r, const float *router_bias, float *router_logits,
                      int32_t *topk_idx, float *topk_w, uint8_t *dropped_mask,
                      int32_t *expert_counts, int32_t *kept_counts, void *y,
                      const ShardArgs *shard, cudaEvent_t *ev, cudaStream_t stream,
                      const GatherArgs *gather = nullptr)
{
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    const bool gate = !shard || (shard->phases & 1);
    const bool fused = gate && router_fused(c) && aligned16(x) && aligned16(W_r);
    const int lsplit = fused || !gate ? 1 : router_splits(c);
    float *lpart = lsplit > 1 ? reinterpret_cast<float *>(ws + L.lpart) : nullptr;
    if (!cuda_ok(record_stage(ev, 0, stream)))
        return MOE_ERR_CUDA;
    cudaError_t err = cudaSuccess;
    // E4M3 token rows for the gather: every token row quantized once
    if (gather)
        err = launch_quantize_e4m3_act(c.T, c.d_model, x, false, gather->src, gather->scale,
                                       nullptr, stream);
    if (!cuda_ok(err))
        return MOE_ERR_CUDA;
    if (gate && !fused) {
        if (c.dtype == MOE_DTYPE_BF16)
            err = launch_router_tc(c, x, W_r, lsplit > 1 ? lpart : router_logits, lsplit, status,
                                   stream);
        else
            err = launch_router_simt(c, x, W_r, router_logits, stream);
    }
    if (!cuda_ok(err) || !cuda_ok(record_stage(ev, 1, stream)))
        return MOE_ERR_CUDA;
    if (!cuda_ok(launch_dispatch(c, L, ws, x, W_r, fused, router_logits, lpart, lsplit,
                                 router_bias, topk_idx, topk_w, dropped_mask, expert_counts,
                                 kept_counts, y, stream, shard, gather)) ||
        !cuda_ok(record_stage(ev, 2, stream)))
        return MOE_ERR_CUDA;
    return MOE_OK;
}

// The experts (routed segments and the shared expert; the first expert
// kernel also evaluates the balance loss of `aux`) and the weighted combine,
// unless the down projection already wrote y.
moe_status expert_step(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws, const void *x,
                       const void *W_gate, const void *W_up, const void *W_down,
                       const void *Ws_gate, const void *Ws_up, const void *Ws_down, void *y,
                       const float *topk_w, const AuxArgs &aux, cudaEvent_t *ev,
                       cudaStream_t stream, const ExpertW8 *w8)
{
    cudaError_t err;
    if (w8 && w8->a8)
        err = launch_experts_w8a8(c, L, ws, x, *w8, y, aux, stream, ev);
    else if (w8)
        err = launch_experts_w8(c, L, ws, x, *w8, y, aux, stream, ev);
    else if (c.dtype == MOE_DTYPE_BF16)
        err = launch_experts_tc(c, L, ws, x, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, y,
                                aux, stream, ev);
    else
        err = launch_experts_simt(c, L, ws, x, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down,
                                  aux, stream, ev);
    if (!cuda_ok(err))
        return MOE_ERR_CUDA;
    if (!(direct_y(c) && c.dtype == MOE_DTYPE_BF16)) {
        if (!cuda_ok(launch_combine(c, L, ws, topk_w, y, stream)))
            return MOE_ERR_CUDA;
    }
    if (!cuda_ok(record_stage(ev, 7, stream)))
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace

// The layer on a validated config and workspace.  clear_status: zero the
// status word and counters first (otherwise the caller already has, on the
// same stream, and an earlier kernel's error is kept).
moe_status forward_body(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                        const void *x, const void *W_r, const float *router_bias,
                        const void *W_gate, const void *W_up, const void *W_down,
                        const void *Ws_gate, const void *Ws_up, const void *Ws_down, void *y,
                        float *router_logits, int32_t *topk_idx, float *topk_w,
                        uint8_t *dropped_mask, int32_t *expert_counts, int32_t *kept_counts,
                        float *aux_loss, bool clear_status, cudaStream_t stream,
                        const ExpertW8 *w8)
{
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    const int E = c.n_experts;
    if (clear_status && !cuda_ok(cudaMemsetAsync(status, 0, 64, stream)))
        return MOE_ERR_CUDA;
    if (c.T == 0) {
        if (!cuda_ok(cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * E, stream)) ||
            !cuda_ok(cudaMemsetAsync(kept_counts, 0, sizeof(int32_t) * E, stream)) ||
            !cuda_ok(cudaMemsetAsync(aux_loss, 0, sizeof(float), stream)))
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    cudaEvent_t *ev = g_stage_events.load();
    // E4M3 activations: every token row is quantized once, and the dispatch
    // gathers its codes (and scale) into expert order instead of the bf16 row
    GatherArgs g{};
    if (w8 && w8->a8) {
        const A8Layout A = a8_layout_of(c, L);
        g.src = ws + A.sxq;
        g.row_bytes = (size_t)c.d_model;
        g.scale = reinterpret_cast<float *>(ws + A.sxs);
        g.dst = ws + A.xq;
        g.scale_dst = reinterpret_cast<float *>(ws + A.xs);
    }
    moe_status st = route_step(c, L, ws, x, W_r, router_bias, router_logits, topk_idx, topk_w,
                               dropped_mask, expert_counts, kept_counts, y, nullptr, ev, stream,
                               w8 && w8->a8 ? &g : nullptr);
    if (st != MOE_OK)
        return st;
    AuxArgs aux;
    aux.psum = reinterpret_cast<const double *>(ws + L.psum);
    aux.counts = expert_counts;
    aux.out = aux_loss;
    aux.E = E;
    aux.T = c.T;
    aux.k = c.top_k;
    aux.alpha = c.aux_alpha;
    return expert_step(c, L, ws, x, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, y, topk_w,
                       aux, ev, stream, w8);
}

}  // namespace moe

extern "C" {

moe_status moe_forward(const moe_config *cfg, const void *x, const void *W_r,
                       const float *router_bias, const void *W_gate, const void *W_up,
                       const void *W_down, const void *Ws_gate, const void *Ws_up,
                       const void *Ws_down, void *y, float *router_logits, int32_t *topk_idx,
                       float *topk_w, uint8_t *dropped_mask, int32_t *expert_counts,
                       int32_t *kept_counts, float *aux_loss, void *workspace,
                       size_t workspace_bytes, cudaStream_t stream)
{
    moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    const moe_config &c = *cfg;
    if (!expert_counts || !kept_counts || !aux_loss)
        return MOE_ERR_INVALID_ARG;
    // with T == 0 nothing per token or per weight is touched (empty tensors
    // may have null data pointers)
    if (c.T > 0) {
        if (!x || !W_r || !W_gate || !W_up || !W_down || !y || !router_logits || !topk_idx ||
            !topk_w || !dropped_mask)
            return MOE_ERR_INVALID_ARG;
        if (c.d_shared > 0 && (!Ws_gate || !Ws_up || !Ws_down))
            return MOE_ERR_INVALID_ARG;
    }
    const WorkspaceLayout L = layout_of(cfg);
    if (!workspace || workspace_bytes < L.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MOE_ERR_WORKSPACE;
    if (c.dtype == MOE_DTYPE_BF16) {
        // tensor-map bases and 16-byte vector accesses
        if (!aligned16(x) || !aligned16(W_r) || !aligned16(W_gate) || !aligned16(W_up) ||
            !aligned16(W_down) || !aligned16(y) ||
            (c.d_shared > 0 && (!aligned16(Ws_gate) || !aligned16(Ws_up) || !aligned16(Ws_down))))
            return MOE_ERR_INVALID_ARG;
    }
    return forward_body(c, L, static_cast<uint8_t *>(workspace), x, W_r, router_bias, W_gate,
                        W_up, W_down, Ws_gate, Ws_up, Ws_down, y, router_logits, topk_idx,
                        topk_w, dropped_mask, expert_counts, kept_counts, aux_loss, true,
                        stream);
}

// Latent layout: the layer's own workspace, then x_lat [T][L] and y_lat [T][L].
static bool latent_layout(const moe_config *cfg, int32_t d_outer, size_t *x_lat, size_t *y_lat,
                          size_t *total)
{
    if (validate_config(cfg) != MOE_OK || d_outer < 1 || d_outer > kMaxWidth)
        return false;
    if (cfg->dtype == MOE_DTYPE_BF16 && d_outer % 64)
        return false;
    const size_t esz = cfg->dtype == MOE_DTYPE_BF16 ? 2 : 4;
    const size_t lat = esz * (size_t)cfg->T * (size_t)cfg->d_model;
    *x_lat = align_up(layout_of(cfg).total, 1024);
    *y_lat = align_up(*x_lat + lat, 1024);
    *total = align_up(*y_lat + lat, 1024);
    return true;
}

moe_status moe_latent_workspace_size(const moe_config *cfg, int32_t d_outer, size_t *bytes)
{
    if (!bytes)
        return MOE_ERR_INVALID_ARG;
    const moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    size_t xo, yo, total;
    if (!latent_layout(cfg, d_outer, &xo, &yo, &total))
        return d_outer < 1 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
    *bytes = total;
    return MOE_OK;
}

moe_status moe_latent_offsets(const moe_config *cfg, int32_t d_outer, size_t *x_lat_offset,
                              size_t *y_lat_offset)
{
    if (!x_lat_offset || !y_lat_offset)
        return MOE_ERR_INVALID_ARG;
    const moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    size_t xo, yo, total;
    if (!latent_layout(cfg, d_outer, &xo, &yo, &total))
        return d_outer < 1 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
    *x_lat_offset = xo;
    *y_lat_offset = yo;
    return MOE_OK;
}

moe_status moe_latent_forward(const moe_config *cfg, int32_t d_outer, const void *x,
                              const void *W_in, const void *W_out, const void *W_r,
                              const float *router_bias, const void *W_gate, const void *W_up,
                              const void *W_down, const void *Ws_gate, const void *Ws_up,
                              const void *Ws_down, void *y, float *router_logits,
                              int32_t *topk_idx, float *topk_w, uint8_t *dropped_mask,
                              int32_t *expert_counts, int32_t *kept_counts, float *aux_loss,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    const moe_config &c = *cfg;
    size_t xo, yo, total;
    if (!latent_layout(cfg, d_outer, &xo, &yo, &total))
        return d_outer < 1 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED;
    if (!expert_counts || !kept_counts || !aux_loss)
        return MOE_ERR_INVALID_ARG;
    if (c.T > 0) {
        if (!x || !W_in || !W_out || !W_r || !W_gate || !W_up || !W_down || !y ||
            !router_logits || !topk_idx || !topk_w || !dropped_mask)
            return MOE_ERR_INVALID_ARG;
        if (c.d_shared > 0 && (!Ws_gate || !Ws_up || !Ws_down))
            return MOE_ERR_INVALID_ARG;
    }
    if (!workspace || workspace_bytes < total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MOE_ERR_WORKSPACE;
    if (c.dtype == MOE_DTYPE_BF16) {
        if (!aligned16(x) || !aligned16(W_in) || !aligned16(W_out) || !aligned16(W_r) ||
            !aligned16(W_gate) || !aligned16(W_up) || !aligned16(W_down) || !aligned16(y) ||
            (c.d_shared > 0 && (!aligned16(Ws_gate) || !aligned16(Ws_up) || !aligned16(Ws_down))))
            return MOE_ERR_INVALID_ARG;
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const WorkspaceLayout L = layout_of(cfg);
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    if (cudaMemsetAsync(status, 0, 64, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    void *x_lat = ws + xo, *y_lat = ws + yo;
    const int T = c.T, Ld = c.d_model;
    // x_lat = x W_in^T
    cudaError_t err = c.dtype == MOE_DTYPE_BF16
                          ? launch_dense_tc(T, Ld, d_outer, x, W_in, x_lat, status, stream)
                          : launch_dense_simt(T, Ld, d_outer, static_cast<const float *>(x),
                                              static_cast<const float *>(W_in),
                                              static_cast<float *>(x_lat), status, stream);
    if (err != cudaSuccess)
        return MOE_ERR_CUDA;
    // the layer at the latent width
    st = forward_body(c, L, ws, x_lat, W_r, router_bias, W_gate, W_up, W_down, Ws_gate, Ws_up,
                      Ws_down, y_lat, router_logits, topk_idx, topk_w, dropped_mask,
                      expert_counts, kept_counts, aux_loss, false, stream);
    if (st != MOE_OK || T == 0)
        return st;
    // y = y_lat W_out^T
    err = c.dtype == MOE_DTYPE_BF16
              ? launch_dense_tc(T, d_outer, Ld, y_lat, W_out, y, status, stream)
              : launch_dense_simt(T, d_outer, Ld, static_cast<const float *>(y_lat),
                                  static_cast<const float *>(W_out), static_cast<float *>(y),
                                  status, stream);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---- one rank's share of a batch split over several ranks

static moe_status validate_shard(const moe_config *cfg, int64_t T_global)
{
    const moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    if (T_global < cfg->T)
        return MOE_ERR_INVALID_ARG;
    if (T_global * cfg->top_k >= (1ll << 31))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status moe_sharded_workspace_size(const moe_config *cfg, int64_t T_global, size_t *bytes)
{
    if (!bytes)
        return MOE_ERR_INVALID_ARG;
    const moe_status st = validate_shard(cfg, T_global);
    if (st != MOE_OK)
        return st;
    *bytes = layout_of(cfg, T_global).total;
    return MOE_OK;
}

moe_status moe_sharded_route(const moe_config *cfg, int64_t T_global, const void *x,
                             const void *W_r, const float *router_bias, float *router_logits,
                             int32_t *topk_idx, float *topk_w, int32_t *expert_counts,
                             double *prob_sums, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream)
{
    moe_status st = validate_shard(cfg, T_global);
    if (st != MOE_OK)
        return st;
    const moe_config &c = *cfg;
    if (!expert_counts || !prob_sums)
        return MOE_ERR_INVALID_ARG;
    if (c.T > 0 && (!x || !W_r || !router_logits || !topk_idx || !topk_w))
        return MOE_ERR_INVALID_ARG;
    const WorkspaceLayout L = layout_of(cfg, T_global);
    if (!workspace || workspace_bytes < L.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MOE_ERR_WORKSPACE;
    if (c.dtype == MOE_DTYPE_BF16 && (!aligned16(x) || !aligned16(W_r)))
        return MOE_ERR_INVALID_ARG;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (!cuda_ok(cudaMemsetAsync(ws + L.status, 0, 64, stream)))
        return MOE_ERR_CUDA;
    if (c.T == 0) {
        if (!cuda_ok(cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * c.n_experts, stream)) ||
            !cuda_ok(cudaMemsetAsync(prob_sums, 0, sizeof(double) * c.n_experts, stream)))
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    ShardArgs sh{};
    sh.phases = 1;
    sh.n_ranks = 1;
    sh.T_global = T_global;
    sh.psum_out = prob_sums;
    return route_step(c, L, ws, x, W_r, router_bias, router_logits, topk_idx, topk_w, nullptr,
                      expert_counts, nullptr, nullptr, &sh, nullptr, stream);
}

moe_status moe_sharded_finish(const moe_config *cfg, int64_t T_global, int32_t n_ranks,
                              int32_t rank, const int32_t *all_expert_counts,
                              const double *all_prob_sums, const void *x, const void *W_gate,
                              const void *W_up, const void *W_down, const void *Ws_gate,
                              const void *Ws_up, const void *Ws_down, const int32_t *topk_idx,
                              const float *topk_w, void *y, uint8_t *dropped_mask,
                              int32_t *kept_counts, float *aux_loss, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream)
{
    moe_status st = validate_shard(cfg, T_global);
    if (st != MOE_OK)
        return st;
    const moe_config &c = *cfg;
    if (n_ranks < 1 || rank < 0 || rank >= n_ranks || !kept_counts || !aux_loss)
        return MOE_ERR_INVALID_ARG;
    if (T_global > 0 && (!all_expert_counts || !all_prob_sums))
        return MOE_ERR_INVALID_ARG;
    if (c.T > 0) {
        if (!x || !W_gate || !W_up || !W_down || !y || !topk_idx || !topk_w || !dropped_mask)
            return MOE_ERR_INVALID_ARG;
        if (c.d_shared > 0 && (!Ws_gate || !Ws_up || !Ws_down))
            return MOE_ERR_INVALID_ARG;
    }
    const WorkspaceLayout L = layout_of(cfg, T_global);
    if (!workspace || workspace_bytes < L.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MOE_ERR_WORKSPACE;
    if (c.dtype == MOE_DTYPE_BF16) {
        if (!aligned16(x) || !aligned16(W_gate) || !aligned16(W_up) || !aligned16(W_down) ||
            !aligned16(y) ||
            (c.d_shared > 0 && (!aligned16(Ws_gate) || !aligned16(Ws_up) || !aligned16(Ws_down))))
            return MOE_ERR_INVALID_ARG;
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int E = c.n_experts;
    if (!cuda_ok(cudaMemsetAsync(kept_counts, 0, sizeof(int32_t) * E, stream)))
        return MOE_ERR_CUDA;
    if (T_global == 0)
        return cuda_ok(cudaMemsetAsync(aux_loss, 0, sizeof(float), stream)) ? MOE_OK
                                                                             : MOE_ERR_CUDA;
    AuxArgs aux;
    aux.psum = reinterpret_cast<const double *>(ws + L.psum);
    aux.counts = reinterpret_cast<const int32_t *>(ws + L.gcount);
    aux.out = aux_loss;
    aux.E = E;
    aux.T = (int)T_global;
    aux.k = c.top_k;
    aux.alpha = c.aux_alpha;
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    if (c.T == 0) {
        // nothing routed here: only the statistics over all ranks and the loss
        return cuda_ok(launch_shard_stats(all_expert_counts, all_prob_sums, n_ranks, rank,
                                          T_global * c.top_k,
                                          reinterpret_cast<int32_t *>(ws + L.gcount),
                                          reinterpret_cast<double *>(ws + L.psum), aux, status,
                                          stream))
                   ? MOE_OK
                   : MOE_ERR_CUDA;
    }
    ShardArgs sh{};
    sh.phases = 2;
    sh.all_counts = all_expert_counts;
    sh.all_psum = all_prob_sums;
    sh.n_ranks = n_ranks;
    sh.rank = rank;
    sh.T_global = T_global;
    // the placement phase only reads the gate's indices and weights
    st = route_step(c, L, ws, x, nullptr, nullptr, nullptr, const_cast<int32_t *>(topk_idx),
                    const_cast<float *>(topk_w), dropped_mask, nullptr, kept_counts, y, &sh,
                    nullptr, stream);
    if (st != MOE_OK)
        return st;
    return expert_step(c, L, ws, x, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, y, topk_w,
                       aux, nullptr, stream, nullptr);
}

// ---- e4m3 expert weights

moe_status moe_quantize_e4m3_rows(int64_t rows, int64_t cols, const void *W, uint8_t *q,
                                  float *scale, cudaStream_t stream)
{
    if (rows < 0 || cols < 1 || cols % 16 || rows * cols >= (1ll << 40))
        return MOE_ERR_INVALID_ARG;
    if (rows == 0)
        return MOE_OK;
    if (!W || !q || !scale || !aligned16(W) || !aligned16(q) ||
        (reinterpret_cast<uintptr_t>(scale) & 3u))
        return MOE_ERR_INVALID_ARG;
    return cuda_ok(launch_quantize_e4m3(rows, cols, W, q, scale, stream)) ? MOE_OK : MOE_ERR_CUDA;
}

namespace {

// Shared argument checks and the call of the E4M3-weight forward passes.
moe_status forward_e4m3(const moe_config *cfg, const void *x, const void *W_r,
                        const float *router_bias, const uint8_t *W_gate_q,
                        const float *W_gate_scale, const uint8_t *W_up_q, const float *W_up_scale,
                        const uint8_t *W_down_q, const float *W_down_scale,
                        const uint8_t *Ws_gate_q, const float *Ws_gate_scale,
                        const uint8_t *Ws_up_q, const float *Ws_up_scale,
                        const uint8_t *Ws_down_q, const float *Ws_down_scale, void *y,
                        float *router_logits, int32_t *topk_idx, float *topk_w,
                        uint8_t *dropped_mask, int32_t *expert_counts, int32_t *kept_counts,
                        float *aux_loss, void *workspace, size_t workspace_bytes,
                        cudaStream_t stream, bool a8)
{
    moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    const moe_config &c = *cfg;
    if (c.dtype != MOE_DTYPE_BF16)
        return MOE_ERR_UNSUPPORTED;
    // E4M3 operands: 128-element reduction steps, and the shared down
    // projection is cut into as many pieces as for the bf16 layer; with
    // d_expert = 64 a piece could get no step
    if (a8 && c.d_shared > 0 && c.d_expert < 128)
        return MOE_ERR_UNSUPPORTED;
    if (!expert_counts || !kept_counts || !aux_loss)
        return MOE_ERR_INVALID_ARG;
    const bool shared = c.d_shared > 0;
    if (c.T > 0) {
        if (!x || !W_r || !W_gate_q || !W_gate_scale || !W_up_q || !W_up_scale || !W_down_q ||
            !W_down_scale || !y || !router_logits || !topk_idx || !topk_w || !dropped_mask)
            return MOE_ERR_INVALID_ARG;
        if (shared && (!Ws_gate_q || !Ws_gate_scale || !Ws_up_q || !Ws_up_scale || !Ws_down_q ||
                       !Ws_down_scale))
            return MOE_ERR_INVALID_ARG;
        if (!aligned16(x) || !aligned16(W_r) || !aligned16(y) || !aligned16(W_gate_q) ||
            !aligned16(W_up_q) || !aligned16(W_down_q) ||
            (shared && (!aligned16(Ws_gate_q) || !aligned16(Ws_up_q) || !aligned16(Ws_down_q))))
            return MOE_ERR_INVALID_ARG;
    }
    const WorkspaceLayout L = layout_of(cfg);
    const size_t need = a8 ? a8_layout_of(c, L).total : L.total;
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MOE_ERR_WORKSPACE;
    ExpertW8 w{};
    w.gate = W_gate_q;
    w.up = W_up_q;
    w.down = W_down_q;
    w.gate_s = W_gate_scale;
    w.up_s = W_up_scale;
    w.down_s = W_down_scale;
    w.sgate = Ws_gate_q;
    w.sup = Ws_up_q;
    w.sdown = Ws_down_q;
    w.sgate_s = Ws_gate_scale;
    w.sup_s = Ws_up_scale;
    w.sdown_s = Ws_down_scale;
    w.a8 = a8;
    return forward_body(c, L, static_cast<uint8_t *>(workspace), x, W_r, router_bias, nullptr,
                        nullptr, nullptr, nullptr, nullptr, nullptr, y, router_logits, topk_idx,
                        topk_w, dropped_mask, expert_counts, kept_counts, aux_loss, true, stream,
                        &w);
}

}  // namespace

moe_status moe_forward_w8(const moe_config *cfg, const void *x, const void *W_r,
                          const float *router_bias, const uint8_t *W_gate_q,
                          const float *W_gate_scale, const uint8_t *W_up_q,
                          const float *W_up_scale, const uint8_t *W_down_q,
                          const float *W_down_scale, const uint8_t *Ws_gate_q,
                          const float *Ws_gate_scale, const uint8_t *Ws_up_q,
                          const float *Ws_up_scale, const uint8_t *Ws_down_q,
                          const float *Ws_down_scale, void *y, float *router_logits,
                          int32_t *topk_idx, float *topk_w, uint8_t *dropped_mask,
                          int32_t *expert_counts, int32_t *kept_counts, float *aux_loss,
                          void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return forward_e4m3(cfg, x, W_r, router_bias, W_gate_q, W_gate_scale, W_up_q, W_up_scale,
                        W_down_q, W_down_scale, Ws_gate_q, Ws_gate_scale, Ws_up_q, Ws_up_scale,
                        Ws_down_q, Ws_down_scale, y, router_logits, topk_idx, topk_w,
                        dropped_mask, expert_counts, kept_counts, aux_loss, workspace,
                        workspace_bytes, stream, false);
}

moe_status moe_w8a8_workspace_size(const moe_config *cfg, size_t *bytes)
{
    if (!bytes)
        return MOE_ERR_INVALID_ARG;
    const moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    if (cfg->dtype != MOE_DTYPE_BF16)
        return MOE_ERR_UNSUPPORTED;
    *bytes = a8_layout_of(*cfg, layout_of(cfg)).total;
    return MOE_OK;
}

moe_status moe_w8a8_offsets(const moe_config *cfg, size_t *x_codes, size_t *x_scales,
                            size_t *h_values, size_t *h_codes, size_t *h_scales)
{
    if (!x_codes || !x_scales || !h_values || !h_codes || !h_scales)
        return MOE_ERR_INVALID_ARG;
    const moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    if (cfg->dtype != MOE_DTYPE_BF16)
        return MOE_ERR_UNSUPPORTED;
    const A8Layout A = a8_layout_of(*cfg, layout_of(cfg));
    *x_codes = A.xq;
    *x_scales = A.xs;
    *h_values = A.hf;
    *h_codes = A.hq;
    *h_scales = A.hsc;
    return MOE_OK;
}

moe_status moe_forward_w8a8(const moe_config *cfg, const void *x, const void *W_r,
                            const float *router_bias, const uint8_t *W_gate_q,
                            const float *W_gate_scale, const uint8_t *W_up_q,
                            const float *W_up_scale, const uint8_t *W_down_q,
                            const float *W_down_scale, const uint8_t *Ws_gate_q,
                            const float *Ws_gate_scale, const uint8_t *Ws_up_q,
                            const float *Ws_up_scale, const uint8_t *Ws_down_q,
                            const float *Ws_down_scale, void *y, float *router_logits,
                            int32_t *topk_idx, float *topk_w, uint8_t *dropped_mask,
                            int32_t *expert_counts, int32_t *kept_counts, float *aux_loss,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    return forward_e4m3(cfg, x, W_r, router_bias, W_gate_q, W_gate_scale, W_up_q, W_up_scale,
                        W_down_q, W_down_scale, Ws_gate_q, Ws_gate_scale, Ws_up_q, Ws_up_scale,
                        Ws_down_q, Ws_down_scale, y, router_logits, topk_idx, topk_w,
                        dropped_mask, expert_counts, kept_counts, aux_loss, workspace,
                        workspace_bytes, stream, true);
}

moe_status moe_read_device_status(const moe_config *cfg, const void *workspace,
                                  cudaStream_t stream, int32_t *code)
{
    const moe_status st = validate_config(cfg);
    if (st != MOE_OK)
        return st;
    if (!workspace || !code)
        return MOE_ERR_INVALID_ARG;
    const WorkspaceLayout L = layout_of(cfg);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, static_cast<const uint8_t *>(workspace) + L.status, sizeof(v),
                        cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    *code = v;
    return v == MOE_DEVICE_OK ? MOE_OK : MOE_ERR_DEVICE_STATUS;
}

moe_status moe_set_stage_events(cudaEvent_t *events, int n_events)
{
    if (events && n_events != MOE_NUM_STAGE_EVENTS)
        return MOE_ERR_INVALID_ARG;
    g_stage_events.store(events);
    return MOE_OK;
}

const char *moe_status_string(moe_status s)
{
    switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: unsupported shape or option";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small or misaligned";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_DEVICE_STATUS: return "MOE_ERR_DEVICE_STATUS: a kernel reported an error";
    }
    return "unknown moe_status";
}

}  // extern "C"
