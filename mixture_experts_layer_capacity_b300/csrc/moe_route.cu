// moe_route.cu -- router scores and gating.
//
//   router_simt: scores on SIMT cores, one warp per (token, expert), for
//                small T and fp32 (large bf16 batches use the tensor-core
//                router in moe_gemm_tc.cu);
//   gate:        one block per chunk of 32 tokens, one warp per token:
//                (optionally the router GEMM itself, with W_r staged in shared
//                memory), softmax over all E, top-k with the lower index first
//                on equal scores, gate weights, per-chunk expert histograms,
//                per-chunk probability sums, and the rank of each assignment
//                among its chunk's tokens (for token-order capacity).
//
// Sources: "Mixture of Experts: More Parameters, Same FLOPs" ('The router':
// scores x W_r, softmax, top-k, renormalised weights); "Mixture of Experts"
// (module 17), 17.2 (softmax over the selected vs over all experts) and 17.4
// (f_i and P_i of the balance loss); "Mixture of experts" (frontiers track),
// gate equation of 'Where the experts live'.
#include <cfloat>
#include <climits>
#include <cuda_bf16.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

// ------------------------------------------------------------- router (SIMT)
// One warp per (token, expert): s[t][e] = sum_d x[t][d] * W_r[e][d], fp32
// accumulation.  bf16 rows are read as 16-byte vectors (D % 8 == 0).
__global__ void router_simt_bf16_kernel(const __nv_bfloat16 *__restrict__ x,
                                        const __nv_bfloat16 *__restrict__ W,
                                        float *__restrict__ logits, int T, int D, int E)
{
    griddep_wait();
    griddep_launch_dependents();
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= (long long)T * E)
        return;
    const int t = (int)(wid / E), e = (int)(wid % E);
    const uint4 *a = reinterpret_cast<const uint4 *>(x + (size_t)t * D);
    const uint4 *b = reinterpret_cast<const uint4 *>(W + (size_t)e * D);
    const int nv = D / 8;
    float acc = 0.f;
    for (int v = lane; v < nv; v += 32) {
        uint4 av = __ldg(a + v), bv = __ldg(b + v);
        const __nv_bfloat162 *ah = reinterpret_cast<const __nv_bfloat162 *>(&av);
        const __nv_bfloat162 *bh = reinterpret_cast<const __nv_bfloat162 *>(&bv);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 af = __bfloat1622float2(ah[i]), bf = __bfloat1622float2(bh[i]);
            acc = fmaf(af.x, bf.x, acc);
            acc = fmaf(af.y, bf.y, acc);
        }
    }
    acc = warp_sum_bcast(acc);
    if (lane == 0)
        logits[(size_t)t * E + e] = acc;
}

__global__ void router_simt_f32_kernel(const float *__restrict__ x, const float *__restrict__ W,
                                       float *__restrict__ logits, int T, int D, int E)
{
    griddep_wait();
    griddep_launch_dependents();
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= (long long)T * E)
        return;
    const int t = (int)(wid / E), e = (int)(wid % E);
    const float *a = x + (size_t)t * D;
    const float *b = W + (size_t)e * D;
    float acc = 0.f;
    for (int d = lane; d < D; d += 32)
        acc = fmaf(__ldg(a + d), __ldg(b + d), acc);
    acc = warp_sum_bcast(acc);
    if (lane == 0)
        logits[(size_t)t * E + e] = acc;
}

cudaError_t launch_router_simt(const moe_config &c, const void *x, const void *W_r,
                               float *logits, cudaStream_t stream)
{
    const long long warps = (long long)c.T * c.n_experts;
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    if (c.dtype == MOE_DTYPE_BF16)
        return launch_pdl(router_simt_bf16_kernel, dim3((unsigned)blocks), dim3(threads), 0,
                          stream, (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)W_r, logits,
                          c.T, c.d_model, c.n_experts);
    return launch_pdl(router_simt_f32_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                      (const float *)x, (const float *)W_r, logits, c.T, c.d_model,
                      c.n_experts);
}

// --------------------------------------------------------------------- gate
struct GateParams {
    float *logits;          // [T,E]: raw scores in (unless fused), scores (+bias) out
    const float *bias;      // [E] or null
    const void *x;          // [T,D] (fused router only)
    const void *W_r;        // [E,D] (fused router only)
    int T, E, k, mode, nchunk, D;
    int32_t *topk_idx;      // [T,k]
    float *topk_w;          // [T,k]
    int32_t *hist;          // [E][nchunk]
    float *ppart;           // [E][nchunk]
    uint8_t *rank;          // [T*k]
    int32_t *status;
};

constexpr int kGateWarps = kChunk;  // one warp per token of the chunk
constexpr int kFusedMaxE = 16;      // fused router: experts held by one lane each
constexpr int kFusedMaxWrBytes = 64 * 1024;

enum { ROUTER_NONE = 0, ROUTER_BF16 = 1, ROUTER_F32 = 2 };

// Partial dot products of one 8-element slice of x against W_r rows in
// shared memory; acc[e] accumulates expert e.
template <int RT>
__device__ __forceinline__ void fused_router_slice(const void *x_row, const uint8_t *wr_s, int D,
                                                   int E, int v, float (&acc)[kFusedMaxE])
{
    float xf[8];
    if (RT == ROUTER_BF16) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(x_row) + v);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            xf[2 * i] = f.x;
            xf[2 * i + 1] = f.y;
        }
    } else {
        const float4 *xr = reinterpret_cast<const float4 *>(x_row) + 2 * v;
        const float4 a = __ldg(xr), b = __ldg(xr + 1);
        xf[0] = a.x; xf[1] = a.y; xf[2] = a.z; xf[3] = a.w;
        xf[4] = b.x; xf[5] = b.y; xf[6] = b.z; xf[7] = b.w;
    }
#pragma unroll
    for (int e = 0; e < kFusedMaxE; ++e) {
        if (e < E) {
            float wf[8];
            if (RT == ROUTER_BF16) {
                const uint4 q = reinterpret_cast<const uint4 *>(wr_s + (size_t)e * D * 2)[v];
                const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __bfloat1622float2(h[i]);
                    wf[2 * i] = f.x;
                    wf[2 * i + 1] = f.y;
                }
            } else {
                const float4 *wr = reinterpret_cast<const float4 *>(wr_s + (size_t)e * D * 4) + 2 * v;
                const float4 a = wr[0], b = wr[1];
                wf[0] = a.x; wf[1] = a.y; wf[2] = a.z; wf[3] = a.w;
                wf[4] = b.x; wf[5] = b.y; wf[6] = b.z; wf[7] = b.w;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
                acc[e] = fmaf(xf[i], wf[i], acc[e]);
        }
    }
}

// One block per chunk of 32 tokens, one warp per token; lane l holds experts
// l, l+32, ...  Dynamic shared memory: [W_r (fused)] [pbuf 32 x E floats]
// [ibuf 32 x k ints] [mask E words].
template <int EPL, int RT>
__global__ void __launch_bounds__(kGateWarps * 32) gate_kernel(GateParams p)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    const int E = p.E, k = p.k;
    const size_t wr_bytes =
        RT == ROUTER_NONE ? 0 : (size_t)E * p.D * (RT == ROUTER_BF16 ? 2 : 4);
    float *pbuf = reinterpret_cast<float *>(dsm + wr_bytes);
    int32_t *ibuf = reinterpret_cast<int32_t *>(pbuf + kChunk * E);
    uint32_t *mask = reinterpret_cast<uint32_t *>(ibuf + kChunk * k);

    const int chunk = blockIdx.x;
    const int tt = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = chunk * kChunk + tt;

    griddep_wait();
    griddep_launch_dependents();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        mask[e] = 0u;
    if constexpr (RT != ROUTER_NONE) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.W_r);
        uint4 *dst = reinterpret_cast<uint4 *>(dsm);
        for (size_t i = threadIdx.x; i < wr_bytes / 16; i += blockDim.x)
            dst[i] = __ldg(src + i);
    }
    __syncthreads();

    if (t < p.T) {
        float s[EPL];
        if (RT != ROUTER_NONE) {
            // the router GEMM for this token: s_e = x_t . W_r[e]
            float acc[kFusedMaxE];
#pragma unroll
            for (int e = 0; e < kFusedMaxE; ++e)
                acc[e] = 0.f;
            const size_t row_bytes = (size_t)p.D * (RT == ROUTER_BF16 ? 2 : 4);
            const void *x_row = static_cast<const uint8_t *>(p.x) + (size_t)t * row_bytes;
            for (int v = lane; v < p.D / 8; v += 32)
                fused_router_slice<RT>(x_row, dsm, p.D, E, v, acc);
            s[0] = -FLT_MAX;
#pragma unroll
            for (int e = 0; e < kFusedMaxE; ++e) {
                if (e < E) {
                    const float v = warp_sum_bcast(acc[e]);
                    if (lane == e)
                        s[0] = v;
                }
            }
#pragma unroll
            for (int i = 1; i < EPL; ++i)
                s[i] = -FLT_MAX;
        }
        bool bad = false;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                float v = (RT != ROUTER_NONE) ? s[i] : p.logits[(size_t)t * E + e];
                if (p.bias)
                    v += p.bias[e];
                if (RT != ROUTER_NONE || p.bias)
                    p.logits[(size_t)t * E + e] = v;
                bad |= !isfinite(v);
                s[i] = v;
            } else {
                s[i] = -FLT_MAX;
            }
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0)
            set_status(p.status, MOE_DEVICE_NONFINITE_SCORE);

        // softmax over all E (max subtracted)
        float m = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (lane + 32 * i < E)
                m = fmaxf(m, s[i]);
        m = warp_max(m);
        float z = 0.f;
        float ex[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            ex[i] = (lane + 32 * i < E) ? expf(s[i] - m) : 0.f;
            z += ex[i];
        }
        z = warp_sum_bcast(z);
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E)
                pbuf[tt * E + e] = ex[i] / z;
        }

        // top-k: k rounds of a warp arg-max; equal scores go to the lower index
        uint32_t taken = 0u;
        float sel_s[kMaxTopK];
        int sel_e[kMaxTopK];
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            sel_s[j] = 0.f;
            sel_e[j] = 0;
            if (j < k) {
                float bv = -FLT_MAX;
                int be = INT_MAX;
#pragma unroll
                for (int i = 0; i < EPL; ++i) {
                    const int e = lane + 32 * i;
                    if (e < E && !((taken >> i) & 1u)) {
                        if (be == INT_MAX || s[i] > bv) {
                            bv = s[i];
                            be = e;
                        }
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                    if (oe != INT_MAX &&
                        (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
                        bv = ov;
                        be = oe;
                    }
                }
                if (be == INT_MAX || be >= E)
                    be = 0;  // unreachable with k <= E; keeps indices in bounds
                sel_s[j] = bv;
                sel_e[j] = be;
                if ((be & 31) == lane)
                    taken |= 1u << (be >> 5);
            }
        }

        // gate weights (every lane computes the same values)
        float w[kMaxTopK];
        if (p.mode == MOE_GATE_SOFTMAX_SELECTED) {
            float zs = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                w[j] = (j < k) ? expf(sel_s[j] - sel_s[0]) : 0.f;
                zs += w[j];
            }
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)
                w[j] = w[j] / zs;
        } else {
            float zs = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                w[j] = (j < k) ? expf(sel_s[j] - m) / z : 0.f;
                zs += w[j];
            }
            if (p.mode == MOE_GATE_SOFTMAX_ALL_RENORM) {
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j)
                    w[j] = w[j] / zs;
            }
        }
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            if (j < k && lane == j) {
                p.topk_idx[(size_t)t * k + j] = sel_e[j];
                p.topk_w[(size_t)t * k + j] = w[j];
                atomicOr(&mask[sel_e[j]], 1u << tt);
                ibuf[tt * k + j] = sel_e[j];
            }
        }
    } else {
        for (int e = lane; e < E; e += 32)
            pbuf[tt * E + e] = 0.f;
    }
    __syncthreads();

    // per-expert chunk statistics: count, and the probability sum in token order
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        p.hist[(size_t)e * p.nchunk + chunk] = __popc(mask[e]);
        float acc = 0.f;
#pragma unroll 8
        for (int u = 0; u < kChunk; ++u)
            acc += pbuf[u * E + e];
        p.ppart[(size_t)e * p.nchunk + chunk] = acc;
    }
    // rank of (t, j) among the chunk's earlier tokens that chose the same expert
    for (int i = threadIdx.x; i < kChunk * k; i += blockDim.x) {
        const int u = i / k, j = i % k;
        const int tok = chunk * kChunk + u;
        if (tok < p.T) {
            const int e = ibuf[u * k + j];
            p.rank[(size_t)tok * k + j] = (uint8_t)__popc(mask[e] & ((1u << u) - 1u));
        }
    }
}

bool router_fused(const moe_config &c)
{
    const size_t esz = c.dtype == MOE_DTYPE_BF16 ? 2 : 4;
    return c.n_experts <= kFusedMaxE && c.d_model % 8 == 0 &&
           (size_t)c.n_experts * c.d_model * esz <= (size_t)kFusedMaxWrBytes;
}

template <int EPL, int RT>
static cudaError_t launch_gate_t(const GateParams &p, size_t smem, cudaStream_t stream)
{
    auto kern = gate_kernel<EPL, RT>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    static uint64_t configured = 0;
    if (dev < 64 && !(configured & (1ull << dev))) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kFusedMaxWrBytes + kChunk * (kMaxExperts + kMaxTopK) * 4 +
                                       kMaxExperts * 4);
        if (err != cudaSuccess)
            return err;
        configured |= 1ull << dev;
    }
    return launch_pdl(kern, dim3(p.nchunk), dim3(kGateWarps * 32), smem, stream, p);
}

cudaError_t launch_gate(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                        const void *x, const void *W_r, float *logits, const float *bias,
                        int32_t *topk_idx, float *topk_w, cudaStream_t stream)
{
    GateParams p;
    p.logits = logits;
    p.bias = bias;
    p.x = x;
    p.W_r = W_r;
    p.T = c.T;
    p.E = c.n_experts;
    p.k = c.top_k;
    p.mode = c.gating_mode;
    p.nchunk = L.nchunk;
    p.D = c.d_model;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.hist = reinterpret_cast<int32_t *>(ws + L.hist);
    p.ppart = reinterpret_cast<float *>(ws + L.ppart);
    p.rank = ws + L.rank;
    p.status = reinterpret_cast<int32_t *>(ws + L.status);
    const bool fused = x != nullptr && W_r != nullptr;
    const size_t esz = c.dtype == MOE_DTYPE_BF16 ? 2 : 4;
    const size_t smem = (fused ? (size_t)c.n_experts * c.d_model * esz : 0) +
                        (size_t)kChunk * (c.n_experts + c.top_k) * 4 + (size_t)c.n_experts * 4;
    if (fused)
        return c.dtype == MOE_DTYPE_BF16 ? launch_gate_t<1, ROUTER_BF16>(p, smem, stream)
                                         : launch_gate_t<1, ROUTER_F32>(p, smem, stream);
    const int epl = (c.n_experts + 31) / 32;
    if (epl <= 1)
        return launch_gate_t<1, ROUTER_NONE>(p, smem, stream);
    if (epl <= 2)
        return launch_gate_t<2, ROUTER_NONE>(p, smem, stream);
    if (epl <= 4)
        return launch_gate_t<4, ROUTER_NONE>(p, smem, stream);
    return launch_gate_t<8, ROUTER_NONE>(p, smem, stream);
}

}  // namespace moe
