// moe_route.cu -- router scores on SIMT cores (small T and fp32), and the
// gating kernel: softmax, top-k with lower-index tie-break, gate weights,
// per-chunk expert histograms, per-chunk probability sums, and the rank of
// each assignment among its chunk's tokens (for token-order capacity).
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
        router_simt_bf16_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
            (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)W_r, logits, c.T, c.d_model,
            c.n_experts);
    else
        router_simt_f32_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
            (const float *)x, (const float *)W_r, logits, c.T, c.d_model, c.n_experts);
    return cudaGetLastError();
}

// --------------------------------------------------------------------- gate
struct GateParams {
    float *logits;          // [T,E] raw scores in, scores (+bias) out
    const float *bias;      // [E] or null
    int T, E, k, mode, nchunk;
    int32_t *topk_idx;      // [T,k]
    float *topk_w;          // [T,k]
    int32_t *hist;          // [E][nchunk]
    float *ppart;           // [E][nchunk]
    uint8_t *rank;          // [T*k]
    int32_t *status;
};

constexpr int kGateWarps = 8;

// One block per chunk of 32 tokens; each warp routes tokens of the chunk,
// one token at a time, with lane l holding experts l, l+32, ...
template <int EPL>
__global__ void __launch_bounds__(kGateWarps * 32) gate_kernel(GateParams p)
{
    __shared__ uint32_t mask[kMaxExperts];            // bit tt: token tt chose e
    __shared__ float pbuf[kChunk][kMaxExperts];       // softmax probabilities
    __shared__ int32_t ibuf[kChunk][kMaxTopK];        // chosen experts

    const int chunk = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E, k = p.k;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        mask[e] = 0u;
    __syncthreads();

    for (int tt = warp; tt < kChunk; tt += kGateWarps) {
        const int t = chunk * kChunk + tt;
        if (t >= p.T) {
            for (int e = lane; e < E; e += 32)
                pbuf[tt][e] = 0.f;
            continue;
        }
        float s[EPL];
        bool bad = false;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            s[i] = -FLT_MAX;
            if (e < E) {
                float v = p.logits[(size_t)t * E + e];
                if (p.bias) {
                    v += p.bias[e];
                    p.logits[(size_t)t * E + e] = v;
                }
                bad |= !isfinite(v);
                s[i] = v;
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
                pbuf[tt][e] = ex[i] / z;
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
                // be is valid: k <= E leaves an untaken expert in some lane.
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
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j) {
                if (j < k) {
                    atomicOr(&mask[sel_e[j]], 1u << tt);
                    ibuf[tt][j] = sel_e[j];
                }
            }
        }
    }
    __syncthreads();

    // per-expert chunk statistics: count, and the probability sum in token order
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        p.hist[(size_t)e * p.nchunk + chunk] = __popc(mask[e]);
        float acc = 0.f;
#pragma unroll 8
        for (int tt = 0; tt < kChunk; ++tt)
            acc += pbuf[tt][e];
        p.ppart[(size_t)e * p.nchunk + chunk] = acc;
    }
    // rank of (t, j) among the chunk's earlier tokens that chose the same expert
    for (int i = threadIdx.x; i < kChunk * k; i += blockDim.x) {
        const int tt = i / k, j = i % k;
        const int t = chunk * kChunk + tt;
        if (t < p.T) {
            const int e = ibuf[tt][j];
            p.rank[(size_t)t * k + j] = (uint8_t)__popc(mask[e] & ((1u << tt) - 1u));
        }
    }
}

cudaError_t launch_gate(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                        float *logits, const float *bias, int32_t *topk_idx, float *topk_w,
                        cudaStream_t stream)
{
    GateParams p;
    p.logits = logits;
    p.bias = bias;
    p.T = c.T;
    p.E = c.n_experts;
    p.k = c.top_k;
    p.mode = c.gating_mode;
    p.nchunk = L.nchunk;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.hist = reinterpret_cast<int32_t *>(ws + L.hist);
    p.ppart = reinterpret_cast<float *>(ws + L.ppart);
    p.rank = ws + L.rank;
    p.status = reinterpret_cast<int32_t *>(ws + L.status);
    const dim3 grid(L.nchunk), block(kGateWarps * 32);
    const int epl = (c.n_experts + 31) / 32;
    if (epl <= 1)
        gate_kernel<1><<<grid, block, 0, stream>>>(p);
    else if (epl <= 2)
        gate_kernel<2><<<grid, block, 0, stream>>>(p);
    else if (epl <= 4)
        gate_kernel<4><<<grid, block, 0, stream>>>(p);
    else
        gate_kernel<8><<<grid, block, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace moe
