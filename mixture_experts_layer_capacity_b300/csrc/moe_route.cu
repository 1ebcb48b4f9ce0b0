// moe_route.cu -- router scores s = x W_r^T on SIMT cores, one warp per
// (token, expert), fp32 accumulation.  Used for small T and fp32 when the
// router is too large to run inside the dispatch kernel; large bf16 batches
// use the tensor-core router in moe_gemm_tc.cu.
//
// Source: "Mixture of Experts: More Parameters, Same FLOPs" ('The router':
// one score per expert, x W_r); "Mixture of experts" (frontiers track),
// 'Where the experts live' (s = W_r x).
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
    static DeviceOnce configured;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (configured.pending(dev)) {
        err = prefer_max_shared_carveout(router_simt_bf16_kernel);
        if (err == cudaSuccess)
            err = prefer_max_shared_carveout(router_simt_f32_kernel);
        if (err != cudaSuccess)
            return err;
        configured.done(dev);
    }
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

}  // namespace moe
