// moe_combine.cu -- the weighted combine:
//   y_t = sum_{j<k, kept} w_tj z[row_tj] (+ z_shared[t])
// with fp32 accumulation in the fixed order j = 0..k-1, then the shared
// expert.  Dropped assignments contribute nothing and the remaining weights
// are not renormalised; the residual connection is the caller's.
//
// Sources: "Mixture of Experts" (module 17), 17.2 equation (shared expert plus
// the gate-weighted routed experts) and 17.5 (a dropped token keeps its other
// experts and the residual); "Mixture of Experts: Sparse FFNs, Routers, and
// Shared Experts" (the combine loop: out[tok] += weight * expert(x[tok])).
#include <cuda_bf16.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kCombineThreads = 128;

// y_t = sum_{j<k, kept} w_tj z[row_tj] (+ zs[t]), fp32 accumulation in the
// fixed order j = 0..k-1, then the shared expert.  Block b covers 128
// 16-byte vectors (8 elements each) of one token (token b / nchunk, chunk
// b % nchunk); each thread issues the loads of all of its token's rows before
// accumulating, so that they overlap.  The shared expert's output is bf16
// [T][D] (zs), or fp32 partial sums [zsplit][T][D] (zs_part) added in split
// order.
__global__ void __launch_bounds__(kCombineThreads)
    combine_bf16_kernel(const __nv_bfloat16 *__restrict__ z, const __nv_bfloat16 *__restrict__ zs,
                        const float *__restrict__ zs_part, int zsplit,
                        const float *__restrict__ topk_w, const int32_t *__restrict__ row_of,
                        __nv_bfloat16 *__restrict__ y, int T, int k, int D, int nchunk,
                        long long R_max, int32_t *status)
{
    __shared__ int rows[kMaxTopK];
    __shared__ float ws[kMaxTopK];
    griddep_wait();
    griddep_launch_dependents();
    if (*(volatile const int32_t *)status != 0)
        return;  // an earlier kernel failed; y is left unspecified
    const int t = blockIdx.x / nchunk, chunk = blockIdx.x - (blockIdx.x / nchunk) * nchunk;
    if ((int)threadIdx.x < k) {
        int r = row_of[(size_t)t * k + threadIdx.x];
        if (kDebugBounds && r >= R_max) {
            set_status(status, MOE_DEVICE_INDEX_OUT_OF_RANGE);
            r = -1;
        }
        rows[threadIdx.x] = r;
        ws[threadIdx.x] = topk_w[(size_t)t * k + threadIdx.x];
    }
    __syncthreads();
    const int v = chunk * kCombineThreads + threadIdx.x;
    if (v >= D / 8)
        return;
    uint4 q[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
        if (j < k && rows[j] >= 0)
            q[j] = reinterpret_cast<const uint4 *>(z + (size_t)rows[j] * D)[v];
    uint4 qs = make_uint4(0u, 0u, 0u, 0u);
    if (zs)
        qs = reinterpret_cast<const uint4 *>(zs + (size_t)t * D)[v];
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        if (j < k && rows[j] >= 0) {
            const float wj = ws[j];
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&q[j]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h[i]);
                acc[2 * i] = fmaf(wj, f.x, acc[2 * i]);
                acc[2 * i + 1] = fmaf(wj, f.y, acc[2 * i + 1]);
            }
        }
    }
    if (zs) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&qs);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            acc[2 * i] += f.x;
            acc[2 * i + 1] += f.y;
        }
    } else if (zs_part) {
        float sh[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            sh[i] = 0.f;
        for (int q0 = 0; q0 < zsplit; ++q0) {
            const float4 *src =
                reinterpret_cast<const float4 *>(zs_part + ((size_t)q0 * T + t) * D) + 2 * v;
            const float4 a = src[0], b = src[1];
            sh[0] += a.x; sh[1] += a.y; sh[2] += a.z; sh[3] += a.w;
            sh[4] += b.x; sh[5] += b.y; sh[6] += b.z; sh[7] += b.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] += sh[i];
    }
    uint4 out;
    __nv_bfloat162 *o = reinterpret_cast<__nv_bfloat162 *>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    reinterpret_cast<uint4 *>(y + (size_t)t * D)[v] = out;
}

__global__ void __launch_bounds__(128)
    combine_f32_kernel(const float *__restrict__ z, const float *__restrict__ zs,
                       const float *__restrict__ topk_w, const int32_t *__restrict__ row_of,
                       float *__restrict__ y, int k, int D, long long R_max, int32_t *status)
{
    __shared__ int rows[kMaxTopK];
    __shared__ float ws[kMaxTopK];
    griddep_wait();
    griddep_launch_dependents();
    if (*(volatile const int32_t *)status != 0)
        return;  // an earlier kernel failed; y is left unspecified
    const int t = blockIdx.x;
    if ((int)threadIdx.x < k) {
        int r = row_of[(size_t)t * k + threadIdx.x];
        if (kDebugBounds && r >= R_max) {
            set_status(status, MOE_DEVICE_INDEX_OUT_OF_RANGE);
            r = -1;
        }
        rows[threadIdx.x] = r;
        ws[threadIdx.x] = topk_w[(size_t)t * k + threadIdx.x];
    }
    __syncthreads();
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float acc = 0.f;
        for (int j = 0; j < k; ++j) {
            const int r = rows[j];
            if (r >= 0)
                acc = fmaf(ws[j], z[(size_t)r * D + d], acc);
        }
        if (zs)
            acc += zs[(size_t)t * D + d];
        y[(size_t)t * D + d] = acc;
    }
}

cudaError_t launch_combine(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                           const float *topk_w, void *y, cudaStream_t stream)
{
    static DeviceOnce configured;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (configured.pending(dev)) {
        err = prefer_max_shared_carveout(combine_bf16_kernel);
        if (err == cudaSuccess)
            err = prefer_max_shared_carveout(combine_f32_kernel);
        if (err != cudaSuccess)
            return err;
        configured.done(dev);
    }
    const int32_t *row_of = reinterpret_cast<const int32_t *>(ws + L.row_of);
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    const bool shared = c.d_shared > 0;
    if (c.dtype == MOE_DTYPE_BF16) {
        const int nchunk = (c.d_model / 8 + kCombineThreads - 1) / kCombineThreads;
        const int zsplit = shared ? shared_down_splits(c) : 1;
        const __nv_bfloat16 *zs = shared && zsplit == 1
                                      ? reinterpret_cast<const __nv_bfloat16 *>(ws + L.zs)
                                      : nullptr;
        const float *zs_part =
            shared && zsplit > 1 ? reinterpret_cast<const float *>(ws + L.zs) : nullptr;
        return launch_pdl(combine_bf16_kernel, dim3((unsigned)((long long)c.T * nchunk)),
                          dim3(kCombineThreads), 0, stream,
                          reinterpret_cast<const __nv_bfloat16 *>(ws + L.z), zs, zs_part, zsplit,
                          topk_w, row_of, (__nv_bfloat16 *)y, c.T, c.top_k, c.d_model, nchunk,
                          (long long)L.R_max, status);
    }
    return launch_pdl(combine_f32_kernel, dim3(c.T), dim3(128), 0, stream,
                      reinterpret_cast<const float *>(ws + L.z),
                      shared ? reinterpret_cast<const float *>(ws + L.zs) : nullptr, topk_w,
                      row_of, (float *)y, c.top_k, c.d_model, (long long)L.R_max, status);
}

}  // namespace moe
