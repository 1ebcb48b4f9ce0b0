// moe_permute.cu -- token-order capacity and the expert-contiguous layout.
//
//   scan:     per expert, exclusive prefix over chunks of the chunk counts
//             (so base + rank = the number of earlier tokens that chose the
//             expert), the demand count n_e, and the probability sum P_sum_e;
//   finalize: kept_e = min(n_e, C), segment offsets, tile prefix, and the
//             balance loss alpha * E * sum_e (n_e / (T k)) (P_sum_e / T);
//   scatter:  position of each assignment, capacity drop, x row gathered into
//             its expert's segment;
//   combine:  y_t = sum_{j, kept} w_tj z[row_tj] + z_shared[t].
//
// Sources: "Mixture of Experts" (module 17), 17.5 (capacity equation; tokens
// beyond C are dropped by that expert only) and 17.4 (balance loss);
// "Mixture of Experts: Sparse FFNs, Routers, and Shared Experts", 'Capacity
// factor' (dropped tokens skip the expert) and the dispatch/combine loop;
// "Mixture of experts" (AI engineering visualised), 'Capacity'.
#include <type_traits>

#include <cuda_bf16.h>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kScanThreads = 256;

// Exclusive scan of one int per thread over a 256-thread block; *total gets
// the block sum.  `sh` must hold 8 ints.
__device__ __forceinline__ int block_excl_scan_256(int v, int *sh, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += n;
    }
    if (lane == 31)
        sh[warp] = incl;
    __syncthreads();
    int wbase = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kScanThreads / 32; ++w) {
        const int s = sh[w];
        if (w < warp)
            wbase += s;
        tot += s;
    }
    __syncthreads();
    *total = tot;
    return wbase + incl - v;
}

// Fixed-order tree sum of one double per thread over a 256-thread block.
__device__ __forceinline__ double block_sum_256(double v, double *sh)
{
    sh[threadIdx.x] = v;
    __syncthreads();
    for (int s = kScanThreads / 2; s > 0; s >>= 1) {
        if ((int)threadIdx.x < s)
            sh[threadIdx.x] += sh[threadIdx.x + s];
        __syncthreads();
    }
    const double r = sh[0];
    __syncthreads();
    return r;
}

// One block per expert: exclusive prefix of the chunk counts, the demand
// count n_e and P_sum_e.  The last block to finish (block counter) then
// computes kept_e = min(n_e, C), the segment offsets, the 128-row tile prefix
// and the balance loss from all experts' results.
__global__ void __launch_bounds__(kScanThreads)
    scan_finalize_kernel(int32_t *hist, const float *ppart, double *psum, int32_t *expert_counts,
                         int nchunk, int E, int T, int k, long long C, float alpha,
                         int32_t *kept_counts, int32_t *seg_off, int32_t *mtile, float *aux_loss,
                         int32_t *block_counter)
{
    __shared__ int shi[8];
    __shared__ double shd[kScanThreads];
    __shared__ int is_last;
    griddep_wait();
    griddep_launch_dependents();
    const int e = blockIdx.x;
    {
        int32_t *h = hist + (size_t)e * nchunk;
        const float *pp = ppart + (size_t)e * nchunk;
        const int per = (nchunk + kScanThreads - 1) / kScanThreads;
        const int beg = min(nchunk, (int)threadIdx.x * per), end = min(nchunk, beg + per);
        int local = 0;
        double pl = 0.0;
        for (int c = beg; c < end; ++c) {
            local += h[c];
            pl += (double)pp[c];
        }
        int total;
        int run = block_excl_scan_256(local, shi, &total);
        for (int c = beg; c < end; ++c) {
            const int v = h[c];
            h[c] = run;
            run += v;
        }
        const double ps = block_sum_256(pl, shd);
        if (threadIdx.x == 0) {
            expert_counts[e] = total;
            psum[e] = ps;
            __threadfence();
            is_last = (atomicAdd(block_counter, 1) == E - 1);
        }
        __syncthreads();
    }
    if (!is_last)
        return;
    __threadfence();

    const int x = threadIdx.x;  // expert handled by this thread in the finalize
    const int n = x < E ? __ldcg(expert_counts + x) : 0;
    const int kept = (C < 0) ? n : (int)min((long long)n, C);
    if (x < E)
        kept_counts[x] = kept;
    int total;
    const int off = block_excl_scan_256(kept, shi, &total);
    if (x < E)
        seg_off[x] = off;
    if (x == 0)
        seg_off[E] = total;
    const int mt = (kept + kTileM - 1) / kTileM;
    int mt_total;
    const int moff = block_excl_scan_256(mt, shi, &mt_total);
    if (x < E)
        mtile[x] = moff;
    if (x == 0)
        mtile[E] = mt_total;
    double term = 0.0;
    if (x < E && T > 0)
        term = ((double)n / ((double)T * (double)k)) * (__ldcg(psum + x) / (double)T);
    const double sum = block_sum_256(term, shd);
    if (x == 0)
        *aux_loss = (float)((double)alpha * (double)E * sum);
}

cudaError_t launch_scan_finalize(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                                 int32_t *expert_counts, int32_t *kept_counts, float *aux_loss,
                                 cudaStream_t stream)
{
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    return launch_pdl(scan_finalize_kernel, dim3(c.n_experts), dim3(kScanThreads), 0, stream,
                      reinterpret_cast<int32_t *>(ws + L.hist),
                      reinterpret_cast<const float *>(ws + L.ppart),
                      reinterpret_cast<double *>(ws + L.psum), expert_counts, L.nchunk,
                      c.n_experts, c.T, c.top_k, (long long)L.C, c.aux_alpha, kept_counts,
                      reinterpret_cast<int32_t *>(ws + L.seg_off),
                      reinterpret_cast<int32_t *>(ws + L.mtile), aux_loss, status + 8);
}

// -------------------------------------------------------------------- scatter
// One block per token.  VEC = bytes per copy unit (16 or 4).
template <int VEC>
__global__ void __launch_bounds__(128)
    scatter_kernel(const uint8_t *__restrict__ x, const int32_t *__restrict__ topk_idx,
                   const uint8_t *__restrict__ rank, const int32_t *__restrict__ base,
                   const int32_t *__restrict__ seg_off, long long C, int k, int nchunk,
                   size_t row_bytes, uint8_t *dropped, int32_t *row_of, uint8_t *x_perm)
{
    __shared__ long long rows[kMaxTopK];
    griddep_wait();
    griddep_launch_dependents();
    const int t = blockIdx.x;
    if ((int)threadIdx.x < k) {
        const int j = threadIdx.x;
        const int e = topk_idx[(size_t)t * k + j];
        const long long pos =
            (long long)base[(size_t)e * nchunk + t / kChunk] + rank[(size_t)t * k + j];
        const bool kept = (C < 0) || (pos < C);
        const long long row = kept ? (long long)seg_off[e] + pos : -1;
        rows[j] = row;
        dropped[(size_t)t * k + j] = kept ? 0 : 1;
        row_of[(size_t)t * k + j] = (int32_t)row;
    }
    __syncthreads();
    using V = typename std::conditional<VEC == 16, uint4, uint32_t>::type;
    const size_t nv = row_bytes / VEC;
    const V *src = reinterpret_cast<const V *>(x + (size_t)t * row_bytes);
    for (size_t v = threadIdx.x; v < nv; v += blockDim.x) {
        const V val = src[v];
        for (int j = 0; j < k; ++j) {
            const long long r = rows[j];
            if (r >= 0)
                reinterpret_cast<V *>(x_perm + (size_t)r * row_bytes)[v] = val;
        }
    }
}

cudaError_t launch_scatter(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                           const void *x, const int32_t *topk_idx, uint8_t *dropped_mask,
                           cudaStream_t stream)
{
    const size_t esz = c.dtype == MOE_DTYPE_BF16 ? 2 : 4;
    const size_t row_bytes = (size_t)c.d_model * esz;
    auto *args_base = reinterpret_cast<const int32_t *>(ws + L.hist);
    auto *seg = reinterpret_cast<const int32_t *>(ws + L.seg_off);
    auto *row_of = reinterpret_cast<int32_t *>(ws + L.row_of);
    if (row_bytes % 16 == 0)
        return launch_pdl(scatter_kernel<16>, dim3(c.T), dim3(128), 0, stream, (const uint8_t *)x,
                          topk_idx, (const uint8_t *)(ws + L.rank), args_base, seg, (long long)L.C,
                          c.top_k, L.nchunk, row_bytes, dropped_mask, row_of, ws + L.x_perm);
    return launch_pdl(scatter_kernel<4>, dim3(c.T), dim3(128), 0, stream, (const uint8_t *)x,
                      topk_idx, (const uint8_t *)(ws + L.rank), args_base, seg, (long long)L.C,
                      c.top_k, L.nchunk, row_bytes, dropped_mask, row_of, ws + L.x_perm);
}

// -------------------------------------------------------------------- combine
// One block per token: y_t = sum_{j<k, kept} w_tj z[row_tj] (+ zs[t]), fp32
// accumulation in the fixed order j = 0..k-1, then the shared expert.
__global__ void __launch_bounds__(128)
    combine_bf16_kernel(const __nv_bfloat16 *__restrict__ z, const __nv_bfloat16 *__restrict__ zs,
                        const float *__restrict__ topk_w, const int32_t *__restrict__ row_of,
                        __nv_bfloat16 *__restrict__ y, int k, int D)
{
    __shared__ int rows[kMaxTopK];
    __shared__ float ws[kMaxTopK];
    griddep_wait();
    griddep_launch_dependents();
    const int t = blockIdx.x;
    if ((int)threadIdx.x < k) {
        rows[threadIdx.x] = row_of[(size_t)t * k + threadIdx.x];
        ws[threadIdx.x] = topk_w[(size_t)t * k + threadIdx.x];
    }
    __syncthreads();
    const int nv = D / 8;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] = 0.f;
        for (int j = 0; j < k; ++j) {
            const int r = rows[j];
            if (r < 0)
                continue;
            const float wj = ws[j];
            const uint4 q = reinterpret_cast<const uint4 *>(z + (size_t)r * D)[v];
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h[i]);
                acc[2 * i] = fmaf(wj, f.x, acc[2 * i]);
                acc[2 * i + 1] = fmaf(wj, f.y, acc[2 * i + 1]);
            }
        }
        if (zs) {
            const uint4 q = reinterpret_cast<const uint4 *>(zs + (size_t)t * D)[v];
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h[i]);
                acc[2 * i] += f.x;
                acc[2 * i + 1] += f.y;
            }
        }
        uint4 out;
        __nv_bfloat162 *o = reinterpret_cast<__nv_bfloat162 *>(&out);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        reinterpret_cast<uint4 *>(y + (size_t)t * D)[v] = out;
    }
}

__global__ void __launch_bounds__(128)
    combine_f32_kernel(const float *__restrict__ z, const float *__restrict__ zs,
                       const float *__restrict__ topk_w, const int32_t *__restrict__ row_of,
                       float *__restrict__ y, int k, int D)
{
    __shared__ int rows[kMaxTopK];
    __shared__ float ws[kMaxTopK];
    griddep_wait();
    griddep_launch_dependents();
    const int t = blockIdx.x;
    if ((int)threadIdx.x < k) {
        rows[threadIdx.x] = row_of[(size_t)t * k + threadIdx.x];
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
    const int32_t *row_of = reinterpret_cast<const int32_t *>(ws + L.row_of);
    const bool shared = c.d_shared > 0;
    if (c.dtype == MOE_DTYPE_BF16)
        return launch_pdl(combine_bf16_kernel, dim3(c.T), dim3(128), 0, stream,
                          reinterpret_cast<const __nv_bfloat16 *>(ws + L.z),
                          shared ? reinterpret_cast<const __nv_bfloat16 *>(ws + L.zs) : nullptr,
                          topk_w, row_of, (__nv_bfloat16 *)y, c.top_k, c.d_model);
    return launch_pdl(combine_f32_kernel, dim3(c.T), dim3(128), 0, stream,
                      reinterpret_cast<const float *>(ws + L.z),
                      shared ? reinterpret_cast<const float *>(ws + L.zs) : nullptr, topk_w,
                      row_of, (float *)y, c.top_k, c.d_model);
}

}  // namespace moe
