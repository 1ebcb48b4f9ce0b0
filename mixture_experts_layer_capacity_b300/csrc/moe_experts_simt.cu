// moe_experts_simt.cu -- the expert feed-forward networks on SIMT cores, for
// the fp32 dtype (exact-precision checks and small layers).  One thread per
// output element, fp32 accumulation:
//   h[r][f] = silu(sum_d x_perm[r][d] W_gate[e][f][d]) * (sum_d x_perm[r][d] W_up[e][f][d])
//   z[r][d] = sum_f h[r][f] W_down[e][d][f]
// where e is the expert whose segment holds row r ("Mixture of Experts: More
// Parameters, Same FLOPs", 'An MoE tiny GPT': the SwiGLU expert).  The shared
// expert is the same computation over all T rows of x with one segment.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

// Largest segment e in [0, nseg) with seg_off[e] <= r (skips empty segments).
__device__ __forceinline__ int segment_of(const int32_t *seg_off, int nseg, int r)
{
    int lo = 0, hi = nseg;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (seg_off[mid] <= r)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

template <bool SWIGLU>
__global__ void simt_seg_gemm_f32_kernel(const float *__restrict__ A, const float *__restrict__ B0,
                                         const float *__restrict__ B1, long long b_seg_elems,
                                         int N, int K, const int32_t *__restrict__ seg_off,
                                         int nseg, int dense_rows, float *__restrict__ out,
                                         const int32_t *status, AuxArgs aux)
{
    griddep_wait();
    griddep_launch_dependents();
    if (*(volatile const int32_t *)status != 0)
        return;  // an earlier kernel failed
    if (aux.out && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.y == 0)
        balance_loss_warp(aux);
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    const int r = blockIdx.y * blockDim.y + threadIdx.y;
    const int rows = seg_off ? seg_off[nseg] : dense_rows;
    if (r >= rows || n >= N)
        return;
    const int e = seg_off ? segment_of(seg_off, nseg, r) : 0;
    const float *a = A + (size_t)r * K;
    const float *b0 = B0 + (size_t)e * b_seg_elems + (size_t)n * K;
    float g = 0.f, u = 0.f;
    if (SWIGLU) {
        const float *b1 = B1 + (size_t)e * b_seg_elems + (size_t)n * K;
        for (int kk = 0; kk < K; ++kk) {
            const float av = a[kk];
            g = fmaf(av, __ldg(b0 + kk), g);
            u = fmaf(av, __ldg(b1 + kk), u);
        }
        out[(size_t)r * N + n] = (g / (1.0f + expf(-g))) * u;
    } else {
        for (int kk = 0; kk < K; ++kk)
            g = fmaf(a[kk], __ldg(b0 + kk), g);
        out[(size_t)r * N + n] = g;
    }
}

cudaError_t launch_experts_simt(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                                const void *x, const void *W_gate, const void *W_up,
                                const void *W_down, const void *Ws_gate, const void *Ws_up,
                                const void *Ws_down, const AuxArgs &aux, cudaStream_t stream,
                                cudaEvent_t *ev)
{
    if (c.dtype != MOE_DTYPE_FP32)
        return cudaErrorInvalidValue;
    const int D = c.d_model, F = c.d_expert, S = c.d_shared, E = c.n_experts;
    const int32_t *seg = reinterpret_cast<const int32_t *>(ws + L.seg_off);
    const int32_t *status = reinterpret_cast<const int32_t *>(ws + L.status);
    float *xp = reinterpret_cast<float *>(ws + L.x_perm);
    float *h = reinterpret_cast<float *>(ws + L.h);
    float *z = reinterpret_cast<float *>(ws + L.z);
    const dim3 block(32, 8);
    const unsigned rb = (unsigned)((L.R_max + 7) / 8);
    const float *nil = nullptr;
    const int32_t *noseg = nullptr;
    AuxArgs none = aux;
    none.out = nullptr;
    cudaError_t err = launch_pdl(simt_seg_gemm_f32_kernel<true>, dim3((F + 31) / 32, rb), block, 0,
                                 stream, (const float *)xp, (const float *)W_gate,
                                 (const float *)W_up, (long long)F * D, F, D, seg, E, 0, h, status, aux);
    if (err == cudaSuccess)
        err = record_stage(ev, 3, stream);
    if (err == cudaSuccess)
        err = launch_pdl(simt_seg_gemm_f32_kernel<false>, dim3((D + 31) / 32, rb), block, 0,
                         stream, (const float *)h, (const float *)W_down, nil,
                         (long long)D * F, D, F, seg, E, 0, z, status, none);
    if (err == cudaSuccess)
        err = record_stage(ev, 4, stream);
    if (err != cudaSuccess)
        return err;
    if (S > 0) {
        float *hs = reinterpret_cast<float *>(ws + L.hs);
        float *zs = reinterpret_cast<float *>(ws + L.zs);
        const unsigned tb = (unsigned)((c.T + 7) / 8);
        err = launch_pdl(simt_seg_gemm_f32_kernel<true>, dim3((S + 31) / 32, tb), block, 0,
                         stream, (const float *)x, (const float *)Ws_gate, (const float *)Ws_up,
                         0LL, S, D, noseg, 1, c.T, hs, status, none);
        if (err == cudaSuccess)
            err = record_stage(ev, 5, stream);
        if (err == cudaSuccess)
            err = launch_pdl(simt_seg_gemm_f32_kernel<false>, dim3((D + 31) / 32, tb), block, 0,
                             stream, (const float *)hs, (const float *)Ws_down, nil, 0LL, D, S,
                             noseg, 1, c.T, zs, status, none);
        if (err == cudaSuccess)
            err = record_stage(ev, 6, stream);
        if (err != cudaSuccess)
            return err;
    } else {
        record_stage(ev, 5, stream);
        record_stage(ev, 6, stream);
    }
    return cudaGetLastError();
}

cudaError_t launch_dense_simt(int rows, int N, int K, const float *A, const float *B, float *out,
                              const int32_t *status, cudaStream_t stream)
{
    if (rows <= 0)
        return cudaSuccess;
    AuxArgs none{};
    const dim3 block(32, 8);
    return launch_pdl(simt_seg_gemm_f32_kernel<false>, dim3((N + 31) / 32, (rows + 7) / 8), block,
                      0, stream, A, B, (const float *)nullptr, 0LL, N, K,
                      (const int32_t *)nullptr, 1, rows, out, status, none);
}

}  // namespace moe
