// moe_dispatch.cu -- routing and dispatch in one cooperative kernel:
//
//   phase 1 (gate):     per chunk of 32 tokens, one warp per token: (the
//                       router GEMM itself when W_r fits in shared memory),
//                       softmax over all E, top-k with the lower index first on
//                       equal scores, gate weights, the chunk's per-expert
//                       counts and probability sums, and each assignment's rank
//                       among the chunk's earlier tokens;
//   phase 2 (scan):     per expert, exclusive prefix of the chunk counts, so
//                       that base + rank = the number of earlier tokens that
//                       chose the expert; demand count n_e; P_sum_e.  The last
//                       block to finish computes kept_e = min(n_e, C), the
//                       segment offsets, the 128-row tile prefix and the
//                       balance loss;
//   phase 3 (scatter):  one warp per token: position of each assignment, the
//                       capacity decision, and x copied into the rows of its
//                       experts' segments.
// Phases are separated by grid-wide barriers (all blocks are co-resident:
// cooperative launch); every barrier wait is bounded in time.
//
// Sources: "Mixture of Experts: More Parameters, Same FLOPs" ('The router');
// "Mixture of Experts" (module 17), 17.2 (softmax over the selected vs over
// all experts), 17.4 (balance loss) and 17.5 (capacity equation; tokens beyond
// C are dropped by that expert only); "Mixture of Experts: Sparse FFNs,
// Routers, and Shared Experts" ('Capacity factor'); "Mixture of experts"
// (frontiers track), gate equation of 'Where the experts live'.
#include <cfloat>
#include <climits>
#include <cuda_bf16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "tc_ptx.cuh"

namespace moe {

constexpr int kDispatchThreads = kChunk * 32;  // one warp per token of a chunk
constexpr int kFusedMaxE = 16;
constexpr int kFusedMaxWrBytes = 64 * 1024;
constexpr uint64_t kBarrierLimitNs = 2000000000ull;

enum { ROUTER_NONE = 0, ROUTER_BF16 = 1, ROUTER_F32 = 2 };

struct DispatchParams {
    float *logits;          // [T,E]: raw scores in (unless fused), scores (+bias) out
    const float *bias;      // [E] or null
    const void *x;          // [T,D]
    const void *W_r;        // [E,D] (fused router only)
    int T, E, k, mode, nchunk, D;
    long long C;            // capacity, -1 = dropless
    float alpha;
    size_t row_bytes;       // D * element size
    int32_t *topk_idx;      // [T,k]
    float *topk_w;          // [T,k]
    uint8_t *dropped;       // [T,k]
    int32_t *expert_counts; // [E]
    int32_t *kept_counts;   // [E]
    float *aux_loss;        // [1]
    int32_t *hist;          // [E][nchunk] chunk counts, then exclusive bases
    float *ppart;           // [E][nchunk]
    uint8_t *rank;          // [T*k]
    double *psum;           // [E]
    int32_t *seg_off;       // [E+1]
    int32_t *mtile;         // [E+1]
    int32_t *row_of;        // [T*k]
    uint8_t *x_perm;        // [R_max, D]
    int32_t *row_tok;       // [R_max] token of each x_perm row (direct-y mode), or null
    float *row_w;           // [R_max] gate weight of each row (direct-y mode), or null
    uint8_t *y_zero;        // y [T,D]: rows of fully dropped tokens are zeroed (direct-y)
    int32_t *status;        // [0] status word, [8] scan counter, [9] barrier counter
};

// ------------------------------------------------------------ block helpers
// Exclusive scan over the block (blockDim.x a multiple of 32, <= 1024);
// *total = block sum.  sh: 33 ints.
__device__ __forceinline__ int block_excl_scan(int v, int *sh, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
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
    if (warp == 0) {
        const int wv = lane < nw ? sh[lane] : 0;
        int wi = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o)
                wi += n;
        }
        if (lane < nw)
            sh[lane] = wi - wv;
        if (lane == 31)
            sh[32] = wi;
    }
    __syncthreads();
    const int r = sh[warp] + incl - v;
    *total = sh[32];
    __syncthreads();
    return r;
}

// Fixed-order tree sum of one double per thread (blockDim.x a power of two).
__device__ __forceinline__ double block_sum(double v, double *sh)
{
    sh[threadIdx.x] = v;
    __syncthreads();
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if ((int)threadIdx.x < s)
            sh[threadIdx.x] += sh[threadIdx.x + s];
        __syncthreads();
    }
    const double r = sh[0];
    __syncthreads();
    return r;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier on a monotonically increasing counter; `target` = number
// of arrivals this barrier completes at.  Bounded: on timeout the status word
// records MOE_DEVICE_PIPELINE_TIMEOUT and false is returned (the caller then
// stops; downstream kernels see the status and skip their work).
__device__ bool grid_barrier(unsigned *counter, unsigned target, int32_t *status, int *sh_ok)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(counter, 1u);
        bool ok = true;
        if (ld_acquire(counter) < target) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire(counter) < target) {
                __nanosleep(64);
                if (global_timer_ns() - t0 > kBarrierLimitNs) {
                    set_status(status, MOE_DEVICE_PIPELINE_TIMEOUT);
                    ok = false;
                    break;
                }
            }
        }
        __threadfence();
        *sh_ok = ok;
    }
    __syncthreads();
    return *sh_ok != 0;
}

// ------------------------------------------------------------ fused router
template <int RT>
__device__ __forceinline__ void router_slice(const uint8_t *x_row, const uint8_t *wr_s, int D,
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

// ------------------------------------------------------------ phase 1: gate
// Routes token t (one warp); returns nothing, writes outputs and the chunk's
// shared-memory statistics (pbuf row, mask bits, ibuf row).
template <int EPL, int RT>
__device__ __forceinline__ void gate_token(const DispatchParams &p, const uint8_t *wr_s, int t,
                                           int tt, float *pbuf, int32_t *ibuf, uint32_t *mask)
{
    const int lane = threadIdx.x & 31;
    const int E = p.E, k = p.k;
    float s[EPL];
    if constexpr (RT != ROUTER_NONE) {
        float acc[kFusedMaxE];
#pragma unroll
        for (int e = 0; e < kFusedMaxE; ++e)
            acc[e] = 0.f;
        const uint8_t *x_row = static_cast<const uint8_t *>(p.x) + (size_t)t * p.row_bytes;
        for (int v = lane; v < p.D / 8; v += 32)
            router_slice<RT>(x_row, wr_s, p.D, E, v, acc);
        s[0] = -FLT_MAX;
#pragma unroll
        for (int e = 0; e < kFusedMaxE; ++e) {
            if (e < E) {
                const float v = warp_sum_bcast(acc[e]);
                if (lane == e)
                    s[0] = v;
            }
        }
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
                if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
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
}

// --------------------------------------------------------- the whole kernel
template <int EPL, int RT>
__global__ void __launch_bounds__(kDispatchThreads, 1) dispatch_kernel(DispatchParams p)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ int sh_int[33];
    __shared__ double sh_dbl[kDispatchThreads];
    __shared__ int sh_flag;
    const int E = p.E, k = p.k;
    const size_t wr_bytes =
        RT == ROUTER_NONE ? 0 : (size_t)E * p.D * (RT == ROUTER_BF16 ? 2 : 4);
    float *pbuf = reinterpret_cast<float *>(dsm + wr_bytes);
    int32_t *ibuf = reinterpret_cast<int32_t *>(pbuf + kChunk * E);
    uint32_t *mask = reinterpret_cast<uint32_t *>(ibuf + kChunk * k);
    unsigned *bar_counter = reinterpret_cast<unsigned *>(p.status + 9);
    const unsigned G = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if constexpr (RT != ROUTER_NONE) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.W_r);
        uint4 *dst = reinterpret_cast<uint4 *>(dsm);
        for (size_t i = threadIdx.x; i < wr_bytes / 16; i += blockDim.x)
            dst[i] = __ldg(src + i);
    }

    // ---- phase 1: gate, chunk by chunk
    for (int chunk = blockIdx.x; chunk < p.nchunk; chunk += G) {
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            mask[e] = 0u;
        __syncthreads();
        const int t = chunk * kChunk + warp;
        if (t < p.T) {
            gate_token<EPL, RT>(p, dsm, t, warp, pbuf, ibuf, mask);
        } else {
            for (int e = lane; e < E; e += 32)
                pbuf[warp * E + e] = 0.f;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            p.hist[(size_t)e * p.nchunk + chunk] = __popc(mask[e]);
            float acc = 0.f;
#pragma unroll 8
            for (int u = 0; u < kChunk; ++u)
                acc += pbuf[u * E + e];
            p.ppart[(size_t)e * p.nchunk + chunk] = acc;
        }
        for (int i = threadIdx.x; i < kChunk * k; i += blockDim.x) {
            const int u = i / k, j = i % k;
            const int tok = chunk * kChunk + u;
            if (tok < p.T) {
                const int e = ibuf[u * k + j];
                p.rank[(size_t)tok * k + j] = (uint8_t)__popc(mask[e] & ((1u << u) - 1u));
            }
        }
        __syncthreads();
    }
    if (!grid_barrier(bar_counter, G, p.status, &sh_flag))
        return;

    // ---- phase 2: per-expert scan; the last expert done finalizes
    for (int e = blockIdx.x; e < E; e += G) {
        int32_t *h = p.hist + (size_t)e * p.nchunk;
        const float *pp = p.ppart + (size_t)e * p.nchunk;
        const int per = (p.nchunk + blockDim.x - 1) / blockDim.x;
        const int beg = min(p.nchunk, (int)threadIdx.x * per);
        const int end = min(p.nchunk, beg + per);
        int local = 0;
        double pl = 0.0;
        for (int c = beg; c < end; ++c) {
            local += __ldcg(h + c);
            pl += (double)__ldcg(pp + c);
        }
        int total;
        int run = block_excl_scan(local, sh_int, &total);
        for (int c = beg; c < end; ++c) {
            const int v = __ldcg(h + c);
            h[c] = run;
            run += v;
        }
        const double ps = block_sum(pl, sh_dbl);
        if (threadIdx.x == 0) {
            p.expert_counts[e] = total;
            p.psum[e] = ps;
            __threadfence();
            sh_flag = (atomicAdd(reinterpret_cast<unsigned *>(p.status + 8), 1u) ==
                       (unsigned)E - 1u);
        }
        __syncthreads();
        if (sh_flag) {
            __threadfence();
            const int x = threadIdx.x;  // this thread's expert in the finalize
            const int n = x < E ? __ldcg(p.expert_counts + x) : 0;
            const int kept = (p.C < 0) ? n : (int)min((long long)n, p.C);
            if (x < E)
                p.kept_counts[x] = kept;
            int tot;
            const int off = block_excl_scan(kept, sh_int, &tot);
            if (x < E)
                p.seg_off[x] = off;
            if (x == 0)
                p.seg_off[E] = tot;
            const int mt = (kept + kTileM - 1) / kTileM;
            int mt_total;
            const int moff = block_excl_scan(mt, sh_int, &mt_total);
            if (x < E)
                p.mtile[x] = moff;
            if (x == 0)
                p.mtile[E] = mt_total;
            double term = 0.0;
            if (x < E && p.T > 0)
                term = ((double)n / ((double)p.T * (double)k)) *
                       (__ldcg(p.psum + x) / (double)p.T);
            const double sum = block_sum(term, sh_dbl);
            if (x == 0)
                *p.aux_loss = (float)((double)p.alpha * (double)E * sum);
        }
        __syncthreads();
    }
    if (!grid_barrier(bar_counter, 2 * G, p.status, &sh_flag))
        return;

    // ---- phase 3: scatter, one warp per token
    const size_t nv = p.row_bytes / 16;
    for (int t = blockIdx.x * kChunk + warp; t < p.T; t += G * kChunk) {
        long long row = -1;
        if (lane < k) {
            const int e = __ldcg(p.topk_idx + (size_t)t * k + lane);
            const long long pos = (long long)__ldcg(p.hist + (size_t)e * p.nchunk + t / kChunk) +
                                  __ldcg(p.rank + (size_t)t * k + lane);
            const bool kept = (p.C < 0) || (pos < p.C);
            row = kept ? (long long)__ldcg(p.seg_off + e) + pos : -1;
            p.dropped[(size_t)t * k + lane] = kept ? 0 : 1;
            p.row_of[(size_t)t * k + lane] = (int32_t)row;
            if (p.row_tok && row >= 0) {
                p.row_tok[row] = t;
                p.row_w[row] = __ldcg(p.topk_w + (size_t)t * k + lane);
            }
        }
        long long rows[kMaxTopK];
        bool any = false;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            rows[j] = __shfl_sync(0xffffffffu, row, j);
            any |= (j < k && rows[j] >= 0);
        }
        const uint8_t *src = static_cast<const uint8_t *>(p.x) + (size_t)t * p.row_bytes;
        if (nv * 16 == p.row_bytes) {
            for (size_t v = lane; v < nv; v += 32) {
                const uint4 val = __ldg(reinterpret_cast<const uint4 *>(src) + v);
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j)
                    if (j < k && rows[j] >= 0)
                        reinterpret_cast<uint4 *>(p.x_perm + (size_t)rows[j] * p.row_bytes)[v] =
                            val;
            }
        } else {  // fp32 rows whose size is not a multiple of 16 bytes
            for (size_t v = lane; v < p.row_bytes / 4; v += 32) {
                const uint32_t val = __ldg(reinterpret_cast<const uint32_t *>(src) + v);
#pragma unroll
                for (int j = 0; j < kMaxTopK; ++j)
                    if (j < k && rows[j] >= 0)
                        reinterpret_cast<uint32_t *>(p.x_perm + (size_t)rows[j] * p.row_bytes)[v] =
                            val;
            }
        }
        if (p.y_zero && !any) {
            uint4 *dst = reinterpret_cast<uint4 *>(p.y_zero + (size_t)t * p.row_bytes);
            for (size_t v = lane; v < nv; v += 32)
                dst[v] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

bool router_fused(const moe_config &c)
{
    const size_t esz = c.dtype == MOE_DTYPE_BF16 ? 2 : 4;
    return c.n_experts <= kFusedMaxE && c.d_model % 8 == 0 &&
           (size_t)c.n_experts * c.d_model * esz <= (size_t)kFusedMaxWrBytes;
}

bool direct_y(const moe_config &c) { return c.top_k == 1 && c.d_shared == 0; }

template <int EPL, int RT>
static cudaError_t launch_dispatch_t(const DispatchParams &p, size_t smem, cudaStream_t stream)
{
    auto kern = dispatch_kernel<EPL, RT>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    static uint64_t configured = 0;
    static int max_blocks[64] = {0};
    if (dev < 64 && !(configured & (1ull << dev))) {
        const size_t smem_max = kFusedMaxWrBytes + kChunk * (kMaxExperts + kMaxTopK) * 4 +
                                kMaxExperts * 4;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem_max);
        if (err != cudaSuccess)
            return err;
        int per_sm = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDispatchThreads,
                                                            smem_max);
        if (err != cudaSuccess)
            return err;
        max_blocks[dev] = std::max(1, per_sm) * sm_count();
        configured |= 1ull << dev;
    }
    const int want = std::max(p.nchunk, p.E);
    const int grid = std::max(1, std::min(want, dev < 64 ? max_blocks[dev] : sm_count()));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDispatchThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_dispatch(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                            const void *x, const void *W_r, bool fused, float *logits,
                            const float *bias, int32_t *topk_idx, float *topk_w,
                            uint8_t *dropped_mask, int32_t *expert_counts, int32_t *kept_counts,
                            float *aux_loss, void *y, cudaStream_t stream)
{
    DispatchParams p;
    const size_t esz = c.dtype == MOE_DTYPE_BF16 ? 2 : 4;
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
    p.C = L.C;
    p.alpha = c.aux_alpha;
    p.row_bytes = (size_t)c.d_model * esz;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.dropped = dropped_mask;
    p.expert_counts = expert_counts;
    p.kept_counts = kept_counts;
    p.aux_loss = aux_loss;
    p.hist = reinterpret_cast<int32_t *>(ws + L.hist);
    p.ppart = reinterpret_cast<float *>(ws + L.ppart);
    p.rank = ws + L.rank;
    p.psum = reinterpret_cast<double *>(ws + L.psum);
    p.seg_off = reinterpret_cast<int32_t *>(ws + L.seg_off);
    p.mtile = reinterpret_cast<int32_t *>(ws + L.mtile);
    p.row_of = reinterpret_cast<int32_t *>(ws + L.row_of);
    p.x_perm = ws + L.x_perm;
    const bool dy = direct_y(c) && c.dtype == MOE_DTYPE_BF16;
    p.row_tok = dy ? reinterpret_cast<int32_t *>(ws + L.row_tok) : nullptr;
    p.row_w = dy ? reinterpret_cast<float *>(ws + L.row_w) : nullptr;
    p.y_zero = dy ? static_cast<uint8_t *>(y) : nullptr;
    p.status = reinterpret_cast<int32_t *>(ws + L.status);
    const size_t smem = (fused ? (size_t)c.n_experts * c.d_model * esz : 0) +
                        (size_t)kChunk * (c.n_experts + c.top_k) * 4 + (size_t)c.n_experts * 4;
    if (fused)
        return c.dtype == MOE_DTYPE_BF16 ? launch_dispatch_t<1, ROUTER_BF16>(p, smem, stream)
                                         : launch_dispatch_t<1, ROUTER_F32>(p, smem, stream);
    const int epl = (c.n_experts + 31) / 32;
    if (epl <= 1)
        return launch_dispatch_t<1, ROUTER_NONE>(p, smem, stream);
    if (epl <= 2)
        return launch_dispatch_t<2, ROUTER_NONE>(p, smem, stream);
    if (epl <= 4)
        return launch_dispatch_t<4, ROUTER_NONE>(p, smem, stream);
    return launch_dispatch_t<8, ROUTER_NONE>(p, smem, stream);
}

}  // namespace moe
