// moe_dispatch.cu -- routing and dispatch in one cooperative kernel with a
// single grid-wide barrier.  Block b owns a contiguous run of tokens (whole
// chunks of cs = 8, 16 or 32 tokens):
//
//   phase 1 (gate):     chunk by chunk, one warp per token: (the router GEMM
//                       itself when W_r fits in shared memory), softmax over
//                       all E, top-k with the lower index first on equal
//                       scores, gate weights; the chunk's per-expert
//                       probability sums; each assignment's rank among the
//                       block's earlier tokens that chose the same expert
//                       (a running count plus the popcount of a per-chunk
//                       token bitmask); finally the block's per-expert counts;
//   -- grid barrier --
//   phase 2 (scatter):  every block reads all blocks' counts and derives,
//                       identically, the demand counts n_e, kept_e = min(n_e, C),
//                       the segment offsets and the 128-row tile prefix, plus
//                       its own per-expert base (tokens of earlier blocks).
//                       The global token-order position of an assignment is
//                       base + rank; it is kept iff position < C.  The block
//                       writes its assignments' rows and copies x into the
//                       rows of its experts' segments.  Per-expert
//                       probability sums (fp64, fixed order) are spread over
//                       the blocks; the first expert kernel, which starts
//                       after this one completes, evaluates the balance loss.
// All blocks are co-resident (cooperative launch); the barrier wait is
// bounded in time.
//
// A batch split over several ranks runs the kernel twice with an exchange
// of per-expert statistics in between (phases): the first launch gates and
// stops after the demand counts and probability sums of this rank's tokens;
// the second, given every rank's counts, places this rank's assignments at
// global token-order positions (the counts of earlier ranks come first), so
// that capacity drops fall exactly where they would for the whole batch.
//
// Sources: "Mixture of Experts: More Parameters, Same FLOPs" ('The router');
// "Mixture of Experts" (module 17), 17.2 (softmax over the selected vs over
// all experts), 17.4 (balance loss) and 17.5 (capacity equation; tokens beyond
// C are dropped by that expert only); "Mixture of Experts: Sparse FFNs,
// Routers, and Shared Experts" ('Capacity factor'); "Mixture of experts"
// (frontiers track), gate equation of 'Where the experts live'.
#include <algorithm>
#include <atomic>
#include <cfloat>
#include <climits>
#include <cuda_bf16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "tc_ptx.cuh"

namespace moe {

constexpr int kDispatchThreads = kChunk * 32;  // 32 warps: one per token of a chunk
constexpr int kFusedMaxE = 16;
constexpr int kFusedMaxWrBytes = 64 * 1024;
constexpr uint64_t kBarrierLimitNs = 2000000000ull;
constexpr size_t kStageMaxBytes = 96 * 1024;  // most x bytes a block stages in shared memory

enum { ROUTER_NONE = 0, ROUTER_BF16 = 1, ROUTER_F32 = 2 };

struct DispatchParams {
    float *logits;          // [T,E]: raw scores in (unless fused), scores (+bias) out
    const float *lpart;     // [lsplit][T][E] router partial scores, or null
    int lsplit;
    const float *bias;      // [E] or null
    int bias_sel_only;      // 1: the bias shifts only the selection keys
    const void *x;          // [T,D]
    const void *W_r;        // [E,D] (fused router only)
    int T, E, k, mode, D;
    int cs;                 // tokens per chunk (1, 2, 4, 8, 16 or 32)
    int nchunk;             // ceil(T / cs)
    int cpb;                // chunks per block
    int x_staged;           // 1: the block's x rows are staged in shared memory (cpb == 1)
    long long C;            // capacity, -1 = dropless
    float alpha;
    size_t row_bytes;       // D * element size
    int32_t *topk_idx;      // [T,k]
    float *topk_w;          // [T,k]
    uint8_t *dropped;       // [T,k]
    int32_t *expert_counts; // [E]
    int32_t *kept_counts;   // [E]
    int32_t *bcount;        // [E][gridDim.x] per-block expert counts
    float *ppart;           // [E][nchunk] per-chunk probability sums
    int32_t *rank;          // [T*k] rank among the block's earlier tokens of the expert
    double *psum;           // [E]
    int32_t *seg_off;       // [E+1]
    int32_t *mtile;         // [E+1]
    int32_t *row_of;        // [T*k]
    uint8_t *x_perm;        // [R_max, D]
    int32_t *row_tok;       // [R_max] token of each x_perm row (direct-y mode), or null
    float *row_w;           // [R_max] gate weight of each row (direct-y mode), or null
    uint8_t *y_zero;        // y [T,D]: rows of fully dropped tokens are zeroed (direct-y)
    int32_t *status;        // [0] status word, [9] barrier counter
    // split batch (all_counts non-null): phases 1 = gate and statistics only,
    // 2 = placement only (the gate's results are in the workspace), 3 = both
    int phases;
    const int32_t *all_counts;  // [n_ranks][E] demand counts of every rank, or null
    const double *all_psum;     // [n_ranks][E] probability sums of every rank
    int n_ranks, rank_id;
    long long TK_global;        // assignments over all ranks (T_global * k)
    int32_t *gcount;            // [E] out: demand counts over all ranks
    // the grid barrier waits for gridDim.x + barrier_extra arrivals, for at
    // most barrier_limit_ns (barrier_extra is 0 except under the test hook
    // moe_debug_barrier_fault, which makes the barrier run out)
    unsigned barrier_extra;
    unsigned long long barrier_limit_ns;
    long long R_max;            // rows of x_perm (bound of every row index)
    // gather source other than x (E4M3 token rows): rows of g_row_bytes
    // copied into x_perm (then rows of g_row_bytes too), and each row's
    // scale gscale[t] into gscale_perm[row]; gx null: x rows are copied
    const uint8_t *gx;
    size_t g_row_bytes;
    const float *gscale;
    float *gscale_perm;
};

// Phase stamps of each dispatch block (builds with MOE_TIMELINE; read
// through moe_timeline_read): 8 global-timer words per block, block < 4096.
constexpr int kDispatchTimelineBlocks = 4096;
#ifdef MOE_TIMELINE
__device__ unsigned long long g_dispatch_timeline[kDispatchTimelineBlocks * 8];
#else
__device__ unsigned long long g_dispatch_timeline[8];
#endif

__device__ __forceinline__ void dispatch_stamp(int word)
{
    if constexpr (kTimeline) {
        if (threadIdx.x == 0 && blockIdx.x < kDispatchTimelineBlocks)
            g_dispatch_timeline[blockIdx.x * 8 + word] = global_timer_ns();
    }
}

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

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier on a counter that starts at zero; `target` = number of
// blocks.  Bounded: after limit_ns the status word records
// MOE_DEVICE_PIPELINE_TIMEOUT and false is returned (the caller then stops;
// downstream kernels see the status and skip their work).
__device__ bool grid_barrier(unsigned *counter, unsigned target, int32_t *status, int *sh_ok,
                             unsigned long long limit_ns)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(counter, 1u);
        bool ok = true;
        if (ld_acquire(counter) < target) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire(counter) < target) {
                __nanosleep(32);
                if (global_timer_ns() - t0 > limit_ns) {
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
__device__ __forceinline__ void cvt8(const uint4 &q, float (&f)[8])
{
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 g = __bfloat1622float2(h[i]);
        f[2 * i] = g.x;
        f[2 * i + 1] = g.y;
    }
}

__device__ __forceinline__ void cvt8(const float4 &a, const float4 &b, float (&f)[8])
{
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr)
                 : "memory");
    return r;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t r;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(r) : "r"(addr) : "memory");
    return r;
}

// Eight consecutive elements (8-element vector v of a bf16 or fp32 row that
// starts at shared-memory address `row`) as fp32.
template <int RT>
__device__ __forceinline__ void lds8(uint32_t row, int v, float (&f)[8])
{
    if (RT == ROUTER_BF16) {
        cvt8(lds128(row + (uint32_t)v * 16u), f);
    } else {
        const uint4 a = lds128(row + (uint32_t)v * 32u), b = lds128(row + (uint32_t)v * 32u + 16u);
        cvt8(make_float4(__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z),
                         __uint_as_float(a.w)),
             make_float4(__uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z),
                         __uint_as_float(b.w)),
             f);
    }
}

// acc[e] += x[8v .. 8v+7] . W_r[r_e][8v .. 8v+7] for e < EM, r_e = min(e, E-1)
// (W_r staged in shared memory at `wr`, row stride `wstride` bytes): no
// branch on E, so the loads of all EM rows can be issued together; the sums
// of e >= E are discarded later.
template <int RT, int EM>
__device__ __forceinline__ void router_fma(const float (&xf)[8], uint32_t wr, uint32_t wstride,
                                           int E, int v, float (&acc)[EM])
{
#pragma unroll
    for (int e = 0; e < EM; ++e) {
        float wf[8];
        lds8<RT>(wr + (uint32_t)min(e, E - 1) * wstride, v, wf);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[e] = fmaf(xf[i], wf[i], acc[e]);
    }
}

// Sum of each of the EM values over the warp's 32 lanes, halving the vector
// at each exchange (EM - 1 + 5 - log2(EM) shuffles instead of 5 * EM).
// Afterwards lane L holds the sum of value L / (32 / EM).
template <int EM>
__device__ __forceinline__ float warp_sum_vector(float (&a)[EM])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int half = EM / 2, o = 16; half >= 1; half /= 2, o /= 2) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? a[i] : a[i + half];
            const float keep = up ? a[i + half] : a[i];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float r = a[0];
#pragma unroll
    for (int o = 16 / EM; o > 0; o >>= 1)
        r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

// CUDA-core router, one warp's part of one token's scores: the 8-element
// vectors part*32+lane, part*32+lane + nparts*32, ... of the token's row
// against W_r (staged in shared memory).  The row is in shared memory
// (x_smem, staged) or in global memory (x_glob; read several vectors at a
// time so that the loads overlap).  Writes out[e] (e < E) = this part's sum.
template <int RT, int EM>
__device__ __forceinline__ void router_part(uint32_t x_smem, const uint8_t *x_glob, uint32_t wr,
                                            uint32_t wstride, int D, int E, int part, int nparts,
                                            float *out)
{
    const int lane = threadIdx.x & 31;
    float acc[EM];
#pragma unroll
    for (int e = 0; e < EM; ++e)
        acc[e] = 0.f;
    const int nv = D / 8, step = nparts * 32;
    if (!x_glob) {
        for (int v = part * 32 + lane; v < nv; v += step) {
            float xf[8];
            lds8<RT>(x_smem, v, xf);
            router_fma<RT, EM>(xf, wr, wstride, E, v, acc);
        }
    } else {
        constexpr int B = RT == ROUTER_BF16 ? 4 : 2;
        for (int v0 = part * 32 + lane; v0 < nv; v0 += step * B) {
            if (RT == ROUTER_BF16) {
                const uint4 *src = reinterpret_cast<const uint4 *>(x_glob);
                uint4 q[B];
#pragma unroll
                for (int u = 0; u < B; ++u)
                    if (v0 + step * u < nv)
                        q[u] = __ldg(src + v0 + step * u);
#pragma unroll
                for (int u = 0; u < B; ++u)
                    if (v0 + step * u < nv) {
                        float xf[8];
                        cvt8(q[u], xf);
                        router_fma<RT, EM>(xf, wr, wstride, E, v0 + step * u, acc);
                    }
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(x_glob);
                float4 qa[B], qb[B];
#pragma unroll
                for (int u = 0; u < B; ++u)
                    if (v0 + step * u < nv) {
                        qa[u] = __ldg(src + 2 * (v0 + step * u));
                        qb[u] = __ldg(src + 2 * (v0 + step * u) + 1);
                    }
#pragma unroll
                for (int u = 0; u < B; ++u)
                    if (v0 + step * u < nv) {
                        float xf[8];
                        cvt8(qa[u], qb[u], xf);
                        router_fma<RT, EM>(xf, wr, wstride, E, v0 + step * u, acc);
                    }
            }
        }
    }
    const float r = warp_sum_vector<EM>(acc);
    constexpr int kGroup = 32 / EM;
    const int e = lane / kGroup;
    if (lane % kGroup == 0 && e < E)
        out[e] = r;
}

// D += A * B on the tensor cores, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kRouterMmaWarps = 8;

// Tensor-core router for bf16: scores of the chunk's nt (<= 32) tokens,
// staged in shared memory (rows at xs, stride xstride bytes), against W_r
// (rows at wr, stride wstride).  Warp q < kRouterMmaWarps takes the 16-wide
// k-steps q, q+8, ... of D; the A fragments are token rows (tokens >= nt
// read as zero), the B fragments W_r rows (rows >= E clamped to E-1, their
// sums unused).  Writes this warp's partial sums to rp[(q*32 + token)*16 + e].
template <int EM>
__device__ __forceinline__ void router_mma(uint32_t xs, uint32_t xstride, int nt, uint32_t wr,
                                           uint32_t wstride, int D, int E, int q, float *rp)
{
    constexpr int NT = EM > 8 ? 2 : 1;  // 8-expert n-tiles
    const int lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
    const int mt = nt > 16 ? 2 : 1;
    float c[2][NT][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                c[m][n][i] = 0.f;
    for (int ks = q; ks < D / 16; ks += kRouterMmaWarps) {
        const uint32_t kb = (uint32_t)(ks * 16 + tq * 2) * 2u;
        uint32_t b[NT][2];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const uint32_t row = wr + (uint32_t)min(n * 8 + g, E - 1) * wstride + kb;
            b[n][0] = lds32(row);
            b[n][1] = lds32(row + 16u);
        }
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            if (m < mt) {
                const int r0 = m * 16 + g, r1 = r0 + 8;
                const uint32_t a0 = r0 < nt ? lds32(xs + (uint32_t)r0 * xstride + kb) : 0u;
                const uint32_t a1 = r1 < nt ? lds32(xs + (uint32_t)r1 * xstride + kb) : 0u;
                const uint32_t a2 = r0 < nt ? lds32(xs + (uint32_t)r0 * xstride + kb + 16u) : 0u;
                const uint32_t a3 = r1 < nt ? lds32(xs + (uint32_t)r1 * xstride + kb + 16u) : 0u;
#pragma unroll
                for (int n = 0; n < NT; ++n)
                    mma_16816(c[m][n], a0, a1, a2, a3, b[n][0], b[n][1]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        if (m < mt) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int r0 = m * 16 + g, col = n * 8 + tq * 2;
                if (r0 < nt) {
                    rp[(q * 32 + r0) * kFusedMaxE + col] = c[m][n][0];
                    rp[(q * 32 + r0) * kFusedMaxE + col + 1] = c[m][n][1];
                }
                if (r0 + 8 < nt) {
                    rp[(q * 32 + r0 + 8) * kFusedMaxE + col] = c[m][n][2];
                    rp[(q * 32 + r0 + 8) * kFusedMaxE + col + 1] = c[m][n][3];
                }
            }
        }
    }
}

// Integer key with the order of the finite floats (-0 and +0 equal).
__device__ __forceinline__ int order_key(float v)
{
    const int i = __float_as_int(v + 0.0f);
    return i >= 0 ? i : i ^ 0x7FFFFFFF;
}

__device__ __forceinline__ float key_value(int key)
{
    return __int_as_float(key >= 0 ? key : key ^ 0x7FFFFFFF);
}

// ------------------------------------------------------------ phase 1: gate
// Routes token t (one warp, slot tt of the chunk); writes the per-token
// outputs and the chunk's shared-memory statistics (pbuf row, mask bits,
// ibuf row).  x_row: the token's row (shared or global memory).
// rpart: the token's router partial sums (fused router), nparts of them at
// a stride of pstride floats, summed in order.
template <int EPL, int RT>
__device__ __forceinline__ void gate_token(const DispatchParams &p, const float *rpart,
                                           int nparts, int pstride, int t, int tt, float *pbuf,
                                           int32_t *ibuf, float *wbuf, uint32_t *mask)
{
    const int lane = threadIdx.x & 31;
    const int E = p.E, k = p.k;
    float s[EPL];
    // scores: the fused router's partial sums (parts in order), or the
    // router GEMM's output; then the optional bias.  All loads come before
    // the stores to the scores so that they overlap.
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        float v = -FLT_MAX;
        if (e < E) {
            if (RT != ROUTER_NONE) {
                v = rpart[e];
                for (int q = 1; q < nparts; ++q)
                    v += rpart[q * pstride + e];
            } else if (p.lpart) {
                // all partial loads first, then the sum in split order
                float part[kMaxRouterSplits];
#pragma unroll
                for (int q = 0; q < kMaxRouterSplits; ++q)
                    part[q] = q < p.lsplit ? p.lpart[((size_t)q * p.T + t) * E + e] : 0.f;
                v = part[0];
#pragma unroll
                for (int q = 1; q < kMaxRouterSplits; ++q)
                    if (q < p.lsplit)
                        v += part[q];
            } else {
                v = p.logits[(size_t)t * E + e];
            }
        }
        s[i] = v;
    }
    // the bias: part of the scores, or (selection-only) of the top-k keys
    const bool sel_bias = p.bias && p.bias_sel_only;
    float bv[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        bv[i] = p.bias && lane + 32 * i < E ? __ldg(p.bias + lane + 32 * i) : 0.f;
    if (p.bias && !sel_bias) {
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            s[i] += bv[i];
    }
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            if (RT != ROUTER_NONE || (p.bias && !sel_bias) || p.lpart)
                p.logits[(size_t)t * E + e] = s[i];
            bad |= !isfinite(s[i]) || !isfinite(bv[i]);
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0)
        set_status(p.status, MOE_DEVICE_NONFINITE_SCORE);

    // router probabilities over all E: softmax (max subtracted), or for the
    // sigmoid mode the sigmoids normalised over all E (balance loss only)
    const bool sigm = p.mode == MOE_GATE_SIGMOID_SELECTED;
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
        ex[i] = (lane + 32 * i < E) ? (sigm ? 1.f / (1.f + expf(-s[i])) : expf(s[i] - m)) : 0.f;
        z += ex[i];
    }
    z = warp_sum_bcast(z);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E)
            pbuf[tt * E + e] = ex[i] / z;
    }

    // top-k: k rounds of a warp arg-max over order keys (redux max), equal
    // keys resolved to the lower expert index (redux min); lane j keeps
    // round j's expert and (unbiased) score
    int key[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        key[i] = (lane + 32 * i < E) ? order_key(sel_bias ? s[i] + bv[i] : s[i]) : INT_MIN;
    uint32_t taken = 0u;
    float my_s = 0.f, s_top = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; ++j) {
        int bk = INT_MIN, be = INT_MAX;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            if (lane + 32 * i < E && !((taken >> i) & 1u) && (be == INT_MAX || key[i] > bk)) {
                bk = key[i];
                be = lane + 32 * i;
            }
        }
        const int mk = __reduce_max_sync(0xffffffffu, bk);
        int win = __reduce_min_sync(0xffffffffu, bk == mk ? be : INT_MAX);
        if (win == INT_MAX || win >= E)
            win = 0;  // unreachable with k <= E; keeps indices in bounds
        if ((win & 31) == lane)
            taken |= 1u << (win >> 5);
        float sv = key_value(mk);
        if (sel_bias) {
            // the winner's score without the bias, from the lane that holds it
            float cand = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (i == (win >> 5))
                    cand = s[i];
            sv = __shfl_sync(0xffffffffu, cand, win & 31);
        }
        if (lane == j) {
            my_s = sv;
            my_e = win;
        }
    }
    // largest selected score (subtracted for range only)
    s_top = warp_max(lane < k ? my_s : -FLT_MAX);

    // gate weights, lane j for assignment j
    float w = 0.f;
    if (p.mode == MOE_GATE_SOFTMAX_SELECTED) {
        const float ev = lane < k ? expf(my_s - s_top) : 0.f;
        w = ev / warp_sum_bcast(ev);
    } else if (sigm) {
        const float a = lane < k ? 1.f / (1.f + expf(-my_s)) : 0.f;
        w = a / warp_sum_bcast(a);
    } else {
        w = lane < k ? expf(my_s - m) / z : 0.f;
        if (p.mode == MOE_GATE_SOFTMAX_ALL_RENORM)
            w = w / warp_sum_bcast(w);
    }
    if (lane < k) {
        p.topk_idx[(size_t)t * k + lane] = my_e;
        p.topk_w[(size_t)t * k + lane] = w;
        atomicOr(&mask[my_e], 1u << tt);
        ibuf[tt * k + lane] = my_e;
        wbuf[tt * k + lane] = w;
    }
}

// ---------------------------------------------------------- phase 2 helpers
// Sum of v over the block (every thread receives it).
__device__ __forceinline__ long long block_sum_ll(long long v)
{
    __shared__ long long sh[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0)
        sh[warp] = v;
    __syncthreads();
    long long t = 0;
    for (int w = 0; w < nw; ++w)
        t += sh[w];
    __syncthreads();
    return t;
}

// Copies token t's row (src: shared or global memory, row_bytes long) into
// its kept rows of x_perm; this warp handles the 16-byte vectors
// part*32+lane, stepping by nparts*32 (four loads in flight before their
// stores).
__device__ __forceinline__ void copy_row(const DispatchParams &p, const uint8_t *src,
                                         size_t row_bytes, const long long (&rows)[kMaxTopK],
                                         int part, int nparts)
{
    const int lane = threadIdx.x & 31, k = p.k;
    const size_t nv = row_bytes / 16;
    if (nv * 16 == row_bytes) {
        const size_t step = (size_t)nparts * 32;
        size_t v = (size_t)part * 32 + lane;
        for (; v + 3 * step < nv; v += 4 * step) {
            uint4 q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                q[u] = reinterpret_cast<const uint4 *>(src)[v + u * step];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)
                if (j < k && rows[j] >= 0) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.x_perm + (size_t)rows[j] * row_bytes);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        dst[v + u * step] = q[u];
                }
        }
        for (; v < nv; v += step) {
            const uint4 q = reinterpret_cast<const uint4 *>(src)[v];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)
                if (j < k && rows[j] >= 0)
                    reinterpret_cast<uint4 *>(p.x_perm + (size_t)rows[j] * row_bytes)[v] = q;
        }
    } else {  // fp32 rows whose size is not a multiple of 16 bytes
        const size_t nw = row_bytes / 4;
        for (size_t v = (size_t)part * 32 + lane; v < nw; v += (size_t)nparts * 32) {
            const uint32_t q = reinterpret_cast<const uint32_t *>(src)[v];
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)
                if (j < k && rows[j] >= 0)
                    reinterpret_cast<uint32_t *>(p.x_perm + (size_t)rows[j] * row_bytes)[v] = q;
        }
    }
}

// Probability sums of the experts e = b, b+G, ... (this warp; fp64, lanes
// over chunks in a fixed order, then a fixed butterfly).  The balance loss
// itself is evaluated by the first expert kernel.
__device__ __forceinline__ void prob_sums(const DispatchParams &p, int b, int G)
{
    const int lane = threadIdx.x & 31, E = p.E;
    for (int e = b; e < E; e += G) {
        const float *pp = p.ppart + (size_t)e * p.nchunk;
        double acc = 0.0;
        for (int c0 = lane; c0 < p.nchunk; c0 += 32 * 4) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = c0 + 32 * u < p.nchunk ? __ldcg(pp + c0 + 32 * u) : 0.f;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                acc += (double)v[u];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0)
            p.psum[e] = acc;
    }
}

// --------------------------------------------------------- the whole kernel
// EPL: experts per lane (ceil(E / 32)); RT: fused router type; EM: the
// fused router's expert count rounded up to 4, 8 or 16; SPLIT: 0 = the whole
// layer's dispatch, 1 = a split batch's gate and statistics, 2 = a split
// batch's placement (separate instantiations keep the whole-layer kernel
// free of the split-batch code).
template <int EPL, int RT, int EM, int SPLIT>
__global__ void __launch_bounds__(kDispatchThreads, 1) dispatch_kernel(DispatchParams p)
{
    extern __shared__ __align__(16) uint8_t dsm[];
    __shared__ int sh_int[33];
    __shared__ int sh_flag;
    const int E = p.E, k = p.k, cs = p.cs;
    // staged rows carry 16 bytes of padding so that the tensor-core router's
    // fragment loads from consecutive rows fall in different banks
    const uint32_t wrow = RT == ROUTER_NONE ? 0u : (uint32_t)p.D * (RT == ROUTER_BF16 ? 2u : 4u);
    const uint32_t wstride = wrow + 16u;
    const size_t wr_bytes = RT == ROUTER_NONE ? 0 : (size_t)E * wstride;
    const uint32_t xstride = (uint32_t)p.row_bytes + 16u;
    const int G = gridDim.x, b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c_beg = b * p.cpb, c_end = min(p.nchunk, c_beg + p.cpb);
    const int t_beg = c_beg * cs, t_end = min(p.T, c_end * cs);
    const int ntok = t_end - t_beg;
    const size_t xs_bytes = p.x_staged ? (size_t)cs * xstride : 0;
    uint8_t *xs = dsm + wr_bytes;                                   // staged x rows
    float *pbuf = reinterpret_cast<float *>(xs + xs_bytes);         // [cs][E]
    int32_t *ibuf = reinterpret_cast<int32_t *>(pbuf + kChunk * E); // [cs][k]
    uint32_t *mask = reinterpret_cast<uint32_t *>(ibuf + kChunk * k);  // [E]
    int32_t *run = reinterpret_cast<int32_t *>(mask + E);          // [E] block-local counts
    int32_t *s_base = run + E;                                      // [E] counts of earlier blocks
    int32_t *s_n = s_base + E;                                      // [E] demand counts
    int32_t *s_seg = s_n + E;                                       // [E+1] segment offsets
    int32_t *s_rb = s_seg + E + 1;                                  // [E] earlier ranks' counts
    float *rpart = reinterpret_cast<float *>(s_rb + E);             // [8][32][16] router parts
    int32_t *rbuf = reinterpret_cast<int32_t *>(rpart + kRouterMmaWarps * kChunk * kFusedMaxE);
    float *wbuf = reinterpret_cast<float *>(rbuf + kChunk * kMaxTopK);  // [32][k] ranks, weights
    unsigned *bar_counter = reinterpret_cast<unsigned *>(p.status + 9);
    // the layout above must fit the shared memory this launch received (the
    // same test in every block, so no block is left waiting at the barrier)
    if ((size_t)(reinterpret_cast<uint8_t *>(wbuf + kChunk * kMaxTopK) - dsm) >
        dynamic_smem_bytes()) {
        if (b == 0 && threadIdx.x == 0)
            set_status(p.status, MOE_DEVICE_LAUNCH_MISMATCH);
        return;
    }

    constexpr bool gate = SPLIT != 2;
    // a one-chunk block keeps its assignments in shared memory from phase 1
    // to phase 2 when both run in this launch
    const bool held = gate && p.cpb == 1;
    // timeline: [0] start; [1] rows staged, [2] router done, [3] tokens
    // gated (the block's first chunk; a block without chunks keeps [0]);
    // [4] phase 1 done, [5] past the grid barrier, [6] segment tables done,
    // [7] the block's last copy warp done
    if constexpr (kTimeline) {
        if (threadIdx.x == 0 && b < kDispatchTimelineBlocks) {
            const unsigned long long t0 = global_timer_ns();
            unsigned long long *rec = g_dispatch_timeline + b * 8;
            rec[0] = rec[1] = rec[2] = rec[3] = t0;
            rec[7] = 0;
        }
    }

    // W_r (fused router) and this block's x rows (when staged) into shared
    // memory, four 16-byte loads in flight per thread
    if (gate) {
        const long long vpw = wrow > 0 ? wrow / 16 : 1, vpx = (long long)(p.row_bytes / 16);
        const long long n_w = RT == ROUTER_NONE ? 0 : (long long)E * vpw;
        const long long n = n_w + (p.x_staged ? (long long)ntok * vpx : 0);
        const uint4 *wsrc = reinterpret_cast<const uint4 *>(p.W_r);
        const uint4 *xsrc = reinterpret_cast<const uint4 *>(
            static_cast<const uint8_t *>(p.x) + (size_t)t_beg * p.row_bytes);
        for (long long i0 = threadIdx.x; i0 < n; i0 += 4 * blockDim.x) {
            uint4 q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const long long i = i0 + (long long)u * blockDim.x;
                if (i < n_w)
                    q[u] = __ldg(wsrc + i);
                else if (i < n)
                    q[u] = __ldg(xsrc + (i - n_w));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const long long i = i0 + (long long)u * blockDim.x;
                if (i < n_w)
                    *reinterpret_cast<uint4 *>(dsm + (i / vpw) * wstride + (i % vpw) * 16) = q[u];
                else if (i < n)
                    *reinterpret_cast<uint4 *>(xs + ((i - n_w) / vpx) * xstride +
                                               ((i - n_w) % vpx) * 16) = q[u];
            }
        }
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        run[e] = 0;

    // ---- phase 1: gate this block's chunks in token order
    for (int chunk = c_beg; gate && chunk < c_end; ++chunk) {
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            mask[e] = 0u;
        __syncthreads();
        if (chunk == c_beg)
            dispatch_stamp(1);
        // fused router: on the tensor cores for staged bf16 rows, else on
        // the CUDA cores with 32 / cs warps per token, each over a slice of D
        const bool mma_router = RT == ROUTER_BF16 && p.x_staged && cs >= 8;
        const int wpt = kChunk / cs;
        if constexpr (RT != ROUTER_NONE) {
            const uint32_t wr = smem_u32(dsm);
            if (mma_router) {
                if (warp < kRouterMmaWarps)
                    router_mma<EM>(smem_u32(xs), xstride, min(cs, p.T - chunk * cs), wr, wstride,
                                   p.D, E, warp, rpart);
            } else {
                const int tt = warp / wpt, part = warp - (warp / wpt) * wpt;
                const int t = chunk * cs + tt;
                if (t < p.T) {
                    const uint32_t x_smem = smem_u32(xs) + (uint32_t)(t - t_beg) * xstride;
                    const uint8_t *x_glob =
                        p.x_staged ? nullptr
                                   : static_cast<const uint8_t *>(p.x) + (size_t)t * p.row_bytes;
                    router_part<RT, EM>(x_smem, x_glob, wr, wstride, p.D, E, part, wpt,
                                        rpart + (size_t)warp * kFusedMaxE);
                }
            }
            __syncthreads();
        }
        if (chunk == c_beg)
            dispatch_stamp(2);
        const int t = chunk * cs + warp;
        if (warp < cs) {
            if (t < p.T) {
                if (mma_router)
                    gate_token<EPL, RT>(p, rpart + (size_t)warp * kFusedMaxE, kRouterMmaWarps,
                                        kChunk * kFusedMaxE, t, warp, pbuf, ibuf, wbuf, mask);
                else
                    gate_token<EPL, RT>(p, rpart + (size_t)warp * wpt * kFusedMaxE, wpt,
                                        kFusedMaxE, t, warp, pbuf, ibuf, wbuf, mask);
            } else {
                for (int e = lane; e < E; e += 32)
                    pbuf[warp * E + e] = 0.f;
            }
        }
        __syncthreads();
        if (chunk == c_beg)
            dispatch_stamp(3);
        // ranks: tokens of earlier chunks of this block (run, before this
        // chunk's counts are added) plus earlier tokens of this chunk
        for (int i = threadIdx.x; i < cs * k; i += blockDim.x) {
            const int u = i / k, j = i - (i / k) * k;
            const int tok = chunk * cs + u;
            if (tok < p.T) {
                int e = ibuf[u * k + j];
                if (kDebugBounds && (unsigned)e >= (unsigned)E) {
                    set_status(p.status, MOE_DEVICE_INDEX_OUT_OF_RANGE);
                    e = 0;
                }
                const int r = run[e] + __popc(mask[e] & ((1u << u) - 1u));
                p.rank[(size_t)tok * k + j] = r;
                rbuf[u * k + j] = r;
            }
        }
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            float acc = 0.f;
            for (int u = 0; u < cs; ++u)
                acc += pbuf[u * E + e];
            p.ppart[(size_t)e * p.nchunk + chunk] = acc;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            run[e] += __popc(mask[e]);
    }
    __syncthreads();
    dispatch_stamp(4);
    if (gate) {
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            p.bcount[(size_t)e * G + b] = run[e];
        // (no copy or other asynchronous work of this block is in flight
        // here, so a block whose wait runs out simply returns)
        if (!grid_barrier(bar_counter, (unsigned)G + p.barrier_extra, p.status, &sh_flag,
                          p.barrier_limit_ns))
            return;
    }
    dispatch_stamp(5);

    // ---- phase 2a: per expert, tokens of earlier blocks and the total
    // (warp w: experts w, w+32, ..., four at a time)
    for (int e0 = warp; e0 < E; e0 += 32 * 4) {
        int pre[4] = {0, 0, 0, 0}, tot[4] = {0, 0, 0, 0};
        for (int bb = lane; bb < G; bb += 32) {
            int v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + 32 * u;
                v[u] = e < E ? __ldcg(p.bcount + (size_t)e * G + bb) : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                tot[u] += v[u];
                pre[u] += bb < b ? v[u] : 0;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + 32 * u;
            const int ps = __reduce_add_sync(0xffffffffu, pre[u]);
            const int ts = __reduce_add_sync(0xffffffffu, tot[u]);
            if (lane == 0 && e < E) {
                s_base[e] = ps;
                s_n[e] = ts;
            }
        }
    }
    __syncthreads();
    if constexpr (SPLIT == 1) {
        // gate and statistics only: this rank's demand counts and
        // probability sums, for the exchange between the ranks
        if (b == 0)
            for (int e = threadIdx.x; e < E; e += blockDim.x)
                p.expert_counts[e] = s_n[e];
        if (warp == 31)
            prob_sums(p, b, G);
        return;
    }
    // ---- split batch: per expert, the assignments of earlier ranks (they
    // precede this rank's in global token order) and of all ranks; the
    // exchanged counts must hold this rank's own and add up to T_global * k
    if constexpr (SPLIT == 2) {
        const int x = threadIdx.x;
        long long before = 0, all = 0, own = 0;
        double ps = 0.0;
        if (x < E) {
            for (int r = 0; r < p.n_ranks; ++r) {
                const long long v = __ldg(p.all_counts + (size_t)r * E + x);
                before += r < p.rank_id ? v : 0;
                all += v;
                own = r == p.rank_id ? v : own;
                ps += __ldg(p.all_psum + (size_t)r * E + x);  // rank order: fixed rounding
            }
        }
        const bool bad_e = x < E && (own != s_n[x] || before < 0 || all > INT_MAX);
        const long long tot = block_sum_ll(all);
        if (__syncthreads_or(bad_e) || tot != p.TK_global) {
            if (b == 0 && threadIdx.x == 0)
                set_status(p.status, MOE_DEVICE_SHARD_MISMATCH);
            return;
        }
        if (x < E) {
            s_rb[x] = (int32_t)min(before, (long long)INT_MAX);
            if (b == 0) {
                p.gcount[x] = (int32_t)all;
                p.psum[x] = ps;
            }
        }
    } else {
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            s_rb[e] = 0;
    }
    __syncthreads();
    // ---- phase 2b: kept counts, segment offsets, 128-row tile prefix (the
    // same in every block; block 0 publishes them).  An expert keeps the
    // assignments whose global position (earlier ranks' count + position
    // here) is below C.
    {
        const int x = threadIdx.x;
        const int n = x < E ? s_n[x] : 0;
        const long long room = x < E ? p.C - (long long)s_rb[x] : 0;
        const int kept = (p.C < 0) ? n : (int)max(0ll, min((long long)n, room));
        int tot;
        const int off = block_excl_scan(kept, sh_int, &tot);
        if (x < E)
            s_seg[x] = off;
        if (x == 0)
            s_seg[E] = tot;
        const int mt = (kept + kTileM - 1) / kTileM;
        int mt_total;
        const int moff = block_excl_scan(mt, sh_int, &mt_total);
        if (b == 0) {
            if (x < E) {
                if (p.expert_counts)
                    p.expert_counts[x] = n;
                p.kept_counts[x] = kept;
                p.seg_off[x] = off;
                p.mtile[x] = moff;
            }
            if (x == 0) {
                p.seg_off[E] = tot;
                p.mtile[E] = mt_total;
            }
        }
    }
    __syncthreads();
    dispatch_stamp(6);

    // ---- phase 2c/2d: the last warp computes this block's probability sums;
    // the other warps place the block's assignments and copy x into x_perm
    if (warp == 31) {
        if constexpr (SPLIT == 0)
            prob_sums(p, b, G);
        return;
    }
    constexpr int kCopyWarps = 31;
    const int nparts = ntok >= kCopyWarps ? 1 : ntok >= 16 ? 2 : ntok >= 8 ? 4 : ntok >= 4 ? 8 : 31;
    for (int task = warp; task < ntok * nparts; task += kCopyWarps) {
        const int t = t_beg + task / nparts, part = task - (task / nparts) * nparts;
        long long row = -1;
        if (lane < k) {
            const size_t tk = (size_t)t * k + lane;
            // a one-chunk block still holds its assignments in shared memory
            const int u = (t - t_beg) * k + lane;
            const int e = held ? ibuf[u] : __ldcg(p.topk_idx + tk);
            // the finish launch of a split batch reads topk_idx as the caller
            // hands it back: an expert index outside [0, E), or a kept row
            // outside its expert's segment, is refused rather than followed
            // (every index is checked in a MOE_DEBUG_BOUNDS build)
            constexpr bool kCheck = SPLIT == 2 || kDebugBounds;
            bool idx_ok = !kCheck || (unsigned)e < (unsigned)E;
            const int es = idx_ok ? e : 0;
            const long long pos = (long long)s_base[es] + (held ? rbuf[u] : __ldcg(p.rank + tk));
            bool kept = idx_ok && ((p.C < 0) || (pos + s_rb[es] < p.C));
            row = kept ? (long long)s_seg[es] + pos : -1;
            if (kCheck && kept && (pos < 0 || row >= s_seg[es + 1] || row >= p.R_max)) {
                idx_ok = kept = false;
                row = -1;
            }
            if (kCheck && !idx_ok)
                set_status(p.status, MOE_DEVICE_INDEX_OUT_OF_RANGE);
            if (part == 0) {
                p.dropped[tk] = kept ? 0 : 1;
                p.row_of[tk] = (int32_t)row;
                if (p.row_tok && row >= 0) {
                    p.row_tok[row] = t;
                    p.row_w[row] = held ? wbuf[u] : __ldcg(p.topk_w + tk);
                }
                if (p.gscale_perm && row >= 0)
                    p.gscale_perm[row] = __ldg(p.gscale + t);
            }
        }
        long long rows[kMaxTopK];
        bool any = false;
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j) {
            rows[j] = __shfl_sync(0xffffffffu, row, j);
            any |= (j < k && rows[j] >= 0);
        }
        const uint8_t *src = p.gx ? p.gx + (size_t)t * p.g_row_bytes
                             : p.x_staged && gate
                                 ? xs + (size_t)(t - t_beg) * xstride
                                 : static_cast<const uint8_t *>(p.x) + (size_t)t * p.row_bytes;
        copy_row(p, src, p.gx ? p.g_row_bytes : p.row_bytes, rows, part, nparts);
        if (p.y_zero && !any) {
            uint4 *dst = reinterpret_cast<uint4 *>(p.y_zero + (size_t)t * p.row_bytes);
            for (size_t v = (size_t)part * 32 + lane; v < p.row_bytes / 16; v += (size_t)nparts * 32)
                dst[v] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if constexpr (kTimeline) {
        if (lane == 0 && b < kDispatchTimelineBlocks)
            atomicMax(g_dispatch_timeline + b * 8 + 7, (unsigned long long)global_timer_ns());
    }
}

// A rank without tokens in a split batch: the demand counts and probability
// sums over all ranks (rank order), then the balance loss.  One warp.
__global__ void shard_stats_kernel(const int32_t *all_counts, const double *all_psum,
                                   int n_ranks, int rank, long long TK_global, int32_t *gcount,
                                   double *gpsum, AuxArgs aux, int32_t *status)
{
    const int lane = threadIdx.x & 31, E = aux.E;
    long long tot = 0;
    bool bad = false;
    for (int e = lane; e < E; e += 32) {
        long long all = 0;
        double ps = 0.0;
        for (int r = 0; r < n_ranks; ++r) {
            const long long v = all_counts[(size_t)r * E + e];
            bad |= (r == rank && v != 0) || v < 0;
            all += v;
            ps += all_psum[(size_t)r * E + e];
        }
        gcount[e] = (int32_t)min(all, (long long)INT_MAX);
        gpsum[e] = ps;
        tot += all;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (__any_sync(0xffffffffu, bad) || tot != TK_global) {
        if (lane == 0)
            set_status(status, MOE_DEVICE_SHARD_MISMATCH);
        return;
    }
    __threadfence();
    __syncwarp();
    balance_loss_warp(aux);
}

cudaError_t launch_shard_stats(const int32_t *all_counts, const double *all_psum, int n_ranks,
                               int rank, long long TK_global, int32_t *gcount, double *gpsum,
                               const AuxArgs &aux, int32_t *status, cudaStream_t stream)
{
    shard_stats_kernel<<<1, 32, 0, stream>>>(all_counts, all_psum, n_ranks, rank, TK_global,
                                             gcount, gpsum, aux, status);
    return cudaGetLastError();
}

bool router_fused(const moe_config &c)
{
    const size_t esz = c.dtype == MOE_DTYPE_BF16 ? 2 : 4;
    return c.n_experts <= kFusedMaxE && c.d_model % 8 == 0 &&
           (size_t)c.n_experts * c.d_model * esz <= (size_t)kFusedMaxWrBytes;
}

bool direct_y(const moe_config &c) { return c.top_k == 1 && c.d_shared == 0; }

// Dynamic shared memory of the dispatch kernel: staged W_r rows (fused
// router; wr_bytes = E * (row bytes + 16)), staged x rows (xs_bytes =
// chunk * (row bytes + 16)), pbuf [32][E] floats, ibuf [32][k], then mask,
// run, base, n [E], the segment offsets [E+1], the earlier ranks' counts
// [E], the router's partial sums [8][32][16], and the chunk's ranks and gate
// weights [32][8].
static size_t dispatch_smem(size_t wr_bytes, size_t xs_bytes, int E, int k)
{
    return wr_bytes + xs_bytes + (size_t)kChunk * (E + k) * 4 + (size_t)4 * E * 4 +
           (size_t)(E + 1) * 4 + (size_t)E * 4 +
           (size_t)kRouterMmaWarps * kChunk * kFusedMaxE * 4 +
           (size_t)2 * kChunk * kMaxTopK * 4;
}

template <int EPL, int RT, int EM, int SPLIT>
static cudaError_t launch_dispatch_t(DispatchParams &p, size_t wr_bytes, cudaStream_t stream)
{
    auto kern = dispatch_kernel<EPL, RT, EM, SPLIT>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    // One block per SM (a 1024-thread block whose largest layout takes most
    // of an SM's shared memory), so the launch geometry depends only on T and
    // the SM count: the two launches of a split batch see the same chunks.
    static DeviceOnce configured;
    if (configured.pending(dev)) {
        const size_t smem_max = dispatch_smem(kFusedMaxWrBytes + kFusedMaxE * 16,
                                              kStageMaxBytes + kChunk * 16, kMaxExperts, kMaxTopK);
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem_max);
        if (err == cudaSuccess)
            err = prefer_max_shared_carveout(kern);
        if (err != cudaSuccess)
            return err;
        int per_sm = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDispatchThreads,
                                                            smem_max);
        if (err != cudaSuccess)
            return err;
        if (per_sm < 1)
            return cudaErrorInvalidConfiguration;
        configured.done(dev);
    }
    const int maxb = std::max(1, std::min(kMaxDispatchBlocks, sm_count()));
    // The smallest chunk (1, 2, ..., 32 tokens) whose chunk count fits one
    // chunk per co-resident block; else 32-token chunks, several per block.
    int cs = kChunk;
    for (int c = 1; c < kChunk; c *= 2)
        if ((p.T + c - 1) / c <= maxb) {
            cs = c;
            break;
        }
    p.cs = cs;
    p.nchunk = (p.T + cs - 1) / cs;
    p.cpb = (p.nchunk + maxb - 1) / maxb;
    const int grid = std::max(1, (p.nchunk + p.cpb - 1) / p.cpb);
    p.x_staged = ((p.phases & 1) && p.cpb == 1 && p.row_bytes % 16 == 0 &&
                  (size_t)cs * p.row_bytes <= kStageMaxBytes) ? 1 : 0;
    const size_t smem = dispatch_smem(wr_bytes, p.x_staged ? (size_t)cs * (p.row_bytes + 16) : 0,
                                      p.E, p.k);
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

// The instantiation for the router type and expert count.
template <int SPLIT>
static cudaError_t launch_dispatch_s(const moe_config &c, DispatchParams &p, bool fused,
                                     size_t wr_bytes, cudaStream_t stream)
{
    const int E = c.n_experts;
    if constexpr (SPLIT != 2) {
        if (fused) {
            if (c.dtype == MOE_DTYPE_BF16)
                return E <= 4   ? launch_dispatch_t<1, ROUTER_BF16, 4, SPLIT>(p, wr_bytes, stream)
                       : E <= 8 ? launch_dispatch_t<1, ROUTER_BF16, 8, SPLIT>(p, wr_bytes, stream)
                                : launch_dispatch_t<1, ROUTER_BF16, 16, SPLIT>(p, wr_bytes, stream);
            return E <= 4   ? launch_dispatch_t<1, ROUTER_F32, 4, SPLIT>(p, wr_bytes, stream)
                   : E <= 8 ? launch_dispatch_t<1, ROUTER_F32, 8, SPLIT>(p, wr_bytes, stream)
                            : launch_dispatch_t<1, ROUTER_F32, 16, SPLIT>(p, wr_bytes, stream);
        }
    }
    const int epl = (E + 31) / 32;
    if (epl <= 1)
        return launch_dispatch_t<1, ROUTER_NONE, 1, SPLIT>(p, wr_bytes, stream);
    if (epl <= 2)
        return launch_dispatch_t<2, ROUTER_NONE, 1, SPLIT>(p, wr_bytes, stream);
    if (epl <= 4)
        return launch_dispatch_t<4, ROUTER_NONE, 1, SPLIT>(p, wr_bytes, stream);
    return launch_dispatch_t<8, ROUTER_NONE, 1, SPLIT>(p, wr_bytes, stream);
}

// The test hook's settings (moe_debug_barrier_fault): extra arrivals the
// grid barrier waits for, and its wait limit (0 = the default).
static std::atomic<unsigned> g_barrier_extra{0};
static std::atomic<unsigned long long> g_barrier_limit_ns{0};

cudaError_t launch_dispatch(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                            const void *x, const void *W_r, bool fused, float *logits,
                            const float *lpart, int lsplit, const float *bias,
                            int32_t *topk_idx, float *topk_w, uint8_t *dropped_mask,
                            int32_t *expert_counts, int32_t *kept_counts, void *y,
                            cudaStream_t stream, const ShardArgs *shard, const GatherArgs *gather)
{
    DispatchParams p{};
    p.phases = shard ? shard->phases : 3;
    p.all_counts = shard ? shard->all_counts : nullptr;
    p.all_psum = shard ? shard->all_psum : nullptr;
    p.n_ranks = shard ? shard->n_ranks : 1;
    p.rank_id = shard ? shard->rank : 0;
    p.TK_global = (shard ? shard->T_global : (long long)c.T) * c.top_k;
    p.gcount = shard ? reinterpret_cast<int32_t *>(ws + L.gcount) : nullptr;
    const size_t esz = c.dtype == MOE_DTYPE_BF16 ? 2 : 4;
    p.logits = logits;
    p.lpart = lpart;
    p.lsplit = lsplit;
    p.bias = bias;
    p.bias_sel_only = c.bias_selection_only;
    p.x = x;
    p.W_r = W_r;
    p.T = c.T;
    p.E = c.n_experts;
    p.k = c.top_k;
    p.mode = c.gating_mode;
    p.D = c.d_model;
    p.C = L.C;
    p.alpha = c.aux_alpha;
    p.row_bytes = (size_t)c.d_model * esz;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.dropped = dropped_mask;
    p.expert_counts = expert_counts;
    p.kept_counts = kept_counts;
    p.bcount = reinterpret_cast<int32_t *>(ws + L.bcount);
    p.ppart = reinterpret_cast<float *>(ws + L.ppart);
    p.rank = reinterpret_cast<int32_t *>(ws + L.rank);
    p.psum = shard && shard->psum_out ? shard->psum_out : reinterpret_cast<double *>(ws + L.psum);
    p.seg_off = reinterpret_cast<int32_t *>(ws + L.seg_off);
    p.mtile = reinterpret_cast<int32_t *>(ws + L.mtile);
    p.row_of = reinterpret_cast<int32_t *>(ws + L.row_of);
    p.x_perm = gather ? gather->dst : ws + L.x_perm;
    p.R_max = L.R_max;
    if (gather) {
        p.gx = gather->src;
        p.g_row_bytes = gather->row_bytes;
        p.gscale = gather->scale;
        p.gscale_perm = gather->scale_dst;
    }
    const bool dy = direct_y(c) && c.dtype == MOE_DTYPE_BF16;
    p.row_tok = dy ? reinterpret_cast<int32_t *>(ws + L.row_tok) : nullptr;
    p.row_w = dy ? reinterpret_cast<float *>(ws + L.row_w) : nullptr;
    p.y_zero = dy ? static_cast<uint8_t *>(y) : nullptr;
    p.status = reinterpret_cast<int32_t *>(ws + L.status);
    p.barrier_extra = g_barrier_extra.load(std::memory_order_relaxed);
    const unsigned long long lim = g_barrier_limit_ns.load(std::memory_order_relaxed);
    p.barrier_limit_ns = lim ? lim : kBarrierLimitNs;
    const size_t wr_bytes = fused ? (size_t)c.n_experts * (c.d_model * esz + 16) : 0;
    const int split = !shard ? 0 : shard->phases == 1 ? 1 : 2;
    if (split == 2)  // placement only: no router, no gating
        return launch_dispatch_s<2>(c, p, false, wr_bytes, stream);
    return split == 1 ? launch_dispatch_s<1>(c, p, fused, wr_bytes, stream)
                      : launch_dispatch_s<0>(c, p, fused, wr_bytes, stream);
}

cudaError_t dispatch_timeline_copy(uint64_t *host, size_t words)
{
    return cudaMemcpyFromSymbol(host, g_dispatch_timeline,
                                std::min(words, sizeof(g_dispatch_timeline) / 8) * 8);
}

cudaError_t dispatch_timeline_clear()
{
    static const unsigned long long zero[sizeof(g_dispatch_timeline) / 8] = {};
    return cudaMemcpyToSymbol(g_dispatch_timeline, zero, sizeof(zero));
}

}  // namespace moe

extern "C" moe_status moe_debug_barrier_fault(int32_t extra_arrivals, uint64_t limit_ns)
{
    if (extra_arrivals < 0 || extra_arrivals > 1 || limit_ns > moe::kBarrierLimitNs ||
        (limit_ns != 0 && limit_ns < 1000))
        return MOE_ERR_INVALID_ARG;
    moe::g_barrier_extra.store((unsigned)extra_arrivals, std::memory_order_relaxed);
    moe::g_barrier_limit_ns.store(limit_ns, std::memory_order_relaxed);
    return MOE_OK;
}
