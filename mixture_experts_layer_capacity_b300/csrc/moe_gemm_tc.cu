// moe_gemm_tc.cu -- tensor-core GEMMs of the MoE layer for bf16 (sm_103a):
//   router:  logits[T,E]  = x[T,D] . W_r[E,D]^T                  (fp32 out)
//   GEMM1:   h[r,F]       = silu(x_perm[r,:] . W_gate[e]^T) * (x_perm[r,:] . W_up[e]^T)
//   GEMM2:   z[r,D]       = h[r,:] . W_down[e]^T
// for every row r of expert e's segment, plus the same two GEMMs over all T
// rows for the shared expert ("Mixture of Experts: More Parameters, Same
// FLOPs", 'An MoE tiny GPT': the SwiGLU expert; "Mixture of Experts"
// (module 17), 17.2 equation: the shared expert on every token).
//
// Design (one CTA per SM, persistent over a tile list built on the device):
//   - tile = 128 rows of one segment x BN output columns; tiles are ordered
//     segment-major, then column tile, then row tile, so the CTAs running at
//     the same time share weight tiles through L2;
//   - warp 0: TMA producer (128-byte-swizzled K-major boxes of 64 elements)
//     into a STAGES-deep shared-memory ring guarded by mbarriers;
//   - warp 1: allocates TMEM and issues tcgen05.mma (M=128, N=BN*NB, K=16)
//     into one of two TMEM accumulators, committing to the ring's "empty"
//     barriers and to the accumulator's "full" barrier;
//   - warps 2-5: epilogue; each thread owns one accumulator row (TMEM lane),
//     loads it with tcgen05.ld, applies SiLU*up (GEMM1) or converts, and
//     stores straight to global memory, then frees the accumulator so the
//     next tile's MMAs overlap this epilogue.
// For GEMM1 the gate and up tiles of the same columns are stacked in one
// 256-row B operand, so one N=256 MMA produces both accumulators.
// Every mbarrier wait is bounded; on timeout the CTA records
// MOE_DEVICE_PIPELINE_TIMEOUT, drains its own copies and MMAs, frees TMEM and
// returns.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "tc_ptx.cuh"

namespace moe {

// Epilogues: fp32 store (router scores), bf16 store (z), SiLU(gate) * up in
// bf16 (h), and bf16 store of w_row * acc straight into the row's token of y
// (down projection when every token has one expert and no shared expert).
enum { EPI_F32 = 0, EPI_BF16 = 1, EPI_SWIGLU = 2, EPI_BF16_Y = 3 };

struct TcParams {
    const int32_t *seg_off;  // grouped: [nseg+1] first A row of each segment; null = dense
    const int32_t *mtile;    // grouped: [nseg+1] prefix sum of 128-row tiles per segment
    int nseg;
    int dense_rows;          // rows of A when dense
    int K;                   // reduction length (multiple of 64)
    int n_tiles;             // output column tiles per segment
    int N_valid;             // output columns that exist
    int b_seg_rows;          // B rows per segment (F or D), 0 when dense
    void *out;
    long long ld_out;        // output row stride, elements
    const int32_t *row_tok;  // EPI_BF16_Y: token of each A row
    const float *row_w;      // EPI_BF16_Y: gate weight of each A row
    int32_t *status;
    AuxArgs aux;             // balance loss to evaluate (aux.out null: none)
    int ksplit;              // splits of the reduction (single-CTA kernel, EPI_F32); 0 or 1 = none
    long long part_stride;   // elements between the splits' fp32 outputs
    // single-CTA kernel: a second, dense problem (the shared expert next to
    // the routed ones) whose tiles come first in the tile list; its operands
    // are the kernel's second set of tensor maps.  sh_tiles = 0: none.
    int sh_tiles;            // dense tiles of the second problem (row tiles x column tiles)
    int sh_rows, sh_K, sh_n_tiles, sh_N_valid;
    // grouped problems split between the CTA-pair kernel (full 256-row tiles)
    // and the single-CTA kernel (each segment's remaining rows, 128-row tiles):
    int pair_full_only;      // pair kernel: only the floor(n / 256) full tiles of a segment
    int tail_after;          // single-CTA kernel: > 0: only the rows after the first
                             // floor(n / tail_after) * tail_after rows of each segment
    int sh_ksplit;           // splits of the second problem's reduction (fp32 partial
                             // outputs part_stride apart, EPI_BF16 kernels only); 0/1 = none
    void *sh_out;
    long long sh_ld_out;
};

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far beyond any tile
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s
constexpr int kThreads = 192;

template <int BN, int NB, int STAGES>
struct TcShape {
    static constexpr int UMMA_N = BN * NB;
    static constexpr int A_BYTES = kTileM * 64 * 2;
    static constexpr int B_BYTES = BN * 64 * 2;
    static constexpr int STAGE_BYTES = A_BYTES + NB * B_BYTES;
    static constexpr int TMEM_COLS = 2 * UMMA_N <= 32    ? 32
                                     : 2 * UMMA_N <= 64  ? 64
                                     : 2 * UMMA_N <= 128 ? 128
                                     : 2 * UMMA_N <= 256 ? 256
                                                         : 512;
    static constexpr int TABLE_BYTES = 2 * (kMaxExperts + 1) * 4 + 8;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 256 + TABLE_BYTES + 1024;
    static_assert(UMMA_N % 16 == 0 && UMMA_N >= 16 && UMMA_N <= 256, "UMMA N");
    static_assert(B_BYTES % 1024 == 0, "B tile must keep 1024-byte alignment");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct TileInfo {
    int a_row0, rows, seg, n_idx;
};

// The fewest workers (CTAs or CTA pairs) that finish n equal units in as
// many rounds as w workers would.  With w workers some would take one unit
// more than the rest, and the final round would run on those few alone; an
// HBM-bound GEMM then streams its last tiles at a few SMs' bandwidth.  With
// every worker taking the same number of units (give or take one in the
// first round), the bandwidth stays shared by all of them to the end.
__device__ __forceinline__ int balanced_workers(int n, int w)
{
    if (n <= 0)
        return w;
    const int rounds = (n + w - 1) / w;
    return (n + rounds - 1) / rounds;
}

// The segment tables (seg_off, mtile) are copied into shared memory at
// kernel start; s_seg/s_mt point there (null when dense).
__device__ __forceinline__ int tile_count(const TcParams &p, const int *s_mt)
{
    if (!s_mt)
        return ((p.dense_rows + kTileM - 1) / kTileM) * p.n_tiles;
    return s_mt[p.nseg] * p.n_tiles;
}

__device__ __forceinline__ TileInfo tile_info(const TcParams &p, const int *s_seg,
                                              const int *s_mt, int g)
{
    TileInfo ti;
    if (!s_mt) {
        const int mt = (p.dense_rows + kTileM - 1) / kTileM;
        ti.n_idx = g / mt;
        const int m = g - ti.n_idx * mt;
        ti.seg = 0;
        ti.a_row0 = m * kTileM;
        ti.rows = min(kTileM, p.dense_rows - ti.a_row0);
        return ti;
    }
    int lo = 0, hi = p.nseg;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_mt[mid] * p.n_tiles <= g)
            lo = mid;
        else
            hi = mid;
    }
    const int mt0 = s_mt[lo], mt_e = s_mt[lo + 1] - mt0;
    const int local = g - mt0 * p.n_tiles;
    ti.n_idx = local / mt_e;
    const int m = local - ti.n_idx * mt_e;
    ti.seg = lo;
    int s0 = s_seg[lo];
    if (p.tail_after > 0)
        s0 += (s_seg[lo + 1] - s_seg[lo]) / p.tail_after * p.tail_after;
    ti.a_row0 = s0 + m * kTileM;
    ti.rows = min(kTileM, s_seg[lo + 1] - ti.a_row0);
    return ti;
}

// Work unit u of the combined list: the second problem's units first
// (tile u / sh_ksplit, split u % sh_ksplit; ti.seg = -1), then the first
// problem's (tile v / ks_n, split v % ks_n).  [kb0, kb1): the unit's 64-wide
// reduction steps.
struct UnitInfo {
    TileInfo ti;
    int ks, kb0, kb1;
    bool second;
};

__device__ __forceinline__ UnitInfo unit_info(const TcParams &p, const int *s_seg,
                                              const int *s_mt, int u, int ks_n)
{
    UnitInfo w;
    const int sh_ks = p.sh_ksplit > 1 ? p.sh_ksplit : 1;
    const int sh_units = p.sh_tiles * sh_ks;
    int n_split, nk;
    if (u < sh_units) {
        const int g = u / sh_ks;
        w.ks = u - g * sh_ks;
        const int mt = (p.sh_rows + kTileM - 1) / kTileM;
        w.ti.n_idx = g / mt;
        const int m = g - w.ti.n_idx * mt;
        w.ti.seg = -1;
        w.ti.a_row0 = m * kTileM;
        w.ti.rows = min(kTileM, p.sh_rows - w.ti.a_row0);
        w.second = true;
        n_split = sh_ks;
        nk = (p.sh_K + 63) / 64;
    } else {
        const int v = u - sh_units;
        const int g = v / ks_n;
        w.ks = v - g * ks_n;
        w.ti = tile_info(p, s_seg, s_mt, g);
        w.second = false;
        n_split = ks_n;
        nk = (p.K + 63) / 64;
    }
    w.kb0 = w.ks * nk / n_split;
    w.kb1 = (w.ks + 1) * nk / n_split;
    return w;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Stores 32 bf16 values (as 16 packed words) of one output row.
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16 *dst, const uint32_t (&pk)[16],
                                               int col, int n_valid)
{
    if (col + 32 <= n_valid) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(&pk[i]);
            if (col + 2 * i < n_valid)
                dst[2 * i] = v.x;
            if (col + 2 * i + 1 < n_valid)
                dst[2 * i + 1] = v.y;
        }
    }
}

// Epilogue of one accumulator row (TMEM lane) of a tile: this thread owns
// output row `orow` (stored only when row_ok), columns n_idx*BN ... of the
// tile.  taddr: TMEM address of the row's first accumulator column.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_row(const TcParams &p, void *out, long long ld_out,
                                             int n_valid, uint32_t taddr, bool row_ok,
                                             long long orow, int n_idx, int ks = 0)
{
    if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t gv[32], uv[32];
            tmem_ld32(taddr + c0, gv);
            tmem_ld32(taddr + BN + c0, uv);
            tmem_wait_ld();
            if (row_ok) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float g0 = __uint_as_float(gv[2 * i]);
                    const float g1 = __uint_as_float(gv[2 * i + 1]);
                    const float u0 = __uint_as_float(uv[2 * i]);
                    const float u1 = __uint_as_float(uv[2 * i + 1]);
                    pk[i] = pack_bf16x2(silu_f32(g0) * u0, silu_f32(g1) * u1);
                }
                const int col = n_idx * BN + c0;
                __nv_bfloat16 *dst =
                    reinterpret_cast<__nv_bfloat16 *>(out) + orow * ld_out + col;
                store_row_bf16(dst, pk, col, n_valid);
            }
        }
    } else if constexpr (EPI == EPI_BF16_Y) {
        int tok = 0;
        float wr = 0.f;
        if (row_ok) {
            tok = p.row_tok[orow];
            wr = p.row_w[orow];
        }
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(taddr + c0, v);
            tmem_wait_ld();
            if (row_ok) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(wr * __uint_as_float(v[2 * i]),
                                        wr * __uint_as_float(v[2 * i + 1]));
                const int col = n_idx * BN + c0;
                __nv_bfloat16 *dst =
                    reinterpret_cast<__nv_bfloat16 *>(out) + (long long)tok * ld_out + col;
                store_row_bf16(dst, pk, col, n_valid);
            }
        }
    } else if constexpr (EPI == EPI_BF16) {
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(taddr + c0, v);
            tmem_wait_ld();
            if (row_ok) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]),
                                        __uint_as_float(v[2 * i + 1]));
                const int col = n_idx * BN + c0;
                __nv_bfloat16 *dst =
                    reinterpret_cast<__nv_bfloat16 *>(out) + orow * ld_out + col;
                store_row_bf16(dst, pk, col, n_valid);
            }
        }
    } else {
        constexpr int CH = BN < 32 ? 16 : 32;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += CH) {
            uint32_t v[32];
            if constexpr (CH == 16) {
                uint32_t v16[16];
                tmem_ld16(taddr + c0, v16);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = v16[i];
            } else {
                tmem_ld32(taddr + c0, v);
                tmem_wait_ld();
            }
            if (row_ok) {
                const int col = n_idx * BN + c0;
                float *dst = reinterpret_cast<float *>(out) + ks * p.part_stride + orow * ld_out + col;
                // 16-byte stores when the whole chunk is in range and aligned
                const bool vec = col + CH <= n_valid && ((ld_out | p.part_stride) & 3) == 0 &&
                                 (reinterpret_cast<uintptr_t>(out) & 15) == 0;
                if (vec) {
#pragma unroll
                    for (int i = 0; i < CH; i += 4)
                        *reinterpret_cast<float4 *>(dst + i) =
                            make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                                        __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                } else {
#pragma unroll
                    for (int i = 0; i < CH; ++i)
                        if (col + i < n_valid)
                            dst[i] = __uint_as_float(v[i]);
                }
            }
        }
    }
}

template <int BN, int NB, int EPI, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB0,
                   const __grid_constant__ CUtensorMap mB1, const __grid_constant__ CUtensorMap sA,
                   const __grid_constant__ CUtensorMap sB0, const __grid_constant__ CUtensorMap sB1,
                   const TcParams p)
{
    using S = TcShape<BN, NB, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * S::STAGE_BYTES);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = bars + 2 * STAGES + 2;
    uint64_t *mma_done = bars + 2 * STAGES + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *tables = reinterpret_cast<int *>(smem + STAGES * S::STAGE_BYTES + 256);
    const int *s_seg = p.mtile ? tables : nullptr;
    const int *s_mt = p.mtile ? tables + (kMaxExperts + 1) : nullptr;

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4 * 32);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&mA);
        tma_prefetch_desc(&mB0);
        if (NB == 2)
            tma_prefetch_desc(&mB1);
        if (p.sh_tiles > 0) {
            tma_prefetch_desc(&sA);
            tma_prefetch_desc(&sB0);
            if (NB == 2)
                tma_prefetch_desc(&sB1);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, S::TMEM_COLS);
        tmem_relinquish();
    }
    // everything above touched only this CTA's shared memory and TMEM; from
    // here on global memory written by the previous kernel is read
    griddep_wait();
    griddep_launch_dependents();
    // an earlier kernel of this forward pass failed: do no work
    const bool failed = *(volatile const int32_t *)p.status != 0;
    if (p.mtile && !failed) {
        for (int i = threadIdx.x; i <= p.nseg; i += blockDim.x) {
            tables[i] = p.seg_off[i];
            if (p.tail_after <= 0)
                tables[kMaxExperts + 1 + i] = p.mtile[i];
        }
    }
    __syncthreads();
    if (p.tail_after > 0 && p.mtile && !failed && warp == 0) {
        // 128-row tiles of each segment's rows past its last full
        // tail_after-row block, prefix-summed
        int carry = 0;
        for (int e0 = 0; e0 < p.nseg; e0 += 32) {
            const int e = e0 + lane;
            const int n = e < p.nseg ? tables[e + 1] - tables[e] : 0;
            const int v = (n - n / p.tail_after * p.tail_after + kTileM - 1) / kTileM;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += t;
            }
            if (e < p.nseg)
                tables[kMaxExperts + 1 + e + 1] = carry + incl;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0)
            tables[kMaxExperts + 1] = 0;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    // work units: tiles x reduction splits (unit u: tile u / ks_n, split u % ks_n)
    const int ks_n = p.ksplit > 1 ? p.ksplit : 1;
    const int tiles_all =
        failed ? 0 : p.sh_tiles * (p.sh_ksplit > 1 ? p.sh_ksplit : 1) + tile_count(p, s_mt) * ks_n;
    const int G = balanced_workers(tiles_all, (int)gridDim.x);
    const int ntiles = (int)blockIdx.x < G ? tiles_all : 0;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int s = 0;
            uint32_t ph = 0;
            long long fills = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < ntiles && ok; u += G) {
                const UnitInfo w = unit_info(p, s_seg, s_mt, u, ks_n);
                const TileInfo &ti = w.ti;
                const bool second = w.second;
                const int kb0 = w.kb0, kb1 = w.kb1;
                const int b_row = second ? ti.n_idx * BN : ti.seg * p.b_seg_rows + ti.n_idx * BN;
                const CUtensorMap *ma = second ? &sA : &mA;
                const CUtensorMap *mb0 = second ? &sB0 : &mB0;
                const CUtensorMap *mb1 = second ? &sB1 : &mB1;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + s * S::STAGE_BYTES;
                    uint8_t *sb = sa + S::A_BYTES;
                    mbar_arrive_expect_tx(&full[s], S::STAGE_BYTES);
                    tma_load_2d(sa, ma, &full[s], kb * 64, ti.a_row0);
                    tma_load_2d(sb, mb0, &full[s], kb * 64, b_row);
                    if (NB == 2)
                        tma_load_2d(sb + S::B_BYTES, mb1, &full[s], kb * 64, b_row);
                    ++fills;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
                // wait (bounded) for this CTA's copies still in flight
                const long long first = fills > STAGES ? fills - STAGES : 0;
                for (long long f = first; f < fills; ++f)
                    mbar_wait(&full[f % STAGES], (uint32_t)((f / STAGES) & 1), nullptr,
                              kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(kTileM, S::UMMA_N);
            int s = 0;
            uint32_t ph = 0, b = 0, tph = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < ntiles && ok; u += G) {
                const UnitInfo w = unit_info(p, s_seg, s_mt, u, ks_n);
                const int kb0 = w.kb0, kb1 = w.kb1;
                if (!mbar_wait(&tempty[b], tph ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * S::UMMA_N;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = smem_u32(smem + s * S::STAGE_BYTES);
                    const uint64_t adesc = sdesc_kmajor_sw128(sa);
                    const uint64_t bdesc = sdesc_kmajor_sw128(sa + S::A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                                  (kb > kb0 || kk > 0) ? 1u : 0u);
                    umma_commit(&empty[s]);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit(&tfull[b]);
                b ^= 1u;
                if (b == 0)
                    tph ^= 1u;
            }
            if (!ok) {
                *abort_flag = 1;
                set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
            }
            // all MMAs of this CTA complete before TMEM is released
            umma_commit(mma_done);
            mbar_wait(mma_done, 0, nullptr, kDrainLimitNs);
        }
    } else {
        // ---------------------------------------------------- epilogue
        // (the first epilogue warp of CTA 0 first evaluates the balance loss,
        // while the first tile's operands are still in flight)
        if (p.aux.out && !failed && blockIdx.x == 0 && warp == 2)
            balance_loss_warp(p.aux);
        const int q = warp & 3;             // TMEM lane quarter this warp may access
        const int r = q * 32 + lane;        // accumulator row of this thread
        uint32_t b = 0, tph = 0;
        for (int u = blockIdx.x; u < ntiles; u += G) {
            const UnitInfo w = unit_info(p, s_seg, s_mt, u, ks_n);
            const TileInfo &ti = w.ti;
            const int ks = w.ks;
            if (!mbar_wait(&tfull[b], tph, abort_flag, kWaitLimitNs)) {
                *abort_flag = 1;
                set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + b * S::UMMA_N + ((uint32_t)(q * 32) << 16);
            const bool row_ok = r < ti.rows;
            const long long orow = (long long)ti.a_row0 + r;
            if (w.second) {
                if constexpr (EPI == EPI_BF16) {
                    if (p.sh_ksplit > 1)  // fp32 partial sums of a piece of the reduction
                        epilogue_row<BN, EPI_F32>(p, p.sh_out, p.sh_ld_out, p.sh_N_valid, taddr,
                                                  row_ok, orow, ti.n_idx, ks);
                    else
                        epilogue_row<BN, EPI>(p, p.sh_out, p.sh_ld_out, p.sh_N_valid, taddr,
                                              row_ok, orow, ti.n_idx, ks);
                } else {
                    epilogue_row<BN, EPI>(p, p.sh_out, p.sh_ld_out, p.sh_N_valid, taddr, row_ok,
                                          orow, ti.n_idx, ks);
                }
            } else
                epilogue_row<BN, EPI>(p, p.out, p.ld_out, p.N_valid, taddr, row_ok, orow,
                                      ti.n_idx, ks);
            tc_fence_before_sync();
            mbar_arrive(&tempty[b]);
            b ^= 1u;
            if (b == 0)
                tph ^= 1u;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, S::TMEM_COLS);
    }
}

// ------------------------------------------------------- CTA-pair GEMM
// The same GEMMs on pairs of CTAs (clusters of 2 on two SMs): a pair tile is
// 256 rows x UMMA_N columns, computed by tcgen05.mma.cta_group::2 (M = 256)
// issued by the even CTA.  Each CTA stages its own 128 rows of A and half of
// the B rows (for GEMM1 the leader holds the gate rows and the peer the up
// rows), so per SM a k-step moves A + B/2 instead of A + B: less L2 -> shared
// memory traffic per FLOP and room for deeper pipelines.  Each CTA's TMEM
// holds the accumulator rows of its own 128 A rows, all UMMA_N columns, so
// the epilogue is that of the single-CTA kernel.
//   - the producers of both CTAs signal the leader's "full" barriers
//     (transaction bytes of both halves; only the leader arrives);
//   - the leader's MMA commits arrive on the "empty" and "tfull" barriers of
//     both CTAs (multicast);
//   - both CTAs' epilogue warps arrive on the leader's "tempty" barriers.
// Pair tiles are 256 rows of one segment; their per-segment counts are
// derived here from the segment offsets.
template <int BN, int NB, int STAGES>
struct PairShape {
    static constexpr int UMMA_N = BN * NB;
    static constexpr int B_HALF_ROWS = UMMA_N / 2;   // B rows staged by each CTA
    static constexpr int A_BYTES = kTileM * 64 * 2;
    static constexpr int B_BYTES = B_HALF_ROWS * 64 * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * UMMA_N <= 256 ? 256 : 512;
    static constexpr int TABLE_BYTES = 2 * (kMaxExperts + 1) * 4 + 8;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 256 + TABLE_BYTES + 1024;
    static_assert(UMMA_N == 128 || UMMA_N == 256, "pair UMMA N");
    static_assert(NB == 1 || B_HALF_ROWS == BN, "gate/up halves");
    static_assert(B_BYTES % 1024 == 0, "B tile must keep 1024-byte alignment");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

constexpr int kPairRows = 2 * kTileM;

__device__ __forceinline__ int pair_tile_count(const TcParams &p, const int *s_mt)
{
    if (!s_mt)
        return ((p.dense_rows + kPairRows - 1) / kPairRows) * p.n_tiles;
    return s_mt[p.nseg] * p.n_tiles;
}

// a_row0 / rows: the pair tile's first A row and its valid rows (<= 256).
__device__ __forceinline__ TileInfo pair_tile_info(const TcParams &p, const int *s_seg,
                                                   const int *s_mt, int g)
{
    TileInfo ti;
    if (!s_mt) {
        const int mt = (p.dense_rows + kPairRows - 1) / kPairRows;
        ti.n_idx = g / mt;
        const int m = g - ti.n_idx * mt;
        ti.seg = 0;
        ti.a_row0 = m * kPairRows;
        ti.rows = min(kPairRows, p.dense_rows - ti.a_row0);
        return ti;
    }
    int lo = 0, hi = p.nseg;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_mt[mid] * p.n_tiles <= g)
            lo = mid;
        else
            hi = mid;
    }
    const int mt0 = s_mt[lo], mt_e = s_mt[lo + 1] - mt0;
    const int local = g - mt0 * p.n_tiles;
    ti.n_idx = local / mt_e;
    const int m = local - ti.n_idx * mt_e;
    ti.seg = lo;
    ti.a_row0 = s_seg[lo] + m * kPairRows;
    ti.rows = min(kPairRows, s_seg[lo + 1] - ti.a_row0);
    return ti;
}

template <int BN, int NB, int EPI, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap mA,
                        const __grid_constant__ CUtensorMap mB0,
                        const __grid_constant__ CUtensorMap mB1, const TcParams p)
{
    using S = PairShape<BN, NB, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * S::STAGE_BYTES);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *tfull = bars + 2 * STAGES;
    uint64_t *tempty = bars + 2 * STAGES + 2;
    uint64_t *mma_done = bars + 2 * STAGES + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *tables = reinterpret_cast<int *>(smem + STAGES * S::STAGE_BYTES + 256);
    int *s_seg = p.mtile ? tables : nullptr;
    int *s_mt = p.mtile ? tables + (kMaxExperts + 1) : nullptr;

    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster_id = (int)(blockIdx.x >> 1), nclusters = (int)(gridDim.x >> 1);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 2 * 4);  // one arrival per epilogue warp of each CTA
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&mA);
        tma_prefetch_desc(&mB0);
        if (NB == 2)
            tma_prefetch_desc(&mB1);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, S::TMEM_COLS);
        tmem_relinquish_pair();
    }
    griddep_wait();
    griddep_launch_dependents();
    const bool failed = *(volatile const int32_t *)p.status != 0;
    if (p.mtile && !failed)
        for (int i = threadIdx.x; i <= p.nseg; i += blockDim.x)
            s_seg[i] = p.seg_off[i];
    __syncthreads();
    // pair tiles per segment (256 rows each), prefix-summed by warp 0
    if (p.mtile && !failed && warp == 0) {
        int carry = 0;
        for (int e0 = 0; e0 < p.nseg; e0 += 32) {
            const int e = e0 + lane;
            const int n = e < p.nseg ? s_seg[e + 1] - s_seg[e] : 0;
            const int v = p.pair_full_only ? n / kPairRows : (n + kPairRows - 1) / kPairRows;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += n;
            }
            if (e < p.nseg)
                s_mt[e + 1] = carry + incl;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0)
            s_mt[0] = 0;
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    const int tiles_all = failed ? 0 : pair_tile_count(p, s_mt);
    const int NC = balanced_workers(tiles_all, nclusters);
    const int ntiles = cluster_id < NC ? tiles_all : 0;
    const int nk = (p.K + 63) / 64;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint32_t full_leader = mapa_shared(smem_u32(&full[0]), 0);
            int s = 0;
            uint32_t ph = 0;
            long long fills = 0;
            bool ok = true;
            for (int g = cluster_id; g < ntiles && ok; g += NC) {
                const TileInfo ti = pair_tile_info(p, s_seg, s_mt, g);
                const int a_row = ti.a_row0 + (int)rank * kTileM;
                const int b_row = ti.seg * p.b_seg_rows + ti.n_idx * BN +
                                  (NB == 1 ? (int)rank * S::B_HALF_ROWS : 0);
                const CUtensorMap *mb = (NB == 2 && !leader) ? &mB1 : &mB0;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + s * S::STAGE_BYTES;
                    uint8_t *sb = sa + S::A_BYTES;
                    const uint32_t fb = full_leader + (uint32_t)s * 8u;
                    if (leader)
                        mbar_arrive_expect_tx(&full[s], 2 * S::STAGE_BYTES);
                    tma_load_2d_pair(sa, &mA, fb, kb * 64, a_row);
                    tma_load_2d_pair(sb, mb, fb, kb * 64, b_row);
                    ++fills;
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
                if (leader) {
                    // wait (bounded) for the copies still in flight
                    const long long first = fills > STAGES ? fills - STAGES : 0;
                    for (long long f = first; f < fills; ++f)
                        mbar_wait(&full[f % STAGES], (uint32_t)((f / STAGES) & 1), nullptr,
                                  kDrainLimitNs);
                } else {
                    // this CTA's copies complete on the leader's barriers:
                    // give them time to land before the pair's final sync
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 1000000ull)
                        __nanosleep(1000);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (even CTA)
            constexpr uint32_t idesc = idesc_bf16_f32(kPairRows, S::UMMA_N);
            int s = 0;
            uint32_t ph = 0, b = 0, tph = 0;
            bool ok = true;
            for (int g = cluster_id; g < ntiles && ok; g += NC) {
                if (!mbar_wait(&tempty[b], tph ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * S::UMMA_N;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = smem_u32(smem + s * S::STAGE_BYTES);
                    const uint64_t adesc = sdesc_kmajor_sw128(sa);
                    const uint64_t bdesc = sdesc_kmajor_sw128(sa + S::A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16_pair(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                                       (kb > 0 || kk > 0) ? 1u : 0u);
                    umma_commit_pair(&empty[s], 0x3);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit_pair(&tfull[b], 0x3);
                b ^= 1u;
                if (b == 0)
                    tph ^= 1u;
            }
            if (!ok) {
                *abort_flag = 1;
                set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
            }
            // all MMAs of the pair complete before either CTA releases TMEM
            umma_commit_pair(mma_done, 0x1);
            mbar_wait(mma_done, 0, nullptr, kDrainLimitNs);
        }
    } else {
        // ---------------------------------------------------- epilogue (both CTAs)
        if (p.aux.out && !failed && blockIdx.x == 0 && warp == 2)
            balance_loss_warp(p.aux);
        const int q = warp & 3;             // TMEM lane quarter this warp may access
        const int r = q * 32 + lane;        // accumulator row of this thread
        const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[0]), 0);
        uint32_t b = 0, tph = 0;
        for (int g = cluster_id; g < ntiles; g += NC) {
            const TileInfo ti = pair_tile_info(p, s_seg, s_mt, g);
            if (!mbar_wait(&tfull[b], tph, abort_flag, kWaitLimitNs)) {
                *abort_flag = 1;
                set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + b * S::UMMA_N + ((uint32_t)(q * 32) << 16);
            const int my_rows = ti.rows - (int)rank * kTileM;
            const bool row_ok = r < my_rows;
            const long long orow = (long long)ti.a_row0 + (int)rank * kTileM + r;
            epilogue_row<BN, EPI>(p, p.out, p.ld_out, p.N_valid, taddr, row_ok, orow, ti.n_idx);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(&tempty[b]);
                else
                    mbar_arrive_cluster(tempty_leader + b * 8u);
            }
            b ^= 1u;
            if (b == 0)
                tph ^= 1u;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // neither CTA frees TMEM or exits while the pair may use it
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, S::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2-D bf16 tensor [rows, k] (k contiguous), boxes of 64 x box_rows, 128-byte
// swizzle; out-of-range elements read as zero.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t k, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn || rows == 0 || k == 0 || (reinterpret_cast<uintptr_t>(base) & 15u))
        return false;
    cuuint64_t dims[2] = {k, rows};
    cuuint64_t strides[1] = {k * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte tensor [rows, k] (e4m3 weights, k contiguous), boxes of 128 x
// box_rows with 128-byte swizzle; out-of-range bytes read as zero.
bool make_map_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t k, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn || rows == 0 || k == 0 || (reinterpret_cast<uintptr_t>(base) & 15u) || (k & 15u))
        return false;
    cuuint64_t dims[2] = {k, rows};
    cuuint64_t strides[1] = {k};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {


// The second problem's operands (TcParams::sh_tiles > 0).
struct SecondMaps {
    CUtensorMap a, b0, b1;
};

template <int BN, int NB, int EPI, int STAGES>
cudaError_t launch_tc(const CUtensorMap &mA, const CUtensorMap &mB0, const CUtensorMap &mB1,
                      const TcParams &p, long long max_tiles, cudaStream_t stream,
                      const SecondMaps *second = nullptr)
{
    using S = TcShape<BN, NB, STAGES>;
    auto kern = tc_gemm_kernel<BN, NB, EPI, STAGES>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    static DeviceOnce configured;
    if (configured.pending(dev)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   S::SMEM_BYTES);
        if (err == cudaSuccess)
            err = prefer_max_shared_carveout(kern);
        if (err != cudaSuccess)
            return err;
        configured.done(dev);
    }
    const long long grid =
        std::min<long long>(max_tiles + (long long)p.sh_tiles * std::max(1, p.sh_ksplit), sm_count());
    if (grid < 1)
        return cudaSuccess;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), (size_t)S::SMEM_BYTES, stream,
                      mA, mB0, mB1, second ? second->a : mA, second ? second->b0 : mB0,
                      second ? second->b1 : mB1, p);
}

// Launches the CTA-pair kernel as clusters of 2 (persistent: at most as
// many pairs as can be resident at once, and no more than there are pair
// tiles).
template <int BN, int NB, int EPI, int STAGES>
cudaError_t launch_tc_pair(const CUtensorMap &mA, const CUtensorMap &mB0, const CUtensorMap &mB1,
                           const TcParams &p, long long max_tiles, cudaStream_t stream)
{
    using S = PairShape<BN, NB, STAGES>;
    auto kern = tc_gemm_pair_kernel<BN, NB, EPI, STAGES>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    static DeviceOnce configured;
    static std::atomic<int> max_pairs[64];
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = S::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    int pairs_max = 0;
    if (configured.pending(dev)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   S::SMEM_BYTES);
        if (err == cudaSuccess)
            err = prefer_max_shared_carveout(kern);
        if (err != cudaSuccess)
            return err;
        cfg.gridDim = dim3((unsigned)(sm_count() & ~1));
        cfg.numAttrs = 1;
        int n = 0;
        err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (err != cudaSuccess)
            return err;
        n = std::max(1, n);
        if (dev >= 0 && dev < 64)
            max_pairs[dev].store(n, std::memory_order_relaxed);
        configured.done(dev);
        pairs_max = n;
    } else {
        pairs_max = max_pairs[dev].load(std::memory_order_relaxed);
    }
    const long long pairs = std::min<long long>(max_tiles, pairs_max);
    if (pairs < 1)
        return cudaSuccess;
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, mA, mB0, mB1, p);
}

}  // namespace

cudaError_t launch_router_tc(const moe_config &c, const void *x, const void *W_r, float *out,
                             int splits, int32_t *status, cudaStream_t stream)
{
    const int E = c.n_experts, D = c.d_model, T = c.T;
    const int bn = E <= 16 ? 16 : E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256;
    CUtensorMap mA, mB;
    if (!make_map(&mA, x, (uint64_t)T, (uint64_t)D, kTileM) ||
        !make_map(&mB, W_r, (uint64_t)E, (uint64_t)D, (uint32_t)bn))
        return cudaErrorInvalidValue;
    TcParams p{};
    p.seg_off = nullptr;
    p.mtile = nullptr;
    p.nseg = 1;
    p.dense_rows = T;
    p.K = D;
    p.n_tiles = 1;
    p.N_valid = E;
    p.b_seg_rows = 0;
    p.out = out;
    p.ld_out = E;
    p.status = status;
    p.ksplit = splits;
    p.part_stride = (long long)T * E;
    const long long tiles = (T + kTileM - 1) / kTileM * std::max(1, splits);
    switch (bn) {
    case 16: return launch_tc<16, 1, EPI_F32, 6>(mA, mB, mB, p, tiles, stream);
    case 32: return launch_tc<32, 1, EPI_F32, 6>(mA, mB, mB, p, tiles, stream);
    case 64: return launch_tc<64, 1, EPI_F32, 6>(mA, mB, mB, p, tiles, stream);
    case 128: return launch_tc<128, 1, EPI_F32, 6>(mA, mB, mB, p, tiles, stream);
    default: return launch_tc<256, 1, EPI_F32, 4>(mA, mB, mB, p, tiles, stream);
    }
}

cudaError_t launch_experts_tc(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                              const void *x, const void *W_gate, const void *W_up,
                              const void *W_down, const void *Ws_gate, const void *Ws_up,
                              const void *Ws_down, void *y, const AuxArgs &aux,
                              cudaStream_t stream, cudaEvent_t *ev)
{
    const int D = c.d_model, F = c.d_expert, S = c.d_shared, E = c.n_experts, T = c.T;
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    const int32_t *seg = reinterpret_cast<const int32_t *>(ws + L.seg_off);
    const int32_t *mtile = reinterpret_cast<const int32_t *>(ws + L.mtile);
    void *xp = ws + L.x_perm, *h = ws + L.h, *z = ws + L.z;
    void *hs = ws + L.hs, *zs = ws + L.zs;
    const long long R = L.R_max;
    const long long mt_bound = R / kTileM + E;     // >= sum_e ceil(kept_e / 128)
    const long long mt2_bound = R / kPairRows + E; // >= sum_e ceil(kept_e / 256)
    const long long mt_s = (T + kTileM - 1) / kTileM, mt2_s = (T + kPairRows - 1) / kPairRows;
    const bool wide_down = D > 1024;              // 256-column tiles for the down projection
    const int bn_down = wide_down ? 256 : 128;
    const LaunchPlan plan = plan_of(c);
    const bool pair_routed = plan.pair_routed, pair_shared = plan.pair_shared;
    // shared expert tiles in the routed launches (single-CTA kernels): they
    // share the machine with the routed tiles instead of running alone on a
    // few SMs (at decode sizes the shared GEMMs have only a handful of tiles)
    const bool fused = plan.shared_fused;
    cudaError_t err;

    // GEMM1 (routed): h = silu(x_perm W_gate^T) * (x_perm W_up^T)
    //   (+ fused: hs = silu(x Ws_gate^T) * (x Ws_up^T))
    {
        CUtensorMap mA, mG, mU;
        if (!make_map(&mA, xp, (uint64_t)R, (uint64_t)D, kTileM) ||
            !make_map(&mG, W_gate, (uint64_t)E * F, (uint64_t)D, 128) ||
            !make_map(&mU, W_up, (uint64_t)E * F, (uint64_t)D, 128))
            return cudaErrorInvalidValue;
        TcParams p{};
        p.seg_off = seg;
        p.mtile = mtile;
        p.nseg = E;
        p.K = D;
        p.n_tiles = (F + 127) / 128;
        p.N_valid = F;
        p.b_seg_rows = F;
        p.out = h;
        p.ld_out = F;
        p.status = status;
        p.aux = aux;
        SecondMaps sm;
        if (fused) {
            if (!make_map(&sm.a, x, (uint64_t)T, (uint64_t)D, kTileM) ||
                !make_map(&sm.b0, Ws_gate, (uint64_t)S, (uint64_t)D, 128) ||
                !make_map(&sm.b1, Ws_up, (uint64_t)S, (uint64_t)D, 128))
                return cudaErrorInvalidValue;
            p.sh_n_tiles = (S + 127) / 128;
            p.sh_tiles = (int)(mt_s * p.sh_n_tiles);
            p.sh_rows = T;
            p.sh_K = D;
            p.sh_N_valid = S;
            p.sh_out = hs;
            p.sh_ld_out = S;
        }
        if (pair_routed && plan.pair_tails) {
            // full 256-row tiles on CTA pairs, then each segment's remaining
            // rows (< 256) in 128-row single-CTA tiles: a 256-row tile over a
            // short remainder would compute mostly padding
            p.pair_full_only = 1;
            err = launch_tc_pair<128, 2, EPI_SWIGLU, 6>(mA, mG, mU, p, mt2_bound * p.n_tiles,
                                                        stream);
            if (err == cudaSuccess) {
                TcParams q = p;
                q.pair_full_only = 0;
                q.tail_after = kPairRows;
                q.aux.out = nullptr;  // evaluated by the pair launch
                err = launch_tc<128, 2, EPI_SWIGLU, 4>(mA, mG, mU, q, 2LL * E * q.n_tiles, stream);
            }
        } else if (pair_routed) {
            err = launch_tc_pair<128, 2, EPI_SWIGLU, 6>(mA, mG, mU, p, mt2_bound * p.n_tiles,
                                                        stream);
        } else {
            err = launch_tc<128, 2, EPI_SWIGLU, 4>(mA, mG, mU, p, mt_bound * p.n_tiles, stream,
                                                   fused ? &sm : nullptr);
        }
        if (err == cudaSuccess)
            err = record_stage(ev, 3, stream);
        if (err != cudaSuccess)
            return err;
    }
    // GEMM2 (routed): z = h W_down^T  (+ fused: zs = hs Ws_down^T)
    {
        CUtensorMap mA, mB;
        if (!make_map(&mA, h, (uint64_t)R, (uint64_t)F, kTileM) ||
            !make_map(&mB, W_down, (uint64_t)E * D, (uint64_t)F,
                      (uint32_t)(pair_routed ? bn_down / 2 : bn_down)))
            return cudaErrorInvalidValue;
        TcParams p{};
        p.seg_off = seg;
        p.mtile = mtile;
        p.nseg = E;
        p.K = F;
        p.n_tiles = (D + bn_down - 1) / bn_down;
        p.N_valid = D;
        p.b_seg_rows = D;
        p.out = z;
        p.ld_out = D;
        p.status = status;
        SecondMaps sm;
        if (fused) {
            if (!make_map(&sm.a, hs, (uint64_t)T, (uint64_t)S, kTileM) ||
                !make_map(&sm.b0, Ws_down, (uint64_t)D, (uint64_t)S, (uint32_t)bn_down))
                return cudaErrorInvalidValue;
            sm.b1 = sm.b0;
            p.sh_n_tiles = p.n_tiles;
            p.sh_tiles = (int)(mt_s * p.sh_n_tiles);
            p.sh_rows = T;
            p.sh_K = S;
            p.sh_N_valid = D;
            p.sh_out = zs;
            p.sh_ld_out = D;
            p.sh_ksplit = shared_down_splits(c);
            p.part_stride = (long long)T * D;
        }
        const SecondMaps *second = fused ? &sm : nullptr;
        const long long tiles = (pair_routed ? mt2_bound : mt_bound) * p.n_tiles;
        // pair tails: full 256-row tiles on pairs, the remainders on single CTAs
        const bool tails = pair_routed && plan.pair_tails;
        p.pair_full_only = tails ? 1 : 0;
        TcParams q = p;
        q.pair_full_only = 0;
        q.tail_after = kPairRows;
        const long long tail_tiles = 2LL * E * p.n_tiles;
        CUtensorMap mBt;  // the single-CTA kernel's B boxes hold bn_down rows
        if (tails && !make_map(&mBt, W_down, (uint64_t)E * D, (uint64_t)F, (uint32_t)bn_down))
            return cudaErrorInvalidValue;
        if (plan.direct_y) {
            p.out = y;
            p.row_tok = reinterpret_cast<const int32_t *>(ws + L.row_tok);
            p.row_w = reinterpret_cast<const float *>(ws + L.row_w);
            q.out = p.out;
            q.row_tok = p.row_tok;
            q.row_w = p.row_w;
            if (pair_routed) {
                err = wide_down ? launch_tc_pair<256, 1, EPI_BF16_Y, 6>(mA, mB, mB, p, tiles, stream)
                                : launch_tc_pair<128, 1, EPI_BF16_Y, 8>(mA, mB, mB, p, tiles, stream);
                if (err == cudaSuccess && tails)
                    err = wide_down
                              ? launch_tc<256, 1, EPI_BF16_Y, 4>(mA, mBt, mBt, q, tail_tiles, stream)
                              : launch_tc<128, 1, EPI_BF16_Y, 6>(mA, mBt, mBt, q, tail_tiles, stream);
            } else
                err = wide_down ? launch_tc<256, 1, EPI_BF16_Y, 4>(mA, mB, mB, p, tiles, stream)
                                : launch_tc<128, 1, EPI_BF16_Y, 6>(mA, mB, mB, p, tiles, stream);
        } else {
            if (pair_routed) {
                err = wide_down ? launch_tc_pair<256, 1, EPI_BF16, 6>(mA, mB, mB, p, tiles, stream)
                                : launch_tc_pair<128, 1, EPI_BF16, 8>(mA, mB, mB, p, tiles, stream);
                if (err == cudaSuccess && tails)
                    err = wide_down
                              ? launch_tc<256, 1, EPI_BF16, 4>(mA, mBt, mBt, q, tail_tiles, stream)
                              : launch_tc<128, 1, EPI_BF16, 6>(mA, mBt, mBt, q, tail_tiles, stream);
            } else
                err = wide_down
                          ? launch_tc<256, 1, EPI_BF16, 4>(mA, mB, mB, p, tiles, stream, second)
                          : launch_tc<128, 1, EPI_BF16, 6>(mA, mB, mB, p, tiles, stream, second);
        }
        if (err == cudaSuccess)
            err = record_stage(ev, 4, stream);
        if (err != cudaSuccess)
            return err;
    }
    if (S > 0 && !fused) {
        // the shared expert on its own: CTA pairs for large T, else one CTA
        // per tile
        {
            CUtensorMap mA, mG, mU;
            if (!make_map(&mA, x, (uint64_t)T, (uint64_t)D, kTileM) ||
                !make_map(&mG, Ws_gate, (uint64_t)S, (uint64_t)D, 128) ||
                !make_map(&mU, Ws_up, (uint64_t)S, (uint64_t)D, 128))
                return cudaErrorInvalidValue;
            TcParams p{};
            p.nseg = 1;
            p.dense_rows = T;
            p.K = D;
            p.n_tiles = (S + 127) / 128;
            p.N_valid = S;
            p.out = hs;
            p.ld_out = S;
            p.status = status;
            err = pair_shared
                      ? launch_tc_pair<128, 2, EPI_SWIGLU, 6>(mA, mG, mU, p, mt2_s * p.n_tiles, stream)
                      : launch_tc<128, 2, EPI_SWIGLU, 4>(mA, mG, mU, p, mt_s * p.n_tiles, stream);
            if (err == cudaSuccess)
                err = record_stage(ev, 5, stream);
            if (err != cudaSuccess)
                return err;
        }
        {
            CUtensorMap mA, mB;
            if (!make_map(&mA, hs, (uint64_t)T, (uint64_t)S, kTileM) ||
                !make_map(&mB, Ws_down, (uint64_t)D, (uint64_t)S,
                          (uint32_t)(pair_shared ? bn_down / 2 : bn_down)))
                return cudaErrorInvalidValue;
            TcParams p{};
            p.nseg = 1;
            p.dense_rows = T;
            p.K = S;
            p.n_tiles = (D + bn_down - 1) / bn_down;
            p.N_valid = D;
            p.out = zs;
            p.ld_out = D;
            p.status = status;
            if (pair_shared)
                err = wide_down
                          ? launch_tc_pair<256, 1, EPI_BF16, 6>(mA, mB, mB, p, mt2_s * p.n_tiles, stream)
                          : launch_tc_pair<128, 1, EPI_BF16, 8>(mA, mB, mB, p, mt2_s * p.n_tiles, stream);
            else
                err = wide_down ? launch_tc<256, 1, EPI_BF16, 4>(mA, mB, mB, p, mt_s * p.n_tiles, stream)
                                : launch_tc<128, 1, EPI_BF16, 6>(mA, mB, mB, p, mt_s * p.n_tiles, stream);
            if (err == cudaSuccess)
                err = record_stage(ev, 6, stream);
            if (err != cudaSuccess)
                return err;
        }
    } else {
        err = record_stage(ev, 5, stream);
        if (err == cudaSuccess)
            err = record_stage(ev, 6, stream);
        if (err != cudaSuccess)
            return err;
    }
    return cudaSuccess;
}

cudaError_t launch_dense_tc(int rows, int N, int K, const void *A, const void *B, void *out,
                            int32_t *status, cudaStream_t stream)
{
    if (rows <= 0)
        return cudaSuccess;
    // few rows: 32-column tiles so that enough CTAs stream the weights;
    // many rows: CTA pairs with 256-row tiles
    const bool narrow = rows <= 2 * kTileM;
    const bool pair = rows >= kPairMinRows / 4;
    const int bn = narrow ? 32 : (N > 1024 ? 256 : 128);
    CUtensorMap mA, mB;
    if (!make_map(&mA, A, (uint64_t)rows, (uint64_t)K, kTileM) ||
        !make_map(&mB, B, (uint64_t)N, (uint64_t)K, (uint32_t)(pair ? bn / 2 : bn)))
        return cudaErrorInvalidValue;
    TcParams p{};
    p.nseg = 1;
    p.dense_rows = rows;
    p.K = K;
    p.n_tiles = (N + bn - 1) / bn;
    p.N_valid = N;
    p.out = out;
    p.ld_out = N;
    p.status = status;
    const long long mt = (rows + kTileM - 1) / kTileM, mt2 = (rows + kPairRows - 1) / kPairRows;
    if (pair)
        return bn == 256 ? launch_tc_pair<256, 1, EPI_BF16, 6>(mA, mB, mB, p, mt2 * p.n_tiles, stream)
                         : launch_tc_pair<128, 1, EPI_BF16, 8>(mA, mB, mB, p, mt2 * p.n_tiles, stream);
    if (narrow)
        return launch_tc<32, 1, EPI_BF16, 8>(mA, mB, mB, p, mt * p.n_tiles, stream);
    return bn == 256 ? launch_tc<256, 1, EPI_BF16, 4>(mA, mB, mB, p, mt * p.n_tiles, stream)
                     : launch_tc<128, 1, EPI_BF16, 6>(mA, mB, mB, p, mt * p.n_tiles, stream);
}

}  // namespace moe
