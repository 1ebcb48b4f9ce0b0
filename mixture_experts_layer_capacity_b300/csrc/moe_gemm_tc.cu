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
//     stores it, then frees the accumulator so the next tile's MMAs overlap
//     this epilogue.
// For GEMM1 the gate and up tiles of the same columns are stacked in one
// 256-row B operand, so one N=256 MMA produces both accumulators.  The
// CTA-pair kernel (tc_gemm_pair_kernel, below) runs the same roles on
// 256-row tiles with cta_group::2 MMAs.  Both kernels have an E4M3 form for
// moe_forward_w8a8 (E4M3 token or hidden rows times E4M3 weights,
// kind::f8f6f4 with 128-element reduction steps in the same 128-byte rows;
// the epilogue scales by the row's and the weight row's fp32 scales and, as
// its main loop is short, stages its output rows and column scales in shared
// memory).
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

// Per-unit timeline of the routed pair GEMMs (builds with MOE_TIMELINE; see
// moe_timeline_read): 2 regions x 4096 units x 8 words, region 1 for the
// down projection.
constexpr int kTimelineUnits = 4096;
constexpr int kTimelineGemmWords = 2 * kTimelineUnits * 8;
static_assert(kTimelineGemmWords + 4096 * 8 == MOE_TIMELINE_WORDS, "timeline layout");
#ifdef MOE_TIMELINE
__device__ unsigned long long g_timeline[2 * 4096 * 8];
#else
__device__ unsigned long long g_timeline[8];
#endif

// Epilogues: fp32 store (router scores), bf16 store (z), SiLU(gate) * up in
// bf16 (h), bf16 store of w_row * acc straight into the row's token of y
// (down projection when every token has one expert and no shared expert),
// and SiLU(gate) * up in fp32 (h of the E4M3-activation path, quantized next).
enum { EPI_F32 = 0, EPI_BF16 = 1, EPI_SWIGLU = 2, EPI_BF16_Y = 3, EPI_SWIGLU_F32 = 4 };

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
    int sh_ksplit;           // splits of the second problem's reduction (fp32 partial
                             // outputs part_stride apart, EPI_BF16 kernels only); 0/1 = none
    void *sh_out;
    long long sh_ld_out;
    // single-CTA kernel with E4M3 operands (its F8 instantiation): the fp32
    // row scales of A (one per A row: token or hidden row) and of B (one per
    // B row, i.e. output column; for GEMM1 the gate and the up rows), for the
    // main and the second problem; the accumulator is scaled by both
    const float *a_scale, *b_scale0, *b_scale1;
    const float *sh_a_scale, *sh_b_scale0, *sh_b_scale1;
    // pair kernel, grouped: each segment's 256-row tiles as usual, except
    // that a small segment (fewer rows than one swap chunk) runs as swap
    // units in the same launch: the weights become the MMA's M = 256
    // operand and the few token rows its N operand (padded to a multiple of
    // 32, not to 256 rows)
    int swap_tails;
};

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far beyond any tile
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s
constexpr int kThreads = 192;

// Per-warp staging tile of the epilogues: 32 rows of one 32-column chunk
// (64 bytes of bf16 or 128 of fp32 per row), rows padded by 16 bytes so that
// the row-per-lane writes and the row-major reads spread over the banks.
constexpr int kEpiRowBytes = 128 + 16;
// and, for E4M3 tiles, the warp's copy of the tile's 256 column scales
constexpr int kEpiScaleFloats = 256;
constexpr int kEpiStageBytes = 4 * (32 * kEpiRowBytes + kEpiScaleFloats * 4);   // four warps

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
    // the epilogue warps' staging tiles, after the ring, barriers and tables
    static constexpr int EPI_OFF = (STAGES * STAGE_BYTES + 256 + TABLE_BYTES + 127) / 128 * 128;
    static constexpr int SMEM_BYTES = EPI_OFF + kEpiStageBytes + 1024;
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
    ti.a_row0 = s_seg[lo] + m * kTileM;
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
                                              const int *s_mt, int u, int ks_n, int kstep = 64)
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
        nk = (p.sh_K + kstep - 1) / kstep;
    } else {
        const int v = u - sh_units;
        const int g = v / ks_n;
        w.ks = v - g * ks_n;
        w.ti = tile_info(p, s_seg, s_mt, g);
        w.second = false;
        n_split = ks_n;
        nk = (p.K + kstep - 1) / kstep;
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

// Scales of an E4M3 tile's accumulator row: the A row's scale and the B
// rows' scales of the tile's columns (gate and up for GEMM1), copied into
// the epilogue warp's shared-memory scale buffer before the tile's
// accumulators are ready (stage_col_scales); b0 null: the operands are bf16
// and nothing is scaled.
struct EpiScale {
    float a;
    const float *b0, *b1;
};

// Copies n column scales of a tile (b: the first column's B row scale; col:
// that column's index in the output) into sb, 0 past the n_valid columns.
// Every lane of the warp calls it, between tiles; the warp's later reads
// see the copy.
__device__ __forceinline__ void stage_col_scales(const float *b, int col, int n_valid, float *sb,
                                                 int n)
{
    const int lane = threadIdx.x & 31;
    __syncwarp();   // the previous tile's reads of sb are done
    for (int c = lane; c < n; c += 32)
        sb[c] = col + c < n_valid ? __ldg(b + c) : 0.f;
    __syncwarp();
}

// Scales of 32 consecutive columns: the row scale a times each staged column
// scale (sb: the chunk's first entry of the warp's scale buffer in shared
// memory, 16-byte aligned; all lanes read the same words).
__device__ __forceinline__ void chunk_scales(const float *sb, float a, float (&cs)[32])
{
    const float4 *b4 = reinterpret_cast<const float4 *>(sb);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float4 t = b4[j];
        cs[4 * j] = a * t.x;
        cs[4 * j + 1] = a * t.y;
        cs[4 * j + 2] = a * t.z;
        cs[4 * j + 3] = a * t.w;
    }
}

// The rows a lane stores in warp_store_chunk: with PPR 16-byte pieces per
// row, pass `it` of a chunk stores piece lane % PPR of the warp's row
// it * (32 / PPR) + lane / PPR.  Those rows' first bytes and validity are
// fetched from their lanes once per tile (warp_rows), not once per chunk.
template <int PPR>
struct WarpRows {
    uint8_t *base[PPR];
    uint32_t ok;   // bit `it`: pass it's row is inside the tile
};

template <int PPR>
__device__ __forceinline__ WarpRows<PPR> warp_rows(uint8_t *row_base, bool row_ok)
{
    const int lane = threadIdx.x & 31;
    WarpRows<PPR> w;
    w.ok = 0;
#pragma unroll
    for (int it = 0; it < PPR; ++it) {
        const int r = it * (32 / PPR) + lane / PPR;
        w.base[it] = reinterpret_cast<uint8_t *>(
            __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(row_base), r));
        w.ok |= (__shfl_sync(0xffffffffu, row_ok ? 1u : 0u, r) & 1u) << it;
    }
    return w;
}

// Stores one 32-column chunk of the warp's 32 rows: each lane holds its own
// row's NW packed words (w); the words pass through the warp's staging tile
// so that each store instruction writes whole 64- or 128-byte row segments
// (4 or 8 lanes per row) instead of one 16-byte piece of 32 different rows.
// rows: the destinations (warp_rows of each row's first byte); off: the
// chunk's byte offset in its row; valid_bytes: bytes of each row inside the
// output's columns (<= NW * 4); es: element size (2 or 4) for a ragged tail.
// Every lane of the warp calls it.
template <int NW>
__device__ __forceinline__ void warp_store_chunk(uint8_t *stile, const uint32_t (&w)[NW],
                                                 const WarpRows<NW / 4> &rows, long long off,
                                                 int valid_bytes, int es)
{
    constexpr int PPR = NW / 4;                 // 16-byte pieces per row
    const int lane = threadIdx.x & 31;
    uint4 *srow = reinterpret_cast<uint4 *>(stile + lane * kEpiRowBytes);
#pragma unroll
    for (int j = 0; j < PPR; ++j)
        srow[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    __syncwarp();
    const int c = lane % PPR;
#pragma unroll
    for (int it = 0; it < PPR; ++it) {
        if (!((rows.ok >> it) & 1u) || c * 16 >= valid_bytes)
            continue;
        const int r = it * (32 / PPR) + lane / PPR;
        const uint8_t *src = stile + r * kEpiRowBytes + c * 16;
        uint8_t *g = rows.base[it] + off + c * 16;
        if ((c + 1) * 16 <= valid_bytes && (reinterpret_cast<uintptr_t>(g) & 15) == 0) {
            *reinterpret_cast<uint4 *>(g) = *reinterpret_cast<const uint4 *>(src);
        } else if (es == 2) {
            for (int e = 0; e < 8 && c * 16 + e * 2 < valid_bytes; ++e)
                reinterpret_cast<uint16_t *>(g)[e] = reinterpret_cast<const uint16_t *>(src)[e];
        } else {
            for (int e = 0; e < 4 && c * 16 + e * 4 < valid_bytes; ++e)
                reinterpret_cast<uint32_t *>(g)[e] = reinterpret_cast<const uint32_t *>(src)[e];
        }
    }
    __syncwarp();   // the tile is rewritten by the next chunk
}

// Bytes of a 32-column chunk starting at output column `col` that lie inside
// n_valid columns of es-byte elements.
__device__ __forceinline__ int chunk_valid_bytes(int col, int n_valid, int es)
{
    return max(0, min(32, n_valid - col)) * es;
}

// Stores a 32-column bf16 chunk of this lane's row (row_base: the row's
// first byte).  E4M3 tiles (STAGED), whose epilogue runs about as long as
// their short main loop, pass it through the warp's staging tile; bf16
// tiles store their 64 contiguous bytes directly (their epilogue hides
// behind the main loop, and staging measured slower for the small layers
// whose last epilogue is on the critical path).
template <bool STAGED>
__device__ __forceinline__ void store_chunk_bf16(uint8_t *stile, const uint32_t (&pk)[16],
                                                 const WarpRows<4> &rows, bool row_ok,
                                                 uint8_t *row_base, int col, int n_valid)
{
    if constexpr (STAGED) {
        warp_store_chunk<16>(stile, pk, rows, (long long)col * 2,
                             chunk_valid_bytes(col, n_valid, 2), 2);
    } else {
        if (row_ok)
            store_row_bf16(reinterpret_cast<__nv_bfloat16 *>(row_base) + col, pk, col,
                           n_valid);
    }
}

// Epilogue of one accumulator row (TMEM lane) of a tile: this thread owns
// output row `orow` (stored only when row_ok), columns n_idx*BN ... of the
// tile.  taddr: TMEM address of the row's first accumulator column.
// SCALED: E4M3 operands, the accumulator is multiplied by the row's and the
// column's scales (sc) first.  stile: the warp's staging tile (all lanes of
// the warp call this together; the E4M3 tiles' outputs are stored through
// it, whole row segments at a time).
template <int BN, int EPI, bool SCALED = false>
__device__ __forceinline__ void epilogue_row(const TcParams &p, void *out, long long ld_out,
                                             int n_valid, uint32_t taddr, bool row_ok,
                                             long long orow, int n_idx, int ks = 0,
                                             EpiScale sc = EpiScale{1.f, nullptr, nullptr},
                                             uint8_t *stile = nullptr)
{
    if constexpr (EPI == EPI_SWIGLU_F32) {
        uint8_t *row_base =
            reinterpret_cast<uint8_t *>(reinterpret_cast<float *>(out) + orow * ld_out);
        const WarpRows<8> rows = warp_rows<8>(row_base, row_ok);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t gv[32], uv[32];
            tmem_ld32(taddr + c0, gv);
            tmem_ld32(taddr + BN + c0, uv);
            tmem_wait_ld();
            const int col = n_idx * BN + c0;
            float gs[32], us[32];
            if constexpr (SCALED) {   // sc.a is 0 for rows outside the tile
                chunk_scales(sc.b0 + c0, sc.a, gs);
                chunk_scales(sc.b1 + c0, sc.a, us);
            }
            uint32_t hw[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float g = __uint_as_float(gv[i]), u = __uint_as_float(uv[i]);
                if constexpr (SCALED) {
                    g *= gs[i];
                    u *= us[i];
                }
                hw[i] = __float_as_uint(silu_f32(g) * u);
            }
            warp_store_chunk<32>(stile, hw, rows, (long long)col * 4,
                                 chunk_valid_bytes(col, n_valid, 4), 4);
        }
    } else if constexpr (EPI == EPI_SWIGLU) {
        uint8_t *row_base = reinterpret_cast<uint8_t *>(
            reinterpret_cast<__nv_bfloat16 *>(out) + orow * ld_out);
        WarpRows<4> rows{};
        if constexpr (SCALED)
            rows = warp_rows<4>(row_base, row_ok);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t gv[32], uv[32];
            tmem_ld32(taddr + c0, gv);
            tmem_ld32(taddr + BN + c0, uv);
            tmem_wait_ld();
            const int col = n_idx * BN + c0;
            uint32_t pk[16];
            float gs[32], us[32];
            if constexpr (SCALED) {   // sc.a is 0 for rows outside the tile
                chunk_scales(sc.b0 + c0, sc.a, gs);
                chunk_scales(sc.b1 + c0, sc.a, us);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float g0 = __uint_as_float(gv[2 * i]);
                float g1 = __uint_as_float(gv[2 * i + 1]);
                float u0 = __uint_as_float(uv[2 * i]);
                float u1 = __uint_as_float(uv[2 * i + 1]);
                if constexpr (SCALED) {
                    g0 *= gs[2 * i];
                    g1 *= gs[2 * i + 1];
                    u0 *= us[2 * i];
                    u1 *= us[2 * i + 1];
                }
                pk[i] = pack_bf16x2(silu_f32(g0) * u0, silu_f32(g1) * u1);
            }
            store_chunk_bf16<SCALED>(stile, pk, rows, row_ok, row_base, col, n_valid);
        }
    } else if constexpr (EPI == EPI_BF16_Y || EPI == EPI_BF16) {
        // EPI_BF16_Y: the row goes, times its gate weight, to its token's row of y
        int tok = 0;
        float wr = 1.f;
        if constexpr (EPI == EPI_BF16_Y) {
            wr = 0.f;
            if (row_ok) {
                tok = p.row_tok[orow];
                wr = p.row_w[orow];
            }
        }
        const long long drow = EPI == EPI_BF16_Y ? (long long)tok : orow;
        uint8_t *row_base = reinterpret_cast<uint8_t *>(
            reinterpret_cast<__nv_bfloat16 *>(out) + drow * ld_out);
        if constexpr (SCALED) {
            // E4M3 tiles: 64 columns per pass, so that each staged store
            // instruction writes four whole 128-byte row segments (with 32
            // columns, eight half segments: the down projection's 256-column
            // tiles then drained slowly enough to hold up the next tile's
            // MMAs)
            static_assert(BN % 64 == 0, "E4M3 bf16 tiles are multiples of 64 columns");
            const WarpRows<8> rows = warp_rows<8>(row_base, row_ok);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 64) {
                uint32_t v[2][32];
                tmem_ld32(taddr + c0, v[0]);
                tmem_ld32(taddr + c0 + 32, v[1]);
                tmem_wait_ld();
                uint32_t pk[32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float cs[32];   // sc.a is 0 for rows outside the tile
                    chunk_scales(sc.b0 + c0 + 32 * h, sc.a, cs);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float a0 = __uint_as_float(v[h][2 * i]);
                        float a1 = __uint_as_float(v[h][2 * i + 1]);
                        if constexpr (EPI == EPI_BF16_Y) {
                            a0 *= wr;
                            a1 *= wr;
                        }
                        pk[16 * h + i] = pack_bf16x2(a0 * cs[2 * i], a1 * cs[2 * i + 1]);
                    }
                }
                const int col = n_idx * BN + c0;
                warp_store_chunk<32>(stile, pk, rows, (long long)col * 2,
                                     max(0, min(64, n_valid - col)) * 2, 2);
            }
        } else {
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                tmem_ld32(taddr + c0, v);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float a0 = __uint_as_float(v[2 * i]);
                    float a1 = __uint_as_float(v[2 * i + 1]);
                    if constexpr (EPI == EPI_BF16_Y) {
                        a0 *= wr;
                        a1 *= wr;
                    }
                    pk[i] = pack_bf16x2(a0, a1);
                }
                const int col = n_idx * BN + c0;
                if (row_ok)
                    store_row_bf16(reinterpret_cast<__nv_bfloat16 *>(row_base) + col, pk, col,
                                   n_valid);
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
                if constexpr (SCALED) {
                    static_assert(CH % 32 == 0 || !SCALED, "scaled fp32 chunks of 32 columns");
#pragma unroll
                    for (int h = 0; h < CH; h += 32) {
                        float cs[32];
                        chunk_scales(sc.b0 + c0 + h, sc.a, cs);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[h + i] = __float_as_uint(__uint_as_float(v[h + i]) * cs[i]);
                    }
                }
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

// F8: E4M3 operands (tensor maps of bytes, 128-element reduction steps in
// the same 128-byte rows, kind::f8f6f4 MMAs with K = 32) and the scaled
// epilogue; otherwise bf16 operands, 64-element steps, kind::f16 with K = 16.
template <int BN, int NB, int EPI, int STAGES, bool F8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB0,
                   const __grid_constant__ CUtensorMap mB1, const __grid_constant__ CUtensorMap sA,
                   const __grid_constant__ CUtensorMap sB0, const __grid_constant__ CUtensorMap sB1,
                   const TcParams p)
{
    using S = TcShape<BN, NB, STAGES>;
    constexpr int KSTEP = F8 ? 128 : 64;   // reduction elements per 128-byte row of a stage
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
            tables[kMaxExperts + 1 + i] = p.mtile[i];
        }
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
                const UnitInfo w = unit_info(p, s_seg, s_mt, u, ks_n, KSTEP);
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
                    tma_load_2d(sa, ma, &full[s], kb * KSTEP, ti.a_row0);
                    tma_load_2d(sb, mb0, &full[s], kb * KSTEP, b_row);
                    if (NB == 2)
                        tma_load_2d(sb + S::B_BYTES, mb1, &full[s], kb * KSTEP, b_row);
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
            constexpr uint32_t idesc =
                F8 ? idesc_e4m3_f32(kTileM, S::UMMA_N) : idesc_bf16_f32(kTileM, S::UMMA_N);
            int s = 0;
            uint32_t ph = 0, b = 0, tph = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < ntiles && ok; u += G) {
                const UnitInfo w = unit_info(p, s_seg, s_mt, u, ks_n, KSTEP);
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
                    // four MMAs per stage, each over a 32-byte slice of the
                    // 128-byte rows (16 bf16 or 32 E4M3 elements)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if constexpr (F8)
                            umma_e4m3(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                                      (kb > kb0 || kk > 0) ? 1u : 0u);
                        else
                            umma_bf16(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                                      (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
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
        // this warp's staging tile for the stores and its column-scale
        // buffer (warps 2-5)
        uint8_t *stile = smem + S::EPI_OFF + (warp - 2) * 32 * kEpiRowBytes;
        float *sbuf = reinterpret_cast<float *>(smem + S::EPI_OFF + 4 * 32 * kEpiRowBytes) +
                      (warp - 2) * kEpiScaleFloats;
        (void)sbuf;
        uint32_t b = 0, tph = 0;
        for (int u = blockIdx.x; u < ntiles; u += G) {
            const UnitInfo w = unit_info(p, s_seg, s_mt, u, ks_n, KSTEP);
            const TileInfo &ti = w.ti;
            const int ks = w.ks;
            if constexpr (F8) {
                // the tile's column scales into this warp's buffer while its
                // accumulators are still being computed
                const long long b0 = (long long)(w.second ? 0 : ti.seg * p.b_seg_rows) +
                                     (long long)ti.n_idx * BN;
                const int nv = w.second ? p.sh_N_valid : p.N_valid;
                stage_col_scales((w.second ? p.sh_b_scale0 : p.b_scale0) + b0, ti.n_idx * BN, nv,
                                 sbuf, BN);
                if (NB == 2)
                    stage_col_scales((w.second ? p.sh_b_scale1 : p.b_scale1) + b0,
                                     ti.n_idx * BN, nv, sbuf + BN, BN);
            }
            if (!mbar_wait(&tfull[b], tph, abort_flag, kWaitLimitNs)) {
                *abort_flag = 1;
                set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + b * S::UMMA_N + ((uint32_t)(q * 32) << 16);
            const bool row_ok = r < ti.rows;
            const long long orow = (long long)ti.a_row0 + r;
            // E4M3 operands: the row's and the tile's column scales
            EpiScale sc{1.f, nullptr, nullptr};
            if constexpr (F8) {
                const float *as = w.second ? p.sh_a_scale : p.a_scale;
                sc.a = row_ok ? __ldg(as + orow) : 0.f;
                sc.b0 = sbuf;
                sc.b1 = NB == 2 ? sbuf + BN : sbuf;
            }
            if (w.second) {
                if constexpr (EPI == EPI_BF16) {
                    if (p.sh_ksplit > 1)  // fp32 partial sums of a piece of the reduction
                        epilogue_row<BN, EPI_F32, F8>(p, p.sh_out, p.sh_ld_out, p.sh_N_valid,
                                                      taddr, row_ok, orow, ti.n_idx, ks, sc);
                    else
                        epilogue_row<BN, EPI, F8>(p, p.sh_out, p.sh_ld_out, p.sh_N_valid, taddr,
                                                  row_ok, orow, ti.n_idx, ks, sc, stile);
                } else {
                    epilogue_row<BN, EPI, F8>(p, p.sh_out, p.sh_ld_out, p.sh_N_valid, taddr,
                                              row_ok, orow, ti.n_idx, ks, sc, stile);
                }
            } else
                epilogue_row<BN, EPI, F8>(p, p.out, p.ld_out, p.N_valid, taddr, row_ok, orow,
                                          ti.n_idx, ks, sc, stile);
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
    // a stage: the A slot and the B slot (full tiles), then the token rows of
    // a swap unit, which fills both slots with weight rows.  8 KB: GEMM1 swap
    // units take up to 128 token rows, GEMM2's up to 64 (two reduction steps
    // per stage); a smaller area cut the small experts into more chunks,
    // each streaming the same weight rows (4 KB: 218 + 288 chunks at the
    // DeepSeek-V3 shape, 8 KB: 189 + 218, both GEMMs ~4 % faster)
    static constexpr int TOK_BYTES = 8192;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + TOK_BYTES;
    static constexpr int TMEM_COLS = 2 * UMMA_N <= 256 ? 256 : 512;
    // segment offsets, full-tile prefix, swap-chunk prefix
    static constexpr int TABLE_BYTES = 3 * (kMaxExperts + 1) * 4 + 8;
    // reduction steps (64 wide) per swap stage: GEMM1 takes one (gate rows in
    // the A slot, up rows in the B slot), GEMM2 two when the B slot holds 128
    // weight rows (a 64-wide step each in the A and B slots), else one
    static constexpr int SWAP_KPS = (NB == 1 && B_HALF_ROWS == kTileM) ? 2 : 1;
    // token rows per swap unit: each CTA stages half of them per step
    static constexpr int SWAP_ROWS = 2 * TOK_BYTES / (SWAP_KPS * 128);
    static constexpr int EPI_OFF = (STAGES * STAGE_BYTES + 256 + TABLE_BYTES + 127) / 128 * 128;
    static constexpr int SMEM_BYTES = EPI_OFF + kEpiStageBytes + 1024;
    static_assert(UMMA_N == 128 || UMMA_N == 256, "pair UMMA N");
    static_assert(NB == 1 || B_HALF_ROWS == BN, "gate/up halves");
    static_assert(B_BYTES % 1024 == 0, "B tile must keep 1024-byte alignment");
    static_assert(SWAP_ROWS % 32 == 0 && SWAP_ROWS <= UMMA_N && SWAP_ROWS <= 128,
                  "swap unit columns fit the accumulator (GEMM1: gate and up halves)");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

constexpr int kPairRows = 2 * kTileM;
constexpr int kSwapBoxRows = 16;   // token rows per TMA box of a swap unit
constexpr int kSwapFeat = 256;     // features per swap unit: 128 weight rows per CTA
                                   // (GEMM1: of both the gate and the up matrix)

__device__ __forceinline__ int pair_tile_count(const TcParams &p, const int *s_mt)
{
    if (!s_mt)
        return ((p.dense_rows + kPairRows - 1) / kPairRows) * p.n_tiles;
    return s_mt[p.nseg] * p.n_tiles;
}

// Row tiles per raster group of a pair launch.  Pairs running at the same
// time take consecutive tiles; within a group of kRowGroup row tiles the
// column tile changes slowest, so the ~74 concurrent tiles touch about
// kRowGroup A row tiles and 74 / kRowGroup B column tiles.  At the
// DeepSeek-V3 shape (D = 7168: 3.7 MB per A or B tile) that is ~63 MB, which
// L2 holds; walking all of a large expert's row tiles per column tile
// instead (its x rows: up to ~230 MB) re-read them from DRAM for every
// column tile (GEMM1 read 2.9x its weight bytes).
constexpr int kRowGroup = 8;

// Tile `local` of an mt x nt grid of row and column tiles in grouped raster
// order: groups of kRowGroup row tiles; within a group, column-major.
__device__ __forceinline__ void grouped_raster(int local, int mt, int nt, int &m, int &n)
{
    const int grp = local / (kRowGroup * nt);
    const int rows = min(kRowGroup, mt - grp * kRowGroup);
    const int within = local - grp * kRowGroup * nt;
    n = within / rows;
    m = grp * kRowGroup + (within - n * rows);
}

// a_row0 / rows: the pair tile's first A row and its valid rows (<= 256).
__device__ __forceinline__ TileInfo pair_tile_info(const TcParams &p, const int *s_seg,
                                                   const int *s_mt, int g)
{
    TileInfo ti;
    int m;
    if (!s_mt) {
        const int mt = (p.dense_rows + kPairRows - 1) / kPairRows;
        grouped_raster(g, mt, p.n_tiles, m, ti.n_idx);
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
    grouped_raster(g - mt0 * p.n_tiles, mt_e, p.n_tiles, m, ti.n_idx);
    ti.seg = lo;
    ti.a_row0 = s_seg[lo] + m * kPairRows;
    ti.rows = min(kPairRows, s_seg[lo + 1] - ti.a_row0);
    return ti;
}

// One CTA pair's work list with swap units: its share of the full tiles
// (g = cluster, cluster + NC, ...), then its share of the swap units
// (likewise).  Every role of both CTAs walks the same sequence.  (Spreading
// the swap units evenly among the full tiles, or putting them first, was
// slower at the DeepSeek-V3 prefill shape: same box, alternating runs, down
// projection 3.85 / 3.76 ms against 3.72 ms with them last; the gate/up
// GEMM was unchanged.)
struct PairSched {
    int cid, NC, a, b, i, j;
    __device__ __forceinline__ PairSched(int cid_, int NC_, int n_full, int n_swap)
        : cid(cid_), NC(NC_), i(0), j(0)
    {
        a = n_full > cid ? (n_full - cid + NC - 1) / NC : 0;
        b = n_swap > cid ? (n_swap - cid + NC - 1) / NC : 0;
    }
    // Next unit: returns false when none is left; `swap` tells the kind and
    // `g` its index in that kind's list.
    __device__ __forceinline__ bool next(bool &swap, int &g)
    {
        if (i >= a && j >= b)
            return false;
        swap = i >= a;
        g = cid + NC * (swap ? j++ : i++);
        return true;
    }
};

// A swap unit: token rows [r0, r0 + rv) of segment `seg` (rv <= swap_rows,
// n = rv rounded up to 32, the MMA's N), feature block fb (kSwapFeat
// features: weight rows fb * kSwapFeat + rank * 128 ... of each CTA).
struct SwapInfo {
    int seg, fb, r0, rv, n;
};

// Swap unit u: chunk-major (a small segment is one chunk of at most
// swap_rows rows), feature block minor, so the units of one chunk run
// at about the same time on neighbouring pairs and share its token rows in
// L2.  s_sw: prefix sum of chunks per segment.
__device__ __forceinline__ SwapInfo swap_info(const int *s_seg, const int *s_sw, int nseg,
                                              int n_fb, int swap_rows, int u)
{
    SwapInfo si;
    const int gc = u / n_fb;
    si.fb = u - gc * n_fb;
    int lo = 0, hi = nseg;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_sw[mid] <= gc)
            lo = mid;
        else
            hi = mid;
    }
    si.seg = lo;
    si.r0 = s_seg[lo] + (gc - s_sw[lo]) * swap_rows;
    si.rv = min(swap_rows, s_seg[lo + 1] - si.r0);
    si.n = (si.rv + 31) & ~31;
    return si;
}

// Epilogue of a swap unit (pair kernel).  The accumulator holds weight rows
// (this CTA's 128 features) in TMEM lanes and token rows in columns: column c
// is token row si.r0 + c, valid for c < si.rv.
//   GEMM1 (EPI_SWIGLU): gate in columns [0, n), up in [128, 128 + n) of the
//     same lanes, so each thread combines its own two values;
//   GEMM2 (EPI_BF16 / EPI_BF16_Y): one output feature per lane.
// A thread stores one value per token row; a warp's 32 lanes write 64
// contiguous bytes of the row (128 for EPI_SWIGLU_F32's fp32 h).  taddr: this
// warp's lane quarter of the buffer.  F8: E4M3 operands; each accumulator is
// scaled by its weight row's scale (b_scale0 / b_scale1: gate / up, or down)
// and its token row's scale (a_scale) first.
template <int EPI, bool F8 = false>
__device__ __forceinline__ void swap_epilogue(const TcParams &p, uint32_t taddr, int q, int lane,
                                              int rank, const SwapInfo &si)
{
    constexpr bool kGlu = EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_F32;
    __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.out);
    const int f = si.fb * kSwapFeat + rank * kTileM + q * 32 + lane;
    const bool f_ok = f < p.N_valid;
    float wg = 1.f, wu = 1.f;
    if constexpr (F8) {
        const long long wr = (long long)si.seg * p.b_seg_rows + f;
        wg = f_ok ? __ldg(p.b_scale0 + wr) : 0.f;
        if constexpr (kGlu)
            wu = f_ok ? __ldg(p.b_scale1 + wr) : 0.f;
    }
#pragma unroll 1
    for (int c0 = 0; c0 < si.n; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(taddr + c0, v);
        if constexpr (kGlu) {
            uint32_t u[32];
            tmem_ld32(taddr + kTileM + c0, u);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float g = __uint_as_float(v[c]), uu = __uint_as_float(u[c]);
                if constexpr (F8) {
                    // token rows past the unit's valid ones read a clamped scale
                    const float ts = __ldg(p.a_scale + si.r0 + min(c0 + c, si.rv - 1));
                    g *= wg * ts;
                    uu *= wu * ts;
                }
                v[c] = __float_as_uint(silu_f32(g) * uu);
            }
        } else {
            tmem_wait_ld();
            if constexpr (F8) {
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    v[c] = __float_as_uint(__uint_as_float(v[c]) * wg *
                                           __ldg(p.a_scale + si.r0 + min(c0 + c, si.rv - 1)));
            }
        }
        if (f_ok) {
            const int nc = si.rv - c0;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                if (c >= nc)
                    break;
                const int row = si.r0 + c0 + c;
                if constexpr (EPI == EPI_SWIGLU_F32) {
                    reinterpret_cast<float *>(p.out)[(long long)row * p.ld_out + f] =
                        __uint_as_float(v[c]);
                } else if constexpr (EPI == EPI_BF16_Y) {
                    const int tok = p.row_tok[row];
                    out[(long long)tok * p.ld_out + f] =
                        __float2bfloat16_rn(p.row_w[row] * __uint_as_float(v[c]));
                } else {
                    out[(long long)row * p.ld_out + f] = __float2bfloat16_rn(__uint_as_float(v[c]));
                }
            }
        }
    }
}

// F8: E4M3 operands as in tc_gemm_kernel (128-element reduction steps in the
// same 128-byte rows, kind::f8f6f4 MMAs, both scales in the epilogues).
template <int BN, int NB, int EPI, int STAGES, bool F8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap mA,
                        const __grid_constant__ CUtensorMap mB0,
                        const __grid_constant__ CUtensorMap mB1,
                        const __grid_constant__ CUtensorMap wS0,
                        const __grid_constant__ CUtensorMap wS1,
                        const __grid_constant__ CUtensorMap tS, const TcParams p)
{
    using S = PairShape<BN, NB, STAGES>;
    static_assert((EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_F32) ? NB == 2 : NB == 1,
                  "pair epilogues");
    static_assert(!F8 || EPI != EPI_SWIGLU, "E4M3 GEMM1 writes fp32 h");
    constexpr int KSTEP = F8 ? 128 : 64;   // reduction elements per 128-byte row
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
    int *s_sw = p.mtile ? tables + 2 * (kMaxExperts + 1) : nullptr;

    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster_id = (int)(blockIdx.x >> 1), nclusters = (int)(gridDim.x >> 1);
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    const bool swap_mode = p.swap_tails && p.mtile;

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
        if (swap_mode) {
            tma_prefetch_desc(&wS0);
            if (NB == 2)
                tma_prefetch_desc(&wS1);
            tma_prefetch_desc(&tS);
        }
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
    // pair tiles per segment (256 rows each, the last one padded) and, with
    // swap units, the chunks of each small segment (which then has no pair
    // tile), prefix-summed by warp 0.  A segment with pair tiles keeps its
    // remainder in a padded pair tile next to its other row tiles, so its
    // weight tiles are still shared through L2.  Small: fewer rows than one
    // swap chunk holds (SWAP_ROWS: 128 in the gate/up GEMM, 64 in the wide
    // down projection), since every further chunk streams the expert's
    // weight rows again while a padded pair tile streams them once per
    // column tile (DeepSeek-V3 prefill shape, same box, alternating runs,
    // against a 256-row threshold: GEMM1 7.29 -> 7.10 ms and GEMM2 3.98 ->
    // 3.81 ms in bf16, GEMM1 3.88 -> 3.78 ms with E4M3 activations; 192 rows
    // for GEMM1, 32 or none for GEMM2 were slower).
    if (p.mtile && !failed && warp == 0) {
        int carry = 0, carry_sw = 0;
        for (int e0 = 0; e0 < p.nseg; e0 += 32) {
            const int e = e0 + lane;
            const int n = e < p.nseg ? s_seg[e + 1] - s_seg[e] : 0;
            const bool small = swap_mode && n < S::SWAP_ROWS;
            const int v = small ? 0 : (n + kPairRows - 1) / kPairRows;
            const int vs = small ? (n + S::SWAP_ROWS - 1) / S::SWAP_ROWS : 0;
            int incl = v, incl_s = vs;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n1 = __shfl_up_sync(0xffffffffu, incl, o);
                const int n2 = __shfl_up_sync(0xffffffffu, incl_s, o);
                if (lane >= o) {
                    incl += n1;
                    incl_s += n2;
                }
            }
            if (e < p.nseg) {
                s_mt[e + 1] = carry + incl;
                s_sw[e + 1] = carry_sw + incl_s;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
            carry_sw += __shfl_sync(0xffffffffu, incl_s, 31);
        }
        if (lane == 0) {
            s_mt[0] = 0;
            s_sw[0] = 0;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    // feature blocks of the swap units (kSwapFeat features each)
    const int n_fb = (p.N_valid + kSwapFeat - 1) / kSwapFeat;
    const int n_full = failed ? 0 : pair_tile_count(p, s_mt);
    const int n_swap = (failed || !swap_mode) ? 0 : s_sw[p.nseg] * n_fb;
    const int NC = balanced_workers(n_full + n_swap, nclusters);
    const bool active = cluster_id < NC;
    const int nk = (p.K + KSTEP - 1) / KSTEP;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint32_t full_leader = mapa_shared(smem_u32(&full[0]), 0);
            int s = 0;
            uint32_t ph = 0;
            long long fills = 0;
            bool ok = true;
            PairSched sched(cluster_id, NC, active ? n_full : 0, active ? n_swap : 0);
            bool sw;
            int g;
            while (ok && sched.next(sw, g)) {
                int a_row, b_row, t_row = 0, half = 0;
                const CUtensorMap *ma = &mA, *mb = (NB == 2 && !leader) ? &mB1 : &mB0;
                uint32_t tx;
                if (!sw) {
                    const TileInfo ti = pair_tile_info(p, s_seg, s_mt, g);
                    a_row = ti.a_row0 + (int)rank * kTileM;
                    b_row = ti.seg * p.b_seg_rows + ti.n_idx * BN +
                            (NB == 1 ? (int)rank * S::B_HALF_ROWS : 0);
                    tx = 2 * (S::A_BYTES + S::B_BYTES);   // both CTAs' slots
                } else {
                    const SwapInfo si = swap_info(s_seg, s_sw, p.nseg, n_fb, S::SWAP_ROWS, g);
                    // this CTA's 128 weight rows of the unit's features (GEMM1:
                    // of W_gate into the A slot and of W_up into the B slot;
                    // GEMM2: of W_down, one reduction step per slot) and its
                    // half of the token rows into the token area
                    a_row = si.seg * p.b_seg_rows + si.fb * kSwapFeat + (int)rank * kTileM;
                    half = si.n / 2;
                    t_row = si.r0 + (int)rank * half;
                    b_row = 0;
                    tx = 0;   // per stage below: its last one may hold a single step
                }
                const int n_stages = sw ? (nk + S::SWAP_KPS - 1) / S::SWAP_KPS : nk;
                for (int st = 0; st < n_stages; ++st) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + s * S::STAGE_BYTES;
                    uint8_t *sb = sa + S::A_BYTES;
                    uint8_t *stok = sb + S::B_BYTES;
                    const uint32_t fb = full_leader + (uint32_t)s * 8u;
                    if (!sw) {
                        if (leader)
                            mbar_arrive_expect_tx(&full[s], tx);
                        tma_load_2d_pair(sa, ma, fb, st * KSTEP, a_row);
                        tma_load_2d_pair(sb, mb, fb, st * KSTEP, b_row);
                    } else {
                        const int k0 = st * S::SWAP_KPS;
                        const int steps = min(S::SWAP_KPS, nk - k0);
                        const uint32_t wbytes = NB == 2 ? 2u * S::A_BYTES : (uint32_t)steps * S::A_BYTES;
                        if (leader)
                            mbar_arrive_expect_tx(&full[s],
                                                  2u * (wbytes + (uint32_t)(steps * half * 128)));
                        if (NB == 2) {
                            tma_load_2d_pair(sa, &wS0, fb, k0 * KSTEP, a_row);
                            tma_load_2d_pair(sb, &wS1, fb, k0 * KSTEP, a_row);
                        } else {
                            for (int j = 0; j < steps; ++j)
                                tma_load_2d_pair(sa + j * S::A_BYTES, &wS0, fb, (k0 + j) * KSTEP,
                                                 a_row);
                        }
                        for (int j = 0; j < steps; ++j)
                            for (int r = 0; r < half; r += kSwapBoxRows)
                                tma_load_2d_pair(stok + j * (S::TOK_BYTES / S::SWAP_KPS) + r * 128,
                                                 &tS, fb, (k0 + j) * KSTEP, t_row + r);
                    }
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
            constexpr uint32_t idesc_full = F8 ? idesc_e4m3_f32(kPairRows, S::UMMA_N)
                                               : idesc_bf16_f32(kPairRows, S::UMMA_N);
            // one K = 16 (bf16) or K = 32 (E4M3) step of the pair
            auto mma = [](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
                if constexpr (F8)
                    umma_e4m3_pair(d, a, b, id, acc);
                else
                    umma_bf16_pair(d, a, b, id, acc);
            };
            int s = 0;
            uint32_t ph = 0, b = 0, tph = 0;
            bool ok = true;
            PairSched sched(cluster_id, NC, active ? n_full : 0, active ? n_swap : 0);
            bool sw;
            int g;
            int tl_i = 0;
            while (ok && sched.next(sw, g)) {
                const uint64_t tl0 = kTimeline ? global_timer_ns() : 0;
                uint32_t idesc = idesc_full;
                if (sw) {
                    const SwapInfo si = swap_info(s_seg, s_sw, p.nseg, n_fb, S::SWAP_ROWS, g);
                    idesc = F8 ? idesc_e4m3_f32(kPairRows, si.n) : idesc_bf16_f32(kPairRows, si.n);
                }
                if (!mbar_wait(&tempty[b], tph ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t tl1 = kTimeline ? global_timer_ns() : 0;
                uint64_t tl2 = 0;
                const uint32_t d_tmem = tmem_base + b * S::UMMA_N;
                const int n_stages = sw ? (nk + S::SWAP_KPS - 1) / S::SWAP_KPS : nk;
                for (int st = 0; st < n_stages; ++st) {
                    if (!mbar_wait(&full[s], ph, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (kTimeline && st == 0)
                        tl2 = global_timer_ns();
                    const uint32_t sa = smem_u32(smem + s * S::STAGE_BYTES);
                    if (!sw) {
                        const uint64_t adesc = sdesc_kmajor_sw128(sa);
                        const uint64_t bdesc = sdesc_kmajor_sw128(sa + S::A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma(d_tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                                (st > 0 || kk > 0) ? 1u : 0u);
                    } else if (NB == 2) {
                        // gate rows (A slot) into columns [0, n), up rows (B
                        // slot) into [128, 128 + n); tokens from the token area
                        const uint64_t gdesc = sdesc_kmajor_sw128(sa);
                        const uint64_t udesc = sdesc_kmajor_sw128(sa + S::A_BYTES);
                        const uint64_t tdesc = sdesc_kmajor_sw128(sa + S::A_BYTES + S::B_BYTES);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t acc = (st > 0 || kk > 0) ? 1u : 0u;
                            mma(d_tmem, gdesc + 2u * kk, tdesc + 2u * kk, idesc, acc);
                            mma(d_tmem + kTileM, udesc + 2u * kk, tdesc + 2u * kk, idesc, acc);
                        }
                    } else {
                        // one or two reduction steps: weights in the A (and B)
                        // slot, their token rows in the halves of the token area
                        const int steps = min(S::SWAP_KPS, nk - st * S::SWAP_KPS);
                        for (int j = 0; j < steps; ++j) {
                            const uint64_t wdesc = sdesc_kmajor_sw128(sa + j * S::A_BYTES);
                            const uint64_t tdesc = sdesc_kmajor_sw128(
                                sa + S::A_BYTES + S::B_BYTES + j * (S::TOK_BYTES / S::SWAP_KPS));
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma(d_tmem, wdesc + 2u * kk, tdesc + 2u * kk, idesc,
                                    (st > 0 || j > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    umma_commit_pair(&empty[s], 0x3);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                if constexpr (kTimeline) {
                    if (blockIdx.x == 0 && p.mtile && tl_i < kTimelineUnits) {
                        unsigned long long *rec =
                            g_timeline + (EPI == EPI_BF16 || EPI == EPI_BF16_Y ? kTimelineUnits * 8 : 0) +
                            tl_i * 8;
                        rec[0] = tl0;
                        rec[1] = tl1;
                        rec[2] = tl2;
                        rec[3] = global_timer_ns();
                        rec[6] = sw ? 1 : 0;
                    }
                    ++tl_i;
                }
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
        // this warp's staging tile for the stores and its column-scale
        // buffer (warps 2-5)
        uint8_t *stile = smem + S::EPI_OFF + (warp - 2) * 32 * kEpiRowBytes;
        float *sbuf = reinterpret_cast<float *>(smem + S::EPI_OFF + 4 * 32 * kEpiRowBytes) +
                      (warp - 2) * kEpiScaleFloats;
        (void)sbuf;
        const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[0]), 0);
        uint32_t b = 0, tph = 0;
        PairSched sched(cluster_id, NC, active ? n_full : 0, active ? n_swap : 0);
        bool sw;
        int g;
        int tl_e = 0;
        while (sched.next(sw, g)) {
            const uint64_t te0 = kTimeline ? global_timer_ns() : 0;
            TileInfo ti{};
            if (!sw) {
                ti = pair_tile_info(p, s_seg, s_mt, g);
                if constexpr (F8) {
                    // the tile's column scales into this warp's buffer while
                    // its accumulators are still being computed
                    const long long b0 =
                        (long long)ti.seg * p.b_seg_rows + (long long)ti.n_idx * BN;
                    stage_col_scales(p.b_scale0 + b0, ti.n_idx * BN, p.N_valid, sbuf, BN);
                    if (NB == 2)
                        stage_col_scales(p.b_scale1 + b0, ti.n_idx * BN, p.N_valid, sbuf + BN,
                                         BN);
                }
            }
            if (!mbar_wait(&tfull[b], tph, abort_flag, kWaitLimitNs)) {
                *abort_flag = 1;
                set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + b * S::UMMA_N + ((uint32_t)(q * 32) << 16);
            const uint64_t te1 = kTimeline ? global_timer_ns() : 0;
            if (!sw) {
                const int my_rows = ti.rows - (int)rank * kTileM;
                const bool row_ok = r < my_rows;
                const long long orow = (long long)ti.a_row0 + (int)rank * kTileM + r;
                EpiScale sc{1.f, nullptr, nullptr};
                if constexpr (F8) {
                    sc.a = row_ok ? __ldg(p.a_scale + orow) : 0.f;
                    sc.b0 = sbuf;
                    sc.b1 = NB == 2 ? sbuf + BN : sbuf;
                }
                epilogue_row<BN, EPI, F8>(p, p.out, p.ld_out, p.N_valid, taddr, row_ok, orow,
                                          ti.n_idx, 0, sc, stile);
            } else {
                const SwapInfo si = swap_info(s_seg, s_sw, p.nseg, n_fb, S::SWAP_ROWS, g);
                swap_epilogue<EPI, F8>(p, taddr, q, lane, (int)rank, si);
            }
            if constexpr (kTimeline) {
                if (blockIdx.x == 0 && p.mtile && warp == 2 && lane == 0 && tl_e < kTimelineUnits) {
                    unsigned long long *rec =
                        g_timeline + (EPI == EPI_BF16 || EPI == EPI_BF16_Y ? kTimelineUnits * 8 : 0) +
                        tl_e * 8;
                    rec[4] = te1;
                    rec[5] = global_timer_ns();
                    rec[7] = te0;
                }
                ++tl_e;
            }
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

template <int BN, int NB, int EPI, int STAGES, bool F8 = false>
cudaError_t launch_tc(const CUtensorMap &mA, const CUtensorMap &mB0, const CUtensorMap &mB1,
                      const TcParams &p, long long max_tiles, cudaStream_t stream,
                      const SecondMaps *second = nullptr)
{
    using S = TcShape<BN, NB, STAGES>;
    auto kern = tc_gemm_kernel<BN, NB, EPI, STAGES, F8>;
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

// The swap units' operands (TcParams::swap_tails): weight maps (GEMM1: W_gate
// and W_up in 16-row boxes; GEMM2: W_down in 128-row boxes) and the token
// rows (x_perm or h) in 16-row boxes.
struct SwapMaps {
    CUtensorMap w0, w1, t;
};

// Launches the CTA-pair kernel as clusters of 2 (persistent: at most as
// many pairs as can be resident at once, and no more than there are units).
template <int BN, int NB, int EPI, int STAGES, bool F8 = false>
cudaError_t launch_tc_pair(const CUtensorMap &mA, const CUtensorMap &mB0, const CUtensorMap &mB1,
                           const TcParams &p, long long max_tiles, cudaStream_t stream,
                           const SwapMaps *swap = nullptr)
{
    using S = PairShape<BN, NB, STAGES>;
    auto kern = tc_gemm_pair_kernel<BN, NB, EPI, STAGES, F8>;
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
    if (p.swap_tails && !swap)
        return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, kern, mA, mB0, mB1, swap ? swap->w0 : mA, swap ? swap->w1 : mA,
                              swap ? swap->t : mA, p);
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
        if (pair_routed) {
            // 256-row tiles on CTA pairs and, in the same launch, the small
            // experts as swap units: a 256-row tile over a few rows would
            // compute mostly padding
            SwapMaps sw;
            if (!make_map(&sw.w0, W_gate, (uint64_t)E * F, (uint64_t)D, kTileM) ||
                !make_map(&sw.w1, W_up, (uint64_t)E * F, (uint64_t)D, kTileM) ||
                !make_map(&sw.t, xp, (uint64_t)R, (uint64_t)D, kSwapBoxRows))
                return cudaErrorInvalidValue;
            p.swap_tails = 1;
            const long long units = mt2_bound * p.n_tiles + 8LL * E * ((F + kSwapFeat - 1) / kSwapFeat);
            err = launch_tc_pair<128, 2, EPI_SWIGLU, 5>(mA, mG, mU, p, units, stream, &sw);
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
        long long tiles = (pair_routed ? mt2_bound : mt_bound) * p.n_tiles;
        // pairs: 256-row tiles and the small experts as swap units (W_down
        // rows in 128-row boxes, h rows in 16-row boxes)
        SwapMaps sw;
        if (pair_routed) {
            if (!make_map(&sw.w0, W_down, (uint64_t)E * D, (uint64_t)F, kTileM) ||
                !make_map(&sw.t, h, (uint64_t)R, (uint64_t)F, kSwapBoxRows))
                return cudaErrorInvalidValue;
            sw.w1 = sw.w0;
            p.swap_tails = 1;
            tiles += 8LL * E * ((D + kSwapFeat - 1) / kSwapFeat);
        }
        if (plan.direct_y) {
            p.out = y;
            p.row_tok = reinterpret_cast<const int32_t *>(ws + L.row_tok);
            p.row_w = reinterpret_cast<const float *>(ws + L.row_w);
            if (pair_routed)
                err = wide_down
                          ? launch_tc_pair<256, 1, EPI_BF16_Y, 5>(mA, mB, mB, p, tiles, stream, &sw)
                          : launch_tc_pair<128, 1, EPI_BF16_Y, 6>(mA, mB, mB, p, tiles, stream, &sw);
            else
                err = wide_down ? launch_tc<256, 1, EPI_BF16_Y, 4>(mA, mB, mB, p, tiles, stream)
                                : launch_tc<128, 1, EPI_BF16_Y, 6>(mA, mB, mB, p, tiles, stream);
        } else {
            if (pair_routed)
                err = wide_down
                          ? launch_tc_pair<256, 1, EPI_BF16, 5>(mA, mB, mB, p, tiles, stream, &sw)
                          : launch_tc_pair<128, 1, EPI_BF16, 6>(mA, mB, mB, p, tiles, stream, &sw);
            else
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
                      ? launch_tc_pair<128, 2, EPI_SWIGLU, 5>(mA, mG, mU, p, mt2_s * p.n_tiles, stream)
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
                          ? launch_tc_pair<256, 1, EPI_BF16, 5>(mA, mB, mB, p, mt2_s * p.n_tiles, stream)
                          : launch_tc_pair<128, 1, EPI_BF16, 6>(mA, mB, mB, p, mt2_s * p.n_tiles, stream);
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
        return bn == 256 ? launch_tc_pair<256, 1, EPI_BF16, 5>(mA, mB, mB, p, mt2 * p.n_tiles, stream)
                         : launch_tc_pair<128, 1, EPI_BF16, 6>(mA, mB, mB, p, mt2 * p.n_tiles, stream);
    if (narrow)
        return launch_tc<32, 1, EPI_BF16, 8>(mA, mB, mB, p, mt * p.n_tiles, stream);
    return bn == 256 ? launch_tc<256, 1, EPI_BF16, 4>(mA, mB, mB, p, mt * p.n_tiles, stream)
                     : launch_tc<128, 1, EPI_BF16, 6>(mA, mB, mB, p, mt * p.n_tiles, stream);
}

namespace {

// launch_experts_w8a8 for layers large enough for CTA pairs (plan.pair_routed):
// the routed GEMMs on the pair kernel (256-row tiles, small experts as swap
// units), the shared expert's GEMMs on their own launches (pairs
// when plan.pair_shared).
cudaError_t experts_w8a8_pairs(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                               const ExpertW8 &w, void *y, const AuxArgs &aux,
                               cudaStream_t stream, cudaEvent_t *ev)
{
    const int D = c.d_model, F = c.d_expert, S = c.d_shared, E = c.n_experts, T = c.T;
    const A8Layout A = a8_layout_of(c, L);
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    const int32_t *seg = reinterpret_cast<const int32_t *>(ws + L.seg_off);
    const int32_t *mtile = reinterpret_cast<const int32_t *>(ws + L.mtile);
    const long long R = L.R_max;
    const long long mt2_bound = R / kPairRows + E;
    const long long mt_s = (T + kTileM - 1) / kTileM, mt2_s = (T + kPairRows - 1) / kPairRows;
    const LaunchPlan plan = plan_of(c);
    const bool shared = S > 0, pair_shared = plan.pair_shared;
    const bool wide_down = D > 1024;
    const int bn_down = wide_down ? 256 : 128;
    uint8_t *xq = ws + A.xq, *hq = ws + A.hq, *sxq = ws + A.sxq, *shq = ws + A.shq;
    float *xs = reinterpret_cast<float *>(ws + A.xs), *hsc = reinterpret_cast<float *>(ws + A.hsc);
    float *sxs = reinterpret_cast<float *>(ws + A.sxs), *shs = reinterpret_cast<float *>(ws + A.shs);
    float *hf = reinterpret_cast<float *>(ws + A.hf), *shf = reinterpret_cast<float *>(ws + A.shf);
    cudaError_t err;

    // GEMM1, routed: hf = silu(xq Wg^T) * (xq Wu^T), fp32
    {
        CUtensorMap mA, mG, mU;
        SwapMaps sw;
        if (!make_map_u8(&mA, xq, (uint64_t)R, (uint64_t)D, kTileM) ||
            !make_map_u8(&mG, w.gate, (uint64_t)E * F, (uint64_t)D, 128) ||
            !make_map_u8(&mU, w.up, (uint64_t)E * F, (uint64_t)D, 128) ||
            !make_map_u8(&sw.w0, w.gate, (uint64_t)E * F, (uint64_t)D, kTileM) ||
            !make_map_u8(&sw.w1, w.up, (uint64_t)E * F, (uint64_t)D, kTileM) ||
            !make_map_u8(&sw.t, xq, (uint64_t)R, (uint64_t)D, kSwapBoxRows))
            return cudaErrorInvalidValue;
        TcParams p{};
        p.seg_off = seg;
        p.mtile = mtile;
        p.nseg = E;
        p.K = D;
        p.n_tiles = (F + 127) / 128;
        p.N_valid = F;
        p.b_seg_rows = F;
        p.out = hf;
        p.ld_out = F;
        p.status = status;
        p.aux = aux;
        p.a_scale = xs;
        p.b_scale0 = w.gate_s;
        p.b_scale1 = w.up_s;
        p.swap_tails = 1;
        const long long units =
            mt2_bound * p.n_tiles + 8LL * E * ((F + kSwapFeat - 1) / kSwapFeat);
        err = launch_tc_pair<128, 2, EPI_SWIGLU_F32, 5, true>(mA, mG, mU, p, units, stream, &sw);
        if (err != cudaSuccess)
            return err;
    }
    err = launch_quantize_e4m3_act(R, F, hf, true, hq, hsc, seg + E, stream);
    if (err == cudaSuccess)
        err = record_stage(ev, 3, stream);
    if (err != cudaSuccess)
        return err;
    // GEMM2, routed: z = hq Wd^T (or w * ... into y)
    {
        CUtensorMap mA, mB;
        SwapMaps sw;
        if (!make_map_u8(&mA, hq, (uint64_t)R, (uint64_t)F, kTileM) ||
            !make_map_u8(&mB, w.down, (uint64_t)E * D, (uint64_t)F, (uint32_t)(bn_down / 2)) ||
            !make_map_u8(&sw.w0, w.down, (uint64_t)E * D, (uint64_t)F, kTileM) ||
            !make_map_u8(&sw.t, hq, (uint64_t)R, (uint64_t)F, kSwapBoxRows))
            return cudaErrorInvalidValue;
        sw.w1 = sw.w0;
        TcParams p{};
        p.seg_off = seg;
        p.mtile = mtile;
        p.nseg = E;
        p.K = F;
        p.n_tiles = (D + bn_down - 1) / bn_down;
        p.N_valid = D;
        p.b_seg_rows = D;
        p.out = ws + L.z;
        p.ld_out = D;
        p.status = status;
        p.a_scale = hsc;
        p.b_scale0 = w.down_s;
        p.b_scale1 = w.down_s;
        p.swap_tails = 1;
        const long long units =
            mt2_bound * p.n_tiles + 8LL * E * ((D + kSwapFeat - 1) / kSwapFeat);
        if (plan.direct_y) {
            p.out = y;
            p.row_tok = reinterpret_cast<const int32_t *>(ws + L.row_tok);
            p.row_w = reinterpret_cast<const float *>(ws + L.row_w);
            err = wide_down
                      ? launch_tc_pair<256, 1, EPI_BF16_Y, 5, true>(mA, mB, mB, p, units, stream, &sw)
                      : launch_tc_pair<128, 1, EPI_BF16_Y, 6, true>(mA, mB, mB, p, units, stream, &sw);
        } else {
            err = wide_down
                      ? launch_tc_pair<256, 1, EPI_BF16, 5, true>(mA, mB, mB, p, units, stream, &sw)
                      : launch_tc_pair<128, 1, EPI_BF16, 6, true>(mA, mB, mB, p, units, stream, &sw);
        }
        if (err == cudaSuccess)
            err = record_stage(ev, 4, stream);
        if (err != cudaSuccess)
            return err;
    }
    // GEMM1, shared expert: shf = silu(sxq Wsg^T) * (sxq Wsu^T), fp32
    if (shared) {
        CUtensorMap mA, mG, mU;
        if (!make_map_u8(&mA, sxq, (uint64_t)T, (uint64_t)D, kTileM) ||
            !make_map_u8(&mG, w.sgate, (uint64_t)S, (uint64_t)D, 128) ||
            !make_map_u8(&mU, w.sup, (uint64_t)S, (uint64_t)D, 128))
            return cudaErrorInvalidValue;
        TcParams p{};
        p.nseg = 1;
        p.dense_rows = T;
        p.K = D;
        p.n_tiles = (S + 127) / 128;
        p.N_valid = S;
        p.out = shf;
        p.ld_out = S;
        p.status = status;
        p.a_scale = sxs;
        p.b_scale0 = w.sgate_s;
        p.b_scale1 = w.sup_s;
        err = pair_shared ? launch_tc_pair<128, 2, EPI_SWIGLU_F32, 5, true>(
                                mA, mG, mU, p, mt2_s * p.n_tiles, stream)
                          : launch_tc<128, 2, EPI_SWIGLU_F32, 4, true>(mA, mG, mU, p,
                                                                       mt_s * p.n_tiles, stream);
        if (err != cudaSuccess)
            return err;
    }
    if (shared)
        err = launch_quantize_e4m3_act(T, S, shf, true, shq, shs, nullptr, stream);
    if (err == cudaSuccess)
        err = record_stage(ev, 5, stream);
    if (err != cudaSuccess)
        return err;
    // GEMM2, shared expert: zs = shq Wsd^T (bf16: the combine adds it)
    if (shared) {
        CUtensorMap mA, mB;
        if (!make_map_u8(&mA, shq, (uint64_t)T, (uint64_t)S, kTileM) ||
            !make_map_u8(&mB, w.sdown, (uint64_t)D, (uint64_t)S,
                         (uint32_t)(pair_shared ? bn_down / 2 : bn_down)))
            return cudaErrorInvalidValue;
        TcParams p{};
        p.nseg = 1;
        p.dense_rows = T;
        p.K = S;
        p.n_tiles = (D + bn_down - 1) / bn_down;
        p.N_valid = D;
        p.out = ws + L.zs;
        p.ld_out = D;
        p.status = status;
        p.a_scale = shs;
        p.b_scale0 = w.sdown_s;
        p.b_scale1 = w.sdown_s;
        if (pair_shared)
            err = wide_down ? launch_tc_pair<256, 1, EPI_BF16, 5, true>(mA, mB, mB, p,
                                                                        mt2_s * p.n_tiles, stream)
                            : launch_tc_pair<128, 1, EPI_BF16, 6, true>(mA, mB, mB, p,
                                                                        mt2_s * p.n_tiles, stream);
        else
            err = wide_down ? launch_tc<256, 1, EPI_BF16, 4, true>(mA, mB, mB, p,
                                                                   mt_s * p.n_tiles, stream)
                            : launch_tc<128, 1, EPI_BF16, 6, true>(mA, mB, mB, p,
                                                                   mt_s * p.n_tiles, stream);
    }
    if (err == cudaSuccess)
        err = record_stage(ev, 6, stream);
    return err;
}

}  // namespace

cudaError_t launch_experts_w8a8(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                                const void *x, const ExpertW8 &w, void *y, const AuxArgs &aux,
                                cudaStream_t stream, cudaEvent_t *ev)
{
    const int D = c.d_model, F = c.d_expert, S = c.d_shared, E = c.n_experts, T = c.T;
    const A8Layout A = a8_layout_of(c, L);
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    const int32_t *seg = reinterpret_cast<const int32_t *>(ws + L.seg_off);
    const int32_t *mtile = reinterpret_cast<const int32_t *>(ws + L.mtile);
    const long long R = L.R_max;
    const long long mt_bound = R / kTileM + E;
    const long long mt_s = (T + kTileM - 1) / kTileM;
    const LaunchPlan plan = plan_of(c);
    const bool shared = S > 0;
    // the shared expert always runs as the second problem of the routed
    // launches; its down projection is cut into fp32 pieces exactly when the
    // combine expects them (shared_down_splits)
    const int zsplit = shared ? shared_down_splits(c) : 1;
    const bool wide_down = D > 1024;
    const int bn_down = wide_down ? 256 : 128;
    uint8_t *xq = ws + A.xq, *hq = ws + A.hq, *sxq = ws + A.sxq, *shq = ws + A.shq;
    float *xs = reinterpret_cast<float *>(ws + A.xs), *hsc = reinterpret_cast<float *>(ws + A.hsc);
    float *sxs = reinterpret_cast<float *>(ws + A.sxs), *shs = reinterpret_cast<float *>(ws + A.shs);
    float *hf = reinterpret_cast<float *>(ws + A.hf), *shf = reinterpret_cast<float *>(ws + A.shf);
    cudaError_t err;

    // few rows per expert: weights as the 128-row MMA operand instead
    if (w8a8_swap(c))
        return launch_experts_w8a8_swap(c, L, ws, w, y, aux, stream, ev);
    // many rows: CTA pairs
    if (plan_of(c).pair_routed)
        return experts_w8a8_pairs(c, L, ws, w, y, aux, stream, ev);
    // the token rows' codes and scales were written before the dispatch
    // (sxq, sxs: one per token) and gathered by it into expert order (xq, xs)
    (void)x;
    // GEMM1: hf = silu(xq Wg^T) * (xq Wu^T), fp32 (+ shf from the shared expert)
    {
        CUtensorMap mA, mG, mU;
        if (!make_map_u8(&mA, xq, (uint64_t)R, (uint64_t)D, kTileM) ||
            !make_map_u8(&mG, w.gate, (uint64_t)E * F, (uint64_t)D, 128) ||
            !make_map_u8(&mU, w.up, (uint64_t)E * F, (uint64_t)D, 128))
            return cudaErrorInvalidValue;
        TcParams p{};
        p.seg_off = seg;
        p.mtile = mtile;
        p.nseg = E;
        p.K = D;
        p.n_tiles = (F + 127) / 128;
        p.N_valid = F;
        p.b_seg_rows = F;
        p.out = hf;
        p.ld_out = F;
        p.status = status;
        p.aux = aux;
        p.a_scale = xs;
        p.b_scale0 = w.gate_s;
        p.b_scale1 = w.up_s;
        SecondMaps sm;
        if (shared) {
            if (!make_map_u8(&sm.a, sxq, (uint64_t)T, (uint64_t)D, kTileM) ||
                !make_map_u8(&sm.b0, w.sgate, (uint64_t)S, (uint64_t)D, 128) ||
                !make_map_u8(&sm.b1, w.sup, (uint64_t)S, (uint64_t)D, 128))
                return cudaErrorInvalidValue;
            p.sh_n_tiles = (S + 127) / 128;
            p.sh_tiles = (int)(mt_s * p.sh_n_tiles);
            p.sh_rows = T;
            p.sh_K = D;
            p.sh_N_valid = S;
            p.sh_out = shf;
            p.sh_ld_out = S;
            p.sh_a_scale = sxs;
            p.sh_b_scale0 = w.sgate_s;
            p.sh_b_scale1 = w.sup_s;
        }
        err = launch_tc<128, 2, EPI_SWIGLU_F32, 4, true>(mA, mG, mU, p, mt_bound * p.n_tiles,
                                                         stream, shared ? &sm : nullptr);
        if (err == cudaSuccess)
            err = launch_quantize_e4m3_act(R, F, hf, true, hq, hsc, seg + E, stream);
        if (err == cudaSuccess && shared)
            err = launch_quantize_e4m3_act(T, S, shf, true, shq, shs, nullptr, stream);
        if (err == cudaSuccess)
            err = record_stage(ev, 3, stream);
        if (err != cudaSuccess)
            return err;
    }
    // GEMM2: z = hq Wd^T (or w * ... into y), (+ zs from the shared expert)
    {
        CUtensorMap mA, mB;
        if (!make_map_u8(&mA, hq, (uint64_t)R, (uint64_t)F, kTileM) ||
            !make_map_u8(&mB, w.down, (uint64_t)E * D, (uint64_t)F, (uint32_t)bn_down))
            return cudaErrorInvalidValue;
        TcParams p{};
        p.seg_off = seg;
        p.mtile = mtile;
        p.nseg = E;
        p.K = F;
        p.n_tiles = (D + bn_down - 1) / bn_down;
        p.N_valid = D;
        p.b_seg_rows = D;
        p.out = ws + L.z;
        p.ld_out = D;
        p.status = status;
        p.a_scale = hsc;
        p.b_scale0 = w.down_s;
        p.b_scale1 = w.down_s;
        SecondMaps sm;
        if (shared) {
            if (!make_map_u8(&sm.a, shq, (uint64_t)T, (uint64_t)S, kTileM) ||
                !make_map_u8(&sm.b0, w.sdown, (uint64_t)D, (uint64_t)S, (uint32_t)bn_down))
                return cudaErrorInvalidValue;
            sm.b1 = sm.b0;
            p.sh_n_tiles = p.n_tiles;
            p.sh_tiles = (int)(mt_s * p.sh_n_tiles);
            p.sh_rows = T;
            p.sh_K = S;
            p.sh_N_valid = D;
            p.sh_out = ws + L.zs;
            p.sh_ld_out = D;
            p.sh_ksplit = zsplit;
            p.part_stride = (long long)T * D;
            p.sh_a_scale = shs;
            p.sh_b_scale0 = w.sdown_s;
            p.sh_b_scale1 = w.sdown_s;
        }
        const SecondMaps *second = shared ? &sm : nullptr;
        const long long tiles = mt_bound * p.n_tiles;
        if (plan.direct_y) {
            p.out = y;
            p.row_tok = reinterpret_cast<const int32_t *>(ws + L.row_tok);
            p.row_w = reinterpret_cast<const float *>(ws + L.row_w);
            err = wide_down ? launch_tc<256, 1, EPI_BF16_Y, 4, true>(mA, mB, mB, p, tiles, stream)
                            : launch_tc<128, 1, EPI_BF16_Y, 6, true>(mA, mB, mB, p, tiles, stream);
        } else {
            err = wide_down
                      ? launch_tc<256, 1, EPI_BF16, 4, true>(mA, mB, mB, p, tiles, stream, second)
                      : launch_tc<128, 1, EPI_BF16, 6, true>(mA, mB, mB, p, tiles, stream, second);
        }
        if (err == cudaSuccess)
            err = record_stage(ev, 4, stream);
        if (err == cudaSuccess)
            err = record_stage(ev, 5, stream);
        if (err == cudaSuccess)
            err = record_stage(ev, 6, stream);
    }
    return err;
}

}  // namespace moe

extern "C" moe_status moe_timeline_clear(void)
{
    if (!moe::kTimeline)
        return MOE_ERR_UNSUPPORTED;
    static const unsigned long long zero[2 * 4096 * 8] = {};
    return cudaMemcpyToSymbol(moe::g_timeline, zero, sizeof(zero)) == cudaSuccess &&
                   moe::dispatch_timeline_clear() == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
}

extern "C" moe_status moe_timeline_read(uint64_t *host_words, int64_t n_words)
{
    if (!moe::kTimeline)
        return MOE_ERR_UNSUPPORTED;
    if (!host_words || n_words < 0 || n_words > MOE_TIMELINE_WORDS)
        return MOE_ERR_INVALID_ARG;
    const int64_t g = std::min<int64_t>(n_words, moe::kTimelineGemmWords);
    if (g > 0 && cudaMemcpyFromSymbol(host_words, moe::g_timeline, (size_t)g * 8) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (n_words > g &&
        moe::dispatch_timeline_copy(host_words + g, (size_t)(n_words - g)) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
