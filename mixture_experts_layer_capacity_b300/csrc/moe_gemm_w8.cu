// moe_gemm_w8.cu -- the SwiGLU expert GEMMs with e4m3 (FP8) weights for
// decode-sized batches, and the row-wise e4m3 quantizer.
//
// At small T the expert GEMMs stream weights from HBM and do ~2 FLOPs per
// weight ("Mixture of Experts: More Parameters, Same FLOPs", 'What experts
// cost at serving time': decoding is memory-bound, and the same page sizes
// serving memory at 8 bits per weight).  One byte per weight halves the
// bytes.  Each weight row (output feature) r carries a fp32 scale s_r:
//   W[r][c] = decode_e4m3(q[r][c]) * s_r,
// so a dot product over c is s_r * sum_c decode(q[r][c]) * x_c: the scale is
// applied once, in the epilogue.
//
// Design (one CTA per SM, persistent over a unit list built on the device):
//   - roles are swapped relative to the bf16 kernels: the weights are the
//     MMA's A operand (M = 128 output features per tile) and the token rows
//     are B (N = 16 or 32 rows, one unit covers up to 32 rows of a segment), so
//     a decode batch with a few rows per expert does not pad A to 128 rows;
//   - warp 0: TMA producer: per 128-wide reduction step, two 128-row e4m3
//     weight tiles (128-byte rows, 128-byte swizzle) and the token rows in
//     16-row boxes (two 64-element halves, 128-byte swizzle, K-major) into a
//     5-stage shared-memory ring (160 KB of weights in flight per SM);
//   - warps 6-13: converters, two groups of four taking alternate reduction
//     steps (so that two steps convert at once): each thread owns one weight
//     row of a tile (its
//     TMEM lane), reads its 64 e4m3 bytes, converts them to f16 (one cvt per
//     pair; every e4m3 value is an f16 value) and writes them into TMEM with
//     tcgen05.st, where the MMA reads A directly (no second pass through
//     shared memory).  The MMA takes f16 A and f16 B, so the activations are
//     f16 too: GEMM1 converts its bf16 token rows to f16 in place in shared
//     memory (the converters, saturating at +-65504) and writes h in f16,
//     which GEMM2 reads as is.  (An exact e4m3 -> bf16 conversion costs
//     several integer operations per pair and left the kernel ALU-bound.)
//   - warp 1: tcgen05.mma kind::f16 (f16 inputs, fp32 accumulate), A from
//     TMEM, B from shared memory, into one of two TMEM accumulators per tile;
//   - warps 2-5: epilogue: TMEM lane = output feature, column = token row;
//     scale, SiLU * up (GEMM1, f16 h), bf16 z or y (GEMM2); 32 consecutive
//     features per warp and token row.
// GEMM1 units hold the gate and up tiles of the same 128 features; GEMM2
// units hold 256 consecutive output features.
// A8 form (E4M3 token rows too, moe_forward_w8a8 at decode sizes): both
// operands are E4M3, so the MMA (kind::f8f6f4, K = 32) reads the weight
// tiles straight from the shared-memory ring as its A operand: no
// converters, no TMEM staging of A.  The token rows arrive as codes (one
// 16-row box of 128-byte rows per 16 rows and reduction step), a 6-stage
// ring of 36 KB stages; the epilogue scales each accumulator by the weight
// row's and the token row's scales, and GEMM1 writes h in fp32 for the row
// quantizer.  A second, dense problem (the
// shared expert) may precede the grouped one in the unit list, as in the
// bf16 kernels.  Every wait is bounded; on timeout the CTA records
// MOE_DEVICE_PIPELINE_TIMEOUT, drains its own copies and MMAs, frees TMEM and
// returns.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

enum { W8_SWIGLU = 0, W8_BF16 = 1, W8_BF16_Y = 2 };

constexpr int kW8Threads = 448;  // warps 0 TMA, 1 MMA, 2-5 epilogue, 6-13 converters
constexpr int kW8Tok = 32;       // most token rows per unit (MMA N)
constexpr int kW8K = 128;        // reduction elements per stage
constexpr int kW8Stages = 5;     // shared-memory ring
constexpr int kW8AStages = 3;    // converted weight stages in TMEM
constexpr int kW8Rows = 128;     // weight rows per A tile (MMA M)
constexpr int kW8FP8Bytes = kW8Rows * kW8K;                        // 16 KB per A tile
constexpr int kW8BHalf = kW8Tok * 128;                             // token rows x 64 elements
constexpr int kW8DCols = 2 * kW8Tok;                               // accumulator buffer
constexpr int kW8ACols = kW8K / 2;                                 // TMEM columns of an A tile
constexpr int kW8ACol0 = 2 * kW8DCols;                             // first A column
constexpr int kW8TmemCols = 512;
constexpr int kW8TableInts = 2 * (kMaxExperts + 1);
constexpr uint64_t kW8WaitNs = 2000000000ull;
constexpr uint64_t kW8DrainNs = 200000000ull;
static_assert(kW8ACol0 + kW8AStages * 2 * kW8ACols <= kW8TmemCols, "TMEM columns");
static_assert(kW8BHalf % 1024 == 0, "1024-byte swizzle atoms");

// The shared-memory ring of each form: bf16 token rows (two 64-element
// halves per stage) or E4M3 token rows (one 128-byte half, A8).
template <bool A8>
struct W8Ring {
    static constexpr int STAGES = A8 ? 6 : kW8Stages;
    static constexpr int B_BYTES = A8 ? kW8BHalf : 2 * kW8BHalf;
    static constexpr int STAGE_BYTES = 2 * kW8FP8Bytes + B_BYTES;
    static constexpr int BARS = 2 * STAGES + 2 * kW8AStages + 4 + 1;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 512 + kW8TableInts * 4 + 1024;
    static_assert(STAGE_BYTES % 1024 == 0, "1024-byte swizzle atoms");
    static_assert(BARS * 8 + 8 <= 512, "barrier area");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct W8Problem {
    const int32_t *seg_off;  // [nseg+1] first row of each segment; null = dense
    int nseg, rows;          // rows: dense row count
    int K;                   // reduction length (multiple of 64)
    int feat;                // output features per segment
    int w_seg_rows;          // weight rows per segment in the maps (0 dense)
    int ftiles;              // feature tiles (128 features for SwiGLU, 256 otherwise)
    int ksplit;              // reduction pieces, fp32 partial outputs (1 = none)
    const float *s0, *s1;    // per weight row scales: gate/up, or down/unused
    const float *tscale;     // A8: per token row scales (rows of the B operand)
    void *out;
    long long ld_out;        // output row stride, elements
    long long part_stride;   // ksplit > 1: elements between the pieces' outputs
};

struct W8Params {
    W8Problem pr[2];         // pr[0]: dense second problem (its units first); pr[1]: main
    const int32_t *row_tok;  // W8_BF16_Y: token of each row
    const float *row_w;      // W8_BF16_Y: gate weight of each row
    int32_t *status;
    AuxArgs aux;
};

struct W8Unit {
    int prob, seg, row0, n, f, ks, kb0, kb1;
};

// Units of a problem: token tiles x feature tiles x reduction pieces.
__device__ __forceinline__ int w8_units(const W8Problem &pr, const int *s_tt)
{
    const int tt = pr.seg_off ? s_tt[pr.nseg] : (pr.rows + kW8Tok - 1) / kW8Tok;
    return tt * pr.ftiles * pr.ksplit;
}

// Unit u of the list: pr[0]'s units, then pr[1]'s.  Within a problem:
// segment-major, then feature tile, then token tile, then reduction piece.
__device__ __forceinline__ W8Unit w8_unit(const W8Params &p, const int *s_seg, const int *s_tt,
                                          int u, int n0)
{
    W8Unit w;
    w.prob = u < n0 ? 0 : 1;
    const W8Problem &pr = p.pr[w.prob];
    const int v = u < n0 ? u : u - n0;
    const int g = v / pr.ksplit;
    w.ks = v - g * pr.ksplit;
    if (!pr.seg_off) {
        const int tt = (pr.rows + kW8Tok - 1) / kW8Tok;
        w.f = g / tt;
        const int m = g - w.f * tt;
        w.seg = 0;
        w.row0 = m * kW8Tok;
        w.n = min(kW8Tok, pr.rows - w.row0);
    } else {
        int lo = 0, hi = pr.nseg;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_tt[mid] * pr.ftiles <= g)
                lo = mid;
            else
                hi = mid;
        }
        const int tt_e = s_tt[lo + 1] - s_tt[lo];
        const int local = g - s_tt[lo] * pr.ftiles;
        w.f = local / tt_e;
        const int m = local - w.f * tt_e;
        w.seg = lo;
        w.row0 = s_seg[lo] + m * kW8Tok;
        w.n = min(kW8Tok, s_seg[lo + 1] - w.row0);
    }
    const int nk = (pr.K + kW8K - 1) / kW8K;
    w.kb0 = w.ks * nk / pr.ksplit;
    w.kb1 = (w.ks + 1) * nk / pr.ksplit;
    return w;
}

// Two e4m3 values (low byte first) to two f16 (low half first), exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)two));
    return h;
}

// Two bf16 (low half first) to two f16, round to nearest, saturating at
// +-65504.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w)
{
    uint32_t d;
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Instruction descriptor, kind::f16 with f16 A and B (format 0), fp32
// accumulator, both K-major: the bf16 descriptor's layout with A/B format 0.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ int balanced_w8(int n, int w)
{
    if (n <= 0)
        return w;
    const int rounds = (n + w - 1) / w;
    return (n + rounds - 1) / rounds;
}

template <int EPI, bool A8>
__global__ void __launch_bounds__(kW8Threads, 1)
    w8_gemm_kernel(const __grid_constant__ CUtensorMap w00, const __grid_constant__ CUtensorMap w01,
                   const __grid_constant__ CUtensorMap b0, const __grid_constant__ CUtensorMap w10,
                   const __grid_constant__ CUtensorMap w11, const __grid_constant__ CUtensorMap b1,
                   const W8Params p)
{
    using RG = W8Ring<A8>;
    extern __shared__ uint8_t smem_raw[];
    // the layout below must fit the shared memory this launch received
    if (dynamic_smem_bytes() < (uint32_t)RG::SMEM_BYTES) {
        if (threadIdx.x == 0)
            set_status(p.status, MOE_DEVICE_LAUNCH_MISMATCH);
        return;
    }
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + RG::STAGES * RG::STAGE_BYTES);
    uint64_t *full = bars;
    uint64_t *empty = full + RG::STAGES;
    uint64_t *afull = empty + RG::STAGES;
    uint64_t *aempty = afull + kW8AStages;
    uint64_t *tfull = aempty + kW8AStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *mma_done = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *tables = reinterpret_cast<int *>(smem + RG::STAGES * RG::STAGE_BYTES + 512);
    int *s_seg = tables;                    // [nseg+1] segment offsets of pr[1]
    int *s_tt = tables + kMaxExperts + 1;   // [nseg+1] prefix of 64-row token tiles

    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RG::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < kW8AStages; ++s) {
            mbar_init(&afull[s], 4 * 32);
            mbar_init(&aempty[s], 1);
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
        tma_prefetch_desc(&w10);
        tma_prefetch_desc(&w11);
        tma_prefetch_desc(&b1);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kW8TmemCols);
        tmem_relinquish();
    }
    griddep_wait();
    griddep_launch_dependents();
    const bool failed = *(volatile const int32_t *)p.status != 0;
    const W8Problem &pg = p.pr[1];
    if (pg.seg_off && !failed) {
        for (int i = threadIdx.x; i <= pg.nseg; i += blockDim.x)
            s_seg[i] = pg.seg_off[i];
    }
    __syncthreads();
    if (pg.seg_off && !failed && warp == 0) {
        int carry = 0;
        for (int e0 = 0; e0 < pg.nseg; e0 += 32) {
            const int e = e0 + lane;
            const int v = e < pg.nseg ? (s_seg[e + 1] - s_seg[e] + kW8Tok - 1) / kW8Tok : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += n;
            }
            if (e < pg.nseg)
                s_tt[e + 1] = carry + incl;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0)
            s_tt[0] = 0;
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    const int n0 = failed ? 0 : w8_units(p.pr[0], s_tt);
    const int n_all = failed ? 0 : n0 + w8_units(p.pr[1], s_tt);
    const int G = balanced_w8(n_all, (int)gridDim.x);
    const int nunits = (int)blockIdx.x < G ? n_all : 0;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int s = 0;
            uint32_t ph = 0;
            long long fills = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < nunits && ok; u += G) {
                const W8Unit w = w8_unit(p, s_seg, s_tt, u, n0);
                const W8Problem &pr = p.pr[w.prob];
                const CUtensorMap *mw0 = w.prob ? &w10 : &w00;
                const CUtensorMap *mw1 = w.prob ? &w11 : &w01;
                const CUtensorMap *mb = w.prob ? &b1 : &b0;
                const int fr = w.f * (EPI == W8_SWIGLU ? kW8Rows : 2 * kW8Rows);
                const int wrow = w.seg * pr.w_seg_rows + fr;
                const int nb = (w.n + 15) / 16;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, kW8WaitNs)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = smem + s * RG::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[s],
                                          2 * kW8FP8Bytes + (A8 ? 1 : 2) * nb * 16 * 128);
                    tma_load_2d(st, mw0, &full[s], kb * kW8K, wrow);
                    if (EPI == W8_SWIGLU)
                        tma_load_2d(st + kW8FP8Bytes, mw1, &full[s], kb * kW8K, wrow);
                    else
                        tma_load_2d(st + kW8FP8Bytes, mw0, &full[s], kb * kW8K, wrow + kW8Rows);
                    // reduction elements past K (a last half block) read as zero;
                    // E4M3 token rows: one 128-byte box row per token row
                    for (int h = 0; h < (A8 ? 1 : 2); ++h)
                        for (int j = 0; j < nb; ++j)
                            tma_load_2d(st + 2 * kW8FP8Bytes + h * kW8BHalf + j * 16 * 128, mb,
                                        &full[s], kb * kW8K + h * 64, w.row0 + 16 * j);
                    ++fills;
                    if (++s == RG::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
                const long long first = fills > RG::STAGES ? fills - RG::STAGES : 0;
                for (long long f = first; f < fills; ++f)
                    mbar_wait(&full[f % RG::STAGES], (uint32_t)((f / RG::STAGES) & 1), nullptr,
                              kW8DrainNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int s = 0, sa = 0;
            uint32_t ph = 0, aph = 0, b = 0, tph = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < nunits && ok; u += G) {
                const W8Unit w = w8_unit(p, s_seg, s_tt, u, n0);
                const int nb = (w.n + 15) / 16;
                const uint32_t idesc =
                    A8 ? idesc_e4m3_f32(kW8Rows, 16 * nb) : idesc_f16_f32(kW8Rows, 16 * nb);
                if (!mbar_wait(&tempty[b], tph ^ 1u, abort_flag, kW8WaitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d0 = tmem_base + b * kW8DCols;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if ((!A8 && !mbar_wait(&afull[sa], aph, abort_flag, kW8WaitNs)) ||
                        !mbar_wait(&full[s], ph, abort_flag, kW8WaitNs)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t st = smem_u32(smem + s * RG::STAGE_BYTES);
                    const uint32_t sb = st + 2 * kW8FP8Bytes;
                    if constexpr (A8) {
                        // weights (A) and token rows (B) from the ring, both
                        // 128-byte rows of 128 codes: four K = 32 steps each
                        const uint64_t bdesc = sdesc_kmajor_sw128(sb);
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const uint64_t adesc = sdesc_kmajor_sw128(st + t * kW8FP8Bytes);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                umma_e4m3(d0 + t * kW8Tok, adesc + 2u * kk, bdesc + 2u * kk, idesc,
                                          (kb > w.kb0 || kk > 0) ? 1u : 0u);
                        }
                        umma_commit(&empty[s]);
                    } else {
                        const uint64_t bdesc[2] = {sdesc_kmajor_sw128(sb),
                                                   sdesc_kmajor_sw128(sb + kW8BHalf)};
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const uint32_t a =
                                tmem_base + kW8ACol0 + (uint32_t)(sa * 2 + t) * kW8ACols;
#pragma unroll
                            for (int kk = 0; kk < kW8K / 16; ++kk)
                                umma_bf16_ta(d0 + t * kW8Tok, a + kk * 8,
                                             bdesc[kk >> 2] + 2u * (kk & 3), idesc,
                                             (kb > w.kb0 || kk > 0) ? 1u : 0u);
                        }
                        umma_commit(&empty[s]);
                        umma_commit(&aempty[sa]);
                        if (++sa == kW8AStages) {
                            sa = 0;
                            aph ^= 1u;
                        }
                    }
                    if (++s == RG::STAGES) {
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
            umma_commit(mma_done);
            mbar_wait(mma_done, 0, nullptr, kW8DrainNs);
        }
    } else if (warp >= 6) {
        // ---------------------------------------------------- converters
        // (none in the A8 form: the MMA reads the E4M3 weights directly)
        if constexpr (!A8) {
        // group grp converts the reduction steps i with i % 2 == grp (i counts
        // this CTA's steps over all its units)
        const int grp = (warp - 6) >> 2;
        const int q = warp & 3;
        const int r = q * 32 + lane;  // weight row within each A tile = TMEM lane
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        long long i = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < nunits && ok; u += G) {
            const W8Unit w = w8_unit(p, s_seg, s_tt, u, n0);
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++i) {
                if ((int)(i & 1) != grp)
                    continue;
                const int s = (int)(i % RG::STAGES), sa = (int)(i % kW8AStages);
                const uint32_t ph = (uint32_t)((i / RG::STAGES) & 1);
                const uint32_t aph = (uint32_t)((i / kW8AStages) & 1);
                if (!mbar_wait(&full[s], ph, abort_flag, kW8WaitNs) ||
                    !mbar_wait(&aempty[sa], aph ^ 1u, abort_flag, kW8WaitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint8_t *st = smem + s * RG::STAGE_BYTES;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    // row r's 16-byte chunk c sits at chunk c ^ (r & 7)
                    // (128-byte swizzle of the TMA box)
                    const uint8_t *row = st + t * kW8FP8Bytes + r * 128;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v[32];
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const int c = hh * 4 + c4;
                            const uint4 qv =
                                *reinterpret_cast<const uint4 *>(row + ((c ^ (r & 7)) << 4));
                            v[8 * c4 + 0] = e4m3x2_to_f16x2(qv.x);
                            v[8 * c4 + 1] = e4m3x2_to_f16x2(qv.x >> 16);
                            v[8 * c4 + 2] = e4m3x2_to_f16x2(qv.y);
                            v[8 * c4 + 3] = e4m3x2_to_f16x2(qv.y >> 16);
                            v[8 * c4 + 4] = e4m3x2_to_f16x2(qv.z);
                            v[8 * c4 + 5] = e4m3x2_to_f16x2(qv.z >> 16);
                            v[8 * c4 + 6] = e4m3x2_to_f16x2(qv.w);
                            v[8 * c4 + 7] = e4m3x2_to_f16x2(qv.w >> 16);
                        }
                        tmem_st32(tmem_base + lanes + kW8ACol0 +
                                      (uint32_t)(sa * 2 + t) * kW8ACols + hh * 32,
                                  v);
                    }
                }
                if constexpr (EPI == W8_SWIGLU) {
                    // GEMM1's token rows arrive as bf16: to f16 in place (element
                    // by element, so the swizzled layout is kept), then make the
                    // writes visible to the tensor cores' reads
                    const int nb = (w.n + 15) / 16;
                    const int tc = (warp - 6 - 4 * grp) * 32 + lane;
                    for (int h = 0; h < 2; ++h) {
                        uint4 *bt = reinterpret_cast<uint4 *>(smem + s * RG::STAGE_BYTES +
                                                              2 * kW8FP8Bytes + h * kW8BHalf);
                        for (int ci = tc; ci < nb * 16 * 8; ci += 128) {
                            uint4 x = bt[ci];
                            x.x = bf16x2_to_f16x2(x.x);
                            x.y = bf16x2_to_f16x2(x.y);
                            x.z = bf16x2_to_f16x2(x.z);
                            x.w = bf16x2_to_f16x2(x.w);
                            bt[ci] = x;
                        }
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive(&afull[sa]);
            }
        }
        if (!ok) {
            *abort_flag = 1;
            set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
        }
        }
    } else {
        // ---------------------------------------------------- epilogue
        if (p.aux.out && !failed && blockIdx.x == 0 && warp == 2)
            balance_loss_warp(p.aux);
        const int q = warp & 3;
        const int r = q * 32 + lane;  // output feature within the tile = TMEM lane
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        uint32_t b = 0, tph = 0;
        for (int u = blockIdx.x; u < nunits; u += G) {
            const W8Unit w = w8_unit(p, s_seg, s_tt, u, n0);
            const W8Problem &pr = p.pr[w.prob];
            if (!mbar_wait(&tfull[b], tph, abort_flag, kW8WaitNs)) {
                *abort_flag = 1;
                set_status(p.status, MOE_DEVICE_PIPELINE_TIMEOUT);
                break;
            }
            tc_fence_after_sync();
            const uint32_t tb = tmem_base + lanes + b * kW8DCols;
            const int ncol = 16 * ((w.n + 15) / 16);
            if constexpr (EPI == W8_SWIGLU) {
                const int f = w.f * kW8Rows + r;
                const bool fok = f < pr.feat;
                const float sg = fok ? pr.s0[(long long)w.seg * pr.w_seg_rows + f] : 0.f;
                const float su = fok ? pr.s1[(long long)w.seg * pr.w_seg_rows + f] : 0.f;
                for (int j0 = 0; j0 < ncol; j0 += 16) {
                    uint32_t gv[16], uv[16];
                    tmem_ld16(tb + j0, gv);
                    tmem_ld16(tb + kW8Tok + j0, uv);
                    tmem_wait_ld();
                    if (fok) {
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int j = j0 + jj;
                            if (j < w.n) {
                                const long long row = w.row0 + j;
                                if constexpr (A8) {
                                    // fp32 h for the row quantizer
                                    const float ts = __ldg(pr.tscale + row);
                                    const float g = __uint_as_float(gv[jj]) * (sg * ts);
                                    const float uu = __uint_as_float(uv[jj]) * (su * ts);
                                    static_cast<float *>(pr.out)[row * pr.ld_out + f] =
                                        silu_f32(g) * uu;
                                } else {
                                    const float g = __uint_as_float(gv[jj]) * sg;
                                    const float uu = __uint_as_float(uv[jj]) * su;
                                    const float hv =
                                        fminf(fmaxf(silu_f32(g) * uu, -65504.f), 65504.f);
                                    static_cast<__half *>(pr.out)[row * pr.ld_out + f] =
                                        __float2half_rn(hv);
                                }
                            }
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int t = 0; t < 2; ++t) {
                    const int f = w.f * 2 * kW8Rows + t * kW8Rows + r;
                    const bool fok = f < pr.feat;
                    const float sc = fok ? pr.s0[(long long)w.seg * pr.w_seg_rows + f] : 0.f;
                    for (int j0 = 0; j0 < ncol; j0 += 16) {
                        uint32_t v[16];
                        tmem_ld16(tb + t * kW8Tok + j0, v);
                        tmem_wait_ld();
                        if (!fok)
                            continue;
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) {
                            const int j = j0 + jj;
                            if (j >= w.n)
                                continue;
                            const long long row = w.row0 + j;
                            const float a = __uint_as_float(v[jj]) *
                                            (A8 ? sc * __ldg(pr.tscale + row) : sc);
                            if (pr.ksplit > 1) {
                                static_cast<float *>(pr.out)[w.ks * pr.part_stride +
                                                             row * pr.ld_out + f] = a;
                            } else if (EPI == W8_BF16_Y) {
                                const int tok = p.row_tok[row];
                                static_cast<__nv_bfloat16 *>(pr.out)[(long long)tok * pr.ld_out +
                                                                     f] =
                                    __float2bfloat16_rn(p.row_w[row] * a);
                            } else {
                                static_cast<__nv_bfloat16 *>(pr.out)[row * pr.ld_out + f] =
                                    __float2bfloat16_rn(a);
                            }
                        }
                    }
                }
            }
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
        tmem_dealloc(tmem_base, kW8TmemCols);
    }
}

template <int EPI, bool A8 = false>
cudaError_t launch_w8(const CUtensorMap (&m)[6], const W8Params &p, long long max_units,
                      cudaStream_t stream)
{
    using RG = W8Ring<A8>;
    auto kern = w8_gemm_kernel<EPI, A8>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    static DeviceOnce configured;
    if (configured.pending(dev)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   RG::SMEM_BYTES);
        if (err == cudaSuccess)
            err = prefer_max_shared_carveout(kern);
        if (err != cudaSuccess)
            return err;
        configured.done(dev);
    }
    const long long grid = std::min<long long>(max_units, sm_count());
    if (grid < 1)
        return cudaSuccess;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kW8Threads), (size_t)RG::SMEM_BYTES, stream,
                      m[0], m[1], m[2], m[3], m[4], m[5], p);
}

// Eight consecutive values of a row as fp32 (v-th group of eight).
__device__ __forceinline__ void load8(const __nv_bfloat16 *row, long long v, float (&f)[8])
{
    const uint4 x = reinterpret_cast<const uint4 *>(row)[v];
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&x);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ void load8(const float *row, long long v, float (&f)[8])
{
    const float4 a = reinterpret_cast<const float4 *>(row)[2 * v];
    const float4 b = reinterpret_cast<const float4 *>(row)[2 * v + 1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

// q[r][c] = e4m3(W[r][c] / s_r), s_r = max_c |W[r][c]| / 448 (1 for an
// all-zero row); fp32 division, round to nearest even, saturating to +-448.
// GROUP warps per row (1, 2, 4 or 8 of the block's 8; long rows take more
// warps, so that a few long rows still spread over many SMs), 8 columns per
// lane and step; the row maximum is combined over the group in shared
// memory (a maximum: the same value in any order).  TIN: bf16 (weights,
// token rows) or fp32 (hidden rows).  rows_dev non-null: only the first
// min(rows, *rows_dev) rows (a row count the previous kernel wrote).
template <typename TIN, int GROUP>
__global__ void __launch_bounds__(256)
    quantize_e4m3_kernel(long long rows, long long cols, const TIN *__restrict__ W,
                         uint8_t *__restrict__ q, float *__restrict__ scale,
                         const int32_t *__restrict__ rows_dev)
{
    constexpr int RPB = 8 / GROUP;   // rows per block and pass
    __shared__ float s_max[8];
    griddep_wait();   // the rows (and their count) come from the previous kernel
    if (rows_dev)
        rows = min(rows, (long long)*(volatile const int32_t *)rows_dev);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = warp / GROUP, gw = warp - slot * GROUP;
    const long long nv = cols / 8;
    const long long per_pass = (long long)gridDim.x * RPB;
    // the same number of passes for every thread of the block (barriers)
    const long long passes = (rows + per_pass - 1) / per_pass;
    for (long long it = 0; it < passes; ++it) {
        const long long r = it * per_pass + (long long)blockIdx.x * RPB + slot;
        const bool valid = r < rows;
        const TIN *src = W + (valid ? r : 0) * cols;
        float amax = 0.f;
        if (valid) {
#pragma unroll 4
            for (long long v = gw * 32 + lane; v < nv; v += GROUP * 32) {
                float f[8];
                load8(src, v, f);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    amax = fmaxf(amax, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
            }
        }
        amax = warp_max(amax);
        if constexpr (GROUP > 1) {
            if (lane == 0)
                s_max[warp] = amax;
            __syncthreads();
#pragma unroll
            for (int i = 0; i < GROUP; ++i)
                amax = fmaxf(amax, s_max[slot * GROUP + i]);
            __syncthreads();   // s_max is rewritten in the next pass
        }
        if (!valid)
            continue;
        const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        if (gw == 0 && lane == 0)
            scale[r] = s;
        uint2 *dst = reinterpret_cast<uint2 *>(q + r * cols);
#pragma unroll 4
        for (long long v = gw * 32 + lane; v < nv; v += GROUP * 32) {
            float f[8];
            load8(src, v, f);
            uint32_t word[2] = {0u, 0u};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t c0 = __nv_cvt_float_to_fp8(__fdiv_rn(f[2 * i], s), __NV_SATFINITE, __NV_E4M3);
                const uint32_t c1 = __nv_cvt_float_to_fp8(__fdiv_rn(f[2 * i + 1], s), __NV_SATFINITE, __NV_E4M3);
                word[i >> 1] |= (c0 | (c1 << 8)) << (16 * (i & 1));
            }
            dst[v] = make_uint2(word[0], word[1]);
        }
    }
}

// Warps per row for rows of `cols` values: at least two 8-value steps per
// lane, at most the block's 8 warps.
int quantize_group(long long cols)
{
    const long long steps = cols / (8 * 32);   // per warp
    return steps >= 16 ? 8 : steps >= 8 ? 4 : steps >= 4 ? 2 : 1;
}

template <typename TIN>
cudaError_t launch_quantize_t(long long rows, long long cols, const TIN *X, uint8_t *q,
                              float *scale, const int32_t *rows_dev, bool pdl,
                              cudaStream_t stream)
{
    const int group = quantize_group(cols);
    const long long rpb = 8 / group;
    const unsigned blocks = (unsigned)std::min<long long>((rows + rpb - 1) / rpb, 16LL * sm_count());
    auto kern = group == 8   ? quantize_e4m3_kernel<TIN, 8>
                : group == 4 ? quantize_e4m3_kernel<TIN, 4>
                : group == 2 ? quantize_e4m3_kernel<TIN, 2>
                             : quantize_e4m3_kernel<TIN, 1>;
    if (pdl)
        return launch_pdl(kern, dim3(blocks), dim3(256), 0, stream, rows, cols, X, q, scale,
                          rows_dev);
    kern<<<blocks, 256, 0, stream>>>(rows, cols, X, q, scale, rows_dev);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_e4m3(long long rows, long long cols, const void *W, uint8_t *q,
                                 float *scale, cudaStream_t stream)
{
    if (rows <= 0)
        return cudaSuccess;
    return launch_quantize_t(rows, cols, static_cast<const __nv_bfloat16 *>(W), q, scale,
                             nullptr, false, stream);
}

cudaError_t launch_quantize_e4m3_act(long long rows, long long cols, const void *X, bool fp32,
                                     uint8_t *q, float *scale, const int32_t *rows_dev,
                                     cudaStream_t stream)
{
    if (rows <= 0)
        return cudaSuccess;
    if (fp32)
        return launch_quantize_t(rows, cols, static_cast<const float *>(X), q, scale, rows_dev,
                                 true, stream);
    return launch_quantize_t(rows, cols, static_cast<const __nv_bfloat16 *>(X), q, scale,
                             rows_dev, true, stream);
}

cudaError_t launch_experts_w8(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                              const void *x, const ExpertW8 &w, void *y, const AuxArgs &aux,
                              cudaStream_t stream, cudaEvent_t *ev)
{
    const int D = c.d_model, F = c.d_expert, S = c.d_shared, E = c.n_experts, T = c.T;
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    const int32_t *seg = reinterpret_cast<const int32_t *>(ws + L.seg_off);
    void *xp = ws + L.x_perm, *h = ws + L.h, *z = ws + L.z;
    void *hs = ws + L.hs, *zs = ws + L.zs;
    const long long R = L.R_max;
    const long long tt_bound = R / kW8Tok + E;            // >= sum_e ceil(kept_e / 32)
    const long long tt_s = (T + kW8Tok - 1) / kW8Tok;
    const LaunchPlan plan = plan_of(c);
    cudaError_t err;

    // GEMM1: h = silu(x_perm W_gate^T) * (x_perm W_up^T); hs likewise from x
    {
        CUtensorMap m[6];
        W8Params p{};
        W8Problem &g = p.pr[1];
        g.seg_off = seg;
        g.nseg = E;
        g.K = D;
        g.feat = F;
        g.w_seg_rows = F;
        g.ftiles = (F + kW8Rows - 1) / kW8Rows;
        g.ksplit = 1;
        g.s0 = w.gate_s;
        g.s1 = w.up_s;
        g.out = h;
        g.ld_out = F;
        if (!make_map_u8(&m[3], w.gate, (uint64_t)E * F, (uint64_t)D, kW8Rows) ||
            !make_map_u8(&m[4], w.up, (uint64_t)E * F, (uint64_t)D, kW8Rows) ||
            !make_map(&m[5], xp, (uint64_t)R, (uint64_t)D, 16))
            return cudaErrorInvalidValue;
        W8Problem &sh = p.pr[0];
        sh.ftiles = 1;
        sh.ksplit = 1;
        sh.K = D;
        if (S > 0) {
            sh.rows = T;
            sh.feat = S;
            sh.ftiles = (S + kW8Rows - 1) / kW8Rows;
            sh.s0 = w.sgate_s;
            sh.s1 = w.sup_s;
            sh.out = hs;
            sh.ld_out = S;
            if (!make_map_u8(&m[0], w.sgate, (uint64_t)S, (uint64_t)D, kW8Rows) ||
                !make_map_u8(&m[1], w.sup, (uint64_t)S, (uint64_t)D, kW8Rows) ||
                !make_map(&m[2], x, (uint64_t)T, (uint64_t)D, 16))
                return cudaErrorInvalidValue;
        } else {
            m[0] = m[3];
            m[1] = m[4];
            m[2] = m[5];
        }
        p.status = status;
        p.aux = aux;
        const long long units = tt_bound * g.ftiles + (S > 0 ? tt_s * sh.ftiles : 0);
        err = launch_w8<W8_SWIGLU>(m, p, units, stream);
        if (err == cudaSuccess)
            err = record_stage(ev, 3, stream);
        if (err != cudaSuccess)
            return err;
    }
    // GEMM2: z = h W_down^T (or y directly); zs = hs Ws_down^T
    {
        CUtensorMap m[6];
        W8Params p{};
        W8Problem &g = p.pr[1];
        g.seg_off = seg;
        g.nseg = E;
        g.K = F;
        g.feat = D;
        g.w_seg_rows = D;
        g.ftiles = (D + 2 * kW8Rows - 1) / (2 * kW8Rows);
        g.ksplit = 1;
        g.s0 = w.down_s;
        g.out = plan.direct_y ? y : z;
        g.ld_out = D;
        if (!make_map_u8(&m[3], w.down, (uint64_t)E * D, (uint64_t)F, kW8Rows) ||
            !make_map(&m[5], h, (uint64_t)R, (uint64_t)F, 16))
            return cudaErrorInvalidValue;
        m[4] = m[3];
        W8Problem &sh = p.pr[0];
        sh.ftiles = 1;
        sh.ksplit = 1;
        sh.K = F;
        if (S > 0) {
            sh.rows = T;
            sh.K = S;
            sh.feat = D;
            sh.ftiles = g.ftiles;
            sh.ksplit = shared_down_splits(c);
            sh.s0 = w.sdown_s;
            sh.out = zs;
            sh.ld_out = D;
            sh.part_stride = (long long)T * D;
            if (!make_map_u8(&m[0], w.sdown, (uint64_t)D, (uint64_t)S, kW8Rows) ||
                !make_map(&m[2], hs, (uint64_t)T, (uint64_t)S, 16))
                return cudaErrorInvalidValue;
            m[1] = m[0];
        } else {
            m[0] = m[3];
            m[1] = m[4];
            m[2] = m[5];
        }
        p.status = status;
        p.aux.out = nullptr;
        const long long units = tt_bound * g.ftiles + (S > 0 ? tt_s * sh.ftiles * sh.ksplit : 0);
        if (plan.direct_y) {
            p.row_tok = reinterpret_cast<const int32_t *>(ws + L.row_tok);
            p.row_w = reinterpret_cast<const float *>(ws + L.row_w);
            err = launch_w8<W8_BF16_Y>(m, p, units, stream);
        } else {
            err = launch_w8<W8_BF16>(m, p, units, stream);
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

cudaError_t launch_experts_w8a8_swap(const moe_config &c, const WorkspaceLayout &L, uint8_t *ws,
                                     const ExpertW8 &w, void *y, const AuxArgs &aux,
                                     cudaStream_t stream, cudaEvent_t *ev)
{
    const int D = c.d_model, F = c.d_expert, S = c.d_shared, E = c.n_experts, T = c.T;
    const A8Layout A = a8_layout_of(c, L);
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    const int32_t *seg = reinterpret_cast<const int32_t *>(ws + L.seg_off);
    uint8_t *xq = ws + A.xq, *hq = ws + A.hq, *sxq = ws + A.sxq, *shq = ws + A.shq;
    const float *xs = reinterpret_cast<const float *>(ws + A.xs);
    const float *sxs = reinterpret_cast<const float *>(ws + A.sxs);
    float *hf = reinterpret_cast<float *>(ws + A.hf), *shf = reinterpret_cast<float *>(ws + A.shf);
    float *hsc = reinterpret_cast<float *>(ws + A.hsc), *shs = reinterpret_cast<float *>(ws + A.shs);
    const long long R = L.R_max;
    const long long tt_bound = R / kW8Tok + E;            // >= sum_e ceil(kept_e / 32)
    const long long tt_s = (T + kW8Tok - 1) / kW8Tok;
    const LaunchPlan plan = plan_of(c);
    cudaError_t err;

    // GEMM1: hf = silu(xq Wg^T) * (xq Wu^T) in fp32; shf likewise from the
    // token rows' codes; then both quantized row-wise
    {
        CUtensorMap m[6];
        W8Params p{};
        W8Problem &g = p.pr[1];
        g.seg_off = seg;
        g.nseg = E;
        g.K = D;
        g.feat = F;
        g.w_seg_rows = F;
        g.ftiles = (F + kW8Rows - 1) / kW8Rows;
        g.ksplit = 1;
        g.s0 = w.gate_s;
        g.s1 = w.up_s;
        g.tscale = xs;
        g.out = hf;
        g.ld_out = F;
        if (!make_map_u8(&m[3], w.gate, (uint64_t)E * F, (uint64_t)D, kW8Rows) ||
            !make_map_u8(&m[4], w.up, (uint64_t)E * F, (uint64_t)D, kW8Rows) ||
            !make_map_u8(&m[5], xq, (uint64_t)R, (uint64_t)D, 16))
            return cudaErrorInvalidValue;
        W8Problem &sh = p.pr[0];
        sh.ftiles = 1;
        sh.ksplit = 1;
        sh.K = D;
        if (S > 0) {
            sh.rows = T;
            sh.feat = S;
            sh.ftiles = (S + kW8Rows - 1) / kW8Rows;
            sh.s0 = w.sgate_s;
            sh.s1 = w.sup_s;
            sh.tscale = sxs;
            sh.out = shf;
            sh.ld_out = S;
            if (!make_map_u8(&m[0], w.sgate, (uint64_t)S, (uint64_t)D, kW8Rows) ||
                !make_map_u8(&m[1], w.sup, (uint64_t)S, (uint64_t)D, kW8Rows) ||
                !make_map_u8(&m[2], sxq, (uint64_t)T, (uint64_t)D, 16))
                return cudaErrorInvalidValue;
        } else {
            m[0] = m[3];
            m[1] = m[4];
            m[2] = m[5];
        }
        p.status = status;
        p.aux = aux;
        const long long units = tt_bound * g.ftiles + (S > 0 ? tt_s * sh.ftiles : 0);
        err = launch_w8<W8_SWIGLU, true>(m, p, units, stream);
        if (err == cudaSuccess)
            err = launch_quantize_e4m3_act(R, F, hf, true, hq, hsc, seg + E, stream);
        if (err == cudaSuccess && S > 0)
            err = launch_quantize_e4m3_act(T, S, shf, true, shq, shs, nullptr, stream);
        if (err == cudaSuccess)
            err = record_stage(ev, 3, stream);
        if (err != cudaSuccess)
            return err;
    }
    // GEMM2: z = hq Wd^T (or y directly); zs = shq Ws_down^T
    {
        CUtensorMap m[6];
        W8Params p{};
        W8Problem &g = p.pr[1];
        g.seg_off = seg;
        g.nseg = E;
        g.K = F;
        g.feat = D;
        g.w_seg_rows = D;
        g.ftiles = (D + 2 * kW8Rows - 1) / (2 * kW8Rows);
        g.ksplit = 1;
        g.s0 = w.down_s;
        g.tscale = hsc;
        g.out = plan.direct_y ? y : ws + L.z;
        g.ld_out = D;
        if (!make_map_u8(&m[3], w.down, (uint64_t)E * D, (uint64_t)F, kW8Rows) ||
            !make_map_u8(&m[5], hq, (uint64_t)R, (uint64_t)F, 16))
            return cudaErrorInvalidValue;
        m[4] = m[3];
        W8Problem &sh = p.pr[0];
        sh.ftiles = 1;
        sh.ksplit = 1;
        sh.K = F;
        if (S > 0) {
            sh.rows = T;
            sh.K = S;
            sh.feat = D;
            sh.ftiles = g.ftiles;
            sh.ksplit = shared_down_splits(c);
            sh.s0 = w.sdown_s;
            sh.tscale = shs;
            sh.out = ws + L.zs;
            sh.ld_out = D;
            sh.part_stride = (long long)T * D;
            if (!make_map_u8(&m[0], w.sdown, (uint64_t)D, (uint64_t)S, kW8Rows) ||
                !make_map_u8(&m[2], shq, (uint64_t)T, (uint64_t)S, 16))
                return cudaErrorInvalidValue;
            m[1] = m[0];
        } else {
            m[0] = m[3];
            m[1] = m[4];
            m[2] = m[5];
        }
        p.status = status;
        p.aux.out = nullptr;
        const long long units = tt_bound * g.ftiles + (S > 0 ? tt_s * sh.ftiles * sh.ksplit : 0);
        if (plan.direct_y) {
            p.row_tok = reinterpret_cast<const int32_t *>(ws + L.row_tok);
            p.row_w = reinterpret_cast<const float *>(ws + L.row_w);
            err = launch_w8<W8_BF16_Y, true>(m, p, units, stream);
        } else {
            err = launch_w8<W8_BF16, true>(m, p, units, stream);
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
