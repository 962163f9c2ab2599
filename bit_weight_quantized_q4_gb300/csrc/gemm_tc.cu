// gemm_tc.cu -- prefill GEMM on the fifth-generation tensor cores (tcgen05,
// accumulators in tensor memory) for Q4_0 and Q8_0 weights and batches wider
// than 16 rows: y[nb][n] = x[nb][k] W^T (crate inferencelayer, Functions:
// gemm_q4_src -- a blocked GEMM whose column tile shares one weight stream).
//
// The per-block scales stay exact without per-block partial sums: every
// weight enters the tensor core as two f16 values hi + lo whose sum is
// exactly d * q * P (Q4_0: q - 8 for its nibble q; Q8_0: its signed byte),
// where P is a power of two per weight row chosen so that the row's largest
// |q|max |d| P lies in [2^14, 2^15) (|q|max = 8 or 128: no f16 overflow, no
// subnormal scales).  hi = f16(d' q) with d' = d P, and lo = f16(d' q - hi)
// is exact: d' q has at most 14 (Q8_0: 18) significant bits and lies on the
// grid of ulp(d').  The activations enter as one f16
// per value after a power-of-two scale per row of x that puts the row's
// largest magnitude in [2^14, 2^15), so the only rounding before the fp32
// accumulation is the activation's (relative 2^-11).  The K sum then runs
// whole inside the tensor core, and the epilogue multiplies by the two
// powers of two back.
//
// Two launches.  q4gemm_tc_stage_kernel writes the activation image: per
// BN-row column tile (BN = 512 over 256 rows, 256 over 128, else 128) and
// stage of BK columns (32 at BN = 512, else 64), K = 16 slabs in the
// K-major, unswizzled operand layout (tc_common.cuh), with the columns of
// each 32-column block in the order of the weight records' lanes (tc_col),
// plus each row's factor back.
// q4gemm_tc_kernel gives each CTA 128 weight rows (eight 16-row record
// tiles) by BN activation rows, one 128 x BN fp32 accumulator in tensor
// memory (a 512-wide tile fills all 512 columns, two N = 256 MMAs per step),
// and three warp roles (q4gemm_tc_kernel):
//   * a copy warp brings each stage's image slice in by bulk copies (TMA
//     engine; a ring of six, three or four slots);
//   * sixteen dequant warps read their lanes' record words straight from
//     global memory, three 128-column chunks ahead, and turn each stage's
//     records into hi / lo operand slabs (a ring of four slots, six at
//     BN = 512), one 16-byte store per lane and slab;
//   * an MMA warp issues each stage's MMAs (BK / 16 steps of K = 16, hi and
//     lo, M = 128, N = min(BN, 256)) and commits them to the stage's mbarrier,
//     which frees the operand and activation slots;
//   * at the end the dequant warps read the accumulator out of tensor memory
//     (warp w: lanes 32 (w % 4) .., columns (BN / 4) (w / 4) ..), scale and
//     store.
// Every wait is bounded; a wait that gives up records error 4, lets what is
// in flight land, frees the tensor memory and stores nothing.
#include "gemv_launch.cuh"
#include "tc_common.cuh"

namespace q4 {
namespace dev {

constexpr int kTcBM = 128;           // weight rows per CTA (eight record tiles)
constexpr int kTcDW = 16;                    // dequant warps (two per record tile)
constexpr int kTcThreads = 32 * (kTcDW + 2);  // and a copy warp, an MMA warp
constexpr int kTcSlab = kTcBM * 16 * 2;              // one K = 16 slab of 128 rows (4 KB)
constexpr int kTcOffFlags = 512;                     // tensor-memory address, abort flag
constexpr int kTcOffRowP = 1024;                     // [128] fp32 row factors P, then [128] their inverses
constexpr int kTcOffA = 2048;
// Per column-tile width BN (activation rows per CTA: 128, 256 or 512; the
// MMA's N is BN up to 256, and a 512-wide tile takes two N = 256 MMAs per
// step into the two halves of the tensor memory): the operand and
// activation slots and the shared-memory map.
template <int BN>
struct TcCfg {
    static_assert(BN == 128 || BN == 256 || BN == 512, "column tile");
    static constexpr int NN = BN > 256 ? 256 : BN;             // the MMA's N
    static constexpr int NH = BN / NN;                          // MMAs per step and operand
    // columns per stage: 32 for the 512-wide tile (four operand slots in
    // flight instead of two: 105 -> 96 us at nb = 512), else 64 (fewer
    // hand-offs: 32-column stages measured 52 -> 67 us at nb = 128)
    static constexpr int BK = BN == 512 ? 32 : 64;
    static constexpr int BPS = BK / 32;               // blocks per stage
    static constexpr int SPC = 4 / BPS;               // stages per 128-column record chunk
    static constexpr int AHalf = (BK / 16) * kTcSlab;  // hi (or lo) of one stage
    static constexpr int ASlot = 2 * AHalf;           // hi + lo
    // hi / lo operand slots and activation slots: 224 KB between them
    static constexpr int SA = BN == 512 ? 6 : 4;
    static constexpr int SB = BN == 128 ? 6 : BN == 256 ? 3 : 4;
    // stage completions: a waiter for stage k's must find it the slot's
    // latest or the one before, so the ring is as deep as both rings
    static constexpr int MD = SA > SB ? SA : SB;
    static constexpr int BSlot = BN * BK * 2;  // activations of one stage
    static constexpr int OffB = kTcOffA + SA * ASlot;
    static constexpr int Smem = OffB + SB * BSlot;
    static_assert(Smem <= (int)kSmemMax, "tcgen05 GEMM shared memory");
    static_assert(8 * (SB + SA + MD) <= kTcOffFlags, "barrier area");
};
// the column tile of a batch: 512 rows above 256, 256 above 128, else 128
// (one wave of 112 CTAs at 512 rows on a 14336-row matrix, and twice the
// tensor work per hand-off: 116 -> 105 us there)
Q4_HD constexpr int tc_bn(int nb) { return nb > 256 ? 512 : nb > 128 ? 256 : 128; }

// Bytes of the activation image (the row factors follow it): rows padded to
// whole column tiles, columns to whole chunks.
Q4_HD inline size_t tc_image_bytes(int nb, int C) {
    const int BN = tc_bn(nb);
    return (size_t)((nb + BN - 1) / BN) * BN * (size_t)C * kChunkK * 2;
}

// ---------------------------------------------------------------- staging

// Column order of the operands.  Inside each 32-column block the eight
// columns 8 t .. 8 t + 7 of the operands hold the block's elements
// 8 m + 2 t + b (i = 2 m + b): the elements one lane of a weight record
// holds, so that the dequant stores them with one 16-byte store.  The
// activations take the same order, so every product pairs the same element.
Q4_HD constexpr int tc_col(int t, int i) { return 8 * (i >> 1) + 2 * t + (i & 1); }

// One CTA per activation row (rows up to the column tile's end): the row's
// largest magnitude (each thread's column groups loaded at once, then a CTA
// reduction), its power-of-two scale, then the row's f16 values into the
// image in the operands' column order (zeros for rows at or beyond nb and
// columns at or beyond K up to whole chunks).  Rows of up to 8192 columns
// keep their values in registers; longer rows read them again.
constexpr int kTcStageG = 4;  // 8-column groups a thread keeps (256 threads x 4 x 8 = 8192)
__device__ __forceinline__ void tc_load_group(const float *xr, int gi, float2 (&v)[4]) {
    const int j = gi >> 2, t = gi & 3;  // block, lane-position
#pragma unroll
    for (int m = 0; m < 4; ++m) v[m] = __ldg(reinterpret_cast<const float2 *>(xr + 32 * j + tc_col(t, 2 * m)));
}
template <int BN>
__global__ void __launch_bounds__(256) q4gemm_tc_stage_kernel(const __grid_constant__ GemmParams p) {
    using Cf = TcCfg<BN>;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float red[8];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = blockIdx.x;  // activation row
    const int NS = Cf::SPC * p.C, KT = p.C * kChunkK, KG = KT / 8, KGv = p.K / 8;
    const bool live = r < p.nb;
    const float *xr = p.x + (size_t)r * p.K;
    float2 v[kTcStageG][4];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < kTcStageG; ++i) {
        const int gi = tid + 256 * i;
#pragma unroll
        for (int q = 0; q < 4; ++q) v[i][q] = make_float2(0.f, 0.f);
        if (live && gi < KGv) tc_load_group(xr, gi, v[i]);
    }
#pragma unroll
    for (int i = 0; i < kTcStageG; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(v[i][q].x), fabsf(v[i][q].y)));
    for (int gi = tid + 256 * kTcStageG; live && gi < KGv; gi += 256) {  // rows over 8192 columns
        float2 u[4];
        tc_load_group(xr, gi, u);
#pragma unroll
        for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(u[q].x), fabsf(u[q].y)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) m = fmaxf(m, red[w]);
    // m = f 2^e with f in [0.5, 1): scale 2^(15 - e) puts m in [2^14, 2^15)
    float sc = 1.f, back = 0.f;
    if (m > 0.f) {
        int e;
        frexpf(m, &e);
        const int se = min(15 - e, 127);
        sc = ldexpf(1.f, se);
        back = ldexpf(1.f, -se);
    }
    if (tid == 0) reinterpret_cast<float *>(p.img + tc_image_bytes(p.nb, p.C))[r] = live ? back : 0.f;
    const int nt = r / BN, rr = r % BN;
    uint8_t *base = p.img + (size_t)nt * NS * Cf::BSlot;
    // operand columns 8 gi .. 8 gi + 7
    auto put = [&](int gi, const float2 (&u)[4]) {
        uint32_t hw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __half2 h2 = __floats2half2_rn(u[q].x * sc, u[q].y * sc);
            hw[q] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        const int k = 8 * gi, s = k / Cf::BK, sl = (k % Cf::BK) / 16;
        *reinterpret_cast<uint4 *>(base + (size_t)s * Cf::BSlot + sl * (BN * 32) + tc::slab_off(rr, k % 16)) =
            make_uint4(hw[0], hw[1], hw[2], hw[3]);
    };
#pragma unroll
    for (int i = 0; i < kTcStageG; ++i)
        if (tid + 256 * i < KG) put(tid + 256 * i, v[i]);
    for (int gi = tid + 256 * kTcStageG; gi < KG; gi += 256) {
        float2 u[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        if (live && gi < KGv) tc_load_group(xr, gi, u);
        put(gi, u);
    }
}

// ---------------------------------------------------------------- GEMM

// global -> shared bulk copy completing on mbarrier `bar`, default L2 policy
// (the weights of a row tile are read by every column tile's CTA, the image
// by every row tile's).
__device__ __forceinline__ void bulk_g2s_keep(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Record geometry of the formats this GEMM takes: Q4_0 (the nibble words of
// rows 0..7 and 8..15 at 0 and 512, the scale words at 1024) and Q8_0 (the
// biased bytes at 0 and 1024, blocks 2-3 512 bytes after blocks 0-1, the
// scale words at 2048), and the largest |q| of each (|q - 8| <= 8, |q| <= 128).
template <int FMT>
struct TcFmt {
    static_assert(FMT == 0 || FMT == 2, "Q4_0 or Q8_0");
    static constexpr int REC = rec_bytes(FMT);
    static constexpr int SOFF = FMT == 2 ? 2048 : 1024;
    static constexpr float QMAX = FMT == 2 ? 128.f : 8.f;
};

// The row factors P (and 1 / P) of this lane's rows 16 w + g and 16 w + g + 8
// from the largest |d| of each row over all chunks: lane (g, cp) reads the
// scale words of chunks cp, cp + 4, ...; a butterfly over the four lanes of
// g gives the row maxima.
template <int FMT>
__device__ __forceinline__ void tc_row_factors(const GemmParams &p, int tile, bool live, float *rowP, int w,
                                               int lane) {
    using Fm = TcFmt<FMT>;
    const int g = lane >> 2, cp = lane & 3;
    float m0 = 0.f, m1 = 0.f;
    if (live) {
        const uint8_t *base = p.w + (size_t)tile * p.C * Fm::REC + Fm::SOFF + g * 16;
#pragma unroll 4
        for (int c = cp; c < p.C; c += 4) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(base + (size_t)c * Fm::REC));
            const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 d = __half22float2(*reinterpret_cast<const __half2 *>(&ws[j]));
                m0 = fmaxf(m0, fabsf(d.x));
                m1 = fmaxf(m1, fabsf(d.y));
            }
        }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    }
    if (cp == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float m = Fm::QMAX * (h ? m1 : m0);
            float P = 1.f, Pi = 1.f;
            if (m > 0.f) {  // m = f 2^e, f in [0.5, 1): m P in [2^14, 2^15)
                int e;
                frexpf(m, &e);
                P = ldexpf(1.f, 15 - e);
                Pi = ldexpf(1.f, e - 15);
            }
            rowP[16 * w + 8 * h + g] = P;
            rowP[kTcBM + 16 * w + 8 * h + g] = Pi;
        }
    }
}

// A dequant lane's words of one chunk, read straight from global memory:
// rows 16 tile + 8 h + g (g = lane % 8), lane-position tp = lane / 8.  Q4_0:
// the 16-byte nibble word (blocks 0..3); Q8_0: the 8 bytes of each block
// (blocks 0-1, then 2-3); both: the four blocks' scale words (rows g | g + 8).
template <int FMT>
struct TcWords {
    uint4 w[FMT == 2 ? 2 : 1];
    uint4 sc;
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < (FMT == 2 ? 2 : 1); ++i) w[i] = make_uint4(0u, 0u, 0u, 0u);
        sc = make_uint4(0u, 0u, 0u, 0u);
    }
    __device__ __forceinline__ void load(const uint8_t *rec, int h, int g, int tp) {
        using Fm = TcFmt<FMT>;
        if constexpr (FMT == 2) {
            w[0] = __ldg(reinterpret_cast<const uint4 *>(rec + h * 1024 + (4 * g + tp) * 16));
            w[1] = __ldg(reinterpret_cast<const uint4 *>(rec + h * 1024 + 512 + (4 * g + tp) * 16));
        } else {
            w[0] = __ldg(reinterpret_cast<const uint4 *>(rec + h * 512 + (4 * g + tp) * 16));
        }
        sc = __ldg(reinterpret_cast<const uint4 *>(rec + Fm::SOFF + g * 16));
    }
};

__device__ __forceinline__ uint32_t word_at(const uint4 &v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}
// Element pair m (the block's elements at operand columns 8 tp + 2 m, + 1)
// as f16x2 (q, q') exactly: Q4_0 from nibbles m and m + 4 of the block's
// word (q - 8), Q8_0 from bytes 2 m and 2 m + 1 of its 8 (u - 128); a value
// v <= 255 in the low byte of a half with exponent bits 0x64 is 1024 + v.
template <int FMT>
__device__ __forceinline__ __half2 tc_pair(const TcWords<FMT> &x, int j, int m) {
    uint32_t b;
    __half2 bias;
    if constexpr (FMT == 2) {
        const uint4 v = (j >> 1) ? x.w[FMT == 2 ? 1 : 0] : x.w[0];  // a select, not a dynamic index
        const uint32_t word = (j & 1) ? ((m >> 1) ? v.w : v.z) : ((m >> 1) ? v.y : v.x);
        if (m & 1)
            asm("prmt.b32 %0, %1, 0x64, 0x4342;" : "=r"(b) : "r"(word));
        else
            asm("prmt.b32 %0, %1, 0x64, 0x4140;" : "=r"(b) : "r"(word));
        bias = __float2half2_rn(1152.f);
    } else {
        b = ((word_at(x.w[0], j) >> (4 * m)) & 0x000F000Fu) | 0x64006400u;
        bias = __float2half2_rn(1032.f);
    }
    return __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
}

// One stage's share of a dequant warp: blocks BPS part .. BPS part + BPS - 1
// of the chunk for its row.  Lane-position tp holds the block's elements at
// operand columns 8 tp .. 8 tp + 7 (tc_col), so each of hi and lo is one
// 16-byte store at `rowoff` (+ the block's slabs).
template <int FMT, int BPS>
__device__ __forceinline__ void tc_dequant(const TcWords<FMT> &x, float P, int h, int part, uint32_t a_hi,
                                           uint32_t a_lo, uint32_t rowoff) {
#pragma unroll
    for (int jj = 0; jj < BPS; ++jj) {
        const int j = BPS * part + jj;
        const uint32_t sw = word_at(x.sc, j);
        const __half dh = __ushort_as_half((unsigned short)(h ? sw >> 16 : sw & 0xFFFFu));
        const __half2 d2 = __float2half2_rn(__half2float(dh) * P);  // d P: exact
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const __half2 q2 = tc_pair<FMT>(x, j, m);
            const __half2 hi = __hmul2(q2, d2);
            const __half2 lo = __hfma2(q2, d2, __hneg2(hi));
            hv[m] = *reinterpret_cast<const uint32_t *>(&hi);
            lv[m] = *reinterpret_cast<const uint32_t *>(&lo);
        }
        const uint32_t off = (uint32_t)(2 * jj * kTcSlab) + rowoff;
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a_hi + off), "r"(hv[0]), "r"(hv[1]), "r"(hv[2]),
                     "r"(hv[3])
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a_lo + off), "r"(lv[0]), "r"(lv[1]), "r"(lv[2]),
                     "r"(lv[3])
                     : "memory");
    }
}

// Warp roles: warps 0-15 dequantise (warp w: half w % 2 of record tile
// w / 2) and run the epilogue, warp 16 lane 0 issues the bulk copies, warp 17
// lane 0 issues the MMAs (warp 17 also owns the tensor memory).  They hand
// slots over through mbarriers only:
//   b_full[s % SB]    stage s's image slice landed       (copy; producer arms)
//   a_full[s % SA]    stage s's hi / lo slabs written    (16 arrivals)
//   mma_done[s % MD]  stage s's MMAs completed           (tcgen05.commit)
// A dequant warp writes stage s's operand slot after mma_done of stage
// s - SA; the producer loads stage s's image slice after mma_done of stage
// s - SB.  With MD >= SA, SB each such ordering keeps every barrier within
// one phase of its waiters.  (The records went through a shared-memory ring
// of bulk copies before: reading them into registers freed 27 KB for a
// fourth (sixth) operand slot, 97 -> 89 us at nb = 512 and 52 -> 44 us at
// nb = 128.)
template <int FMT, int BN>
__global__ void __launch_bounds__(kTcThreads, 1) q4gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    using Cf = TcCfg<BN>;
    using Fm = TcFmt<FMT>;
    constexpr int SA = Cf::SA, SB = Cf::SB, MD = Cf::MD;
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nt = blockIdx.x, mt = blockIdx.y;  // activation (column) tile fastest, weight row tile
    const int t0 = 8 * mt, tiles = min(8, p.T - t0);
    const int C = p.C, NS = Cf::SPC * C;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t b_full = sbase, a_full = b_full + 8 * SB, mma_done = a_full + 8 * SA;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + kTcOffFlags);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kTcOffFlags + 4);
    float *rowP = reinterpret_cast<float *>(smem + kTcOffRowP);
    const uint32_t a_base = sbase + kTcOffA, b_base = sbase + Cf::OffB;
    const uint8_t *img = p.img + (size_t)nt * NS * Cf::BSlot;
    const long long lim = p.wait_cycles;
    auto fail = [&]() {
        *abort_flag = 1;
        atomicExch(p.err, 4);
    };

    if (tid == 0) {
        for (int i = 0; i < SB; ++i) mbar_init(b_full + 8 * i, 1);
        for (int i = 0; i < MD; ++i) mbar_init(mma_done + 8 * i, 1);
        for (int i = 0; i < SA; ++i) mbar_init(a_full + 8 * i, kTcDW);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcDW + 1) {
        tc::tmem_alloc(smem_u32(tslot), BN);
        tc::tmem_relinquish();
    }
    if (warp < 8) tc_row_factors<FMT>(p, t0 + warp, warp < tiles, rowP, warp, lane);  // warp w: tile w
    tc::fence_before_sync();
    __syncthreads();  // barriers, tensor memory, row factors
    tc::fence_after_sync();
    const uint32_t taddr = *tslot;

    int b_issued = 0, mma_issued = 0;  // the issuing lanes' counts
    if (warp == kTcDW) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            auto issue_b = [&](int s) {
                const uint32_t bar = b_full + 8 * (s % SB);
                // extra_tx: testing the give-up path only
                mbar_expect_tx(bar, Cf::BSlot + (s == 0 ? (uint32_t)p.extra_tx : 0u));
                bulk_g2s_keep(b_base + (s % SB) * Cf::BSlot, img + (size_t)s * Cf::BSlot, Cf::BSlot, bar);
            };
            asm volatile("griddepcontrol.wait;" ::: "memory");
            for (; b_issued < min(SB, NS); ++b_issued) issue_b(b_issued);
            // then, in stage order, each slot as soon as its MMAs are done
            for (; b_issued < NS; ++b_issued) {
                if (*abort_flag) break;
                const int s = b_issued;
                if (!mbar_wait(mma_done + 8 * ((s - SB) % MD), (uint32_t)((s - SB) / MD) & 1u, lim)) {
                    fail();
                    break;
                }
                issue_b(s);
            }
        }
    } else if (warp == kTcDW + 1) {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_f16(kTcBM, Cf::NN);
            const uint64_t a0 = tc::smem_desc(a_base, 128, 256), b0 = tc::smem_desc(b_base, 128, 256);
            // at BN >= 256 stage s + 1's barriers are waited while stage s's
            // last MMAs are still queued, so the tensor pipe does not drain at
            // each hand-off (nb = 256: 52.3 -> 50.2 us, nb = 512: 88.9 ->
            // 86.5); at BN = 128 the stage is committed first (that order
            // measured 45.1 against 45.8 us there)
            constexpr int KS = Cf::BK / 16, PRE = BN >= 256 ? KS - 1 : KS;
            bool ready = mbar_wait(a_full, 0u, lim) && mbar_wait(b_full, 0u, lim);
            for (int s = 0; s < NS; ++s) {
                if (!ready || *abort_flag) {
                    if (!ready) fail();
                    break;
                }
                tc::fence_after_sync();
                // descriptors advance by (byte offset >> 4) in their start field
                const uint64_t ad = a0 + (uint64_t)(((s % SA) * Cf::ASlot) >> 4);
                const uint64_t bd = b0 + (uint64_t)(((s % SB) * Cf::BSlot) >> 4);
                auto step = [&](int ks) {
#pragma unroll
                    for (int nh = 0; nh < Cf::NH; ++nh) {  // activation rows NN nh .. into columns NN nh ..
                        const uint64_t bk = bd + (uint64_t)((ks * (BN * 32) + nh * (Cf::NN * 32)) >> 4);
                        const uint32_t d = taddr + (uint32_t)(nh * Cf::NN);
                        tc::mma_f16(d, ad + (uint64_t)((ks * kTcSlab) >> 4), bk, idesc, (s | ks) != 0);
                        tc::mma_f16(d, ad + (uint64_t)((Cf::AHalf + ks * kTcSlab) >> 4), bk, idesc, 1u);
                    }
                };
#pragma unroll
                for (int ks = 0; ks < PRE; ++ks) step(ks);
                if constexpr (PRE == KS) {
                    tc::commit(mma_done + 8 * (s % MD));
                    mma_issued = s + 1;
                }
                if (s + 1 < NS)
                    ready = mbar_wait(a_full + 8 * ((s + 1) % SA), (uint32_t)((s + 1) / SA) & 1u, lim) &&
                            mbar_wait(b_full + 8 * ((s + 1) % SB), (uint32_t)((s + 1) / SB) & 1u, lim);
                if constexpr (PRE < KS) {
#pragma unroll
                    for (int ks = PRE; ks < KS; ++ks) step(ks);
                    tc::commit(mma_done + 8 * (s % MD));
                    mma_issued = s + 1;
                }
            }
        }
    } else {
        // ---------------------------------------------------------- dequant
        // warp w: record tile w / 2, rows 8 (w % 2) + g.  Each lane reads its
        // 16-byte nibble word and the 16-byte scale word of a chunk straight
        // from global memory, three chunks ahead of their use.
        // lanes 8 tp .. 8 tp + 7 take lane-position tp of rows g = 0..7, so
        // that each quarter-warp's 16-byte stores fill 128 contiguous bytes
        const int tile = warp >> 1, h = warp & 1, g = lane & 7, tp = lane >> 3;
        const bool live = tile < tiles;
        const float P = rowP[16 * tile + 8 * h + g];
        // columns 8 tp .. 8 tp + 7 of a block: slab tp / 2 of its two, core
        // matrix half tp % 2
        const uint32_t rowoff = (uint32_t)((tp >> 1) * kTcSlab + (2 * tile + h) * 256 + (tp & 1) * 128 + g * 16);
        const uint8_t *wrec = p.w + (size_t)(t0 + tile) * C * Fm::REC;
        auto load = [&](int c, TcWords<FMT> &x) {
            if (live && c < C) x.load(wrec + (size_t)c * Fm::REC, h, g, tp);
        };
        TcWords<FMT> x0, x1, x2;
        x0.zero();
        x1.zero();
        x2.zero();
        load(0, x0);
        load(1, x1);
        load(2, x2);
        for (int s = 0; s < NS; ++s) {
            const int c = s / Cf::SPC, jh = s % Cf::SPC;  // chunk, part
            if (*abort_flag) break;
            if (jh == 0 && c > 0) {  // the next chunk's words; chunk c + 2's load goes out
                x0 = x1;
                x1 = x2;
                load(c + 2, x2);
            }
            // the operand slot is free once the MMAs of stage s - SA are done
            const bool ok = s < SA || mbar_wait(mma_done + 8 * ((s - SA) % MD), (uint32_t)((s - SA) / MD) & 1u, lim);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail();
                break;
            }
            tc::fence_after_sync();
            const uint32_t a_hi = a_base + (s % SA) * Cf::ASlot;
            if (live) tc_dequant<FMT, Cf::BPS>(x0, P, h, jh, a_hi, a_hi + Cf::AHalf, rowoff);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the slabs, for the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(a_full + 8 * (s % SA));
        }
    }

    // every role is done (or gave up): the products must have landed before
    // the accumulator is read or freed; the epilogue reads the staging
    // kernel's row factors
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    bool ok = !*abort_flag;
    if (ok && warp < kTcDW) {
        const bool done = mbar_wait(mma_done + 8 * ((NS - 1) % MD), (uint32_t)((NS - 1) / MD) & 1u, lim);
        if (!__all_sync(0xffffffffu, done) && lane == 0) fail();
    }
    __syncthreads();
    ok = !*abort_flag;
    if (!ok) {
        // let the copies and products in flight land, free the tensor
        // memory, store nothing
        if (warp == kTcDW && lane == 0) {
            for (int s = max(0, b_issued - SB); s < b_issued; ++s)
                mbar_wait(b_full + 8 * (s % SB), (uint32_t)(s / SB) & 1u, kWaitCycles);
        }
        if (warp == kTcDW + 1 && lane == 0 && mma_issued > 0)
            mbar_wait(mma_done + 8 * ((mma_issued - 1) % MD), (uint32_t)((mma_issued - 1) / MD) & 1u, kWaitCycles);
        tc::fence_before_sync();
        __syncthreads();
        if (warp == kTcDW + 1) {
            tc::fence_after_sync();
            tc::tmem_dealloc(taddr, BN);
        }
        return;
    }
    tc::fence_after_sync();

    // epilogue: dequant warp w reads lanes 32 (w % 4) .. (weight rows) and
    // columns (BN / 4) (w / 4) .. (activation rows) of the accumulator
    if (warp < kTcDW) {
        const float *F = reinterpret_cast<const float *>(p.img + tc_image_bytes(p.nb, p.C));
        const int q = warp & 3, cg = warp >> 2;
        const int rl = 32 * q + lane, row = kTcBM * mt + rl;
        const float pinv = rowP[kTcBM + rl];
#pragma unroll 1
        for (int cb = 0; cb < BN / 64; ++cb) {
            const int c0 = (BN / 4) * cg + 16 * cb;
            float v[16];
            tc::ld16(taddr + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, v);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int col = BN * nt + c0 + i;
                if (row < p.n && col < p.nb) {
                    float *dst = p.y + (size_t)col * p.n + row;
                    const float r = v[i] * pinv * F[col];
                    *dst = p.accumulate ? *dst + r : r;
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kTcDW + 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(taddr, BN);
    }
}

}  // namespace dev

size_t gemm_tc_image_bytes(int nb, int C) {
    const int BN = dev::tc_bn(nb);
    return dev::tc_image_bytes(nb, C) + (size_t)((nb + BN - 1) / BN) * BN * sizeof(float);
}

// Q4_0 and Q8_0 batches wider than 16 rows: the staging kernel, then the GEMM as its
// programmatic dependent.
template <int FMT, int BN>
static int launch_gemm_tc_bn(const GemmParams &p, cudaStream_t stream) {
    using Cf = dev::TcCfg<BN>;
    static size_t smem_set[64] = {0};
    if (!raise_smem(dev::q4gemm_tc_kernel<FMT, BN>, (size_t)Cf::Smem, smem_set)) return -1;
    const int NT = (p.nb + BN - 1) / BN;
    dev::q4gemm_tc_stage_kernel<BN><<<NT * BN, 256, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)NT, (unsigned)((p.T + 7) / 8), 1);
    cfg.blockDim = dim3(dev::kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = Cf::Smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dev::q4gemm_tc_kernel<FMT, BN>, p) == cudaSuccess ? 0 : -1;
}

template <int FMT>
static int launch_gemm_tc_fmt(const GemmParams &p, cudaStream_t stream) {
    switch (dev::tc_bn(p.nb)) {
        case 512: return launch_gemm_tc_bn<FMT, 512>(p, stream);
        case 256: return launch_gemm_tc_bn<FMT, 256>(p, stream);
        default: return launch_gemm_tc_bn<FMT, 128>(p, stream);
    }
}

int launch_gemm_tc(const GemmParams &p, int fmt, void *stream_) {
    cudaStream_t stream = (cudaStream_t)stream_;
    if (fmt == 2) return launch_gemm_tc_fmt<2>(p, stream);
    if (fmt == 0) return launch_gemm_tc_fmt<0>(p, stream);
    return -1;
}

}  // namespace q4
