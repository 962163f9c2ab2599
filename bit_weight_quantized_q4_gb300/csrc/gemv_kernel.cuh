// gemv_kernel.cuh -- the dequant-in-GEMV kernel family for sm_103a.
//
// What it computes (per activation row r and output row n):
//   Q4_0:   y = sum_b d_b * sum_j (q_bj - 8) * x_bj          (w = d*(q-8))
//   affine: y = sum_b s_b * sum_j q_bj * x_bj + m_b * gsum_b  (w = s*q + m)
// with an optional RMSNorm prologue (x -> x / sqrt(mean x^2 + eps) * gamma)
// and one of four epilogues: store, residual add, SwiGLU over a gate/up pair,
// or a per-group (max, index) for the greedy argmax.  The value formulas are
// crate inferencelayer's q4_0_to_q8_0n (Q4_0) and Module gpu's Q / HalfSet
// (affine weights, activation group sums); the fused neighbours follow
// honeycrisp/mod.rs, forward_decode_fused_layers.
//
// How (GB300-first, not the pages' Metal/WGSL shapes):
//  * One CTA (16 warps; 8 for nb > 8) owns a group of 16-row tile pairs and
//    one K-slice, at most one CTA per SM; a thread-block cluster of S CTAs
//    splits K and folds its partial sums over distributed shared memory in
//    rank order (deterministic, no atomics).
//  * The unit of work is one 128-column chunk of a tile pair: two weight
//    records that share one set of activation fragments.  Each warp streams
//    its contiguous range of units through a private two-stage shared-memory
//    ring filled by TMA bulk copies on mbarriers, a stage ahead of its
//    compute.
//  * A nibble masked in place is an exact f16 subnormal (q * 2^-24, or
//    q * 2^-20 for the upper nibble of a byte), so a 32-bit word of eight
//    nibbles becomes four tensor-core A registers with one shift and four
//    ANDs.  The activation operand carries the factor 16 at the positions
//    of the lower nibbles, and products land in units of 2^-20.
//  * Activations are staged once per CTA in shared memory in mma B-fragment
//    order, each 32-column block scaled by its own power of two: as an f16
//    hi + lo pair (about 22 significant bits) for nb <= 4, where hi and lo
//    of a row are two n columns of one product, and as one f16 for nb > 4.
//    The block's factor back to the input's units multiplies its weight
//    scale.
//  * mma.sync m16n8k16 (f16 in, fp32 accumulate) forms the per-block dot
//    products.  The block's offset term (the -8 of Q4_0, the min m of the
//    affine format) multiplies the block's activation sum: for Q4_0 that sum
//    is the same tensor-core product with every nibble equal to 8, so a
//    block of all-8 weights cancels exactly; for the affine format it is the
//    fp32 group sum.  Each block's result is scaled by its fp32 scale and
//    accumulated in fp32, so weights are never rounded.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cooperative_groups.h>
#include <math.h>

#include <type_traits>

#include "q4_internal.h"

namespace q4 {
namespace dev {

namespace cg = cooperative_groups;

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
template <int OFF>
__device__ __forceinline__ uint4 lds128_at(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+%5];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a), "n"(OFF)
                 : "memory");
    return v;
}
// A 16-byte shared load into v where p is non-zero; elsewhere v keeps its
// value (a predicated load, no select).
template <int OFF>
__device__ __forceinline__ void lds128_if(uint4 &v, uint32_t a, uint32_t p) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %5, 0;\n\t@q ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+%6];\n\t}"
                 : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
                 : "r"(a), "r"(p), "n"(OFF)
                 : "memory");
}
// mbarrier and bulk-copy (TMA engine) primitives for the weight ring.
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// global -> shared bulk copy of `bytes` (16-byte aligned, multiple of 16),
// completing on mbarrier `bar`; evict-first in L2 (weights stream once)
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// Wait for phase `parity` of mbarrier `bar` to complete; false after `limit`
// SM clock cycles (the caller records the failure and stops).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit) {
    long long t0 = 0;
    for (int it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{ .reg .pred P; mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2; selp.b32 %0, 1, 0, P; }"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (it == 0) {
            t0 = clock64();
        } else if (clock64() - t0 > limit) {
            return false;
        }
    }
}

// Barrier over the NW warps of a CTA (named barrier 1): every warp of the
// kernels, used by the engine's functions.
template <int NW>
__device__ __forceinline__ void csync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

// D = A * B + (z0..z3), m16n8k16, f16 inputs, fp32 accumulate; the caller
// passes four zero registers that stay live across the loop.
__device__ __forceinline__ void mma16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1, float z0, float z1, float z2, float z3) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z0), "f"(z1), "f"(z2), "f"(z3));
}

// D = A * B + C, m16n8k16, f16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One nibble word -> four tensor-core A registers of exact f16 subnormals:
//   r0 = (nib0, nib4) * 2^-24   r1 = (nib1, nib5) * 2^-20
//   r2 = (nib2, nib6) * 2^-24   r3 = (nib3, nib7) * 2^-20
// (a nibble at bits 0..3 of a half is the mantissa q * 2^-24; at bits 4..7
// it is q * 2^-20).  r0/r2 cover k positions 0..7 of their k16 step, r1/r3
// positions 8..15.
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
    const uint32_t w8 = w >> 8;
    r0 = w & 0x000F000Fu;
    r1 = w & 0x00F000F0u;
    r2 = w8 & 0x000F000Fu;
    r3 = w8 & 0x00F000F0u;
}
// The A registers of a block whose every nibble is 8 (Q4_0), and of a Q8_0
// block whose every weight is 0 (every biased byte 128): the value of a zero
// weight in the format's A encoding, for the registers of k positions 0..7
// (lo) and 8..15 (hi) of a k16 step.
constexpr uint32_t kEightLo = 0x00080008u;
constexpr uint32_t kEightHi = 0x00800080u;
template <int FMT>
__device__ __forceinline__ constexpr uint32_t zero_lo() { return FMT == 2 ? 0x00800080u : kEightLo; }

// Two biased Q8_0 bytes -> one tensor-core A register of exact f16
// subnormals u * 2^-24: bytes 0-1 of w (sel 0x4140) or bytes 2-3 (0x4342)
// into the low byte of each half.
template <unsigned SEL>
__device__ __forceinline__ uint32_t bytes_to_half2(uint32_t w) {
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(w), "n"(SEL));
    return r;
}
// A registers of one block of a Q8_0 record for rows g (a[0], a[2], a[4],
// a[6]) and g + 8 (odd): lo / hi are the lane's two words of the block.
__device__ __forceinline__ void unpack_q8(uint32_t lo, uint32_t hi, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    r0 = bytes_to_half2<0x4140>(lo);
    r1 = bytes_to_half2<0x4342>(lo);
    r2 = bytes_to_half2<0x4140>(hi);
    r3 = bytes_to_half2<0x4342>(hi);
}

// Q1: the tensor-core A register rho of a lane's sign word -- bits rho and
// 16 + rho (stored inverted) become the f16 sign bits of +1.0 halves.
__device__ __forceinline__ uint32_t q1_signs(uint32_t w, int rho) {
    return ((w << (15 - rho)) & 0x80008000u) | 0x3C003C00u;  // one shift, one lop3 (rho is unrolled)
}

// The two 16-bit scales (or mins) of a scale word as fp32.
template <int FMT>
__device__ __forceinline__ float2 scale_pair(uint32_t w) {
    if (FMT != 1) {  // fp16 scales (Q4_0, Q8_0); affine: bf16
        __half2 h = *reinterpret_cast<const __half2 *>(&w);
        return __half22float2(h);
    } else {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
}

// Q4_K: the rows' fp16 d and dmin (words {row g, row g+8}) as d * 2^24 and
// -dmin * 2^24, the factors q4k_pair takes.
__device__ __forceinline__ void q4k_rows(uint32_t dw, uint32_t mw, float2 &dd, float2 &dm) {
    const float2 d = __half22float2(*reinterpret_cast<const __half2 *>(&dw));
    const float2 m = __half22float2(*reinterpret_cast<const __half2 *>(&mw));
    constexpr float P = 16777216.f;  // 2^24
    dd = make_float2(d.x * P, d.y * P);
    dm = make_float2(-m.x * P, -m.y * P);
}
// Q4_K: block scale d*sc and min -dmin*mn of rows g and g+8 from the record's
// byte word {sc(g), mn(g), sc(g+8), mn(g+8)}.  prmt makes each 6-bit byte an
// exact f16 subnormal v * 2^-24, so with dd, dm from q4k_rows both products
// are exact in fp32.
__device__ __forceinline__ void q4k_pair(uint32_t w, float2 dd, float2 dm, float2 &s2, float2 &m2) {
    const uint32_t scw = bytes_to_half2<0x4240>(w), mnw = bytes_to_half2<0x4341>(w);
    const float2 sc = __half22float2(*reinterpret_cast<const __half2 *>(&scw));
    const float2 mn = __half22float2(*reinterpret_cast<const __half2 *>(&mnw));
    s2 = make_float2(dd.x * sc.x, dd.y * sc.y);
    m2 = make_float2(dm.x * mn.x, dm.y * mn.y);
}

__device__ __forceinline__ void map_tile(const GemvParams &p, int t, int &m, int &tm) {
    if (p.mode == MODE_PAIRS) {
        m = t & 1;
        tm = t >> 1;
        return;
    }
    m = 0;
    tm = t;
    while (m + 1 < p.nmat && tm >= p.tiles[m]) {
        tm -= p.tiles[m];
        ++m;
    }
}

// Total order used by the argmax: larger value first, then lower index; NaN
// ranks below every number.
__device__ __forceinline__ void am_take(float &bv, int &bi, float v, int i) {
    float key = isnan(v) ? -INFINITY : v;
    if (key > bv || (key == bv && i < bi)) {
        bv = key;
        bi = i;
    }
}

__device__ __forceinline__ void am_warp(float &bv, int &bi) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
        }
    }
}

// ---------------------------------------------------------------------------
// The engine shared by the per-call kernel and the persistent decode-step
// kernel.  A "job" (GemvParams) is one GEMV-shaped launch: up to three
// matrices over one activation batch with one prologue and one epilogue.
// Within a job, group g of `groups` owns a contiguous range of tile pairs
// (gate/up pairs for SwiGLU) and cluster rank r its K-slice; the CTA's
// (pair, chunk) units are split into contiguous ranges, one per warp.

template <int CLS>
struct Cls {
    static constexpr bool HLN = CLS <= 1;    // hi / lo of an activation row in two n columns
    static constexpr int NT = CLS == 3 ? 2 : 1;  // 8-column n-tiles
    static constexpr int NW = cls_warps(CLS);
    static constexpr int DU = cls_depth(CLS);     // ring stages per warp
    static constexpr int SU = cls_stage(CLS);     // pair units per stage: stages of 2*SU records
    static constexpr int GSW = cls_gsw(CLS);
    static constexpr int NGR = HLN ? 1 : 2 * NT;    // group-sum rows one lane uses
    static constexpr int NACC = HLN ? 2 : 4 * NT;   // accumulators per record and lane
};

struct Geo {
    int t0, tiles_here, np;      // the group's first tile, its tiles and tile pairs
    int c0, cs, kb, ke;          // K-slice: chunks [c0, c0 + cs), columns [kb, ke)
    int U, ub, ue, n_my, fp;     // units of the CTA; this warp's [ub, ue) and its first pair
};

// a / b for 0 <= a < 2^24 and b >= 1: a float quotient (a few units off at
// most), corrected to the floor
__device__ __forceinline__ int div_small(int a, int b) {
    int d = (int)__fdividef((float)a, (float)b);
    while (d > 0 && d * b > a) --d;
    while ((d + 1) * b <= a) ++d;
    return d;
}
// The group's span of a job: balanced contiguous ranges of the job's
// P = T / upt units (pairs, or single tiles).
__device__ __forceinline__ JobSpan span_of(const GemvParams &p, int group) {
    JobSpan sp;
    const int P = p.upt == 2 ? (p.T + 1) >> 1 : p.T;  // units of upt (1 or 2) tiles
    int p0 = 0, p1 = 0;
    if (group < p.groups) {  // a job with fewer units than CTAs leaves the rest without work
        if ((long long)(group + 1) * P < (1 << 24)) {
            p0 = div_small(group * P, p.groups);
            p1 = div_small((group + 1) * P, p.groups);
        } else {
            p0 = (int)((unsigned long long)group * P / p.groups);
            p1 = (int)((unsigned long long)(group + 1) * P / p.groups);
        }
    }
    sp.np = p1 - p0;
    sp.t0 = p.upt * p0;
    sp.tiles = min(p.upt * sp.np, p.T - sp.t0);
    sp.pad = 0;
    return sp;
}
// One warp's geometry of a job from the group's span: the K-slice of `rank`
// and the warp's contiguous run [ub, ue) of the group's (pair, chunk) units.
template <int NW>
__device__ __forceinline__ Geo geo_of(const GemvParams &p, const JobSpan &sp, int rank, int warp) {
    Geo q;
    q.np = sp.np;
    q.t0 = sp.t0;
    q.tiles_here = sp.tiles;
    q.c0 = rank * p.Cs;
    q.cs = max(0, min(p.Cs, p.C - q.c0));
    q.kb = q.c0 * kChunkK;
    q.ke = min(p.K, q.kb + p.Cs * kChunkK);
    q.U = q.np * q.cs;
    q.ub = (int)((long long)warp * q.U / NW);
    q.ue = (int)((long long)(warp + 1) * q.U / NW);
    q.n_my = q.ue - q.ub;
    q.fp = q.cs > 0 ? (q.U < (1 << 24) ? div_small(q.ub, q.cs) : q.ub / q.cs) : 0;
    return q;
}
template <int NW>
__device__ __forceinline__ Geo make_geo(const GemvParams &p, int group, int rank, int warp) {
    return geo_of<NW>(p, span_of(p, group), rank, warp);
}

template <int REC>
__device__ __forceinline__ const uint8_t *tile_base(const GemvParams &p, int t) {
    int m, tm;
    map_tile(p, t, m, tm);
    return p.w[m] + (size_t)tm * p.C * REC;
}

// Units in the next ring stage: at most SU tile-pair units (2*SU single-tile
// units), never past the end of the current pair's K-slice (`to_pair_end`
// units) or the warp's range (`left`).  Producer and consumer both use it.
template <int SU>
__device__ __forceinline__ int stage_units(int upt, int to_pair_end, int left) {
    int n = upt == 2 ? SU : 2 * SU;
    if (n > to_pair_end) n = to_pair_end;
    if (n > left) n = left;
    return n;
}

// The weight units a warp streams, in order, across the jobs of a launch:
// each job's [ub, ue) range of this warp, job after job.  The load side runs
// up to DU-1 units ahead of the compute side, across job boundaries.
template <int REC, int NW>
struct WeightStream {
    const GemvParams *jobs;
    const JobSpan *spans;  // the group's span of every job, or null (computed)
    int njobs, group, rank, warp;
    int job, c0, cs, t0, pl, c, left, upt;
    const uint8_t *ptr0, *ptr1;  // the next unit's records (ptr1 null: the unit has one tile)

    __device__ __forceinline__ void pair_ptrs() {
        const GemvParams &p = jobs[job];
        const int ta = t0 + p.upt * pl;
        const size_t off = (size_t)(c0 + c) * REC;
        ptr0 = tile_base<REC>(p, ta) + off;
        ptr1 = p.upt == 2 && ta + 1 < p.T ? tile_base<REC>(p, ta + 1) + off : nullptr;
    }
    __device__ __forceinline__ void start(const Geo &q) {
        if (q.n_my > 0) {
            upt = jobs[job].upt;
            t0 = q.t0;
            c0 = q.c0;
            cs = q.cs;
            pl = q.fp;
            c = q.ub - q.fp * q.cs;
            left = q.n_my;
            pair_ptrs();
        }
    }
    __device__ __forceinline__ void next_job() {
        while (left == 0 && job + 1 < njobs) {
            ++job;
            start(spans != nullptr ? geo_of<NW>(jobs[job], spans[job], rank, warp)
                                   : make_geo<NW>(jobs[job], group, rank, warp));
        }
    }
    __device__ __forceinline__ void init(const GemvParams *j, const JobSpan *sp, int n, int grp, int rk, int w) {
        jobs = j;
        spans = sp;
        njobs = n;
        group = grp;
        rank = rk;
        warp = w;
        job = -1;
        left = 0;
        ptr0 = ptr1 = nullptr;
        next_job();
    }
    // one job whose geometry the caller already has
    __device__ __forceinline__ void init_one(const GemvParams *j, const Geo &q) {
        jobs = j;
        spans = nullptr;
        njobs = 1;
        job = 0;
        left = 0;
        ptr0 = ptr1 = nullptr;
        start(q);
    }
    // copy the next stage -- up to SU units of the current tile pair (2*SU
    // for single-tile units), never past the pair or the warp's range -- into
    // the ring stage at shared address `dst` with the TMA engine, completing
    // on mbarrier `bar`: one copy of n consecutive records per tile (the
    // second tile's records at dst + SU*REC).  The issuer issues; every
    // thread that holds this stream advances its state.
    template <int SU>
    __device__ __forceinline__ void issue(uint32_t dst, uint32_t bar, bool issuer, uint64_t policy, int extra_tx) {
        const int n = stage_units<SU>(upt, cs - c, left);
        if (issuer) {
            // the warp's reads of this stage (ordered by the caller's
            // __syncwarp) come before the async-proxy writes that refill it
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_expect_tx(bar, (ptr1 != nullptr ? 2 : 1) * n * REC + extra_tx);
            bulk_g2s(dst, ptr0, n * REC, bar, policy);
            if (ptr1 != nullptr) bulk_g2s(dst + SU * REC, ptr1, n * REC, bar, policy);
        }
        left -= n;
        c += n;
        if (c == cs) {
            c = 0;
            ++pl;
            if (left > 0) pair_ptrs();
        } else {
            ptr0 += (size_t)n * REC;
            if (ptr1 != nullptr) ptr1 += (size_t)n * REC;
        }
        // the move to the warp's next job (next_job) is left to the caller
    }
};

// One warp's ring of DU stages of SREC bytes, with an mbarrier per stage.
// `fill` counts stages issued, `cons` stages consumed; stage k lives in
// slot k mod DU and completes phase (k / DU) mod 2 of its barrier.  A slot is
// refilled as soon as the warp has consumed it, so between two jobs of the
// persistent kernel (and before the first one) all DU stages are in flight.
template <int DU, int SU, int SREC>
struct Ring {
    uint32_t base, bars;  // this warp's stages and barriers (shared addresses)
    uint32_t fill, cons;
    bool ok;              // false once a wait gave up
    uint64_t policy;
    long long limit;      // bound of one wait (cycles)
    int extra_tx;         // expected bytes beyond the copies (testing only; 0)
    __device__ __forceinline__ void init(uint32_t b, uint32_t br, int lane, long long lim, int extra) {
        base = b;
        bars = br;
        fill = cons = 0;
        ok = true;
        limit = lim;
        extra_tx = extra;
        policy = evict_first_policy();
        if (lane == 0) {
#pragma unroll
            for (int i = 0; i < DU; ++i) mbar_init(bars + 8 * i, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
    }
    __device__ __forceinline__ uint32_t stage(uint32_t k) const { return base + (k % DU) * SREC; }
    __device__ __forceinline__ uint32_t bar(uint32_t k) const { return bars + (k % DU) * 8; }
    // Refill one free slot from the stream; with cross == false only from
    // the stream's current job (moving to the next job recomputes its
    // geometry, which the persistent kernel does while it waits at a grid
    // barrier).  True if a stage was issued.
    template <class WS>
    __device__ __forceinline__ bool push(WS &ws, int lane, bool cross = true) {
        if (!ok || fill - cons >= (uint32_t)DU) return false;
        if (ws.left == 0) {
            if (!cross) return false;
            ws.next_job();
            if (ws.left == 0) return false;
        }
        ws.template issue<SU>(stage(fill), bar(fill), lane == 0, policy, extra_tx);
        ++fill;
        return true;
    }
    // wait for the unit `cons`; the warp agrees on the outcome
    __device__ __forceinline__ bool wait(int *err, int lane) {
        const bool mine = ok && mbar_wait(bar(cons), (cons / DU) & 1, limit);
        const bool all = __all_sync(0xffffffffu, mine);
        if (!all && ok) {
            ok = false;
            if (lane == 0 && err != nullptr) atomicExch(err, 2);
        }
        return ok;
    }
    // after a failed wait: wait (bounded, always by the full second, whatever
    // `limit` is) for the copies still in flight into this warp's stages
    // before the CTA may exit
    __device__ __forceinline__ void drain() {
        if (ok) return;
        for (uint32_t k = cons; k < fill; ++k) mbar_wait(bar(k), (k / DU) & 1, kWaitCycles);
        cons = fill;
    }
};

// Shared-memory regions of one CTA (sizes: engine_smem()).
struct Smem {
    uint8_t *xs;     // activation slice, f16 (hi + lo for nb <= 4) in mma B-fragment order
    float *gs;       // affine block sums of x (* gamma) [chunk][GSW rows][4 blocks]
    float *fs;       // block factors back to the input's units (times 2^20), same shape
    float *red;      // cluster fold (S > 1): partials pushed by each rank [S][slice]
    float *slots;    // per-warp tile partials [warp][SW][16][nb]
    float *rbuf;     // reductions [4][warp][kMaxNb]
    float *nx;       // per row [8][kMaxNb]: 0 this slice's sum of squares, 5 output factor
    int *wtab;       // the warps' unit ranges: ub[NW + 1], fp[NW] (tail of rbuf)
    uint64_t *bars;  // ring barriers [warp][DU]
    uint8_t *ring;   // weight stages [warp][DU][2*SU records]
};

template <int CLS>
__device__ __forceinline__ Smem carve(uint8_t *smem, int nb, int Cs, int TG, int SW, int S) {
    using C = Cls<CLS>;
    Smem m;
    m.xs = smem;
    m.gs = reinterpret_cast<float *>(smem + (size_t)4 * cls_xrow(CLS) * nb * Cs);
    m.fs = m.gs + (size_t)4 * C::GSW * Cs;
    m.red = m.fs + (size_t)4 * C::GSW * Cs;
    m.slots = m.red + (S > 1 ? (size_t)(TG + 2 * S) * kTileRows * nb : 0);
    m.rbuf = m.slots + (size_t)C::NW * SW * kTileRows * nb;
    m.nx = m.rbuf + 4 * C::NW * kMaxNb;
    m.wtab = reinterpret_cast<int *>(m.rbuf + 3 * C::NW * kMaxNb);
    m.bars = reinterpret_cast<uint64_t *>(m.nx + 8 * kMaxNb);
    m.ring = reinterpret_cast<uint8_t *>(m.bars + C::NW * C::DU);
    return m;
}

// The activation scale of a block: 2^e with bound * 2^e in [2^10, 2^11), from
// the exponent field of `bound` (e clamped to [-100, 100]; 0 for a zero or
// non-finite bound), and the factor back 2^(U-e), which also undoes the 2^-U
// unit of the products: U = 20 for the nibble formats (their lower nibbles
// meet activations times 16), 24 for Q8_0 (bytes are f16 subnormals u * 2^-24),
// 0 for Q1 (signs are f16 +-1).
template <int FMT>
__device__ __forceinline__ void block_scale(float bound, float &scale, float &back) {
    constexpr int U = FMT == 2 ? 24 : FMT == 4 ? 0 : 20;
    int e = 0;
    if (bound > 0.f && bound <= 3.0e38f) {
        const int be = (int)((__float_as_uint(bound) >> 23) & 0xFF);  // bound in [2^(be-127), 2^(be-126))
        e = max(-100, min(100, 10 - (be - 127)));
    }
    scale = __uint_as_float((uint32_t)(127 + e) << 23);
    back = __uint_as_float((uint32_t)(127 + U - e) << 23);
}

// Byte offset in the staged slice of element kk (0..31) of 32-column block
// b, activation row r, half `part` (0 hi, 1 lo); elements kk and kk+1 (kk
// even) share one f16x2 word.  Within a k16 step s, position pp = 2t + 8h + e
// belongs to lane-position t, B register h and half e.
//   nb <= 4: per block [column 2r+part][t][s][h]         (16 bytes per lane)
//   nb >  4: per block [n-tile][row][t][s][part][h]        (32 bytes per lane)
template <int CLS>
__device__ __forceinline__ int xs_off(int b, int r, int kk, int part, int xbs) {
    const int s = kk >> 4, pp = kk & 15, h = pp >> 3, tt = (pp & 7) >> 1;
    if (Cls<CLS>::HLN) return b * xbs + ((2 * r + part) * 4 + tt) * 16 + (2 * s + h) * 4;
    return b * xbs + (r >> 3) * 512 + ((r & 7) * 4 + tt) * 16 + s * 8 + h * 4;  // f16 value only (part 0)
}

// Store columns (kl, kl+1) of row r, already scaled, as hi + lo f16 pairs;
// for the nibble formats, positions 0..7 of a k16 step carry the factor 16 of
// the lower nibbles.
template <int FMT, int CLS>
__device__ __forceinline__ void put_pair(uint8_t *xs, int xbs, int r, int kl, float v0, float v1) {
    const int b = kl >> 5, kk = kl & 31;
    if (is_nibble(FMT) && (kk & 8) == 0) {
        v0 *= 16.f;
        v1 *= 16.f;
    }
    const __half2 hi = __floats2half2_rn(v0, v1);
    const float2 hf = __half22float2(hi);
    const __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
    *reinterpret_cast<__half2 *>(xs + xs_off<CLS>(b, r, kk, 0, xbs)) = hi;
    *reinterpret_cast<__half2 *>(xs + xs_off<CLS>(b, r, kk, 1, xbs)) = lo;
}

__device__ __forceinline__ int gs_idx(int b, int row, int GSW) { return ((b >> 2) * GSW + row) * 4 + (b & 3); }

// Activation staging.  Each 32-column block of a row gets its own power-of-
// two scale, chosen from the block's largest magnitude (of x * gamma when
// gamma is given) so that it lands in [2^10, 2^11); the scaled values go to
// shared memory in mma B-fragment order (xs_off) as f16 hi + lo parts (nb <= 4)
// or as f16 alone (nb > 4), the first 8 of every 16 columns times 16 (see
// unpack_word).  The block's factor back to the input's units, times the
// 2^20 of the nibble unpack, goes to fs, and run_units folds it into the
// block's weight scale.  For the affine format gs holds the block sums of
// x (* gamma) in the input's units: in-kernel in the order of q4_group_sums
// (pairs, then a butterfly), or the caller's group sums.  (Q4_0's offset
// products are formed in run_units.)  With gamma, the RMS factor of each row
// multiplies the row's outputs at the end (nx[5]); its sum of squares is
// reduced per warp here and per row after the staging barrier.  Activation
// loads bypass L1 (.cg): in the persistent kernel another SM may have
// rewritten them since this SM last read them.

// nb = 1 (class 0).  The tensor-core products of a chunk run as one chain of
// eight m16n8k16 products (two k16 steps per 32-column block) in which block
// j's activations occupy only the column pair (2j, 2j+1) -- hi and lo -- and
// are zero in the other columns; a lane's B registers are kept when its
// column belongs to the block and zeroed otherwise.  At the end of the chain
// lane (g, t) holds block t's hi and lo products of rows g and g+8.
// chunk_b() loads those B registers for block j of a chunk.
__device__ __forceinline__ uint4 chunk_b(const uint8_t *xchunk, int j, int boff, int g) {
    uint4 b = *reinterpret_cast<const uint4 *>(xchunk + j * 128 + boff);
    if ((g >> 1) != j) b = make_uint4(0u, 0u, 0u, 0u);
    return b;
}

// The offset products of Q4_0 (and Q8_0) for nb = 1: per chunk, the product
// chain above with every weight at its zero code (nibble 8, byte 128), once
// per CTA and job; block j's hi + lo goes to the block-sum slot of block j.
// A weight block of all zero codes then gives exactly the same chain values,
// so (hi + lo) - offset is exactly zero for it.
template <int FMT, int CLS>
__device__ __forceinline__ void eights_chunk(const Smem &m, int c, int lane) {
    constexpr uint32_t EL = zero_lo<FMT>();
    constexpr int GSW = Cls<CLS>::GSW;
    const int g = lane >> 2, t = lane & 3;
    const int boff = (g & 1) * 64 + t * 16;
    const float z = 0.f;
    const uint8_t *xchunk = m.xs + c * kBlocksPerChunk * 128;
    float d[4];
#pragma unroll
    for (int j = 0; j < kBlocksPerChunk; ++j) {
        const uint4 b = chunk_b(xchunk, j, boff, g);
        if (j == 0) {
            mma16816_c(d, EL, EL, kEightHi, kEightHi, b.x, b.y, z, z, z, z);
        } else {
            mma16816(d, EL, EL, kEightHi, kEightHi, b.x, b.y);
        }
        mma16816(d, EL, EL, kEightHi, kEightHi, b.z, b.w);
    }
    if (g == 0) m.gs[gs_idx(c * kBlocksPerChunk + t, 0, GSW)] = d[0] + d[1];
}
// All chunks, after the staging barrier (the generic staging path of nb = 1,
// slices over 8192 columns); ends with a CTA barrier.
template <int FMT, int CLS>
__device__ void eights_c0(const Smem &m, int Cs, int warp, int lane) {
    for (int c = warp; c < Cs; c += Cls<CLS>::NW) eights_chunk<FMT, CLS>(m, c, lane);
    csync<Cls<CLS>::NW>();
}

// Activation loads of the staging: columns (k, k+1) or (k .. k+3) of the row
// starting at element `roff` of x, read from the fp32 rows, or from the
// HalfSet streams (Module gpu, Struct HalfSet), where x[2i] is element i of
// the even stream and x[2i+1] element i of the odd stream, each an f16.
__device__ __forceinline__ float half_at(const uint16_t *s, size_t i) {
    return __half2float(__ushort_as_half(__ldcg(reinterpret_cast<const unsigned short *>(s) + i)));
}
__device__ __forceinline__ float2 load_x2(const GemvParams &p, size_t roff, int k) {
    if (p.xe == nullptr) return __ldcg(reinterpret_cast<const float2 *>(p.x + roff + k));
    const size_t i = (roff + k) >> 1;
    return make_float2(half_at(p.xe, i), half_at(p.xo, i));
}
__device__ __forceinline__ float4 load_x4(const GemvParams &p, size_t roff, int k) {
    if (p.xe == nullptr) return __ldcg(reinterpret_cast<const float4 *>(p.x + roff + k));
    const size_t i = (roff + k) >> 1;  // even: one f16 pair per stream
    const unsigned e = __ldcg(reinterpret_cast<const unsigned *>(p.xe + i));
    const unsigned o = __ldcg(reinterpret_cast<const unsigned *>(p.xo + i));
    const float2 fe = __half22float2(*reinterpret_cast<const __half2 *>(&e));
    const float2 fo = __half22float2(*reinterpret_cast<const __half2 *>(&o));
    return make_float4(fe.x, fo.x, fe.y, fo.y);
}

// After the writes: the staging barrier, then each row's output factor --
// its inverse RMS from the warps' partial sums of squares in warp order (and,
// for a split K, the cluster ranks' slice sums in rank order), or 1.
template <int CLS>
__device__ void stage_finish(const GemvParams &p, const Smem &m, int S, int nb, int tid) {
    constexpr int NW = Cls<CLS>::NW;
    const bool norm = p.gamma != nullptr;
    csync<NW>();
    // every CTA of the cluster has started (the kernel's first arrive): from
    // here on the ranks may access each other's shared memory
    if (S > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (!norm) {
        if (tid < nb) m.nx[5 * kMaxNb + tid] = 1.f;
        return;
    }
    // warp w adds the NW warps' partial sums of rows w and w + NW by a fixed
    // butterfly (lane l < NW holds warp l's partial)
    const int warp = tid >> 5, lane = tid & 31;
    float tss[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = warp + h * NW;
        if (r < nb) {  // warp-uniform
            float v = lane < NW ? m.rbuf[r * NW + lane] : 0.f;
#pragma unroll
            for (int off = NW / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            tss[h] = v;
        }
    }
    if (S > 1) {
        cg::cluster_group cluster = cg::this_cluster();
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (warp + h * NW < nb && lane == 0) m.nx[warp + h * NW] = tss[h];
        cluster.sync();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = warp + h * NW;
            if (r < nb && lane == 0) {
                tss[h] = 0.f;
                for (int rr = 0; rr < S; ++rr) tss[h] += cluster.map_shared_rank(m.nx, rr)[r];
            }
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = warp + h * NW;
        if (r < nb && lane == 0) m.nx[5 * kMaxNb + r] = 1.0f / sqrtf(tss[h] / (float)p.K + p.eps);
    }
}

// One activation row whose slice has at most 8192 columns (nb = 1).  Warp w
// stages the 128-column chunks w, w + NW, ...: lane l converts column pairs
// l and l + 32 of a chunk (a block's 32 columns are the pairs of 16 lanes).
// For Q4_0 the warp then forms the eights product of each of its chunks
// (eights_chunk) as soon as the chunk is written, so no CTA barrier is added
// for it.
template <int FMT, int CLS>
__device__ void stage_row1(const GemvParams &p, const Geo &q, const Smem &m, int tid, int warp, int lane) {
    using C = Cls<CLS>;
    constexpr int NW = C::NW, NTH = NW * 32, GSW = C::GSW;
    constexpr int RP = 8192 / (2 * NTH);  // pairs per lane at most
    const int Cs = p.Cs;                  // staged chunks; columns at or beyond ke are zero
    const int kb = q.kb, ke = q.ke;
    const bool norm = p.gamma != nullptr;
    const bool given = has_min(FMT) && p.gsum != nullptr && !norm;  // block sums from the caller
    const int nch = warp < Cs ? (Cs - 1 - warp) / NW + 1 : 0;   // chunks of this warp
    float2 xv[RP], gv[RP];
    // every load first (guarded, not a loop exit, so that they can all be in
    // flight together); pass qq: chunk warp + (qq / 2) * NW, half qq & 1
#pragma unroll
    for (int qq = 0; qq < RP; ++qq) {
        float2 v = make_float2(0.f, 0.f), gm = make_float2(1.f, 1.f);
        const int kl = 128 * (warp + (qq >> 1) * NW) + 64 * (qq & 1) + 2 * lane;
        if ((qq >> 1) < nch && kb + kl < ke) {
            v = load_x2(p, 0, kb + kl);
            if (norm) gm = *reinterpret_cast<const float2 *>(p.gamma + kb + kl);
        }
        xv[qq] = v;
        gv[qq] = gm;
    }
    float ss = 0.f;
#pragma unroll
    for (int qq = 0; qq < RP; ++qq) {
        if ((qq >> 1) >= nch) break;  // warp-uniform
        const int c = warp + (qq >> 1) * NW;
        const int kl = 128 * c + 64 * (qq & 1) + 2 * lane;
        float a0 = xv[qq].x, a1 = xv[qq].y;
        ss = fmaf(a0, a0, ss);
        ss = fmaf(a1, a1, ss);
        if (norm) {
            a0 *= gv[qq].x;
            a1 *= gv[qq].y;
        }
        float bm = fmaxf(fabsf(a0), fabsf(a1));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        float sc, back;
        block_scale<FMT>(bm, sc, back);
        put_pair<FMT, CLS>(m.xs, 128, 0, kl, a0 * sc, a1 * sc);
        float bsum = 0.f;
        if (has_min(FMT) && !given) bsum = half_warp_sum(a0 + a1);
        if ((lane & 15) == 0) {
            m.fs[gs_idx(kl >> 5, 0, GSW)] = back;
            if (has_min(FMT) && !given) m.gs[gs_idx(kl >> 5, 0, GSW)] = bsum;
        }
        if (has_offset(FMT) && (qq & 1)) {  // the chunk is written: its eights (zero-weight) product
            __syncwarp();
            eights_chunk<FMT, CLS>(m, c, lane);
        }
    }
    if (given) {
        for (int b = tid; b < Cs * kBlocksPerChunk; b += NTH)
            m.gs[gs_idx(b, 0, GSW)] = kb + 32 * b < ke ? __ldcg(p.gsum + kb / 32 + b) : 0.f;
    }
    if (norm) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) m.rbuf[warp] = ss;
    }
}

// Stage this CTA's activation slice of job p.  One row of at most 8192
// columns takes stage_row1.  Otherwise the slice is nb rows x Cs chunks of
// 128 columns; a segment is one row of one chunk, a float4 per lane (a
// block's 32 columns are 8 lanes).  Warp w takes a contiguous range of
// segments in row-major order, SEG at a time with all their loads in flight
// (with PIPE, the next SEG load while the current SEG are converted).
template <int FMT, int CLS, int SEG, bool PIPE>
__device__ void stage_x(const GemvParams &p, const Geo &q, const Smem &m, int S, int tid, int warp, int lane) {
    using C = Cls<CLS>;
    constexpr int NW = C::NW, NTH = NW * 32, GSW = C::GSW;
    const int nb = CLS == 0 ? 1 : p.nb;
    const int Cs = p.Cs;
    if (CLS == 0 && Cs * kChunkK <= 8192) {
        stage_row1<FMT, CLS>(p, q, m, tid, warp, lane);
        stage_finish<CLS>(p, m, S, 1, tid);
        return;
    }
    const int kb = q.kb, ke = q.ke;
    const int xbs = cls_xrow(CLS) * nb;
    const bool norm = p.gamma != nullptr;
    const bool given = has_min(FMT) && p.gsum != nullptr && !norm;  // block sums from the caller
    const int nseg = nb * Cs;
    const int spw = (nseg + NW - 1) / NW;
    const int s0 = min(warp * spw, nseg), s1 = min(s0 + spw, nseg);
    const int r0 = CLS == 0 ? 0 : s0 / Cs, c0 = s0 - r0 * Cs;  // row and chunk of this warp's first segment

    // with gamma: this warp's partial sums of squares, [nb][NW], zero for
    // every row until a flush below overwrites the rows it touches
    float *part = m.rbuf;
    if (norm && lane < nb) part[lane * NW + warp] = 0.f;
    __syncwarp();
    float ss = 0.f;
    int rcur = r0;

    const float f16x = !is_nibble(FMT) || (lane & 2) ? 1.f : 16.f;  // the lower nibbles' factor 16
    constexpr int LO = 64, P2 = 16;  // lo part (nb <= 4), second column pair
    const int lane_off = (lane >> 3) * xbs + (lane & 1) * 32 + ((lane >> 2) & 1) * 8 + ((lane >> 1) & 1) * 4;
    // a batch's loads are predicated, not branched around, so that they are
    // all in flight together; segments past the range read as zeros
    auto load_batch = [&](float4 (&xv)[SEG], float4 (&gv)[SEG], int base, int r, int c) {
#pragma unroll
        for (int j = 0; j < SEG; ++j) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f), g = make_float4(1.f, 1.f, 1.f, 1.f);
            const int k = kb + 128 * c + 4 * lane;
            if (base + j < s1 && k < ke) {
                v = load_x4(p, (size_t)r * p.K, k);
                if (norm) g = __ldg(reinterpret_cast<const float4 *>(p.gamma + k));
            }
            xv[j] = v;
            gv[j] = g;
            if (++c == Cs) {
                c = 0;
                ++r;
            }
        }
    };
    // convert a batch; (r, c) advance past it
    auto convert_batch = [&](const float4 (&xv)[SEG], const float4 (&gv)[SEG], int base, int &r, int &c) {
#pragma unroll
        for (int j = 0; j < SEG; ++j) {
            const bool valid = base + j < s1;  // warp-uniform
            if (norm && valid && r != rcur) {  // a new row: this warp's sum for the previous one
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (lane == 0) part[rcur * NW + warp] = ss;
                ss = 0.f;
                rcur = r;
            }
            const int kl = 128 * c + 4 * lane;
            const float4 v = xv[j];
            float4 a = v;
            if (norm) {
                ss = fmaf(v.x, v.x, ss);
                ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss);
                ss = fmaf(v.w, v.w, ss);
                a.x *= gv[j].x;
                a.y *= gv[j].y;
                a.z *= gv[j].z;
                a.w *= gv[j].w;
            }
            float bm = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w)));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
            float sc, back;
            block_scale<FMT>(bm, sc, back);
            const float f = sc * f16x;
            const __half2 h0 = __floats2half2_rn(a.x * f, a.y * f);
            const __half2 h1 = __floats2half2_rn(a.z * f, a.w * f);
            __half2 l0 = h0, l1 = h1;
            if (C::HLN) {
                const float2 b0 = __half22float2(h0), b1 = __half22float2(h1);
                l0 = __floats2half2_rn(a.x * f - b0.x, a.y * f - b0.y);
                l1 = __floats2half2_rn(a.z * f - b1.x, a.w * f - b1.y);
            }
            float bsum = 0.f;
            if (has_min(FMT) && !given) bsum = block8_sum(a);
            if (valid) {
                const int seg = C::HLN ? 4 * c * xbs + 128 * r : 4 * c * xbs + (r >> 3) * 512 + (r & 7) * 64;
                uint8_t *d = m.xs + seg + lane_off;
                *reinterpret_cast<__half2 *>(d) = h0;
                *reinterpret_cast<__half2 *>(d + P2) = h1;
                if (C::HLN) {
                    *reinterpret_cast<__half2 *>(d + LO) = l0;
                    *reinterpret_cast<__half2 *>(d + P2 + LO) = l1;
                }
                if ((lane & 7) == 0) {
                    m.fs[gs_idx(kl >> 5, r, GSW)] = back;
                    if (has_min(FMT) && !given) m.gs[gs_idx(kl >> 5, r, GSW)] = bsum;
                }
            }
            if (++c == Cs) {
                c = 0;
                ++r;
            }
        }
    };
    auto advance = [&](int &r, int &c, int n) {
        c += n;
        while (c >= Cs) {
            c -= Cs;
            ++r;
        }
    };
    int rc = r0, cc = c0;  // the next segment to convert
    if (PIPE) {
        // two batches in registers: the next one's loads are in flight while
        // the current one is converted
        float4 xa[SEG], ga[SEG], xb[SEG], gb[SEG];
        int rl = r0, cl = c0;  // the next segment to load
        if (s0 < s1) load_batch(xa, ga, s0, rl, cl);
        advance(rl, cl, SEG);
        for (int base = s0; base < s1; base += 2 * SEG) {
            if (base + SEG < s1) load_batch(xb, gb, base + SEG, rl, cl);
            advance(rl, cl, SEG);
            convert_batch(xa, ga, base, rc, cc);
            if (base + 2 * SEG < s1) load_batch(xa, ga, base + 2 * SEG, rl, cl);
            advance(rl, cl, SEG);
            if (base + SEG < s1) convert_batch(xb, gb, base + SEG, rc, cc);
        }
    } else {
        float4 xa[SEG], ga[SEG];
        for (int base = s0; base < s1; base += SEG) {
            load_batch(xa, ga, base, rc, cc);
            convert_batch(xa, ga, base, rc, cc);
        }
    }
    if (norm && s0 < s1) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) part[rcur * NW + warp] = ss;
    }
    if (given) {
        const int nblk = Cs * kBlocksPerChunk;
        for (int i = tid; i < nb * nblk; i += NTH) {
            const int r = i / nblk, b = i - r * nblk;
            m.gs[gs_idx(b, r, GSW)] = kb + 32 * b < ke ? __ldcg(p.gsum + (size_t)r * (p.K / 32) + kb / 32 + b) : 0.f;
        }
    }
    stage_finish<CLS>(p, m, S, nb, tid);
    if (CLS == 0 && has_offset(FMT)) eights_c0<FMT, CLS>(m, Cs, warp, lane);
}

template <int I>
__device__ __forceinline__ uint32_t word_of(const uint4 &v) {
    return I == 0 ? v.x : I == 1 ? v.y : I == 2 ? v.z : v.w;
}

// This warp's units of one job: per unit, the activation fragments and
// offset sums of its chunk, then for each of the pair's records and each of
// the chunk's four blocks: unpack, tensor-core products, offset, scale.
// Each tile's partial over this warp's chunks goes to one of its slots.
// Consumes one ring stage per unit and refills it from `ws`.
template <int FMT, int CLS>
using RingOf = Ring<Cls<CLS>::DU, stage_su(FMT, CLS), 2 * stage_su(FMT, CLS) * rec_bytes(FMT)>;
template <int FMT, int CLS>
using StreamOf = WeightStream<rec_bytes(FMT), Cls<CLS>::NW>;

// nb = 1: the unit loop on the chunk-wide product chain (see chunk_b).  Per
// record: the chain's eight products as two independent chains of four
// (blocks 0-1 and 2-3; their sum is the single chain's value, since each
// column only ever adds exact zeros from the other chain's blocks), then one
// block's offset and scale per lane -- block t's (hi + lo - offset) * d * f
// for rows g and g+8 (Q4_0; affine: s * f * (hi + lo) + m * block sum) --
// added to the lane's running sums; the four lanes of a row are added at the
// end of each tile's slice.  Two records are in flight at a time: the two
// tiles of a pair unit, or two consecutive chunks of a single-tile stage.

// The chunk's activation registers (chunk_b) and block t's offset term and
// activation factor, for lane (g, t).
struct ChunkX {
    uint4 B[kBlocksPerChunk];
    float G, F;
};
template <int CLS>
__device__ __forceinline__ void load_chunk(ChunkX &x, const Smem &m, int cc, int boff, int g, int t) {
    const uint8_t *xchunk = m.xs + cc * kBlocksPerChunk * 128;
#pragma unroll
    for (int j = 0; j < kBlocksPerChunk; ++j) x.B[j] = chunk_b(xchunk, j, boff, g);
    const int gi = gs_idx(cc * kBlocksPerChunk + t, 0, Cls<CLS>::GSW);
    x.G = m.gs[gi];
    x.F = m.fs[gi];
}

// load_chunk into registers kept over a warp's units: only the lane's own
// block (g >> 1) is loaded; its other three B registers were zeroed once
// (zero_chunk) and stay zero, so no select is needed per chunk.
template <int CLS>
__device__ __forceinline__ void refresh_chunk(ChunkX &x, const Smem &m, int cc, int boff, int g, int t) {
    const uint32_t a = smem_u32(m.xs + cc * kBlocksPerChunk * 128 + boff);
    const uint32_t jj = (uint32_t)(g >> 1);
    lds128_if<0>(x.B[0], a, jj == 0u);
    lds128_if<128>(x.B[1], a, jj == 1u);
    lds128_if<256>(x.B[2], a, jj == 2u);
    lds128_if<384>(x.B[3], a, jj == 3u);
    const int gi = gs_idx(cc * kBlocksPerChunk + t, 0, Cls<CLS>::GSW);
    x.G = m.gs[gi];
    x.F = m.fs[gi];
}
__device__ __forceinline__ void zero_chunk(ChunkX &x) {
#pragma unroll
    for (int j = 0; j < kBlocksPerChunk; ++j) x.B[j] = make_uint4(0u, 0u, 0u, 0u);
}

// A lane's weight words of one record: the nibble formats' two 16-byte words
// (rows g and g+8, word j for block j), or Q8_0's four (rows g and g+8,
// blocks 0-1 and 2-3).  regs<J>() gives the eight tensor-core A registers of
// block J: rows g (even) and g+8 (odd), k positions in unpack_word's order.
template <int FMT>
struct RecWords {
    uint4 w[FMT == 2 ? 4 : FMT == 4 ? 1 : 2];  // Q1: w[0].x, .y = the sign words of rows g, g + 8
    __device__ __forceinline__ void load(uint32_t ra, int lane) {
        if constexpr (FMT == 4) {
            asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(w[0].x), "=r"(w[0].y) : "r"(ra + lane * 8) : "memory");
            return;
        }
        w[0] = lds128_at<0>(ra + lane * 16);
        w[1] = lds128_at<FMT == 2 ? 1024 : 512>(ra + lane * 16);
        if constexpr (FMT == 2) {
            w[2] = lds128_at<512>(ra + lane * 16);
            w[3] = lds128_at<1536>(ra + lane * 16);
        }
    }
    template <int J>
    __device__ __forceinline__ void regs(uint32_t (&a)[8]) const {
        if constexpr (FMT == 4) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[2 * i] = q1_signs(w[0].x, 4 * J + i);
                a[2 * i + 1] = q1_signs(w[0].y, 4 * J + i);
            }
        } else if constexpr (FMT == 2) {
            const uint4 &r0 = w[J < 2 ? 0 : 2], &r1 = w[J < 2 ? 1 : 3];
            unpack_q8((J & 1) ? r0.z : r0.x, (J & 1) ? r0.w : r0.y, a[0], a[2], a[4], a[6]);
            unpack_q8((J & 1) ? r1.z : r1.x, (J & 1) ? r1.w : r1.y, a[1], a[3], a[5], a[7]);
        } else {
            unpack_word(J == 0 ? w[0].x : J == 1 ? w[0].y : J == 2 ? w[0].z : w[0].w, a[0], a[2], a[4], a[6]);
            unpack_word(J == 0 ? w[1].x : J == 1 ? w[1].y : J == 2 ? w[1].z : w[1].w, a[1], a[3], a[5], a[7]);
        }
    }
};
// Byte offset of the scale words in a record, and of the mins (affine).
template <int FMT>
__device__ __forceinline__ constexpr int scale_off() { return FMT == 2 ? 2048 : FMT == 4 ? 256 : 1024; }

// One record at shared address ra against chunk x: this lane's block's share
// of rows g and g+8, added to a0 and a1.
template <int FMT>
__device__ __forceinline__ void record_c0(uint32_t ra, const ChunkX &x, int lane, float &a0, float &a1) {
    RecWords<FMT> rw;
    rw.load(ra, lane);
    uint32_t sw, mw = 0u;                            // scales (mins) of (row g, block t), (row g + 8, block t)
    uint32_t dw = 0u, dmw = 0u;                      // Q4_K: d and dmin of rows g, g + 8
    if constexpr (FMT == 4)  // Q1: one scale per row and chunk
        asm volatile("ld.shared.u32 %0, [%1+256];" : "=r"(sw) : "r"(ra + (lane >> 2) * 4) : "memory");
    else
        asm volatile("ld.shared.u32 %0, [%1+%2];" : "=r"(sw) : "r"(ra + lane * 4), "n"(scale_off<FMT>()) : "memory");
    if (FMT == 1) asm volatile("ld.shared.u32 %0, [%1+1152];" : "=r"(mw) : "r"(ra + lane * 4) : "memory");
    if (FMT == 3) {
        asm volatile("ld.shared.u32 %0, [%1+1152];" : "=r"(dw) : "r"(ra + (lane >> 2) * 4) : "memory");
        asm volatile("ld.shared.u32 %0, [%1+1184];" : "=r"(dmw) : "r"(ra + (lane >> 2) * 4) : "memory");
    }
    const float z = 0.f;
    float dA[4], dB[4];
    uint32_t a[8], b[8];
    rw.template regs<0>(a);
    rw.template regs<2>(b);
    mma16816_c(dA, a[0], a[1], a[2], a[3], x.B[0].x, x.B[0].y, z, z, z, z);
    mma16816_c(dB, b[0], b[1], b[2], b[3], x.B[2].x, x.B[2].y, z, z, z, z);
    mma16816(dA, a[4], a[5], a[6], a[7], x.B[0].z, x.B[0].w);
    mma16816(dB, b[4], b[5], b[6], b[7], x.B[2].z, x.B[2].w);
    rw.template regs<1>(a);
    rw.template regs<3>(b);
    mma16816(dA, a[0], a[1], a[2], a[3], x.B[1].x, x.B[1].y);
    mma16816(dB, b[0], b[1], b[2], b[3], x.B[3].x, x.B[3].y);
    mma16816(dA, a[4], a[5], a[6], a[7], x.B[1].z, x.B[1].w);
    mma16816(dB, b[4], b[5], b[6], b[7], x.B[3].z, x.B[3].w);
    const float T0 = (dA[0] + dB[0]) + (dA[1] + dB[1]);  // block t, row g: hi + lo
    const float T2 = (dA[2] + dB[2]) + (dA[3] + dB[3]);  // row g + 8
    float2 s2, m2 = make_float2(0.f, 0.f);
    if constexpr (FMT == 3) {
        float2 dd, dm;
        q4k_rows(dw, dmw, dd, dm);
        q4k_pair(sw, dd, dm, s2, m2);
    } else {
        s2 = scale_pair<FMT>(sw);
        if (FMT == 1) m2 = scale_pair<FMT>(mw);
    }
    if (has_offset(FMT)) {
        a0 = fmaf(s2.x * x.F, T0 - x.G, a0);
        a1 = fmaf(s2.y * x.F, T2 - x.G, a1);
    } else if (!has_min(FMT)) {  // Q1: the signs' product alone
        a0 = fmaf(s2.x * x.F, T0, a0);
        a1 = fmaf(s2.y * x.F, T2, a1);
    } else {
        a0 = fmaf(m2.x, x.G, fmaf(s2.x * x.F, T0, a0));
        a1 = fmaf(m2.y, x.G, fmaf(s2.y * x.F, T2, a1));
    }
}

// OWNB: the chunk registers persist over the warp's units (refresh_chunk);
// the per-call kernel takes it, the persistent step keeps load_chunk (there
// the longer-lived registers measured slower).
template <int FMT, bool OWNB, class RING>
__device__ void run_units_c0(const GemvParams &p, const Geo &q, const Smem &m, StreamOf<FMT, 0> &ws,
                             RING &ring, int warp, int lane, bool cross) {
    using C = Cls<0>;
    constexpr int REC = rec_bytes(FMT);
    constexpr int SU = stage_su(FMT, 0);
    const int g = lane >> 2, t = lane & 3;
    const int boff = (g & 1) * 64 + t * 16;
    const int cs = q.cs;
    float acc[2][2];  // [record][row g, row g + 8]: this lane's block's share
#pragma unroll
    for (int rc = 0; rc < 2; ++rc) acc[rc][0] = acc[rc][1] = 0.f;
    int pl = q.fp, cc = q.ub - q.fp * cs;
    const int upt = p.upt;
    if (lane == 0) {  // this warp's range for the fold (visible after the caller's barrier)
        m.wtab[warp] = q.ub;
        m.wtab[C::NW + 1 + warp] = q.fp;
        if (warp == C::NW - 1) m.wtab[C::NW] = q.ue;
    }
    float *my_slots = m.slots + (size_t)warp * p.SW * kTileRows;
    ChunkX k0, k1;  // OWNB: the persistent chunk registers
    if constexpr (OWNB) {
        zero_chunk(k0);
        zero_chunk(k1);
    }

    // a tile's slice is done: add the four lanes of each row (a fixed
    // butterfly) and hand the sums to the fold
    auto flush = [&](int pair, bool two) {
#pragma unroll
        for (int rc = 0; rc < 2; ++rc) {
            if (rc == 0 || two) {
                float a0 = acc[rc][0], a1 = acc[rc][1];
                a0 += __shfl_xor_sync(0xffffffffu, a0, 1);
                a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
                a0 += __shfl_xor_sync(0xffffffffu, a0, 2);
                a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
                if (t == 0) {
                    float *dst = my_slots + (size_t)(upt * (pair - q.fp) + rc) * kTileRows;
                    dst[g] = a0;
                    dst[g + 8] = a1;
                }
            }
            acc[rc][0] = acc[rc][1] = 0.f;
        }
    };

    for (int i = 0; i < q.n_my;) {
        const int n_st = stage_units<SU>(upt, cs - cc, q.n_my - i);  // units of this stage
        if (!ring.wait(p.err, lane)) break;  // gave up: stop (the error is recorded)
        const uint32_t st_base = ring.stage(ring.cons);
        i += n_st;
        if (upt == 2) {
            for (int su = 0; su < n_st; ++su) {  // a pair unit: its two records side by side
                const uint32_t st_a = st_base + su * REC;
                const bool two = q.t0 + 2 * pl + 1 < p.T;
                ChunkX x;
                if constexpr (OWNB) {
                    refresh_chunk<0>(k0, m, cc, boff, g, t);
                    x = k0;
                } else {
                    load_chunk<0>(x, m, cc, boff, g, t);
                }
                // both records without a branch, so that their products
                // interleave; a pair whose second tile is past the end has
                // no record in that slot (stale bytes of the stage), and
                // flush drops what it gave
                record_c0<FMT>(st_a, x, lane, acc[0][0], acc[0][1]);
                record_c0<FMT>(st_a + SU * REC, x, lane, acc[1][0], acc[1][1]);
                if (++cc == cs) {  // end of this pair's slice: hand the tiles over
                    flush(pl, two);
                    cc = 0;
                    ++pl;
                }
            }
        } else {
            // single-tile units: consecutive chunks of one tile (a stage never
            // crosses the tile's slice), two at a time
            int su = 0;
            for (; su + 1 < n_st; su += 2) {
                ChunkX x0, x1;
                if constexpr (OWNB) {
                    refresh_chunk<0>(k0, m, cc, boff, g, t);
                    refresh_chunk<0>(k1, m, cc + 1, boff, g, t);
                    x0 = k0;
                    x1 = k1;
                } else {
                    load_chunk<0>(x0, m, cc, boff, g, t);
                    load_chunk<0>(x1, m, cc + 1, boff, g, t);
                }
                float b0 = 0.f, b1 = 0.f;
                record_c0<FMT>(st_base + su * REC, x0, lane, acc[0][0], acc[0][1]);
                record_c0<FMT>(st_base + (su + 1) * REC, x1, lane, b0, b1);
                acc[0][0] += b0;
                acc[0][1] += b1;
                cc += 2;
                if (cc == cs) {
                    flush(pl, false);
                    cc = 0;
                    ++pl;
                }
            }
            if (su < n_st) {
                ChunkX x0;
                if constexpr (OWNB) {
                    refresh_chunk<0>(k0, m, cc, boff, g, t);
                    x0 = k0;
                } else {
                    load_chunk<0>(x0, m, cc, boff, g, t);
                }
                record_c0<FMT>(st_base + su * REC, x0, lane, acc[0][0], acc[0][1]);
                if (++cc == cs) {
                    flush(pl, false);
                    cc = 0;
                    ++pl;
                }
            }
        }
        __syncwarp();             // every lane is done with this stage: refill its slot
        ++ring.cons;
        ring.push(ws, lane, cross);
    }
    if (ring.ok && q.n_my > 0 && cc != 0) flush(pl, upt == 2 && q.t0 + 2 * pl + 1 < p.T);  // ended inside a unit
}

// cross: whether a refill may move the stream to its next job (false in the
// persistent kernel, which refills across jobs at the grid barrier).  OWNB:
// see run_units_c0.
template <int FMT, int CLS, bool OWNB, class RING>
__device__ void run_units(const GemvParams &p, const Geo &q, const Smem &m, StreamOf<FMT, CLS> &ws,
                          RING &ring, int warp, int lane, bool cross) {
    if constexpr (CLS == 0) {
        run_units_c0<FMT, OWNB>(p, q, m, ws, ring, warp, lane, cross);
        return;
    }
    using C = Cls<CLS>;
    constexpr int REC = rec_bytes(FMT);
    constexpr int SU = stage_su(FMT, CLS);
    constexpr int NT = C::NT, NGR = C::NGR, NACC = C::NACC;
    const int g = lane >> 2, t = lane & 3;
    const int nb = CLS == 0 ? 1 : p.nb;
    const int xbs = cls_xrow(CLS) * nb;
    const int cs = q.cs;
    // this lane's B-fragment slot in a block (lanes past the batch read a
    // duplicate column: their outputs are never stored)
    int boff[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        if (C::HLN) {
            boff[nt] = ((g % (2 * nb)) * 4 + t) * 16;
        } else {
            const int cnt = min(8, nb - 8 * nt);
            boff[nt] = nt * 512 + ((g % cnt) * 4 + t) * 16;
        }
    }
    int grow[NGR];  // this lane's offset-sum rows
#pragma unroll
    for (int j = 0; j < NGR; ++j) grow[j] = C::HLN ? t : 8 * (j >> 1) + 2 * t + (j & 1);
    float acc[2][NACC];
#pragma unroll
    for (int rc = 0; rc < 2; ++rc)
#pragma unroll
        for (int j = 0; j < NACC; ++j) acc[rc][j] = 0.f;
    const float z = 0.f;
    int pl = q.fp, cc = q.ub - q.fp * cs;
    const int upt = p.upt;
    if (lane == 0) {  // this warp's range for the fold (visible after the caller's barrier)
        m.wtab[warp] = q.ub;
        m.wtab[C::NW + 1 + warp] = q.fp;
        if (warp == C::NW - 1) m.wtab[C::NW] = q.ue;
    }
    float *my_slots = m.slots + (size_t)warp * p.SW * kTileRows * nb;

    auto flush = [&](int pair, bool two) {
#pragma unroll
        for (int rc = 0; rc < 2; ++rc) {
            if (rc == 0 || two) {
                float *dst = my_slots + (size_t)(upt * (pair - q.fp) + rc) * kTileRows * nb;
                if (C::HLN) {
                    if (t < nb) {
                        dst[g * nb + t] = acc[rc][0];
                        dst[(g + 8) * nb + t] = acc[rc][1];
                    }
                } else {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int r0 = 8 * nt + 2 * t;
                        if (r0 < nb) {
                            dst[g * nb + r0] = acc[rc][4 * nt + 0];
                            dst[(g + 8) * nb + r0] = acc[rc][4 * nt + 2];
                        }
                        if (r0 + 1 < nb) {
                            dst[g * nb + r0 + 1] = acc[rc][4 * nt + 1];
                            dst[(g + 8) * nb + r0 + 1] = acc[rc][4 * nt + 3];
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < NACC; ++j) acc[rc][j] = 0.f;
        }
    };

    for (int i = 0; i < q.n_my;) {
        const int n_st = stage_units<SU>(upt, cs - cc, q.n_my - i);  // units of this stage
        if (!ring.wait(p.err, lane)) break;  // gave up: stop (the error is recorded)
        const uint32_t st_base = ring.stage(ring.cons);
        i += n_st;
      for (int su = 0; su < n_st; ++su) {
        // unit su of the stage: its record(s) at st_base + su*REC (and + SU*REC)
        const uint32_t st_a = st_base + su * REC;
        const bool two = upt == 2 && q.t0 + 2 * pl + 1 < p.T;
        // the chunk's four block factors of this lane's activation rows, and
        // for the formats with a min their block sums (Q4_0 and Q8_0 form
        // their offset products per block below; Q1 has neither)
        float G[NGR][4], F[NGR][4];
#pragma unroll
        for (int j = 0; j < NGR; ++j) {
            const float4 fv = *reinterpret_cast<const float4 *>(m.fs + (cc * C::GSW + grow[j]) * 4);
            F[j][0] = fv.x;
            F[j][1] = fv.y;
            F[j][2] = fv.z;
            F[j][3] = fv.w;
            if (has_min(FMT)) {
                const float4 gv = *reinterpret_cast<const float4 *>(m.gs + (cc * C::GSW + grow[j]) * 4);
                G[j][0] = gv.x;
                G[j][1] = gv.y;
                G[j][2] = gv.z;
                G[j][3] = gv.w;
            } else if (!has_offset(FMT)) {  // Q1: no offset term
                G[j][0] = G[j][1] = G[j][2] = G[j][3] = 0.f;
            }
        }
        // the records' words: weights of rows g and g+8, scales (and mins)
        RecWords<FMT> rw[2];
        uint4 sw[2], mw[2];
        float2 dd[2], dm[2];  // Q4_K: the rows' d and dmin factors (q4k_rows)
#pragma unroll
        for (int rc = 0; rc < 2; ++rc) {
            sw[rc] = mw[rc] = make_uint4(0u, 0u, 0u, 0u);
            dd[rc] = dm[rc] = make_float2(0.f, 0.f);
            {
                // both records without a branch (as for nb = 1); what a second
                // record that is not there gives is dropped at the flush.  A
                // pair's second slot (stale bytes if its tile is past the end)
                // lies inside the stage; single-tile units (upt 1) have no
                // second slot, so theirs reads the first record again.
                const uint32_t ra = st_a + (upt == 2 ? rc * SU * REC : 0);
                rw[rc].load(ra, lane);
                if constexpr (FMT == 4) {  // Q1: one scale word per row pair, for every block
                    uint32_t w1;
                    asm volatile("ld.shared.u32 %0, [%1+256];" : "=r"(w1) : "r"(ra + g * 4) : "memory");
                    sw[rc] = make_uint4(w1, w1, w1, w1);
                } else {
                    sw[rc] = lds128_at<scale_off<FMT>()>(ra + g * 16);
                }
                if (FMT == 1) mw[rc] = lds128_at<1152>(ra + g * 16);
                if (FMT == 3) {
                    uint32_t dw, dmw;
                    asm volatile("ld.shared.u32 %0, [%1+1152];" : "=r"(dw) : "r"(ra + g * 4) : "memory");
                    asm volatile("ld.shared.u32 %0, [%1+1184];" : "=r"(dmw) : "r"(ra + g * 4) : "memory");
                    q4k_rows(dw, dmw, dd[rc], dm[rc]);
                }
            }
        }
        const uint8_t *xchunk = m.xs + cc * kBlocksPerChunk * xbs;

        auto block = [&](auto blk_c) {
            constexpr int blk = decltype(blk_c)::value;
            const uint8_t *xa = xchunk + blk * xbs;
            uint4 B[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) B[nt] = *reinterpret_cast<const uint4 *>(xa + boff[nt]);
            if (has_offset(FMT)) {
                // the block's offset product: the same tensor-core chain as the
                // weights' below, with every weight zero (every nibble 8 for
                // Q4_0, every biased byte 128 for Q8_0): exactly what such a
                // block gives, so it cancels to zero.  Kept times minus the
                // activation row's block factor F (a power of two: exact), for
                // both records: fma(F, T, -F G) is F (T - G) rounded once
                constexpr uint32_t EL = zero_lo<FMT>();
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float e[4];
                    mma16816_c(e, EL, EL, kEightHi, kEightHi, B[nt].x, B[nt].y, z, z, z, z);
                    mma16816(e, EL, EL, kEightHi, kEightHi, B[nt].z, B[nt].w);
                    if (C::HLN) {
                        G[0][blk] = -(F[0][blk] * (e[0] + e[1]));
                    } else {
                        G[2 * nt][blk] = -(F[2 * nt][blk] * e[0]);
                        G[2 * nt + 1][blk] = -(F[2 * nt + 1][blk] * e[1]);
                    }
                }
            }
#pragma unroll
            for (int rc = 0; rc < 2; ++rc) {
                uint32_t a[8];
                rw[rc].template regs<blk>(a);  // rows g (even) and g + 8 (odd)
                float2 s2, m2 = make_float2(0.f, 0.f);
                if constexpr (FMT == 3) {
                    q4k_pair(word_of<blk>(sw[rc]), dd[rc], dm[rc], s2, m2);
                } else {
                    s2 = scale_pair<FMT>(word_of<blk>(sw[rc]));
                    if (FMT == 1) m2 = scale_pair<FMT>(word_of<blk>(mw[rc]));
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float d[4];
                    if (C::HLN) {
                        // columns (2t, 2t+1) = (hi, lo) of activation row t
                        mma16816_c(d, a[0], a[1], a[2], a[3], B[nt].x, B[nt].y, z, z, z, z);
                        mma16816(d, a[4], a[5], a[6], a[7], B[nt].z, B[nt].w);
                        const float T0 = d[0] + d[1], T2 = d[2] + d[3];
                        const float fb = F[0][blk];
                        if (has_offset(FMT)) {
                            acc[rc][0] = fmaf(s2.x, fmaf(fb, T0, G[0][blk]), acc[rc][0]);
                            acc[rc][1] = fmaf(s2.y, fmaf(fb, T2, G[0][blk]), acc[rc][1]);
                        } else if (!has_min(FMT)) {
                            acc[rc][0] = fmaf(s2.x * fb, T0, acc[rc][0]);
                            acc[rc][1] = fmaf(s2.y * fb, T2, acc[rc][1]);
                        } else {
                            acc[rc][0] = fmaf(m2.x, G[0][blk], fmaf(s2.x * fb, T0, acc[rc][0]));
                            acc[rc][1] = fmaf(m2.y, G[0][blk], fmaf(s2.y * fb, T2, acc[rc][1]));
                        }
                    } else {
                        // columns (2t, 2t+1) = activation rows 8nt+2t, 8nt+2t+1
                        mma16816_c(d, a[0], a[1], a[2], a[3], B[nt].x, B[nt].y, z, z, z, z);
                        mma16816(d, a[4], a[5], a[6], a[7], B[nt].z, B[nt].w);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float sj = (j < 2 ? s2.x : s2.y) * F[2 * nt + (j & 1)][blk];
                            const float gj = G[2 * nt + (j & 1)][blk];
                            float &ac = acc[rc][4 * nt + j];
                            if (has_offset(FMT)) {
                                ac = fmaf(j < 2 ? s2.x : s2.y, fmaf(F[2 * nt + (j & 1)][blk], d[j], gj), ac);
                            } else if (!has_min(FMT)) {
                                ac = fmaf(sj, d[j], ac);
                            } else {
                                const float mj = j < 2 ? m2.x : m2.y;
                                ac = fmaf(mj, gj, fmaf(sj, d[j], ac));
                            }
                        }
                    }
                }
            }
        };
        block(std::integral_constant<int, 0>());
        block(std::integral_constant<int, 1>());
        block(std::integral_constant<int, 2>());
        block(std::integral_constant<int, 3>());
        if (++cc == cs) {  // end of this pair's slice: hand the tiles over
            flush(pl, two);
            cc = 0;
            ++pl;
        }
      }
        __syncwarp();             // every lane is done with this stage: refill its slot
        ++ring.cons;
        ring.push(ws, lane, cross);
    }
    if (ring.ok && q.n_my > 0 && cc != 0) flush(pl, upt == 2 && q.t0 + 2 * pl + 1 < p.T);  // ended inside a unit
}

// The warps' unit ranges, from the table run_units leaves in shared memory:
// warp w holds units [ub[w], ub[w+1]) and its first unit lies in tile unit
// fp[w].  Held in registers by each folding thread.
template <int NW>
struct WarpTable {
    int ub[NW + 1], fp[NW];
    __device__ __forceinline__ void load(const int *tab) {
#pragma unroll
        for (int w = 0; w <= NW; ++w) ub[w] = tab[w];
#pragma unroll
        for (int w = 0; w < NW; ++w) fp[w] = tab[NW + 1 + w];
    }
};

// Sum of the partials of output (tile tl, row, activation row r) over the
// warps whose unit range touched the tile, in warp order.
template <int CLS>
__device__ __forceinline__ float fold_one(const GemvParams &p, const Geo &q, const Smem &m,
                                          const WarpTable<Cls<CLS>::NW> &wt, int tl, int row, int r, int nb) {
    constexpr int NW = Cls<CLS>::NW;
    const int pl = tl / p.upt, sub = tl - pl * p.upt;
    const int u0 = pl * q.cs, u1 = u0 + q.cs;  // the tile's units
    const float *base = m.slots + (size_t)row * nb + r;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (max(wt.ub[w], u0) < min(wt.ub[w + 1], u1))
            v += base[(size_t)(w * p.SW + p.upt * (pl - wt.fp[w]) + sub) * kTileRows * nb];
    }
    return v;
}

// Cluster K-split (S > 1): each rank folds its warps' partials of all the
// group's outputs (its K-slice's share, output factor applied) and pushes
// each into the shared memory of the rank that finishes that output's tile
// (distributed shared memory stores into `red`); after one cluster barrier
// each rank adds the ranks' shares of its slice in rank order from its own
// memory and writes the slice (store, residual, SwiGLU on whole gate/up
// pairs).  For the argmax, each rank reduces its slice to (max, index) pairs
// and pushes them to rank 0, which combines them in rank order after a
// second barrier.  No rank reads another's shared memory after the first
// barrier here (the RMSNorm exchange of the staging comes before it), so
// none has to wait for the others before it exits.
template <int CLS>
__device__ void cluster_finish(const GemvParams &p, const Geo &q, const Smem &m, int S, int rank, int group, int tid,
                               int warp, int lane) {
    constexpr int NW = Cls<CLS>::NW, NTH = NW * 32;
    const int nb = CLS == 0 ? 1 : p.nb;
    const int tile_vals = kTileRows * nb;
    // rank j finishes units [j*nu/S, (j+1)*nu/S): whole tiles (whole gate/up
    // pairs for SwiGLU).  Every rank pushes its partials of a unit into the
    // owner's shared memory, at red[source rank][position in the slice]
    const int tpu = p.epi == EPI_SWIGLU ? 2 : 1;
    const int nu = q.tiles_here / tpu, uv = tpu * tile_vals;
    const int L = (nu + S - 1) / S * uv;  // the longest slice
    cg::cluster_group cluster = cg::this_cluster();
    {
        // thread tid folds output `rem` of tiles tl0, tl0 + per, ... (a tile's
        // 16 * nb outputs fit the CTA's threads)
        const int per = NTH / tile_vals;
        const int tl0 = tid / tile_vals, rem = tid - tl0 * tile_vals;
        if (tl0 < per && tl0 < q.tiles_here) {
            WarpTable<NW> wt;
            wt.load(m.wtab);
            const int row = rem / nb, r = rem - row * nb;
            const float fr = m.nx[5 * kMaxNb + r];
            for (int tl = tl0; tl < q.tiles_here; tl += per) {
                const float v = fold_one<CLS>(p, q, m, wt, tl, row, r, nb) * fr;
                const int u = tpu == 2 ? tl >> 1 : tl;
                const int j = ((u + 1) * S - 1) / nu;  // the owner of unit u
                *cluster.map_shared_rank(m.red + rank * L + tl * tile_vals + rem - (j * nu / S) * uv, j) = v;
            }
        }
    }
    cluster.sync();  // every partial is in its owner's shared memory
    const int i0 = (rank * nu / S) * uv, i1 = ((rank + 1) * nu / S) * uv;
    // this rank's slice: the sources in rank order (the sum replaces source
    // 0's entry, which only this thread reads)
    for (int i = tid; i < i1 - i0; i += NTH) {
        float v = 0.f;
        for (int rr = 0; rr < S; ++rr) v += m.red[rr * L + i];
        m.red[i] = v;
    }
    __syncthreads();
    if (group < p.groups) {
        if (p.epi == EPI_ARGMAX) {
            const int N = p.n[0];
            float *bvs = m.rbuf;  // [warp], then every rank's pairs [S][kMaxNb] (rank 0's copy is read)
            int *bis = reinterpret_cast<int *>(m.rbuf + NW);
            float *rv = m.rbuf + 2 * NW;
            int *ri_ = reinterpret_cast<int *>(m.rbuf + 2 * NW + kMaxCluster * kMaxNb);
            const int row0 = i0 / nb, row1 = i1 / nb;  // rows (tile * 16 + row) of the slice
            for (int r = 0; r < nb; ++r) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
                for (int ri = row0 + tid; ri < row1; ri += NTH) {
                    const int n = (q.t0 + ri / kTileRows) * kTileRows + (ri % kTileRows);
                    if (n >= N) continue;
                    const float v = m.red[ri * nb + r - i0];
                    if (p.out[0] != nullptr) p.out[0][(size_t)r * N + n] = v;
                    am_take(bv, bi, v, n);
                }
                am_warp(bv, bi);
                if (lane == 0) {
                    bvs[warp] = bv;
                    bis[warp] = bi;
                }
                __syncthreads();
                if (tid == 0) {
                    float fv = bvs[0];
                    int fi = bis[0];
                    for (int w = 1; w < NW; ++w) {
                        if (bvs[w] > fv || (bvs[w] == fv && bis[w] < fi)) {
                            fv = bvs[w];
                            fi = bis[w];
                        }
                    }
                    *cluster.map_shared_rank(rv + rank * kMaxNb + r, 0) = fv;
                    *cluster.map_shared_rank(ri_ + rank * kMaxNb + r, 0) = fi;
                }
                __syncthreads();
            }
            cluster.sync();  // every rank's pairs are in rank 0's shared memory
            if (rank == 0 && tid < nb) {
                float fv = -INFINITY;
                int fi = 0x7fffffff;
                for (int rr = 0; rr < S; ++rr) {
                    const float v = rv[rr * kMaxNb + tid];
                    const int k = ri_[rr * kMaxNb + tid];
                    if (v > fv || (v == fv && k < fi)) {
                        fv = v;
                        fi = k;
                    }
                }
                p.am_val[(size_t)tid * p.groups + group] = fv;
                p.am_idx[(size_t)tid * p.groups + group] = fi;
            }
        } else {
            for (int idx = i0 + tid; idx < i1; idx += NTH) {
                const int tl = idx / tile_vals;
                const int rem = idx - tl * tile_vals;
                const int row = rem / nb, r = rem - row * nb;
                int mi, tm;
                map_tile(p, q.t0 + tl, mi, tm);
                const int n = tm * kTileRows + row;
                const int N = p.n[mi];
                if (n >= N) continue;
                const float v = m.red[idx - i0];
                if (p.epi == EPI_STORE) {
                    p.out[mi][(size_t)r * N + n] = v;
                } else if (p.epi == EPI_RESIDUAL) {
                    p.out[0][(size_t)r * N + n] = v + __ldcg(p.res + (size_t)r * N + n);
                } else if (mi == 0) {  // EPI_SWIGLU: gate tile tl, up tile tl + 1 (same slice)
                    const float u = m.red[idx - i0 + tile_vals];
                    p.out[0][(size_t)r * N + n] = v / (1.0f + expf(-v)) * u;
                }
            }
        }
    }
}

// Single K-slice logits job: this group's (max, index) per activation row
// over its folded outputs (and the outputs themselves when asked for).
template <int CLS>
__device__ void argmax_epilogue(const GemvParams &p, const Geo &q, const Smem &m, int group, int tid, int warp,
                                int lane) {
    constexpr int NW = Cls<CLS>::NW, NTH = NW * 32;
    const int nb = CLS == 0 ? 1 : p.nb;
    if (group >= p.groups) return;  // no tiles, no partials
    const int N = p.n[0];
    float *bvs = m.rbuf;  // [warp]
    int *bis = reinterpret_cast<int *>(m.rbuf + NW);
    WarpTable<NW> wt;
    wt.load(m.wtab);
    for (int r = 0; r < nb; ++r) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int ri = tid; ri < q.tiles_here * kTileRows; ri += NTH) {
            const int n = (q.t0 + ri / kTileRows) * kTileRows + (ri % kTileRows);
            if (n >= N) continue;
            const float v = fold_one<CLS>(p, q, m, wt, ri / kTileRows, ri % kTileRows, r, nb) * m.nx[5 * kMaxNb + r];
            if (p.out[0] != nullptr) p.out[0][(size_t)r * N + n] = v;
            am_take(bv, bi, v, n);
        }
        am_warp(bv, bi);
        if (lane == 0) {
            bvs[warp] = bv;
            bis[warp] = bi;
        }
        csync<NW>();
        if (tid == 0) {
            float fv = bvs[0];
            int fi = bis[0];
            for (int w = 1; w < NW; ++w) {
                if (bvs[w] > fv || (bvs[w] == fv && bis[w] < fi)) {
                    fv = bvs[w];
                    fi = bis[w];
                }
            }
            p.am_val[(size_t)r * p.groups + group] = fv;
            p.am_idx[(size_t)r * p.groups + group] = fi;
        }
        csync<NW>();
    }
}

// The residual a folding thread adds to its first output (fold_store's
// thread mapping), loaded as soon as the job starts so that its latency is
// hidden behind the staging and the unit loop; 0 when there is none.
template <int CLS>
__device__ __forceinline__ float residual_prefetch(const GemvParams &p, const Geo &q, int tid) {
    constexpr int NTH = Cls<CLS>::NW * 32;
    const int nb = CLS == 0 ? 1 : p.nb;
    const int tile_vals = kTileRows * nb;
    const int tp0 = tid / tile_vals, rem = tid - tp0 * tile_vals;
    const int row = rem / nb, r = rem - row * nb;
    if (p.epi != EPI_RESIDUAL || tp0 >= NTH / tile_vals || tp0 >= q.tiles_here) return 0.f;
    const int n = (q.t0 + tp0) * kTileRows + row;  // single-matrix job
    return n < p.n[0] ? __ldcg(p.res + (size_t)r * p.n[0] + n) : 0.f;
}

// Single K-slice, store / residual / SwiGLU jobs: fold each output's warp
// partials and write it at once.  res0: this thread's first residual, from
// residual_prefetch.
template <int CLS>
__device__ void fold_store(const GemvParams &p, const Geo &q, const Smem &m, int group, int tid, float res0) {
    constexpr int NTH = Cls<CLS>::NW * 32;
    const int nb = CLS == 0 ? 1 : p.nb;
    if (group >= p.groups) return;  // no tiles
    WarpTable<Cls<CLS>::NW> wt;
    wt.load(m.wtab);
    const int tile_vals = kTileRows * nb;
    const bool pairs = p.epi == EPI_SWIGLU;
    const int ntp = pairs ? q.tiles_here / 2 : q.tiles_here;  // tiles, or gate/up pairs
    // thread tid handles output `rem` of tiles (pairs) tp0, tp0 + per, ...
    const int per = NTH / tile_vals;
    const int tp0 = tid / tile_vals, rem = tid - tp0 * tile_vals;
    const int row = rem / nb, r = rem - row * nb;
    for (int tp = tp0 < per ? tp0 : ntp; tp < ntp; tp += per) {
        const int tl = pairs ? 2 * tp : tp;
        int mi, tm;
        map_tile(p, q.t0 + tl, mi, tm);
        const int n = tm * kTileRows + row;
        const int N = p.n[mi];
        if (n >= N) continue;
        const float f = m.nx[5 * kMaxNb + r];
        const float v = fold_one<CLS>(p, q, m, wt, tl, row, r, nb) * f;
        if (p.epi == EPI_STORE) {
            p.out[mi][(size_t)r * N + n] = v;
        } else if (p.epi == EPI_RESIDUAL) {
            p.out[0][(size_t)r * N + n] = v + (tp == tp0 ? res0 : __ldcg(p.res + (size_t)r * N + n));
        } else {  // SwiGLU: gate tile, then its up tile
            const float u = fold_one<CLS>(p, q, m, wt, tl + 1, row, r, nb) * f;
            p.out[0][(size_t)r * N + n] = v / (1.0f + expf(-v)) * u;
        }
    }
    csync<Cls<CLS>::NW>();
}

// Copy a job's parameter block into shared memory with one round of
// independent 8-byte loads (a first touch of the constant bank costs a
// miss per line; this takes them all at once).  Visible after a barrier.
static_assert(sizeof(GemvParams) % 8 == 0, "parameter block must be whole 8-byte words");
constexpr int kParamWords = (int)(sizeof(GemvParams) / 8);
__device__ __forceinline__ void copy_params(GemvParams *dst, const GemvParams *src, int tid) {
    if (tid < kParamWords)
        reinterpret_cast<unsigned long long *>(dst)[tid] = reinterpret_cast<const unsigned long long *>(src)[tid];
}

// ---------------------------------------------------------------------------
// Per-call kernel: one job, one group of tile pairs per cluster.
template <int FMT, int CLS>
__global__ void __launch_bounds__(Cls<CLS>::NW * 32, 1) q4gemv_engine_kernel(const __grid_constant__ GemvParams prm) {
    using C = Cls<CLS>;
    constexpr int REC = rec_bytes(FMT);
    constexpr int NW = C::NW;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ GemvParams ps;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    copy_params(&ps, &prm, tid);
    __syncthreads();
    const GemvParams &p = ps;
    const int S = p.S;
    const int group = blockIdx.x / S, rank = blockIdx.x - group * S;
    const int nb = CLS == 0 ? 1 : p.nb;
    const Smem m = carve<CLS>(smem, nb, p.Cs, p.TG, p.SW, S);
    RingOf<FMT, CLS> ring;
    ring.init(smem_u32(m.ring) + warp * C::DU * 2 * stage_su(FMT, CLS) * REC, smem_u32(m.bars) + warp * C::DU * 8, lane,
              p.wait_cycles, p.extra_tx);
    // this CTA has started; the matching wait ends the activation staging
    if (S > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    // the next kernel may launch now; it waits for this one before it reads
    // what this one writes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // weights do not depend on the previous kernel: each warp starts its
    // first stage's copies before waiting for it, and the rest of its ring
    // once the activations are staged (with the whole ring in flight the
    // staging's activation loads wait behind the copies: 9.6 against 8.9 us
    // for the 14336 x 4096 matvec)
    const Geo q = make_geo<NW>(p, group, rank, warp);
    StreamOf<FMT, CLS> ws;
    ws.init_one(&p, q);
    ring.push(ws, lane);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float res0 = S == 1 ? residual_prefetch<CLS>(p, q, tid) : 0.f;

    stage_x<FMT, CLS, CLS == 3 ? 8 : 4, CLS != 0>(p, q, m, S, tid, warp, lane);
    for (int s = 1; s < C::DU; ++s) ring.push(ws, lane);
    run_units<FMT, CLS, true>(p, q, m, ws, ring, warp, lane, true);
    ring.drain();
    __syncthreads();
    if (S == 1 && p.epi != EPI_ARGMAX) {
        fold_store<CLS>(p, q, m, group, tid, res0);
        return;
    }
    if (S > 1) {
        cluster_finish<CLS>(p, q, m, S, rank, group, tid, warp, lane);
        return;
    }
    argmax_epilogue<CLS>(p, q, m, group, tid, warp, lane);
}

}  // namespace dev
}  // namespace q4
#include "step_attn.cuh"
namespace q4 {
namespace dev {

// ---------------------------------------------------------------------------
// Persistent decode-step kernel: one CTA per SM runs the step's jobs in
// order, separated by grid-wide barriers; the weight stream of every warp
// runs ahead across job boundaries, so weights keep arriving while the CTA
// waits at a barrier or stages the next job's activations.

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier number `b` (1-based) over the NW warps of every CTA.  Each
// CTA adds one to the arrival counter with a release reduction (no reply to
// wait for), then polls the counter with acquire loads until all
// b * gridDim.x (+ extra) arrivals are in.  The wait is bounded: after
// `polls` polls the CTA records the failure in *err and the caller stops.
// Between its arrival and its wait, each warp runs `work` (the persistent
// kernel refills its weight ring there).
template <int NW, class Work>
__device__ __forceinline__ bool grid_barrier(unsigned *counter, int *err, unsigned b, long long polls,
                                             unsigned extra, Work &&work) {
    csync<NW>();
    __shared__ int fail;
    if (threadIdx.x == 0) {
        fail = 0;
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
    }
    work();
    if (threadIdx.x == 0) {
        const unsigned target = b * gridDim.x + extra;
        long long it = 0;
        while (ld_acquire_u32(counter) < target) {
            if (++it > polls) {
                atomicExch(err, 1);
                fail = 1;
                break;
            }
        }
    }
    csync<NW>();
    return fail == 0;
}

// ATT: the jobs include the layers' decode attention (EPI_ATTN jobs,
// q4_decode_step_attn; nb = 1), each run by step_attn_job.  Without it the
// kernel is the stand-in step's, unchanged.
template <int FMT, int CLS, bool ATT>
__global__ void __launch_bounds__(Cls<CLS>::NW * 32, 1) q4gemv_step_kernel(const __grid_constant__ StepParams sp) {
    using C = Cls<CLS>;
    constexpr int REC = rec_bytes(FMT);
    constexpr int NW = C::NW;
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int group = blockIdx.x;
    const int nb = CLS == 0 ? 1 : sp.nb;
    const int cs_max = (sp.Kmax + kChunkK - 1) / kChunkK;  // as the host sized it
    const Smem m = carve<CLS>(smem, nb, cs_max, sp.TGmax, sp.SWmax, 1);
    RingOf<FMT, CLS> ring;
    ring.init(smem_u32(m.ring) + warp * C::DU * 2 * stage_su(FMT, CLS) * REC, smem_u32(m.bars) + warp * C::DU * 8, lane,
              sp.jobs[0].wait_cycles, sp.jobs[0].extra_tx);

    // every job's parameter block in shared memory (after the engine's
    // regions), copied once: the weight stream and the job loop read them there
    GemvParams *jobs = reinterpret_cast<GemvParams *>(m.ring + (size_t)NW * C::DU * 2 * stage_su(FMT, CLS) * REC);
    for (int i = tid; i < sp.njobs * kParamWords; i += NW * 32)
        reinterpret_cast<unsigned long long *>(jobs)[i] = reinterpret_cast<const unsigned long long *>(sp.jobs)[i];
    csync<NW>();
    // and this group's span of every job (the divisions, once)
    JobSpan *spans = reinterpret_cast<JobSpan *>(jobs + sp.njobs);
    for (int j = tid; j < sp.njobs; j += NW * 32) spans[j] = span_of(jobs[j], group);
    csync<NW>();
    StreamOf<FMT, CLS> ws;
    ws.init(jobs, spans, sp.njobs, group, 0, warp);
    for (int s = 0; s < C::DU; ++s) ring.push(ws, lane);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // at a grid barrier: refill every free slot, moving across jobs
    auto refill = [&]() {
        while (ring.push(ws, lane)) {
        }
    };

    for (int j = 0; j < sp.njobs; ++j) {
        const GemvParams &p = jobs[j];
        if (j > 0 &&
            !grid_barrier<NW>(sp.counter, sp.err, (unsigned)j, sp.barrier_polls, (unsigned)sp.barrier_extra, refill)) {
            ring.drain();
            return;
        }
        if constexpr (ATT) {
            if (p.epi == EPI_ATTN) {  // CTA-uniform
                step_attn_job<NW>(sp.att, p.layer, m.xs, group, tid, warp, lane);
                continue;
            }
        }
        const Geo q = geo_of<NW>(p, spans[j], 0, warp);
        if (q.tiles_here == 0) continue;  // no work in this job (CTA-uniform)
        const float res0 = residual_prefetch<CLS>(p, q, tid);
        stage_x<FMT, CLS, 4, false>(p, q, m, 1, tid, warp, lane);
        run_units<FMT, CLS, false>(p, q, m, ws, ring, warp, lane, false);
        csync<NW>();
        if (p.epi != EPI_ARGMAX) {
            fold_store<CLS>(p, q, m, group, tid, res0);
        } else {
            argmax_epilogue<CLS>(p, q, m, group, tid, warp, lane);
        }
    }
    ring.drain();
    // the last job is the logits argmax: fold the groups' pairs in order
    if (!grid_barrier<NW>(sp.counter, sp.err, (unsigned)sp.njobs, sp.barrier_polls, (unsigned)sp.barrier_extra,
                          [] {}))
        return;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const GemvParams &pl = jobs[sp.njobs - 1];
    if (group == 0 && tid < 32) {
        for (int r = 0; r < nb; ++r) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int i = lane; i < pl.groups; i += 32) {
                const float v = __ldcg(pl.am_val + (size_t)r * pl.groups + i);
                const int k = __ldcg(pl.am_idx + (size_t)r * pl.groups + i);
                if (v > bv || (v == bv && k < bi)) {
                    bv = v;
                    bi = k;
                }
            }
            am_warp(bv, bi);
            if (lane == 0) {
                sp.idx[r] = bi;
                if (sp.val) sp.val[r] = bv;
            }
        }
    }
}

}  // namespace dev
}  // namespace q4
