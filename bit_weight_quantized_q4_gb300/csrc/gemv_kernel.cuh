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
//  * One CTA = 8 warps owns a group of 16-row tiles and one K-slice, at most
//    one CTA per SM; a thread-block cluster of S CTAs splits K and folds its
//    partial sums over distributed shared memory in rank order
//    (deterministic, no atomics).
//  * At kernel start each CTA lets the next kernel in the stream launch and
//    starts its first weight copies (and loads gamma); only then does it wait
//    for the previous kernel.  Each warp streams its contiguous range of
//    (tile, chunk) records through a private shared-memory ring with 16-byte
//    cp.async copies, seven records in flight per warp.
//  * Each 32-bit nibble word becomes four f16x2 registers of (q - 8) (or q)
//    with one lop3 and one packed fma each -- exact integers in f16.
//  * Activations are staged once per CTA in shared memory as an exact
//    power-of-two-scaled hi + lo pair of f16 values (about 22 significant
//    bits), laid out so each lane loads its mma B fragment with one 64-bit
//    shared load.
//  * mma.sync m16n8k16 (f16 in, fp32 accumulate) forms the per-block dot
//    products of 16 rows x 8 activation rows, the hi and lo halves as two
//    k-steps into the same accumulator; each block's result is scaled by its
//    fp32 scale and accumulated in fp32, so weights are never rounded.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cooperative_groups.h>
#include <math.h>

#include "q4_internal.h"

namespace q4 {
namespace dev {

namespace cg = cooperative_groups;

// 128-bit streaming load: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ldg_stream(const uint8_t *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte asynchronous copy global -> shared (L2 only), and its group fences.
__device__ __forceinline__ void cp_async16(uint8_t *dst, const uint8_t *src) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
template <int OFF>
__device__ __forceinline__ void cp_async16_at(uint32_t dst, const uint8_t *src) {
    asm volatile("cp.async.cg.shared.global [%0+%2], [%1+%2], 16;" ::"r"(dst), "l"(src), "n"(OFF) : "memory");
}
template <int OFF>
__device__ __forceinline__ uint4 lds128_at(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+%5];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a), "n"(OFF)
                 : "memory");
    return v;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// (a & b) | c
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
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

// One nibble word -> four f16x2 registers holding (q - 8) for Q4_0 or q for
// affine, exactly.  OR-ing a nibble into the mantissa of f16 1024.0 gives
// 1024 + q (or 1024 + 16q for the upper nibble of a byte), and one packed
// fma removes the bias (and the 16x):
//   r0 = (nib0, nib4)  r1 = (nib1, nib5)  r2 = (nib2, nib6)  r3 = (nib3, nib7)
template <int FMT>
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
    const uint32_t kMagic = 0x64006400u;                                // 1024.0
    const uint32_t kOne = 0x3C003C00u;                                  // 1.0
    const uint32_t kSixteenth = 0x2C002C00u;                            // 1/16
    const uint32_t kBiasLo = FMT == 0 ? 0xE408E408u : 0xE400E400u;      // -1032 / -1024
    const uint32_t kBiasHi = FMT == 0 ? 0xD480D480u : 0xD400D400u;      // -72 / -64
    const uint32_t w8 = w >> 8;
    r0 = hfma2(lop3_and_or(w, 0x000F000Fu, kMagic), kOne, kBiasLo);
    r1 = hfma2(lop3_and_or(w, 0x00F000F0u, kMagic), kSixteenth, kBiasHi);
    r2 = hfma2(lop3_and_or(w8, 0x000F000Fu, kMagic), kOne, kBiasLo);
    r3 = hfma2(lop3_and_or(w8, 0x00F000F0u, kMagic), kSixteenth, kBiasHi);
}

// The two 16-bit scales (or mins) of a scale word as fp32.
template <int FMT>
__device__ __forceinline__ float2 scale_pair(uint32_t w) {
    if (FMT == 0) {
        __half2 h = *reinterpret_cast<const __half2 *>(&w);
        return __half22float2(h);
    } else {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
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
// Within a job, group g of `groups` owns a contiguous range of 16-row tiles
// (gate/up pairs for SwiGLU) and cluster rank r its K-slice; the CTA's
// (tile, chunk) records are split into contiguous ranges, one per warp.

struct Geo {
    int t0, tiles_here;              // this group's tiles [t0, t0 + tiles_here)
    int c0, cs_here, Ks, kb, ke;     // K-slice: chunks [c0, c0 + cs_here), columns [kb, ke)
    int U, ub, ue, n_my, first_tl;   // records of the CTA; this warp's [ub, ue)
};

template <int NW>
__device__ __forceinline__ Geo make_geo(const GemvParams &p, int group, int rank, int warp) {
    Geo q;
    const int pw = p.mode == MODE_PAIRS ? 2 : 1;
    const int P = p.T / pw;
    if (group < p.groups) {
        q.t0 = (int)(((long long)group * P) / p.groups) * pw;
        const int t1 = (int)(((long long)(group + 1) * P) / p.groups) * pw;
        q.tiles_here = t1 - q.t0;
    } else {  // a job with fewer tile units than CTAs: this CTA has none
        q.t0 = 0;
        q.tiles_here = 0;
    }
    q.c0 = rank * p.Cs;
    q.cs_here = max(0, min(p.Cs, p.C - q.c0));
    q.Ks = p.Cs * kChunkK;
    q.kb = q.c0 * kChunkK;
    q.ke = min(p.K, q.kb + q.Ks);
    q.U = q.tiles_here * q.cs_here;
    q.ub = (warp * q.U) / NW;
    q.ue = ((warp + 1) * q.U) / NW;
    q.n_my = q.ue - q.ub;
    q.first_tl = q.cs_here > 0 ? q.ub / q.cs_here : 0;
    return q;
}

template <int REC>
__device__ __forceinline__ const uint8_t *tile_ptr(const GemvParams &p, int t0, int c0, int tl) {
    int m, tm;
    map_tile(p, t0 + tl, m, tm);
    return p.w[m] + ((size_t)tm * p.C + (size_t)c0) * REC;
}

// The weight records a warp streams, in order, across the jobs of a launch:
// each job's [ub, ue) range of this warp, job after job.  The load side runs
// up to DEPTH-1 records ahead of the compute side, across job boundaries.
template <int REC, int NW>
struct WeightStream {
    const GemvParams *jobs;
    int njobs, group, rank, warp;
    int job, t0, c0, cs, tl, c, left, tiles;
    const uint8_t *ptr;

    __device__ __forceinline__ void next_job() {
        while (left == 0 && job + 1 < njobs) {
            ++job;
            const Geo q = make_geo<NW>(jobs[job], group, rank, warp);
            if (q.n_my > 0) {
                t0 = q.t0;
                c0 = q.c0;
                cs = q.cs_here;
                tiles = q.tiles_here;
                tl = q.first_tl;
                c = q.ub - tl * cs;
                left = q.n_my;
                ptr = tile_ptr<REC>(jobs[job], t0, c0, tl) + (size_t)c * REC;
            }
        }
    }
    __device__ __forceinline__ void init(const GemvParams *j, int n, int grp, int rk, int w) {
        jobs = j;
        njobs = n;
        group = grp;
        rank = rk;
        warp = w;
        job = -1;
        left = 0;
        ptr = nullptr;
        next_job();
    }
    // copy the next record into the ring stage at shared address `dst`:
    // each lane its two 16-byte nibble pieces, lanes 0..7 (0..15 affine) the
    // scale (and min) words
    __device__ __forceinline__ void issue(uint32_t dst, int lane) {
        const uint8_t *src = ptr + lane * 16;
        const uint32_t d = dst + lane * 16;
        cp_async16_at<0>(d, src);
        cp_async16_at<512>(d, src);
        if (lane < (REC - 1024) / 16) cp_async16_at<1024>(d, src);
        ptr += REC;
        --left;
        if (++c == cs) {
            c = 0;
            if (++tl < tiles && left > 0) ptr = tile_ptr<REC>(jobs[job], t0, c0, tl);
        }
        if (left == 0) next_job();
    }
};

// Shared-memory regions of one CTA (sizes: engine_smem()).
struct Smem {
    uint8_t *xs;     // activation slice, hi/lo f16 in mma B-fragment order
    float *gs;       // affine: group sums [blocks][GSW]
    float *red;      // CTA results [TG][16][nb]
    float *slots;    // per-warp tile partials [warp][TG][16][nb]
    float *rbuf;     // reductions [4][warp][kMaxNb]
    float *nx;       // row stats [8][kMaxNb]: 2 inv_rms, 3 scale, 5 inv_scale
    uint8_t *ring;   // weight records [warp][DEPTH][REC]
};

template <int NW>
__device__ __forceinline__ Smem carve(uint8_t *smem, int fmt, int nb, int Cs, int GSW, int TG) {
    Smem m;
    m.xs = smem;
    m.gs = reinterpret_cast<float *>(smem + (size_t)4 * nb * Cs * kChunkK);
    m.red = m.gs + (fmt == 1 ? Cs * kBlocksPerChunk * GSW : 0);
    m.slots = m.red + TG * kTileRows * nb;
    m.rbuf = m.slots + NW * TG * kTileRows * nb;
    m.nx = m.rbuf + 4 * NW * kMaxNb;
    m.ring = reinterpret_cast<uint8_t *>(m.nx + 8 * kMaxNb);
    return m;
}

// The activation scale of a row: 2^e with bound * 2^e in [2^14, 2^15), from
// the exponent field of `bound` (e clamped to [-100, 100]; 1 for 0 or
// non-finite bounds; subnormal bounds take the clamp).
__device__ __forceinline__ void row_scale(float bound, float &scale, float &inv_scale) {
    scale = 1.f;
    inv_scale = 1.f;
    if (bound > 0.f && bound <= 3.0e38f) {
        const int be = (int)((__float_as_uint(bound) >> 23) & 0xFF);  // bound in [2^(be-127), 2^(be-126))
        int e = 14 - (be - 127);
        e = max(-100, min(100, e));
        scale = __uint_as_float((uint32_t)(127 + e) << 23);
        inv_scale = __uint_as_float((uint32_t)(127 - e) << 23);
    }
}

// Stage this CTA's activation slice of job p: per row, scale by a power of
// two chosen from its largest magnitude (after RMSNorm when gamma is given)
// and split into f16 hi + lo, stored in B-fragment order:
//   per 32-column block: [n-tile][k16 step][lane g*4+t][hi(k=2t,2t+1), hi(2t+8,2t+9), lo(..), lo(..)]
// Activation loads bypass L1 (.cg): in the persistent kernel another SM may
// have rewritten them since this SM last read them.
template <int FMT, int NT, bool NB1, int NW>
__device__ void stage_x(const GemvParams &p, const Geo &q, const Smem &m, int S, int tid, int warp, int lane) {
    constexpr int GSW = 8 * NT;
    constexpr int NTH = NW * 32;
    const int nb = NB1 ? 1 : p.nb;
    const int Ks = q.Ks, kb = q.kb, ke = q.ke;
    const int xbs = 128 * nb;
    const bool norm = p.gamma != nullptr;
    constexpr int RP = 8192 / (2 * NTH);  // nb == 1: a slice up to 8192 columns passes through registers
    if (NB1 && Ks <= 2 * NTH * RP) {
        const int npass = (Ks / 2 + NTH - 1) / NTH;  // pairs per thread actually used
        float2 xv[RP], gv[RP];
        float ss = 0.f, mx = 0.f;
#pragma unroll
        for (int qq = 0; qq < RP; ++qq) {
            if (qq >= npass) break;
            float2 v = make_float2(0.f, 0.f), gm = make_float2(1.f, 1.f);
            const int k = kb + 2 * (tid + qq * NTH);
            if (k < ke) {
                v = __ldcg(reinterpret_cast<const float2 *>(p.x + k));
                if (norm) gm = *reinterpret_cast<const float2 *>(p.gamma + k);
            }
            xv[qq] = v;
            gv[qq] = gm;
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            mx = fmaxf(mx, fmaxf(fabsf(norm ? v.x * gm.x : v.x), fabsf(norm ? v.y * gm.y : v.y)));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        }
        if (lane == 0) {
            m.rbuf[warp] = ss;
            m.rbuf[NW + warp] = mx;
        }
        __syncthreads();
        float tss = 0.f, tmx = 0.f;  // every thread adds the warps in the same order
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            tss += m.rbuf[w];
            tmx = fmaxf(tmx, m.rbuf[NW + w]);
        }
        if (norm && S > 1) {
            // the RMS needs the whole row: add the slices' sums in rank order
            cg::cluster_group cluster = cg::this_cluster();
            if (tid == 0) m.nx[0] = tss;
            cluster.sync();
            tss = 0.f;
            for (int r = 0; r < S; ++r) tss += cluster.map_shared_rank(m.nx, r)[0];
        }
        const float inv_rms = norm ? 1.0f / sqrtf(tss / (float)p.K + p.eps) : 1.f;
        float scale, inv_scale;
        row_scale(tmx * inv_rms, scale, inv_scale);
        if (tid == 0) {
            m.nx[2 * kMaxNb] = inv_rms;
            m.nx[3 * kMaxNb] = scale;
            m.nx[5 * kMaxNb] = inv_scale;
        }
#pragma unroll
        for (int qq = 0; qq < RP; ++qq) {
            if (qq >= npass) break;
            const int kl = 2 * (tid + qq * NTH);
            if (kl < Ks) {
                float v0 = xv[qq].x, v1 = xv[qq].y;
                if (norm) {
                    v0 = v0 * inv_rms * gv[qq].x;
                    v1 = v1 * inv_rms * gv[qq].y;
                }
                v0 *= scale;
                v1 *= scale;
                __half2 hi = __floats2half2_rn(v0, v1);
                float2 hf = __half22float2(hi);
                __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
                const int kk = kl & 31, k16 = kk & 15;
                const int off = (kl >> 5) * 128 + (kk >> 4) * 64 + ((k16 & 7) >> 1) * 16 + (k16 >> 3) * 4;
                *reinterpret_cast<__half2 *>(m.xs + off) = hi;
                *reinterpret_cast<__half2 *>(m.xs + off + 8) = lo;
            }
        }
        if (FMT == 1) {
            const int nblk = p.Cs * kBlocksPerChunk;
            for (int i = tid; i < GSW * nblk; i += NTH) {
                const int r = i / nblk, bl = i - r * nblk;
                const int kblk = kb + 32 * bl;
                float sacc = 0.f;
                if (r == 0 && kblk < ke) {
                    if (p.gsum != nullptr && !norm) {
                        sacc = __ldcg(p.gsum + kblk / 32);
                    } else {
                        float vv[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) vv[e] = __ldcg(p.x + kblk + e);
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            float v = vv[e];
                            if (norm) v = v * inv_rms * p.gamma[kblk + e];
                            sacc += v;
                        }
                    }
                    sacc *= scale;
                }
                m.gs[bl * GSW + r] = sacc;
            }
        }
        __syncthreads();
        return;
    }
    // general nb: two passes over the slice
    for (int r = 0; r < nb; ++r) {
        float ss = 0.f, mx = 0.f;
        const float *xr = p.x + (size_t)r * p.K;
        for (int k = kb + 2 * tid; k < ke; k += 2 * NTH) {
            float2 v = __ldcg(reinterpret_cast<const float2 *>(xr + k));
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            if (norm) {
                float2 gm = *reinterpret_cast<const float2 *>(p.gamma + k);
                mx = fmaxf(mx, fmaxf(fabsf(v.x * gm.x), fabsf(v.y * gm.y)));
            } else {
                mx = fmaxf(mx, fmaxf(fabsf(v.x), fabsf(v.y)));
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        }
        if (lane == 0) {
            m.rbuf[warp * kMaxNb + r] = ss;
            m.rbuf[NW * kMaxNb + warp * kMaxNb + r] = mx;
        }
    }
    __syncthreads();
    if (tid < nb) {
        float ss = 0.f, mx = 0.f;
        for (int w = 0; w < NW; ++w) {
            ss += m.rbuf[w * kMaxNb + tid];
            mx = fmaxf(mx, m.rbuf[NW * kMaxNb + w * kMaxNb + tid]);
        }
        m.nx[0 * kMaxNb + tid] = ss;  // this slice's sum of squares
        m.nx[1 * kMaxNb + tid] = mx;
    }
    if (norm && S > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (tid < nb) {
            float tot = 0.f;
            for (int r = 0; r < S; ++r) tot += cluster.map_shared_rank(m.nx, r)[tid];
            m.nx[4 * kMaxNb + tid] = tot;
        }
    } else if (tid < nb) {
        m.nx[4 * kMaxNb + tid] = m.nx[tid];
    }
    __syncthreads();
    if (tid < nb) {
        float inv_rms = 1.f;
        if (norm) inv_rms = 1.0f / sqrtf(m.nx[4 * kMaxNb + tid] / (float)p.K + p.eps);
        float scale, inv_scale;
        row_scale(m.nx[1 * kMaxNb + tid] * inv_rms, scale, inv_scale);
        m.nx[2 * kMaxNb + tid] = inv_rms;
        m.nx[3 * kMaxNb + tid] = scale;
        m.nx[5 * kMaxNb + tid] = inv_scale;
    }
    __syncthreads();
    const int half_ks = Ks >> 1;
    for (int i = tid; i < nb * half_ks; i += NTH) {
        const int r = i / half_ks, kp = i - r * half_ks;
        const int kl = 2 * kp, k = kb + kl;
        float v0 = 0.f, v1 = 0.f;
        if (k < ke) {
            float2 v = __ldcg(reinterpret_cast<const float2 *>(p.x + (size_t)r * p.K + k));
            v0 = v.x;
            v1 = v.y;
            if (norm) {
                const float ir = m.nx[2 * kMaxNb + r];
                float2 gm = *reinterpret_cast<const float2 *>(p.gamma + k);
                v0 = v0 * ir * gm.x;
                v1 = v1 * ir * gm.y;
            }
        }
        const float sc = m.nx[3 * kMaxNb + r];
        v0 *= sc;
        v1 *= sc;
        __half2 hi = __floats2half2_rn(v0, v1);
        float2 hf = __half22float2(hi);
        __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
        const int bl = kl >> 5, kk = kl & 31, st = kk >> 4, k16 = kk & 15;
        const int nt = r >> 3, cols = min(8, nb - 8 * nt);
        const int off = bl * xbs + nt * 1024 + st * 64 * cols + (4 * (r & 7) + ((k16 & 7) >> 1)) * 16 +
                        (k16 >> 3) * 4;
        *reinterpret_cast<__half2 *>(m.xs + off) = hi;
        *reinterpret_cast<__half2 *>(m.xs + off + 8) = lo;
    }
    if (FMT == 1) {
        const int nblk = p.Cs * kBlocksPerChunk;
        for (int i = tid; i < GSW * nblk; i += NTH) {
            const int r = i / nblk, bl = i - r * nblk;
            const int kblk = kb + 32 * bl;
            float s = 0.f;
            if (r < nb && kblk < ke) {
                if (p.gsum != nullptr && !norm) {
                    s = __ldcg(p.gsum + (size_t)r * (p.K / 32) + kblk / 32);
                } else {
                    const float *xr = p.x + (size_t)r * p.K + kblk;
                    const float ir = m.nx[2 * kMaxNb + r];
                    float vv[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) vv[e] = __ldcg(xr + e);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float v = vv[e];
                        if (norm) v = v * ir * p.gamma[kblk + e];
                        s += v;
                    }
                }
                s *= m.nx[3 * kMaxNb + r];
            }
            m.gs[bl * GSW + r] = s;
        }
    }
    __syncthreads();
}

// This warp's records of one job: dequantise, tensor-core dot products,
// per-block scaling; each tile's partial goes to this warp's slot.
// Consumes one ring stage per record and refills it from `ws`.
template <int FMT, int NT, bool NB1, int DEPTH, int NW>
__device__ void run_units(const GemvParams &p, const Geo &q, const Smem &m,
                          WeightStream<FMT == 0 ? kRecQ4_0 : kRecAffine, NW> &ws, uint32_t &st_a, uint32_t &fill_a,
                          uint32_t ring_a, int warp, int lane) {
    constexpr int REC = FMT == 0 ? kRecQ4_0 : kRecAffine;
    constexpr int GSW = 8 * NT;
    const int g = lane >> 2, tq = lane & 3;
    const int nb = NB1 ? 1 : p.nb;
    const int xbs = 128 * nb;
    const int cs_here = q.cs_here;
    const uint32_t ring_end = ring_a + DEPTH * REC;
    // lanes beyond the batch read a duplicate column: its mma outputs are
    // never stored, and every lane loads unconditionally
    const uint32_t xs_a = smem_u32(m.xs);
    uint32_t xoff[NT];
    int hstr[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int cols = min(8, nb - 8 * nt);
        xoff[nt] = xs_a + nt * 1024 + (4 * (g % cols) + tq) * 16;
        hstr[nt] = 64 * cols;
    }
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    int ctl = q.first_tl, cc = q.ub - q.first_tl * cs_here;
    const float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
    float *my_slots = m.slots + (size_t)warp * p.TG * kTileRows * nb;

    auto flush = [&](int tl) {
        float *dst = my_slots + (size_t)tl * kTileRows * nb;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int a0 = 8 * j + 2 * tq;
            if (a0 < nb) {
                dst[g * nb + a0] = acc[j][0];
                dst[(g + 8) * nb + a0] = acc[j][2];
            }
            if (!NB1 && a0 + 1 < nb) {
                dst[g * nb + a0 + 1] = acc[j][1];
                dst[(g + 8) * nb + a0 + 1] = acc[j][3];
            }
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        }
    };

    // One 32-column block: two nibble words (rows g, g+8) -> A fragments;
    // per n-tile two 16-byte B loads and four mma (hi and lo halves of both
    // k16 steps); the block scale applied in fp32.
    auto block = [&](uint32_t w0, uint32_t w1, uint32_t scw, uint32_t mnw, uint32_t xblk, int blk) {
        uint32_t a[8];
        unpack_word<FMT>(w0, a[0], a[2], a[4], a[6]);  // row g
        unpack_word<FMT>(w1, a[1], a[3], a[5], a[7]);  // row g + 8
        const float2 d = scale_pair<FMT>(scw);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint32_t xa = xblk + xoff[nt];
            uint4 b0, b1;
            if (NB1) {
                b0 = lds128_at<0>(xa);
                b1 = lds128_at<64>(xa);
            } else {
                b0 = lds128_at<0>(xa);
                b1 = lds128_at<0>(xa + hstr[nt]);
            }
            float dd[4];
            mma16816_c(dd, a[0], a[1], a[2], a[3], b0.x, b0.y, z0, z1, z2, z3);  // k 0..15, hi
            mma16816(dd, a[0], a[1], a[2], a[3], b0.z, b0.w);                      // k 0..15, lo
            mma16816(dd, a[4], a[5], a[6], a[7], b1.x, b1.y);                      // k 16..31, hi
            mma16816(dd, a[4], a[5], a[6], a[7], b1.z, b1.w);                      // k 16..31, lo
            acc[nt][0] = fmaf(d.x, dd[0], acc[nt][0]);
            acc[nt][2] = fmaf(d.y, dd[2], acc[nt][2]);
            if (!NB1) {
                acc[nt][1] = fmaf(d.x, dd[1], acc[nt][1]);
                acc[nt][3] = fmaf(d.y, dd[3], acc[nt][3]);
            }
            if (FMT == 1) {
                const float2 mm = scale_pair<FMT>(mnw);
                const float2 gv = *reinterpret_cast<const float2 *>(m.gs + blk * GSW + 8 * nt + 2 * tq);
                acc[nt][0] = fmaf(mm.x, gv.x, acc[nt][0]);
                acc[nt][2] = fmaf(mm.y, gv.x, acc[nt][2]);
                if (!NB1) {
                    acc[nt][1] = fmaf(mm.x, gv.y, acc[nt][1]);
                    acc[nt][3] = fmaf(mm.y, gv.y, acc[nt][3]);
                }
            }
        }
    };

    for (int i = 0; i < q.n_my; ++i) {
        cp_async_wait<DEPTH - 2>();  // this lane's copies of the record have landed
        __syncwarp();                 // ... and every lane's; the previous stage is free
        if (ws.left > 0) ws.issue(fill_a, lane);
        cp_async_commit();
        fill_a += REC;
        if (fill_a == ring_end) fill_a = ring_a;
        const uint4 q0 = lds128_at<0>(st_a + lane * 16);
        const uint4 q1 = lds128_at<512>(st_a + lane * 16);
        const uint4 sc = lds128_at<1024>(st_a + g * 16);
        uint4 mn = make_uint4(0u, 0u, 0u, 0u);
        if (FMT == 1) mn = lds128_at<1152>(st_a + g * 16);
        st_a += REC;
        if (st_a == ring_end) st_a = ring_a;
        const uint32_t xu = (uint32_t)(cc * kBlocksPerChunk * xbs);
        const int blk0 = cc * kBlocksPerChunk;
        block(q0.x, q1.x, sc.x, mn.x, xu, blk0);
        block(q0.y, q1.y, sc.y, mn.y, xu + xbs, blk0 + 1);
        block(q0.z, q1.z, sc.z, mn.z, xu + 2 * xbs, blk0 + 2);
        block(q0.w, q1.w, sc.w, mn.w, xu + 3 * xbs, blk0 + 3);
        if (++cc == cs_here) {  // end of this tile's slice: hand the tile over
            flush(ctl);
            cc = 0;
            ++ctl;
        }
    }
    if (q.n_my > 0 && cc != 0) flush(ctl);  // the range ended inside a tile
}

// Sum the warps' partials of each tile in warp order (only the warps whose
// record range touched the tile), undo the activation scale; then (cluster)
// fold the K-slices into rank 0.  Returns false on cluster ranks other than
// 0, which have nothing left to do.
template <bool NB1, int NW>
__device__ bool fold_tiles(const GemvParams &p, const Geo &q, const Smem &m, int S, int rank, int tid) {
    constexpr int NTH = NW * 32;
    const int nb = NB1 ? 1 : p.nb;
    const int cs = q.cs_here, U = q.U;
    const int total = q.tiles_here * kTileRows * nb;
    const size_t wstride = (size_t)p.TG * kTileRows * nb;
    for (int idx = tid; idx < total; idx += NTH) {
        const int tl = idx / (kTileRows * nb);
        const int u0 = tl * cs, u1 = u0 + cs;  // this tile's records [u0, u1)
        float v = 0.f;
#pragma unroll 4
        for (int w = 0; w < NW; ++w) {
            const int wub = (w * U) / NW, wue = ((w + 1) * U) / NW;
            if (max(wub, u0) < min(wue, u1)) v += m.slots[(size_t)w * wstride + idx];
        }
        m.red[idx] = v * m.nx[5 * kMaxNb + (idx % nb)];
    }
    if (S > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (rank == 0) {
            for (int idx = tid; idx < total; idx += NTH) {
                float v = m.red[idx];
                for (int r = 1; r < S; ++r) v += cluster.map_shared_rank(m.red, r)[idx];
                m.red[idx] = v;
            }
        }
        cluster.sync();
        if (rank != 0) return false;
    } else {
        __syncthreads();
    }
    return true;
}

// Write the job's outputs from `red`: store, residual add, SwiGLU over a
// gate/up tile pair, or this group's (max, index) per activation row.
template <bool NB1, int NW>
__device__ void epilogue(const GemvParams &p, const Geo &q, const Smem &m, int group, int tid, int warp, int lane) {
    constexpr int NTH = NW * 32;
    const int nb = NB1 ? 1 : p.nb;
    const int total = q.tiles_here * kTileRows * nb;
    if (group >= p.groups) return;  // no tiles, no partials
    if (p.epi == EPI_ARGMAX) {
        const int N = p.n[0];
        float *bvs = m.rbuf;  // [warp]
        int *bis = reinterpret_cast<int *>(m.rbuf + NW);
        for (int r = 0; r < nb; ++r) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int ri = tid; ri < q.tiles_here * kTileRows; ri += NTH) {
                const int n = (q.t0 + ri / kTileRows) * kTileRows + (ri % kTileRows);
                if (n >= N) continue;
                const float v = m.red[ri * nb + r];
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
                p.am_val[(size_t)r * p.groups + group] = fv;
                p.am_idx[(size_t)r * p.groups + group] = fi;
            }
            __syncthreads();
        }
        return;
    }
    for (int idx = tid; idx < total; idx += NTH) {
        const int tl = idx / (kTileRows * nb);
        const int rem = idx - tl * kTileRows * nb;
        const int row = rem / nb, r = rem - row * nb;
        int mi, tm;
        map_tile(p, q.t0 + tl, mi, tm);
        const int n = tm * kTileRows + row;
        const int N = p.n[mi];
        if (n >= N) continue;
        const float v = m.red[idx];
        if (p.epi == EPI_STORE) {
            p.out[mi][(size_t)r * N + n] = v;
        } else if (p.epi == EPI_RESIDUAL) {
            p.out[0][(size_t)r * N + n] = v + __ldcg(p.res + (size_t)r * N + n);
        } else if (mi == 0) {  // EPI_SWIGLU: gate tile tl, up tile tl + 1
            const float u = m.red[idx + kTileRows * nb];
            p.out[0][(size_t)r * N + n] = v / (1.0f + expf(-v)) * u;
        }
    }
    __syncthreads();
}

// Single K-slice, store / residual / SwiGLU jobs: fold each output's warp
// partials (in warp order) and write it at once, with no round trip through
// `red` and one barrier fewer than fold_tiles + epilogue.
template <bool NB1, int NW>
__device__ void fold_store(const GemvParams &p, const Geo &q, const Smem &m, int group, int tid) {
    constexpr int NTH = NW * 32;
    const int nb = NB1 ? 1 : p.nb;
    if (group >= p.groups) return;  // no tiles
    const int cs = q.cs_here, U = q.U;
    const size_t wstride = (size_t)p.TG * kTileRows * nb;
    const int tile_vals = kTileRows * nb;
    auto fold = [&](int idx) -> float {
        const int tl = idx / tile_vals;
        const int u0 = tl * cs, u1 = u0 + cs;  // this tile's records [u0, u1)
        float v = 0.f;
#pragma unroll 4
        for (int w = 0; w < NW; ++w) {
            const int wub = (w * U) / NW, wue = ((w + 1) * U) / NW;
            if (max(wub, u0) < min(wue, u1)) v += m.slots[(size_t)w * wstride + idx];
        }
        return v * m.nx[5 * kMaxNb + (idx % nb)];
    };
    const bool pairs = p.epi == EPI_SWIGLU;
    const int total = (pairs ? q.tiles_here / 2 : q.tiles_here) * tile_vals;
    for (int e = tid; e < total; e += NTH) {
        const int tp = e / tile_vals, rem = e - tp * tile_vals;
        const int idx = (pairs ? 2 * tp : tp) * tile_vals + rem;
        const int row = rem / nb, r = rem - row * nb;
        int mi, tm;
        map_tile(p, q.t0 + idx / tile_vals, mi, tm);
        const int n = tm * kTileRows + row;
        const int N = p.n[mi];
        if (n >= N) continue;
        const float v = fold(idx);
        if (p.epi == EPI_STORE) {
            p.out[mi][(size_t)r * N + n] = v;
        } else if (p.epi == EPI_RESIDUAL) {
            p.out[0][(size_t)r * N + n] = v + __ldcg(p.res + (size_t)r * N + n);
        } else {  // SwiGLU: gate tile, then its up tile
            const float u = fold(idx + tile_vals);
            p.out[0][(size_t)r * N + n] = v / (1.0f + expf(-v)) * u;
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// Per-call kernel: one job, one group of tiles per cluster.
template <int FMT, int NT, bool NB1>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const __grid_constant__ GemvParams p) {
    constexpr int REC = FMT == 0 ? kRecQ4_0 : kRecAffine;
    constexpr int DEPTH = kRingDepth;
    constexpr int NW = kWarps;
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.S;
    const int group = blockIdx.x / S, rank = blockIdx.x - group * S;
    const int nb = NB1 ? 1 : p.nb;
    const Smem m = carve<NW>(smem, FMT, nb, p.Cs, 8 * NT, p.TG);
    const uint32_t ring_a = smem_u32(m.ring) + warp * DEPTH * REC;

    // the next kernel may launch now; it waits for this one before it reads
    // what this one writes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // weights do not depend on the previous kernel: start their copies first
    WeightStream<REC, NW> ws;
    ws.init(&p, 1, group, rank, warp);
    for (int s = 0; s < DEPTH - 1; ++s) {
        if (ws.left > 0) ws.issue(ring_a + s * REC, lane);
        cp_async_commit();
    }
    const Geo q = make_geo<NW>(p, group, rank, warp);
    asm volatile("griddepcontrol.wait;" ::: "memory");

    stage_x<FMT, NT, NB1, NW>(p, q, m, S, tid, warp, lane);
    uint32_t st_a = ring_a, fill_a = ring_a + (DEPTH - 1) * REC;
    run_units<FMT, NT, NB1, DEPTH, NW>(p, q, m, ws, st_a, fill_a, ring_a, warp, lane);
    cp_async_wait<0>();
    __syncthreads();
    if (S == 1 && p.epi != EPI_ARGMAX) {
        fold_store<NB1, NW>(p, q, m, group, tid);
        return;
    }
    if (!fold_tiles<NB1, NW>(p, q, m, S, rank, tid)) return;
    epilogue<NB1, NW>(p, q, m, group, tid, warp, lane);
}

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

// Grid barrier number `b` (1-based).  Each CTA adds one to the arrival
// counter; the CTA that completes the count publishes `b` in the release
// word, which the others poll (a read-only line, away from the atomics).
// The wait is bounded: after kBarrierSpins polls the CTA records the failure
// in *err and the caller stops.
__device__ __forceinline__ bool grid_barrier(unsigned *counter, unsigned *release, int *err, unsigned b) {
    __syncthreads();
    __shared__ int fail;
    if (threadIdx.x == 0) {
        fail = 0;
        __threadfence();
        const unsigned prev = atomicAdd(counter, 1u);
        if (prev + 1 == b * gridDim.x) {
            asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(release), "r"(b) : "memory");
        } else {
            long long it = 0;
            while (ld_acquire_u32(release) < b) {
                if (++it > kBarrierSpins) {
                    atomicExch(err, 1);
                    fail = 1;
                    break;
                }
            }
        }
        __threadfence();
    }
    __syncthreads();
    return fail == 0;
}

template <int FMT, int NT, bool NB1>
__global__ void __launch_bounds__(kStepWarps * 32, 1) decode_kernel(const __grid_constant__ StepParams sp) {
    constexpr int REC = FMT == 0 ? kRecQ4_0 : kRecAffine;
    constexpr int DEPTH = kStepRingDepth;
    constexpr int NW = kStepWarps;
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int group = blockIdx.x;
    const int nb = NB1 ? 1 : sp.nb;
    const int cs_max = (sp.Kmax + kChunkK - 1) / kChunkK;  // as the host sized it
    const Smem m = carve<NW>(smem, FMT, nb, cs_max, 8 * NT, sp.TGmax);
    const uint32_t ring_a = smem_u32(m.ring) + warp * DEPTH * REC;

    WeightStream<REC, NW> ws;
    ws.init(sp.jobs, sp.njobs, group, 0, warp);
    for (int s = 0; s < DEPTH - 1; ++s) {
        if (ws.left > 0) ws.issue(ring_a + s * REC, lane);
        cp_async_commit();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");

    uint32_t st_a = ring_a, fill_a = ring_a + (DEPTH - 1) * REC;
    for (int j = 0; j < sp.njobs; ++j) {
        const GemvParams &p = sp.jobs[j];
        if (j > 0 && !grid_barrier(sp.counter, sp.release, sp.err, (unsigned)j)) return;
        const Geo q = make_geo<NW>(p, group, 0, warp);
        stage_x<FMT, NT, NB1, NW>(p, q, m, 1, tid, warp, lane);
        run_units<FMT, NT, NB1, DEPTH, NW>(p, q, m, ws, st_a, fill_a, ring_a, warp, lane);
        __syncthreads();
        if (p.epi != EPI_ARGMAX) {
            fold_store<NB1, NW>(p, q, m, group, tid);
        } else {
            fold_tiles<NB1, NW>(p, q, m, 1, 0, tid);
            epilogue<NB1, NW>(p, q, m, group, tid, warp, lane);
        }
    }
    cp_async_wait<0>();
    // the last job is the logits argmax: fold the groups' pairs in order
    if (!grid_barrier(sp.counter, sp.release, sp.err, (unsigned)sp.njobs)) return;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const GemvParams &pl = sp.jobs[sp.njobs - 1];
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
