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
    if (p.mode == MODE_SINGLE) {
        m = 0;
        tm = t;
    } else if (p.mode == MODE_CONCAT) {
        m = t < p.tiles[0] ? 0 : 1;
        tm = m ? t - p.tiles[0] : t;
    } else {
        m = t & 1;
        tm = t >> 1;
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

template <int FMT, int NT, bool NB1>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvParams p) {
    constexpr int REC = FMT == 0 ? kRecQ4_0 : kRecAffine;
    constexpr int DEPTH = kRingDepth;  // weight records per warp: 1 in use, the rest in flight
    constexpr int GSW = 8 * NT;     // group-sum row width (activation rows, padded)

    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int nb = NB1 ? 1 : p.nb;
    const int S = p.S;
    const int group = blockIdx.x / S;
    const int rank = blockIdx.x - group * S;
    const int pw = p.mode == MODE_PAIRS ? 2 : 1;
    const int P = p.T / pw;
    const int t0 = (int)(((long long)group * P) / p.groups) * pw;
    const int t1 = (int)(((long long)(group + 1) * P) / p.groups) * pw;
    const int tiles_here = t1 - t0;
    const int c0 = rank * p.Cs;
    const int cs_here = max(0, min(p.Cs, p.C - c0));
    const int Ks = p.Cs * kChunkK;
    const int kb = c0 * kChunkK;
    const int ke = min(p.K, kb + Ks);  // real activations of this slice: [kb, ke)
    const int xbs = 128 * nb;          // bytes of one block's activations in shared memory

    // shared memory carve-up (sizes match smem_bytes())
    uint8_t *xs = smem;                                                  // [Cs*4][nt][2][lanes][16 B]
    float *gs = reinterpret_cast<float *>(smem + (size_t)4 * nb * Ks);  // [Cs*4][GSW]
    float *red = gs + (FMT == 1 ? p.Cs * kBlocksPerChunk * GSW : 0);    // [TG][16][nb]
    float *bslot = red + p.TG * kTileRows * nb;                         // [warp][2][16][nb]
    float *rbuf = bslot + kWarps * 2 * kTileRows * nb;                  // [4][warp][kMaxNb]
    float *nx = rbuf + 4 * kWarps * kMaxNb;                             // [8][kMaxNb] row stats
    uint8_t *ring = reinterpret_cast<uint8_t *>(nx + 8 * kMaxNb) + (size_t)warp * DEPTH * REC;  // this warp's

    auto tile_ptr = [&](int tl) -> const uint8_t * {
        int m, tm;
        map_tile(p, t0 + tl, m, tm);
        return p.w[m] + ((size_t)tm * p.C + (size_t)c0) * REC;
    };

    // the next kernel may launch now; it waits for this one before it reads
    // what this one writes
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int U = tiles_here * cs_here;
    const int ub = (warp * U) / kWarps, ue = ((warp + 1) * U) / kWarps;
    const int n_my = ue - ub;
    const int first_tl = cs_here > 0 ? ub / cs_here : 0;
    int ltl = first_tl, lc = ub - first_tl * cs_here;
    const uint8_t *lptr = n_my > 0 ? tile_ptr(ltl) + (size_t)lc * REC : nullptr;
    // copy the next record of this warp's range into the ring stage at shared
    // address `dst`: each lane its two 16-byte nibble pieces, lanes 0..7
    // (0..15 affine) the scale (and min) words; then advance the cursor
    const uint32_t ring_a = smem_u32(ring);
    auto load_next = [&](uint32_t dst) {
        const uint8_t *src = lptr + lane * 16;
        const uint32_t d = dst + lane * 16;
        cp_async16_at<0>(d, src);
        cp_async16_at<512>(d, src);
        if (lane < (REC - 1024) / 16) cp_async16_at<1024>(d, src);
        lptr += REC;
        if (++lc == cs_here) {
            lc = 0;
            if (++ltl < tiles_here) lptr = tile_ptr(ltl);
        }
    };
    for (int s = 0; s < DEPTH - 1; ++s) {
        if (s < n_my) load_next(ring_a + s * REC);
        cp_async_commit();
    }

    const bool norm = p.gamma != nullptr;
    // nb == 1 and a slice of at most 2 * kThreads * RP columns: the whole
    // activation slice passes through registers in a single global read
    constexpr int RP = 16;
    const bool fast = NB1 && Ks <= 2 * kThreads * RP;
    float2 xv[RP], gv[RP];
    if (NB1 && fast && norm) {
        // gamma is a weight: load it before waiting for the previous kernel
#pragma unroll
        for (int q = 0; q < RP; ++q) {
            const int k = kb + 2 * (tid + q * kThreads);
            gv[q] = k < ke ? *reinterpret_cast<const float2 *>(p.gamma + k) : make_float2(0.f, 0.f);
        }
    }

    // ---- activations are the previous kernel's output: wait for it.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (NB1 && fast) {
        float ss = 0.f, mx = 0.f;
#pragma unroll
        for (int q = 0; q < RP; ++q) {
            const int k = kb + 2 * (tid + q * kThreads);
            float2 v = make_float2(0.f, 0.f);
            if (k < ke) v = *reinterpret_cast<const float2 *>(p.x + k);
            xv[q] = v;
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            const float ax = norm ? fabsf(v.x * gv[q].x) : fabsf(v.x);
            const float ay = norm ? fabsf(v.y * gv[q].y) : fabsf(v.y);
            mx = fmaxf(mx, fmaxf(ax, ay));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        }
        if (lane == 0) {
            rbuf[warp] = ss;
            rbuf[kWarps + warp] = mx;
        }
        __syncthreads();
        float tss = 0.f, tmx = 0.f;  // every thread adds the warps in the same order
        for (int w = 0; w < kWarps; ++w) {
            tss += rbuf[w];
            tmx = fmaxf(tmx, rbuf[kWarps + w]);
        }
        if (norm && S > 1) {
            // the RMS needs the whole row: add the slices' sums in rank order
            cg::cluster_group cluster = cg::this_cluster();
            if (tid == 0) nx[0] = tss;
            cluster.sync();
            tss = 0.f;
            for (int q = 0; q < S; ++q) tss += cluster.map_shared_rank(nx, q)[0];
        }
        const float inv_rms = norm ? 1.0f / sqrtf(tss / (float)p.K + p.eps) : 1.f;
        const float bound = tmx * inv_rms;
        float scale = 1.f, inv_scale = 1.f;
        if (bound > 0.f && bound <= 3.0e38f) {
            int ex;
            frexpf(bound, &ex);  // bound in [2^(ex-1), 2^ex)
            int e = 15 - ex;     // bound * 2^e in [2^14, 2^15)
            e = max(-100, min(100, e));
            scale = ldexpf(1.f, e);
            inv_scale = ldexpf(1.f, -e);
        }
        if (tid == 0) {
            nx[2 * kMaxNb] = inv_rms;
            nx[3 * kMaxNb] = scale;
            nx[5 * kMaxNb] = inv_scale;
        }
#pragma unroll
        for (int q = 0; q < RP; ++q) {
            const int kl = 2 * (tid + q * kThreads);
            if (kl < Ks) {
                float v0 = xv[q].x, v1 = xv[q].y;
                if (norm) {
                    v0 = v0 * inv_rms * gv[q].x;
                    v1 = v1 * inv_rms * gv[q].y;
                }
                v0 *= scale;
                v1 *= scale;
                __half2 hi = __floats2half2_rn(v0, v1);
                float2 hf = __half22float2(hi);
                __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
                const int kk = kl & 31, k16 = kk & 15;
                const int off = (kl >> 5) * 128 + (kk >> 4) * 64 + ((k16 & 7) >> 1) * 16 + (k16 >> 3) * 4;
                *reinterpret_cast<__half2 *>(xs + off) = hi;
                *reinterpret_cast<__half2 *>(xs + off + 8) = lo;
            }
        }
        if (FMT == 1) {
            __syncthreads();  // row stats visible to the group-sum loop
            const int nblk = p.Cs * kBlocksPerChunk;
            for (int i = tid; i < GSW * nblk; i += kThreads) {
                const int r = i / nblk, bl = i - r * nblk;
                const int kblk = kb + 32 * bl;
                float sacc = 0.f;
                if (r == 0 && kblk < ke) {
                    if (p.gsum != nullptr && !norm) {
                        sacc = p.gsum[kblk / 32];
                    } else {
                        for (int e = 0; e < 32; ++e) {
                            float v = p.x[kblk + e];
                            if (norm) v = v * inv_rms * p.gamma[kblk + e];
                            sacc += v;
                        }
                    }
                    sacc *= scale;
                }
                gs[bl * GSW + r] = sacc;
            }
        }
    } else {
        // pass 1: per activation row, sum of squares and max |x*gamma| (or |x|)
        for (int r = 0; r < nb; ++r) {
            float ss = 0.f, mx = 0.f;
            const float *xr = p.x + (size_t)r * p.K;
            for (int k = kb + 2 * tid; k < ke; k += 2 * kThreads) {
                float2 v = *reinterpret_cast<const float2 *>(xr + k);
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
                rbuf[warp * kMaxNb + r] = ss;
                rbuf[kWarps * kMaxNb + warp * kMaxNb + r] = mx;
            }
        }
        __syncthreads();
        if (tid < nb) {
            float ss = 0.f, mx = 0.f;
            for (int w = 0; w < kWarps; ++w) {
                ss += rbuf[w * kMaxNb + tid];
                mx = fmaxf(mx, rbuf[kWarps * kMaxNb + w * kMaxNb + tid]);
            }
            nx[0 * kMaxNb + tid] = ss;  // this slice's sum of squares
            nx[1 * kMaxNb + tid] = mx;
        }
        if (norm && S > 1) {
            // the RMS needs the whole row: add the slices' sums in rank order
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();
            if (tid < nb) {
                float tot = 0.f;
                for (int q = 0; q < S; ++q) tot += cluster.map_shared_rank(nx, q)[tid];
                nx[4 * kMaxNb + tid] = tot;
            }
        } else if (tid < nb) {
            nx[4 * kMaxNb + tid] = nx[tid];
        }
        __syncthreads();
        if (tid < nb) {
            float inv_rms = 1.f;
            if (norm) inv_rms = 1.0f / sqrtf(nx[4 * kMaxNb + tid] / (float)p.K + p.eps);
            float bound = nx[1 * kMaxNb + tid] * inv_rms;
            float scale = 1.f, inv_scale = 1.f;
            if (bound > 0.f && bound <= 3.0e38f) {
                int ex;
                frexpf(bound, &ex);  // bound in [2^(ex-1), 2^ex)
                int e = 15 - ex;     // bound * 2^e in [2^14, 2^15)
                e = max(-100, min(100, e));
                scale = ldexpf(1.f, e);
                inv_scale = ldexpf(1.f, -e);
            }
            nx[2 * kMaxNb + tid] = inv_rms;
            nx[3 * kMaxNb + tid] = scale;
            nx[5 * kMaxNb + tid] = inv_scale;
        }
        __syncthreads();

        // pass 2: scaled (and normed) activations as hi + lo f16 pairs, stored
        // per block in the order the lanes load their mma B fragments:
        //   [n-tile][k16 step][lane g*4+t][hi(k=2t,2t+1), hi(2t+8,2t+9), lo(..), lo(..)]
        {
            const int half_ks = Ks >> 1;
            for (int i = tid; i < nb * half_ks; i += kThreads) {
                const int r = i / half_ks, kp = i - r * half_ks;
                const int kl = 2 * kp, k = kb + kl;
                float v0 = 0.f, v1 = 0.f;
                if (k < ke) {
                    float2 v = *reinterpret_cast<const float2 *>(p.x + (size_t)r * p.K + k);
                    v0 = v.x;
                    v1 = v.y;
                    if (norm) {
                        const float ir = nx[2 * kMaxNb + r];
                        float2 gm = *reinterpret_cast<const float2 *>(p.gamma + k);
                        v0 = v0 * ir * gm.x;
                        v1 = v1 * ir * gm.y;
                    }
                }
                const float sc = nx[3 * kMaxNb + r];
                v0 *= sc;
                v1 *= sc;
                __half2 hi = __floats2half2_rn(v0, v1);
                float2 hf = __half22float2(hi);
                __half2 lo = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
                const int bl = kl >> 5, kk = kl & 31, st = kk >> 4, k16 = kk & 15;
                const int nt = r >> 3, cols = min(8, nb - 8 * nt);
                const int off = bl * xbs + nt * 1024 + st * 64 * cols + (4 * (r & 7) + ((k16 & 7) >> 1)) * 16 +
                                (k16 >> 3) * 4;
                *reinterpret_cast<__half2 *>(xs + off) = hi;
                *reinterpret_cast<__half2 *>(xs + off + 8) = lo;
            }
            if (FMT == 1) {
                // per-32 group sums of the (normed) activations, ascending order
                const int nblk = p.Cs * kBlocksPerChunk;
                for (int i = tid; i < GSW * nblk; i += kThreads) {
                    const int r = i / nblk, bl = i - r * nblk;
                    const int kblk = kb + 32 * bl;
                    float s = 0.f;
                    if (r < nb && kblk < ke) {
                        if (p.gsum != nullptr && !norm) {
                            s = p.gsum[(size_t)r * (p.K / 32) + kblk / 32];
                        } else {
                            const float *xr = p.x + (size_t)r * p.K + kblk;
                            const float ir = nx[2 * kMaxNb + r];
                            for (int e = 0; e < 32; ++e) {
                                float v = xr[e];
                                if (norm) v = v * ir * p.gamma[kblk + e];
                                s += v;
                            }
                        }
                        s *= nx[3 * kMaxNb + r];
                    }
                    gs[bl * GSW + r] = s;
                }
            }
        }
    }
    __syncthreads();

    // ---- main loop over this warp's contiguous (tile, chunk) units
    // lanes beyond the batch read a duplicate column: its mma outputs are
    // never stored, and every lane loads unconditionally
    const uint32_t xs_a = smem_u32(xs);
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
    int ctl = first_tl, cc = ub - first_tl * cs_here;
    const float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;

    auto flush = [&](int tl) {
        const bool complete = tl * cs_here >= ub && (tl + 1) * cs_here <= ue;
        float *dst = complete ? red + (size_t)tl * kTileRows * nb
                              : bslot + (size_t)(warp * 2 + (tl == first_tl ? 0 : 1)) * kTileRows * nb;
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
                const float2 gv = *reinterpret_cast<const float2 *>(gs + blk * GSW + 8 * nt + 2 * tq);
                acc[nt][0] = fmaf(mm.x, gv.x, acc[nt][0]);
                acc[nt][2] = fmaf(mm.y, gv.x, acc[nt][2]);
                if (!NB1) {
                    acc[nt][1] = fmaf(mm.x, gv.y, acc[nt][1]);
                    acc[nt][3] = fmaf(mm.y, gv.y, acc[nt][3]);
                }
            }
        }
    };

    uint32_t st_a = ring_a;                           // stage being consumed
    uint32_t fill_a = ring_a + (DEPTH - 1) * REC;     // stage to refill
    const uint32_t ring_end = ring_a + DEPTH * REC;
    for (int i = 0; i < n_my; ++i) {
        cp_async_wait<DEPTH - 2>();  // this lane's copies of record i have landed
        __syncwarp();                 // ... and every lane's; the previous stage is free
        if (i + DEPTH - 1 < n_my) load_next(fill_a);
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
    cp_async_wait<0>();
    if (n_my > 0 && cc != 0) flush(ctl);  // the range ended inside a tile
    __syncthreads();

    // ---- tiles split between warps: add their parts in warp order; then
    // undo the activation scale
    const int total = tiles_here * kTileRows * nb;
    for (int idx = tid; idx < total; idx += kThreads) {
        const int tl = idx / (kTileRows * nb);
        const int rem = idx - tl * kTileRows * nb;
        float v = 0.f;
        if (cs_here > 0) {
            const int u_first = tl * cs_here, u_last = u_first + cs_here - 1;
            const int w_first = (kWarps * (u_first + 1) + U - 1) / U - 1;
            const int w_last = (kWarps * (u_last + 1) + U - 1) / U - 1;
            if (w_first == w_last) {
                v = red[idx];
            } else {
                for (int w = w_first; w <= w_last; ++w) {
                    const int wub = (w * U) / kWarps;
                    if (((w + 1) * U) / kWarps == wub) continue;  // this warp had no units
                    const int slot = (tl == wub / cs_here) ? 0 : 1;
                    v += bslot[(size_t)(w * 2 + slot) * kTileRows * nb + rem];
                }
            }
        }
        red[idx] = v * nx[5 * kMaxNb + (rem % nb)];
    }
    if (S > 1) {
        // fold the K-slices of the cluster into rank 0, in rank order
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (rank == 0) {
            for (int idx = tid; idx < total; idx += kThreads) {
                float v = red[idx];
                for (int q = 1; q < S; ++q) v += cluster.map_shared_rank(red, q)[idx];
                red[idx] = v;
            }
        }
        cluster.sync();
        if (rank != 0) return;
    } else {
        __syncthreads();
    }

    // ---- epilogue
    if (p.epi == EPI_ARGMAX) {
        const int N = p.n[0];
        float *bvs = rbuf;                       // [warp]
        int *bis = reinterpret_cast<int *>(rbuf + kWarps);
        for (int r = 0; r < nb; ++r) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int ri = tid; ri < tiles_here * kTileRows; ri += kThreads) {
                const int n = (t0 + ri / kTileRows) * kTileRows + (ri % kTileRows);
                if (n >= N) continue;
                const float v = red[ri * nb + r];
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
                for (int w = 1; w < kWarps; ++w) {
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
    for (int idx = tid; idx < total; idx += kThreads) {
        const int tl = idx / (kTileRows * nb);
        const int rem = idx - tl * kTileRows * nb;
        const int row = rem / nb, r = rem - row * nb;
        int m, tm;
        map_tile(p, t0 + tl, m, tm);
        const int n = tm * kTileRows + row;
        const int N = p.n[m];
        if (n >= N) continue;
        const float v = red[idx];
        if (p.epi == EPI_STORE) {
            p.out[m][(size_t)r * N + n] = v;
        } else if (p.epi == EPI_RESIDUAL) {
            p.out[0][(size_t)r * N + n] = v + p.res[(size_t)r * N + n];
        } else if (m == 0) {  // EPI_SWIGLU: gate tile tl, up tile tl + 1
            const float u = red[idx + kTileRows * nb];
            p.out[0][(size_t)r * N + n] = v / (1.0f + expf(-v)) * u;
        }
    }
}

}  // namespace dev
}  // namespace q4
