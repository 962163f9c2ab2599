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
//  * One CTA = 8 warps owns a group of 16-row tiles and one K-slice; a
//    thread-block cluster of S CTAs splits K and folds its partial sums over
//    distributed shared memory in rank order (deterministic, no atomics).
//  * Weights stream once with 128-bit L1-bypassing loads, four records in
//    flight per warp, issued before the programmatic-dependent-launch wait so
//    the weight stream overlaps the previous kernel's tail.
//  * Each 32-bit nibble word becomes four f16x2 registers of (q - 8) (or q)
//    with one lop3 and one packed fma each -- exact integers in f16.
//  * Activations are staged once per CTA in shared memory as an exact
//    power-of-two-scaled hi + lo pair of f16 values (about 22 significant
//    bits), laid out so each lane loads its mma B fragment with one 64-bit
//    shared load.
//  * mma.sync m16n8k16 (f16 in, fp32 accumulate) forms the per-block dot
//    products of 16 rows x (hi, lo) columns; each block's result is scaled
//    by its fp32 scale and accumulated in fp32, so weights are never rounded.
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

template <int FMT, int NT>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvParams p) {
    constexpr int REC = FMT == 0 ? kRecQ4_0 : kRecAffine;
    constexpr int DEPTH = 4;  // weight records per warp: 1 in use + 3 in flight

    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tq = lane & 3;
    const int nb = p.nb, S = p.S, TG = p.TG;
    const int group = blockIdx.x / S;
    const int rank = blockIdx.x - group * S;
    const int t0 = group * TG;
    const int tiles_here = min(TG, p.T - t0);
    const int c0 = rank * p.Cs;
    const int cs_here = max(0, min(p.Cs, p.C - c0));
    const int Ks = p.Cs * kChunkK;
    const int kb = c0 * kChunkK;
    const int ke = min(p.K, kb + Ks);  // real activations of this slice: [kb, ke)

    // shared memory carve-up (sizes match smem_bytes())
    uint8_t *xs = smem;                                              // [Ks/16][2nb][4][2] u32
    float *gs = reinterpret_cast<float *>(smem + (size_t)4 * nb * Ks);  // [Cs*4][nb]
    float *slots = gs + (FMT == 1 ? nb * p.Cs * kBlocksPerChunk : 0);   // [warp][TG][16][nb]
    float *red = slots + kWarps * TG * kTileRows * nb;                 // [TG][16][nb]
    float *rbuf = red + TG * kTileRows * nb;                           // [2][warp][kMaxNb]
    float *nx = rbuf + 4 * kWarps * kMaxNb;                            // [8][kMaxNb] row stats

    // ---- weights first: they do not depend on the previous kernel.
    const int n_units = tiles_here * cs_here;
    const int my_units = n_units > warp ? (n_units - warp + kWarps - 1) / kWarps : 0;
    uint4 rp0[DEPTH], rp1[DEPTH], rsc[DEPTH], rmn[DEPTH];

    auto unit_ptr = [&](int i) -> const uint8_t * {
        const int u = warp + i * kWarps;
        const int tl = u / cs_here, cl = u - tl * cs_here;
        int m, tm;
        map_tile(p, t0 + tl, m, tm);
        return p.w[m] + ((size_t)tm * p.C + (size_t)(c0 + cl)) * REC;
    };
    auto load_unit = [&](int i, uint4 &a, uint4 &b, uint4 &s, uint4 &mn) {
        const uint8_t *q = unit_ptr(i);
        a = ldg_stream(q + lane * 16);
        b = ldg_stream(q + 512 + lane * 16);
        s = ldg_stream(q + 1024 + g * 16);
        if (FMT == 1) mn = ldg_stream(q + 1152 + g * 16);
    };
#pragma unroll
    for (int s = 0; s < DEPTH - 1; ++s)
        if (s < my_units) load_unit(s, rp0[s], rp1[s], rsc[s], rmn[s]);

    for (int i = tid; i < kWarps * TG * kTileRows * nb; i += kThreads) slots[i] = 0.f;

    // ---- activations are the previous kernel's output: wait for it.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const bool norm = p.gamma != nullptr;
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

    // pass 2: scaled (and normed) activations as hi + lo f16 in B-fragment order
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
            const int s = kl >> 4, kk = kl & 15;
            const int off = s * 64 * nb + ((kk & 7) >> 1) * 8 + (kk >> 3) * 4;
            *reinterpret_cast<__half2 *>(xs + off + (2 * r) * 32) = hi;
            *reinterpret_cast<__half2 *>(xs + off + (2 * r + 1) * 32) = lo;
        }
        if (FMT == 1) {
            // per-32 group sums of the (normed) activations, ascending order
            const int nblk = p.Cs * kBlocksPerChunk;
            for (int i = tid; i < nb * nblk; i += kThreads) {
                const int r = i / nblk, bl = i - r * nblk;
                const int kblk = kb + 32 * bl;
                float s = 0.f;
                if (kblk < ke) {
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
                }
                gs[bl * nb + r] = s * nx[3 * kMaxNb + r];
            }
        }
    }
    __syncthreads();

    // ---- main loop: warp-strided (tile, chunk) units
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    int cur_tl = -1;

    auto flush = [&](int tl) {
        float *sl = slots + ((size_t)(warp * TG + tl) * kTileRows) * nb;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int r = 4 * j + tq;
            if (r < nb) {
                sl[g * nb + r] = acc[j][0] + acc[j][1];
                sl[(g + 8) * nb + r] = acc[j][2] + acc[j][3];
            }
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        }
    };

    auto compute_unit = [&](int i, const uint4 &q0, const uint4 &q1, const uint4 &sc, const uint4 &mn) {
        const int u = warp + i * kWarps;
        const int tl = u / cs_here, cl = u - tl * cs_here;
        if (tl != cur_tl) {
            if (cur_tl >= 0) flush(cur_tl);
            cur_tl = tl;
        }
        const uint32_t w0s[4] = {q0.x, q0.y, q0.z, q0.w};
        const uint32_t w1s[4] = {q1.x, q1.y, q1.z, q1.w};
        const uint32_t scs[4] = {sc.x, sc.y, sc.z, sc.w};
        const uint32_t mns[4] = {mn.x, mn.y, mn.z, mn.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t a[8];
            unpack_word<FMT>(w0s[j], a[0], a[2], a[4], a[6]);  // row g
            unpack_word<FMT>(w1s[j], a[1], a[3], a[5], a[7]);  // row g + 8
            const float2 d = scale_pair<FMT>(scs[j]);
            float2 mm = make_float2(0.f, 0.f);
            if (FMT == 1) mm = scale_pair<FMT>(mns[j]);
            const int step = cl * 8 + 2 * j;  // k16 step of the block's first half
            const uint8_t *xb = xs + (size_t)step * 64 * nb + lane * 8;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                uint2 b0 = make_uint2(0u, 0u), b1 = make_uint2(0u, 0u);
                if (8 * nt + g < 2 * nb) {
                    b0 = *reinterpret_cast<const uint2 *>(xb + nt * 256);
                    b1 = *reinterpret_cast<const uint2 *>(xb + 64 * nb + nt * 256);
                }
                float dd[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(dd, a[0], a[1], a[2], a[3], b0.x, b0.y);
                mma16816(dd, a[4], a[5], a[6], a[7], b1.x, b1.y);
                acc[nt][0] = fmaf(d.x, dd[0], acc[nt][0]);
                acc[nt][1] = fmaf(d.x, dd[1], acc[nt][1]);
                acc[nt][2] = fmaf(d.y, dd[2], acc[nt][2]);
                acc[nt][3] = fmaf(d.y, dd[3], acc[nt][3]);
                if (FMT == 1) {
                    const int r = 4 * nt + tq;
                    if (r < nb) {
                        const float gv = gs[(cl * kBlocksPerChunk + j) * nb + r];
                        acc[nt][0] = fmaf(mm.x, gv, acc[nt][0]);
                        acc[nt][2] = fmaf(mm.y, gv, acc[nt][2]);
                    }
                }
            }
        }
    };

    for (int i0 = 0; i0 < my_units; i0 += DEPTH) {
#pragma unroll
        for (int s = 0; s < DEPTH; ++s) {
            const int i = i0 + s;
            if (i < my_units) {
                const int nx_slot = (s + DEPTH - 1) % DEPTH;
                if (i + DEPTH - 1 < my_units)
                    load_unit(i + DEPTH - 1, rp0[nx_slot], rp1[nx_slot], rsc[nx_slot], rmn[nx_slot]);
                compute_unit(i, rp0[s], rp1[s], rsc[s], rmn[s]);
            }
        }
    }
    if (cur_tl >= 0) flush(cur_tl);

    // the next kernel in the stream may start its own weight stream now
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();

    // ---- fold the warps' partials in warp order, undo the activation scale
    const int total = tiles_here * kTileRows * nb;
    for (int idx = tid; idx < total; idx += kThreads) {
        float v = 0.f;
        for (int w = 0; w < kWarps; ++w) v += slots[(size_t)w * TG * kTileRows * nb + idx];
        red[idx] = v * nx[5 * kMaxNb + (idx % nb)];
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
