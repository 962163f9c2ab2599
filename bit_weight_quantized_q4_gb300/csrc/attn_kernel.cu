// attn_kernel.cu -- decode attention over an f32 KV cache (honeycrisp/mod.rs:
// gpu_attention, and the fused RoPE + KV-append + SDPA dispatch of
// forward_decode_fused_layers).  One token: optional RoPE of q and the new
// k, append of k and v at `position`, then for every query head the softmax
// of scale * q K^T over the attended positions times V.
//
// The work is HBM-bound on the cache rows.  CTA (s, hk) takes kv head hk and
// the s-th chunk of the attended positions: its K and V rows are contiguous
// in the cache, so two TMA bulk copies bring them into shared memory (each on
// its own mbarrier: the scores start while V is still arriving), and every
// query head of the group reuses them.  Chunks are folded in a second pass
// (their maxima and sums, in chunk order) unless there is only one.
#include "gemv_launch.cuh"

namespace q4 {
namespace dev {

// RoPE of a head vector held DL = D/32 elements per lane (lane l holds
// elements l*DL .. l*DL+DL-1): element e pairs with e + D/2, which lane l ^ 16
// holds; (a, b) -> (a c - b s, b c + a s) with the table row of the position.
template <int DL>
__device__ __forceinline__ void rope_lane(float (&x)[DL], const float *cosr, const float *sinr, int lane) {
    constexpr int HALF = 16 * DL;
#pragma unroll
    for (int j = 0; j < DL; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, x[j], 16);
        const int jj = (lane * DL + j) % HALF;
        const float c = __ldg(cosr + jj), s = __ldg(sinr + jj);
        x[j] = lane < 16 ? x[j] * c - other * s : x[j] * c + other * s;
    }
}

template <int DL>
__device__ __forceinline__ void load_row(float (&x)[DL], const float *src) {
    if constexpr (DL == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(src);
        x[0] = v.x;
        x[1] = v.y;
    } else {
        const float4 v = *reinterpret_cast<const float4 *>(src);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
    }
}

// 32 partial sums per lane -> lane l holds the warp-wide sum of value l
// (recursive halving: each round a lane keeps the half of its values whose
// index bit matches its lane bit and adds its partner's share of it).
__device__ __forceinline__ float transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? v[i] : v[i + o];
            const float keep = up ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

constexpr int kAttnWarps = 8;

template <int D, int G>
__global__ void __launch_bounds__(kAttnWarps * 32, 1) q4attn_split_kernel(const __grid_constant__ AttnParams p) {
    constexpr int DL = D / 32, P = 32 / G, NW = kAttnWarps;
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, hk = blockIdx.y;
    const int Lc = p.Lc;
    const int t0 = p.lo + split * Lc;
    const int n = min(Lc, p.total - t0);  // >= 1
    const bool owner = t0 + n == p.total;  // this chunk ends with the new token
    const uint32_t barK = smem_u32(smem), barV = barK + 8;
    float *Ks = reinterpret_cast<float *>(smem + 16);
    float *Vs = Ks + (size_t)Lc * D;
    float *sc = Vs + (size_t)Lc * D;  // [G][Lc]: scores, then exp(score - max)
    float *red = sc + (size_t)G * Lc;  // [NW][G * D]
    float *stat = red + NW * G * D;   // max[G], sum[G]
    const size_t row0 = ((size_t)hk * p.max_seq + t0) * D;

    if (tid == 0) {
        mbar_init(barK, 1);
        mbar_init(barV, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)n * D * 4;
        const uint64_t pol = evict_first_policy();
        mbar_expect_tx(barK, bytes);
        bulk_g2s(smem_u32(Ks), p.k_cache + row0, bytes, barK, pol);
        mbar_expect_tx(barV, bytes);
        bulk_g2s(smem_u32(Vs), p.v_cache + row0, bytes, barV, pol);
    }
    // while the rows arrive: this group's query heads (rotated) in registers,
    // and for the last chunk the new token's k (rotated) and v
    const float *cosr = p.rope_cos ? p.rope_cos + (size_t)p.position * (D / 2) : nullptr;
    const float *sinr = p.rope_sin ? p.rope_sin + (size_t)p.position * (D / 2) : nullptr;
    float qr[G][DL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        load_row<DL>(qr[g], p.q + (size_t)(hk * G + g) * D + lane * DL);
        if (cosr) rope_lane<DL>(qr[g], cosr, sinr, lane);
    }
    float kv[DL];
    if (owner && warp < 2) {
        load_row<DL>(kv, (warp == 0 ? p.k_new : p.v_new) + (size_t)hk * D + lane * DL);
        if (warp == 0 && cosr) rope_lane<DL>(kv, cosr, sinr, lane);
    }

    // K rows in
    bool ok = mbar_wait(barK, 0, p.wait_cycles);
    if (!__syncthreads_and(ok)) {
        // gave up: record it, and let the copies land before the CTA leaves
        if (tid == 0) {
            atomicExch(p.err, 3);
            mbar_wait(barK, 0, kWaitCycles);
            mbar_wait(barV, 0, kWaitCycles);
        }
        __syncthreads();
        return;
    }
    if (owner && warp == 0) {  // append k: the cache, and this chunk's copy of it
#pragma unroll
        for (int j = 0; j < DL; ++j) {
            Ks[(size_t)(n - 1) * D + lane * DL + j] = kv[j];
            p.k_cache[row0 + (size_t)(n - 1) * D + lane * DL + j] = kv[j];
        }
    }
    __syncthreads();

    // scores: a warp takes P positions at a time, lane l dims l*DL.., every
    // head of the group; one transpose-reduce gives lane l the score of
    // position l / G, head l % G
    for (int i = warp; i * P < n; i += NW) {
        float v[32];
#pragma unroll
        for (int pp = 0; pp < P; ++pp) {
            const int tl = i * P + pp;
            float kr[DL];
            if (tl < n) {
                load_row<DL>(kr, Ks + (size_t)tl * D + lane * DL);
            } else {
#pragma unroll
                for (int j = 0; j < DL; ++j) kr[j] = 0.f;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float s = 0.f;
#pragma unroll
                for (int j = 0; j < DL; ++j) s = fmaf(qr[g][j], kr[j], s);
                v[pp * G + g] = s;
            }
        }
        const float s = transpose_reduce(v, lane);
        const int tl = i * P + lane / G, g = lane % G;
        if (tl < n) sc[(size_t)g * Lc + tl] = s * p.scale;
    }
    __syncthreads();

    // softmax of each head over the chunk: its maximum, exp(s - max), sum
    for (int g = warp; g < G; g += NW) {
        float* row = sc + (size_t)g * Lc;
        float mx = -INFINITY;
        for (int t = lane; t < n; t += 32) mx = fmaxf(mx, row[t]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
        for (int t = lane; t < n; t += 32) {
            const float e = expf(row[t] - mx);
            row[t] = e;
            sum += e;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) {
            stat[g] = mx;
            stat[G + g] = sum;
        }
    }

    // V rows in (usually long since), and the new token's v
    ok = mbar_wait(barV, 0, p.wait_cycles);
    if (!__syncthreads_and(ok)) {
        if (tid == 0) {
            atomicExch(p.err, 3);
            mbar_wait(barV, 0, kWaitCycles);
        }
        __syncthreads();
        return;
    }
    if (owner && warp == 1) {
#pragma unroll
        for (int j = 0; j < DL; ++j) {
            Vs[(size_t)(n - 1) * D + lane * DL + j] = kv[j];
            p.v_cache[row0 + (size_t)(n - 1) * D + lane * DL + j] = kv[j];
        }
    }
    __syncthreads();

    // sum_t p_t v_t: warp w takes positions w, w + NW, ...; lane l dims
    // l*DL.. of every head; then the warps' shares are added in warp order
    float acc[G][DL];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < DL; ++j) acc[g][j] = 0.f;
    for (int tl = warp; tl < n; tl += NW) {
        float vr[DL];
        load_row<DL>(vr, Vs + (size_t)tl * D + lane * DL);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float pg = sc[(size_t)g * Lc + tl];
#pragma unroll
            for (int j = 0; j < DL; ++j) acc[g][j] = fmaf(pg, vr[j], acc[g][j]);
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < DL; ++j) red[(size_t)warp * G * D + g * D + lane * DL + j] = acc[g][j];
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += NW * 32) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) o += red[(size_t)w * G * D + idx];
        const int g = idx / D, d = idx - g * D, hq = hk * G + g;
        if (p.nsplit == 1) {
            p.out[(size_t)hq * D + d] = o / stat[G + g];
        } else {
            p.ws_o[((size_t)split * p.H + hq) * D + d] = o;
            if (d == 0) {
                p.ws_m[(size_t)split * p.H + hq] = stat[g];
                p.ws_l[(size_t)split * p.H + hq] = stat[G + g];
            }
        }
    }
}

// Fold the chunks of query head blockIdx.x: with M the largest chunk maximum,
// out = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M), in chunk order.
__global__ void q4attn_combine_kernel(const __grid_constant__ AttnParams p) {
    const int hq = blockIdx.x, D = p.D;
    float M = -INFINITY;
    for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, p.ws_m[(size_t)s * p.H + hq]);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float L = 0.f, o = 0.f;
        for (int s = 0; s < p.nsplit; ++s) {
            const float w = expf(p.ws_m[(size_t)s * p.H + hq] - M);
            L = fmaf(p.ws_l[(size_t)s * p.H + hq], w, L);
            o = fmaf(p.ws_o[((size_t)s * p.H + hq) * D + d], w, o);
        }
        p.out[(size_t)hq * D + d] = o / L;
    }
}

}  // namespace dev

size_t attn_smem_bytes(int D, int G, int Lc) {
    return 16 + (size_t)2 * Lc * D * 4 + (size_t)G * Lc * 4 + (size_t)dev::kAttnWarps * G * D * 4 + 2 * G * 4;
}

template <int D, int G>
static int launch_attn_dg(const AttnParams &p, cudaStream_t stream) {
    auto kern = dev::q4attn_split_kernel<D, G>;
    static size_t smem_set[64] = {0};
    const size_t smem = attn_smem_bytes(D, G, p.Lc);
    if (!raise_smem(kern, smem, smem_set)) return -1;
    dim3 grid(p.nsplit, p.Hkv);
    kern<<<grid, dev::kAttnWarps * 32, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    if (p.nsplit > 1) {
        dev::q4attn_combine_kernel<<<p.H, D, 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess) return -1;
    }
    return 0;
}

int launch_attn(const AttnParams &p, void *stream_) {
    cudaStream_t stream = (cudaStream_t)stream_;
    const int G = p.H / p.Hkv;
    if (p.D == 64) {
        switch (G) {
            case 1: return launch_attn_dg<64, 1>(p, stream);
            case 2: return launch_attn_dg<64, 2>(p, stream);
            case 4: return launch_attn_dg<64, 4>(p, stream);
            case 8: return launch_attn_dg<64, 8>(p, stream);
            case 16: return launch_attn_dg<64, 16>(p, stream);
        }
    } else if (p.D == 128) {
        switch (G) {
            case 1: return launch_attn_dg<128, 1>(p, stream);
            case 2: return launch_attn_dg<128, 2>(p, stream);
            case 4: return launch_attn_dg<128, 4>(p, stream);
            case 8: return launch_attn_dg<128, 8>(p, stream);
        }
    }
    return -1;
}

}  // namespace q4
