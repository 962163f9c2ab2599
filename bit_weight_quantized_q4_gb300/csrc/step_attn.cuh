// step_attn.cuh -- the persistent decode step's attention job
// (q4_decode_step_attn): one token's decode attention of one layer inside
// q4gemv_step_kernel, between the layer's q/k/v job and its o job, with a
// grid barrier on either side.  It computes what q4_attn_decode computes
// (honeycrisp/mod.rs: gpu_attention, and the fused RoPE + KV-append + SDPA
// dispatch of forward_decode_fused_layers) at head size 64 and four query
// heads per kv head, arranged for the step's CTAs:
//   * CTA c takes kv head c / cps and split c % cps (Lc positions) of the
//     attended positions [lo, total); the split holding the new token
//     rotates k, appends k and v to the caches and scores them with the rest;
//   * its warps read K and V rows straight from the caches, each keeping a
//     running softmax per head over its positions; the warps merge in warp
//     order;
//   * the last split of a kv head to finish (a ticket, not a wait) folds the
//     splits' shares into the o job's input: each warp combines its splits
//     in order, all their loads at once, then the warps merge in warp order.
// Every load of data another CTA of the launch may have written bypasses L1.
#pragma once
#include "attn_common.cuh"

namespace q4 {
namespace dev {

template <int DL>
__device__ __forceinline__ void load_row_cg(float (&x)[DL], const float *src) {
    static_assert(DL == 2, "head size 64: two values a lane");
    const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
    x[0] = v.x;
    x[1] = v.y;
}

// The job for the CTA of `group`.  scratch: step_attn_scratch_bytes(NW, cps)
// bytes of shared memory that no other job uses meanwhile.  Every return is
// CTA-uniform; the caller's next grid barrier follows.
template <int NW>
__device__ void step_attn_job(const StepAttn &A, int layer, uint8_t *scratch, int group, int tid, int warp,
                              int lane) {
    constexpr int D = kStepAttnD, G = kStepAttnG, DL = D / 32, P = 32 / G;
    const int hk = group / A.cps, s = group - hk * A.cps;
    if (hk >= A.Hkv || s >= A.nsplit) return;  // no positions for this CTA
    const int t0 = A.lo + s * A.Lc;
    const int n = min(A.Lc, A.total - t0);  // >= 1 for s < nsplit
    const bool owner = t0 + n == A.total;   // this split ends with the new token
    float *kc = A.k_cache[layer], *vc = A.v_cache[layer];
    const size_t row0 = ((size_t)hk * A.max_seq + t0) * D;
    float *red = reinterpret_cast<float *>(scratch);  // [NW][G][D]
    float *wm = red + NW * G * D, *wl = wm + NW * G;  // [NW][G]
    float *eb = wl + NW * G, *ab = eb + NW * 32;     // per warp: a step's weights, rescale factors
    int *flag = reinterpret_cast<int *>(ab + NW * G);

    const float *cosr = A.rope_cos ? A.rope_cos + (size_t)A.position * (D / 2) : nullptr;
    const float *sinr = A.rope_sin ? A.rope_sin + (size_t)A.position * (D / 2) : nullptr;
    float qr[G][DL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        load_row_cg<DL>(qr[g], A.q + (size_t)(hk * G + g) * D + lane * DL);
        if (cosr) rope_lane<DL>(qr[g], cosr, sinr, lane);
    }
    if (owner && warp < 2) {  // append the new token: k rotated, v as is
        float kv[DL];
        load_row_cg<DL>(kv, (warp == 0 ? A.k_new : A.v_new) + (size_t)hk * D + lane * DL);
        if (warp == 0 && cosr) rope_lane<DL>(kv, cosr, sinr, lane);
        float *grow = (warp == 0 ? kc : vc) + row0 + (size_t)(n - 1) * D + lane * DL;
#pragma unroll
        for (int e = 0; e < DL; ++e) grow[e] = kv[e];
    }
    csync<NW>();  // the appended row is in the caches before any warp reads it

    // this warp's running softmax: lane l keeps head l % G's maximum and sum,
    // every lane the output share of its dims for every head
    float mh = -INFINITY, lh = 0.f;
    float acc[G][DL];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[g][e] = 0.f;
    float *ew = eb + warp * 32, *aw = ab + warp * G;
    for (int i = warp; i * P < n; i += NW) {
        // positions i*P .. i*P+P-1 of the split: their K and V rows at once
        float v[32], vr[P][DL];
#pragma unroll
        for (int pp = 0; pp < P; ++pp) {
            const int r = i * P + pp;
            float kr[DL];
            if (r < n) {
                load_row_cg<DL>(kr, kc + row0 + (size_t)r * D + lane * DL);
                load_row_cg<DL>(vr[pp], vc + row0 + (size_t)r * D + lane * DL);
            } else {
#pragma unroll
                for (int e = 0; e < DL; ++e) kr[e] = vr[pp][e] = 0.f;
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float sc = 0.f;
#pragma unroll
                for (int e = 0; e < DL; ++e) sc = fmaf(qr[g][e], kr[e], sc);
                v[pp * G + g] = sc;
            }
        }
        // lane l: position l / G, head l % G
        const float t = transpose_reduce(v, lane);
        const bool valid = i * P + lane / G < n;
        const float sl = valid ? t * A.scale : -INFINITY;
        float mx = sl;
#pragma unroll
        for (int o = G; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float mnew = fmaxf(mh, mx);  // finite: position i*P is valid
        const float alpha = expf(mh - mnew);
        const float e = valid ? expf(sl - mnew) : 0.f;
        float sum = e;
#pragma unroll
        for (int o = G; o < 32; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        lh = fmaf(lh, alpha, sum);
        mh = mnew;
        ew[lane] = e;
        if (lane < G) aw[lane] = alpha;
        __syncwarp();
        {
            float a[G];
            load_vec<G>(a, aw);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int q2 = 0; q2 < DL; ++q2) acc[g][q2] *= a[g];
        }
#pragma unroll
        for (int pp = 0; pp < P; ++pp) {
            if (i * P + pp < n) {  // warp-uniform
                float w[G];
                load_vec<G>(w, ew + pp * G);
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int q2 = 0; q2 < DL; ++q2) acc[g][q2] = fmaf(w[g], vr[pp][q2], acc[g][q2]);
            }
        }
        __syncwarp();  // the slots are read before the next step writes them
    }

    // merge the warps in warp order (a warp without positions has m = -inf)
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < DL; ++e) red[(size_t)warp * G * D + g * D + lane * DL + e] = acc[g][e];
    if (lane < G) {
        wm[warp * G + lane] = mh;
        wl[warp * G + lane] = lh;
    }
    csync<NW>();
    for (int idx = tid; idx < G * D; idx += NW * 32) {
        const int g = idx / D, d = idx - g * D, hq = hk * G + g;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w * G + g]);
        float o = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float f = expf(wm[w * G + g] - M);
            o = fmaf(red[(size_t)w * G * D + idx], f, o);
            L = fmaf(wl[w * G + g], f, L);
        }
        if (A.nsplit == 1) {
            A.out[(size_t)hq * D + d] = o / L;
        } else {
            A.ws_o[((size_t)s * A.H + hq) * D + d] = o;
            if (d == 0) {
                A.ws_m[(size_t)s * A.H + hq] = M;
                A.ws_l[(size_t)s * A.H + hq] = L;
            }
        }
    }
    if (A.nsplit == 1) return;

    // the last split of this kv head to finish folds every split's share in
    // split order: out = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M)
    __threadfence();
    csync<NW>();
    if (tid == 0) *flag = atomicAdd(A.ws_count + hk, 1) == A.nsplit - 1;
    csync<NW>();
    if (!*flag) return;
    __threadfence();
    // warp w combines the splits w, w + NW, ... in order, every load of them
    // in flight at once: lane l holds outputs l + 32 k (head (l + 32 k) / D)
    // and the running maximum and sum of those heads; then the warps merge
    // in warp order
    constexpr int OPL = G * D / 32;  // outputs per lane
    float pm[OPL], pl[OPL], po[OPL];
#pragma unroll
    for (int k = 0; k < OPL; ++k) {
        pm[k] = -INFINITY;
        pl[k] = 0.f;
        po[k] = 0.f;
    }
    for (int s2 = warp; s2 < A.nsplit; s2 += NW) {
        const size_t base = (size_t)s2 * A.H + hk * G;
        float om[OPL], ol[OPL], oo[OPL];
#pragma unroll
        for (int k = 0; k < OPL; ++k) {
            const int idx = lane + 32 * k, g = idx / D;
            om[k] = __ldcg(A.ws_m + base + g);
            ol[k] = __ldcg(A.ws_l + base + g);
            oo[k] = __ldcg(A.ws_o + base * D + idx);
        }
#pragma unroll
        for (int k = 0; k < OPL; ++k) {
            const float M = fmaxf(pm[k], om[k]);
            const float fa = expf(pm[k] - M), fb = expf(om[k] - M);
            pl[k] = pl[k] * fa + ol[k] * fb;
            po[k] = po[k] * fa + oo[k] * fb;
            pm[k] = M;
        }
    }
    // red: the warps' output shares; wm, wl (free again): their maxima and
    // sums per head (the same in every lane: lane 0's outputs k = g D / 32
    // are head g's)
#pragma unroll
    for (int k = 0; k < OPL; ++k) red[(size_t)warp * G * D + lane + 32 * k] = po[k];
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            wm[warp * G + g] = pm[g * (D / 32)];
            wl[warp * G + g] = pl[g * (D / 32)];
        }
    }
    csync<NW>();
    for (int idx = tid; idx < G * D; idx += NW * 32) {
        const int g = idx / D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w * G + g]);
        float o = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float f = expf(wm[w * G + g] - M);  // 0 for a warp without splits
            o = fmaf(red[(size_t)w * G * D + idx], f, o);
            L = fmaf(wl[w * G + g], f, L);
        }
        A.out[(size_t)(hk * G) * D + idx] = o / L;
    }
    if (tid == 0) A.ws_count[hk] = 0;  // zero again for the next layer and step
}

}  // namespace dev
}  // namespace q4
