// attn_kernel.cu -- decode attention over an f32 KV cache (honeycrisp/mod.rs:
// gpu_attention, and the fused RoPE + KV-append + SDPA dispatch of
// forward_decode_fused_layers).  One token: optional RoPE of q and the new
// k, append of k and v at `position`, then for every query head the softmax
// of scale * q K^T over the attended positions times V.
//
// The work is HBM-bound on the cache rows.  CTA (s, hk) takes kv head hk and
// the s-th split of the attended positions, about one CTA per SM slot.  Its K
// and V rows are contiguous in the cache: it walks them in sub-chunks of LS
// positions through a ring of shared-memory stages that TMA bulk copies fill
// (K and V on their own mbarriers, two stages ahead), each warp keeping a
// running softmax per head over its positions (flash decoding); every query
// head of the group reuses each row.  The last split of a kv head to finish folds the splits' shares in
// split order: one launch, and a result that does not depend on the order in
// which the CTAs ran.  The launch is a programmatic dependent of the kernel
// before it (the projection that writes q, k and v), so CTAs that find an SM
// free start while it runs and warm L2 with their first cache rows.
#include "attn_common.cuh"
#include "gemv_launch.cuh"

namespace q4 {
namespace dev {

constexpr int kAttnWarps = 8;
constexpr int kAttnStages = 2;  // ring stages of K and V sub-chunks

// Positions per sub-chunk: a stage holds LS rows of K and LS rows of V.
Q4_HD constexpr int attn_sub(int D) { return D == 64 ? 64 : 32; }

// Shared memory of a CTA: 2 mbarriers per stage (64 bytes in all), the ring
// (per stage LS rows of K, then of V; at the end it holds the fold weights),
// the warps' outputs [NW][G * D], their running maxima and sums [NW][G], the
// fold's sums [G], per warp one step's 32 softmax weights and G rescale
// factors, and the last-split flag.
//
// Each warp keeps its own running softmax over the positions it scores (per
// head: maximum, sum, and the output, rescaled whenever the maximum grows), so
// a sub-chunk needs one CTA barrier, the one that frees its stage; the warps'
// states are merged at the end.
template <int D, int G>
__global__ void __launch_bounds__(kAttnWarps * 32, (G * D <= 512 ? 2 : 1))
    q4attn_split_kernel(const __grid_constant__ AttnParams p) {
    constexpr int DL = D / 32, P = 32 / G, NW = kAttnWarps, S = kAttnStages, LS = attn_sub(D);
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, hk = blockIdx.y;
    const int per = p.Lc;  // positions of each split (the last may have fewer)
    const int t0 = p.lo + split * per;
    const int n = min(per, p.total - t0);  // >= 1
    const int nsub = (n + LS - 1) / LS;
    const bool owner = t0 + n == p.total;  // this split ends with the new token
    const uint32_t bars = smem_u32(smem);  // stage s: K barrier at bars + 16 s, V barrier 8 bytes on
    float *ring = reinterpret_cast<float *>(smem + 64);
    float *red = ring + (size_t)S * 2 * LS * D;
    float *wm = red + NW * G * D, *wl = wm + NW * G, *Lg = wl + NW * G;
    float *eb = Lg + G, *ab = eb + NW * 32;  // per warp: this step's exp(s - max) and rescale factors
    int *flag = reinterpret_cast<int *>(ab + NW * G);
    const size_t row0 = ((size_t)hk * p.max_seq + t0) * D;
    const uint64_t pol = evict_first_policy();

    // sub-chunk j's K and V rows into stage j % S (thread 0 only)
    auto issue = [&](int j) {
        const int st = j % S, rows = min(LS, n - j * LS);
        const uint32_t bytes = (uint32_t)rows * D * 4;
        float *kst = ring + (size_t)st * 2 * LS * D;
        const uint32_t bk = bars + 16 * st, bv = bk + 8;
        mbar_expect_tx(bk, bytes + (j == 0 ? p.extra_tx : 0));  // extra_tx: testing the give-up path only
        bulk_g2s(smem_u32(kst), p.k_cache + row0 + (size_t)j * LS * D, bytes, bk, pol);
        mbar_expect_tx(bv, bytes);
        bulk_g2s(smem_u32(kst + LS * D), p.v_cache + row0 + (size_t)j * LS * D, bytes, bv, pol);
    };
    // Launched as a programmatic dependent of the previous kernel, which may
    // still be running: until griddepcontrol.wait nothing it (or anything
    // before it) writes is read -- the first stages' K and V rows only go to
    // L2, a hint that cannot return old data.  The next kernel may launch now;
    // it waits for this one to finish before it reads what this one writes.
    if (tid == 0) {
        const uint32_t pre = (uint32_t)min(n, S * LS) * D * 4;
        bulk_prefetch_l2(p.k_cache + row0, pre);
        bulk_prefetch_l2(p.v_cache + row0, pre);
        for (int st = 0; st < S; ++st) {
            mbar_init(bars + 16 * st, 1);
            mbar_init(bars + 16 * st + 8, 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0)
        for (int j = 0; j < min(S, nsub); ++j) issue(j);

    // while the rows arrive: the group's query heads (rotated) in registers,
    // and for the split with the new token its k (rotated) and v
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
    // this warp's running softmax: lane l keeps head l % G's maximum and sum
    // (the same in every lane of that head), and every lane the output share
    // of its dims for every head
    float mh = -INFINITY, lh = 0.f;
    float acc[G][DL];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[g][e] = 0.f;

    bool ok = true;
    int waited = 0;  // sub-chunks whose copies have landed
    for (int j = 0; j < nsub; ++j) {
        const int st = j % S, rows = min(LS, n - j * LS);
        const uint32_t par = (uint32_t)(j / S) & 1u;
        float *Ks = ring + (size_t)st * 2 * LS * D, *Vs = Ks + LS * D;
        bool mine = mbar_wait(bars + 16 * st, par, p.wait_cycles);
        mine = mine && mbar_wait(bars + 16 * st + 8, par, p.wait_cycles);
        ok = __syncthreads_and(mine);
        if (!ok) break;
        waited = j + 1;
        if (owner && j == nsub - 1) {  // append k and v: the caches, and this stage's copies
            if (warp < 2) {
                float *srow = (warp == 0 ? Ks : Vs) + (size_t)(rows - 1) * D + lane * DL;
                float *grow = (warp == 0 ? p.k_cache : p.v_cache) + row0 + (size_t)(n - 1) * D + lane * DL;
#pragma unroll
                for (int e = 0; e < DL; ++e) {
                    srow[e] = kv[e];
                    grow[e] = kv[e];
                }
            }
            __syncthreads();
        }
        for (int i = warp; i * P < rows; i += NW) {
            // scores of positions i*P .. i*P+P-1 for every head: lane l ends
            // with position l / G, head l % G
            float v[32];
#pragma unroll
            for (int pp = 0; pp < P; ++pp) {
                const int r = i * P + pp;
                float kr[DL];
                if (r < rows) {
                    load_row<DL>(kr, Ks + (size_t)r * D + lane * DL);
                } else {
#pragma unroll
                    for (int e = 0; e < DL; ++e) kr[e] = 0.f;
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float s = 0.f;
#pragma unroll
                    for (int e = 0; e < DL; ++e) s = fmaf(qr[g][e], kr[e], s);
                    v[pp * G + g] = s;
                }
            }
            const float t = transpose_reduce(v, lane);
            const bool valid = i * P + lane / G < rows;
            const float s = valid ? t * p.scale : -INFINITY;
            // the head's maximum over these positions (lanes l, l ^ G, ...),
            // the factor that rescales what came before, exp(s - max), sum
            float mx = s;
#pragma unroll
            for (int o = G; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mnew = fmaxf(mh, mx);  // finite: position i*P is valid
            const float alpha = expf(mh - mnew);  // 0 the first time
            const float e = valid ? expf(s - mnew) : 0.f;
            float sum = e;
#pragma unroll
            for (int o = G; o < 32; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            lh = fmaf(lh, alpha, sum);
            mh = mnew;
            // output: rescale each head (lane g holds head g's factor), then
            // add these positions' rows of V weighted by their exp(s - max);
            // both reach every lane through the warp's own shared-memory slots
            float *ew = eb + warp * 32, *aw = ab + warp * G;
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
                const int r = i * P + pp;
                if (r < rows) {  // warp-uniform
                    float vr[DL], w[G];
                    load_row<DL>(vr, Vs + (size_t)r * D + lane * DL);
                    load_vec<G>(w, ew + pp * G);
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int q2 = 0; q2 < DL; ++q2) acc[g][q2] = fmaf(w[g], vr[q2], acc[g][q2]);
                }
            }
            __syncwarp();  // the slots are read before the next step writes them
        }
        __syncthreads();  // the stage is free again
        if (tid == 0 && j + S < nsub) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(j + S);
        }
    }
    if (!ok) {
        // a wait gave up: record it and let the copies in flight land before
        // the CTA goes on (its share is not valid; it still joins the fold
        // count, so the count is right for the next call)
        if (tid == 0) {
            atomicExch(p.err, 3);
            for (int j = waited; j < min(nsub, waited + S); ++j) {
                const uint32_t par = (uint32_t)(j / S) & 1u;
                mbar_wait(bars + 16 * (j % S), par, kWaitCycles);
                mbar_wait(bars + 16 * (j % S) + 8, par, kWaitCycles);
            }
        }
        __syncthreads();
    }

    // merge the warps, in warp order: M = max_w m_w, L = sum_w l_w e^(m_w - M),
    // o = sum_w o_w e^(m_w - M) (a warp without positions has m_w = -inf)
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < DL; ++e) red[(size_t)warp * G * D + g * D + lane * DL + e] = acc[g][e];
    if (lane < G) {
        wm[warp * G + lane] = mh;
        wl[warp * G + lane] = lh;
    }
    __syncthreads();
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
        if (p.nsplit == 1) {
            p.out[(size_t)hq * D + d] = o / L;
        } else {
            p.ws_o[((size_t)split * p.H + hq) * D + d] = o;
            if (d == 0) {
                p.ws_m[(size_t)split * p.H + hq] = M;
                p.ws_l[(size_t)split * p.H + hq] = L;
            }
        }
    }
    if (p.nsplit == 1) return;

    // the last split of this kv head to finish folds every split's share in
    // split order: out = sum_s o_s e^(m_s - M) / sum_s l_s e^(m_s - M)
    __threadfence();
    __syncthreads();
    if (tid == 0) *flag = atomicAdd(p.ws_count + hk, 1) == p.nsplit - 1;
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    float *wts = ring;  // [nsplit][G]: the splits' weights e^(m_s - M)
    for (int g = warp; g < G; g += NW) {
        const int hq = hk * G + g;
        float M = -INFINITY;
        for (int s2 = lane; s2 < p.nsplit; s2 += 32) M = fmaxf(M, __ldcg(p.ws_m + (size_t)s2 * p.H + hq));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        for (int s2 = lane; s2 < p.nsplit; s2 += 32) {
            const float w = expf(__ldcg(p.ws_m + (size_t)s2 * p.H + hq) - M);
            wts[s2 * G + g] = w;
            L = fmaf(__ldcg(p.ws_l + (size_t)s2 * p.H + hq), w, L);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) Lg[g] = L;
    }
    __syncthreads();
    // warp w adds the splits w, w + NW, ... for every output (lane l: outputs
    // l, l + 32, ...), all their loads in flight together; then the warps'
    // sums are added in warp order
    constexpr int OPL = G * D / 32;
    float part[OPL];
#pragma unroll
    for (int k = 0; k < OPL; ++k) part[k] = 0.f;
    for (int s2 = warp; s2 < p.nsplit; s2 += NW) {
        const float *src = p.ws_o + ((size_t)s2 * p.H + hk * G) * D;
#pragma unroll
        for (int k = 0; k < OPL; ++k) {
            const int idx = lane + 32 * k;
            part[k] = fmaf(__ldcg(src + idx), wts[s2 * G + idx / D], part[k]);
        }
    }
#pragma unroll
    for (int k = 0; k < OPL; ++k) red[(size_t)warp * G * D + lane + 32 * k] = part[k];
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += NW * 32) {
        const int g = idx / D;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) o += red[(size_t)w * G * D + idx];
        p.out[(size_t)(hk * G) * D + idx] = o / Lg[g];
    }
    if (tid == 0) p.ws_count[hk] = 0;  // zero again for the next call
}

}  // namespace dev

size_t attn_smem_bytes(int D, int G) {
    const int LS = dev::attn_sub(D), NW = dev::kAttnWarps;
    return 64 + (size_t)dev::kAttnStages * 2 * LS * D * 4 + (size_t)NW * G * D * 4 +
           (size_t)(2 * NW * G + G + NW * 32 + NW * G) * 4 + 16;
}
// splits one fold can weigh: its weights [nsplit][G] reuse the ring
int attn_max_splits(int D, int G) { return dev::kAttnStages * 2 * dev::attn_sub(D) * D / G; }
int attn_sub_chunk(int D) { return dev::attn_sub(D); }
int attn_ctas_per_sm(int D, int G) { return G * D <= 512 ? 2 : 1; }

template <int D, int G>
static int launch_attn_dg(const AttnParams &p, cudaStream_t stream) {
    auto kern = dev::q4attn_split_kernel<D, G>;
    static size_t smem_set[64] = {0};
    const size_t smem = attn_smem_bytes(D, G);
    if (!raise_smem(kern, smem, smem_set)) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.nsplit, (unsigned)p.Hkv, 1);
    cfg.blockDim = dim3(dev::kAttnWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? 0 : -1;
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
