// gemm_kernel.cu -- prefill GEMM: y[nb][n] = x[nb][k] W^T for wide activation
// batches (crate inferencelayer, Functions: gemm_q4_src -- a blocked GEMM whose
// column tile shares one weight stream, so the weights are read once per
// column tile instead of once per column; gemm_q4_splitk_src for its fold).
//
// Two launches.  q4gemm_stage_kernel converts x once into the tensor-core
// B-fragment image the GEMM reads: per activation tile (64 rows, or 16 for
// batches of at most 16 rows) and 128-column chunk, every 32-column block of
// a row scaled by its own power of two and carried as one f16 per value (as
// the engine's batch classes above four rows), the block's factor back, and
// its offset term (the zero-weight product times minus the factor back for
// Q4_0 and Q8_0, the fp32 block sum for the formats with a min).  q4gemm_kernel then gives each CTA 64
// weight rows (four 16-row tiles) by one activation tile: a two-stage ring of
// TMA bulk copies brings each chunk's four weight records and its image slice
// into shared memory, and each warp runs one weight tile against its share of
// the tile's 8-row n-tiles with the engine's record decoding and per-block
// scale arithmetic.  The activation tile index runs fastest in the grid, so
// the CTAs that share a weight tile group run together and the weights come
// from HBM about once.
#include "gemv_launch.cuh"

namespace q4 {
namespace dev {

constexpr int kGemmWarps = 8;
constexpr int kGemmSC = 2;      // chunks per ring stage
// ring stages: four for the 16-row activation tile (its stages are small and
// the kernel streams weights), two for the 64-row tile (tensor-bound)
Q4_HD constexpr int gemm_stages(int NT) { return NT == 2 ? 4 : 2; }
// Activation tiles of NT n-tiles (NT * 8 rows): 8 for wide batches, 2 for
// batches of at most 16 rows.  Per tile and 128-column chunk the image holds
// the B fragments [block][n-tile][lane] (16 bytes a lane), then the factors
// and the offsets [block][row] in fp32.
Q4_HD constexpr int gemm_img_b(int NT) { return 4 * NT * 32 * 16; }
Q4_HD constexpr int gemm_img(int NT) { return gemm_img_b(NT) + 2 * 4 * NT * 8 * 4; }

// ---------------------------------------------------------------- staging

template <int FMT, int NT>
__global__ void __launch_bounds__(NT * 32) q4gemm_stage_kernel(const __grid_constant__ GemmParams p) {
    constexpr int ROWS = NT * 8;
    // the GEMM (launched as this kernel's dependent) may start now: it
    // streams weights until it waits for this grid
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int c = blockIdx.x, rt = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int nt = warp;                       // n-tile: activation rows rt*ROWS + nt*8 .. +7
    const int r = rt * ROWS + nt * 8 + g;      // this lane's activation row
    uint8_t *img = p.img + ((size_t)rt * p.C + c) * gemm_img(NT);
    float *F = reinterpret_cast<float *>(img + gemm_img_b(NT)), *Gs = F + 4 * ROWS;
    // lane (g, t) holds columns 8m + 2t, 8m + 2t + 1 of the chunk, m = 0..15:
    // block m / 4, k16 step (m % 4) / 2, positions 0..7 (m even) or 8..15
    float2 v[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int col = c * kChunkK + 8 * m + 2 * t;
        v[m] = (r < p.nb && col < p.K) ? __ldg(reinterpret_cast<const float2 *>(p.x + (size_t)r * p.K + col))
                                       : make_float2(0.f, 0.f);
    }
    const float z = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float bm = 0.f, bs = 0.f;
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            const float2 u = v[4 * j + mm];
            bm = fmaxf(bm, fmaxf(fabsf(u.x), fabsf(u.y)));
            bs += u.x + u.y;
        }
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        float sc, back;
        block_scale<FMT>(bm, sc, back);
        uint32_t b[4];
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            // the nibble formats' positions 0..7 of a step carry the factor 16
            const float f = (is_nibble(FMT) && (mm & 1) == 0) ? 16.f * sc : sc;
            const __half2 h = __floats2half2_rn(v[4 * j + mm].x * f, v[4 * j + mm].y * f);
            b[mm] = *reinterpret_cast<const uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(img + ((size_t)(j * NT + nt) * 32 + lane) * 16) = make_uint4(b[0], b[1], b[2], b[3]);
        if (t == 0) F[j * ROWS + nt * 8 + g] = back;
        if constexpr (has_offset(FMT)) {
            // the block's zero-weight product, through the same tensor-core
            // chain as the weights' (so that zero weights give exactly 0):
            // lane (g, t) ends with rows 2t and 2t + 1 of the n-tile.  Stored
            // times minus the rows' factors back (lanes 8t and 8t + 4 hold
            // them): powers of two, so the product is exact and the GEMM's
            // fma(f, d, -f o) equals f * (d - o) rounded once.
            constexpr uint32_t EL = zero_lo<FMT>();
            float e[4];
            mma16816_c(e, EL, EL, kEightHi, kEightHi, b[0], b[1], z, z, z, z);
            mma16816(e, EL, EL, kEightHi, kEightHi, b[2], b[3]);
            const float f0 = __shfl_sync(0xffffffffu, back, 8 * t), f1 = __shfl_sync(0xffffffffu, back, 8 * t + 4);
            if (g == 0) {
                Gs[j * ROWS + nt * 8 + 2 * t] = -(f0 * e[0]);
                Gs[j * ROWS + nt * 8 + 2 * t + 1] = -(f1 * e[1]);
            }
        } else if constexpr (has_min(FMT)) {
            // the block sum of x (its four lanes' shares, added by a butterfly)
            bs += __shfl_xor_sync(0xffffffffu, bs, 1);
            bs += __shfl_xor_sync(0xffffffffu, bs, 2);
            if (t == 0) Gs[j * ROWS + nt * 8 + g] = bs;
        } else {
            if (t == 0) Gs[j * ROWS + nt * 8 + g] = 0.f;
        }
    }
}

// ---------------------------------------------------------------- GEMM

// A record's per-row scale words for this lane's rows g and g + 8.
template <int FMT>
struct RecScales {
    uint4 sw, mw;
    float2 dd, dm;  // Q4_K: d and dmin factors (q4k_rows)
    __device__ __forceinline__ void load(uint32_t ra, int g) {
        mw = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (FMT == 4) {
            uint32_t w1;
            asm volatile("ld.shared.u32 %0, [%1+256];" : "=r"(w1) : "r"(ra + g * 4) : "memory");
            sw = make_uint4(w1, w1, w1, w1);
        } else {
            sw = lds128_at<scale_off<FMT>()>(ra + g * 16);
        }
        if constexpr (FMT == 1) mw = lds128_at<1152>(ra + g * 16);
        if constexpr (FMT == 3) {
            uint32_t dw, dmw;
            asm volatile("ld.shared.u32 %0, [%1+1152];" : "=r"(dw) : "r"(ra + g * 4) : "memory");
            asm volatile("ld.shared.u32 %0, [%1+1184];" : "=r"(dmw) : "r"(ra + g * 4) : "memory");
            q4k_rows(dw, dmw, dd, dm);
        }
    }
    // block J's scales (and mins) of rows g and g + 8
    template <int J>
    __device__ __forceinline__ void block(float2 &s2, float2 &m2) const {
        m2 = make_float2(0.f, 0.f);
        if constexpr (FMT == 3) {
            q4k_pair(word_of<J>(sw), dd, dm, s2, m2);
        } else {
            s2 = scale_pair<FMT>(word_of<J>(sw));
            if constexpr (FMT == 1) m2 = scale_pair<FMT>(word_of<J>(mw));
        }
    }
};

template <int FMT, int NT>
__global__ void __launch_bounds__(kGemmWarps * 32, 2) q4gemm_kernel(const __grid_constant__ GemmParams p) {
    constexpr int REC = rec_bytes(FMT), SC = kGemmSC, S = gemm_stages(NT);
    constexpr int ROWS = NT * 8, NTW = NT / 2, IMG = gemm_img(NT), IMGB = gemm_img_b(NT);
    constexpr int WB = 4 * SC * REC;            // weight bytes of a stage (four tiles)
    constexpr int STAGE = WB + SC * IMG;        // stage bytes
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int rt = blockIdx.x, tg = blockIdx.y;  // activation tile (fastest), weight tile group
    const int wt = warp & 3, ng = warp >> 2;     // this warp: weight tile, n-tiles NTW ng .. NTW ng + NTW - 1
    const int tile = 4 * tg + wt;
    const bool tile_ok = tile < p.T;
    const int nst = (p.C + SC - 1) / SC;
    const uint32_t bars = smem_u32(smem);
    uint8_t *ring = smem + 16 * S;
    const uint64_t pol = evict_first_policy();

    // stage k (chunks k*SC ..): the weight records, then the image slice;
    // both complete on the stage's barrier (thread 0 only)
    auto issue_w = [&](int k) {
        const int c0 = k * SC, n = min(SC, p.C - c0);
        uint8_t *st = ring + (size_t)(k % S) * STAGE;
        const uint32_t bar = bars + 8 * (k % S);
        const int tiles = min(4, p.T - 4 * tg);
        // extra_tx: testing the give-up path only
        mbar_expect_tx(bar, (uint32_t)(tiles * n * REC + n * IMG) + (k == 0 ? (uint32_t)p.extra_tx : 0u));
        for (int i = 0; i < tiles; ++i)
            bulk_g2s(smem_u32(st + i * SC * REC), p.w + ((size_t)(4 * tg + i) * p.C + c0) * REC, n * REC, bar, pol);
    };
    auto issue_img = [&](int k) {
        const int c0 = k * SC, n = min(SC, p.C - c0);
        uint8_t *st = ring + (size_t)(k % S) * STAGE;
        bulk_g2s(smem_u32(st + WB), p.img + ((size_t)rt * p.C + c0) * IMG, n * IMG, bars + 8 * (k % S), pol);
    };
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bars + 8 * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // weights do not depend on the staging kernel: their first copies go out
    // before waiting for it, the image slices after
    if (tid == 0)
        for (int k = 0; k < min(S, nst); ++k) issue_w(k);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0)
        for (int k = 0; k < min(S, nst); ++k) issue_img(k);

    float acc[NTW][4];
#pragma unroll
    for (int i = 0; i < NTW; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
    const float z = 0.f;
    bool ok = true;
    int waited = 0;
    for (int k = 0; k < nst; ++k) {
        ok = __syncthreads_and(mbar_wait(bars + 8 * (k % S), (uint32_t)(k / S) & 1u, p.wait_cycles));
        if (!ok) break;
        waited = k + 1;
        const int n = min(SC, p.C - k * SC);
        const uint8_t *st = ring + (size_t)(k % S) * STAGE;
        if (tile_ok) {  // warp-uniform
            for (int cc = 0; cc < n; ++cc) {
                const uint32_t ra = smem_u32(st + wt * SC * REC + cc * REC);
                const uint8_t *img = st + WB + cc * IMG;
                const float *F = reinterpret_cast<const float *>(img + IMGB), *Gs = F + 4 * ROWS;
                RecWords<FMT> rw;
                rw.load(ra, lane);
                RecScales<FMT> rs;
                rs.load(ra, g);
                auto block = [&](auto jc) {
                    constexpr int J = decltype(jc)::value;
                    uint32_t a[8];
                    rw.template regs<J>(a);
                    float2 s2, m2;
                    rs.template block<J>(s2, m2);
#pragma unroll
                    for (int i = 0; i < NTW; ++i) {
                        const int ntl = NTW * ng + i;
                        const uint4 B = *reinterpret_cast<const uint4 *>(img + ((size_t)(J * NT + ntl) * 32 + lane) * 16);
                        float d[4];
                        mma16816_c(d, a[0], a[1], a[2], a[3], B.x, B.y, z, z, z, z);
                        mma16816(d, a[4], a[5], a[6], a[7], B.z, B.w);
                        const float2 f = *reinterpret_cast<const float2 *>(F + J * ROWS + ntl * 8 + 2 * t);
                        const float2 o = *reinterpret_cast<const float2 *>(Gs + J * ROWS + ntl * 8 + 2 * t);
                        // d: (row g, cols 2t, 2t+1), (row g+8, cols 2t, 2t+1)
                        if constexpr (has_offset(FMT)) {  // o = -f * offset: s * f * (d - offset)
                            acc[i][0] = fmaf(s2.x, fmaf(f.x, d[0], o.x), acc[i][0]);
                            acc[i][1] = fmaf(s2.x, fmaf(f.y, d[1], o.y), acc[i][1]);
                            acc[i][2] = fmaf(s2.y, fmaf(f.x, d[2], o.x), acc[i][2]);
                            acc[i][3] = fmaf(s2.y, fmaf(f.y, d[3], o.y), acc[i][3]);
                        } else if constexpr (has_min(FMT)) {
                            acc[i][0] = fmaf(m2.x, o.x, fmaf(s2.x * f.x, d[0], acc[i][0]));
                            acc[i][1] = fmaf(m2.x, o.y, fmaf(s2.x * f.y, d[1], acc[i][1]));
                            acc[i][2] = fmaf(m2.y, o.x, fmaf(s2.y * f.x, d[2], acc[i][2]));
                            acc[i][3] = fmaf(m2.y, o.y, fmaf(s2.y * f.y, d[3], acc[i][3]));
                        } else {
                            acc[i][0] = fmaf(s2.x * f.x, d[0], acc[i][0]);
                            acc[i][1] = fmaf(s2.x * f.y, d[1], acc[i][1]);
                            acc[i][2] = fmaf(s2.y * f.x, d[2], acc[i][2]);
                            acc[i][3] = fmaf(s2.y * f.y, d[3], acc[i][3]);
                        }
                    }
                };
                block(std::integral_constant<int, 0>());
                block(std::integral_constant<int, 1>());
                block(std::integral_constant<int, 2>());
                block(std::integral_constant<int, 3>());
            }
        }
        __syncthreads();  // the stage is free again
        if (tid == 0 && k + S < nst) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_w(k + S);
            issue_img(k + S);
        }
    }
    if (!ok) {
        // a wait gave up: record it, let the copies in flight land, store nothing
        if (tid == 0) {
            atomicExch(p.err, 4);
            for (int k = waited; k < min(nst, waited + S); ++k)
                mbar_wait(bars + 8 * (k % S), (uint32_t)(k / S) & 1u, kWaitCycles);
        }
        __syncthreads();
        return;
    }
    if (!tile_ok) return;
#pragma unroll
    for (int i = 0; i < NTW; ++i) {
        const int col0 = rt * ROWS + (NTW * ng + i) * 8 + 2 * t;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int row = tile * 16 + g + (e >= 2 ? 8 : 0), col = col0 + (e & 1);
            if (row < p.n && col < p.nb) {
                float *dst = p.y + (size_t)col * p.n + row;
                *dst = p.accumulate ? *dst + acc[i][e] : acc[i][e];
            }
        }
    }
}

}  // namespace dev

// activation tile of a batch: 16 rows (2 n-tiles) up to 16 rows, else 64
static int gemm_nt(int nb) { return nb <= 16 ? 2 : 8; }
size_t gemm_image_bytes(int nb, int C) {
    const int NT = gemm_nt(nb);
    return (size_t)((nb + NT * 8 - 1) / (NT * 8)) * C * dev::gemm_img(NT);
}
size_t gemm_smem_bytes(int fmt, int nb) {
    const int NT = gemm_nt(nb), S = dev::gemm_stages(NT);
    return 16 * S + (size_t)S * (4 * dev::kGemmSC * rec_bytes(fmt) + dev::kGemmSC * dev::gemm_img(NT));
}

template <int FMT, int NT>
static int launch_gemm_nt(const GemmParams &p, cudaStream_t stream) {
    auto kern = dev::q4gemm_kernel<FMT, NT>;
    static size_t smem_set[64] = {0};
    const size_t smem = gemm_smem_bytes(FMT, NT == 2 ? 16 : 64);
    if (!raise_smem(kern, smem, smem_set)) return -1;
    const int RT = (p.nb + NT * 8 - 1) / (NT * 8);
    // staging: an ordinary launch (it overwrites the image a previous call's
    // GEMM may still be reading)
    dev::q4gemm_stage_kernel<FMT, NT><<<dim3(p.C, RT), NT * 32, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -1;
    // the GEMM as its programmatic dependent
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)RT, (unsigned)((p.T + 3) / 4), 1);
    cfg.blockDim = dim3(dev::kGemmWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? 0 : -1;
}

template <int FMT>
static int launch_gemm_fmt(const GemmParams &p, cudaStream_t stream) {
    return gemm_nt(p.nb) == 2 ? launch_gemm_nt<FMT, 2>(p, stream) : launch_gemm_nt<FMT, 8>(p, stream);
}

int launch_gemm(const GemmParams &p, int fmt, void *stream_) {
    cudaStream_t stream = (cudaStream_t)stream_;
    switch (fmt) {
        case 0: return launch_gemm_fmt<0>(p, stream);
        case 1: return launch_gemm_fmt<1>(p, stream);
        case 2: return launch_gemm_fmt<2>(p, stream);
        case 3: return launch_gemm_fmt<3>(p, stream);
        case 4: return launch_gemm_fmt<4>(p, stream);
    }
    return -1;
}

}  // namespace q4
