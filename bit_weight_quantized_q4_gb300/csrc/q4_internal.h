// q4_internal.h -- shared definitions of libq4gemv: the device weight layout,
// the kernel parameter block and the launch planner.
#pragma once
#include <stddef.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define Q4_HD __host__ __device__
#else
#define Q4_HD
#endif

namespace q4 {

// ---------------------------------------------------------------- layout
// A weight matrix is cut into 16-row tiles and, along k, into 128-column
// chunks (4 blocks of 32).  Tile t's chunks are stored one after another;
// one chunk of one tile is one contiguous record:
//
//   bytes [   0,  512)  nibble words of rows 0..7   (32 lanes x 16 B)
//   bytes [ 512, 1024)  nibble words of rows 8..15  (32 lanes x 16 B)
//   bytes [1024, 1152)  scales: 8 groups x 4 words; word j of group g holds
//                       the 16-bit scale of (row g, block j) in its low half
//                       and of (row g+8, block j) in its high half
//   bytes [1152, 1280)  affine only: the mins, laid out like the scales
//
// Lane L = 4*g + t (g = 0..7, t = 0..3) owns 16 bytes = 4 words, word j for
// block j of the chunk.  The 8 nibbles of that word are the weights lane L
// needs for the tensor-core A fragment of row g (or g+8) in that block:
// nibble i (bits 4i..4i+3) holds block element kNibElem[t][i].
constexpr int kTileRows = 16;
constexpr int kChunkK = 128;
constexpr int kBlocksPerChunk = 4;
constexpr int kRecQ4_0 = 1152;
constexpr int kRecAffine = 1280;
// Q8_0 records (2176 bytes): the biased bytes u = q + 128 of rows 0..7 in
// [0, 1024) and of rows 8..15 in [1024, 2048), then the scales as for Q4_0
// at [2048, 2176).  In each half, blocks 0-1 come first ([0, 512)) and
// blocks 2-3 after ([512, 1024)); lane L owns 16 bytes of each: the 8 bytes of
// its row's first block of the pair, then of the second.  Byte i of a lane's
// 8 holds block element q8_elem(t, i).
constexpr int kRecQ8_0 = 2176;
// Q4_K records (1216 bytes): the nibble words as for Q4_0 at [0, 1024); at
// [1024, 1152) word j of group g holds the bytes sc(g, j), mn(g, j),
// sc(g+8, j), mn(g+8, j) -- the 6-bit scale and min of block j of rows g and
// g+8; at [1152, 1184) word g holds the fp16 d of rows g (low half) and g+8
// (high half) of the superblock the chunk belongs to, and at [1184, 1216) their
// fp16 dmin.  A 256-column superblock spans two chunks; each carries d, dmin.
constexpr int kRecQ4_K = 1216;
// Q1 records (288 bytes): a 128-column chunk is one Q1 superblock.  Lane
// L = 4g + t owns 8 bytes at [8L, 8L + 8): the 32 sign bits of row g, then of
// row g + 8, each bit inverted (a set stored bit is -d), bit rho (0..15) for
// element q1_elem(t, rho) and bit 16 + rho for the element after it; then at
// [256, 288) word g holds the fp16 d of rows g (low half) and g + 8.
constexpr int kRecQ1 = 288;

// Chunk element (0..127) of Q1 bit rho (0..15) of lane-position t: register
// rho = 2s + h of the tensor-core A fragment of k16 step s, its first k
// (h = 0: columns 2t, 2t+1 of the step; h = 1: 2t+8, 2t+9).
inline int q1_elem(int t, int rho) { return 16 * (rho >> 1) + 8 * (rho & 1) + 2 * t; }

// Block element (0..31) stored in nibble i of lane-position t's word.
// Pairs (i, i+4) are (k, k+1) of one f16x2 fragment register:
//   i=0/4: k = 2t, 2t+1        (first k16 step, columns 0..7)
//   i=1/5: k = 2t+8, 2t+9      (first k16 step, columns 8..15)
//   i=2/6: k = 16+2t, 17+2t    (second k16 step, columns 0..7)
//   i=3/7: k = 24+2t, 25+2t    (second k16 step, columns 8..15)
inline int nib_elem(int t, int i) {
    const int base[4] = {0, 8, 16, 24};
    return base[i & 3] + 2 * t + (i >> 2);
}

// Block element (0..31) stored in byte i of lane-position t's 8 bytes of a
// Q8_0 block: pairs (i, i+1) are (k, k+1) of one f16x2 fragment register
// (bytes 0-1: k = 2t, 2t+1; 2-3: 2t+8, 2t+9; 4-5: 16+2t, 17+2t; 6-7: 24+2t,
// 25+2t).
inline int q8_elem(int t, int i) {
    const int base[4] = {0, 8, 16, 24};
    return base[i >> 1] + 2 * t + (i & 1);
}

Q4_HD constexpr int rec_bytes(int fmt) {
    return fmt == 0 ? kRecQ4_0 : fmt == 1 ? kRecAffine : fmt == 2 ? kRecQ8_0 : fmt == 3 ? kRecQ4_K : kRecQ1;
}
// Formats whose weights carry a per-block min (w = s*q + m): the products
// need the activation block sums.
Q4_HD constexpr bool has_min(int fmt) { return fmt == 1 || fmt == 3; }
// Formats stored with an offset (Q4_0's q - 8, Q8_0's bias of 128): the
// products need the block's zero-weight (offset) product.
Q4_HD constexpr bool has_offset(int fmt) { return fmt == 0 || fmt == 2; }
// Nibble formats: a lower nibble meets its activation times 16.
Q4_HD constexpr bool is_nibble(int fmt) { return fmt == 0 || fmt == 1 || fmt == 3; }
inline int64_t tiles_of(int64_t n) { return (n + kTileRows - 1) / kTileRows; }
inline int64_t chunks_of(int64_t k) { return (k + kChunkK - 1) / kChunkK; }

// ---------------------------------------------------------------- kernel
enum Mode { MODE_SINGLE = 0, MODE_CONCAT = 1, MODE_PAIRS = 2 };
enum Epi { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SWIGLU = 2, EPI_ARGMAX = 3, EPI_ATTN = 4 };


constexpr int kMaxNb = 16;
constexpr int kMaxCluster = 8;
constexpr size_t kXsCap = 64 * 1024;          // activation slice staged per CTA
constexpr size_t kSmemMax = 227 * 1024;       // dynamic shared memory of one CTA
constexpr int kMaxMats = 3;                   // matrices of one job (q, k, v share one input)

// Batch classes.  The activation rows of a launch become the n columns of
// the m16n8k16 tensor-core products:
//   class 0 (nb = 1) and 1 (nb = 2..4): the hi and lo halves of row r are
//     columns 2r and 2r+1 -- two mma per 32-weight block;
//   class 2 (nb = 5..8): row r is column r, hi and lo are two k-steps into
//     one accumulator -- four mma per block;
//   class 3 (nb = 9..16): as class 2 over two 8-column n-tiles -- eight.
Q4_HD constexpr int cls_of(int nb) { return nb <= 1 ? 0 : nb <= 4 ? 1 : nb <= 8 ? 2 : 3; }
Q4_HD constexpr int cls_warps(int c) { return c == 3 ? 8 : 16; }     // warps per CTA
Q4_HD constexpr int cls_depth(int c) { return (void)c, 2; }  // ring stages per warp
Q4_HD constexpr int cls_stage(int c) { return c == 2 ? 1 : 2; }  // pair units per stage (2x as many single-tile units)
// pair units per ring stage for a format: Q8_0 records are nearly twice as
// large, so its stages hold one; Q1 records a quarter, so its stages hold
// four times as many
Q4_HD constexpr int stage_su(int fmt, int c) { return fmt == 2 ? 1 : fmt == 4 ? 4 * cls_stage(c) : cls_stage(c); }
Q4_HD constexpr int cls_gsw(int c) { return c <= 1 ? 4 : c == 2 ? 8 : 16; }  // group-sum rows per chunk
// bytes of one activation row per 32-column block in shared memory: f16 hi
// and lo parts for nb <= 4, the f16 value alone for larger batches
Q4_HD constexpr int cls_xrow(int c) { return c <= 1 ? 128 : 64; }

// A unit of work is one 128-column chunk of upt consecutive 16-row tiles
// (upt records).  upt is 2 -- a tile pair (2p, 2p+1), for gate/up jobs
// (gate tile p, up tile p) -- unless a job has fewer pairs than the CTAs
// that run it, then 1.
struct GemvParams {
    const uint8_t *w[kMaxMats];  // packed weights
    int n[kMaxMats];             // output rows of each matrix
    int tiles[kMaxMats];         // 16-row tiles of each matrix
    int nmat;                    // matrices in use
    int mode;                    // Mode
    int T;                       // tiles of the job (sum, or 2x for pairs)
    int K;                       // input length
    int C;                       // 128-column chunks per row
    int nb;                      // activation rows
    int TG;                      // most tiles one group holds (sizes shared memory)
    int SW;                      // tile slots per warp for partial sums (sizes shared memory)
    int upt;                     // tiles per unit: 2, or 1 for jobs with few tiles
    int S;                       // K-split: CTAs per cluster
    int Cs;                      // chunks per K-slice
    int groups;                  // groups; group g holds units [g*P/groups, (g+1)*P/groups) of the P = T/upt
    const float *x;              // [nb][K], or nullptr when the activations come as a HalfSet (xe, xo)
    const uint16_t *xe, *xo;     // HalfSet: f16 bits of x[r][2i] and x[r][2i+1], [nb][K/2] each; or nullptr
    const float *gamma;          // [K] or nullptr (no RMSNorm)
    float eps;
    const float *gsum;           // affine: caller group sums [nb][K/32] or nullptr
    int epi;                     // Epi
    float *out[kMaxMats];        // y per matrix (swiglu: out[0] = h; argmax: logits or nullptr)
    const float *res;            // residual [nb][n0]
    float *am_val;               // argmax partials [nb][groups]
    int *am_idx;
    int *err;                    // set nonzero if a kernel wait gave up
    long long wait_cycles;       // bound of one weight-copy wait (SM clock cycles)
    int extra_tx;                // bytes a copy stage expects beyond its copies (0; testing the give-up path only)
    int layer;                   // EPI_ATTN (persistent step only): the layer, an index into StepAttn's caches
};

// One CTA group's share of a job: its first tile, tile pairs (units of upt
// tiles) and tiles.  The persistent kernel computes every job's once at
// start, so that moving to the next job costs no division.
struct JobSpan {
    int t0, np, tiles, pad;
};

// The persistent decode-step kernel runs these jobs in order, one CTA per SM.
constexpr int kMaxStepJobs = 4 * 32 + 1;      // four jobs per layer, up to 32 layers, + logits
constexpr int kMaxStepLayers = 32;

// The persistent step's decode attention (q4_decode_step_attn): one job per
// layer between the q/k/v job and the o job.  Geometry fixed at head size
// 64 and four query heads per kv head.  CTA c takes kv head c / cps and
// split c % cps of the attended positions [lo, total) -- Lc positions each,
// nsplit of them in use -- and the last split of a kv head to finish folds
// the splits' shares (ws_count[hk], zero again when it has).
constexpr int kStepAttnD = 64, kStepAttnG = 4;
struct StepAttn {
    const float *q, *k_new, *v_new;            // the q/k/v job's outputs: [H][D], [Hkv][D], [Hkv][D]
    const float *rope_cos, *rope_sin;          // [max_seq][D/2], or nullptr (no RoPE)
    float *out;                                // [H][D]: the o job's input
    float *ws_o, *ws_m, *ws_l;                 // [nsplit][H][D], [nsplit][H], [nsplit][H]
    int *ws_count;                             // [Hkv]
    float *k_cache[kMaxStepLayers];            // per layer [Hkv][max_seq][D]
    float *v_cache[kMaxStepLayers];
    int max_seq, position, H, Hkv, lo, total, Lc, nsplit, cps;
    float scale;
};
constexpr long long kBarrierSpins = 1ll << 22;  // polls before a grid barrier gives up
constexpr long long kWaitCycles = 1ll << 31;    // about a second: bound of one mbarrier wait

struct StepParams {
    int njobs;
    int nb;
    int Kmax;                    // largest K of the jobs (sizes the activation slice)
    int TGmax;                   // most tiles any group holds in any job
    int SWmax;                   // most tile slots per warp of any job
    unsigned *counter;           // grid-barrier arrivals (zeroed before each launch)
    unsigned *release;           // number of the last completed barrier (zeroed before each launch)
    int *err;                    // set to 1 if a barrier gave up
    int32_t *idx;                // [nb] argmax of the last job
    float *val;                  // [nb] or nullptr
    long long barrier_polls;     // polls before a grid barrier gives up
    int barrier_extra;           // arrivals a barrier expects beyond the CTAs (0; testing the give-up path only)
    int attn;                    // the jobs include EPI_ATTN jobs (q4_decode_step_attn)
    GemvParams jobs[kMaxStepJobs];
    StepAttn att;                // their parameters (attn only)
};

#if defined(__CUDACC__)
// Block sum of 32 activations held as a float4 by each of 8 consecutive
// lanes: (v.x + v.y) + (v.z + v.w) per lane, then a butterfly over lane xor
// 1, 2, 4; every lane of the 8 ends with the same value.  The affine block
// sums of the staged activations and q4_group_sums both add this way, so the
// two give the same bits.  half_warp_sum over column pairs (lanes 0..15 and
// 16..31 holding x[2j] + x[2j+1]) adds in the same order: its first step
// forms the same four-column sums, its other three the same butterfly.
__device__ __forceinline__ float block8_sum(float4 v) {
    float t = (v.x + v.y) + (v.z + v.w);
    t += __shfl_xor_sync(0xffffffffu, t, 1);
    t += __shfl_xor_sync(0xffffffffu, t, 2);
    t += __shfl_xor_sync(0xffffffffu, t, 4);
    return t;
}
__device__ __forceinline__ float half_warp_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    return v;
}
#endif

// Dynamic shared memory of one engine CTA: activation slice (B fragments),
// group sums, tile results (only for a cluster fold, S > 1), per-warp tile
// partials, reductions, weight ring.
inline size_t engine_smem(int fmt, int nb, int TG, int Cs, int SW, int S) {
    const int c = cls_of(nb);
    const size_t NW = (size_t)cls_warps(c);
    const size_t xs = (size_t)4 * cls_xrow(c) * nb * Cs;
    const size_t gs = (size_t)2 * 16 * cls_gsw(c) * Cs;  // block sums and block factors
    const size_t red = S > 1 ? (size_t)64 * (TG + 2 * S) * nb : 0;  // S slices of at most TG / S + 2 tiles
    const size_t slots = (size_t)64 * NW * SW * nb;
    const size_t misc = (size_t)16 * NW * kMaxNb + 32 * kMaxNb + 8 * NW * cls_depth(c);  // + ring barriers
    const size_t ring = NW * cls_depth(c) * 2 * stage_su(fmt, c) * rec_bytes(fmt);
    return xs + gs + red + slots + misc + ring;
}

// Most tile units one warp's contiguous unit range touches, over the group
// sizes np in {np_a, np_b} and K-slice widths cs in {cs_a, cs_b}; upt times
// that is the warp's tile-slot count.  A range of len units of a cs-chunk pair
// sequence touches at most ceil(len / cs) + 1 pairs; this is the exact
// maximum for the warp split the kernel uses.
inline int slots_per_warp(int np_a, int np_b, int cs_a, int cs_b, int NW, int upt) {
    int best = 1;
    const int nps[2] = {np_a, np_b}, css[2] = {cs_a, cs_b};
    for (int i = 0; i < 2; ++i) {
        for (int j = 0; j < 2; ++j) {
            const long long np = nps[i], cs = css[j];
            if (np <= 0 || cs <= 0) continue;
            const long long U = np * cs;
            for (int w = 0; w < NW; ++w) {
                const long long ub = w * U / NW, ue = (w + 1) * U / NW;
                if (ue > ub) {
                    const int touched = (int)((ue - 1) / cs - ub / cs + 1);
                    if (touched > best) best = touched;
                }
            }
        }
    }
    return upt * best;
}

struct Plan {
    int TG, S, Cs, groups, ctas, SW, upt;
    size_t smem;
};

// Tiles per unit: pairs unless that leaves CTAs idle (gate/up jobs: always
// pairs, so a gate tile and its up tile share a CTA).
inline int units_of(int T, bool pairs, int ctas, int &upt) {
    upt = pairs || (T + 1) / 2 >= ctas ? 2 : 1;
    return (T + upt - 1) / upt;
}

// Launch plan for T tiles x C chunks.  One group of tile pairs per cluster of
// S CTAs (S splits K); at most one CTA per SM where the work allows, so that
// the next kernel in the stream can be resident beside it.  Chooses the
// split whose busiest SM streams the fewest records; ties go to the smaller
// split.  A plan whose shared memory exceeds kSmemMax is never chosen while
// another fits.
inline Plan make_plan(int fmt, int T, int C, int nb, bool pairs, int num_sms) {
    const int NW = cls_warps(cls_of(nb));
    Plan best{};
    long long best_cost = -1;
    bool best_fits = false;
    for (int S = 1; S <= kMaxCluster; S *= 2) {
        if (S > 1 && S > C) break;
        const int Cs = (C + S - 1) / S;
        if ((size_t)4 * cls_xrow(cls_of(nb)) * nb * Cs > kXsCap && S < kMaxCluster) continue;
        int G0 = num_sms / S;
        if (G0 < 1) G0 = 1;
        int upt = 2;
        const int P = units_of(T, pairs, G0, upt);
        // one wave of groups where the partial sums fit, else more groups
        // (fewer pairs each) until they do
        Plan pl;
        for (int mult = 1;; ++mult) {
            const int G = (int)((long long)G0 * mult < P ? (long long)G0 * mult : P);
            const int per = (P + G - 1) / G, per_lo = P / G;
            const int cs_last = C - ((C - 1) / Cs) * Cs;  // chunks of the last non-empty K-slice
            pl.S = S;
            pl.Cs = Cs;
            pl.groups = G;
            pl.ctas = G * S;
            pl.upt = upt;
            pl.TG = upt * per < T ? upt * per : T;
            pl.SW = slots_per_warp(per, per_lo, Cs, cs_last, NW, upt);
            pl.smem = engine_smem(fmt, nb, pl.TG, Cs, pl.SW, S);
            if (pl.smem <= kSmemMax || G == P) break;
        }
        const int per = (P + pl.groups - 1) / pl.groups;
        const bool fits = pl.smem <= kSmemMax;
        const int waves = (pl.ctas + num_sms - 1) / num_sms;
        // records on the busiest SM, plus about a microsecond of one SM's
        // share of HBM (~40 records) for each cluster-wide exchange and
        // about 1.5 us (~60 records) of staging and folding per extra wave
        const long long cost = (long long)per * upt * Cs * waves + (S > 1 ? 40 : 0) + 60 * (waves - 1);
        if (best_cost < 0 || (fits && !best_fits) || (fits == best_fits && cost < best_cost)) {
            best_cost = cost;
            best_fits = fits;
            best = pl;
        }
    }
    return best;
}

// Shared-memory scratch of the persistent step's attention job (step_attn.cuh,
// NW warps): the warps' output shares, maxima and sums, per-warp softmax
// slots, a flag.
inline size_t step_attn_scratch_bytes(int NW) {
    const size_t G = kStepAttnG, D = kStepAttnD;
    return ((size_t)NW * G * D + 2 * (size_t)NW * G + (size_t)NW * 32 + (size_t)NW * G) * 4 + 16;
}

// Dynamic shared memory of one decode-step CTA: the engine's regions plus a
// copy of every job's parameter block and the CTA's span of every job.
inline size_t step_smem_bytes(int fmt, int nb, int TGmax, int Kmax, int SWmax, int njobs) {
    const int Cs = (Kmax + kChunkK - 1) / kChunkK;
    return engine_smem(fmt, nb, TGmax, Cs, SWmax, 1) + (size_t)njobs * (sizeof(GemvParams) + sizeof(JobSpan));
}

// Launchers, one per kernel instantiation family (defined in the .cu files).
// Decode attention (attn_kernel.cu): one token against an f32 KV cache.
// CTA (s, hk) takes kv head hk and split s -- Lc positions -- of the attended
// positions [lo, total); with nsplit > 1 the last split of each kv head to
// finish folds the splits' shares (ws_count[hk] counts them, and is zero
// again when the call ends).
struct AttnParams {
    const float *q, *k_new, *v_new;   // [H][D], [Hkv][D], [Hkv][D]
    float *k_cache, *v_cache;         // [Hkv][max_seq][D]
    const float *rope_cos, *rope_sin; // [max_seq][D/2] or nullptr
    float *out;                       // [H][D]
    float *ws_o, *ws_m, *ws_l;        // split shares [nsplit][H][D], maxima and sums [nsplit][H]
    int *ws_count;                    // [Hkv] splits finished (zero between calls)
    int *err;                         // set nonzero if a copy wait gave up
    long long wait_cycles;            // bound of one copy wait (SM clock cycles)
    int extra_tx;                     // bytes the first K copy expects beyond its rows (0; testing only)
    int max_seq, position, H, Hkv, D, lo, total, Lc, nsplit;
    float scale;
};
size_t attn_smem_bytes(int D, int G);
int attn_sub_chunk(int D);         // positions per pipeline stage
int attn_ctas_per_sm(int D, int G);
int attn_max_splits(int D, int G);
int launch_attn(const AttnParams &p, void *stream);

// Prefill GEMM (gemm_kernel.cu): y[nb][n] (=, or +=) x[nb][K] W^T for any nb;
// x is first staged into `img` (B fragments, block factors and offsets per 64
// activation rows and 128-column chunk).
struct GemmParams {
    const uint8_t *w;   // packed weights
    const float *x;     // [nb][K]
    uint8_t *img;       // staged activations, gemm_image_bytes(nb, C)
    float *y;           // [nb][n]
    int n, T, C, K, nb, accumulate;
    int *err;           // set nonzero if a copy wait gave up
    long long wait_cycles;
    int extra_tx;       // bytes the first stage expects beyond its copies (testing only; 0)
};
size_t gemm_image_bytes(int nb, int C);
size_t gemm_smem_bytes(int fmt, int nb);
int launch_gemm(const GemmParams &p, int fmt, void *stream);
// The tensor-memory GEMM (Q4_0 and Q8_0, nb > 16): its activation image and
// row factors, and its two launches.
size_t gemm_tc_image_bytes(int nb, int C);
int launch_gemm_tc(const GemmParams &p, int fmt, void *stream);
constexpr int kGemmTcMinNb = 17;  // up to 16 rows the 16-row mma.sync tile is faster

int launch_gemv_q4_0(const GemvParams &p, const Plan &plan, void *stream);
int launch_gemv_affine(const GemvParams &p, const Plan &plan, void *stream);
int launch_gemv_q8_0(const GemvParams &p, const Plan &plan, void *stream);
int launch_gemv_q4_k(const GemvParams &p, const Plan &plan, void *stream);
int launch_gemv_q1(const GemvParams &p, const Plan &plan, void *stream);
// Cooperative launch of the decode-step kernel: one CTA per SM.
int launch_step_q4_0(const StepParams &p, int ctas, size_t smem, void *stream);
int launch_step_affine(const StepParams &p, int ctas, size_t smem, void *stream);
int launch_step_q8_0(const StepParams &p, int ctas, size_t smem, void *stream);
int launch_step_q4_k(const StepParams &p, int ctas, size_t smem, void *stream);
int launch_step_q1(const StepParams &p, int ctas, size_t smem, void *stream);
// Decode-step CTAs that can be resident on one SM (0 on error).
int step_occupancy_q4_0(int nb, size_t smem, bool attn);
int step_occupancy_affine(int nb, size_t smem, bool attn);
int step_occupancy_q8_0(int nb, size_t smem, bool attn);
int step_occupancy_q4_k(int nb, size_t smem, bool attn);
int step_occupancy_q1(int nb, size_t smem, bool attn);

}  // namespace q4
