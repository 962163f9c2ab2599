// q4_internal.h -- shared definitions of libq4gemv: the device weight layout,
// the kernel parameter block and the launch planner.
#pragma once
#include <stddef.h>
#include <stdint.h>

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

inline int rec_bytes(int fmt) { return fmt == 0 ? kRecQ4_0 : kRecAffine; }
inline int64_t tiles_of(int64_t n) { return (n + kTileRows - 1) / kTileRows; }
inline int64_t chunks_of(int64_t k) { return (k + kChunkK - 1) / kChunkK; }

// ---------------------------------------------------------------- kernel
enum Mode { MODE_SINGLE = 0, MODE_CONCAT = 1, MODE_PAIRS = 2 };
enum Epi { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SWIGLU = 2, EPI_ARGMAX = 3 };

constexpr int kThreads = 256;                 // per-call kernel: 8 warps per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kStepWarps = 16;               // persistent decode-step kernel: 16 warps per CTA
constexpr int kMaxNb = 16;
constexpr int kMaxCluster = 8;
constexpr size_t kXsCap = 64 * 1024;          // activation slice staged per CTA
constexpr int kRingDepth = 8;                 // weight records per warp in the cp.async ring

constexpr int kMaxMats = 3;                // matrices of one job (q, k, v share one input)

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
    int S;                       // K-split: CTAs per cluster
    int Cs;                      // chunks per K-slice
    int groups;                  // tile groups; group g holds tile units [g*P/groups, (g+1)*P/groups)
    const float *x;              // [nb][K]
    const float *gamma;          // [K] or nullptr (no RMSNorm)
    float eps;
    const float *gsum;           // affine: caller group sums [nb][K/32] or nullptr
    int epi;                     // Epi
    float *out[kMaxMats];        // y per matrix (swiglu: out[0] = h; argmax: logits or nullptr)
    const float *res;            // residual [nb][n0]
    float *am_val;               // argmax partials [nb][groups]
    int *am_idx;
};

// The persistent decode-step kernel runs these jobs in order, one CTA per SM.
constexpr int kMaxStepJobs = 4 * 32 + 1;      // four jobs per layer, up to 32 layers, + logits
constexpr int kStepRingDepth = 8;             // weight records per warp of the decode-step kernel
constexpr long long kBarrierSpins = 1ll << 22;  // polls before a grid barrier gives up

struct StepParams {
    int njobs;
    int nb;
    int Kmax;                    // largest K of the jobs (sizes the activation slice)
    int TGmax;                   // most tiles any group holds in any job
    unsigned *counter;           // grid-barrier arrivals (zeroed before each launch)
    unsigned *release;           // number of the last completed barrier (zeroed before each launch)
    int *err;                    // set to 1 if a barrier gave up
    int32_t *idx;                // [nb] argmax of the last job
    float *val;                  // [nb] or nullptr
    GemvParams jobs[kMaxStepJobs];
};

inline int ntiles_for(int nb) { return nb <= 8 ? 1 : 2; }

// Dynamic shared memory of one CTA of the engine: activation slice, group
// sums (affine), per-warp tile partials, reductions, the weight ring.
inline size_t engine_smem(int fmt, int TG, int Cs, int nb, int warps, int depth) {
    size_t xs = (size_t)4 * nb * Cs * kChunkK;
    size_t gs = fmt == 1 ? (size_t)4 * Cs * kBlocksPerChunk * 8 * ntiles_for(nb) : 0;
    size_t red = (size_t)4 * TG * kTileRows * nb;
    size_t slots = (size_t)4 * warps * TG * kTileRows * nb;
    size_t misc = (size_t)4 * 4 * warps * kMaxNb + 4 * 8 * kMaxNb;
    size_t ring = (size_t)warps * depth * rec_bytes(fmt);
    return xs + gs + red + slots + misc + ring;
}

inline size_t smem_bytes(int fmt, int TG, int Cs, int nb) {
    return engine_smem(fmt, TG, Cs, nb, kWarps, kRingDepth);
}

// Dynamic shared memory of one decode-step CTA.
inline size_t step_smem_bytes(int fmt, int TGmax, int Kmax, int nb) {
    const int Cs = (Kmax + kChunkK - 1) / kChunkK;
    return engine_smem(fmt, TGmax, Cs, nb, kStepWarps, kStepRingDepth);
}

struct Plan {
    int TG, S, Cs, groups, ctas;
    size_t smem;
};

// Launch plan for T tiles x C chunks.  One group of tiles per cluster of S
// CTAs (S splits K); at most one CTA per SM where the work allows, so that
// the next kernel in the stream can be resident beside it.  Chooses the
// split whose busiest CTA has the least work; ties go to the smaller split.
inline Plan make_plan(int fmt, int T, int C, int nb, bool pairs, int num_sms) {
    const int pw = pairs ? 2 : 1;
    const int P = T / pw;                       // allocation units (tiles or gate/up pairs)
    Plan best{};
    long long best_cost = -1;
    for (int S = 1; S <= kMaxCluster; S *= 2) {
        if (S > 1 && S > C) break;
        const int Cs = (C + S - 1) / S;
        if ((size_t)4 * nb * Cs * kChunkK > kXsCap && S < kMaxCluster) continue;
        int G = num_sms / S;
        if (G < 1) G = 1;
        if (G > P) G = P;
        int per = (P + G - 1) / G;                      // units of the busiest group
        const int cap = 128 / (nb * pw) > 0 ? 128 / (nb * pw) : 1;  // per-warp partials fit shared memory
        if (per > cap) {
            per = cap;
            G = (P + per - 1) / per;
        }
        const int ctas = G * S;
        const int waves = (ctas + num_sms - 1) / num_sms;
        // records on the busiest SM, plus about a microsecond of one SM's
        // share of HBM (~40 records) for each cluster-wide exchange
        const long long cost = (long long)per * pw * Cs * waves + (S > 1 ? 40 : 0);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best.TG = per * pw;
            best.S = S;
            best.Cs = Cs;
            best.groups = G;
            best.ctas = ctas;
        }
    }
    best.smem = smem_bytes(fmt, best.TG, best.Cs, nb);
    return best;
}

// Launchers, one per kernel instantiation family (defined in the .cu files).
int launch_gemv_q4_0(const GemvParams &p, const Plan &plan, void *stream);
int launch_gemv_affine(const GemvParams &p, const Plan &plan, void *stream);
// Cooperative launch of the decode-step kernel: one CTA per SM.
int launch_step_q4_0(const StepParams &p, int ctas, size_t smem, void *stream);
int launch_step_affine(const StepParams &p, int ctas, size_t smem, void *stream);
// Decode-step CTAs that can be resident on one SM (0 on error).
int step_occupancy_q4_0(int nb, size_t smem);
int step_occupancy_affine(int nb, size_t smem);

}  // namespace q4
