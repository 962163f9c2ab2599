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

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxNb = 16;
constexpr int kMaxCluster = 8;

struct GemvParams {
    const uint8_t *w[2];   // packed weights of (up to) two matrices
    int n[2];              // output rows of each matrix
    int tiles[2];          // 16-row tiles of each matrix
    int mode;              // Mode
    int T;                 // tiles of the launch (sum, or 2x for pairs)
    int K;                 // input length
    int C;                 // 128-column chunks per row
    int nb;                // activation rows
    int TG;                // tiles per group (one group = one cluster)
    int S;                 // K-split: CTAs per cluster
    int Cs;                // chunks per K-slice
    const float *x;        // [nb][K]
    const float *gamma;    // [K] or nullptr (no RMSNorm)
    float eps;
    const float *gsum;     // affine: caller group sums [nb][K/32] or nullptr
    int epi;               // Epi
    float *out[2];         // y per matrix (swiglu: out[0] = h; argmax: logits or nullptr)
    const float *res;      // residual [nb][n0]
    float *am_val;         // argmax partials [nb][groups]
    int *am_idx;
    int groups;
};

// Dynamic shared memory of one CTA.
inline size_t smem_bytes(int fmt, int TG, int Cs, int nb) {
    size_t xs = (size_t)4 * nb * Cs * kChunkK;                     // hi/lo f16 activations
    size_t gs = fmt == 1 ? (size_t)4 * nb * Cs * kBlocksPerChunk : 0;  // affine group sums
    size_t slots = (size_t)4 * kWarps * TG * kTileRows * nb;       // per-warp partials
    size_t red = (size_t)4 * TG * kTileRows * nb;                  // CTA partials
    size_t misc = (size_t)4 * 4 * kWarps * kMaxNb + 4 * 8 * kMaxNb;  // reductions
    return xs + gs + slots + red + misc;
}

struct Plan {
    int TG, S, Cs, groups, ctas;
    size_t smem;
};

// Tiles per group and K-split for a launch of T tiles x C chunks.
inline Plan make_plan(int fmt, int T, int C, int nb, bool pairs, int num_sms) {
    Plan p{};
    const size_t xs_cap = 64 * 1024;
    int S = 1;
    // the activation slice must fit in shared memory
    while (S < kMaxCluster && (size_t)4 * nb * ((C + S - 1) / S) * kChunkK > xs_cap) S *= 2;
    // split K further when there are too few tiles to cover every SM
    while (S < kMaxCluster && (int64_t)T * S < num_sms && (C + 2 * S - 1) / (2 * S) >= 2) S *= 2;
    if (S > C) S = 1 << (31 - __builtin_clz((unsigned)C));   // at least one chunk per slice
    int Cs = (C + S - 1) / S;
    const int target = 2 * num_sms;        // two 256-thread CTAs per SM
    int TG = (int)(((int64_t)T * S + target - 1) / target);
    if (TG < 1) TG = 1;
    int tg_cap = 64 / nb;
    if (tg_cap < 1) tg_cap = 1;
    if (TG > tg_cap) TG = tg_cap;
    if (pairs) {
        if (TG < 2) TG = 2;
        TG += TG & 1;
    }
    p.TG = TG;
    p.S = S;
    p.Cs = Cs;
    p.groups = (T + TG - 1) / TG;
    p.ctas = p.groups * S;
    p.smem = smem_bytes(fmt, TG, Cs, nb);
    return p;
}

// Launchers, one per kernel instantiation family (defined in the .cu files).
int launch_gemv_q4_0(const GemvParams &p, const Plan &plan, void *stream);
int launch_gemv_affine(const GemvParams &p, const Plan &plan, void *stream);

}  // namespace q4
