/*
 * q4_oracle.c -- plain, slow, obviously correct CPU oracle for the weight-only
 * dequant-in-GEMV family (Q4_0 blocks, affine-Q4 groups, Q8_0 blocks, Q4_K
 * superblocks and Q1 sign-bit superblocks) and its fused
 * neighbours (RMSNorm, SwiGLU, residual add, greedy argmax).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this code.  The CUDA library never
 * includes, links or calls it, and it shares no source with the CUDA path.
 *
 * Everything is computed in IEEE double precision, one output at a time:
 * dequantise a weight row to f64 from its stored bytes, then a sequential dot
 * product in ascending k.  No blocking, no reordering, no group-sum rewrite.
 * Build with -ffp-contract=off so that no multiply-add is fused on any host.
 *
 * Sources (the pages this code follows):
 *  - Q4_0 block (32 weights in 18 bytes: fp16 scale d, then 16 nibble bytes;
 *    weight = d * (q - 8)): crate inferencelayer, Functions, entries
 *    q4_0_to_q8_0n (the lossless upcast keeps d and maps q to nib - 8) and
 *    gemv_q1_k_lcpp_src (Q4_0's 18-byte 32-weight block).  Nibble order inside
 *    the 16 bytes is not stated on the pages; the reading taken is the GGUF
 *    order the pages read as-is (gemv_q8_0n_k_lcpp_src): byte i holds element i
 *    in its low nibble and element i+16 in its high nibble.
 *  - Q8_0 block (32 weights in 34 bytes: fp16 scale d, then 32 signed bytes;
 *    weight = d * q): crate inferencelayer, Functions, entries q4_0_to_q8_0n
 *    (the lossless upcast of a Q4_0 block keeps d and maps q to nib - 8) and
 *    gemv_q8_0n_k_lcpp_src (Q8_0 blocks read as-is).
 *  - Q4_K superblock (256 weights in 144 bytes: fp16 d, fp16 dmin, 12 bytes
 *    of 6-bit sub-scales sc and sub-mins mn for eight 32-weight sub-blocks,
 *    128 nibble bytes; weight = d * sc * q - dmin * mn): crate inferencelayer,
 *    Functions, entries gemv_q5k_k_lcpp_src (the superblock's fields in this
 *    order, "the SAME 6-bit pack as Q4_K", and w = d*sc*nib - dmin*mn with the
 *    fifth bit plane, which Q4_K does not have) and honeycrisp/mod.rs
 *    (quant_matmul's Q4_K branch: k a multiple of 256).  The pages do not
 *    print the 6-bit pack or the nibble order; the reading taken is the GGUF
 *    one the pages load as-is.  Sub-blocks 0-3 keep sc and mn in the low six
 *    bits of scale bytes 0-3 and 4-7; sub-blocks 4-7 keep their low four bits
 *    in the two nibbles of bytes 8-11 (sc low, mn high) and their top two bits
 *    in the top two bits of bytes 0-3 (sc) and 4-7 (mn).  The 128 nibble bytes
 *    are four runs of 32: run r holds sub-block 2r in its low nibbles and
 *    sub-block 2r+1 in its high nibbles, in element order.
 *  - Q1 superblock (128 binary weights in 18 bytes: fp16 scale d, then 16
 *    bytes of sign bits; weight = +d for a set bit, -d for a clear one):
 *    crate inferencelayer, Functions, entries gemv_q1_k_lcpp_src (bit i of a
 *    weight word is element i's sign, 1 -> +1 and 0 -> -1; one f16 scale per
 *    128 weights; 4.5 bytes per 32 weights) and gemm_q1_src (the sign bits
 *    and one f16 scale per 128-weight superblock).  Reading: the scale comes
 *    first, as in Q4_0's block, and the bits follow as little-endian words,
 *    so byte i holds elements 8i..8i+7 from its lowest bit up.
 *  - Affine-Q4 group (32 weights, bf16 scale s and bf16 min m, weight =
 *    s*q + m): Module gpu (qwen4_exp), Structs Q (affine-Q4 projection with
 *    byte offsets into a bf16 weight buffer) and HalfSet (even/odd streams plus
 *    per-32 group sums).  Reading: nibbles are planar [n][k/2] with byte i of a
 *    row holding element 2i (low nibble) and 2i+1 (high nibble); s and m are
 *    planar [n][k/32].
 *  - RMSNorm with eps and width d = len(gamma): honeycrisp/mod.rs, Op::RmsNorm
 *    and forward_decode_fused_layers step "1+2 Q matmul with inline
 *    input_norm".  Reading: xhat = x / sqrt(mean(x^2) + eps) * gamma.
 *  - SwiGLU mid = silu(gate) * up: honeycrisp/mod.rs, fused_ffn_residual step 4.
 *  - Residual y = matmul(x, w) + residual: honeycrisp/mod.rs, fused
 *    matmul + residual dispatch in forward_decode_fused_layers.
 *  - Greedy argmax over logits: Module gpu, module sampling.  Reading: ties go
 *    to the lowest index.
 *  - Decode attention with KV append, GQA, sliding window and RoPE tables:
 *    honeycrisp/mod.rs, attn_state (f32 caches of kv_heads x max_seq x
 *    head_dim per layer; RoPE tables theta = pos / rope_theta^(2j/head_dim)),
 *    gpu_attention (append k and v at position, then scores = q K^T, softmax,
 *    times V over total_seq = position + 1 with a window and a scale) and the
 *    fused RoPE + KV-append + SDPA dispatch of forward_decode_fused_layers.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/* IEEE 754 binary16 -> double, from the bit fields. */
double q4o_half(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25);    /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 (the upper half of an IEEE binary32) -> double, from the bit fields. */
double q4o_bf16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* subnormal: f * 2^-133 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x80), e - 134);    /* 1.f * 2^(e-127) */
    return sign ? -v : v;
}

/* One row of Q4_0 weights, dequantised to f64.
 * blocks: [n][k/32][18] bytes; w: [k]. */
void q4o_q4_0_row(const uint8_t *blocks, int64_t k, int64_t row, double *w)
{
    int64_t nblk = k / 32;
    const uint8_t *r = blocks + row * nblk * 18;
    for (int64_t b = 0; b < nblk; ++b) {
        const uint8_t *blk = r + b * 18;
        double d = q4o_half((uint16_t)(blk[0] | (blk[1] << 8)));
        const uint8_t *qs = blk + 2;
        for (int j = 0; j < 32; ++j) {
            int q = (j < 16) ? (qs[j] & 0x0f) : (qs[j - 16] >> 4);
            w[b * 32 + j] = d * (double)(q - 8);
        }
    }
}

/* One row of Q8_0 weights, dequantised to f64: blocks of 34 bytes, the fp16
 * scale d (little endian) then 32 signed bytes q; weight = d * q.
 * blocks: [n][k/32][34] bytes; w: [k]. */
void q4o_q8_0_row(const uint8_t *blocks, int64_t k, int64_t row, double *w)
{
    int64_t nblk = k / 32;
    const uint8_t *r = blocks + row * nblk * 34;
    for (int64_t b = 0; b < nblk; ++b) {
        const uint8_t *blk = r + b * 34;
        double d = q4o_half((uint16_t)(blk[0] | (blk[1] << 8)));
        for (int j = 0; j < 32; ++j) {
            int q = blk[2 + j] < 128 ? blk[2 + j] : blk[2 + j] - 256;   /* two's complement byte */
            w[b * 32 + j] = d * (double)q;
        }
    }
}

/* Sub-block j's 6-bit scale and min of a Q4_K superblock's 12 scale bytes. */
void q4o_q4_k_scale_min(const uint8_t *sb, int j, int *sc, int *mn)
{
    if (j < 4) {
        *sc = sb[j] & 63;
        *mn = sb[j + 4] & 63;
    } else {
        *sc = (sb[j + 4] & 0x0f) | ((sb[j - 4] >> 6) << 4);
        *mn = (sb[j + 4] >> 4) | ((sb[j] >> 6) << 4);
    }
}

/* One row of Q4_K weights, dequantised to f64: superblocks of 144 bytes,
 * fp16 d and dmin (little endian), 12 scale bytes, 128 nibble bytes;
 * weight = d * sc * q - dmin * mn.  blocks: [n][k/256][144] bytes; w: [k]. */
void q4o_q4_k_row(const uint8_t *blocks, int64_t k, int64_t row, double *w)
{
    int64_t nsb = k / 256;
    const uint8_t *r = blocks + row * nsb * 144;
    for (int64_t b = 0; b < nsb; ++b) {
        const uint8_t *blk = r + b * 144;
        double d = q4o_half((uint16_t)(blk[0] | (blk[1] << 8)));
        double dmin = q4o_half((uint16_t)(blk[2] | (blk[3] << 8)));
        const uint8_t *sb = blk + 4, *qs = blk + 16;
        for (int e = 0; e < 256; ++e) {
            int j = e / 32;                       /* sub-block */
            int l = e % 32;                       /* element within it */
            int byte = qs[32 * (j / 2) + l];
            int q = (j & 1) ? (byte >> 4) : (byte & 0x0f);
            int sc, mn;
            q4o_q4_k_scale_min(sb, j, &sc, &mn);
            w[b * 256 + e] = d * (double)sc * (double)q - dmin * (double)mn;
        }
    }
}

/* One row of Q1 weights, dequantised to f64: superblocks of 18 bytes, the
 * fp16 scale d (little endian) then 16 bytes of sign bits; weight = d for a
 * set bit, -d for a clear one.  blocks: [n][k/128][18] bytes; w: [k]. */
void q4o_q1_row(const uint8_t *blocks, int64_t k, int64_t row, double *w)
{
    int64_t nsb = k / 128;
    const uint8_t *r = blocks + row * nsb * 18;
    for (int64_t b = 0; b < nsb; ++b) {
        const uint8_t *blk = r + b * 18;
        double d = q4o_half((uint16_t)(blk[0] | (blk[1] << 8)));
        for (int e = 0; e < 128; ++e) {
            int bit = (blk[2 + e / 8] >> (e % 8)) & 1;
            w[b * 128 + e] = bit ? d : -d;
        }
    }
}

/* One row of affine-Q4 weights, dequantised to f64.
 * nib: [n][k/2] bytes; s, m: [n][k/32] bf16 bits; w: [k]. */
void q4o_affine_row(const uint8_t *nib, const uint16_t *s, const uint16_t *m,
                    int64_t k, int64_t row, double *w)
{
    const uint8_t *r = nib + row * (k / 2);
    const uint16_t *sr = s + row * (k / 32);
    const uint16_t *mr = m + row * (k / 32);
    for (int64_t e = 0; e < k; ++e) {
        int byte = r[e / 2];
        int q = (e & 1) ? (byte >> 4) : (byte & 0x0f);
        double sg = q4o_bf16(sr[e / 32]);
        double mg = q4o_bf16(mr[e / 32]);
        w[e] = sg * (double)q + mg;
    }
}

/* y[r][i] = sum_k w[i][k] * x[r][k], summed sequentially in ascending k, and
 * bound[r][i] = sum_k |w[i][k]| * |x[r][k]| (the scale of the parity tolerance),
 * for the output rows i in [row0, row1) (rows are independent; callers may
 * run disjoint ranges at the same time, each with its own scratch).
 * fmt 0: a = Q4_0 blocks.  fmt 1: a = nibbles, b = s, c = m.  fmt 2: a = Q8_0 blocks.
 * fmt 3: a = Q4_K superblocks.  fmt 4: a = Q1 superblocks.
 * x: [nb][k] f64; y, bound: [nb][n]; wrow: scratch of k doubles. */
void q4o_gemv_rows(int fmt, const void *a, const void *b, const void *c,
                   int64_t n, int64_t k, const double *x, int64_t nb,
                   double *y, double *bound, double *wrow, int64_t row0, int64_t row1)
{
    for (int64_t i = row0; i < row1; ++i) {
        if (fmt == 0)
            q4o_q4_0_row((const uint8_t *)a, k, i, wrow);
        else if (fmt == 2)
            q4o_q8_0_row((const uint8_t *)a, k, i, wrow);
        else if (fmt == 3)
            q4o_q4_k_row((const uint8_t *)a, k, i, wrow);
        else if (fmt == 4)
            q4o_q1_row((const uint8_t *)a, k, i, wrow);
        else
            q4o_affine_row((const uint8_t *)a, (const uint16_t *)b,
                           (const uint16_t *)c, k, i, wrow);
        for (int64_t r = 0; r < nb; ++r) {
            const double *xr = x + r * k;
            double acc = 0.0, mag = 0.0;
            for (int64_t e = 0; e < k; ++e) {
                acc += wrow[e] * xr[e];
                mag += fabs(wrow[e]) * fabs(xr[e]);
            }
            y[r * n + i] = acc;
            if (bound)
                bound[r * n + i] = mag;
        }
    }
}

/* All n output rows of the GEMV above. */
void q4o_gemv(int fmt, const void *a, const void *b, const void *c,
              int64_t n, int64_t k, const double *x, int64_t nb,
              double *y, double *bound, double *wrow)
{
    q4o_gemv_rows(fmt, a, b, c, n, k, x, nb, y, bound, wrow, 0, n);
}

/* HalfSet activations (Module gpu, Struct HalfSet: half even/odd streams)
 * as f64 rows: x[r][2i] = half(xe[r][i]), x[r][2i+1] = half(xo[r][i]).
 * xe, xo: [nb][k/2] f16 bits; x: [nb][k]. */
void q4o_halfset_rows(const uint16_t *xe, const uint16_t *xo, int64_t nb, int64_t k, double *x)
{
    for (int64_t r = 0; r < nb; ++r)
        for (int64_t i = 0; i < k / 2; ++i) {
            x[r * k + 2 * i] = q4o_half(xe[r * (k / 2) + i]);
            x[r * k + 2 * i + 1] = q4o_half(xo[r * (k / 2) + i]);
        }
}

/* xhat[r][e] = x[r][e] / sqrt(mean_e' x[r][e']^2 + eps) * gamma[e]. */
void q4o_rmsnorm(const double *x, const double *gamma, int64_t nb, int64_t k,
                 double eps, double *xhat)
{
    for (int64_t r = 0; r < nb; ++r) {
        const double *xr = x + r * k;
        double ss = 0.0;
        for (int64_t e = 0; e < k; ++e)
            ss += xr[e] * xr[e];
        double rms = sqrt(ss / (double)k + eps);
        for (int64_t e = 0; e < k; ++e)
            xhat[r * k + e] = xr[e] / rms * gamma[e];
    }
}

/* silu(t) = t / (1 + exp(-t)) */
double q4o_silu(double t)
{
    return t / (1.0 + exp(-t));
}

/* h = silu(g) * u, elementwise. */
void q4o_swiglu(const double *g, const double *u, int64_t count, double *h)
{
    for (int64_t i = 0; i < count; ++i)
        h[i] = q4o_silu(g[i]) * u[i];
}

/* out = a + b, elementwise. */
void q4o_add(const double *a, const double *b, int64_t count, double *out)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = a[i] + b[i];
}

/* Index of the largest value; the lowest index wins a tie. */
int64_t q4o_argmax(const double *v, int64_t n)
{
    int64_t best = 0;
    for (int64_t i = 1; i < n; ++i)
        if (v[i] > v[best])
            best = i;
    return best;
}

/* RoPE tables (honeycrisp/mod.rs, attn_state: theta = pos / rope_theta^(2j /
 * head_dim) for j < rope_dim / 2, tables of cos and sin per position):
 * cosv[p][j], sinv[p][j] for p < max_seq, j < d / 2 (rope_dim = d). */
void q4o_rope_table(int64_t max_seq, int64_t d, double rope_theta, double *cosv, double *sinv)
{
    for (int64_t p = 0; p < max_seq; ++p)
        for (int64_t j = 0; j < d / 2; ++j) {
            double th = (double)p / pow(rope_theta, 2.0 * (double)j / (double)d);
            cosv[p * (d / 2) + j] = cos(th);
            sinv[p * (d / 2) + j] = sin(th);
        }
}

/* Rotate one head vector x[d] in place by the table row (c, s) of its
 * position.  Reading (the pages do not print the pairing): element j pairs
 * with element j + d/2 (the rotate-half form of the transformers models the
 * pages mirror): (a, b) -> (a c - b s, b c + a s). */
void q4o_rope_apply(double *x, int64_t d, const double *c, const double *s)
{
    for (int64_t j = 0; j < d / 2; ++j) {
        double a = x[j], b = x[j + d / 2];
        x[j] = a * c[j] - b * s[j];
        x[j + d / 2] = b * c[j] + a * s[j];
    }
}

/* Decode attention of the token at `position` (honeycrisp/mod.rs,
 * gpu_attention and the fused RoPE + KV-append + SDPA dispatch of
 * forward_decode_fused_layers):
 *  1. with tables, q (every head) and k_new (every kv head) are rotated by
 *     the table rows of `position`;
 *  2. k_new and v_new are appended: cache[hk][position] = k, v;
 *  3. total = position + 1; the attended positions are [lo, total) with
 *     lo = max(0, total - window) for window > 0, else 0;
 *  4. query head h reads kv head h / (H / Hkv) (consecutive heads share one);
 *     its scores are scale * q_h . k_t, softmax over the attended positions
 *     (shifted by their maximum), and out_h = sum_t p_t v_t.
 * q: [H][d]; k_new, v_new: [Hkv][d]; k_cache, v_cache: [Hkv][max_seq][d]
 * (updated); cosv, sinv: [max_seq][d/2] or NULL (no rotation);
 * out, bound: [H][d] (bound = sum_t p_t |v_t|, the tolerance scale);
 * scratch: max_seq + 2 d doubles. */
void q4o_attn_decode(const double *q, const double *k_new, const double *v_new,
                     double *k_cache, double *v_cache, int64_t max_seq, int64_t position,
                     int64_t H, int64_t Hkv, int64_t d, int64_t window, double scale,
                     const double *cosv, const double *sinv, double *out, double *bound,
                     double *scratch)
{
    double *p = scratch, *qh = scratch + max_seq, *kh = qh + d;
    int64_t G = H / Hkv;
    for (int64_t hk = 0; hk < Hkv; ++hk) {
        for (int64_t e = 0; e < d; ++e)
            kh[e] = k_new[hk * d + e];
        if (cosv)
            q4o_rope_apply(kh, d, cosv + position * (d / 2), sinv + position * (d / 2));
        for (int64_t e = 0; e < d; ++e) {
            k_cache[(hk * max_seq + position) * d + e] = kh[e];
            v_cache[(hk * max_seq + position) * d + e] = v_new[hk * d + e];
        }
    }
    int64_t total = position + 1;
    int64_t lo = (window > 0 && total > window) ? total - window : 0;
    for (int64_t h = 0; h < H; ++h) {
        int64_t hk = h / G;
        for (int64_t e = 0; e < d; ++e)
            qh[e] = q[h * d + e];
        if (cosv)
            q4o_rope_apply(qh, d, cosv + position * (d / 2), sinv + position * (d / 2));
        double mx = -INFINITY;
        for (int64_t t = lo; t < total; ++t) {
            double s = 0.0;
            for (int64_t e = 0; e < d; ++e)
                s += qh[e] * k_cache[(hk * max_seq + t) * d + e];
            p[t] = scale * s;
            if (p[t] > mx)
                mx = p[t];
        }
        double z = 0.0;
        for (int64_t t = lo; t < total; ++t) {
            p[t] = exp(p[t] - mx);
            z += p[t];
        }
        for (int64_t e = 0; e < d; ++e) {
            double acc = 0.0, mag = 0.0;
            for (int64_t t = lo; t < total; ++t) {
                double v = v_cache[(hk * max_seq + t) * d + e];
                acc += p[t] / z * v;
                mag += p[t] / z * fabs(v);
            }
            out[h * d + e] = acc;
            bound[h * d + e] = mag;
        }
    }
}
