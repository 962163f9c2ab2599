// repack.cpp -- host-side lossless re-layout of Q4_0 / affine-Q4 / Q8_0 / Q4_K / Q1 weights into
// the coalesced device layout described in q4_internal.h, and its inverse.
//
// The pages re-lay block formats once at load time so that the GEMV reads
// aligned vectors (honeycrisp/mod.rs: transpose_q8_blocks; crate
// inferencelayer: q1_rp4_repack_src, the ROWPACK4 layout).  Here each 16-row x
// 128-column tile chunk becomes one contiguous record whose 16-byte lanes are
// exactly the tensor-core operand fragments of the kernel's warps.
#include <math.h>
#include <string.h>

#include "../../include/q4gemv.h"
#include "q4_internal.h"

namespace {

inline uint32_t load_u32(const uint8_t *p) {
    uint32_t v;
    memcpy(&v, p, 4);
    return v;
}
inline void store_u32(uint8_t *p, uint32_t v) { memcpy(p, &v, 4); }

bool shape_ok(int32_t n, int32_t k) {
    return n >= 1 && k >= 32 && k % 32 == 0 && k <= 65536 && n <= (1 << 24);
}

// Byte offset in a Q8_0 record of element e (0..31) of block j (0..3) of row
// rr (0..15): the lane-position t and byte i with q8_elem(t, i) == e.
inline int q8_off(int rr, int j, int e) {
    const int h = rr >> 3, g = rr & 7;
    const int t = (e & 7) >> 1, i = 2 * (e >> 3) + (e & 1);  // inverse of q8_elem
    return h * 1024 + (j >> 1) * 512 + (4 * g + t) * 16 + (j & 1) * 8 + i;
}

// Nibble q of element e (0..31) of block `blk` of a Q4_0 row (GGUF order).
inline int q4_0_nib(const uint8_t *blk, int e) {
    const uint8_t *qs = blk + 2;
    return e < 16 ? (qs[e] & 15) : (qs[e - 16] >> 4);
}

// Nibble of element e of an affine row (even element in the low nibble).
inline int affine_nib(const uint8_t *row, int64_t e) {
    int b = row[e >> 1];
    return (e & 1) ? (b >> 4) : (b & 15);
}

// Q4_K superblock (144 bytes: fp16 d, fp16 dmin, 12 scale bytes, 128
// nibble bytes).  Sub-block j's 6-bit scale and min: for j < 4 the low six
// bits of bytes j and j + 4; for j >= 4 the low and high nibbles of byte
// j + 4, topped by the upper two bits of bytes j - 4 and j.
inline void q4k_get(const uint8_t *sb, int j, int &sc, int &mn) {
    const uint8_t *s = sb + 4;
    if (j < 4) {
        sc = s[j] & 0x3F;
        mn = s[j + 4] & 0x3F;
    } else {
        sc = (s[j + 4] & 0x0F) | ((s[j - 4] & 0xC0) >> 2);
        mn = (s[j + 4] >> 4) | ((s[j] & 0xC0) >> 2);
    }
}
inline void q4k_put(uint8_t *sb, int j, int sc, int mn) {
    uint8_t *s = sb + 4;
    if (j < 4) {
        s[j] = (uint8_t)((s[j] & 0xC0) | sc);
        s[j + 4] = (uint8_t)((s[j + 4] & 0xC0) | mn);
    } else {
        s[j + 4] = (uint8_t)((sc & 0x0F) | ((mn & 0x0F) << 4));
        s[j - 4] = (uint8_t)((s[j - 4] & 0x3F) | ((sc >> 4) << 6));
        s[j] = (uint8_t)((s[j] & 0x3F) | ((mn >> 4) << 6));
    }
}
// Nibble of element e (0..31) of sub-block j: runs of 32 bytes, sub-block 2r
// in the low nibbles of run r and 2r + 1 in the high ones.
inline int q4k_nib(const uint8_t *sb, int j, int e) {
    const int b = sb[16 + 32 * (j >> 1) + e];
    return (j & 1) ? (b >> 4) : (b & 15);
}

}  // namespace

inline bool fmt_ok(int32_t fmt) {
    return fmt == Q4_FMT_Q4_0 || fmt == Q4_FMT_AFFINE || fmt == Q4_FMT_Q8_0 || fmt == Q4_FMT_Q4_K || fmt == Q4_FMT_Q1;
}
// Q4_K rows are whole 256-column superblocks, Q1 rows whole 128-column ones.
inline bool fmt_shape_ok(int32_t fmt, int32_t n, int32_t k) {
    return fmt_ok(fmt) && shape_ok(n, k) && (fmt != Q4_FMT_Q4_K || k % 256 == 0) && (fmt != Q4_FMT_Q1 || k % 128 == 0);
}

extern "C" size_t q4_packed_bytes(int32_t fmt, int32_t n, int32_t k) {
    if (!fmt_shape_ok(fmt, n, k)) return 0;
    return (size_t)q4::tiles_of(n) * (size_t)q4::chunks_of(k) * (size_t)q4::rec_bytes(fmt);
}

extern "C" size_t q4_weight_bytes(int32_t fmt, int32_t n, int32_t k) {
    if (!fmt_shape_ok(fmt, n, k)) return 0;
    if (fmt == Q4_FMT_Q4_K) return (size_t)n * (size_t)(k / 256) * 144u;
    if (fmt == Q4_FMT_Q1) return (size_t)n * (size_t)(k / 128) * 18u;
    return (size_t)n * (size_t)(k / 32) * (fmt == Q4_FMT_Q4_0 ? 18u : fmt == Q4_FMT_AFFINE ? 20u : 34u);
}

// Generic packer: `get_q(row, blk, e)` gives the nibble of element e of a
// block, `get_s` / `get_m` the 16-bit scale / min of a block.
template <class GetQ, class GetS, class GetM>
static void pack(int fmt, int32_t n, int32_t k, uint8_t *out, GetQ get_q, GetS get_s, GetM get_m) {
    const int64_t T = q4::tiles_of(n), C = q4::chunks_of(k), B = k / 32;
    const int rec = q4::rec_bytes(fmt);
    const uint32_t pad_word = fmt == Q4_FMT_Q4_0 ? 0x88888888u : 0u;  // zero weights
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < C; ++c) {
            uint8_t *r = out + (t * C + c) * rec;
            for (int h = 0; h < 2; ++h)
                for (int g = 0; g < 8; ++g)
                    for (int tp = 0; tp < 4; ++tp)
                        for (int j = 0; j < 4; ++j) {
                            int64_t row = t * 16 + h * 8 + g, blk = c * 4 + j;
                            uint32_t word = pad_word;
                            if (row < n && blk < B) {
                                word = 0;
                                for (int i = 0; i < 8; ++i)
                                    word |= (uint32_t)get_q(row, blk, q4::nib_elem(tp, i)) << (4 * i);
                            }
                            store_u32(r + h * 512 + (4 * g + tp) * 16 + j * 4, word);
                        }
            for (int g = 0; g < 8; ++g)
                for (int j = 0; j < 4; ++j) {
                    int64_t blk = c * 4 + j, r0 = t * 16 + g, r1 = r0 + 8;
                    uint32_t s0 = (r0 < n && blk < B) ? get_s(r0, blk) : 0;
                    uint32_t s1 = (r1 < n && blk < B) ? get_s(r1, blk) : 0;
                    store_u32(r + 1024 + g * 16 + j * 4, s0 | (s1 << 16));
                    if (fmt == Q4_FMT_AFFINE) {
                        uint32_t m0 = (r0 < n && blk < B) ? get_m(r0, blk) : 0;
                        uint32_t m1 = (r1 < n && blk < B) ? get_m(r1, blk) : 0;
                        store_u32(r + 1152 + g * 16 + j * 4, m0 | (m1 << 16));
                    }
                }
        }
    }
}

extern "C" q4_status q4_repack_q4_0(const void *host_blocks, int32_t n, int32_t k, void *host_out,
                                    size_t out_bytes) {
    if (!host_blocks || !host_out) return Q4_ERR_NULL;
    if (!shape_ok(n, k)) return Q4_ERR_SHAPE;
    if (out_bytes < q4_packed_bytes(Q4_FMT_Q4_0, n, k)) return Q4_ERR_SHAPE;
    const uint8_t *src = (const uint8_t *)host_blocks;
    const int64_t B = k / 32;
    auto blk_ptr = [&](int64_t row, int64_t blk) { return src + (row * B + blk) * 18; };
    pack(Q4_FMT_Q4_0, n, k, (uint8_t *)host_out,
         [&](int64_t row, int64_t blk, int e) { return q4_0_nib(blk_ptr(row, blk), e); },
         [&](int64_t row, int64_t blk) {
             const uint8_t *b = blk_ptr(row, blk);
             return (uint32_t)b[0] | ((uint32_t)b[1] << 8);
         },
         [&](int64_t, int64_t) { return 0u; });
    return Q4_OK;
}

extern "C" q4_status q4_repack_affine(const uint8_t *nib, const uint16_t *s, const uint16_t *m,
                                      int32_t n, int32_t k, void *host_out, size_t out_bytes) {
    if (!nib || !s || !m || !host_out) return Q4_ERR_NULL;
    if (!shape_ok(n, k)) return Q4_ERR_SHAPE;
    if (out_bytes < q4_packed_bytes(Q4_FMT_AFFINE, n, k)) return Q4_ERR_SHAPE;
    const int64_t B = k / 32;
    pack(Q4_FMT_AFFINE, n, k, (uint8_t *)host_out,
         [&](int64_t row, int64_t blk, int e) { return affine_nib(nib + row * (k / 2), blk * 32 + e); },
         [&](int64_t row, int64_t blk) { return (uint32_t)s[row * B + blk]; },
         [&](int64_t row, int64_t blk) { return (uint32_t)m[row * B + blk]; });
    return Q4_OK;
}

extern "C" q4_status q4_repack_q4_k(const void *host_blocks, int32_t n, int32_t k, void *host_out,
                                    size_t out_bytes) {
    if (!host_blocks || !host_out) return Q4_ERR_NULL;
    if (!fmt_shape_ok(Q4_FMT_Q4_K, n, k)) return Q4_ERR_SHAPE;
    if (out_bytes < q4_packed_bytes(Q4_FMT_Q4_K, n, k)) return Q4_ERR_SHAPE;
    const uint8_t *src = (const uint8_t *)host_blocks;
    uint8_t *out = (uint8_t *)host_out;
    const int64_t NS = k / 256;
    auto sb_ptr = [&](int64_t row, int64_t blk) { return src + (row * NS + blk / 8) * 144; };
    // nibble words, and the 6-bit scale and min of each block as the two
    // bytes of its 16-bit "scale" (padding: all zero, d = 0)
    pack(Q4_FMT_Q4_K, n, k, out,
         [&](int64_t row, int64_t blk, int e) { return q4k_nib(sb_ptr(row, blk), (int)(blk % 8), e); },
         [&](int64_t row, int64_t blk) {
             int sc, mn;
             q4k_get(sb_ptr(row, blk), (int)(blk % 8), sc, mn);
             return (uint32_t)sc | ((uint32_t)mn << 8);
         },
         [&](int64_t, int64_t) { return 0u; });
    const int64_t T = q4::tiles_of(n), C = q4::chunks_of(k);
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            uint8_t *r = out + (t * C + c) * q4::kRecQ4_K;
            for (int g = 0; g < 8; ++g) {
                uint32_t dw = 0, mw = 0;
                for (int h = 0; h < 2; ++h) {
                    const int64_t row = t * 16 + h * 8 + g;
                    if (row >= n) continue;
                    const uint8_t *sb = src + (row * NS + c / 2) * 144;
                    dw |= ((uint32_t)sb[0] | ((uint32_t)sb[1] << 8)) << (16 * h);
                    mw |= ((uint32_t)sb[2] | ((uint32_t)sb[3] << 8)) << (16 * h);
                }
                store_u32(r + 1152 + g * 4, dw);
                store_u32(r + 1184 + g * 4, mw);
            }
        }
    return Q4_OK;
}

// Q1 superblock (18 bytes: fp16 d, 16 bytes of sign bits, byte i holding
// elements 8i..8i+7 from its lowest bit; 1 is +d).  The device record keeps
// each bit inverted, so that a set bit is the f16 sign of -1.
inline int q1_bit(const uint8_t *sb, int e) { return (sb[2 + (e >> 3)] >> (e & 7)) & 1; }

extern "C" q4_status q4_repack_q1(const void *host_blocks, int32_t n, int32_t k, void *host_out, size_t out_bytes) {
    if (!host_blocks || !host_out) return Q4_ERR_NULL;
    if (!fmt_shape_ok(Q4_FMT_Q1, n, k)) return Q4_ERR_SHAPE;
    if (out_bytes < q4_packed_bytes(Q4_FMT_Q1, n, k)) return Q4_ERR_SHAPE;
    const uint8_t *src = (const uint8_t *)host_blocks;
    uint8_t *out = (uint8_t *)host_out;
    const int64_t T = q4::tiles_of(n), C = k / 128;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            uint8_t *r = out + (t * C + c) * q4::kRecQ1;
            for (int g = 0; g < 8; ++g) {
                uint32_t dw = 0;
                for (int h = 0; h < 2; ++h) {
                    const int64_t row = t * 16 + h * 8 + g;
                    const uint8_t *sb = row < n ? src + (row * C + c) * 18 : nullptr;
                    for (int tp = 0; tp < 4; ++tp) {
                        uint32_t word = 0;  // padding rows: d = 0, any bits
                        if (sb)
                            for (int rho = 0; rho < 16; ++rho) {
                                const int e = q4::q1_elem(tp, rho);
                                word |= (uint32_t)(q1_bit(sb, e) ^ 1) << rho;
                                word |= (uint32_t)(q1_bit(sb, e + 1) ^ 1) << (16 + rho);
                            }
                        store_u32(r + (4 * g + tp) * 8 + 4 * h, word);
                    }
                    if (sb) dw |= ((uint32_t)sb[0] | ((uint32_t)sb[1] << 8)) << (16 * h);
                }
                store_u32(r + 256 + 4 * g, dw);
            }
        }
    return Q4_OK;
}

extern "C" q4_status q4_unpack_q1(const void *host_packed, size_t packed_bytes, int32_t n, int32_t k,
                                  void *host_blocks) {
    if (!host_packed || !host_blocks) return Q4_ERR_NULL;
    if (!fmt_shape_ok(Q4_FMT_Q1, n, k)) return Q4_ERR_SHAPE;
    if (packed_bytes < q4_packed_bytes(Q4_FMT_Q1, n, k)) return Q4_ERR_SHAPE;
    const uint8_t *in = (const uint8_t *)host_packed;
    uint8_t *dst = (uint8_t *)host_blocks;
    const int64_t C = k / 128;
    memset(dst, 0, (size_t)n * (size_t)C * 18);
    for (int64_t row = 0; row < n; ++row)
        for (int64_t c = 0; c < C; ++c) {
            const uint8_t *r = in + ((row / 16) * C + c) * q4::kRecQ1;
            const int g = (int)(row % 8), h = (int)((row % 16) / 8);
            uint8_t *sb = dst + (row * C + c) * 18;
            const uint16_t d = (uint16_t)(load_u32(r + 256 + 4 * g) >> (16 * h));
            sb[0] = (uint8_t)(d & 0xFF);
            sb[1] = (uint8_t)(d >> 8);
            for (int tp = 0; tp < 4; ++tp) {
                const uint32_t word = load_u32(r + (4 * g + tp) * 8 + 4 * h);
                for (int rho = 0; rho < 16; ++rho) {
                    const int e = q4::q1_elem(tp, rho);
                    sb[2 + (e >> 3)] |= (uint8_t)((((word >> rho) & 1) ^ 1) << (e & 7));
                    sb[2 + ((e + 1) >> 3)] |= (uint8_t)((((word >> (16 + rho)) & 1) ^ 1) << ((e + 1) & 7));
                }
            }
        }
    return Q4_OK;
}

extern "C" q4_status q4_repack_q8_0(const void *host_blocks, int32_t n, int32_t k, void *host_out,
                                    size_t out_bytes) {
    if (!host_blocks || !host_out) return Q4_ERR_NULL;
    if (!shape_ok(n, k)) return Q4_ERR_SHAPE;
    if (out_bytes < q4_packed_bytes(Q4_FMT_Q8_0, n, k)) return Q4_ERR_SHAPE;
    const uint8_t *src = (const uint8_t *)host_blocks;
    uint8_t *out = (uint8_t *)host_out;
    const int64_t T = q4::tiles_of(n), C = q4::chunks_of(k), B = k / 32;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            uint8_t *r = out + (t * C + c) * q4::kRecQ8_0;
            for (int rr = 0; rr < 16; ++rr)
                for (int j = 0; j < 4; ++j) {
                    const int64_t row = t * 16 + rr, blk = c * 4 + j;
                    const bool real = row < n && blk < B;
                    const uint8_t *b = real ? src + (row * B + blk) * 34 : nullptr;
                    // biased bytes u = q + 128; padding is q = 0 with d = 0
                    for (int e = 0; e < 32; ++e) r[q8_off(rr, j, e)] = (uint8_t)(real ? b[2 + e] ^ 0x80u : 0x80u);
                }
            for (int g = 0; g < 8; ++g)
                for (int j = 0; j < 4; ++j) {
                    const int64_t blk = c * 4 + j, r0 = t * 16 + g, r1 = r0 + 8;
                    auto scale = [&](int64_t row) -> uint32_t {
                        if (row >= n || blk >= B) return 0;
                        const uint8_t *b = src + (row * B + blk) * 34;
                        return (uint32_t)b[0] | ((uint32_t)b[1] << 8);
                    };
                    store_u32(r + 2048 + g * 16 + j * 4, scale(r0) | (scale(r1) << 16));
                }
        }
    return Q4_OK;
}

extern "C" q4_status q4_unpack_q8_0(const void *host_packed, size_t packed_bytes, int32_t n, int32_t k,
                                    void *host_blocks) {
    if (!host_packed || !host_blocks) return Q4_ERR_NULL;
    if (!shape_ok(n, k)) return Q4_ERR_SHAPE;
    if (packed_bytes < q4_packed_bytes(Q4_FMT_Q8_0, n, k)) return Q4_ERR_SHAPE;
    const uint8_t *in = (const uint8_t *)host_packed;
    uint8_t *dst = (uint8_t *)host_blocks;
    const int64_t T = q4::tiles_of(n), C = q4::chunks_of(k), B = k / 32;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            const uint8_t *r = in + (t * C + c) * q4::kRecQ8_0;
            for (int rr = 0; rr < 16; ++rr)
                for (int j = 0; j < 4; ++j) {
                    const int64_t row = t * 16 + rr, blk = c * 4 + j;
                    if (row >= n || blk >= B) continue;
                    uint8_t *b = dst + (row * B + blk) * 34;
                    const uint32_t sw = load_u32(r + 2048 + (rr & 7) * 16 + j * 4);
                    const uint16_t sv = (uint16_t)((rr >> 3) ? (sw >> 16) : (sw & 0xFFFF));
                    b[0] = (uint8_t)(sv & 0xFF);
                    b[1] = (uint8_t)(sv >> 8);
                    for (int e = 0; e < 32; ++e) b[2 + e] = (uint8_t)(r[q8_off(rr, j, e)] ^ 0x80u);
                }
        }
    return Q4_OK;
}

// Walk every real (row, block) of a packed buffer and hand its 32 nibbles and
// 16-bit scale / min to `put`.
template <class Put>
static void unpack(int fmt, int32_t n, int32_t k, const uint8_t *in, Put put) {
    const int64_t T = q4::tiles_of(n), C = q4::chunks_of(k), B = k / 32;
    const int rec = q4::rec_bytes(fmt);
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            const uint8_t *r = in + (t * C + c) * rec;
            for (int h = 0; h < 2; ++h)
                for (int g = 0; g < 8; ++g)
                    for (int j = 0; j < 4; ++j) {
                        int64_t row = t * 16 + h * 8 + g, blk = c * 4 + j;
                        if (row >= n || blk >= B) continue;
                        int q[32];
                        for (int tp = 0; tp < 4; ++tp) {
                            uint32_t word = load_u32(r + h * 512 + (4 * g + tp) * 16 + j * 4);
                            for (int i = 0; i < 8; ++i) q[q4::nib_elem(tp, i)] = (word >> (4 * i)) & 15;
                        }
                        uint32_t sw = load_u32(r + 1024 + g * 16 + j * 4);
                        uint16_t sv = (uint16_t)(h ? (sw >> 16) : (sw & 0xFFFF));
                        uint16_t mv = 0;
                        if (fmt == Q4_FMT_AFFINE) {
                            uint32_t mw = load_u32(r + 1152 + g * 16 + j * 4);
                            mv = (uint16_t)(h ? (mw >> 16) : (mw & 0xFFFF));
                        }
                        put(row, blk, q, sv, mv);
                    }
        }
}

extern "C" q4_status q4_unpack_q4_0(const void *host_packed, size_t packed_bytes, int32_t n, int32_t k,
                                    void *host_blocks) {
    if (!host_packed || !host_blocks) return Q4_ERR_NULL;
    if (!shape_ok(n, k)) return Q4_ERR_SHAPE;
    if (packed_bytes < q4_packed_bytes(Q4_FMT_Q4_0, n, k)) return Q4_ERR_SHAPE;
    uint8_t *dst = (uint8_t *)host_blocks;
    const int64_t B = k / 32;
    unpack(Q4_FMT_Q4_0, n, k, (const uint8_t *)host_packed,
           [&](int64_t row, int64_t blk, const int *q, uint16_t s, uint16_t) {
               uint8_t *b = dst + (row * B + blk) * 18;
               b[0] = (uint8_t)(s & 0xFF);
               b[1] = (uint8_t)(s >> 8);
               for (int i = 0; i < 16; ++i) b[2 + i] = (uint8_t)(q[i] | (q[i + 16] << 4));
           });
    return Q4_OK;
}

extern "C" q4_status q4_unpack_affine(const void *host_packed, size_t packed_bytes, int32_t n, int32_t k,
                                      uint8_t *nib, uint16_t *s, uint16_t *m) {
    if (!host_packed || !nib || !s || !m) return Q4_ERR_NULL;
    if (!shape_ok(n, k)) return Q4_ERR_SHAPE;
    if (packed_bytes < q4_packed_bytes(Q4_FMT_AFFINE, n, k)) return Q4_ERR_SHAPE;
    const int64_t B = k / 32;
    unpack(Q4_FMT_AFFINE, n, k, (const uint8_t *)host_packed,
           [&](int64_t row, int64_t blk, const int *q, uint16_t sv, uint16_t mv) {
               uint8_t *r = nib + row * (k / 2) + blk * 16;
               for (int i = 0; i < 16; ++i) r[i] = (uint8_t)(q[2 * i] | (q[2 * i + 1] << 4));
               s[row * B + blk] = sv;
               m[row * B + blk] = mv;
           });
    return Q4_OK;
}

extern "C" q4_status q4_unpack_q4_k(const void *host_packed, size_t packed_bytes, int32_t n, int32_t k,
                                    void *host_blocks) {
    if (!host_packed || !host_blocks) return Q4_ERR_NULL;
    if (!fmt_shape_ok(Q4_FMT_Q4_K, n, k)) return Q4_ERR_SHAPE;
    if (packed_bytes < q4_packed_bytes(Q4_FMT_Q4_K, n, k)) return Q4_ERR_SHAPE;
    const uint8_t *in = (const uint8_t *)host_packed;
    uint8_t *dst = (uint8_t *)host_blocks;
    const int64_t NS = k / 256, C = q4::chunks_of(k);
    memset(dst, 0, (size_t)n * (size_t)NS * 144);
    unpack(Q4_FMT_Q4_K, n, k, in, [&](int64_t row, int64_t blk, const int *q, uint16_t sv, uint16_t) {
        uint8_t *sb = dst + (row * NS + blk / 8) * 144;
        const int j = (int)(blk % 8);
        q4k_put(sb, j, sv & 0xFF, sv >> 8);
        for (int e = 0; e < 32; ++e) sb[16 + 32 * (j >> 1) + e] |= (uint8_t)(q[e] << (4 * (j & 1)));
        if (j == 0) {  // d and dmin from the superblock's first chunk
            const uint8_t *r = in + ((row / 16) * C + blk / 4) * q4::kRecQ4_K;
            const int g = (int)(row % 8), h = (int)((row % 16) / 8);
            const uint32_t dw = load_u32(r + 1152 + g * 4), mw = load_u32(r + 1184 + g * 4);
            const uint16_t d = (uint16_t)(dw >> (16 * h)), dm = (uint16_t)(mw >> (16 * h));
            sb[0] = (uint8_t)(d & 0xFF);
            sb[1] = (uint8_t)(d >> 8);
            sb[2] = (uint8_t)(dm & 0xFF);
            sb[3] = (uint8_t)(dm >> 8);
        }
    });
    return Q4_OK;
}

// RoPE tables (honeycrisp/mod.rs, attn_state: theta = pos / rope_theta^(2j /
// head_dim) for j < head_dim / 2), computed in double and rounded to fp32.
extern "C" q4_status q4_rope_table(int32_t max_seq, int32_t D, double rope_theta, float *host_cos,
                                   float *host_sin) {
    if (!host_cos || !host_sin) return Q4_ERR_NULL;
    if (max_seq < 1 || max_seq > (1 << 24) || D < 2 || D % 2 != 0 || !(rope_theta > 0.0)) return Q4_ERR_SHAPE;
    const int half = D / 2;
    for (int64_t p = 0; p < max_seq; ++p)
        for (int j = 0; j < half; ++j) {
            const double th = (double)p / pow(rope_theta, 2.0 * j / D);
            host_cos[p * half + j] = (float)cos(th);
            host_sin[p * half + j] = (float)sin(th);
        }
    return Q4_OK;
}
