/*
 * q4gemv.h -- C ABI of libq4gemv: weight-only 4-bit dequant-in-GEMV over a
 * small batch of activation rows, fused with its decode-step neighbours.
 *
 * Sources for the operations (page title, then the item on it):
 *  - crate inferencelayer (docs.rs), Functions: gemv_q4_k_lcpp_src (Q4 GEMV,
 *    1-16 activation columns, fp32 accumulation), q4_0_to_q8_0n (Q4_0 weight
 *    = d * (nib - 8)), gemv_q1_k_lcpp_src (a Q4_0 block is 18 bytes per 32
 *    weights), gemm_q4_splitk_reduce_src (split-K partials folded in a fixed
 *    slice order).
 *  - Module gpu (qwen4_exp, docs.cherenkov.io): Struct Q (affine-Q4
 *    projection), Struct HalfSet (per-32 activation group sums feed the
 *    multi-row Q4 matvecs), Constant MAX_NB (rows per step), module
 *    sampling (logits projection and greedy argmax).
 *  - honeycrisp/mod.rs (cyber.page): forward_decode_fused_layers (Q matmul
 *    with inline input_norm; K+V dual with inline input_norm; matmul +
 *    residual; post_norm + gate + up + silu), fused_ffn_residual, Op::RmsNorm.
 *
 * Conventions for every call below:
 *  - Memory: weights, activations, outputs and workspaces are DEVICE
 *    pointers owned by the caller; the library allocates nothing, keeps no
 *    pointer after a call returns and has no host-visible state.  Host
 *    pointers appear only in the repack/unpack calls and are marked "host".
 *  - Layout: activations are row-major [nb][k] fp32, outputs [nb][n] fp32
 *    (row r of a batch is one decode position).  1 <= nb <= 16, k % 32 == 0,
 *    1 <= n, k <= 65536 (one packed weight must stay below 2^31 bytes).
 *  - Alignment: every device pointer must be 16-byte aligned.
 *  - Errors: arguments are validated on the host before anything is
 *    launched; on any error nothing is launched and a status other than
 *    Q4_OK is returned.  A launch failure returns Q4_ERR_CUDA (from
 *    cudaGetLastError).  Kernels never trap and never spin on a flag.
 *  - Asynchrony: calls enqueue work on `stream` and return; they never
 *    synchronise the host.  Kernels are launched with programmatic
 *    dependent launch: each waits for the preceding kernel in the stream
 *    before it reads activations or writes outputs, and only reads weights
 *    (which must not be written concurrently) before that point.
 *  - Aliasing: outputs must not overlap inputs, except y == r in
 *    q4_res_gemv.
 *  - Numerics: fp32 accumulation of exact dequantised weights against the
 *    activations carried to about 22 significant bits; per output
 *    |y - y_exact| <= 1e-3 * sum_k |w_k| |x_k| + 1e-6 for finite inputs.
 */
#ifndef Q4GEMV_H
#define Q4GEMV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    Q4_OK = 0,
    Q4_ERR_NULL = 1,          /* a required pointer is NULL */
    Q4_ERR_SHAPE = 2,         /* n, k or a byte count is out of range / inconsistent */
    Q4_ERR_ALIGN = 3,         /* a device pointer is not 16-byte aligned */
    Q4_ERR_UNSUPPORTED = 4,   /* nb outside 1..16, unknown format, mixed formats */
    Q4_ERR_WORKSPACE = 5,     /* workspace missing or smaller than required */
    Q4_ERR_CUDA = 6           /* a CUDA runtime call failed */
} q4_status;

typedef enum {
    Q4_FMT_Q4_0 = 0,    /* 32 weights: fp16 scale d + 16 nibble bytes; w = d*(q-8) */
    Q4_FMT_AFFINE = 1,  /* 32 weights: bf16 scale s, bf16 min m, 16 nibble bytes; w = s*q + m */
    Q4_FMT_Q8_0 = 2,    /* 32 weights: fp16 scale d + 32 signed bytes; w = d*q */
    Q4_FMT_Q4_K = 3,    /* 256-weight superblocks: fp16 d, dmin, 6-bit sub-scales sc and mins mn
                           per 32 weights, nibbles; w = d*sc*q - dmin*mn (k a multiple of 256) */
    Q4_FMT_Q1 = 4       /* 128-weight superblocks: fp16 d + 128 sign bits; w = +d (bit 1) or -d
                           (bit 0) (k a multiple of 128) */
} q4_format;

/* A non-owning view of one repacked weight matrix in device memory.
 * `dev` points to q4_packed_bytes(fmt, n, k) bytes written by a repack call
 * (copied to the device by the caller); `bytes` is that size. */
typedef struct {
    int32_t fmt;        /* q4_format */
    int32_t n;          /* output rows */
    int32_t k;          /* input length, multiple of 32 (of 256 for Q4_K, of 128 for Q1) */
    const void *dev;    /* device pointer, 16-byte aligned */
    size_t bytes;       /* size of the packed buffer */
} q4_weight;

/* Size in bytes of the device layout of an n x k weight (0 on bad shape).
 * The layout is 16-row tiles x 128-column chunks; rows are padded to a
 * multiple of 16 and columns to a multiple of 128 with zero-valued weights,
 * so the size may exceed the algorithmic 18 (Q4_0) or 20 (affine) bytes per
 * 32 weights when n % 16 or k % 128 is not zero.  Q8_0 takes 2176 bytes per
 * 16 x 128 tile chunk (34 per 32 weights); Q4_K takes 1216 (19 per 32
 * weights: each chunk repeats its superblock's d and dmin); Q1 takes 288
 * (4.5 per 32 weights). */
size_t q4_packed_bytes(int32_t fmt, int32_t n, int32_t k);

/* Algorithmic weight bytes of an n x k matrix: 18 (Q4_0), 20 (affine) or 34
 * (Q8_0) per 32 weights, 144 per 256 (Q4_K), 18 per 128 (Q1); 0 on bad shape. */
size_t q4_weight_bytes(int32_t fmt, int32_t n, int32_t k);

/* Host -> host, lossless, deterministic repack of Q4_0 blocks into the
 * device layout.  host_blocks: [n][k/32] blocks of 18 bytes (fp16 d little
 * endian, then 16 bytes; byte i holds element i in its low nibble and
 * element i+16 in its high nibble).  host_out: q4_packed_bytes(...) bytes. */
q4_status q4_repack_q4_0(const void *host_blocks, int32_t n, int32_t k,
                         void *host_out, size_t out_bytes);

/* Host -> host repack of affine-Q4 weights.  nib: [n][k/2] bytes, byte i
 * holding element 2i (low nibble) and 2i+1 (high nibble); s, m: [n][k/32]
 * bf16 bit patterns; host_out: q4_packed_bytes(...) bytes. */
q4_status q4_repack_affine(const uint8_t *nib, const uint16_t *s, const uint16_t *m,
                           int32_t n, int32_t k, void *host_out, size_t out_bytes);

/* Inverse of q4_repack_q4_0 (host -> host); used to check the round trip. */
q4_status q4_unpack_q4_0(const void *host_packed, size_t packed_bytes, int32_t n, int32_t k,
                         void *host_blocks);

/* Q8_0 host blocks (crate inferencelayer, Functions: q4_0_to_q8_0n,
 * gemv_q8_0n_k_lcpp_src): [n][k/32] blocks of 34 bytes, the fp16 scale d
 * (little endian) then 32 signed bytes q; w = d*q.  Lossless, host -> host,
 * like q4_repack_q4_0; host_out holds q4_packed_bytes(Q4_FMT_Q8_0, n, k). */
q4_status q4_repack_q8_0(const void *host_blocks, int32_t n, int32_t k, void *host_out, size_t out_bytes);

/* Inverse of q4_repack_q8_0 (host -> host). */
q4_status q4_unpack_q8_0(const void *host_packed, size_t packed_bytes, int32_t n, int32_t k, void *host_blocks);

/* Q4_K host superblocks (crate inferencelayer, Functions:
 * gemv_q5k_k_lcpp_src, whose layout minus the fifth-bit plane this is;
 * honeycrisp/mod.rs, quant_matmul's Q4_K branch): [n][k/256] superblocks of
 * 144 bytes -- fp16 d, fp16 dmin (little endian), 12 bytes of 6-bit sub-block
 * scales and mins (sub-blocks 0-3: low six bits of bytes j and j+4; 4-7: the
 * nibbles of byte j+4 topped by bits 6-7 of bytes j-4 and j), 128 nibble bytes
 * (run r of 32 holds sub-block 2r in its low nibbles, 2r+1 in its high ones);
 * w = d*sc*q - dmin*mn.  k must be a multiple of 256 (else Q4_ERR_SHAPE).
 * Lossless, host -> host; host_out holds q4_packed_bytes(Q4_FMT_Q4_K, n, k). */
q4_status q4_repack_q4_k(const void *host_blocks, int32_t n, int32_t k, void *host_out, size_t out_bytes);

/* Inverse of q4_repack_q4_k (host -> host). */
q4_status q4_unpack_q4_k(const void *host_packed, size_t packed_bytes, int32_t n, int32_t k, void *host_blocks);

/* Q1 host superblocks (crate inferencelayer, Functions: gemv_q1_k_lcpp_src,
 * gemm_q1_src): [n][k/128] superblocks of 18 bytes -- the fp16 scale d
 * (little endian), then 16 bytes of sign bits, byte i holding elements
 * 8i..8i+7 from its lowest bit; w = +d for a set bit, -d for a clear one.  k
 * must be a multiple of 128 (else Q4_ERR_SHAPE).  Lossless, host -> host;
 * host_out holds q4_packed_bytes(Q4_FMT_Q1, n, k). */
q4_status q4_repack_q1(const void *host_blocks, int32_t n, int32_t k, void *host_out, size_t out_bytes);

/* Inverse of q4_repack_q1 (host -> host). */
q4_status q4_unpack_q1(const void *host_packed, size_t packed_bytes, int32_t n, int32_t k, void *host_blocks);

/* Inverse of q4_repack_affine (host -> host). */
q4_status q4_unpack_affine(const void *host_packed, size_t packed_bytes, int32_t n, int32_t k,
                           uint8_t *nib, uint16_t *s, uint16_t *m);

/* Per-32 group sums of a row batch (Module gpu, Struct HalfSet):
 * gsum[r][g] = fp32 sum of x[r][32g .. 32g+31], added in ascending order.
 * x: [nb][k] device fp32; gsum: [nb][k/32] device fp32. */
q4_status q4_group_sums(const float *x, int32_t nb, int32_t k, float *gsum, cudaStream_t stream);

/* y[r][i] = sum_k w[i][k] * x[r][k]   (dequant-in-GEMV).
 * x: [nb][k]; y: [nb][n].  gsum: affine weights only, [nb][k/32] group sums
 * of x as q4_group_sums writes them, or NULL to have the kernel compute them
 * (ignored for Q4_0). */
q4_status q4_gemv(const q4_weight *W, const float *x, const float *gsum, int32_t nb,
                  float *y, cudaStream_t stream);

/* RMSNorm prologue then GEMV (honeycrisp/mod.rs, forward_decode_fused_layers,
 * "Q matmul with inline input_norm"):
 *   xhat[r][k] = x[r][k] / sqrt(mean_k x[r][k]^2 + eps) * gamma[k];
 *   y[r][i] = sum_k w[i][k] * xhat[r][k].
 * gamma: [k] device fp32. */
q4_status q4_nrm_gemv(const q4_weight *W, const float *x, const float *gamma, float eps,
                      int32_t nb, float *y, cudaStream_t stream);

/* Two weight streams over one (optionally RMS-normed) activation batch in
 * one launch (forward_decode_fused_layers, K+V dual with inline input_norm):
 *   ya = Wa * xhat, yb = Wb * xhat, xhat = x when gamma is NULL.
 * Wa and Wb must have the same format and k.  ya: [nb][Wa.n], yb: [nb][Wb.n]. */
q4_status q4_dual_gemv(const q4_weight *Wa, const q4_weight *Wb, const float *x,
                       const float *gamma, float eps, int32_t nb, float *ya, float *yb,
                       cudaStream_t stream);

/* RMSNorm, gate and up projections and the SwiGLU epilogue in one launch
 * (forward_decode_fused_layers, post_norm + gate + up + silu; fused_ffn_residual
 * step 4):  h[r][i] = silu(g) * u,  g = (Wg xhat)[r][i], u = (Wu xhat)[r][i],
 * silu(t) = t / (1 + exp(-t)).  Wg and Wu: same format, n and k.  h: [nb][n]. */
q4_status q4_gus_nrm(const q4_weight *Wg, const q4_weight *Wu, const float *x,
                     const float *gamma, float eps, int32_t nb, float *h, cudaStream_t stream);

/* GEMV with a residual-add epilogue (forward_decode_fused_layers, fused
 * matmul + residual):  y[r][i] = sum_k w[i][k] x[r][k] + r_in[r][i].
 * r_in, y: [nb][n]; y may equal r_in (in-place residual stream). */
q4_status q4_res_gemv(const q4_weight *W, const float *x, const float *r_in, int32_t nb,
                      float *y, cudaStream_t stream);

/* HalfSet packing (Module gpu, Struct HalfSet: "half even/odd streams plus
 * per-32 group sums", the input format of the multi-row Q4 matvecs).  For each
 * activation row r of x ([nb][k] fp32, device): x_even[r][i] = f16(x[r][2i])
 * and x_odd[r][i] = f16(x[r][2i+1]) ([nb][k/2] f16 bits each, device;
 * round to nearest, ties to even), and gsum[r][g] ([nb][k/32] fp32, device,
 * or NULL for none) = the fp32 sum of the 32 f16 values of group g, added in
 * the order q4_group_sums and the GEMV's own staging use.  A caller that
 * runs several multi-row matvecs on one batch (speculative verification)
 * converts once.  Same validation as q4_group_sums. */
q4_status q4_pack_half(const float *x, int32_t nb, int32_t k, uint16_t *x_even, uint16_t *x_odd, float *gsum,
                       cudaStream_t stream);

/* y = W x for nb rows (1..16) given as a HalfSet: x[r][2i] = x_even[r][i],
 * x[r][2i+1] = x_odd[r][i] (f16 bits, [nb][k/2] each, device).  gsum
 * ([nb][k/32] fp32, device): for affine weights the group sums of those f16
 * values (q4_pack_half writes them), or NULL to have the kernel form them; it
 * must match the streams; ignored for Q4_0.  Results are those of q4_gemv on
 * the f16 values widened to fp32 (bit for bit). */
q4_status q4_gemv_half(const q4_weight *W, const uint16_t *x_even, const uint16_t *x_odd, const float *gsum,
                       int32_t nb, float *y, cudaStream_t stream);

/* Workspace bytes q4_argmax needs for an n-row logits projection and nb rows. */
size_t q4_argmax_workspace_bytes(int32_t n, int32_t nb);

/* Logits projection (optionally behind an RMSNorm when gamma is not NULL)
 * and greedy argmax per activation row (Module gpu, module sampling), in two
 * passes: pass 1 computes the logits tile by tile and writes one (max, index)
 * pair per thread-block group to `workspace`; pass 2 folds those pairs in
 * group order.  Ties go to the lowest index; a NaN logit ranks below every
 * number.  idx: [nb] int32 (required); val: [nb] the maximum logit, or NULL;
 * logits: [nb][n] all logits, or NULL.  workspace: device memory of at least
 * q4_argmax_workspace_bytes(n, nb) bytes, no initialisation needed. */
q4_status q4_argmax(const q4_weight *W, const float *x, const float *gamma, float eps,
                    int32_t nb, int32_t *idx, float *val, float *logits,
                    void *workspace, size_t ws_bytes, cudaStream_t stream);

/* One decoder layer of the decode step (q4_decode_step).  All seven weights
 * share one format; hidden = Wo.n = Wd.n = the k of Wq, Wk, Wv, Wg, Wu and
 * Wo; inter = Wg.n = Wu.n = Wd.k.  `attn` is the attention output the o
 * projection consumes ([nb][hidden], device), gamma_in / gamma_post the
 * RMSNorm weights before the q/k/v and the gate/up projections. */
typedef struct {
    q4_weight Wq, Wk, Wv, Wo, Wg, Wu, Wd;
    const float *gamma_in;
    const float *gamma_post;
    const float *attn;
} q4_decode_layer;

/* Workspace bytes q4_decode_step needs for nb activation rows. */
size_t q4_decode_workspace_bytes(int32_t nb);

/* One decode step as a single persistent kernel (honeycrisp/mod.rs,
 * forward_decode_fused_layers: the whole stack in one submission; Module
 * gpu, module sampling: logits projection and greedy argmax).  Per layer:
 *   q, k, v = (Wq, Wk, Wv) * rmsnorm(src, gamma_in)    src = x_in, then hid
 *   hid     = src + Wo * attn
 *   h       = silu(Wg * rmsnorm(hid, gamma_post)) * (Wu * rmsnorm(hid, gamma_post))
 *   hid     = hid + Wd * h
 * then idx[r] = argmax_i (Wlogits * rmsnorm(hid, gamma_final))[r][i] (ties to
 * the lowest index), val[r] its logit (val may be NULL).
 * layers: HOST array of n_layers (1..32) descriptors, read during the call.
 * x_in [nb][hidden] is read only; hid [nb][hidden] receives the final hidden
 * state; q, k, v, h ([nb][Wq.n], [nb][Wk.n], [nb][Wv.n], [nb][inter]) receive
 * the last layer's projections and are scratch otherwise.  workspace: device
 * memory of q4_decode_workspace_bytes(nb) bytes; the call zeroes the first
 * 16 bytes (a grid-barrier counter and an error word) on `stream` before the
 * launch.  The kernel is a cooperative launch of one CTA per SM whose jobs
 * are separated by grid-wide barriers; a barrier that does not complete in
 * bounded time sets the error word and the kernel returns early (see
 * q4_decode_check).  Returns Q4_ERR_UNSUPPORTED when the shapes need more
 * shared memory than one CTA has (large nb * inter). */
q4_status q4_decode_step(const q4_decode_layer *layers, int32_t n_layers, const q4_weight *Wlogits,
                         const float *gamma_final, float eps, int32_t nb, const float *x_in, float *hid,
                         float *q, float *k, float *v, float *h, int32_t *idx, float *val, void *workspace,
                         size_t ws_bytes, cudaStream_t stream);

/* The decode attention of q4_decode_step_attn (honeycrisp/mod.rs,
 * gpu_attention and the fused RoPE + KV-append + SDPA dispatch of
 * forward_decode_fused_layers), for one token at `position`: per layer, q,
 * the new k and v (the layer's q/k/v projections, read as heads of
 * head_dim), RoPE of q and k from the tables, k and v appended to the layer's
 * caches at `position`, then out = softmax(scale q K^T) V over the cached
 * positions [lo, position] (lo = position + 1 - window when window > 0 and
 * the context is longer, else 0), query head h reading kv head h / (heads /
 * kv_heads).
 * k_caches, v_caches: HOST arrays of n_layers device pointers, each cache
 * [kv_heads][max_seq][head_dim] fp32 (16-byte aligned), read during the call.
 * rope_cos, rope_sin: device [max_seq][head_dim/2] tables (q4_rope_table), or
 * both NULL for no RoPE.  out: device [heads * head_dim], the attention
 * output the o projections consume (scratch between layers).  scale <= 0
 * means 1/sqrt(head_dim).  Library-specific geometry limits: head_dim 64 and
 * four query heads per kv head (Q4_ERR_UNSUPPORTED otherwise; q4_attn_decode
 * covers the others call by call). */
typedef struct {
    float *const *k_caches;
    float *const *v_caches;
    const float *rope_cos;
    const float *rope_sin;
    float *out;
    int32_t max_seq, position, window, heads, kv_heads, head_dim;
    float scale;
} q4_step_attention;

/* Workspace bytes q4_decode_step_attn needs (nb = 1); 0 for a geometry it
 * does not take. */
size_t q4_decode_attn_workspace_bytes(int32_t heads, int32_t kv_heads, int32_t head_dim);

/* The real decode step as a single persistent kernel: q4_decode_step with
 * each layer's decode attention (q4_step_attention) between its q/k/v and o
 * projections, in place of the `attn` stand-in (layers[l].attn is not read):
 *   q, k, v = (Wq, Wk, Wv) * rmsnorm(src, gamma_in)
 *   out     = attention(q, k, v, caches of layer l)     (appends k, v)
 *   hid     = src + Wo * out,  then gate/up/SwiGLU and down as in q4_decode_step
 * then the logits argmax.  nb = 1 (x_in, hid [1][hidden]); heads * head_dim
 * must equal hidden (Wq.n, Wo.k) and kv_heads * head_dim Wk.n and Wv.n;
 * n_layers 1..25.  workspace: q4_decode_attn_workspace_bytes bytes; the call
 * zeroes its first 80 bytes on `stream` before the launch.  Each attention
 * is a job of the kernel: CTA c takes kv head c / (CTAs / kv_heads) and a
 * split of the positions, and the last split of a kv head to finish folds
 * the splits (no wait; the same result whatever the CTA order).  Failure
 * reporting as for q4_decode_step (q4_decode_check). */
q4_status q4_decode_step_attn(const q4_decode_layer *layers, int32_t n_layers, const q4_step_attention *att,
                              const q4_weight *Wlogits, const float *gamma_final, float eps, const float *x_in,
                              float *hid, float *q, float *k, float *v, float *h, int32_t *idx, float *val,
                              void *workspace, size_t ws_bytes, cudaStream_t stream);

/* Synchronises `stream` and reports whether the last q4_decode_step (or
 * q4_decode_step_attn) on this workspace completed all its grid barriers and
 * weight copies (Q4_OK) or gave up on one (Q4_ERR_CUDA). */
q4_status q4_decode_check(const void *workspace, cudaStream_t stream);

/* Synchronises `stream` and reports whether any GEMV-family kernel of this
 * library on the current device (q4_gemv, q4_nrm_gemv, q4_dual_gemv,
 * q4_gus_nrm, q4_res_gemv, q4_argmax, q4_argmax_noalloc, q4_gemm,
 * q4_attn_decode) gave up waiting for its weight (or K/V) copies since the
 * last check (Q4_ERR_CUDA; the flag is then
 * cleared) or not (Q4_OK).  Each kernel bounds every such wait (about a
 * second); a kernel that gives up records it in a per-device word of the
 * library, stops streaming, waits (bounded) for its copies in flight and
 * returns, leaving its outputs undefined.  The word's address is resolved
 * on the first library call on a device; make that call before any stream
 * capture.  Library-specific: the pages have no counterpart. */
q4_status q4_device_check(cudaStream_t stream);

/* Testing hook for the give-up path of the kernels' bounded waits.  The pages
 * have no counterpart.  Sets, for every later launch of this process:
 * barrier_polls, the polls before a grid barrier of q4_decode_step gives up
 * (<= 0: the default, 2^22); barrier_extra (0 or 1), arrivals each grid
 * barrier expects beyond its CTAs; copy_wait_cycles, the SM clock cycles
 * before a wait for a weight-copy stage gives up (<= 0: the default, 2^31,
 * about a second); copy_extra_bytes (0..4096, a multiple of 16), bytes each
 * weight-copy stage of the GEMV kernels expects beyond its copies (the first
 * stage only for q4_gemm and for each CTA of q4_attn_decode).  A non-zero extra makes every
 * such wait run out: the kernel then records the failure (q4_decode_check,
 * q4_device_check), waits for its copies in flight (always bounded by the
 * default second) and returns with its outputs undefined; nothing faults or
 * hangs.  q4_debug_wait_limits(0, 0, 0, 0) restores the defaults.  Not for
 * use while other threads launch this library's kernels.  Q4_ERR_SHAPE on an
 * argument out of range (nothing changes). */
q4_status q4_debug_wait_limits(int64_t barrier_polls, int32_t barrier_extra, int64_t copy_wait_cycles,
                               int32_t copy_extra_bytes);

/* Allocation-free variant of q4_argmax.  The pages have no counterpart: this
 * exists for callers that cannot allocate device memory where they need the
 * argmax, such as a plug-in whose host application owns all device memory and
 * gives it no allocator, or a decode loop that must not call cudaMalloc once
 * running (a cudaMalloc can synchronise the device and stall the step).
 * Same arguments and results as q4_argmax without the workspace: the pass-1
 * (max, index) pairs live in a 128 KiB array compiled into the library, which
 * every GPU that loads the library holds until the process exits.
 * - Limit: the call needs G x nb (max, index) pairs of 8 bytes, G being the
 *   thread-block groups of its launch plan (G <= ceil(n/16)); it is accepted
 *   when G x nb <= 16384 (4-byte values rounded up to 16 bytes, then the
 *   4-byte indices, within the 131072 bytes).  So ceil(n/16) * nb <= 16384
 *   always fits (the 65536-row logits projection fits at every nb).  A larger
 *   need returns Q4_ERR_WORKSPACE and launches nothing.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and caches it; make that
 *   first call before any stream capture.
 * - Every call shares the one array.  Nothing in it needs to start at zero
 *   (pass 1 writes every pair pass 2 reads), but calls whose kernels overlap
 *   on the GPU (other streams, other threads) race on it: serialise them.
 * - It calls no cudaMalloc, cudaFree or other allocating routine. */
q4_status q4_argmax_noalloc(const q4_weight *W, const float *x, const float *gamma, float eps,
                            int32_t nb, int32_t *idx, float *val, float *logits, cudaStream_t stream);

/* ---------------------------------------------------------------- prefill GEMM
 * y = x W^T for a wide activation batch (crate inferencelayer, Functions:
 * gemm_q4_src, the blocked prefill GEMM whose column tile shares one weight
 * stream; its dims.z = 1 form accumulates into y).  Any nb >= 1 (meant for
 * nb > 16, where the GEMV family re-reads the weights per 16 rows); every
 * weight format.  x: [nb][k] fp32; y: [nb][n] fp32, overwritten, or with
 * accumulate != 0 y += x W^T (y must then hold the values to add to).
 * Numerics: weights exact, products accumulated in fp32, each activation
 * carried as one f16 (relative rounding at most 2^-11) after a power-of-two
 * scale: per 32-column block of a row (as the GEMV calls do above four rows)
 * in the mma.sync form that serves every format (Q4_0 and Q8_0 up to 16 rows);
 * per activation row in the tcgen05 form that serves Q4_0 and Q8_0 from 17 rows (there the
 * weights enter the tensor core as f16 hi + lo pairs with an exact sum, and
 * the fp32 accumulator lives in tensor memory).
 * Workspace: q4_gemm_workspace_bytes(nb, k) device bytes (16-byte aligned,
 * contents need not be initialised) hold the staged activations; the call
 * launches a staging kernel and the GEMM kernel on `stream`.
 * Q4_ERR_SHAPE for nb outside 1..2^20, Q4_ERR_WORKSPACE for a missing or short
 * workspace; the weight and pointer checks are the GEMV family's. */
size_t q4_gemm_workspace_bytes(int32_t nb, int32_t k);
q4_status q4_gemm(const q4_weight *W, const float *x, int32_t nb, float *y, int32_t accumulate, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------- attention
 * Decode attention of one token (honeycrisp/mod.rs: attn_state, gpu_attention
 * and the fused RoPE + KV-append + SDPA dispatch of
 * forward_decode_fused_layers), one call on `stream`:
 *  1. with tables, q (every head) and k_new (every kv head) are rotated by
 *     the tables' row `position`: element j pairs with element j + D/2,
 *     (a, b) -> (a c - b s, b c + a s);
 *  2. k_new (rotated) and v_new are written to row `position` of the caches;
 *  3. the attended positions are [lo, position + 1), lo = max(0, position + 1
 *     - window) for window > 0, else 0;
 *  4. query head h reads kv head h / (H / Hkv); out_h = sum_t p_t v_t with p
 *     the softmax over t of scale * q_h . k_t.
 * Arguments (device pointers, fp32, 16-byte aligned, row-major):
 *   q [H][D], k_new and v_new [Hkv][D]; k_cache and v_cache [Hkv][max_seq][D]
 *   (row `position` is written, rows >= position + 1 are never read); rope_cos
 *   and rope_sin [max_seq][D/2] or both NULL (no rotation; q4_rope_table
 *   fills them); out [H][D].
 * Supported: D = 64 with H / Hkv in {1, 2, 4, 8, 16}, D = 128 with H / Hkv
 * in {1, 2, 4, 8}, else Q4_ERR_UNSUPPORTED; 0 <= position < max_seq <= 2^24
 * and window >= 0, else Q4_ERR_SHAPE.
 * Workspace: a device buffer of q4_attn_workspace_bytes(H, D, max_seq)
 * bytes (16-byte aligned), zero-filled by the caller before its first use:
 * it holds per-kv-head counters (every call leaves them zero) and the
 * partial results of the splits of the attended positions.  It may be NULL
 * when the call needs one split only (Q4_ERR_WORKSPACE if it is needed and
 * missing or short).  Calls that share a workspace must not run at the same
 * time.
 * The caller owns every buffer; out must not overlap the inputs.  Results
 * do not depend on run-to-run scheduling (chunks are folded in order). */
size_t q4_attn_workspace_bytes(int32_t H, int32_t D, int32_t max_seq);
q4_status q4_attn_decode(const float *q, const float *k_new, const float *v_new, float *k_cache, float *v_cache,
                         int32_t max_seq, int32_t position, int32_t H, int32_t Hkv, int32_t D, int32_t window,
                         float scale, const float *rope_cos, const float *rope_sin, float *out, void *workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/* Host: RoPE tables cos and sin [max_seq][D/2] (fp32, computed in double) of
 * the angle pos / rope_theta^(2j/D) (honeycrisp/mod.rs, attn_state).  D even,
 * rope_theta > 0, 1 <= max_seq <= 2^24, else Q4_ERR_SHAPE. */
q4_status q4_rope_table(int32_t max_seq, int32_t D, double rope_theta, float *host_cos, float *host_sin);

/* Launch plan the library uses for a GEMV-shaped call (host-only; exposed
 * for tests and tuning).  tiles: 16-row tiles of the launch, chunks: 128-k
 * chunks per row, pairs: 1 when tiles come in gate/up pairs, num_sms:
 * multiprocessors of the device.  out[0..5] = tiles per group, K-split
 * (cluster size), chunks per K-slice, groups, CTAs, dynamic shared bytes. */
q4_status q4_plan(int32_t fmt, int32_t tiles, int32_t chunks, int32_t nb, int32_t pairs,
                  int32_t num_sms, int32_t out[6]);

/* Human-readable name of a status. */
const char *q4_status_str(q4_status s);

#ifdef __cplusplus
}
#endif

#endif /* Q4GEMV_H */
