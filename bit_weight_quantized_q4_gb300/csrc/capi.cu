// capi.cu -- the C entry points of libq4gemv: argument validation, the launch
// plan, and the kernel launches.  Every check happens before anything is
// enqueued; on any error nothing is launched.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/q4gemv.h"
#include "q4_internal.h"

namespace q4 {
int launch_argmax_fold(const float *am_val, const int *am_idx, int groups, int nb, int32_t *idx,
                       float *val, void *stream);
int launch_group_sums(const float *x, int nb, int k, float *gsum, void *stream);
int launch_pack_half(const float *x, int nb, int k, uint16_t *xe, uint16_t *xo, float *gsum, void *stream);
}  // namespace q4

namespace {

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool shape_ok(int32_t n, int32_t k) {
    return n >= 1 && k >= 32 && k % 32 == 0 && k <= 65536 && n <= (1 << 24);
}

inline bool fmt_known(int32_t fmt) {
    return fmt == Q4_FMT_Q4_0 || fmt == Q4_FMT_AFFINE || fmt == Q4_FMT_Q8_0 || fmt == Q4_FMT_Q4_K || fmt == Q4_FMT_Q1;
}

q4_status check_weight(const q4_weight *W) {
    if (!W || !W->dev) return Q4_ERR_NULL;
    if (!fmt_known(W->fmt)) return Q4_ERR_UNSUPPORTED;
    if (!shape_ok(W->n, W->k)) return Q4_ERR_SHAPE;
    const size_t need = q4_packed_bytes(W->fmt, W->n, W->k);  // 0: k not whole superblocks (Q4_K)
    if (need == 0 || W->bytes < need) return Q4_ERR_SHAPE;
    if (!aligned16(W->dev)) return Q4_ERR_ALIGN;
    return Q4_OK;
}

q4_status check_act(const void *p) {
    if (!p) return Q4_ERR_NULL;
    if (!aligned16(p)) return Q4_ERR_ALIGN;
    return Q4_OK;
}

int num_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return sms;
}

#define Q4_TRY(expr)                      \
    do {                                  \
        q4_status _s = (expr);            \
        if (_s != Q4_OK) return _s;       \
    } while (0)

q4::GemvParams base_params(const q4_weight *W0, const q4_weight *W1, int mode, const float *x,
                           const float *gamma, float eps, int nb) {
    q4::GemvParams p;
    memset(&p, 0, sizeof(p));
    p.w[0] = (const uint8_t *)W0->dev;
    p.n[0] = W0->n;
    p.tiles[0] = (int)q4::tiles_of(W0->n);
    p.nmat = 1;
    if (W1) {
        p.w[1] = (const uint8_t *)W1->dev;
        p.n[1] = W1->n;
        p.tiles[1] = (int)q4::tiles_of(W1->n);
        p.nmat = 2;
    }
    p.mode = mode;
    p.T = mode == q4::MODE_SINGLE ? p.tiles[0]
          : mode == q4::MODE_CONCAT ? p.tiles[0] + p.tiles[1]
                                    : 2 * p.tiles[0];
    p.K = W0->k;
    p.C = (int)q4::chunks_of(W0->k);
    p.nb = nb;
    p.x = x;
    p.gamma = gamma;
    p.eps = eps;
    return p;
}

// Bounds of the kernels' waits and the extra counts a wait expects, applied
// to every launch (q4_debug_wait_limits changes them to test the give-up
// path; the defaults are about a second and nothing extra).
long long g_barrier_polls = q4::kBarrierSpins;
int g_barrier_extra = 0;
long long g_wait_cycles = q4::kWaitCycles;
int g_extra_tx = 0;

// The per-call kernels' error word: set (never cleared) by a kernel whose
// bounded wait for its weight copies gave up; q4_device_check reads and
// clears it.  One word per device, its address resolved once per device.
constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
int *g_err_ptr[kMaxDevices] = {};

}  // namespace

static __device__ int q4_kernel_error_word;

namespace {

q4_status kernel_err_ptr(int **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return Q4_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_err_mu);
    if (g_err_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, q4_kernel_error_word) != cudaSuccess || p == nullptr) return Q4_ERR_CUDA;
        g_err_ptr[dev] = (int *)p;
    }
    *out = g_err_ptr[dev];
    return Q4_OK;
}

// The launch plan of job p on this device.
q4_status plan_of(const q4::GemvParams &p, int fmt, q4::Plan *plan) {
    const int sms = num_sms();
    if (sms <= 0) return Q4_ERR_CUDA;
    *plan = q4::make_plan(fmt, p.T, p.C, p.nb, p.mode == q4::MODE_PAIRS, sms);
    if (plan->smem > q4::kSmemMax) return Q4_ERR_UNSUPPORTED;  // nb * k too large to stage
    return Q4_OK;
}

// Launch job p with `plan` (from plan_of on the same job): the caller sizes
// any per-group buffer from the plan that is launched.
q4_status launch_planned(const q4::GemvParams &p, int fmt, const q4::Plan &plan, cudaStream_t stream) {
    q4::GemvParams pp = p;
    Q4_TRY(kernel_err_ptr(&pp.err));
    pp.wait_cycles = g_wait_cycles;
    pp.extra_tx = g_extra_tx;
    pp.TG = plan.TG;
    pp.SW = plan.SW;
    pp.upt = plan.upt;
    pp.S = plan.S;
    pp.Cs = plan.Cs;
    pp.groups = plan.groups;
    cudaGetLastError();  // clear a stale error so the check below is ours
    int rc = fmt == Q4_FMT_Q4_0     ? q4::launch_gemv_q4_0(pp, plan, stream)
             : fmt == Q4_FMT_AFFINE ? q4::launch_gemv_affine(pp, plan, stream)
             : fmt == Q4_FMT_Q8_0   ? q4::launch_gemv_q8_0(pp, plan, stream)
             : fmt == Q4_FMT_Q4_K   ? q4::launch_gemv_q4_k(pp, plan, stream)
                                    : q4::launch_gemv_q1(pp, plan, stream);
    if (rc != 0 || cudaGetLastError() != cudaSuccess) return Q4_ERR_CUDA;
    return Q4_OK;
}

q4_status run(const q4::GemvParams &p, int fmt, cudaStream_t stream) {
    q4::Plan plan;
    Q4_TRY(plan_of(p, fmt, &plan));
    return launch_planned(p, fmt, plan, stream);
}

inline bool nb_ok(int32_t nb) { return nb >= 1 && nb <= q4::kMaxNb; }

}  // namespace

extern "C" {

const char *q4_status_str(q4_status s) {
    switch (s) {
        case Q4_OK: return "Q4_OK";
        case Q4_ERR_NULL: return "Q4_ERR_NULL: a required pointer is NULL";
        case Q4_ERR_SHAPE: return "Q4_ERR_SHAPE: shape or byte count out of range";
        case Q4_ERR_ALIGN: return "Q4_ERR_ALIGN: device pointer not 16-byte aligned";
        case Q4_ERR_UNSUPPORTED: return "Q4_ERR_UNSUPPORTED: nb, format or combination not supported";
        case Q4_ERR_WORKSPACE: return "Q4_ERR_WORKSPACE: workspace missing or too small";
        case Q4_ERR_CUDA: return "Q4_ERR_CUDA: a CUDA runtime call failed";
    }
    return "unknown q4_status";
}

q4_status q4_plan(int32_t fmt, int32_t tiles, int32_t chunks, int32_t nb, int32_t pairs, int32_t sms,
                  int32_t out[6]) {
    if (!out) return Q4_ERR_NULL;
    if (!fmt_known(fmt)) return Q4_ERR_UNSUPPORTED;
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    if (tiles < 1 || chunks < 1 || sms < 1 || (pairs && (tiles & 1))) return Q4_ERR_SHAPE;
    q4::Plan p = q4::make_plan(fmt, tiles, chunks, nb, pairs != 0, sms);
    out[0] = p.TG;
    out[1] = p.S;
    out[2] = p.Cs;
    out[3] = p.groups;
    out[4] = p.ctas;
    out[5] = (int32_t)p.smem;
    return Q4_OK;
}

q4_status q4_group_sums(const float *x, int32_t nb, int32_t k, float *gsum, cudaStream_t stream) {
    Q4_TRY(check_act(x));
    Q4_TRY(check_act(gsum));
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    if (!shape_ok(1, k)) return Q4_ERR_SHAPE;
    cudaGetLastError();
    if (q4::launch_group_sums(x, nb, k, gsum, stream) != 0 || cudaGetLastError() != cudaSuccess)
        return Q4_ERR_CUDA;
    return Q4_OK;
}

q4_status q4_gemv(const q4_weight *W, const float *x, const float *gsum, int32_t nb, float *y,
                  cudaStream_t stream) {
    Q4_TRY(check_weight(W));
    Q4_TRY(check_act(x));
    Q4_TRY(check_act(y));
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    if (gsum && !aligned16(gsum)) return Q4_ERR_ALIGN;
    q4::GemvParams p = base_params(W, nullptr, q4::MODE_SINGLE, x, nullptr, 0.f, nb);
    p.gsum = q4::has_min(W->fmt) ? gsum : nullptr;
    p.epi = q4::EPI_STORE;
    p.out[0] = y;
    return run(p, W->fmt, stream);
}

q4_status q4_pack_half(const float *x, int32_t nb, int32_t k, uint16_t *x_even, uint16_t *x_odd, float *gsum,
                       cudaStream_t stream) {
    Q4_TRY(check_act(x));
    Q4_TRY(check_act(x_even));
    Q4_TRY(check_act(x_odd));
    if (gsum && !aligned16(gsum)) return Q4_ERR_ALIGN;
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    if (!shape_ok(1, k)) return Q4_ERR_SHAPE;
    cudaGetLastError();
    if (q4::launch_pack_half(x, nb, k, x_even, x_odd, gsum, stream) != 0 || cudaGetLastError() != cudaSuccess)
        return Q4_ERR_CUDA;
    return Q4_OK;
}

q4_status q4_gemv_half(const q4_weight *W, const uint16_t *x_even, const uint16_t *x_odd, const float *gsum,
                       int32_t nb, float *y, cudaStream_t stream) {
    Q4_TRY(check_weight(W));
    Q4_TRY(check_act(x_even));
    Q4_TRY(check_act(x_odd));
    Q4_TRY(check_act(y));
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    if (gsum && !aligned16(gsum)) return Q4_ERR_ALIGN;
    q4::GemvParams p = base_params(W, nullptr, q4::MODE_SINGLE, nullptr, nullptr, 0.f, nb);
    p.xe = x_even;
    p.xo = x_odd;
    p.gsum = q4::has_min(W->fmt) ? gsum : nullptr;
    p.epi = q4::EPI_STORE;
    p.out[0] = y;
    return run(p, W->fmt, stream);
}

q4_status q4_nrm_gemv(const q4_weight *W, const float *x, const float *gamma, float eps, int32_t nb,
                      float *y, cudaStream_t stream) {
    Q4_TRY(check_weight(W));
    Q4_TRY(check_act(x));
    Q4_TRY(check_act(gamma));
    Q4_TRY(check_act(y));
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    q4::GemvParams p = base_params(W, nullptr, q4::MODE_SINGLE, x, gamma, eps, nb);
    p.epi = q4::EPI_STORE;
    p.out[0] = y;
    return run(p, W->fmt, stream);
}

q4_status q4_dual_gemv(const q4_weight *Wa, const q4_weight *Wb, const float *x, const float *gamma,
                       float eps, int32_t nb, float *ya, float *yb, cudaStream_t stream) {
    Q4_TRY(check_weight(Wa));
    Q4_TRY(check_weight(Wb));
    Q4_TRY(check_act(x));
    Q4_TRY(check_act(ya));
    Q4_TRY(check_act(yb));
    if (gamma && !aligned16(gamma)) return Q4_ERR_ALIGN;
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    if (Wa->fmt != Wb->fmt) return Q4_ERR_UNSUPPORTED;
    if (Wa->k != Wb->k) return Q4_ERR_SHAPE;
    q4::GemvParams p = base_params(Wa, Wb, q4::MODE_CONCAT, x, gamma, eps, nb);
    p.epi = q4::EPI_STORE;
    p.out[0] = ya;
    p.out[1] = yb;
    return run(p, Wa->fmt, stream);
}

q4_status q4_gus_nrm(const q4_weight *Wg, const q4_weight *Wu, const float *x, const float *gamma,
                     float eps, int32_t nb, float *h, cudaStream_t stream) {
    Q4_TRY(check_weight(Wg));
    Q4_TRY(check_weight(Wu));
    Q4_TRY(check_act(x));
    Q4_TRY(check_act(gamma));
    Q4_TRY(check_act(h));
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    if (Wg->fmt != Wu->fmt) return Q4_ERR_UNSUPPORTED;
    if (Wg->k != Wu->k || Wg->n != Wu->n) return Q4_ERR_SHAPE;
    q4::GemvParams p = base_params(Wg, Wu, q4::MODE_PAIRS, x, gamma, eps, nb);
    p.epi = q4::EPI_SWIGLU;
    p.out[0] = h;
    return run(p, Wg->fmt, stream);
}

q4_status q4_res_gemv(const q4_weight *W, const float *x, const float *r_in, int32_t nb, float *y,
                      cudaStream_t stream) {
    Q4_TRY(check_weight(W));
    Q4_TRY(check_act(x));
    Q4_TRY(check_act(r_in));
    Q4_TRY(check_act(y));
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    q4::GemvParams p = base_params(W, nullptr, q4::MODE_SINGLE, x, nullptr, 0.f, nb);
    p.epi = q4::EPI_RESIDUAL;
    p.out[0] = y;
    p.res = r_in;
    return run(p, W->fmt, stream);
}

size_t q4_argmax_workspace_bytes(int32_t n, int32_t nb) {
    if (n < 1 || !nb_ok(nb)) return 0;
    // one (value, index) pair per group and activation row; a group has at
    // least one tile, so the tile count bounds the groups of any plan
    const size_t groups = (size_t)q4::tiles_of(n);
    return groups * (size_t)nb * 8u + 16u;
}

q4_status q4_argmax(const q4_weight *W, const float *x, const float *gamma, float eps, int32_t nb,
                    int32_t *idx, float *val, float *logits, void *workspace, size_t ws_bytes,
                    cudaStream_t stream) {
    Q4_TRY(check_weight(W));
    Q4_TRY(check_act(x));
    if (!idx) return Q4_ERR_NULL;
    if (!aligned16(idx) || (val && !aligned16(val)) || (logits && !aligned16(logits)) ||
        (gamma && !aligned16(gamma)))
        return Q4_ERR_ALIGN;
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    if (!workspace) return Q4_ERR_WORKSPACE;
    if (!aligned16(workspace)) return Q4_ERR_ALIGN;
    if (ws_bytes < q4_argmax_workspace_bytes(W->n, nb)) return Q4_ERR_WORKSPACE;
    q4::GemvParams p = base_params(W, nullptr, q4::MODE_SINGLE, x, gamma, eps, nb);
    p.epi = q4::EPI_ARGMAX;
    p.out[0] = logits;
    const size_t groups_max = (size_t)q4::tiles_of(W->n);
    p.am_val = (float *)workspace;
    p.am_idx = (int *)((uint8_t *)workspace + ((groups_max * nb * 4 + 15) & ~(size_t)15));
    q4::Plan plan;
    Q4_TRY(plan_of(p, W->fmt, &plan));
    Q4_TRY(launch_planned(p, W->fmt, plan, stream));
    // pass 2 folds exactly the groups of the plan that was launched
    cudaGetLastError();
    if (q4::launch_argmax_fold(p.am_val, p.am_idx, plan.groups, nb, idx, val, stream) != 0 ||
        cudaGetLastError() != cudaSuccess)
        return Q4_ERR_CUDA;
    return Q4_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free greedy argmax.
//
// q4_argmax needs a caller-provided workspace for its pass-1 (max, index)
// pairs.  Some callers cannot provide one: a plug-in whose host application
// owns all device memory and hands out no allocator, or a decode loop that
// must not touch the allocator once it is running (a cudaMalloc there can
// synchronise the device and stall a latency-critical step).  For them
// q4_argmax_noalloc keeps those pairs in the fixed array below, which is
// compiled into the library: every GPU that loads the library holds these
// 128 KiB until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = 128u * 1024u;
constexpr int kNoAllocMaxDevices = 64;

}  // namespace

static __device__ __align__(256) unsigned char q4_noalloc_argmax_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's
// name in host code is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
q4_status noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return Q4_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, q4_noalloc_argmax_scratch) != cudaSuccess || p == nullptr)
            return Q4_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return Q4_OK;
}

}  // namespace

extern "C" q4_status q4_argmax_noalloc(const q4_weight *W, const float *x, const float *gamma, float eps,
                                       int32_t nb, int32_t *idx, float *val, float *logits,
                                       cudaStream_t stream) {
    Q4_TRY(check_weight(W));
    Q4_TRY(check_act(x));
    if (!idx) return Q4_ERR_NULL;
    if (!aligned16(idx) || (val && !aligned16(val)) || (logits && !aligned16(logits)) ||
        (gamma && !aligned16(gamma)))
        return Q4_ERR_ALIGN;
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    q4::GemvParams p = base_params(W, nullptr, q4::MODE_SINGLE, x, gamma, eps, nb);
    p.epi = q4::EPI_ARGMAX;
    p.out[0] = logits;
    // The pairs this call needs: one per (thread-block group, activation
    // row) of the plan below, which is the plan that is launched.
    q4::Plan plan;
    Q4_TRY(plan_of(p, W->fmt, &plan));
    const size_t val_bytes = ((size_t)plan.groups * nb * 4 + 15) & ~(size_t)15;
    if (val_bytes + (size_t)plan.groups * nb * 4 > kNoAllocScratchBytes) return Q4_ERR_WORKSPACE;
    void *scratch = nullptr;
    Q4_TRY(noalloc_scratch(&scratch));
    p.am_val = (float *)scratch;
    p.am_idx = (int *)((unsigned char *)scratch + val_bytes);
    Q4_TRY(launch_planned(p, W->fmt, plan, stream));
    cudaGetLastError();
    if (q4::launch_argmax_fold(p.am_val, p.am_idx, plan.groups, nb, idx, val, stream) != 0 ||
        cudaGetLastError() != cudaSuccess)
        return Q4_ERR_CUDA;
    return Q4_OK;
}

// ---------------------------------------------------------------------------
// The whole synthetic decode step as one persistent kernel.
namespace {

constexpr int kStepMaxGroups = 1024;  // bound on the CTAs of a step (argmax pairs)

q4_status check_layer_shapes(const q4_decode_layer &L, int fmt, int hidden, int inter, bool need_attn) {
    const q4_weight *ws[7] = {&L.Wq, &L.Wk, &L.Wv, &L.Wo, &L.Wg, &L.Wu, &L.Wd};
    for (const q4_weight *w : ws) {
        Q4_TRY(check_weight(w));
        if (w->fmt != fmt) return Q4_ERR_UNSUPPORTED;
    }
    if (L.Wq.k != hidden || L.Wk.k != hidden || L.Wv.k != hidden || L.Wg.k != hidden || L.Wu.k != hidden)
        return Q4_ERR_SHAPE;
    if (L.Wo.n != hidden || L.Wd.n != hidden || L.Wg.n != inter || L.Wu.n != inter || L.Wd.k != inter)
        return Q4_ERR_SHAPE;
    if (!L.gamma_in || !L.gamma_post || (need_attn && !L.attn)) return Q4_ERR_NULL;
    if (!aligned16(L.gamma_in) || !aligned16(L.gamma_post) || (need_attn && !aligned16(L.attn))) return Q4_ERR_ALIGN;
    return Q4_OK;
}

q4::GemvParams step_job(int G, int nb, int *err) {
    q4::GemvParams p;
    memset(&p, 0, sizeof(p));
    p.err = err;
    p.wait_cycles = g_wait_cycles;
    p.extra_tx = g_extra_tx;
    p.nb = nb;
    p.S = 1;
    p.groups = G;
    return p;
}

void add_mat(q4::GemvParams &p, const q4_weight &W, float *out) {
    const int i = p.nmat++;
    p.w[i] = (const uint8_t *)W.dev;
    p.n[i] = W.n;
    p.tiles[i] = (int)q4::tiles_of(W.n);
    p.out[i] = out;
    p.K = W.k;
    p.C = (int)q4::chunks_of(W.k);
    p.Cs = p.C;
}

void finish_job(q4::GemvParams &p, int &TGmax, int &Kmax, int &SWmax) {
    int T = 0;
    for (int i = 0; i < p.nmat; ++i) T += p.tiles[i];
    if (p.mode == q4::MODE_PAIRS) T = 2 * p.tiles[0];
    p.T = T;
    const int P = q4::units_of(T, p.mode == q4::MODE_PAIRS, p.groups, p.upt);
    if (p.groups > P) p.groups = P;  // never more groups than units
    const int per = (P + p.groups - 1) / p.groups, per_lo = P / p.groups;
    p.TG = p.upt * per < T ? p.upt * per : T;
    p.SW = q4::slots_per_warp(per, per_lo, p.C, p.C, q4::cls_warps(q4::cls_of(p.nb)), p.upt);
    if (p.TG > TGmax) TGmax = p.TG;
    if (p.SW > SWmax) SWmax = p.SW;
    if (p.K > Kmax) Kmax = p.K;
}

// The attention form's workspace: the 16-byte header, the kv heads' split
// tickets (64 bytes: up to 16 kv heads), the argmax pairs, then the splits'
// partial outputs, maxima and sums for up to kStepMaxGroups / kv_heads splits.
constexpr size_t kAttnTicketOff = 16, kAttnPairsOff = 80;
constexpr int kStepAttnMaxKvHeads = 16;
bool step_attn_geometry_ok(int heads, int kv_heads, int head_dim) {
    return head_dim == q4::kStepAttnD && kv_heads >= 1 && kv_heads <= kStepAttnMaxKvHeads &&
           heads == q4::kStepAttnG * kv_heads;
}
size_t step_attn_partials_off() { return kAttnPairsOff + (size_t)8 * kStepMaxGroups; }

}  // namespace

extern "C" size_t q4_decode_workspace_bytes(int32_t nb) {
    if (!nb_ok(nb)) return 0;
    return 16 + (size_t)8 * nb * kStepMaxGroups;
}

extern "C" size_t q4_decode_attn_workspace_bytes(int32_t heads, int32_t kv_heads, int32_t head_dim) {
    if (!step_attn_geometry_ok(heads, kv_heads, head_dim)) return 0;
    const size_t splits = (size_t)kStepMaxGroups / kv_heads;
    return step_attn_partials_off() + splits * heads * (head_dim + 2) * sizeof(float);
}

namespace {
q4_status run_step(const q4_decode_layer *layers, int32_t n_layers, const q4_step_attention *att,
                   const q4_weight *Wlogits, const float *gamma_final, float eps, int32_t nb, const float *x_in,
                   float *hid, float *q, float *k, float *v, float *h, int32_t *idx, float *val, void *workspace,
                   size_t ws_bytes, cudaStream_t stream);
}  // namespace

extern "C" q4_status q4_decode_step_attn(const q4_decode_layer *layers, int32_t n_layers,
                                         const q4_step_attention *att, const q4_weight *Wlogits,
                                         const float *gamma_final, float eps, const float *x_in, float *hid,
                                         float *q, float *k, float *v, float *h, int32_t *idx, float *val,
                                         void *workspace, size_t ws_bytes, cudaStream_t stream) {
    if (!att) return Q4_ERR_NULL;
    return run_step(layers, n_layers, att, Wlogits, gamma_final, eps, 1, x_in, hid, q, k, v, h, idx, val, workspace,
                    ws_bytes, stream);
}

extern "C" q4_status q4_decode_step(const q4_decode_layer *layers, int32_t n_layers, const q4_weight *Wlogits,
                                    const float *gamma_final, float eps, int32_t nb, const float *x_in,
                                    float *hid, float *q, float *k, float *v, float *h, int32_t *idx,
                                    float *val, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    return run_step(layers, n_layers, nullptr, Wlogits, gamma_final, eps, nb, x_in, hid, q, k, v, h, idx, val,
                    workspace, ws_bytes, stream);
}

namespace {
// The step's jobs and launch; with `att` each layer also runs its decode
// attention as a job between the q/k/v and the o job (nb = 1).
q4_status run_step(const q4_decode_layer *layers, int32_t n_layers, const q4_step_attention *att,
                   const q4_weight *Wlogits, const float *gamma_final, float eps, int32_t nb, const float *x_in,
                   float *hid, float *q, float *k, float *v, float *h, int32_t *idx, float *val, void *workspace,
                   size_t ws_bytes, cudaStream_t stream) {
    if (!layers || !Wlogits) return Q4_ERR_NULL;
    const int jobs_per_layer = att ? 5 : 4;
    if (n_layers < 1 || n_layers > q4::kMaxStepLayers || jobs_per_layer * n_layers + 1 > q4::kMaxStepJobs)
        return Q4_ERR_UNSUPPORTED;
    if (!nb_ok(nb)) return Q4_ERR_UNSUPPORTED;
    Q4_TRY(check_weight(Wlogits));
    const int fmt = Wlogits->fmt;
    const int hidden = layers[0].Wo.n, inter = layers[0].Wg.n;
    for (int l = 0; l < n_layers; ++l) {
        Q4_TRY(check_layer_shapes(layers[l], fmt, hidden, inter, att == nullptr));
        if (layers[l].Wq.n != layers[0].Wq.n || layers[l].Wk.n != layers[0].Wk.n ||
            layers[l].Wv.n != layers[0].Wv.n || layers[l].Wo.k != layers[0].Wo.k)
            return Q4_ERR_SHAPE;
    }
    if (layers[0].Wo.k != hidden) return Q4_ERR_SHAPE;  // the attention output has width hidden
    if (Wlogits->k != hidden) return Q4_ERR_SHAPE;
    Q4_TRY(check_act(gamma_final));
    Q4_TRY(check_act(x_in));
    Q4_TRY(check_act(hid));
    Q4_TRY(check_act(q));
    Q4_TRY(check_act(k));
    Q4_TRY(check_act(v));
    Q4_TRY(check_act(h));
    if (!idx) return Q4_ERR_NULL;
    if (!aligned16(idx) || (val && !aligned16(val))) return Q4_ERR_ALIGN;
    if (att) {  // the attention form: its own arguments and geometry
        if (!step_attn_geometry_ok(att->heads, att->kv_heads, att->head_dim)) return Q4_ERR_UNSUPPORTED;
        const int D = att->head_dim;
        if (att->heads * D != hidden || att->heads * D != layers[0].Wq.n || att->kv_heads * D != layers[0].Wk.n ||
            att->kv_heads * D != layers[0].Wv.n)
            return Q4_ERR_SHAPE;
        if (att->max_seq < 1 || att->max_seq > (1 << 24) || att->position < 0 || att->position >= att->max_seq ||
            att->window < 0)
            return Q4_ERR_SHAPE;
        if (!att->k_caches || !att->v_caches) return Q4_ERR_NULL;
        for (int l = 0; l < n_layers; ++l) {
            Q4_TRY(check_act(att->k_caches[l]));
            Q4_TRY(check_act(att->v_caches[l]));
        }
        if ((att->rope_cos == nullptr) != (att->rope_sin == nullptr)) return Q4_ERR_NULL;
        if (att->rope_cos) {
            Q4_TRY(check_act(att->rope_cos));
            Q4_TRY(check_act(att->rope_sin));
        }
        Q4_TRY(check_act(att->out));
    }
    if (!workspace) return Q4_ERR_WORKSPACE;
    if (!aligned16(workspace)) return Q4_ERR_ALIGN;
    if (ws_bytes < (att ? q4_decode_attn_workspace_bytes(att->heads, att->kv_heads, att->head_dim)
                        : q4_decode_workspace_bytes(nb)))
        return Q4_ERR_WORKSPACE;

    const int sms = num_sms();
    if (sms <= 0) return Q4_ERR_CUDA;
    const int G = sms < kStepMaxGroups ? sms : kStepMaxGroups;  // one CTA per SM
    // the attention jobs' split of the positions: cps CTAs per kv head, each
    // Lc positions of [lo, total), nsplit of them in use
    int cps = 0;
    if (att) {
        cps = G / att->kv_heads;
        if (cps < 1) return Q4_ERR_UNSUPPORTED;
    }

    // the step's jobs; the StepParams block travels as the kernel argument
    static thread_local q4::StepParams sp;
    memset(&sp, 0, sizeof(sp));
    unsigned char *wsb = (unsigned char *)workspace;
    sp.counter = (unsigned *)wsb;
    sp.err = (int *)(wsb + 4);
    sp.release = (unsigned *)(wsb + 8);
    sp.idx = idx;
    sp.val = val;
    sp.nb = nb;
    sp.barrier_polls = g_barrier_polls;
    sp.barrier_extra = g_barrier_extra;
    if (att) {
        q4::StepAttn &A = sp.att;
        sp.attn = 1;
        A.q = q;
        A.k_new = k;
        A.v_new = v;
        A.rope_cos = att->rope_cos;
        A.rope_sin = att->rope_sin;
        A.out = att->out;
        const size_t splits = (size_t)kStepMaxGroups / att->kv_heads;
        A.ws_count = (int *)(wsb + kAttnTicketOff);
        A.ws_o = (float *)(wsb + step_attn_partials_off());
        A.ws_m = A.ws_o + splits * att->heads * att->head_dim;
        A.ws_l = A.ws_m + splits * att->heads;
        for (int l = 0; l < n_layers; ++l) {
            A.k_cache[l] = att->k_caches[l];
            A.v_cache[l] = att->v_caches[l];
        }
        A.max_seq = att->max_seq;
        A.position = att->position;
        A.H = att->heads;
        A.Hkv = att->kv_heads;
        A.total = att->position + 1;
        A.lo = (att->window > 0 && A.total > att->window) ? A.total - att->window : 0;
        const int len = A.total - A.lo;
        A.cps = cps;
        A.Lc = (len + cps - 1) / cps;
        A.nsplit = (len + A.Lc - 1) / A.Lc;
        A.scale = att->scale > 0.f ? att->scale : 1.0f / sqrtf((float)att->head_dim);
    }
    int TGmax = 1, Kmax = 0, SWmax = 2;
    int nj = 0;
    for (int l = 0; l < n_layers; ++l) {
        const q4_decode_layer &L = layers[l];
        const float *src = l == 0 ? x_in : hid;
        q4::GemvParams a = step_job(G, nb, sp.err);  // RMSNorm + q, k, v (one input, three weights)
        a.mode = q4::MODE_CONCAT;
        add_mat(a, L.Wq, q);
        add_mat(a, L.Wk, k);
        add_mat(a, L.Wv, v);
        a.x = src;
        a.gamma = L.gamma_in;
        a.eps = eps;
        a.epi = q4::EPI_STORE;
        finish_job(a, TGmax, Kmax, SWmax);
        sp.jobs[nj++] = a;
        if (att) {  // the layer's decode attention: no weights, no tiles
            q4::GemvParams at = step_job(G, nb, sp.err);
            at.epi = q4::EPI_ATTN;
            at.layer = l;
            at.groups = 0;
            at.upt = 2;
            at.K = (int)q4::kChunkK;
            at.C = at.Cs = 1;
            sp.jobs[nj++] = at;
        }
        q4::GemvParams o = step_job(G, nb, sp.err);  // o projection of the attention output + residual
        o.mode = q4::MODE_SINGLE;
        add_mat(o, L.Wo, hid);
        o.x = att ? att->out : L.attn;
        o.res = src;
        o.epi = q4::EPI_RESIDUAL;
        finish_job(o, TGmax, Kmax, SWmax);
        sp.jobs[nj++] = o;
        q4::GemvParams gu = step_job(G, nb, sp.err);  // RMSNorm + gate/up + SwiGLU
        gu.mode = q4::MODE_PAIRS;
        add_mat(gu, L.Wg, h);
        add_mat(gu, L.Wu, nullptr);
        gu.x = hid;
        gu.gamma = L.gamma_post;
        gu.eps = eps;
        gu.epi = q4::EPI_SWIGLU;
        finish_job(gu, TGmax, Kmax, SWmax);
        sp.jobs[nj++] = gu;
        q4::GemvParams d = step_job(G, nb, sp.err);  // down projection + residual, in place
        d.mode = q4::MODE_SINGLE;
        add_mat(d, L.Wd, hid);
        d.x = h;
        d.res = hid;
        d.epi = q4::EPI_RESIDUAL;
        finish_job(d, TGmax, Kmax, SWmax);
        sp.jobs[nj++] = d;
    }
    q4::GemvParams lg = step_job(G, nb, sp.err);  // final RMSNorm + logits + per-group argmax
    lg.mode = q4::MODE_SINGLE;
    add_mat(lg, *Wlogits, nullptr);
    lg.x = hid;
    lg.gamma = gamma_final;
    lg.eps = eps;
    lg.epi = q4::EPI_ARGMAX;
    const size_t pairs = att ? kAttnPairsOff : 16;
    lg.am_val = (float *)(wsb + pairs);
    lg.am_idx = (int *)(wsb + pairs + (size_t)4 * nb * kStepMaxGroups);
    finish_job(lg, TGmax, Kmax, SWmax);
    sp.jobs[nj++] = lg;
    sp.njobs = nj;
    if (att) {
        // the attention job's scratch overlays the activation slice (nb = 1:
        // 512 bytes a 128-column chunk), so that slice is at least that large
        const size_t scratch = q4::step_attn_scratch_bytes(q4::cls_warps(0));
        const int chunks = (int)((scratch + 511) / 512);
        if (Kmax < chunks * (int)q4::kChunkK) Kmax = chunks * (int)q4::kChunkK;
    }
    sp.Kmax = Kmax;
    sp.TGmax = TGmax;
    sp.SWmax = SWmax;
    // every job runs on all G CTAs; a job's groups may be fewer (clipped to
    // its tile units), and the CTAs beyond them skip that job's work

    const size_t smem = q4::step_smem_bytes(fmt, nb, TGmax, Kmax, SWmax, nj);
    if (smem > q4::kSmemMax) return Q4_ERR_UNSUPPORTED;
    const bool an = att != nullptr;
    const int occ = fmt == Q4_FMT_Q4_0     ? q4::step_occupancy_q4_0(nb, smem, an)
                    : fmt == Q4_FMT_AFFINE ? q4::step_occupancy_affine(nb, smem, an)
                    : fmt == Q4_FMT_Q8_0   ? q4::step_occupancy_q8_0(nb, smem, an)
                    : fmt == Q4_FMT_Q4_K   ? q4::step_occupancy_q4_k(nb, smem, an)
                                           : q4::step_occupancy_q1(nb, smem, an);
    if (occ < 1) return Q4_ERR_UNSUPPORTED;
    cudaGetLastError();
    // the barrier counter and error word (and the attention tickets)
    if (cudaMemsetAsync(workspace, 0, att ? kAttnPairsOff : 16, stream) != cudaSuccess) return Q4_ERR_CUDA;
    const int rc = fmt == Q4_FMT_Q4_0     ? q4::launch_step_q4_0(sp, G, smem, stream)
                   : fmt == Q4_FMT_AFFINE ? q4::launch_step_affine(sp, G, smem, stream)
                   : fmt == Q4_FMT_Q8_0   ? q4::launch_step_q8_0(sp, G, smem, stream)
                   : fmt == Q4_FMT_Q4_K   ? q4::launch_step_q4_k(sp, G, smem, stream)
                                          : q4::launch_step_q1(sp, G, smem, stream);
    if (rc != 0 || cudaGetLastError() != cudaSuccess) return Q4_ERR_CUDA;
    return Q4_OK;
}
}  // namespace

extern "C" q4_status q4_decode_check(const void *workspace, cudaStream_t stream) {
    if (!workspace) return Q4_ERR_NULL;
    int err = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return Q4_ERR_CUDA;
    if (cudaMemcpy(&err, (const unsigned char *)workspace + 4, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return Q4_ERR_CUDA;
    return err ? Q4_ERR_CUDA : Q4_OK;
}

// ---------------------------------------------------------------- prefill GEMM

extern "C" size_t q4_gemm_workspace_bytes(int32_t nb, int32_t k) {
    if (nb < 1 || nb > (1 << 20) || !shape_ok(1, k)) return 0;
    // enough for either form (the tensor-memory one takes Q4_0 and Q8_0 from 17 rows)
    const int C = (int)q4::chunks_of(k);
    const size_t a = q4::gemm_image_bytes(nb, C), b = nb >= q4::kGemmTcMinNb ? q4::gemm_tc_image_bytes(nb, C) : 0;
    return a > b ? a : b;
}

extern "C" q4_status q4_gemm(const q4_weight *W, const float *x, int32_t nb, float *y, int32_t accumulate,
                             void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    Q4_TRY(check_weight(W));
    Q4_TRY(check_act(x));
    Q4_TRY(check_act(y));
    if (nb < 1 || nb > (1 << 20)) return Q4_ERR_SHAPE;
    const size_t need = q4_gemm_workspace_bytes(nb, W->k);
    if (!workspace || workspace_bytes < need) return Q4_ERR_WORKSPACE;
    if (!aligned16(workspace)) return Q4_ERR_ALIGN;
    if (q4::gemm_smem_bytes(W->fmt, nb) > q4::kSmemMax) return Q4_ERR_UNSUPPORTED;
    q4::GemmParams p{};
    p.w = (const uint8_t *)W->dev;
    p.x = x;
    p.img = (uint8_t *)workspace;
    p.y = y;
    p.n = W->n;
    p.T = (int)q4::tiles_of(W->n);
    p.C = (int)q4::chunks_of(W->k);
    p.K = W->k;
    p.nb = nb;
    p.accumulate = accumulate != 0;
    Q4_TRY(kernel_err_ptr(&p.err));
    p.wait_cycles = g_wait_cycles;
    p.extra_tx = g_extra_tx;
    cudaGetLastError();
    const bool tc = (W->fmt == Q4_FMT_Q4_0 || W->fmt == Q4_FMT_Q8_0) && nb >= q4::kGemmTcMinNb;
    if ((tc ? q4::launch_gemm_tc(p, W->fmt, stream) : q4::launch_gemm(p, W->fmt, stream)) != 0 ||
        cudaGetLastError() != cudaSuccess)
        return Q4_ERR_CUDA;
    return Q4_OK;
}

// ---------------------------------------------------------------- attention

namespace {
constexpr int kAttnMinChunk = 16;  // positions per split at least (bounds the workspace)
// the per-kv-head split counters at the start of the workspace
inline size_t attn_count_bytes(int32_t H) { return ((size_t)H * sizeof(int) + 15) / 16 * 16; }

bool attn_geometry_ok(int32_t H, int32_t Hkv, int32_t D) {
    if (Hkv < 1 || H < Hkv || H % Hkv != 0 || H > 4096) return false;
    const int G = H / Hkv;
    if (D == 64) return G == 1 || G == 2 || G == 4 || G == 8 || G == 16;
    if (D == 128) return G == 1 || G == 2 || G == 4 || G == 8;
    return false;
}
}  // namespace

extern "C" size_t q4_attn_workspace_bytes(int32_t H, int32_t D, int32_t max_seq) {
    if (H < 1 || max_seq < 1 || (D != 64 && D != 128)) return 0;
    const size_t splits = ((size_t)max_seq + kAttnMinChunk - 1) / kAttnMinChunk;
    return attn_count_bytes(H) + splits * (size_t)H * (size_t)(D + 2) * sizeof(float);
}

extern "C" q4_status q4_attn_decode(const float *q, const float *k_new, const float *v_new, float *k_cache,
                                    float *v_cache, int32_t max_seq, int32_t position, int32_t H, int32_t Hkv,
                                    int32_t D, int32_t window, float scale, const float *rope_cos,
                                    const float *rope_sin, float *out, void *workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
    Q4_TRY(check_act(q));
    Q4_TRY(check_act(k_new));
    Q4_TRY(check_act(v_new));
    Q4_TRY(check_act(k_cache));
    Q4_TRY(check_act(v_cache));
    Q4_TRY(check_act(out));
    if ((rope_cos == nullptr) != (rope_sin == nullptr)) return Q4_ERR_NULL;
    if (rope_cos) {
        Q4_TRY(check_act(rope_cos));
        Q4_TRY(check_act(rope_sin));
    }
    if (!attn_geometry_ok(H, Hkv, D)) return Q4_ERR_UNSUPPORTED;
    if (max_seq < 1 || max_seq > (1 << 24) || position < 0 || position >= max_seq || window < 0)
        return Q4_ERR_SHAPE;
    const int sms = num_sms();
    if (sms <= 0) return Q4_ERR_CUDA;
    q4::AttnParams p{};
    p.q = q;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.rope_cos = rope_cos;
    p.rope_sin = rope_sin;
    p.out = out;
    p.max_seq = max_seq;
    p.position = position;
    p.H = H;
    p.Hkv = Hkv;
    p.D = D;
    p.scale = scale;
    p.total = position + 1;
    p.lo = (window > 0 && p.total > window) ? p.total - window : 0;
    // splits: about one CTA per SM slot over all kv heads, each at least one
    // pipeline stage of positions
    const int len = p.total - p.lo;
    const int G = H / Hkv;
    const int LS = q4::attn_sub_chunk(D);
    const int target = std::max(1, q4::attn_ctas_per_sm(D, G) * sms / Hkv);
    int ns = std::max(1, std::min(std::min(target, q4::attn_max_splits(D, G)), (len + LS - 1) / LS));
    p.Lc = (len + ns - 1) / ns;
    p.nsplit = (len + p.Lc - 1) / p.Lc;
    if (p.nsplit > 1) {
        const size_t need = attn_count_bytes(H) + (size_t)p.nsplit * H * (D + 2) * sizeof(float);
        if (!workspace || workspace_bytes < need) return Q4_ERR_WORKSPACE;
        if (!aligned16(workspace)) return Q4_ERR_ALIGN;
        p.ws_count = (int *)workspace;
        p.ws_o = (float *)((char *)workspace + attn_count_bytes(H));
        p.ws_m = p.ws_o + (size_t)p.nsplit * H * D;
        p.ws_l = p.ws_m + (size_t)p.nsplit * H;
    }
    if (q4::attn_smem_bytes(D, G) > q4::kSmemMax) return Q4_ERR_UNSUPPORTED;
    Q4_TRY(kernel_err_ptr(&p.err));
    p.wait_cycles = g_wait_cycles;
    p.extra_tx = g_extra_tx;
    cudaGetLastError();
    if (q4::launch_attn(p, stream) != 0 || cudaGetLastError() != cudaSuccess) return Q4_ERR_CUDA;
    return Q4_OK;
}

extern "C" q4_status q4_debug_wait_limits(int64_t barrier_polls, int32_t barrier_extra, int64_t copy_wait_cycles,
                                          int32_t copy_extra_bytes) {
    if (barrier_extra < 0 || barrier_extra > 1 || copy_extra_bytes < 0 || copy_extra_bytes > 4096 ||
        copy_extra_bytes % 16 != 0)
        return Q4_ERR_SHAPE;
    g_barrier_polls = barrier_polls > 0 ? (long long)barrier_polls : q4::kBarrierSpins;
    g_barrier_extra = barrier_extra;
    g_wait_cycles = copy_wait_cycles > 0 ? (long long)copy_wait_cycles : q4::kWaitCycles;
    g_extra_tx = copy_extra_bytes;
    return Q4_OK;
}

extern "C" q4_status q4_device_check(cudaStream_t stream) {
    int *dev_err = nullptr;
    Q4_TRY(kernel_err_ptr(&dev_err));
    if (cudaStreamSynchronize(stream) != cudaSuccess) return Q4_ERR_CUDA;
    int err = 0;
    if (cudaMemcpy(&err, dev_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return Q4_ERR_CUDA;
    if (err != 0) {
        const int zero = 0;
        if (cudaMemcpy(dev_err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return Q4_ERR_CUDA;
        return Q4_ERR_CUDA;
    }
    return Q4_OK;
}
