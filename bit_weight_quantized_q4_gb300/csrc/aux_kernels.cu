// aux_kernels.cu -- the argmax fold (pass 2), the activation group sums and
// the HalfSet packing.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "q4_internal.h"

namespace q4 {
namespace dev {

// Pass 2 of the greedy argmax (Module gpu, module sampling): one CTA per
// activation row folds the per-group (max, index) pairs of pass 1.  Larger
// value wins, ties go to the lower index; pass 1 already ranked NaN lowest.
__global__ void __launch_bounds__(256) q4gemv_argmax_fold_kernel(const float *am_val, const int *am_idx,
                                                          int groups, int32_t *idx, float *val) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float sv[8];
    __shared__ int si[8];
    const int r = blockIdx.x, tid = threadIdx.x;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = tid; i < groups; i += 256) {
        float v = am_val[(size_t)r * groups + i];
        int j = am_idx[(size_t)r * groups + i];
        if (v > bv || (v == bv && j < bi)) {
            bv = v;
            bi = j;
        }
    }
    for (int off = 16; off > 0; off >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
        }
    }
    if ((tid & 31) == 0) {
        sv[tid >> 5] = bv;
        si[tid >> 5] = bi;
    }
    __syncthreads();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (tid == 0) {
        bv = sv[0];
        bi = si[0];
        for (int w = 1; w < 8; ++w)
            if (sv[w] > bv || (sv[w] == bv && si[w] < bi)) {
                bv = sv[w];
                bi = si[w];
            }
        idx[r] = bi;
        if (val) val[r] = bv;
    }
}

// gsum[r][g] = sum of x[r][32g .. 32g+31] (Module gpu, Struct HalfSet: per-32
// group sums of a row batch).  Eight lanes per group, four columns each,
// added by block8_sum -- the order the GEMV's staging uses for its own affine
// block sums, so either source gives the same bits.
__global__ void __launch_bounds__(256) q4gemv_group_sums_kernel(const float *x, int nb, int k, float *gsum) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int G = k / 32;
    const int total = nb * G;
    const int lane = threadIdx.x & 31;
    const int gi_all = (blockIdx.x * 256 + threadIdx.x) >> 3;  // (row, group) index
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (gi_all < total) {
        const int r = gi_all / G, gi = gi_all - r * G;
        v = *reinterpret_cast<const float4 *>(x + (size_t)r * k + 32 * gi + 4 * (lane & 7));
    }
    const float t = block8_sum(v);
    if (gi_all < total && (lane & 7) == 0) gsum[gi_all] = t;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// HalfSet packing (Module gpu, Struct HalfSet): each activation rounded to
// f16 (nearest, ties to even), the even-indexed elements of a row into
// x_even, the odd-indexed into x_odd, and the per-32 group sums of the f16
// values (as fp32) into gsum, added by block8_sum -- the order the GEMV's
// staging uses, so either source gives the same bits.  Eight lanes per group,
// four columns each.
__global__ void __launch_bounds__(256) q4gemv_pack_half_kernel(const float *x, int nb, int k, uint16_t *xe,
                                                               uint16_t *xo, float *gsum) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int G = k / 32;
    const int total = nb * G;
    const int lane = threadIdx.x & 31;
    const int gi_all = (blockIdx.x * 256 + threadIdx.x) >> 3;  // (row, group) index
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    size_t e0 = 0;
    if (gi_all < total) {
        const int r = gi_all / G, gi = gi_all - r * G;
        const size_t off = (size_t)r * k + 32 * gi + 4 * (lane & 7);
        const float4 a = *reinterpret_cast<const float4 *>(x + off);
        const __half2 ev = __floats2half2_rn(a.x, a.z), od = __floats2half2_rn(a.y, a.w);
        e0 = off >> 1;
        *reinterpret_cast<__half2 *>(xe + e0) = ev;
        *reinterpret_cast<__half2 *>(xo + e0) = od;
        const float2 fe = __half22float2(ev), fo = __half22float2(od);
        v = make_float4(fe.x, fo.x, fe.y, fo.y);
    }
    const float t = block8_sum(v);
    if (gi_all < total && (lane & 7) == 0 && gsum != nullptr) gsum[gi_all] = t;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace dev

static int launch_pdl(const void *func, dim3 grid, dim3 block, void **args, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, func, args) == cudaSuccess ? 0 : -1;
}

int launch_argmax_fold(const float *am_val, const int *am_idx, int groups, int nb, int32_t *idx,
                       float *val, void *stream) {
    void *args[] = {(void *)&am_val, (void *)&am_idx, (void *)&groups, (void *)&idx, (void *)&val};
    return launch_pdl((const void *)dev::q4gemv_argmax_fold_kernel, dim3(nb), dim3(256), args,
                      (cudaStream_t)stream);
}

int launch_pack_half(const float *x, int nb, int k, uint16_t *xe, uint16_t *xo, float *gsum, void *stream) {
    void *args[] = {(void *)&x, (void *)&nb, (void *)&k, (void *)&xe, (void *)&xo, (void *)&gsum};
    const int total = nb * (k / 32);  // 8 threads per group
    return launch_pdl((const void *)dev::q4gemv_pack_half_kernel, dim3((8 * total + 255) / 256), dim3(256), args,
                      (cudaStream_t)stream);
}

int launch_group_sums(const float *x, int nb, int k, float *gsum, void *stream) {
    void *args[] = {(void *)&x, (void *)&nb, (void *)&k, (void *)&gsum};
    const int total = nb * (k / 32);  // 8 threads per group
    return launch_pdl((const void *)dev::q4gemv_group_sums_kernel, dim3((8 * total + 255) / 256), dim3(256), args,
                      (cudaStream_t)stream);
}

}  // namespace q4
