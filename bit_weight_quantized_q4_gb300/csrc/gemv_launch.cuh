// gemv_launch.cuh -- host launchers for the dequant-in-GEMV kernels: pick the
// batch class from nb, raise the dynamic shared-memory limit once per device
// and kernel, and launch with programmatic dependent launch (plus a cluster
// when K is split, or cooperatively for the decode step).
#pragma once
#include <cuda_runtime.h>

#include "gemv_kernel.cuh"

namespace q4 {

template <typename Kern>
static bool raise_smem(Kern kern, size_t smem, size_t (&set)[64]) {
    int devid = 0;
    if (cudaGetDevice(&devid) != cudaSuccess) return false;
    if (devid < 64 && smem > set[devid]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return false;
        set[devid] = smem;
    } else if (devid >= 64) {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess;
    }
    return true;
}

template <int FMT, int CLS>
static int launch_cls(const GemvParams &p, const Plan &plan, cudaStream_t stream) {
    auto kern = dev::q4gemv_engine_kernel<FMT, CLS>;
    static size_t smem_set[64] = {0};
    if (!raise_smem(kern, plan.smem, smem_set)) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.ctas, 1, 1);
    cfg.blockDim = dim3(cls_warps(CLS) * 32, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (plan.S > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = (unsigned)plan.S;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? 0 : -1;
}

template <int FMT>
static int launch_gemv_fmt(const GemvParams &p, const Plan &plan, cudaStream_t stream) {
    switch (cls_of(p.nb)) {
        case 0: return launch_cls<FMT, 0>(p, plan, stream);
        case 1: return launch_cls<FMT, 1>(p, plan, stream);
        case 2: return launch_cls<FMT, 2>(p, plan, stream);
        default: return launch_cls<FMT, 3>(p, plan, stream);
    }
}

template <int FMT, int CLS, bool ATT>
static int launch_step_cls(const StepParams &p, int ctas, size_t smem, cudaStream_t stream) {
    auto kern = dev::q4gemv_step_kernel<FMT, CLS, ATT>;
    static size_t smem_set[64] = {0};
    if (!raise_smem(kern, smem, smem_set)) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(cls_warps(CLS) * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeCooperative;
    attrs[0].val.cooperative = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? 0 : -1;
}

template <int FMT>
static int launch_step_fmt(const StepParams &p, int ctas, size_t smem, cudaStream_t stream) {
    if (p.attn) return launch_step_cls<FMT, 0, true>(p, ctas, smem, stream);  // nb = 1 (the host checks)
    switch (cls_of(p.nb)) {
        case 0: return launch_step_cls<FMT, 0, false>(p, ctas, smem, stream);
        case 1: return launch_step_cls<FMT, 1, false>(p, ctas, smem, stream);
        case 2: return launch_step_cls<FMT, 2, false>(p, ctas, smem, stream);
        default: return launch_step_cls<FMT, 3, false>(p, ctas, smem, stream);
    }
}

template <int FMT, int CLS, bool ATT>
static int step_occupancy_cls(size_t smem) {
    auto kern = dev::q4gemv_step_kernel<FMT, CLS, ATT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, cls_warps(CLS) * 32, smem) != cudaSuccess)
        return 0;
    return blocks;
}

template <int FMT>
static int step_occupancy_fmt(int nb, size_t smem, bool attn) {
    if (attn) return step_occupancy_cls<FMT, 0, true>(smem);
    switch (cls_of(nb)) {
        case 0: return step_occupancy_cls<FMT, 0, false>(smem);
        case 1: return step_occupancy_cls<FMT, 1, false>(smem);
        case 2: return step_occupancy_cls<FMT, 2, false>(smem);
        default: return step_occupancy_cls<FMT, 3, false>(smem);
    }
}

}  // namespace q4
