// gemv_launch.cuh -- host launcher for the dequant-in-GEMV kernel: picks the
// n-tile count from nb, raises the dynamic shared-memory limit once per
// device, and launches with programmatic dependent launch (and a cluster
// when K is split).
#pragma once
#include <cuda_runtime.h>

#include "gemv_kernel.cuh"

namespace q4 {

template <int FMT, int NT, bool NB1>
static int launch_nt(const GemvParams &p, const Plan &plan, cudaStream_t stream) {
    auto kern = dev::gemv_kernel<FMT, NT, NB1>;
    int devid = 0;
    if (cudaGetDevice(&devid) != cudaSuccess) return -1;
    static size_t smem_set[64] = {0};
    if (devid < 64 && plan.smem > smem_set[devid]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem) !=
            cudaSuccess)
            return -1;
        smem_set[devid] = plan.smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.ctas, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
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
    if (p.nb == 1) return launch_nt<FMT, 1, true>(p, plan, stream);
    if (p.nb <= 8) return launch_nt<FMT, 1, false>(p, plan, stream);
    return launch_nt<FMT, 2, false>(p, plan, stream);
}

template <int FMT, int NT, bool NB1>
static int launch_step_nt(const StepParams &p, int ctas, size_t smem, cudaStream_t stream) {
    auto kern = dev::decode_kernel<FMT, NT, NB1>;
    int devid = 0;
    if (cudaGetDevice(&devid) != cudaSuccess) return -1;
    static size_t smem_set[64] = {0};
    if (devid < 64 && smem > smem_set[devid]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -1;
        smem_set[devid] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(kStepWarps * 32, 1, 1);
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
    if (p.nb == 1) return launch_step_nt<FMT, 1, true>(p, ctas, smem, stream);
    if (p.nb <= 8) return launch_step_nt<FMT, 1, false>(p, ctas, smem, stream);
    return launch_step_nt<FMT, 2, false>(p, ctas, smem, stream);
}

template <int FMT, int NT, bool NB1>
static int step_occupancy(size_t smem) {
    auto kern = dev::decode_kernel<FMT, NT, NB1>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return 0;
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, kStepWarps * 32, smem) != cudaSuccess)
        return 0;
    return blocks;
}

template <int FMT>
static int step_occupancy_fmt(int nb, size_t smem) {
    if (nb == 1) return step_occupancy<FMT, 1, true>(smem);
    if (nb <= 8) return step_occupancy<FMT, 1, false>(smem);
    return step_occupancy<FMT, 2, false>(smem);
}

}  // namespace q4
