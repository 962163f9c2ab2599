// gemv_affine.cu -- affine-Q4 instantiations of the dequant-in-GEMV kernel.
#include "gemv_launch.cuh"

namespace q4 {
int launch_gemv_affine(const GemvParams &p, const Plan &plan, void *stream) {
    return launch_gemv_fmt<1>(p, plan, (cudaStream_t)stream);
}
}  // namespace q4
