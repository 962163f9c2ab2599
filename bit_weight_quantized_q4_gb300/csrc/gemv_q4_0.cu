// gemv_q4_0.cu -- Q4_0 instantiations of the dequant-in-GEMV kernel.
#include "gemv_launch.cuh"

namespace q4 {
int launch_gemv_q4_0(const GemvParams &p, const Plan &plan, void *stream) {
    return launch_gemv_fmt<0>(p, plan, (cudaStream_t)stream);
}
}  // namespace q4
