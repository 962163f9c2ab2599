// gemv_q4_0.cu -- Q4_0 instantiations of the dequant-in-GEMV kernel.
#include "gemv_launch.cuh"

namespace q4 {
int launch_gemv_q4_0(const GemvParams &p, const Plan &plan, void *stream) {
    return launch_gemv_fmt<0>(p, plan, (cudaStream_t)stream);
}
int launch_step_q4_0(const StepParams &p, int ctas, size_t smem, void *stream) {
    return launch_step_fmt<0>(p, ctas, smem, (cudaStream_t)stream);
}
int step_occupancy_q4_0(int nb, size_t smem, bool attn) { return step_occupancy_fmt<0>(nb, smem, attn); }
}  // namespace q4
