// gemv_q4_k.cu -- Q4_K instantiations of the dequant-in-GEMV kernel.
#include "gemv_launch.cuh"

namespace q4 {
int launch_gemv_q4_k(const GemvParams &p, const Plan &plan, void *stream) {
    return launch_gemv_fmt<3>(p, plan, (cudaStream_t)stream);
}
int launch_step_q4_k(const StepParams &p, int ctas, size_t smem, void *stream) {
    return launch_step_fmt<3>(p, ctas, smem, (cudaStream_t)stream);
}
int step_occupancy_q4_k(int nb, size_t smem, bool attn) { return step_occupancy_fmt<3>(nb, smem, attn); }
}  // namespace q4
