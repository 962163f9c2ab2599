// gemv_q1.cu -- Q1 instantiations of the dequant-in-GEMV kernel.
#include "gemv_launch.cuh"

namespace q4 {
int launch_gemv_q1(const GemvParams &p, const Plan &plan, void *stream) {
    return launch_gemv_fmt<4>(p, plan, (cudaStream_t)stream);
}
int launch_step_q1(const StepParams &p, int ctas, size_t smem, void *stream) {
    return launch_step_fmt<4>(p, ctas, smem, (cudaStream_t)stream);
}
int step_occupancy_q1(int nb, size_t smem, bool attn) { return step_occupancy_fmt<4>(nb, smem, attn); }
}  // namespace q4
