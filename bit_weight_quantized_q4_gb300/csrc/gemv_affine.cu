// gemv_affine.cu -- affine-Q4 instantiations of the dequant-in-GEMV kernel.
#include "gemv_launch.cuh"

namespace q4 {
int launch_gemv_affine(const GemvParams &p, const Plan &plan, void *stream) {
    return launch_gemv_fmt<1>(p, plan, (cudaStream_t)stream);
}
int launch_step_affine(const StepParams &p, int ctas, size_t smem, void *stream) {
    return launch_step_fmt<1>(p, ctas, smem, (cudaStream_t)stream);
}
int step_occupancy_affine(int nb, size_t smem, bool attn) { return step_occupancy_fmt<1>(nb, smem, attn); }
}  // namespace q4
