// nvfp4_quant_col.cu -- columnwise and 2D launches (exact quotients; the
// fast-math forms are built in nvfp4_quant_col_approx.cu).
#include "nvfp4_quant_col.cuh"

namespace nvfp4 {

cudaError_t launch_quant_col(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return a.fast_math ? launch_quant_col_approx(a, fp32, mode, rht, s) : quant_col_launch<false>(a, fp32, mode, rht, s);
}

cudaError_t launch_quant_2d(const QArgs &a, bool fp32, cudaStream_t s) {
    return a.fast_math ? launch_quant_2d_approx(a, fp32, s) : quant_2d_launch<false>(a, fp32, s);
}

}  // namespace nvfp4
