// nvfp4_quant_col_approx.cu -- columnwise and 2D kernels with the fast-math
// element quotient y * RN(1/d) (NVFP4_FAST_MATH), in their own translation
// unit so that both forms compile in parallel.
#include "nvfp4_quant_col.cuh"

namespace nvfp4 {

cudaError_t launch_quant_col_approx(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return quant_col_launch<true>(a, fp32, mode, rht, s);
}

cudaError_t launch_quant_2d_approx(const QArgs &a, bool fp32, cudaStream_t s) {
    return quant_2d_launch<true>(a, fp32, s);
}

}  // namespace nvfp4
