// nvfp4_quant_row_approx.cu -- rowwise kernels with the fast-math element
// quotient y * RN(1/d) (NVFP4_FAST_MATH), in their own translation unit so
// that both forms compile in parallel.
#include "nvfp4_quant_row.cuh"

namespace nvfp4 {

cudaError_t launch_quant_row_approx(const QArgs &a, bool fp32, int mode, bool rht, bool scaled_rows,
                                    cudaStream_t s) {
    return quant_row_launch<true>(a, fp32, mode, rht, scaled_rows, s);
}

cudaError_t launch_quant_row_fused_approx(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return quant_row_fused_launch<true>(a, fp32, mode, rht, s);
}

}  // namespace nvfp4
