// nvfp4_quant_row.cu -- rowwise launches (exact quotients; the fast-math
// forms are built in nvfp4_quant_row_approx.cu).
#include "nvfp4_quant_row.cuh"

namespace nvfp4 {

cudaError_t launch_quant_row(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return a.fast_math ? launch_quant_row_approx(a, fp32, mode, rht, false, s)
                       : quant_row_launch<false>(a, fp32, mode, rht, false, s);
}

cudaError_t launch_quant_row_fused(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return a.fast_math ? launch_quant_row_fused_approx(a, fp32, mode, rht, s)
                       : quant_row_fused_launch<false>(a, fp32, mode, rht, s);
}

cudaError_t launch_quant_rowscaled(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return a.fast_math ? launch_quant_row_approx(a, fp32, mode, rht, true, s)
                       : quant_row_launch<false>(a, fp32, mode, rht, true, s);
}

cudaError_t launch_quant_grouped(const QArgs &a, bool fp32, int mode, bool rht, bool *padded, cudaStream_t s) {
    return fp32 ? dispatch_row_grouped<float>(a, mode, rht, padded, s)
                : dispatch_row_grouped<bf16_t>(a, mode, rht, padded, s);
}

}  // namespace nvfp4
