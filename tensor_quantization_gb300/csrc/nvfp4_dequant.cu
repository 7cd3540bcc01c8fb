// nvfp4_dequant.cu -- NVFP4 decode and swizzle pad fill.
//
// Decode ("[nvfp4 training][rl] Add a CuTe DSL fast-path kernel for
// four-over-six quantize #4852", PR description: nvfp4_dequantize, the
// standard NVFP4 decode): out = value(code) * (Sf * g), each product rounded
// to fp32, then to bf16 (round to nearest even) for a bf16 output.  With the
// inverse RHT (codes of an RHT-quantized output), each decoded 16-block is
// mapped back to the source basis before the output rounding: signs on the
// inputs, the butterfly with strides 1, 2, 4, 8, then x 0.25.
#include <cuda_bf16.h>

#include "nvfp4_encode.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {

__global__ void __launch_bounds__(256) k_dequant(const uint8_t *__restrict__ codes, const uint8_t *__restrict__ scales,
                                                 const float *__restrict__ gscale, int64_t rows, int64_t cols,
                                                 int swizzled, int per_row, void *out, int out_fp32, int rht,
                                                 uint32_t sign_mask) {
    f2 sgn[8];  // +-1 per input element of the inverse RHT
#pragma unroll
    for (int k = 0; k < 8; k++)
        sgn[k] = f2{((sign_mask >> (2 * k)) & 1u) ? -1.0f : 1.0f, ((sign_mask >> (2 * k + 1)) & 1u) ? -1.0f : 1.0f};
    const uint32_t CS = (uint32_t)(cols >> 4);
    const uint32_t n = (uint32_t)rows * CS;
    const int64_t csp = (CS + 3) & ~3u;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const uint32_t r = i / CS, j = i - r * CS;
        const float g = per_row ? gscale[r] : gscale[0];
        const uint32_t S = scales[swizzled ? swizzle_offset(r, j, csp) : (int64_t)i];
        const float d = __fmul_rn(e4m3_value(S), g);
        const uint2 c = *reinterpret_cast<const uint2 *>(codes + (int64_t)r * (cols >> 1) + 8 * j);
        f2 o[8];
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const uint32_t w = (k < 4) ? c.x : c.y;
            o[k] = mul2(e2m1x2_value(w >> (8 * (k & 3))), f2{d, d});
        }
        if (rht) {
#pragma unroll
            for (int k = 0; k < 8; k++) o[k] = mul2(o[k], sgn[k]);
            fwht16(o);
#pragma unroll
            for (int k = 0; k < 8; k++) o[k] = mul2(o[k], f2{0.25f, 0.25f});
        }
        const int64_t base = (int64_t)r * cols + 16 * j;
        if (out_fp32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out) + base);
#pragma unroll
            for (int k = 0; k < 4; k++) dst[k] = make_float4(o[2 * k].x, o[2 * k].y, o[2 * k + 1].x, o[2 * k + 1].y);
        } else {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(o[k].x, o[k].y);
                w[k] = *reinterpret_cast<const uint32_t *>(&h);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + base);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
    }
}

// Pad bytes of a swizzled scale array: rows [R, R_p) of every scale column,
// and scale columns [CS, CS_p) of rows [0, R).
__global__ void __launch_bounds__(256) k_scale_pad(uint8_t *scales, int64_t R, int64_t CS) {
    const int64_t Rp = (R + 127) / 128 * 128, CSp = (CS + 3) / 4 * 4;
    const int64_t n1 = (Rp - R) * CSp, n2 = R * (CSp - CS);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n1 + n2; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t r, j;
        if (i < n1) {
            r = R + i / CSp;
            j = i % CSp;
        } else {
            const int64_t k = i - n1, w = CSp - CS;
            r = k / w;
            j = CS + k % w;
        }
        scales[swizzle_offset(r, j, CSp)] = 0;
    }
}

cudaError_t launch_scale_pad(uint8_t *scales, int64_t rows_out, int64_t cs, cudaStream_t s) {
    const int64_t Rp = (rows_out + 127) / 128 * 128, CSp = (cs + 3) / 4 * 4;
    const int64_t n = (Rp - rows_out) * CSp + rows_out * (CSp - cs);
    if (n == 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256;
    k_scale_pad<<<(int)(blocks < 1024 ? blocks : 1024), 256, 0, s>>>(scales, rows_out, cs);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t *codes, const uint8_t *scales, const float *gscale, int64_t rows,
                           int64_t cols, int swizzled, int per_row, void *out, int out_fp32, int rht,
                           uint32_t sign_mask, cudaStream_t s) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_dequant, 256, 0);
    const int64_t want = (rows * (cols >> 4) + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
    const int grid = (int)(want < cap ? (want > 0 ? want : 1) : cap);
    k_dequant<<<grid, 256, 0, s>>>(codes, scales, gscale, rows, cols, swizzled, per_row, out, out_fp32, rht,
                                   sign_mask);
    return cudaGetLastError();
}

}  // namespace nvfp4
