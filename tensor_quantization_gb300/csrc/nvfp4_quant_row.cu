// nvfp4_quant_row.cu -- rowwise 1x16 quantize kernels.
//
//  k_quant_row        per-tensor global scale (amax from the amax pass or
//                     given by the caller); one thread per 16-element block.
//  k_quant_rowscaled  one global scale per row: a CTA owns a row, reduces its
//                     amax, then encodes it (single launch, no amax pass).
#include "nvfp4_encode.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_load.cuh"

namespace nvfp4 {

template <int MODE, bool RHT, typename T>
__global__ void __launch_bounds__(256) k_quant_row(const QArgs a) {
    const uint32_t CS = (uint32_t)(a.cols >> 4);
    const uint32_t n = (uint32_t)a.rows * CS;
    const int64_t csp = (CS + 3) & ~3u;
    const float g = global_scale_of(a.amax[0]);
    if (blockIdx.x == 0 && threadIdx.x == 0) a.gscale[0] = g;
    const T *x = static_cast<const T *>(a.x);
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const uint32_t r = i / CS, j = i - r * CS;
        f2 v[8];
        load_block_row(x + (int64_t)r * a.ld + 16 * j, v);
        if (RHT) rht16(v, a.sign_mask);
        uint4 rnd = make_uint4(0u, 0u, 0u, 0u);
        if (MODE == MODE_SR) rnd = block_random(a.seed, a.offset, i);
        uint32_t S;
        const uint2 c = encode_block<MODE>(v, g, rnd, S);
        *reinterpret_cast<uint2 *>(a.codes_row + (int64_t)r * (a.cols >> 1) + 8 * j) = c;
        a.scales_row[a.swizzled ? swizzle_offset(r, j, csp) : (int64_t)i] = (uint8_t)S;
    }
}

template <int MODE, bool RHT, typename T>
__global__ void __launch_bounds__(256) k_quant_rowscaled(const QArgs a) {
    __shared__ uint32_t red[32];
    const uint32_t CS = (uint32_t)(a.cols >> 4);
    const int64_t csp = (CS + 3) & ~3u;
    const T *x = static_cast<const T *>(a.x);
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const T *xr = x + r * a.ld;
        // pass 1: amax of the row (post-RHT magnitudes; the 0.25 is applied to
        // the maximum, which rounds the same way because rounding is monotone)
        uint32_t m = 0;
        for (uint32_t j = threadIdx.x; j < CS; j += blockDim.x) {
            f2 v[8];
            load_block_row(xr + 16 * j, v);
            if (RHT) fwht16(v);
            m = max(m, amax_bits(v));
        }
        m = block_max_u32(m, red);
        float A = __uint_as_float(m);
        if (RHT) A = __fmul_rn(A, 0.25f);
        const float g = global_scale_of(A);
        if (threadIdx.x == 0) {
            a.amax[r] = A;
            a.gscale[r] = g;
        }
        // pass 2: encode
        for (uint32_t j = threadIdx.x; j < CS; j += blockDim.x) {
            f2 v[8];
            load_block_row(xr + 16 * j, v);
            if (RHT) rht16(v, a.sign_mask);
            uint4 rnd = make_uint4(0u, 0u, 0u, 0u);
            if (MODE == MODE_SR) rnd = block_random(a.seed, a.offset, (uint64_t)r * CS + j);
            uint32_t S;
            const uint2 c = encode_block<MODE>(v, g, rnd, S);
            *reinterpret_cast<uint2 *>(a.codes_row + r * (a.cols >> 1) + 8 * j) = c;
            a.scales_row[a.swizzled ? swizzle_offset(r, j, csp) : r * CS + j] = (uint8_t)S;
        }
    }
}

template <typename K>
static int grid_for(K kernel, int threads, int64_t work_items) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0);
    if (per_sm < 1) per_sm = 1;
    const int64_t want = (work_items + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

template <int MODE, bool RHT, typename T>
static cudaError_t run_row(const QArgs &a, cudaStream_t s) {
    auto k = k_quant_row<MODE, RHT, T>;
    const int grid = grid_for(k, 256, (a.cols >> 4) * a.rows);
    k<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <int MODE, bool RHT, typename T>
static cudaError_t run_rowscaled(const QArgs &a, cudaStream_t s) {
    auto k = k_quant_rowscaled<MODE, RHT, T>;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 256, 0);
    const int64_t cap = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
    const int grid = (int)(a.rows < cap ? (a.rows > 0 ? a.rows : 1) : cap);
    k<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t dispatch_row(const QArgs &a, int mode, bool rht, bool scaled_rows, cudaStream_t s) {
    if (scaled_rows) {
        if (mode == MODE_RNE) return rht ? run_rowscaled<MODE_RNE, true, T>(a, s) : run_rowscaled<MODE_RNE, false, T>(a, s);
        if (mode == MODE_SR) return rht ? run_rowscaled<MODE_SR, true, T>(a, s) : run_rowscaled<MODE_SR, false, T>(a, s);
        return run_rowscaled<MODE_4O6, false, T>(a, s);
    }
    if (mode == MODE_RNE) return rht ? run_row<MODE_RNE, true, T>(a, s) : run_row<MODE_RNE, false, T>(a, s);
    if (mode == MODE_SR) return rht ? run_row<MODE_SR, true, T>(a, s) : run_row<MODE_SR, false, T>(a, s);
    return run_row<MODE_4O6, false, T>(a, s);
}

cudaError_t launch_quant_row(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return fp32 ? dispatch_row<float>(a, mode, rht, false, s) : dispatch_row<bf16_t>(a, mode, rht, false, s);
}

cudaError_t launch_quant_rowscaled(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return fp32 ? dispatch_row<float>(a, mode, rht, true, s) : dispatch_row<bf16_t>(a, mode, rht, true, s);
}

}  // namespace nvfp4
