// nvfp4_quant_row.cu -- rowwise 1x16 quantize kernels.
//
//  k_quant_row        per-tensor global scale (amax from the amax pass or
//                     given by the caller).  Each CTA encodes one contiguous
//                     range of 16-element blocks, a thread one block per
//                     step, with the next block's loads issued before the
//                     current one is encoded.
//  k_quant_rowscaled  one global scale per row: a CTA owns a row, reduces its
//                     amax, prepares that row's divisor table, then encodes
//                     it (single launch, no separate amax pass).
#include "nvfp4_encode.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_load.cuh"

namespace nvfp4 {

// Scale bytes of 4 consecutive blocks of a row go out as one 32-bit store
// (lanes 4m..4m+3 hold blocks j..j+3 with j % 4 == 0); otherwise one byte.
__device__ __forceinline__ void store_scale(const QArgs &a, uint8_t *scales, uint32_t S, int64_t r, uint32_t j,
                                            uint32_t CS, int64_t csp, bool active, bool words) {
    if (words) {
        const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, S, 1);
        const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, S, 2);
        const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, S, 3);
        if (active && (j & 3u) == 0) {
            const int64_t off = a.swizzled ? swizzle_offset(r, j, csp) : r * CS + j;
            *reinterpret_cast<uint32_t *>(scales + off) = S | (s1 << 8) | (s2 << 16) | (s3 << 24);
        }
    } else if (active) {
        scales[a.swizzled ? swizzle_offset(r, j, csp) : r * CS + j] = (uint8_t)S;
    }
}

template <int MODE, bool RHT, typename T>
__global__ void __launch_bounds__(256) k_quant_row(const QArgs a) {
    __shared__ DivTable tab;
    const uint32_t CS = (uint32_t)(a.cols >> 4);
    const uint32_t n = (uint32_t)a.rows * CS;
    const int64_t csp = (CS + 3) & ~3u;
    const float g = global_scale_of(a.amax[0]);
    build_table(tab, g, threadIdx.x, blockDim.x);
    const ScaleDiv sd = make_scale_div(g);
    if (blockIdx.x == 0 && threadIdx.x == 0) a.gscale[0] = g;
    __syncthreads();

    // this CTA's range of blocks: a multiple of 32 long, so warps stay whole
    const uint32_t per = ((n + gridDim.x - 1) / gridDim.x + 31) & ~31u;
    const uint32_t b0 = blockIdx.x * per;
    if (b0 >= n) return;
    const uint32_t b1 = min(n, b0 + per);
    const bool words = (CS & 3u) == 0;
    const T *x = static_cast<const T *>(a.x);

    uint32_t i = b0 + threadIdx.x;
    uint32_t r = i / CS, j = i - r * CS;
    const uint32_t dr = blockDim.x / CS, dj = blockDim.x % CS;
    RawBlock<T> cur, nxt;
    if (i < b1) load_raw(x + (int64_t)r * a.ld + 16 * j, cur);
    for (uint32_t base = b0 + (threadIdx.x & ~31u); base < b1; base += blockDim.x) {
        const bool active = i < b1;
        // next block of this thread
        const uint32_t i2 = i + blockDim.x;
        uint32_t r2 = r + dr, j2 = j + dj;
        if (j2 >= CS) { j2 -= CS; ++r2; }
        if (i2 < b1) load_raw(x + (int64_t)r2 * a.ld + 16 * j2, nxt);
        uint32_t S = 0;
        if (active) {
            f2 v[8];
            unpack(cur, v);
            if (RHT) rht16(v, a.sign_mask);
            uint4 rnd = make_uint4(0u, 0u, 0u, 0u);
            if (MODE == MODE_SR) rnd = block_random(a.seed, a.offset, i);
            const uint2 c = encode_block<MODE>(v, sd, tab, rnd, S);
            *reinterpret_cast<uint2 *>(a.codes_row + (int64_t)r * (a.cols >> 1) + 8 * j) = c;
        }
        store_scale(a, a.scales_row, S, r, j, CS, csp, active, words);
        i = i2;
        r = r2;
        j = j2;
        cur = nxt;
    }
}

template <int MODE, bool RHT, typename T>
__global__ void __launch_bounds__(256) k_quant_rowscaled(const QArgs a) {
    __shared__ DivTable tab;
    __shared__ uint32_t red[32];
    const uint32_t CS = (uint32_t)(a.cols >> 4);
    const int64_t csp = (CS + 3) & ~3u;
    const bool words = (CS & 3u) == 0;
    const T *x = static_cast<const T *>(a.x);
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const T *xr = x + r * a.ld;
        // pass 1: amax of the row (post-RHT magnitudes; the 0.25 is applied to
        // the maximum, which rounds the same way because rounding is monotone)
        float m = 0.0f;
        for (uint32_t j = threadIdx.x; j < CS; j += blockDim.x) {
            RawBlock<T> b;
            load_raw(xr + 16 * j, b);
            f2 v[8];
            unpack(b, v);
            if (RHT) fwht16(v);
            m = absmax_nan(m, block_amax(v));
        }
        float A = __uint_as_float(block_max_u32(__float_as_uint(m), red));
        if (RHT) A = __fmul_rn(A, 0.25f);
        const float g = global_scale_of(A);
        if (threadIdx.x == 0) {
            a.amax[r] = A;
            a.gscale[r] = g;
        }
        build_table(tab, g, threadIdx.x, blockDim.x);
        const ScaleDiv sd = make_scale_div(g);
        __syncthreads();
        // pass 2: encode (warp-uniform trip count for the scale-word shuffles)
        for (uint32_t base = threadIdx.x & ~31u; base < CS; base += blockDim.x) {
            const uint32_t j = base + (threadIdx.x & 31u);
            const bool active = j < CS;
            uint32_t S = 0;
            if (active) {
                RawBlock<T> b;
                load_raw(xr + 16 * j, b);
                f2 v[8];
                unpack(b, v);
                if (RHT) rht16(v, a.sign_mask);
                uint4 rnd = make_uint4(0u, 0u, 0u, 0u);
                if (MODE == MODE_SR) rnd = block_random(a.seed, a.offset, (uint64_t)r * CS + j);
                const uint2 c = encode_block<MODE>(v, sd, tab, rnd, S);
                *reinterpret_cast<uint2 *>(a.codes_row + r * (a.cols >> 1) + 8 * j) = c;
            }
            store_scale(a, a.scales_row, S, r, j, CS, csp, active, words);
        }
        __syncthreads();  // the next row rebuilds the table
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
