// nvfp4_quant_col.cu -- columnwise (X^T) 1x16 quantize and 16x16 (2D) tiles.
//
// A thread owns a strip of 16 X rows x one 16-byte chunk of columns (8 bf16 or
// 4 fp32): a warp reads 512 contiguous bytes per row.  Each column of the
// strip is one 16-element block of an X^T row.
#include "nvfp4_encode.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_load.cuh"

namespace nvfp4 {

// Block of column `cc` of a 16-row strip: pair m = (row 2m, row 2m+1).
template <typename T>
__device__ __forceinline__ void strip_column(const Chunk<T> (&rows)[16], int cc, f2 (&v)[8]) {
#pragma unroll
    for (int m = 0; m < 8; m++) v[m] = f2{rows[2 * m].get(cc), rows[2 * m + 1].get(cc)};
}

template <typename T>
__device__ __forceinline__ void load_strip(const T *x, int64_t ld, int64_t r0, int64_t c0, int valid,
                                           Chunk<T> (&rows)[16]) {
#pragma unroll
    for (int k = 0; k < 16; k++) rows[k].load(x + (r0 + k) * ld + c0, valid);
}

template <int MODE, bool RHT, typename T>
__global__ void __launch_bounds__(256) k_quant_col(const QArgs a) {
    constexpr int CW = Chunk<T>::W;
    __shared__ DivTable tab;
    __shared__ RhtMult rm;
    if (RHT) build_rht_mult(rm, a.sign_mask, threadIdx.x);
    const uint32_t C = (uint32_t)a.cols;
    const uint32_t RB = (uint32_t)(a.rows >> 4);  // blocks per X^T row
    const uint32_t NCH = (C + CW - 1) / CW;
    const uint32_t n = RB * NCH;
    const int64_t csp = (RB + 3) & ~3u;
    const float g = global_scale_of(a.amax[0]);
    build_table(tab, g, threadIdx.x, blockDim.x);
    const ScaleDiv sd = make_scale_div(g);
    if (blockIdx.x == 0 && threadIdx.x == 0) a.gscale[0] = g;
    __syncthreads();
    const T *x = static_cast<const T *>(a.x);
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const uint32_t ch = i % NCH, rb = i / NCH;
        const uint32_t c0 = ch * CW;
        Chunk<T> rows[16];
        load_strip(x, a.ld, (int64_t)rb * 16, c0, (int)min((uint32_t)CW, C - c0), rows);
#pragma unroll
        for (int cc = 0; cc < CW; cc++) {
            const uint32_t o = c0 + cc;  // X column = X^T row
            if (o >= C) break;
            f2 v[8];
            strip_column(rows, cc, v);
            if (RHT) rht16(v, rm);
            const uint64_t blk = (uint64_t)o * RB + rb;
            uint4 rnd = make_uint4(0u, 0u, 0u, 0u);
            if (MODE == MODE_SR) rnd = block_random(a.seed, a.offset, blk);
            uint32_t S;
            const uint2 c = encode_block<MODE>(v, sd, tab, rnd, S);
            *reinterpret_cast<uint2 *>(a.codes_col + (int64_t)o * (a.rows >> 1) + 8 * rb) = c;
            a.scales_col[a.swizzled ? swizzle_offset(o, rb, csp) : (int64_t)blk] = (uint8_t)S;
        }
    }
}

// Codes of NP pairs against divisor entry S (RNE): NP = 4 -> one word, NP = 2
// -> low half of a word.
template <int NP>
__device__ __forceinline__ uint32_t encode_pairs_rne(const f2 (&y)[NP], uint32_t S, const DivTable &T) {
    if (S == 0u) return 0u;
    const Divisor &D = T.e[S & 0x7Fu];
    f2 q[4] = {f2{0.f, 0.f}, f2{0.f, 0.f}, f2{0.f, 0.f}, f2{0.f, 0.f}};
    const bool fast = divisor_fast(D.d);
#pragma unroll
    for (int k = 0; k < NP; k++)
        q[k] = fast ? neg_quot2(y[k], D) : f2{neg_quot_slow(y[k].x, D.d), neg_quot_slow(y[k].y, D.d)};
    return e2m1x8(q[0].x, q[0].y, q[1].x, q[1].y, q[2].x, q[2].y, q[3].x, q[3].y) ^ 0x88888888u;
}

// 16x16 tiles: the 16/CW lanes that share a tile combine their maxima, then
// every lane encodes its rows (half / quarter blocks) and its columns.
template <typename T>
__global__ void __launch_bounds__(256) k_quant_2d(const QArgs a) {
    constexpr int CW = Chunk<T>::W;
    constexpr int LPT = 16 / CW;  // lanes per 16x16 tile
    const uint32_t C = (uint32_t)a.cols;
    const uint32_t RB = (uint32_t)(a.rows >> 4), CB = C >> 4;
    const uint32_t NCH = C / CW;
    const uint32_t n = RB * NCH;  // a multiple of LPT
    const int64_t csp_row = (CB + 3) & ~3u, csp_col = (RB + 3) & ~3u;
    __shared__ DivTable tab;
    const float g = global_scale_of(a.amax[0]);
    build_table(tab, g, threadIdx.x, blockDim.x);
    const ScaleDiv sd = make_scale_div(g);
    if (blockIdx.x == 0 && threadIdx.x == 0) a.gscale[0] = g;
    __syncthreads();
    const T *x = static_cast<const T *>(a.x);
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t base = blockIdx.x * blockDim.x + (threadIdx.x & ~31u); base < n; base += stride) {
        const uint32_t i = base + lane;
        const bool active = i < n;
        const uint32_t ch = active ? i % NCH : 0, rb = active ? i / NCH : 0;
        const uint32_t c0 = ch * CW;
        Chunk<T> rows[16];
        uint32_t m = 0;
        if (active) {
            load_strip(x, a.ld, (int64_t)rb * 16, c0, CW, rows);
#pragma unroll
            for (int k = 0; k < 16; k++)
#pragma unroll
                for (int c = 0; c < CW; c++) m = max(m, mag_bits(rows[k].get(c)));
        }
#pragma unroll
        for (int off = 1; off < LPT; off <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
        if (!active) continue;
        const uint32_t S = block_scale(__uint_as_float(m), sd.m6, sd.fast6);
        const uint32_t cb = c0 >> 4;  // tile column
        if (a.want_row) {
#pragma unroll
            for (int k = 0; k < 16; k++) {
                const int64_t r = (int64_t)rb * 16 + k;
                f2 y[CW / 2];
#pragma unroll
                for (int p = 0; p < CW / 2; p++) y[p] = f2{rows[k].get(2 * p), rows[k].get(2 * p + 1)};
                const uint32_t w = encode_pairs_rne<CW / 2>(y, S, tab);
                uint8_t *dst = a.codes_row + r * (C >> 1) + (c0 >> 1);
                if (CW == 8) *reinterpret_cast<uint32_t *>(dst) = w;
                else *reinterpret_cast<uint16_t *>(dst) = (uint16_t)w;
                if ((ch & (LPT - 1)) == 0)
                    a.scales_row[a.swizzled ? swizzle_offset(r, cb, csp_row) : r * CB + cb] = (uint8_t)S;
            }
        }
        if (a.want_col) {
#pragma unroll
            for (int cc = 0; cc < CW; cc++) {
                const int64_t o = c0 + cc;
                f2 v[8];
                strip_column(rows, cc, v);
                const uint4 none = make_uint4(0u, 0u, 0u, 0u);
                const uint2 c = encode_with_scale<false>(v, S, tab, none);
                *reinterpret_cast<uint2 *>(a.codes_col + o * (a.rows >> 1) + 8 * rb) = c;
                a.scales_col[a.swizzled ? swizzle_offset(o, rb, csp_col) : o * RB + rb] = (uint8_t)S;
            }
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
static cudaError_t run_col(const QArgs &a, cudaStream_t s) {
    auto k = k_quant_col<MODE, RHT, T>;
    const int64_t work = (a.rows >> 4) * ((a.cols + Chunk<T>::W - 1) / Chunk<T>::W);
    k<<<grid_for(k, 256, work), 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t dispatch_col(const QArgs &a, int mode, bool rht, cudaStream_t s) {
    if (mode == MODE_RNE) return rht ? run_col<MODE_RNE, true, T>(a, s) : run_col<MODE_RNE, false, T>(a, s);
    if (mode == MODE_SR) return rht ? run_col<MODE_SR, true, T>(a, s) : run_col<MODE_SR, false, T>(a, s);
    return run_col<MODE_4O6, false, T>(a, s);
}

cudaError_t launch_quant_col(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return fp32 ? dispatch_col<float>(a, mode, rht, s) : dispatch_col<bf16_t>(a, mode, rht, s);
}

template <typename T>
static cudaError_t run_2d(const QArgs &a, cudaStream_t s) {
    auto k = k_quant_2d<T>;
    const int64_t work = (a.rows >> 4) * (a.cols / Chunk<T>::W);
    k<<<grid_for(k, 256, work), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quant_2d(const QArgs &a, bool fp32, cudaStream_t s) {
    return fp32 ? run_2d<float>(a, s) : run_2d<bf16_t>(a, s);
}

}  // namespace nvfp4
