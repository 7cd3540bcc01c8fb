// nvfp4_amax.cu -- global amax reductions.
//
// Per tensor: grid-stride 128-bit loads, magnitude-bit maximum per thread,
// warp (redux.sync) and CTA trees, then ONE atomicMax per CTA into the
// workspace.  The CTA that takes the last ticket publishes amax and
// g = amax / 2688 and returns the workspace to zero, so the pass needs no
// memset and no second launch.  The host never waits: the per-tensor scale
// stays on the device ("nvfp4-sm120" README, section "Results": the amax host
// sync was 86% of the quantizer's time).
//
// With the RHT the maximum is over the post-transform magnitudes.  Signs do
// not change magnitudes and rounding is monotone, so the kernel takes the
// maximum of the raw butterfly outputs and multiplies it by 0.25 once.
#include "nvfp4_encode.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_load.cuh"
#include "nvfp4_tma.cuh"

namespace nvfp4 {

__device__ __forceinline__ void publish_tensor_amax(const QArgs &a, uint32_t m, bool rht) {
    __shared__ uint32_t red[32];
    allow_dependents();  // the quantize pass may start staging its tiles
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) {
        atomicMax(&a.workspace[0], m);
        __threadfence();
        const uint32_t ticket = atomicAdd(&a.workspace[1], 1u);
        if (ticket == gridDim.x - 1) {
            __threadfence();
            const uint32_t bits = atomicExch(&a.workspace[0], 0u);
            atomicExch(&a.workspace[1], 0u);
            float A = __uint_as_float(bits);
            if (rht) A = __fmul_rn(A, 0.25f);
            a.amax[0] = A;
            a.gscale[0] = global_scale_of(A);
        }
    }
}

// No RHT: the maximum over every element, any orientation.  A thread takes
// kPlainUnroll 16-byte chunks per step (all loads issued before any is
// used), so enough bytes are in flight to stream at HBM rate.
constexpr int kPlainUnroll = 4;

template <typename T>
__global__ void __launch_bounds__(256) k_amax_plain(const QArgs a) {
    constexpr int W = Chunk<T>::W;
    const uint32_t NCH = (uint32_t)((a.cols + W - 1) / W);
    const uint32_t n = (uint32_t)a.rows * NCH;
    const T *x = static_cast<const T *>(a.x);
    const uint32_t stride = gridDim.x * blockDim.x;
    uint32_t m = 0;
    for (uint32_t i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < n; i0 += kPlainUnroll * stride) {
        Chunk<T> c[kPlainUnroll];
#pragma unroll
        for (int u = 0; u < kPlainUnroll; u++) {
            const uint32_t i = i0 + u * stride;
            if (i < n) {
                const uint32_t r = i / NCH, ch = i - r * NCH;
                const int64_t c0 = (int64_t)ch * W;
                c[u].load(x + (int64_t)r * a.ld + c0, (int)min((int64_t)W, a.cols - c0));
            }
        }
#pragma unroll
        for (int u = 0; u < kPlainUnroll; u++)
            if (i0 + u * stride < n)
#pragma unroll
                for (int e = 0; e < W; e++) m = max(m, mag_bits(c[u].get(e)));
    }
    publish_tensor_amax(a, m, false);
}

// RHT blocks along rows.  Each CTA scans one contiguous range of blocks; a
// thread keeps kAmaxDepth blocks' loads in flight (consecutive blocks of its
// range, 32 bytes each for bf16) and transforms them as they land.
constexpr int kAmaxDepth = 1;

template <typename T>
__global__ void __launch_bounds__(256) k_amax_rht_row(const QArgs a) {
    const uint32_t CS = (uint32_t)(a.cols >> 4);
    const uint32_t n = (uint32_t)a.rows * CS;
    const uint32_t span = blockDim.x * kAmaxDepth;  // blocks per CTA step
    const uint32_t per = ((n + gridDim.x - 1) / gridDim.x + span - 1) / span * span;
    const uint32_t b0 = blockIdx.x * per, b1 = min(n, b0 + per);
    const T *x = static_cast<const T *>(a.x);
    uint32_t m = 0;
    for (uint32_t base = b0; base < b1; base += span) {
        RawBlock<T> raw[kAmaxDepth];
#pragma unroll
        for (int k = 0; k < kAmaxDepth; k++) {
            const uint32_t i = base + k * blockDim.x + threadIdx.x;
            if (i < b1) {
                const uint32_t r = i / CS, j = i - r * CS;
                load_raw(x + (int64_t)r * a.ld + 16 * j, raw[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < kAmaxDepth; k++) {
            if (base + k * blockDim.x + threadIdx.x < b1) {
                f2 v[8];
                unpack(raw[k], v);
                fwht16(v);
                m = max(m, __float_as_uint(block_amax(v)));
            }
        }
    }
    publish_tensor_amax(a, m, true);
}

// RHT blocks along columns: a thread owns 16 rows x one 16-byte chunk.
template <typename T>
__global__ void __launch_bounds__(256) k_amax_rht_col(const QArgs a) {
    constexpr int CW = Chunk<T>::W;
    const uint32_t C = (uint32_t)a.cols;
    const uint32_t RB = (uint32_t)(a.rows >> 4), NCH = (C + CW - 1) / CW;
    const uint32_t n = RB * NCH;
    const T *x = static_cast<const T *>(a.x);
    uint32_t m = 0;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const uint32_t ch = i % NCH, rb = i / NCH;
        const uint32_t c0 = ch * CW;
        const int valid = (int)min((uint32_t)CW, C - c0);
        Chunk<T> rows[16];
#pragma unroll
        for (int k = 0; k < 16; k++) rows[k].load(x + ((int64_t)rb * 16 + k) * a.ld + c0, valid);
#pragma unroll
        for (int cc = 0; cc < CW; cc++) {
            f2 v[8];
#pragma unroll
            for (int p = 0; p < 8; p++) v[p] = f2{rows[2 * p].get(cc), rows[2 * p + 1].get(cc)};
            fwht16(v);
            // columns past the edge were loaded as zeros and stay zero
            m = max(m, __float_as_uint(block_amax(v)));
        }
    }
    publish_tensor_amax(a, m, true);
}

// Per-row amax of the rowwise orientation: a CTA per row.
template <bool RHT, typename T>
__global__ void __launch_bounds__(256) k_amax_rows(const QArgs a) {
    __shared__ uint32_t red[32];
    const uint32_t CS = (uint32_t)(a.cols >> 4);
    const T *x = static_cast<const T *>(a.x);
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        uint32_t m = 0;
        for (uint32_t j = threadIdx.x; j < CS; j += blockDim.x) {
            f2 v[8];
            load_block_row(x + r * a.ld + 16 * j, v);
            if (RHT) fwht16(v);
            m = max(m, __float_as_uint(block_amax(v)));
        }
        m = block_max_u32(m, red);
        if (threadIdx.x == 0) {
            float A = __uint_as_float(m);
            if (RHT) A = __fmul_rn(A, 0.25f);
            a.amax[r] = A;
            a.gscale[r] = global_scale_of(A);
        }
    }
}

// Grouped rowwise scaling: n_groups row ranges, each its own tensor for the
// amax.  A CTA takes a contiguous range of rows and, for each group segment in
// it, reduces the segment's blocks (post-RHT magnitudes without the 0.25) and
// folds the result into amax[g] with one atomicMax on its bits (the caller
// zeroed amax[]; magnitude bits order like the floats, NaN above +inf).
template <bool RHT, typename T>
__global__ void __launch_bounds__(256) k_amax_groups(const QArgs a) {
    __shared__ uint32_t red[32];
    const uint32_t CS = (uint32_t)(a.cols >> 4);
    const T *x = static_cast<const T *>(a.x);
    const int64_t per = (a.rows + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = (int64_t)blockIdx.x * per, r1 = min(a.rows, r0 + per);
    if (r0 >= r1) return;
    // the group of r0: largest g with offsets[g] <= r0
    int64_t lo = 0, hi = a.n_groups - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (__ldg(a.group_offsets + mid) <= r0) lo = mid;
        else hi = mid - 1;
    }
    uint32_t *bits = reinterpret_cast<uint32_t *>(a.amax);
    for (int64_t g = lo; g < a.n_groups; ++g) {
        const int64_t s0 = max(r0, __ldg(a.group_offsets + g)), s1 = min(r1, __ldg(a.group_offsets + g + 1));
        if (s0 >= r1) break;
        if (s0 >= s1) continue;  // an empty group, or one that ends before this range
        const uint64_t nb = (uint64_t)(s1 - s0) * CS;
        uint32_t m = 0;
        for (uint64_t i = threadIdx.x; i < nb; i += blockDim.x) {
            const int64_t r = s0 + (int64_t)(i / CS);
            const uint32_t j = (uint32_t)(i % CS);
            f2 v[8];
            load_block_row(x + r * a.ld + 16 * j, v);
            if (RHT) fwht16(v);
            m = max(m, __float_as_uint(block_amax(v)) & 0x7FFFFFFFu);
        }
        m = block_max_u32(m, red);
        if (threadIdx.x == 0) atomicMax(bits + g, m);
    }
}

// amax[g] from its bits (x 0.25 for the RHT, unless the caller gave it) and
// global_scale[g] = amax[g] / 2688.
__global__ void k_group_finalize(const QArgs a, int rht, int given) {
    const int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (g >= a.n_groups) return;
    float A = a.amax[g];
    if (!given && rht) A = __fmul_rn(A, 0.25f);
    a.amax[g] = A;
    a.gscale[g] = global_scale_of(A);
}

template <typename K>
static int grid_for(K kernel, int64_t work_items) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0);
    if (per_sm < 1) per_sm = 1;
    const int64_t want = (work_items + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

template <typename T>
static cudaError_t run_amax_tensor(const QArgs &a, bool rht, bool col, cudaStream_t s) {
    constexpr int W = Chunk<T>::W;
    if (!rht) {
        auto k = k_amax_plain<T>;
        k<<<grid_for(k, a.rows * ((a.cols + W - 1) / W)), 256, 0, s>>>(a);
    } else if (!col) {
        auto k = k_amax_rht_row<T>;
        k<<<grid_for(k, a.rows * (a.cols >> 4)), 256, 0, s>>>(a);
    } else {
        auto k = k_amax_rht_col<T>;
        k<<<grid_for(k, (a.rows >> 4) * ((a.cols + W - 1) / W)), 256, 0, s>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_amax_tensor(const QArgs &a, bool fp32, bool rht, bool col, cudaStream_t s) {
    return fp32 ? run_amax_tensor<float>(a, rht, col, s) : run_amax_tensor<bf16_t>(a, rht, col, s);
}

template <bool RHT, typename T>
static cudaError_t run_amax_rows(const QArgs &a, cudaStream_t s) {
    auto k = k_amax_rows<RHT, T>;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 256, 0);
    const int64_t cap = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
    k<<<(int)(a.rows < cap ? (a.rows > 0 ? a.rows : 1) : cap), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_amax_rows(const QArgs &a, bool fp32, bool rht, cudaStream_t s) {
    if (fp32) return rht ? run_amax_rows<true, float>(a, s) : run_amax_rows<false, float>(a, s);
    return rht ? run_amax_rows<true, bf16_t>(a, s) : run_amax_rows<false, bf16_t>(a, s);
}

template <bool RHT, typename T>
static cudaError_t run_amax_groups(const QArgs &a, cudaStream_t s) {
    auto k = k_amax_groups<RHT, T>;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 256, 0);
    const int64_t cap = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
    k<<<(int)(a.rows < cap ? (a.rows > 0 ? a.rows : 1) : cap), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_amax_groups(const QArgs &a, bool fp32, bool rht, cudaStream_t s) {
    if (fp32) return rht ? run_amax_groups<true, float>(a, s) : run_amax_groups<false, float>(a, s);
    return rht ? run_amax_groups<true, bf16_t>(a, s) : run_amax_groups<false, bf16_t>(a, s);
}

cudaError_t launch_group_finalize(const QArgs &a, bool rht, bool given, cudaStream_t s) {
    const int64_t blocks = (a.n_groups + 255) / 256;
    k_group_finalize<<<(unsigned)blocks, 256, 0, s>>>(a, rht ? 1 : 0, given ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace nvfp4
