// nvfp4_load.cuh -- global-memory loaders (128-bit, read-only path).
#pragma once

#include "nvfp4_device.cuh"

namespace nvfp4 {

typedef uint16_t bf16_t;  // bf16 elements are handled as raw 16-bit patterns

__device__ __forceinline__ uint4 ld_nc(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ f2 bf16_pair(uint32_t w) { return f2{bf16_lo(w), bf16_hi(w)}; }

// One 1x16 block of a row (16 consecutive elements, 16-byte aligned).
__device__ __forceinline__ void load_block_row(const bf16_t *p, f2 (&v)[8]) {
    const uint4 a = ld_nc(p), b = ld_nc(p + 8);
    v[0] = bf16_pair(a.x); v[1] = bf16_pair(a.y); v[2] = bf16_pair(a.z); v[3] = bf16_pair(a.w);
    v[4] = bf16_pair(b.x); v[5] = bf16_pair(b.y); v[6] = bf16_pair(b.z); v[7] = bf16_pair(b.w);
}
__device__ __forceinline__ void load_block_row(const float *p, f2 (&v)[8]) {
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const uint4 a = ld_nc(p + 4 * k);
        v[2 * k] = f2{__uint_as_float(a.x), __uint_as_float(a.y)};
        v[2 * k + 1] = f2{__uint_as_float(a.z), __uint_as_float(a.w)};
    }
}

// The raw bytes of one 1x16 block (32 B of bf16 or 64 B of fp32), loaded with
// 128-bit reads so that the loads can be issued ahead of their use.
template <typename T>
struct RawBlock {
    uint4 w[sizeof(T)];  // 16 elements * sizeof(T) bytes / 16 bytes per uint4
};

template <typename T>
__device__ __forceinline__ void load_raw(const T *p, RawBlock<T> &b) {
#pragma unroll
    for (int k = 0; k < (int)sizeof(T); k++) b.w[k] = ld_nc(p + k * (16 / sizeof(T)));
}

__device__ __forceinline__ void unpack(const RawBlock<bf16_t> &b, f2 (&v)[8]) {
    v[0] = bf16_pair(b.w[0].x); v[1] = bf16_pair(b.w[0].y); v[2] = bf16_pair(b.w[0].z); v[3] = bf16_pair(b.w[0].w);
    v[4] = bf16_pair(b.w[1].x); v[5] = bf16_pair(b.w[1].y); v[6] = bf16_pair(b.w[1].z); v[7] = bf16_pair(b.w[1].w);
}
__device__ __forceinline__ void unpack(const RawBlock<float> &b, f2 (&v)[8]) {
#pragma unroll
    for (int k = 0; k < 4; k++) {
        v[2 * k] = f2{__uint_as_float(b.w[k].x), __uint_as_float(b.w[k].y)};
        v[2 * k + 1] = f2{__uint_as_float(b.w[k].z), __uint_as_float(b.w[k].w)};
    }
}

// Unpack a raw block and run the butterfly's first stage, (a, b) ->
// (a + b, a - b) on each pair.  For bf16 the even element a enters the adds
// as a bf16 operand of a mixed-precision add (it widens exactly, so the
// result is the fp32 sum), which saves unpacking it.
__device__ __forceinline__ void fwht_first_bf16(uint32_t w, f2 &o) {
    const float b = bf16_hi(w);
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; add.rn.f32.bf16 %0, lo, %3; sub.rn.f32.bf16 %1, lo, %3; }"
        : "=f"(o.x), "=f"(o.y)
        : "r"(w), "f"(b));
}
__device__ __forceinline__ void unpack_fwht_first(const RawBlock<bf16_t> &b, f2 (&v)[8]) {
    fwht_first_bf16(b.w[0].x, v[0]); fwht_first_bf16(b.w[0].y, v[1]);
    fwht_first_bf16(b.w[0].z, v[2]); fwht_first_bf16(b.w[0].w, v[3]);
    fwht_first_bf16(b.w[1].x, v[4]); fwht_first_bf16(b.w[1].y, v[5]);
    fwht_first_bf16(b.w[1].z, v[6]); fwht_first_bf16(b.w[1].w, v[7]);
}
__device__ __forceinline__ void unpack_fwht_first(const RawBlock<float> &b, f2 (&v)[8]) {
    unpack(b, v);
    fwht16_first(v);
}

// A 16-byte chunk of one row: 8 bf16 or 4 fp32 elements.  When fewer than a
// full chunk of columns remain, the missing elements read as zero.
template <typename T>
struct Chunk {
    static constexpr int W = 16 / sizeof(T);
    uint4 raw;
    __device__ __forceinline__ void load(const T *p, int valid) {
        if (valid >= W) {
            raw = ld_nc(p);
        } else {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int c = 0; c < W; c++)
                if (c < valid) w[c * sizeof(T) / 4] |= elem_bits(p[c]) << (8 * ((c * sizeof(T)) & 3));
            raw = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    static __device__ __forceinline__ uint32_t elem_bits(bf16_t v) { return (uint32_t)v; }
    static __device__ __forceinline__ uint32_t elem_bits(float v) { return __float_as_uint(v); }
    __device__ __forceinline__ float get(int c) const;
};
template <>
__device__ __forceinline__ float Chunk<bf16_t>::get(int c) const {
    const uint32_t w = (c >> 1) == 0 ? raw.x : (c >> 1) == 1 ? raw.y : (c >> 1) == 2 ? raw.z : raw.w;
    return (c & 1) ? bf16_hi(w) : bf16_lo(w);
}
template <>
__device__ __forceinline__ float Chunk<float>::get(int c) const {
    const uint32_t w = c == 0 ? raw.x : c == 1 ? raw.y : c == 2 ? raw.z : raw.w;
    return __uint_as_float(w);
}

// Block-wide maximum of a 32-bit value (every thread must call it).
__device__ __forceinline__ uint32_t block_max_u32(uint32_t m, uint32_t *red) {
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = m;
    __syncthreads();
    uint32_t t = (lane < nw) ? red[lane] : 0u;
    t = __reduce_max_sync(0xFFFFFFFFu, t);
    return t;
}

}  // namespace nvfp4
