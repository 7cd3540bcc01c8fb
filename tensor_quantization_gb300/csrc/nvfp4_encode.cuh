// nvfp4_encode.cuh -- block-level encoders shared by the quantize kernels.
//
// A 1x16 block is held as 8 fp32 pairs (element 2k in .x, 2k+1 in .y).
#pragma once

#include "nvfp4_device.cuh"

namespace nvfp4 {

enum Mode { MODE_RNE = 0, MODE_SR = 1, MODE_4O6 = 2 };

// Unsigned max of magnitude bits: max |v|, with NaN beating every number.
__device__ __forceinline__ uint32_t amax_bits(const f2 (&v)[8]) {
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) m = max(m, max(mag_bits(v[k].x), mag_bits(v[k].y)));
    return m;
}

// Decode scale of the tensor / row: g = A / (6 * 448).
__device__ __forceinline__ float global_scale_of(float A) { return __fdiv_rn(A, 2688.0f); }

// S = e4m3(amax_b / (M * g)); an all-zero block gets 0.
// ("nvfp4-sm120" README, section "Layout": two-level E2M1/E4M3 scaling.)
__device__ __forceinline__ uint32_t block_scale(uint32_t amax_b, float M, float g) {
    if (amax_b == 0u) return 0u;
    float dM = __fmul_rn(M, g);
    return e4m3_rn(__fdiv_rn(__uint_as_float(amax_b), dM));
}

// Random byte of element e (byte e&3 of word e>>2).
__device__ __forceinline__ uint32_t rbyte(const uint4 &r, int e) {
    uint32_t w = (e >> 2) == 0 ? r.x : (e >> 2) == 1 ? r.y : (e >> 2) == 2 ? r.z : r.w;
    return (w >> (8 * (e & 3))) & 0xFFu;
}

// Quotients q = y / (Sf * g) of one block (exactly rounded), then the E2M1
// codes (RNE, or SR with the block's random bytes).  Returns 8 bytes of codes:
// .x = elements 0..7, .y = elements 8..15.
template <bool SR>
__device__ __forceinline__ uint2 encode_with_scale(const f2 (&y)[8], uint32_t S, float g, const uint4 &rnd) {
    const float Sf = e4m3_value(S);
    if (Sf == 0.0f) return make_uint2(0u, 0u);
    const float d = __fmul_rn(Sf, g);
    const Recip R = make_recip(d);
    f2 q[8];
    if (R.fast) {
#pragma unroll
        for (int k = 0; k < 8; k++) q[k] = div2_fast(y[k], R);
    } else {
#pragma unroll
        for (int k = 0; k < 8; k++) q[k] = f2{div_slow(y[k].x, d), div_slow(y[k].y, d)};
    }
    if (SR) {
#pragma unroll
        for (int k = 0; k < 8; k++) q[k] = sr_round2(q[k], rbyte(rnd, 2 * k), rbyte(rnd, 2 * k + 1));
    }
    uint2 c;
    c.x = e2m1x8(q[0].x, q[0].y, q[1].x, q[1].y, q[2].x, q[2].y, q[3].x, q[3].y);
    c.y = e2m1x8(q[4].x, q[4].y, q[5].x, q[5].y, q[6].x, q[6].y, q[7].x, q[7].y);
    return c;
}

// Four-over-six candidate error: squared dequantization error, reduced by
// the clamped shuffle-down tree (offsets 8, 4, 2, 1: lane i += lane i+off).
// (PR #4852 description: pinned width-16 error reduction.)
__device__ __forceinline__ float candidate_error(const f2 (&y)[8], uint2 codes, uint32_t S, float g) {
    const float Sf = e4m3_value(S);
    const float d = (Sf == 0.0f) ? 0.0f : __fmul_rn(Sf, g);
    const f2 dd{d, d};
    f2 p[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const uint32_t w = (k < 4) ? codes.x : codes.y;
        const f2 val = e2m1x2_value(w >> (8 * (k & 3)));
        const f2 e = sub2(y[k], mul2(val, dd));
        p[k] = mul2(e, e);
    }
    // pair k holds (p[2k], p[2k+1]); offset 8 pairs k with k+4, offset 4 with
    // k+2, offset 2 with k+1, offset 1 is the final scalar add.
#pragma unroll
    for (int k = 0; k < 4; k++) p[k] = add2(p[k], p[k + 4]);
#pragma unroll
    for (int k = 0; k < 2; k++) p[k] = add2(p[k], p[k + 2]);
    p[0] = add2(p[0], p[1]);
    return __fadd_rn(p[0].x, p[0].y);
}

// Encode one block in the given mode.  Returns the codes and writes S.
template <int MODE>
__device__ __forceinline__ uint2 encode_block(const f2 (&y)[8], float g, const uint4 &rnd, uint32_t &S_out) {
    const uint32_t am = amax_bits(y);
    if (MODE == MODE_4O6) {
        const uint32_t S6 = block_scale(am, 6.0f, g);
        const uint32_t S4 = block_scale(am, 4.0f, g);
        const uint2 c6 = encode_with_scale<false>(y, S6, g, rnd);
        const uint2 c4 = encode_with_scale<false>(y, S4, g, rnd);
        const float e6 = candidate_error(y, c6, S6, g);
        const float e4 = candidate_error(y, c4, S4, g);
        const bool pick4 = e4 < e6;  // ties and NaN keep map-to-6
        S_out = pick4 ? S4 : S6;
        return pick4 ? c4 : c6;
    } else {
        const uint32_t S = block_scale(am, 6.0f, g);
        S_out = S;
        return encode_with_scale<MODE == MODE_SR>(y, S, g, rnd);
    }
}

// RHT of a block in place: butterfly, then * (+-0.25).
__device__ __forceinline__ void rht16(f2 (&v)[8], uint32_t sign_mask) {
    fwht16(v);
#pragma unroll
    for (int k = 0; k < 8; k++) v[k] = mul2(v[k], rht_mult(sign_mask, k));
}

}  // namespace nvfp4
