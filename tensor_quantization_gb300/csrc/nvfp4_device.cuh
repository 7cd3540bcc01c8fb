// nvfp4_device.cuh -- sm_103a device primitives of the NVFP4 quantizer.
//
// Rounding-critical steps use explicit instructions so that no compiler
// lowering choice can change a result: the hardware E4M3/E2M1 casts
// (cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32) and their exact decodes, an exactly
// rounded division, and fixed butterfly / reduction orders.
// ("[nvfp4 training][rl] Add a CuTe DSL fast-path kernel for four-over-six
// quantize #4852", PR description.)
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

// ------------------------------------------------------------------ bits
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t mag_bits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }
// max(|a|, |b|) that returns NaN if either is NaN.
__device__ __forceinline__ float absmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)));
    return r;
}

// ------------------------------------------------------ packed fp32 pairs
// Blackwell executes two fp32 lanes per instruction (add/sub/mul/fma .f32x2).
struct f2 { float x, y; };

__device__ __forceinline__ unsigned long long pk(f2 a) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
    return r;
}
__device__ __forceinline__ f2 upk(unsigned long long r) {
    f2 a;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
    return a;
}
__device__ __forceinline__ f2 add2(f2 a, f2 b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk(a)), "l"(pk(b)));
    return upk(r);
}
__device__ __forceinline__ f2 sub2(f2 a, f2 b) {
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk(a)), "l"(pk(b)));
    return upk(r);
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk(a)), "l"(pk(b)));
    return upk(r);
}
__device__ __forceinline__ f2 mulrz2(f2 a, f2 b) {
    unsigned long long r;
    asm("mul.rz.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk(a)), "l"(pk(b)));
    return upk(r);
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk(a)), "l"(pk(b)), "l"(pk(c)));
    return upk(r);
}

// ------------------------------------------------------------------ E4M3
// Round-to-nearest-even, saturating (+-inf -> +-448), NaN -> 0x7F.
__device__ __forceinline__ uint32_t e4m3_rn(float s) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
    return r & 0xFFu;
}

// Exact value of an E4M3 byte (E4M3 is a subset of fp16).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
    uint32_t h2;
    uint16_t in = (uint16_t)(b & 0xFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    float f;
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.f32.f16 %0, lo; }" : "=f"(f) : "r"(h2));
    return f;
}

// ------------------------------------------------------------------ E2M1
// Eight fp32 values -> eight RNE/satfinite E2M1 codes packed in a word,
// element k in nibble k (low nibble first).
__device__ __forceinline__ uint32_t e2m1x8(float q0, float q1, float q2, float q3, float q4, float q5,
                                           float q6, float q7) {
    uint32_t w;
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3}; }"
        : "=r"(w)
        : "f"(q0), "f"(q1), "f"(q2), "f"(q3), "f"(q4), "f"(q5), "f"(q6), "f"(q7));
    return w;
}

// Eight fp32 values -> eight codes as e2m1x8, plus each pair's decoded grid
// values as f16x2 (low half = even element), taken from the cast's own byte
// before it is packed.
__device__ __forceinline__ uint32_t e2m1x8_vals(const f2 (&q)[8], int p0, uint32_t (&h)[8]) {
    uint32_t w;
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %8, %7;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %10, %9;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %12, %11;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %4, b3;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3}; }"
        : "=r"(w), "=r"(h[p0]), "=r"(h[p0 + 1]), "=r"(h[p0 + 2]), "=r"(h[p0 + 3])
        : "f"(q[p0].x), "f"(q[p0].y), "f"(q[p0 + 1].x), "f"(q[p0 + 1].y), "f"(q[p0 + 2].x), "f"(q[p0 + 2].y),
          "f"(q[p0 + 3].x), "f"(q[p0 + 3].y));
    return w;
}

// The two fp32 values of an f16x2 word (low half -> .x).
__device__ __forceinline__ f2 f16x2_to_f2(uint32_t h2) {
    f2 v;
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }"
        : "=f"(v.x), "=f"(v.y)
        : "r"(h2));
    return v;
}

// Exact fp32 values of the two codes in byte `b` (low nibble -> .x).
__device__ __forceinline__ f2 e2m1x2_value(uint32_t b) {
    uint32_t h2;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h2) : "r"(b & 0xFFu));
    f2 v;
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }"
        : "=f"(v.x), "=f"(v.y) : "r"(h2));
    return v;
}

// ------------------------------------------------- exactly rounded y / d
// A block divides all of its elements by the same d = Sf * g, and d takes at
// most 128 values per global scale, so the reciprocal is prepared once per d:
//   rd = RD(1/d), rl = RN((1 - d*rd) * rd) >= 0  (the remainder 1 - d*rd is
//   exact by FMA and non-negative), rh = RN(1/d).
// Per element (two at a time, packed):
//   q0 = RN(y*rd + RN(y*rl))   relative error < 2^-46: a faithful rounding of
//                              y/d, with the sign of y even for y = -0
//                              (both products carry y's sign);
//   f  = y - q0*d              exact (remainder of a faithful quotient);
//   q  = RN(q0 + f*rh)         = RN(y/d) by Markstein's theorem (Markstein
//                              1990; Muller et al., Handbook of
//                              Floating-Point Arithmetic, division chapter).
// The sequence is evaluated on negated reciprocals and returns -q, which keeps
// every signed zero exact without a sign fix-up; callers flip the code sign.
// Fast-path precondition: d in [2^-80, 2^100], y finite.  With |y| >= 2^-100
// and |y/d| >= 2^-100 nothing underflows (t and rl err by far less than the
// quotient's ulp, the remainder is representable, the result is normal), so
// the result is exact.  Otherwise |y/d| < 2^-20 and the computed value stays
// that small with the sign of y, which fixes its E2M1 code and its E4M3
// rounding (both 0), also at the 2^-14 scale of sr_pair_f16; a quotient that
// overflows becomes +-inf, which the saturating casts encode as +-6.
struct Divisor {
    float d, nrh, nrd, nrl;  // d, -RN(1/d), -RD(1/d), -rl
};

__device__ __forceinline__ Divisor make_divisor(float d) {
    Divisor D;
    D.d = d;
    const float rd = __frcp_rd(d);
    const float rem = __fmaf_rn(-d, rd, 1.0f);
    D.nrh = -__frcp_rn(d);
    D.nrd = -rd;
    D.nrl = -__fmul_rn(rem, rd);
    return D;
}

__device__ __forceinline__ bool divisor_fast(float d) { return d >= 0x1p-80f && d <= 0x1p100f; }  // NaN: false

// -RN(y/d) for two numerators (fast path).
__device__ __forceinline__ f2 neg_quot2(f2 y, const Divisor &D) {
    const f2 t = mul2(y, f2{D.nrl, D.nrl});
    const f2 nq = fma2(y, f2{D.nrd, D.nrd}, t);
    const f2 f = fma2(nq, f2{D.d, D.d}, y);
    return fma2(f, f2{D.nrh, D.nrh}, nq);
}

// RN(a/d) for a > 0 (scalar, fast path).
__device__ __forceinline__ float quot_pos(float a, const Divisor &D) {
    const float nq = __fmaf_rn(a, D.nrd, __fmul_rn(a, D.nrl));
    const float f = __fmaf_rn(nq, D.d, a);
    return -__fmaf_rn(f, D.nrh, nq);
}

// -RN(y/d) by IEEE division for divisors outside the fast range, clamped to
// [-8, 8] (every |q| >= 6 encodes as 6); NaN becomes -8 so that it encodes as
// +6 once the code sign is flipped.
__device__ __forceinline__ float neg_quot_slow(float y, float d) {
    const float q = __fdiv_rn(y, d);
    if (q != q) return -8.0f;
    return -fminf(fmaxf(q, -8.0f), 8.0f);
}

// --------------------------------------------------- stochastic rounding
// The dither of element e, (r + 0.5) * 2^8 for its random byte r = byte
// (e & 3) of word (e >> 2): one PRMT puts the byte above a constant 0x80 byte.
__device__ __forceinline__ uint32_t dither8(const uint4 &r, int e) {
    const uint32_t w = (e >> 2) == 0 ? r.x : (e >> 2) == 1 ? r.y : (e >> 2) == 2 ? r.z : r.w;
    return __byte_perm(0x80u, w, 0x1140u + 16u * (uint32_t)(e & 3));
}

// Scaling |q| < 8 by 2^-126 (rounding toward zero) puts the E2M1 grid at the
// floats whose low 22 bits are zero, subnormal step 0.5 included; adding the
// dither (r + 0.5) * 2^14 (= dither8 << 6) to the bits and truncating gives
//   up  <=>  (|q| - a)/(b - a) + (r + 0.5)/256 >= 1
// (the truncation only drops bits below the 2^-13 step of the dither, which
// cannot change a ">=" against it).  Returns the chosen grid value, signed.
__device__ __forceinline__ f2 sr_round2(f2 q, uint32_t d0, uint32_t d1) {
    f2 z = mulrz2(q, f2{0x1p-126f, 0x1p-126f});
    uint32_t t0 = ((d0 << 6) + __float_as_uint(z.x)) & 0xFFC00000u;
    uint32_t t1 = ((d1 << 6) + __float_as_uint(z.y)) & 0xFFC00000u;
    return mul2(f2{__uint_as_float(t0), __uint_as_float(t1)}, f2{0x1p126f, 0x1p126f});
}

// The same decision two elements at a time through fp16 (fast path).  The
// divisor carries a factor 2^14, so the negated quotients arrive as
// -q * 2^-14, exact (a power-of-two scaling of RN(y/d) in the normal range;
// only |q| < 2^-112 could round differently, and every such q encodes as 0).
// Converting the pair to f16x2 toward zero truncates each |q| * 2^-14 to a
// multiple of 2^-10 grid steps: q = 1 is the smallest normal f16, so below it
// the subnormal step holds the 0.5 grid step at bit 9, and above it each
// binade keeps one mantissa bit above bit 9.  Adding 2r + 1 to each 16-bit
// lane (the same dither (r + 0.5)/256 of a grid step; no carry leaves a lane)
// and clearing the low 9 bits makes the same decision as sr_round2.  The grid
// values times 2^14 (exact in f16) then go through the f16x2 -> e2m1x2 cast
// (satfinite: 8 and 12 encode as 6).  Pair k holds elements 2k (low half) and
// 2k + 1, whose random bytes are bytes 2k & 3 and (2k & 3) + 1 of word k / 2.
__device__ __forceinline__ uint32_t sr_pair_f16(f2 nq, const uint4 &r, int k) {
    uint32_t h;
    asm("cvt.rz.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(nq.y), "f"(nq.x));
    const uint32_t w = (k >> 1) == 0 ? r.x : (k >> 1) == 1 ? r.y : (k >> 1) == 2 ? r.z : r.w;
    const uint32_t bb = (uint32_t)(2 * k) & 3u;
    const uint32_t t = __byte_perm(w, 0u, 0x4040u | bb | ((bb + 1u) << 8));  // r_odd << 16 | r_even
    const uint32_t m = (h + (t << 1) + 0x00010001u) & 0xFE00FE00u;
    uint32_t o;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o) : "r"(m), "r"(0x74007400u));  // x 2^14
    return o;
}

// Four f16x2 pairs -> eight RNE/satfinite E2M1 codes, element k in nibble k
// (the high half of a pair is the high nibble of its byte).
__device__ __forceinline__ uint32_t e2m1x8_f16(uint32_t h0, uint32_t h1, uint32_t h2, uint32_t h3) {
    uint32_t w;
    asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f16x2 b0, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f16x2 b1, %2;\n\t"
        "cvt.rn.satfinite.e2m1x2.f16x2 b2, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f16x2 b3, %4;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3}; }"
        : "=r"(w)
        : "r"(h0), "r"(h1), "r"(h2), "r"(h3));
    return w;
}

// ----------------------------------------------------------- Philox4x32-10
// Salmon et al., "Parallel random numbers: as easy as 1, 2, 3" (SC'11).
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int i = 0; i < 10; i++) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        c1 = (uint32_t)p1;
        c3 = (uint32_t)p0;
        c0 = n0;
        c2 = n2;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(c0, c1, c2, c3);
}

// The same with the ten round keys given (k0[i] = seed lo + i * 0x9E3779B9,
// k1[i] = seed hi + i * 0xBB67AE85).
__device__ __forceinline__ uint4 philox4x32_10_keyed(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                     const uint32_t (&k0)[10], const uint32_t (&k1)[10]) {
#pragma unroll
    for (int i = 0; i < 10; i++) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0[i];
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1[i];
        c1 = (uint32_t)p1;
        c3 = (uint32_t)p0;
        c0 = n0;
        c2 = n2;
    }
    return make_uint4(c0, c1, c2, c3);
}

// Random bytes of block `blk`: key = seed, counter = (blk, offset).
__device__ __forceinline__ uint4 block_random(uint64_t seed, uint64_t offset, uint64_t blk) {
    return philox4x32_10((uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)offset, (uint32_t)(offset >> 32),
                         (uint32_t)seed, (uint32_t)(seed >> 32));
}

// ------------------------------------------------------------ 16-point RHT
// Butterfly with strides 1, 2, 4, 8 (this order defines the rounding).  The
// block is held as 8 pairs v[k] = (y[2k], y[2k+1]); the stride-1 stage works
// inside a pair, the later stages on whole pairs with packed adds.
__device__ __forceinline__ void fwht16_first(f2 (&v)[8]) {
#pragma unroll
    for (int k = 0; k < 8; k++) {
        float a = v[k].x, b = v[k].y;
        v[k].x = __fadd_rn(a, b);
        v[k].y = __fsub_rn(a, b);
    }
}

__device__ __forceinline__ void fwht16_rest(f2 (&v)[8]) {
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            if ((k & h) == 0) {
                f2 a = v[k], b = v[k + h];
                v[k] = add2(a, b);
                v[k + h] = sub2(a, b);
            }
        }
    }
}

__device__ __forceinline__ void fwht16(f2 (&v)[8]) {
    fwht16_first(v);
    fwht16_rest(v);
}

// Per-pair multipliers (+-0.25) from the sign mask: bit j -> element j.
__device__ __forceinline__ f2 rht_mult(uint32_t mask, int k) {
    return f2{((mask >> (2 * k)) & 1u) ? -0.25f : 0.25f, ((mask >> (2 * k + 1)) & 1u) ? -0.25f : 0.25f};
}

// -------------------------------------------------------------- layouts
__device__ __forceinline__ int64_t swizzle_offset(int64_t r, int64_t j, int64_t cs_p) {
    return ((r >> 7) * (cs_p >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (j & 3);
}
// The same in 32-bit arithmetic, for scale arrays below 4 GiB.
__device__ __forceinline__ uint32_t swizzle_offset32(uint32_t r, uint32_t j, uint32_t cs_p) {
    return ((r >> 7) * (cs_p >> 2) + (j >> 2)) * 512u + (r & 31u) * 16u + ((r & 127u) >> 5) * 4u + (j & 3u);
}

}  // namespace nvfp4
