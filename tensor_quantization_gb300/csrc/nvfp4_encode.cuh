// nvfp4_encode.cuh -- block-level encoders shared by the quantize kernels.
//
// A 1x16 block is held as 8 fp32 pairs (element 2k in .x, 2k+1 in .y).
//
// For one global scale g, the element divisor d = Sf * g takes one of 128
// values (one per non-negative E4M3 byte), so each CTA prepares all of them
// once (DivTable, in shared memory) and a block only looks its divisor up.
#pragma once

#include "nvfp4_device.cuh"

namespace nvfp4 {

enum Mode { MODE_RNE = 0, MODE_SR = 1, MODE_4O6 = 2 };

// Decode scale of the tensor / row: g = A / (6 * 448).
__device__ __forceinline__ float global_scale_of(float A) { return __fdiv_rn(A, 2688.0f); }

// max |v| over a block (NaN if any element is NaN): a tree of 3-input
// max.NaN instructions (sm_100+), written as one asm block so that ptxas
// folds every |.| into their operand modifiers.
__device__ __forceinline__ float block_amax(const f2 (&v)[8]) {
    float m;
    asm("{\n\t.reg .f32 a<16>, b<6>, c<2>;\n\t"
        "abs.f32 a0, %1; abs.f32 a1, %2; abs.f32 a2, %3; abs.f32 a3, %4;\n\t"
        "abs.f32 a4, %5; abs.f32 a5, %6; abs.f32 a6, %7; abs.f32 a7, %8;\n\t"
        "abs.f32 a8, %9; abs.f32 a9, %10; abs.f32 a10, %11; abs.f32 a11, %12;\n\t"
        "abs.f32 a12, %13; abs.f32 a13, %14; abs.f32 a14, %15; abs.f32 a15, %16;\n\t"
        "max.NaN.f32 b0, a0, a1, a2; max.NaN.f32 b1, a3, a4, a5; max.NaN.f32 b2, a6, a7, a8;\n\t"
        "max.NaN.f32 b3, a9, a10, a11; max.NaN.f32 b4, a12, a13, a14;\n\t"
        "max.NaN.f32 c0, b0, b1, b2; max.NaN.f32 c1, b3, b4, a15;\n\t"
        "max.NaN.f32 %0, c0, c1;\n\t}"
        : "=f"(m)
        : "f"(v[0].x), "f"(v[0].y), "f"(v[1].x), "f"(v[1].y), "f"(v[2].x), "f"(v[2].y), "f"(v[3].x), "f"(v[3].y),
          "f"(v[4].x), "f"(v[4].y), "f"(v[5].x), "f"(v[5].y), "f"(v[6].x), "f"(v[6].y), "f"(v[7].x), "f"(v[7].y));
    return m;
}

// The 128 element divisors of one global scale.  Entry s holds
// d = RN(value(s) * g) and its reciprocal pieces; entry 0x7F (NaN) has d = NaN
// and takes the IEEE path.
struct DivTable {
    Divisor e[128];
};

// A divisor times the exact power of two `up` (dn = 1/up): d * up and the
// reciprocal pieces * dn, each exact while everything stays normal.
__device__ __forceinline__ Divisor scale_divisor(Divisor D, float up, float dn) {
    D.d = __fmul_rn(D.d, up);
    D.nrh = __fmul_rn(D.nrh, dn);
    D.nrd = __fmul_rn(D.nrd, dn);
    D.nrl = __fmul_rn(D.nrl, dn);
    return D;
}

// The divisor table of g; with up != 1 every entry is pre-multiplied by the
// fast path's power-of-two factor (FastScale below), so blocks use it as is.
__device__ __forceinline__ void build_table(DivTable &T, float g, int tid, int nthreads, float up = 1.0f) {
    for (int s = tid; s < 128; s += nthreads) {
        Divisor D = make_divisor(__fmul_rn(e4m3_value((uint32_t)s), g));
        if (up != 1.0f) D = scale_divisor(D, up, 1.0f / up);
        T.e[s] = D;
    }
}

// The same entries computed when they are looked up (a block whose global
// scale has no table in shared memory); T.e[s] gives the bits of the table's
// entry s.
struct DivDirect {
    struct Entries {
        float g, up;
        __device__ __forceinline__ Divisor operator[](uint32_t s) const {
            Divisor D = make_divisor(__fmul_rn(e4m3_value(s), g));
            if (up != 1.0f) D = scale_divisor(D, up, 1.0f / up);
            return D;
        }
    } e;
};

// Divisors M*g of the block-scale computation (M = 6, and 4 for four-over-six).
struct ScaleDiv {
    Divisor m6, m4;
    bool fast6, fast4;
};

__device__ __forceinline__ ScaleDiv make_scale_div(float g) {
    ScaleDiv s;
    s.m6 = make_divisor(__fmul_rn(6.0f, g));
    s.m4 = make_divisor(__fmul_rn(4.0f, g));
    s.fast6 = divisor_fast(s.m6.d);
    s.fast4 = divisor_fast(s.m4.d);
    return s;
}

// S = e4m3(amax_b / (M * g)); an all-zero block gets 0; NaN gives 0x7F.
// ("nvfp4-sm120" README, section "Layout": two-level E2M1/E4M3 scaling.)
__device__ __forceinline__ uint32_t block_scale(float amax_b, const Divisor &dm, bool fast) {
    if (amax_b == 0.0f) return 0u;
    return e4m3_rn(fast ? quot_pos(amax_b, dm) : __fdiv_rn(amax_b, dm.d));
}

// E2M1 codes of one block against divisor D (S != 0): exactly rounded
// quotients (negated, see neg_quot2), stochastic rounding when SR, the RN
// cast, and one XOR per 8 codes to restore the sign.  .x = elements 0..7.
template <bool SR>
__device__ __forceinline__ uint2 encode_codes(const f2 (&y)[8], const Divisor &D, const uint4 &rnd) {
    f2 nq[8];
    if (divisor_fast(D.d)) {
#pragma unroll
        for (int k = 0; k < 8; k++) nq[k] = neg_quot2(y[k], D);
    } else {
#pragma unroll
        for (int k = 0; k < 8; k++) nq[k] = f2{neg_quot_slow(y[k].x, D.d), neg_quot_slow(y[k].y, D.d)};
    }
    if (SR) {
#pragma unroll
        for (int k = 0; k < 8; k++) nq[k] = sr_round2(nq[k], dither8(rnd, 2 * k), dither8(rnd, 2 * k + 1));
    }
    uint2 c;
    c.x = e2m1x8(nq[0].x, nq[0].y, nq[1].x, nq[1].y, nq[2].x, nq[2].y, nq[3].x, nq[3].y) ^ 0x88888888u;
    c.y = e2m1x8(nq[4].x, nq[4].y, nq[5].x, nq[5].y, nq[6].x, nq[6].y, nq[7].x, nq[7].y) ^ 0x88888888u;
    return c;
}

template <bool SR, typename Tab>
__device__ __forceinline__ uint2 encode_with_scale(const f2 (&y)[8], uint32_t S, const Tab &T, const uint4 &rnd) {
    if (S == 0u) return make_uint2(0u, 0u);
    return encode_codes<SR>(y, T.e[S & 0x7Fu], rnd);
}

// Four-over-six candidate error: squared dequantization error, reduced by
// the clamped shuffle-down tree (offsets 8, 4, 2, 1: lane i += lane i+off).
// (PR #4852 description: pinned width-16 error reduction.)  Every product and
// sum must round on its own.  ptxas contracts a packed f32x2 multiply into a
// packed add, subtract or FMA that consumes it, even with .rn on both, which
// would round y - val*d (or a square plus its partner) once instead of twice
// and change which candidate wins a near-tie.  So only the dequantized value
// is a packed multiply, and it feeds an FMA as a multiplicand:
//   t = RN(val*d);  e = RN(t*(-1) + y) = RN(y - t);  p = RN(e*e + 0)
// (e*e >= 0, so adding +0 is exact), and the tree adds FMA results only.
// A GPU test compares this with the oracle on a million blocks.  d = 0 when
// S = 0.
__device__ __forceinline__ float candidate_error(const f2 (&y)[8], uint2 codes, float d) {
    const f2 dd{d, d}, m1{-1.0f, -1.0f}, z{0.0f, 0.0f};
    f2 p[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const uint32_t w = (k < 4) ? codes.x : codes.y;
        const f2 e = fma2(mul2(e2m1x2_value(w >> (8 * (k & 3))), dd), m1, y[k]);
        p[k] = fma2(e, e, z);
    }
    // p[k] holds elements 2k, 2k+1: offsets 8, 4, 2 pair p[k] with p[k+4],
    // p[k+2], p[k+1]; offset 1 adds the two halves of p[0]
#pragma unroll
    for (int k = 0; k < 4; k++) p[k] = add2(p[k], p[k + 4]);
    p[0] = add2(p[0], p[2]);
    p[1] = add2(p[1], p[3]);
    p[0] = add2(p[0], p[1]);
    return __fadd_rn(p[0].x, p[0].y);
}

// The same error from the negated candidate values nv = -val (f16x2 pairs,
// as the fast encoder's cast produces them from the negated quotients):
// t = RN(nv * (-d)) = RN(val * d), then exactly the steps above.  (Written as
// t * (+1) + y with t = RN(nv * d), ptxas folds the multiply by one and
// contracts the product into a single FMA.)
__device__ __forceinline__ float candidate_error_neg(const f2 (&y)[8], const uint32_t (&nv)[8], float d) {
    const f2 ndd{-d, -d}, m1{-1.0f, -1.0f}, z{0.0f, 0.0f};
    f2 p[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
        const f2 e = fma2(mul2(f16x2_to_f2(nv[k]), ndd), m1, y[k]);
        p[k] = fma2(e, e, z);
    }
#pragma unroll
    for (int k = 0; k < 4; k++) p[k] = add2(p[k], p[k + 4]);
    p[0] = add2(p[0], p[2]);
    p[1] = add2(p[1], p[3]);
    p[0] = add2(p[0], p[1]);
    return __fadd_rn(p[0].x, p[0].y);
}

// Encode one block in the given mode.  Returns the codes and writes S.
template <int MODE, typename Tab>
__device__ __forceinline__ uint2 encode_block(const f2 (&y)[8], const ScaleDiv &sd, const Tab &T, const uint4 &rnd,
                                              uint32_t &S_out) {
    const float am = block_amax(y);
    if (MODE == MODE_4O6) {
        const uint32_t S6 = block_scale(am, sd.m6, sd.fast6);
        const uint32_t S4 = block_scale(am, sd.m4, sd.fast4);
        const uint2 c6 = encode_with_scale<false>(y, S6, T, rnd);
        const uint2 c4 = encode_with_scale<false>(y, S4, T, rnd);
        const float e6 = candidate_error(y, c6, S6 ? T.e[S6 & 0x7Fu].d : 0.0f);
        const float e4 = candidate_error(y, c4, S4 ? T.e[S4 & 0x7Fu].d : 0.0f);
        const bool pick4 = e4 < e6;  // ties and NaN keep map-to-6
        S_out = pick4 ? S4 : S6;
        return pick4 ? c4 : c6;
    } else {
        const uint32_t S = block_scale(am, sd.m6, sd.fast6);
        S_out = S;
        return encode_with_scale<MODE == MODE_SR>(y, S, T, rnd);
    }
}

// ---------------------------------------------------------------- fast path
// When every divisor of a global scale g is in the fast division range (true
// unless the tensor's amax is extreme, NaN or infinite), blocks skip the
// per-block range test.  With S != 0x7F guaranteed (the block amax is finite),
// an all-zero block is the only special case and is masked to +0 codes.
__device__ __forceinline__ bool scale_all_fast(float g) {
    // smallest divisor 2^-9 * g, largest 448 * g (x 2^16 for the folded RHT
    // and the fp16 stochastic rounding)
    return g >= 0x1p-71f && g <= 0x1p73f;  // false for NaN
}

// The RHT's outputs are y_j = s_j * 0.25 * v'_j (v' = butterfly output).  On
// the fast path the 0.25 goes into the divisor (y/d = v'/(4d) exactly: a
// quotient that could differ, from a v' so small that 0.25 * v' rounds, is
// below 2^-40 and keeps its sign, so its code cannot change) and the signs s_j
// into the code-sign flip.  `signs` holds bit 4e+3 for every negated element
// e of the 8 in one code word.
// The divisor's exact power-of-two factor on the fast path: 4 for the folded
// RHT, 2^14 for stochastic rounding through fp16 (sr_pair_f16).
template <int MODE, bool RHT>
struct FastScale {
    static constexpr float up = MODE == MODE_SR ? (RHT ? 0x1p16f : 0x1p14f) : (RHT ? 4.0f : 1.0f);
};

// PRE: D already carries the factor (a table built with FastScale::up).
template <bool SR, bool AP = false, bool PRE = false>
__device__ __forceinline__ uint2 encode_fast(const f2 (&v)[8], Divisor D, uint32_t S, bool fold4,
                                             uint2 signs, const uint4 &rnd) {
    const float up = SR ? (fold4 ? 0x1p16f : 0x1p14f) : (fold4 ? 4.0f : 1.0f);
    const float dn = SR ? (fold4 ? 0x1p-16f : 0x1p-14f) : (fold4 ? 0.25f : 1.0f);
    if ((SR || fold4) && !PRE) D = scale_divisor(D, up, dn);
    f2 nq[8];
    if (AP) {  // fast math: -(y * RN(1/d)), one multiply
#pragma unroll
        for (int k = 0; k < 8; k++) nq[k] = mul2(v[k], f2{D.nrh, D.nrh});
    } else {
#pragma unroll
        for (int k = 0; k < 8; k++) nq[k] = neg_quot2(v[k], D);
    }
    const uint32_t keep = S ? 0xFFFFFFFFu : 0u;
    uint2 c;
    if (SR) {
        uint32_t h[8];
#pragma unroll
        for (int k = 0; k < 8; k++) h[k] = sr_pair_f16(nq[k], rnd, k);
        c.x = (e2m1x8_f16(h[0], h[1], h[2], h[3]) ^ 0x88888888u ^ signs.x) & keep;
        c.y = (e2m1x8_f16(h[4], h[5], h[6], h[7]) ^ 0x88888888u ^ signs.y) & keep;
        return c;
    }
    c.x = (e2m1x8(nq[0].x, nq[0].y, nq[1].x, nq[1].y, nq[2].x, nq[2].y, nq[3].x, nq[3].y) ^ 0x88888888u ^ signs.x) & keep;
    c.y = (e2m1x8(nq[4].x, nq[4].y, nq[5].x, nq[5].y, nq[6].x, nq[6].y, nq[7].x, nq[7].y) ^ 0x88888888u ^ signs.y) & keep;
    return c;
}

// RNE codes of one block (no RHT) plus the negated grid values of every
// pair for the four-over-six error (the codes are cast from -q and flipped).
__device__ __forceinline__ uint2 encode_fast_vals(const f2 (&v)[8], const Divisor &D, uint32_t S,
                                                  uint32_t (&nv)[8]) {
    f2 nq[8];
#pragma unroll
    for (int k = 0; k < 8; k++) nq[k] = neg_quot2(v[k], D);
    const uint32_t keep = S ? 0xFFFFFFFFu : 0u;
    uint2 c;
    c.x = (e2m1x8_vals(nq, 0, nv) ^ 0x88888888u) & keep;
    c.y = (e2m1x8_vals(nq, 4, nv) ^ 0x88888888u) & keep;
    return c;
}

// One block on the fast path.  v holds the raw block (RHT: the butterfly is
// applied here and the 0.25 / signs are folded as above; STAGE1: v already
// holds the butterfly's first stage).  AP (fast math) replaces the exact
// element quotient by y * RN(1/d); block scales stay exact.
template <int MODE, bool RHT, bool AP = false, bool STAGE1 = false, bool PRE = false, typename Tab = DivTable>
__device__ __forceinline__ uint2 encode_block_fast(f2 (&v)[8], const ScaleDiv &sd, const Tab &T, uint2 signs,
                                                   const uint4 &rnd, uint32_t &S_out) {
    if (RHT && !STAGE1) fwht16_first(v);
    if (RHT) fwht16_rest(v);
    float am = block_amax(v);
    if (RHT) am = __fmul_rn(am, 0.25f);  // = max |y|: rounding is monotone
    if (MODE == MODE_4O6) {
        const uint32_t S6 = am == 0.0f ? 0u : e4m3_rn(quot_pos(am, sd.m6));
        const uint32_t S4 = am == 0.0f ? 0u : e4m3_rn(quot_pos(am, sd.m4));
        const Divisor D6 = T.e[S6], D4 = T.e[S4];
        uint32_t n6[8], n4[8];  // negated candidate values, straight from the casts
        const uint2 c6 = encode_fast_vals(v, D6, S6, n6);
        const uint2 c4 = encode_fast_vals(v, D4, S4, n4);
        const float e6 = candidate_error_neg(v, n6, S6 ? D6.d : 0.0f);
        const float e4 = candidate_error_neg(v, n4, S4 ? D4.d : 0.0f);
        const bool pick4 = e4 < e6;  // ties keep map-to-6
        S_out = pick4 ? S4 : S6;
        return pick4 ? c4 : c6;
    } else {
        const uint32_t S = am == 0.0f ? 0u : e4m3_rn(quot_pos(am, sd.m6));
        S_out = S;
        return encode_fast<MODE == MODE_SR, AP, PRE>(v, T.e[S], S, RHT, signs, rnd);
    }
}

// Code-word sign flips for the RHT sign mask: bit 4e+3 for negated element e.
__device__ __forceinline__ uint2 rht_sign_words(uint32_t mask) {
    uint2 w = make_uint2(0u, 0u);
#pragma unroll
    for (int e = 0; e < 8; e++) {
        w.x |= ((mask >> e) & 1u) << (4 * e + 3);
        w.y |= ((mask >> (8 + e)) & 1u) << (4 * e + 3);
    }
    return w;
}

// The 16 RHT output multipliers (+-0.25 by the sign mask), prepared once per
// CTA in shared memory and read back as 4 x 128-bit per block.
struct RhtMult {
    f2 m[8];
};

__device__ __forceinline__ void build_rht_mult(RhtMult &M, uint32_t sign_mask, int tid) {
    if (tid < 8) M.m[tid] = rht_mult(sign_mask, tid);
}

// RHT of a block in place: butterfly, then * (+-0.25).
__device__ __forceinline__ void rht16(f2 (&v)[8], const RhtMult &M) {
    fwht16(v);
#pragma unroll
    for (int k = 0; k < 8; k++) v[k] = mul2(v[k], M.m[k]);
}

}  // namespace nvfp4
