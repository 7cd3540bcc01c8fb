// gpu_probes.cu -- test-only kernels that run the library's device primitives
// on arrays, so the tests can compare them with the CPU oracle (casts) and
// with CUDA's own IEEE division.  Compiled by tests/test_gpu_primitives.py.
#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"
#include "nvfp4_encode.cuh"

using namespace nvfp4;

__global__ void k_e2m1(const float *q, int64_t n, uint8_t *out) {
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= n) return;
    // element 0 of the packed word = low nibble; feed q twice to also check
    // that element 1 lands in the high nibble
    uint32_t w = e2m1x8(q[i], q[i], 0.f, 0.f, 0.f, 0.f, 0.f, 0.f);
    uint32_t lo = w & 15u, hi = (w >> 4) & 15u;
    out[i] = (lo == hi) ? (uint8_t)lo : (uint8_t)0xFF;
}

__global__ void k_e2m1_order(uint32_t *out) {
    // eight distinct values: codes 1..7 and 0x9 must appear in element order
    out[0] = e2m1x8(0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f, -0.5f);
}

__global__ void k_sr(const float *q, const uint8_t *r, int64_t n, uint8_t *out) {
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= n) return;
    f2 v = sr_round2(f2{q[i], 0.f}, dither8(make_uint4(r[i], 0u, 0u, 0u), 0), 0x80u);  // symmetric: also used on -q
    out[i] = (uint8_t)(e2m1x8(v.x, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 15u);
}

// The fp16 stochastic-rounding pair on q * 2^-14 (as the scaled divisor
// delivers it): element i is paired with a zero partner, alternately in the
// low and the high half (random byte 0 or 1 of word 0), so both lanes and
// both nibbles are checked.
__global__ void k_sr_f16(const float *q, const uint8_t *r, int64_t n, uint8_t *out) {
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float qs = q[i] * 0x1p-14f;
    const bool hi = i & 1;
    const uint4 rw = make_uint4(hi ? (uint32_t)r[i] << 8 : (uint32_t)r[i], 0u, 0u, 0u);
    const uint32_t h = sr_pair_f16(hi ? f2{0.f, qs} : f2{qs, 0.f}, rw, 0);
    const uint32_t w = e2m1x8_f16(h, 0u, 0u, 0u);
    out[i] = (uint8_t)((hi ? w >> 4 : w) & 15u);
}

// The f16x2 -> e2m1x2 cast on every f16 pattern (paired with +0), in both halves.
__global__ void k_e2m1_f16(uint8_t *out) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;  // 0 .. 65535
    const uint32_t lo = e2m1x8_f16(i, 0u, 0u, 0u) & 15u;
    const uint32_t hi = (e2m1x8_f16(i << 16, 0u, 0u, 0u) >> 4) & 15u;
    out[i] = (uint8_t)(lo == hi ? lo : 0xFFu);
}

__global__ void k_e4m3(const float *s, int64_t n, uint8_t *out) {
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i < n) out[i] = (uint8_t)e4m3_rn(s[i]);
}

__global__ void k_e4m3_value(float *out) { out[threadIdx.x] = e4m3_value(threadIdx.x); }

__global__ void k_e2m1_value(float *out) {
    f2 v = e2m1x2_value(threadIdx.x);
    out[2 * threadIdx.x] = v.x;
    out[2 * threadIdx.x + 1] = v.y;
}

__device__ __forceinline__ uint32_t mix(uint64_t x) {
    x ^= x >> 33; x *= 0xff51afd7ed558ccdull; x ^= x >> 33; x *= 0xc4ceb9fe1a85ec53ull; x ^= x >> 33;
    return (uint32_t)x;
}

// Exact division: the library's per-block path (fast when the divisor range
// allows, IEEE otherwise; both return -RN(y/d)) against __fdiv_rn.  Kinds:
// 0 random significands, 1 near-midpoint quotients (y = RN(d*m), m a
// midpoint), 2 random d over the whole fast range, 3 signed zeros.  Quotients
// below 2^-11 only need to stay below 2^-10 with the right sign.  The scalar
// block-scale quotient (positive numerators) is checked on the same pairs.
__global__ void k_div(uint64_t seed, int64_t n, int kind, unsigned long long *bad, float *first) {
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= n) return;
    uint32_t a = mix(seed * 0x9E3779B97F4A7C15ull + 2 * i), b = mix(seed ^ (0xD1B54A32D192ED03ull * (2 * i + 1)));
    float d, y;
    if (kind == 2) {
        d = __uint_as_float(((mix(a) % 180u) + 47u) << 23 | (b & 0x7FFFFFu));   // 2^-80 .. 2^100
    } else if (kind == 4) {
        d = __uint_as_float(((mix(a) % 61u) + 107u) << 23 | (b & 0x7FFFFFu));   // 2^-20 .. 2^40
    } else {
        d = __uint_as_float((127u << 23) | (b & 0x7FFFFFu)) * __uint_as_float(((a >> 27) + 112u) << 23);
    }
    if (kind == 1) {
        // m = the midpoint between a float f in [1, 2) and its successor (not an
        // fp32 value), scaled by 2^k, k in [-12, 3]; y = RN(d * m) puts y / d
        // close to m, often within far less than an ulp.  Every third pair
        // uses d = 1 + j * 2^-23 (few significant bits), which makes d * m
        // nearly representable more often.
        if (a % 3u == 0u) d = 1.0f + (float)(b & 63u) * 0x1p-23f;
        const double m = ((double)__uint_as_float((127u << 23) | (a & 0x7FFFFFu)) + 0x1p-24) *
                         (double)__uint_as_float((uint32_t)(115 + (mix(b) & 15u)) << 23);
        y = __double2float_rn((double)d * m);
    } else if (kind == 3) {
        y = 0.0f;
    } else if (kind == 4) {
        // small quotients, 2^-60 .. 2^-11, with |y| >= 2^-80: the range the
        // stochastic-rounding fast path uses at its 2^-14 scale; exact there
        float q = __uint_as_float(((mix(b) % 50u) + 67u) << 23 | (a & 0x7FFFFFu));
        y = __fmul_rn(d, q);
    } else {
        float q = __uint_as_float((127u << 23) | (a & 0x7FFFFFu)) * __uint_as_float((uint32_t)(112 + (b >> 28)) << 23);
        y = __fmul_rn(d, q);
    }
    if (a & 1u) y = -y;
    const Divisor D = make_divisor(d);
    const bool fast = divisor_fast(d);
    const f2 nq = fast ? neg_quot2(f2{y, y}, D) : f2{neg_quot_slow(y, d), neg_quot_slow(y, d)};
    const float ref = __fdiv_rn(y, d);
    const float want = -(fast ? ref : fminf(fmaxf(ref, -8.f), 8.f));
    bool ok;
    if (kind != 4 && fabsf(ref) < 0x1p-11f && ref != 0.0f) ok = fabsf(nq.x) < 0x1p-10f && signbit(nq.x) != signbit(ref);
    else ok = __float_as_uint(nq.x) == __float_as_uint(want);
    ok = ok && __float_as_uint(nq.x) == __float_as_uint(nq.y);
    if (fast && fabsf(ref) >= 0x1p-11f && isfinite(ref)) {
        const float ay = fabsf(y);
        ok = ok && __float_as_uint(quot_pos(ay, D)) == __float_as_uint(__fdiv_rn(ay, d));
    }
    if (!ok) {
        unsigned long long k = atomicAdd(bad, 1ull);
        if (k < 4) { first[3 * k] = y; first[3 * k + 1] = d; first[3 * k + 2] = nq.x; }
    }
}

// Four-over-six candidate error of block i: values y[16i..], codes packed two
// per byte (low nibble first) in codes[i], element divisor d[i].
// The fast path's form: the candidate's values negated (codes with their
// sign bits flipped), decoded to f16x2 pairs.
__global__ void k_cand_err_neg(const float *y, const uint2 *codes, const float *d, int64_t n, float *out) {
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= n) return;
    f2 v[8];
    uint32_t nv[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
        v[k] = f2{y[16 * i + 2 * k], y[16 * i + 2 * k + 1]};
        const uint32_t w = ((k < 4) ? codes[i].x : codes[i].y) ^ 0x88888888u;
        asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(nv[k]) : "r"((w >> (8 * (k & 3))) & 0xFFu));
    }
    out[i] = candidate_error_neg(v, nv, d[i]);
}

__global__ void k_cand_err(const float *y, const uint2 *codes, const float *d, int64_t n, float *out) {
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= n) return;
    f2 v[8];
#pragma unroll
    for (int k = 0; k < 8; k++) v[k] = f2{y[16 * i + 2 * k], y[16 * i + 2 * k + 1]};
    out[i] = candidate_error(v, codes[i], d[i]);
}

extern "C" {
int probe_cand_err_neg(const float *y, const uint2 *codes, const float *d, int64_t n, float *out) {
    k_cand_err_neg<<<(unsigned)((n + 255) / 256), 256>>>(y, codes, d, n, out);
    return cudaDeviceSynchronize();
}
int probe_cand_err(const float *y, const uint2 *codes, const float *d, int64_t n, float *out) {
    k_cand_err<<<(unsigned)((n + 255) / 256), 256>>>(y, codes, d, n, out);
    return cudaDeviceSynchronize();
}
int probe_e2m1(const float *q, int64_t n, uint8_t *out) {
    k_e2m1<<<(unsigned)((n + 255) / 256), 256>>>(q, n, out);
    return cudaDeviceSynchronize();
}
int probe_sr_f16(const float *q, const uint8_t *r, int64_t n, uint8_t *out) {
    k_sr_f16<<<(unsigned)((n + 255) / 256), 256>>>(q, r, n, out);
    return cudaDeviceSynchronize();
}
int probe_e2m1_f16(uint8_t *out) {
    k_e2m1_f16<<<256, 256>>>(out);
    return cudaDeviceSynchronize();
}
int probe_e2m1_order(uint32_t *out) {
    k_e2m1_order<<<1, 1>>>(out);
    return cudaDeviceSynchronize();
}
int probe_sr(const float *q, const uint8_t *r, int64_t n, uint8_t *out) {
    k_sr<<<(unsigned)((n + 255) / 256), 256>>>(q, r, n, out);
    return cudaDeviceSynchronize();
}
int probe_e4m3(const float *s, int64_t n, uint8_t *out) {
    k_e4m3<<<(unsigned)((n + 255) / 256), 256>>>(s, n, out);
    return cudaDeviceSynchronize();
}
int probe_e4m3_value(float *out) {
    k_e4m3_value<<<1, 256>>>(out);
    return cudaDeviceSynchronize();
}
int probe_e2m1_value(float *out) {
    k_e2m1_value<<<1, 256>>>(out);
    return cudaDeviceSynchronize();
}
int probe_div(uint64_t seed, int64_t n, int kind, unsigned long long *bad, float *first) {
    k_div<<<(unsigned)((n + 255) / 256), 256>>>(seed, n, kind, bad, first);
    return cudaDeviceSynchronize();
}
}
