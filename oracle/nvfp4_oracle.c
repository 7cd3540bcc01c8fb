/*
 * nvfp4_oracle.c -- plain, slow, single-threaded CPU definition of the NVFP4
 * training quantizer.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load this file's shared library; the product
 * path (the CUDA library and its Python binding) never does, and the two share
 * no code.
 *
 * Every floating-point step is one IEEE-754 binary32 operation rounded to
 * nearest-even: build with -O2 -ffp-contract=off -fno-fast-math so that the
 * compiler neither fuses a*b+c nor reorders anything.
 *
 * Sources (web pages; cited by title and section):
 *  [A] "在 RTX 5090 (SM120) 上补全 NVFP4 量化相关 kernel" (harrychen.xyz),
 *      sections "FP4 量化技术" (the E2M1 value set), "随机舍入" (stochastic
 *      rounding, P(round to b) = (x-a)/(b-a)), "随机 Hadamard 变换" (the 16x16
 *      Hadamard applied to 16-element blocks of the last dimension),
 *      "随机舍入指令：（半）软件模拟" (SR as a random decision followed by a
 *      round-to-nearest cast), "Vibe Coding 过程" (Philox counters, nibble
 *      order, NaN propagation are the known hazards).
 *  [B] "nvfp4-sm120" README, sections "Approach" (BlockWise1x16 scales in the
 *      SWIZZLE_32_4_4 layout), "Layout" (two-level E2M1/E4M3 quantization;
 *      Fprop RNE / Dgrad SR / Wgrad RHT+SR), "Results" (scale kept on device).
 *  [C] "[nvfp4 training][rl] Add a CuTe DSL fast-path kernel for four-over-six
 *      quantize #4852", PR description (four-over-six: map-to-6 and 1.5x-scale
 *      map-to-4 candidates, lower error kept; per-tensor or row-scaled global
 *      scales; correctly rounded FP32 division; pinned width-16 clamped
 *      shuffle-down error reduction).
 *
 * Where the pages leave a step open the reading taken here is the one listed
 * in the design notes; each function says which step it is.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_ERR_ARG 1
#define ORA_ERR_UNSUPPORTED 2

enum { ORA_MODE_RNE = 0, ORA_MODE_SR = 1, ORA_MODE_4O6 = 2 };

/* ------------------------------------------------------------------ bits */

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* bf16 -> fp32 is exact: the bf16 pattern is the top half of the fp32 one. */
static float bf16_to_f32(uint16_t h) { return u2f((uint32_t)h << 16); }

/* fp32 -> bf16, round to nearest even; NaN stays a (quiet) NaN. */
uint16_t ora_f32_to_bf16(float f) {
    uint32_t u = f2u(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* ------------------------------------------------------------------ E2M1 */
/* E2M1 ([A] "FP4 量化技术"): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa
 * bit.  Exponent field 0 is subnormal: value = m * 0.5.  Otherwise
 * value = (1 + m/2) * 2^(e-1).  The eight magnitudes are 0, .5, 1, 1.5, 2, 3,
 * 4, 6, in code order 0..7; bit 3 is the sign. */
float ora_e2m1_value(int code) {
    int e = (code >> 1) & 3, m = code & 1;
    float v = (e == 0) ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * ldexpf(1.0f, e - 1);
    return (code & 8) ? -v : v;
}

/* Largest magnitude code c in [0,6] with value(c) <= m (m finite, 0 <= m < 6). */
static int e2m1_floor_code(float m) {
    int c = 0;
    while (c < 6 && ora_e2m1_value(c + 1) <= m) c++;
    return c;
}

/* Round-to-nearest-even cast with saturation to +-6 (".satfinite").  A tie
 * goes to the even code (mantissa bit 0).  NaN encodes as +6 (code 7): E2M1
 * has no NaN, and the saturating hardware cast behaves the same way. */
int ora_e2m1_rne(float q) {
    if (isnan(q)) return 7;
    int sign = signbit(q) ? 8 : 0;
    float m = fabsf(q);
    if (m >= 6.0f) return sign | 7;
    int c = e2m1_floor_code(m);
    float a = ora_e2m1_value(c), b = ora_e2m1_value(c + 1);
    float mid = (a + b) * 0.5f; /* exact: a and b are short dyadic numbers */
    int r;
    if (m < mid) r = c;
    else if (m > mid) r = c + 1;
    else r = (c & 1) ? c + 1 : c;
    return sign | r;
}

/* Stochastic rounding ([A] "随机舍入"): between the grid neighbours a <= m < b,
 * round up with probability (m-a)/(b-a).  The draw is one random byte r
 * (0..255) per element; up iff frac + (r + 0.5)/256 >= 1, i.e. a uniform
 * dither of the grid step followed by truncation.  The comparison is made as
 * 512*frac >= 511 - 2r, where both sides are exact.  |q| >= 6 saturates. */
int ora_e2m1_sr(float q, unsigned r) {
    if (isnan(q)) return 7;
    int sign = signbit(q) ? 8 : 0;
    float m = fabsf(q);
    if (m >= 6.0f) return sign | 7;
    int c = e2m1_floor_code(m);
    float a = ora_e2m1_value(c), b = ora_e2m1_value(c + 1);
    /* m - a is exact (Sterbenz: a <= m < b <= 2a, or a == 0) and 1/(b-a) is a
     * power of two, so frac is the exact ratio. */
    float frac = (m - a) * (1.0f / (b - a));
    int up = frac * 512.0f >= (float)(511 - 2 * (int)(r & 0xFFu));
    return sign | (up ? c + 1 : c);
}

/* ------------------------------------------------------------------ E4M3 */
/* E4M3 (OCP FP8 "e4m3fn"): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN; no infinities; the
 * largest finite value is 0x7E = 448. */
float ora_e4m3_value(unsigned b) {
    b &= 0xFFu;
    int e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    float v = (e == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
    return (b & 0x80u) ? -v : v;
}

/* Round to nearest, ties to even mantissa, saturating to +-448 (".satfinite":
 * also +-inf -> +-448); NaN -> 0x7F. */
unsigned ora_e4m3_rn(float s) {
    if (isnan(s)) return 0x7Fu;
    unsigned sign = signbit(s) ? 0x80u : 0u;
    float a = fabsf(s);
    if (a >= 448.0f) return sign | 0x7Eu;
    /* binary search for the largest code k with value(k) <= a */
    unsigned lo = 0, hi = 0x7E; /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        unsigned mid = (lo + hi) / 2;
        if (ora_e4m3_value(mid) <= a) lo = mid; else hi = mid;
    }
    float vl = ora_e4m3_value(lo), vh = ora_e4m3_value(hi);
    float mid = (vl + vh) * 0.5f; /* exact: 4-bit significands */
    unsigned k;
    if (a < mid) k = lo;
    else if (a > mid) k = hi;
    else k = (lo & 1u) ? hi : lo;
    return sign | k;
}

/* ---------------------------------------------------------- Philox4x32-10 */
/* Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC'11: ten rounds of two 32x32->64 multiplies (multipliers 0xD2511F53,
 * 0xCD9E8D57) with a Weyl key schedule (0x9E3779B9, 0xBB67AE85). */
void ora_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; round++) {
        if (round > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Random bytes of one 16-element block.  Counter layout: key = (seed low 32,
 * seed high 32); counter = (blk low 32, blk high 32, offset low 32, offset
 * high 32), blk being the row-major index of the block in the OUTPUT
 * orientation.  Element e takes byte e&3 (little end first) of word e>>2. */
static void block_random_bytes(uint64_t seed, uint64_t offset, uint64_t blk, uint8_t rb[16]) {
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)offset, (uint32_t)(offset >> 32)};
    uint32_t o[4];
    ora_philox4x32_10(ctr, key, o);
    for (int e = 0; e < 16; e++) rb[e] = (uint8_t)(o[e >> 2] >> (8 * (e & 3)));
}

/* ------------------------------------------------------------------- RHT */
/* [A] "随机 Hadamard 变换": y = v . H16 / 4 . diag(s).  H16 is the Sylvester
 * Hadamard matrix, H[i][j] = (-1)^popcount(i & j), applied as the in-place
 * butterfly with strides h = 1, 2, 4, 8 (this order is the definition).  Then
 * every output is multiplied by 0.25 and negated where bit j of the sign mask
 * is set.  The 0.25 and the sign are exact. */
void ora_rht16(float v[16], uint32_t sign_mask) {
    for (int h = 1; h < 16; h <<= 1)
        for (int i = 0; i < 16; i++)
            if ((i & h) == 0) {
                float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
    for (int j = 0; j < 16; j++) {
        float t = v[j] * 0.25f;
        v[j] = ((sign_mask >> j) & 1u) ? -t : t;
    }
}

/* ------------------------------------------------------- amax and scales */
/* Magnitude maximum as an unsigned maximum of (bits & 0x7FFFFFFF): equal to
 * max |v| for numbers, and any NaN beats every number, so NaN propagates
 * (the reading taken for the pages' conflicting NaN remarks). */
static uint32_t absbits(float v) { return f2u(v) & 0x7FFFFFFFu; }

/* Per-tensor / per-row decode scale g = A / (6 * 448). */
static float global_scale_of(float A) { return A / 2688.0f; }

/* Block scale byte for the map-to-M grid: S = e4m3(amax_b / (M * g)); an
 * all-zero block gets S = 0. */
static unsigned block_scale(float amax_b, float M, float g) {
    if (f2u(amax_b) == 0u) return 0u;
    float dM = M * g;
    float s = amax_b / dM;
    return ora_e4m3_rn(s);
}

/* Encode n values against block scale S: q = y / (Sf * g), correctly rounded
 * ([C]); Sf == 0 encodes every element as +0. */
static void encode_with_scale(const float *y, int n, unsigned S, float g, int sr,
                              const uint8_t *rb, int *code) {
    float Sf = ora_e4m3_value(S);
    if (Sf == 0.0f) { for (int i = 0; i < n; i++) code[i] = 0; return; }
    float d = Sf * g;
    for (int i = 0; i < n; i++) {
        float q = y[i] / d;
        code[i] = sr ? ora_e2m1_sr(q, rb[i]) : ora_e2m1_rne(q);
    }
}

/* Four-over-six error of one 16-element candidate ([C]): squared error of the
 * dequantized value, summed by the clamped shuffle-down tree with offsets 8,
 * 4, 2, 1 -- lane i adds lane i+off -- so the order is
 * (((p0+p8)+(p4+p12)) + ((p2+p10)+(p6+p14))) + (((p1+p9)+(p5+p13)) + ((p3+p11)+(p7+p15))). */
static float candidate_error(const float *y, const int *code, unsigned S, float g) {
    float Sf = ora_e4m3_value(S);
    float d = (Sf == 0.0f) ? 0.0f : Sf * g;
    float p[16];
    for (int i = 0; i < 16; i++) {
        float deq = ora_e2m1_value(code[i]) * d;
        float e = y[i] - deq;
        p[i] = e * e;
    }
    for (int off = 8; off >= 1; off >>= 1)
        for (int i = 0; i < off; i++) p[i] = p[i] + p[i + off];
    return p[0];
}

/* SWIZZLE_32_4_4 ([B] "Approach"; mapping from the public cuBLAS block-scaling
 * layout): pad to R_p = ceil(R/128)*128 rows and Cs_p = ceil(Cs/4)*4 scale
 * columns, 512-byte tiles of 128 rows x 4 columns in row-major tile order,
 * inside a tile (r%32)*16 + ((r%128)/32)*4 + (j%4). */
int64_t ora_swizzle_offset(int64_t r, int64_t j, int64_t cs_p) {
    return ((r / 128) * (cs_p / 4) + j / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4);
}

int64_t ora_scale_bytes(int64_t rows_out, int64_t cols_out, int swizzled) {
    int64_t cs = cols_out / 16;
    if (!swizzled) return rows_out * cs;
    int64_t rp = (rows_out + 127) / 128 * 128, csp = (cs + 3) / 4 * 4;
    return rp * csp;
}

static void put_scale(uint8_t *scales, int64_t r, int64_t j, int64_t cs, int swizzled, unsigned S) {
    if (swizzled) scales[ora_swizzle_offset(r, j, (cs + 3) / 4 * 4)] = (uint8_t)S;
    else scales[r * cs + j] = (uint8_t)S;
}

static unsigned get_scale(const uint8_t *scales, int64_t r, int64_t j, int64_t cs, int swizzled) {
    return swizzled ? scales[ora_swizzle_offset(r, j, (cs + 3) / 4 * 4)] : scales[r * cs + j];
}

/* ------------------------------------------------------------- the input */
typedef struct {
    const void *x;
    int dtype; /* 0 bf16, 1 fp32 */
    int64_t rows, cols, ld;
    int orient; /* 0: rows of X are the output rows; 1: work on X^T */
} view_t;

/* Element (r, c) of the working matrix W (W = X, or X^T for the columnwise
 * orientation), widened to fp32 exactly. */
static float wget(const view_t *v, int64_t r, int64_t c) {
    int64_t i = v->orient ? c : r, k = v->orient ? r : c;
    if (v->dtype == 0) return bf16_to_f32(((const uint16_t *)v->x)[i * v->ld + k]);
    return ((const float *)v->x)[i * v->ld + k];
}

static void load_block(const view_t *v, int64_t r, int64_t j, int rht, uint32_t mask, float y[16]) {
    for (int e = 0; e < 16; e++) y[e] = wget(v, r, 16 * j + e);
    if (rht) ora_rht16(y, mask);
}

/* ------------------------------------------------------------ quantize */
/* Quantize output rows [r0, r1) of W.
 *   mode: 0 RNE, 1 SR (Philox bytes), 2 four-over-six (RNE candidates).
 *   block2d: one scale per 16x16 tile (replicated to 1x16 in the output).
 *   per_row: one global scale per output row (else one per tensor, computed
 *            over the WHOLE tensor whatever [r0, r1) is).
 * codes: [R_out, C_out/2] bytes, low nibble = even element.  scales: linear
 * [R_out, C_out/16] or swizzled.  amax_out / gscale_out: 1 float (per tensor)
 * or R_out floats (per row; only [r0, r1) written).
 *   block_base: added to every block number of the Philox counter, i.e. the
 *            number of this input's first block when it is a shard of a larger
 *            tensor whose blocks keep their numbers (0 for a whole tensor). */
int ora_quantize(const void *x, int dtype, int64_t rows, int64_t cols, int64_t ld,
                 int orient, int mode, int block2d, int per_row, int swizzled,
                 int rht, uint32_t sign_mask, uint64_t seed, uint64_t offset,
                 int64_t r0, int64_t r1, const float *amax_in,
                 uint8_t *codes, uint8_t *scales, float *amax_out, float *gscale_out, uint64_t block_base) {
    view_t v = {x, dtype, rows, cols, ld, orient};
    int64_t R = orient ? cols : rows, C = orient ? rows : cols;
    if (!x || !codes || !scales || !amax_out || !gscale_out) return ORA_ERR_ARG;
    if (rows < 0 || cols < 0 || ld < cols || C % 16 != 0) return ORA_ERR_ARG;
    if (r0 < 0 || r1 > R || r0 > r1) return ORA_ERR_ARG;
    if (block2d && (R % 16 != 0 || r0 % 16 != 0 || r1 % 16 != 0)) return ORA_ERR_ARG;
    if (block2d && (rht || mode == ORA_MODE_SR || mode == ORA_MODE_4O6 || per_row)) return ORA_ERR_UNSUPPORTED;
    if (mode == ORA_MODE_4O6 && rht) return ORA_ERR_UNSUPPORTED;
    int64_t CS = C / 16;
    float y[16];

    /* Global amax over the post-RHT values (per tensor: everything), unless
     * the caller supplies it (amax_in, per tensor only). */
    float g_tensor = 0.0f;
    if (!per_row && amax_in) {
        amax_out[0] = amax_in[0];
        g_tensor = global_scale_of(amax_in[0]);
        gscale_out[0] = g_tensor;
    } else if (!per_row) {
        uint32_t mb = 0;
        for (int64_t r = 0; r < R; r++)
            for (int64_t j = 0; j < CS; j++) {
                load_block(&v, r, j, rht, sign_mask, y);
                for (int e = 0; e < 16; e++) if (absbits(y[e]) > mb) mb = absbits(y[e]);
            }
        float A = u2f(mb);
        g_tensor = global_scale_of(A);
        amax_out[0] = A;
        gscale_out[0] = g_tensor;
    }

    if (block2d) {
        for (int64_t rt = r0; rt < r1; rt += 16)
            for (int64_t j = 0; j < CS; j++) {
                uint32_t mb = 0;
                for (int64_t r = rt; r < rt + 16; r++)
                    for (int e = 0; e < 16; e++) {
                        uint32_t b = absbits(wget(&v, r, 16 * j + e));
                        if (b > mb) mb = b;
                    }
                unsigned S = block_scale(u2f(mb), 6.0f, g_tensor);
                for (int64_t r = rt; r < rt + 16; r++) {
                    int code[16];
                    for (int e = 0; e < 16; e++) y[e] = wget(&v, r, 16 * j + e);
                    encode_with_scale(y, 16, S, g_tensor, 0, NULL, code);
                    for (int k = 0; k < 8; k++)
                        codes[r * (C / 2) + 8 * j + k] = (uint8_t)(code[2 * k] | (code[2 * k + 1] << 4));
                    put_scale(scales, r, j, CS, swizzled, S);
                }
            }
        return ORA_OK;
    }

    for (int64_t r = r0; r < r1; r++) {
        float g = g_tensor;
        if (per_row) {
            uint32_t mb = 0;
            for (int64_t j = 0; j < CS; j++) {
                load_block(&v, r, j, rht, sign_mask, y);
                for (int e = 0; e < 16; e++) if (absbits(y[e]) > mb) mb = absbits(y[e]);
            }
            amax_out[r] = u2f(mb);
            g = global_scale_of(u2f(mb));
            gscale_out[r] = g;
        }
        for (int64_t j = 0; j < CS; j++) {
            load_block(&v, r, j, rht, sign_mask, y);
            uint32_t mb = 0;
            for (int e = 0; e < 16; e++) if (absbits(y[e]) > mb) mb = absbits(y[e]);
            float amax_b = u2f(mb);
            int code[16];
            unsigned S;
            if (mode == ORA_MODE_4O6) {
                int c6[16], c4[16];
                unsigned S6 = block_scale(amax_b, 6.0f, g), S4 = block_scale(amax_b, 4.0f, g);
                encode_with_scale(y, 16, S6, g, 0, NULL, c6);
                encode_with_scale(y, 16, S4, g, 0, NULL, c4);
                float e6 = candidate_error(y, c6, S6, g), e4 = candidate_error(y, c4, S4, g);
                int pick4 = e4 < e6; /* ties and NaN keep map-to-6 */
                S = pick4 ? S4 : S6;
                memcpy(code, pick4 ? c4 : c6, sizeof code);
            } else {
                uint8_t rb[16];
                if (mode == ORA_MODE_SR) block_random_bytes(seed, offset, block_base + (uint64_t)(r * CS + j), rb);
                S = block_scale(amax_b, 6.0f, g);
                encode_with_scale(y, 16, S, g, mode == ORA_MODE_SR, rb, code);
            }
            for (int k = 0; k < 8; k++)
                codes[r * (C / 2) + 8 * j + k] = (uint8_t)(code[2 * k] | (code[2 * k + 1] << 4));
            put_scale(scales, r, j, CS, swizzled, S);
        }
    }
    return ORA_OK;
}

/* ---------------------------------------------------------- dequantize */
/* The standard NVFP4 decode ([C] "nvfp4_dequantize"): out = value(code) *
 * (Sf * g), both products rounded; g is one float (per tensor) or one per
 * row.  out_dtype 0 writes bf16 (RNE of the fp32 result), 1 writes fp32. */
int ora_dequantize(const uint8_t *codes, const uint8_t *scales, const float *gscale,
                   int64_t rows, int64_t cols, int swizzled, int per_row,
                   void *out, int out_dtype) {
    if (!codes || !scales || !gscale || !out || cols % 16 != 0 || rows < 0) return ORA_ERR_ARG;
    int64_t CS = cols / 16;
    for (int64_t r = 0; r < rows; r++) {
        float g = per_row ? gscale[r] : gscale[0];
        for (int64_t c = 0; c < cols; c++) {
            unsigned byte = codes[r * (cols / 2) + c / 2];
            int code = (c & 1) ? (int)(byte >> 4) : (int)(byte & 15u);
            float Sf = ora_e4m3_value(get_scale(scales, r, c / 16, CS, swizzled));
            float d = Sf * g;
            float o = ora_e2m1_value(code) * d;
            if (out_dtype == 0) ((uint16_t *)out)[r * cols + c] = ora_f32_to_bf16(o);
            else ((float *)out)[r * cols + c] = o;
        }
    }
    return ORA_OK;
}

/* Inverse of the 16-point RHT: y = (v.H16).(1/4).diag(s) gives
 * v = ((y.diag(s)).H16).(1/4), because H16.H16 = 16 I.  Steps: the signs on
 * the inputs, the same butterfly (strides 1, 2, 4, 8), then x 0.25. */
void ora_inverse_rht16(float y[16], uint32_t sign_mask) {
    for (int j = 0; j < 16; j++)
        if ((sign_mask >> j) & 1u) y[j] = -y[j];
    for (int h = 1; h < 16; h <<= 1)
        for (int i = 0; i < 16; i++)
            if ((i & h) == 0) {
                float a = y[i], b = y[i + h];
                y[i] = a + b;
                y[i + h] = a - b;
            }
    for (int j = 0; j < 16; j++) y[j] = y[j] * 0.25f;
}

/* Dequantize of an RHT-quantized rowwise output back to the original basis:
 * the standard decode of each 16-block (as ora_dequantize, fp32), then the
 * inverse RHT of the block; a bf16 output takes RN of the result. */
int ora_dequantize_rht(const uint8_t *codes, const uint8_t *scales, const float *gscale,
                       int64_t rows, int64_t cols, int swizzled, int per_row, uint32_t sign_mask,
                       void *out, int out_dtype) {
    if (!codes || !scales || !gscale || !out || cols % 16 != 0 || rows < 0) return ORA_ERR_ARG;
    int64_t CS = cols / 16;
    float y[16];
    for (int64_t r = 0; r < rows; r++) {
        float g = per_row ? gscale[r] : gscale[0];
        for (int64_t j = 0; j < CS; j++) {
            float Sf = ora_e4m3_value(get_scale(scales, r, j, CS, swizzled));
            float d = Sf * g;
            for (int e = 0; e < 16; e++) {
                unsigned byte = codes[r * (cols / 2) + 8 * j + e / 2];
                int code = (e & 1) ? (int)(byte >> 4) : (int)(byte & 15u);
                y[e] = ora_e2m1_value(code) * d;
            }
            ora_inverse_rht16(y, sign_mask);
            for (int e = 0; e < 16; e++) {
                int64_t c = 16 * j + e;
                if (out_dtype == 0) ((uint16_t *)out)[r * cols + c] = ora_f32_to_bf16(y[e]);
                else ((float *)out)[r * cols + c] = y[e];
            }
        }
    }
    return ORA_OK;
}

/* Global amax alone (per tensor, or per output row), same definition as in
 * ora_quantize. */
int ora_amax(const void *x, int dtype, int64_t rows, int64_t cols, int64_t ld, int orient,
             int rht, uint32_t sign_mask, int per_row, float *amax_out, float *gscale_out) {
    view_t v = {x, dtype, rows, cols, ld, orient};
    int64_t R = orient ? cols : rows, C = orient ? rows : cols;
    if (!x || !amax_out || !gscale_out || C % 16 != 0) return ORA_ERR_ARG;
    float y[16];
    uint32_t mt = 0;
    for (int64_t r = 0; r < R; r++) {
        uint32_t mr = 0;
        for (int64_t j = 0; j < C / 16; j++) {
            load_block(&v, r, j, rht, sign_mask, y);
            for (int e = 0; e < 16; e++) if (absbits(y[e]) > mr) mr = absbits(y[e]);
        }
        if (per_row) { amax_out[r] = u2f(mr); gscale_out[r] = global_scale_of(u2f(mr)); }
        if (mr > mt) mt = mr;
    }
    if (!per_row) { amax_out[0] = u2f(mt); gscale_out[0] = global_scale_of(u2f(mt)); }
    return ORA_OK;
}

/* ------------------------------------------- array forms (for the tests) */
void ora_e2m1_rne_n(const float *q, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)ora_e2m1_rne(q[i]);
}
void ora_e2m1_sr_n(const float *q, const uint8_t *r, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)ora_e2m1_sr(q[i], r[i]);
}
void ora_e4m3_rn_n(const float *s, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; i++) out[i] = (uint8_t)ora_e4m3_rn(s[i]);
}
/* Four-over-six candidate errors of n blocks: block b has values y[16b..],
 * codes code[16b..] (4-bit), block scale S[b] and global scale g[b]. */
void ora_candidate_error_n(const float *y, const int32_t *code, const uint32_t *S, const float *g, int64_t n,
                           float *out) {
    for (int64_t b = 0; b < n; b++) {
        int c[16];
        for (int i = 0; i < 16; i++) c[i] = code[16 * b + i];
        out[b] = candidate_error(y + 16 * b, c, S[b], g[b]);
    }
}
