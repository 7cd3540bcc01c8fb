// nvfp4_quant_col.cuh -- columnwise (X^T) 1x16 quantize and 16x16 (2D) tiles
// (included by nvfp4_quant_col.cu for exact division and
// nvfp4_quant_col_approx.cu for NVFP4_FAST_MATH, selected by AP).
//
// Both kernels walk tiles of 128 X rows x one 128-byte column span (64 bf16 or
// 32 fp32 columns) that TMA copies into shared memory, two stages per CTA.  A
// thread takes an 8-byte half chunk of the 16 rows of one row block: each of
// its columns is one 16-element block of an X^T row (columnwise), and 16/HC
// neighbouring threads hold one 16x16 tile (2D).  Column-layout outputs are
// staged in a shared-memory output tile and leave as 128-byte row pieces.
#pragma once

#include "nvfp4_encode.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_load.cuh"
#include "nvfp4_tensor_amax.cuh"
#include "nvfp4_tma.cuh"

namespace nvfp4 {
namespace {  // internal linkage: each including unit has its own kernels

// ------------------------------------------------------------ columnwise
// Tiles of 128 X rows x one 128-byte column span (64 bf16 / 32 fp32 columns)
// arrive by TMA (128-byte swizzle) into one of two stages.  Thread t reads the
// 8-byte half chunk hc = t % 16 of the 16 rows of row block rbl = t / 16 and
// encodes the HC columns in it: each is one 16-element block of an X^T row.
// Codes and scales go to a shared-memory output tile first (RBT row blocks x
// 8 bytes per output row, slots XOR-swizzled so the writes do not collide in
// a bank), then out to global memory as 16-byte pieces, so every output row
// gets RBT x 8 contiguous bytes per tile.  A tile has RBT row blocks and the
// CTA 16 x RBT threads.  Both kernels use RBT = 8 (128-row tiles, four CTAs
// per SM): against RBT = 16 the 2D kernel measured 5% and the columnwise one
// 1% faster per step; RBT = 4 was slower.
constexpr int kColRBT = 8;

template <typename T, int RBT>
struct ColTile {
    static constexpr int TR = 16 * RBT;               // X rows per tile
    static constexpr int NT = 16 * RBT;               // threads per CTA
    static constexpr int TC = 128 / (int)sizeof(T);  // X columns per tile
    static constexpr int HC = 8 / (int)sizeof(T);    // X columns per thread
    static constexpr int kStageBytes = TR * 128;
    static constexpr int kPitch = RBT * 8;            // output tile: TC rows x RBT blocks x 8 bytes
    static constexpr int kCodeBytes = TC * kPitch;
    static constexpr int kScaleBytes = TC * RBT;
    static constexpr int kSmemBytes = 2 * (kStageBytes + kCodeBytes + kScaleBytes) + 1024;
};

// Column cc (0..HC-1) of a thread's 16 x 8-byte strip as block pairs.
template <typename T>
__device__ __forceinline__ void strip_block(const uint2 (&w)[16], int cc, f2 (&v)[8]) {
#pragma unroll
    for (int m = 0; m < 8; m++) {
        if (sizeof(T) == 2) {
            const uint32_t a = (cc < 2) ? w[2 * m].x : w[2 * m].y, b = (cc < 2) ? w[2 * m + 1].x : w[2 * m + 1].y;
            v[m] = (cc & 1) ? f2{__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u)}
                            : f2{__uint_as_float(a << 16), __uint_as_float(b << 16)};
        } else {
            v[m] = (cc == 0) ? f2{__uint_as_float(w[2 * m].x), __uint_as_float(w[2 * m + 1].x)}
                             : f2{__uint_as_float(w[2 * m].y), __uint_as_float(w[2 * m + 1].y)};
        }
    }
}

// The same block with the butterfly's first stage applied, (a, b) ->
// (a + b, a - b) on rows 2m, 2m + 1: for bf16 the even row's element enters
// the adds as a bf16 operand of a mixed-precision add (it widens exactly, so
// the result is the fp32 sum), which saves unpacking it.
template <typename T>
__device__ __forceinline__ void strip_fwht_first(const uint2 (&w)[16], int cc, f2 (&v)[8]) {
    if (sizeof(T) != 2) {
        strip_block<T>(w, cc, v);
        fwht16_first(v);
        return;
    }
#pragma unroll
    for (int m = 0; m < 8; m++) {
        const uint32_t a = (cc < 2) ? w[2 * m].x : w[2 * m].y, b = (cc < 2) ? w[2 * m + 1].x : w[2 * m + 1].y;
        const float fb = (cc & 1) ? bf16_hi(b) : bf16_lo(b);
        if (cc & 1)
            asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; add.rn.f32.bf16 %0, hi, %3; sub.rn.f32.bf16 %1, hi, %3; }"
                : "=f"(v[m].x), "=f"(v[m].y)
                : "r"(a), "f"(fb));
        else
            asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; add.rn.f32.bf16 %0, lo, %3; sub.rn.f32.bf16 %1, lo, %3; }"
                : "=f"(v[m].x), "=f"(v[m].y)
                : "r"(a), "f"(fb));
    }
}

// Writes a staged output tile of the columnwise layout: output rows
// o0..o0+TC-1, row blocks rb0..rb0+RBT-1 (codes as 16-byte pieces, scales as
// words; narrower stores where alignment or the tensor edge requires).  Row
// block rbl of output row ol sits in slot rbl ^ ((ol / HC) % RBT): the writing
// thread's half chunk XOR-swizzles the slots.
template <typename T, int RBT>
__device__ __forceinline__ void write_col_tile(const QArgs &a, const uint8_t *ocs, const uint8_t *oss, uint32_t o0,
                                               uint32_t rb0, uint32_t C, uint32_t RB, uint32_t csp,
                                               int64_t code_pitch, bool codes16, bool words, bool lin_words,
                                               int tid) {
    using CT = ColTile<T, RBT>;
    constexpr int TC = CT::TC, HC = CT::HC, NT = CT::NT, PIECES = RBT / 2, WORDS = RBT / 4;
    // codes: output row ol takes RBT/2 pieces of 16 bytes (row blocks 2q, 2q+1)
    for (int i = tid; i < TC * PIECES; i += NT) {
        const int ol = i / PIECES, q = i % PIECES;
        const uint32_t o = o0 + ol, rba = rb0 + 2 * q;
        if (o >= C || rba >= RB) continue;
        const int f = (ol / HC) & (RBT - 1);
        uint4 v = *reinterpret_cast<const uint4 *>(ocs + ol * CT::kPitch + (((2 * q) ^ (f & (RBT - 2))) << 3));
        if (f & 1) v = make_uint4(v.z, v.w, v.x, v.y);
        uint8_t *dst = a.codes_col + (int64_t)o * code_pitch + (int64_t)rba * 8;
        if (codes16 && rba + 1 < RB) {
            *reinterpret_cast<uint4 *>(dst) = v;
        } else {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(v.x, v.y);
            if (rba + 1 < RB) *reinterpret_cast<uint2 *>(dst + 8) = make_uint2(v.z, v.w);
        }
    }
    // scales: output row ol takes RBT/4 words (row blocks 4q..4q+3)
    for (int i = tid; i < TC * WORDS; i += NT) {
        const int ol = i / WORDS, q = i % WORDS;
        const uint32_t o = o0 + ol, rbq = rb0 + 4 * q;
        if (o >= C || rbq >= RB) continue;
        const uint32_t word = (uint32_t)oss[(4 * q) * TC + ol] | ((uint32_t)oss[(4 * q + 1) * TC + ol] << 8) |
                              ((uint32_t)oss[(4 * q + 2) * TC + ol] << 16) |
                              ((uint32_t)oss[(4 * q + 3) * TC + ol] << 24);
        if (a.swizzled) {  // bytes past RB are pad (zero) and inside the padded row
            uint8_t *dst = a.scales_col + swizzle_offset32(o, rbq, csp);
            if (words) {
                *reinterpret_cast<uint32_t *>(dst) = word;
            } else {
#pragma unroll
                for (int b = 0; b < 4; b++) dst[b] = (uint8_t)(word >> (8 * b));
            }
        } else {
            uint8_t *dst = a.scales_col + (size_t)o * RB + rbq;
            if (lin_words && rbq + 3 < RB) {
                *reinterpret_cast<uint32_t *>(dst) = word;
            } else {
                for (int b = 0; b < 4 && rbq + b < RB; b++) dst[b] = (uint8_t)(word >> (8 * b));
            }
        }
    }
}

// Columnwise kernel: the TMA tiles and thread layout above, but a thread
// encodes its HC columns two at a time (one 32-bit strip word per row for
// bf16), and stores each block's 8 code bytes and its scale byte straight
// from registers: the 16 lanes of a half warp write 16 different output rows,
// and the eight row blocks of a tile complete each row's 64 contiguous bytes
// while they sit in L2.  No shared output tile and half the strip live at a
// time, so five CTAs fit per SM instead of four.  Pad bytes of a swizzled
// scale layout are written by the pad kernel.
template <typename T>
struct ColStrip {  // the 16 rows of two adjacent columns of a thread's half chunk
    uint32_t w[16][sizeof(T) / 2];
};

template <typename T>
__device__ __forceinline__ void load_strip(const uint8_t *stage, int rbl, int hc, int pass, ColStrip<T> &st) {
#pragma unroll
    for (int r = 0; r < 16; r++) {
        const int row = rbl * 16 + r;
        const uint8_t *p = stage + row * 128 + ((((hc >> 1) ^ (row & 7)) << 4) | ((hc & 1) << 3));
        if (sizeof(T) == 2) {
            st.w[r][0] = *reinterpret_cast<const uint32_t *>(p + 4 * pass);
        } else {
            const uint2 v = *reinterpret_cast<const uint2 *>(p);
            st.w[r][0] = v.x;
            st.w[r][sizeof(T) / 2 - 1] = v.y;
        }
    }
}

// Column h (0, 1) of a strip as block pairs (rows 2m, 2m+1); with FIRST the
// butterfly's first stage applied (bf16: the even row's element enters the
// adds as a bf16 operand, which widens exactly).
template <typename T, bool FIRST>
__device__ __forceinline__ void strip_column(const ColStrip<T> &st, int h, f2 (&v)[8]) {
#pragma unroll
    for (int m = 0; m < 8; m++) {
        if (sizeof(T) == 2) {
            const uint32_t a = st.w[2 * m][0], b = st.w[2 * m + 1][0];
            if (!FIRST) {
                v[m] = h ? f2{bf16_hi(a), bf16_hi(b)} : f2{bf16_lo(a), bf16_lo(b)};
            } else {
                const float fb = h ? bf16_hi(b) : bf16_lo(b);
                if (h)
                    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; add.rn.f32.bf16 %0, hi, %3; sub.rn.f32.bf16 %1, hi, %3; }"
                        : "=f"(v[m].x), "=f"(v[m].y) : "r"(a), "f"(fb));
                else
                    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; add.rn.f32.bf16 %0, lo, %3; sub.rn.f32.bf16 %1, lo, %3; }"
                        : "=f"(v[m].x), "=f"(v[m].y) : "r"(a), "f"(fb));
            }
        } else {
            v[m] = f2{__uint_as_float(st.w[2 * m][h]), __uint_as_float(st.w[2 * m + 1][h])};
        }
    }
    if (FIRST && sizeof(T) != 2) fwht16_first(v);
}

template <int MODE, bool RHT, typename T, bool AP>
__global__ void __launch_bounds__(16 * kColRBT) k_quant_col(const __grid_constant__ CUtensorMap tmap, const QArgs a) {
    constexpr int RBT = kColRBT;
    using CT = ColTile<T, RBT>;
    constexpr int TC = CT::TC, HC = CT::HC, PASSES = HC / 2;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ DivTable tab;
    __shared__ RhtMult rm;
    __shared__ __align__(8) uint64_t full[2];
    uint8_t *in = dyn_smem + ((1024u - (smem_addr(dyn_smem) & 1023u)) & 1023u);
    const uint32_t R = (uint32_t)a.rows, C = (uint32_t)a.cols, RB = R >> 4, csp = (RB + 3) & ~3u;
    const uint32_t ntc = (C + TC - 1) / TC, ntr = (R + CT::TR - 1) / CT::TR;
    const uint32_t ntiles = ntc * ntr;
    const int tid = threadIdx.x, hc = tid & 15, rbl = tid >> 4;
    if (tid == 0) {
        for (int s = 0; s < 2; s++) mbar_init(&full[s], 1);
        mbar_init_fence();
        for (int k = 0; k < 2; k++) {
            const uint32_t t = blockIdx.x + k * gridDim.x;
            if (t < ntiles) {
                mbar_arrive_expect_tx(&full[k], CT::kStageBytes);
                tma_load_2d(in + k * CT::kStageBytes, &tmap, (int32_t)(((ntiles - 1 - t) % ntc) * TC),
                            (int32_t)(((ntiles - 1 - t) / ntc) * CT::TR), &full[k]);
            }
        }
    }
    const uint2 signs = RHT ? rht_sign_words(a.sign_mask) : make_uint2(0u, 0u);
    if (RHT) build_rht_mult(rm, a.sign_mask, tid);
    grid_dependency_wait();
    const float A = tensor_amax_read(a, RHT);
    const float g = global_scale_of(A);
    build_table(tab, g, tid, blockDim.x);
    const ScaleDiv sd = make_scale_div(g);
    const bool fast = scale_all_fast(g);
    __syncthreads();
    tensor_amax_done(a, A, g);

    const int64_t code_pitch = R >> 1;
    for (uint32_t k = 0;; ++k) {
        const uint32_t t = blockIdx.x + k * gridDim.x;
        if (t >= ntiles) break;
        const uint32_t s = k & 1u;
        if (!mbar_wait(&full[s], (k >> 1) & 1u)) {
            wait_gave_up(a, a.gscale);
        }
        // tiles from the end of the tensor: the amax pass read the tail last, so
        // with a tensor larger than L2 the first tiles here still come from L2
        const uint32_t tr = (ntiles - 1 - t) / ntc, tc = (ntiles - 1 - t) - tr * ntc;
        const uint32_t rb = tr * RBT + rbl, o0 = tc * TC;
        const uint8_t *stage = in + s * CT::kStageBytes;
#pragma unroll
        for (int pass = 0; pass < PASSES; pass++) {
            ColStrip<T> st;
            load_strip<T>(stage, rbl, hc, pass, st);
            uint4 rnd[2];
#pragma unroll
            for (int h = 0; h < 2; h++) {
                rnd[h] = make_uint4(0u, 0u, 0u, 0u);
                if (MODE == MODE_SR) {
                    const uint64_t blk = a.blk_base + (uint64_t)(o0 + HC * hc + 2 * pass + h) * RB + rb;
                    rnd[h] = philox4x32_10_keyed((uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)a.offset,
                                                 (uint32_t)(a.offset >> 32), a.round_key0, a.round_key1);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint32_t o = o0 + HC * hc + 2 * pass + h;  // output row = X column
                if (rb < RB && o < C) {
                    uint32_t S = 0;
                    uint2 c;
                    f2 v[8];
                    if (fast && RHT) {
                        strip_column<T, true>(st, h, v);
                        c = encode_block_fast<MODE, RHT, AP, true>(v, sd, tab, signs, rnd[h], S);
                    } else if (fast) {
                        strip_column<T, false>(st, h, v);
                        c = encode_block_fast<MODE, RHT, AP>(v, sd, tab, signs, rnd[h], S);
                    } else {
                        strip_column<T, false>(st, h, v);
                        if (RHT) rht16(v, rm);
                        c = encode_block<MODE>(v, sd, tab, rnd[h], S);
                    }
                    *reinterpret_cast<uint2 *>(a.codes_col + (int64_t)o * code_pitch + (int64_t)rb * 8) = c;
                    a.scales_col[a.swizzled ? swizzle_offset32(o, rb, csp) : o * RB + rb] = (uint8_t)S;
                }
            }
        }
        __syncthreads();  // stage s consumed
        if (tid == 0) {
            const uint32_t tn = t + 2 * gridDim.x;
            if (tn < ntiles) {
                fence_async_shared();
                mbar_arrive_expect_tx(&full[s], CT::kStageBytes);
                tma_load_2d(in + s * CT::kStageBytes, &tmap, (int32_t)(((ntiles - 1 - tn) % ntc) * TC),
                            (int32_t)(((ntiles - 1 - tn) / ntc) * CT::TR), &full[s]);
            }
        }
    }
}

// ------------------------------------------------------------ 16x16 tiles
// The same TMA tiles and thread layout as the columnwise kernel.  The 16/HC
// lanes whose strips make up one 16x16 tile combine their magnitude maxima
// with shuffles; the tile's scale S (one divisor for all 256 values) is used
// for both orientations, so every element is divided once and its quotient is
// cast twice: paired along a row for the row codes (written directly; the 16
// lanes of a row block fill 32 or 16 contiguous bytes of each row) and paired
// along a column for the column codes (staged in the shared-memory output
// tile).  Column codes are thereby the exact transpose of the row codes.
template <typename T>
__device__ __forceinline__ f2 strip_pair(const uint2 &w, int p) {
    if (sizeof(T) == 2) {
        const uint32_t x = p == 0 ? w.x : w.y;
        return f2{__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u)};
    }
    return f2{__uint_as_float(w.x), __uint_as_float(w.y)};
}

template <typename T, bool AP>
__global__ void __launch_bounds__(16 * kColRBT, 5) k_quant_2d(const __grid_constant__ CUtensorMap tmap, const QArgs a) {
    constexpr int RBT = kColRBT;
    using CT = ColTile<T, RBT>;
    constexpr int TC = CT::TC, HC = CT::HC, NP = HC / 2, LPT = 16 / HC;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ DivTable tab;
    __shared__ __align__(8) uint64_t full[2];
    uint8_t *in = dyn_smem + ((1024u - (smem_addr(dyn_smem) & 1023u)) & 1023u);
    uint8_t *oc = in + 2 * CT::kStageBytes;
    uint8_t *os = oc + 2 * CT::kCodeBytes;
    const uint32_t R = (uint32_t)a.rows, C = (uint32_t)a.cols, RB = R >> 4, CB = C >> 4;
    const uint32_t csp = (RB + 3) & ~3u, csp_row = (CB + 3) & ~3u;
    const uint32_t ntc = (C + TC - 1) / TC, ntr = (R + CT::TR - 1) / CT::TR;
    const uint32_t ntiles = ntc * ntr;
    const int tid = threadIdx.x, hc = tid & 15, rbl = tid >> 4, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < 2; s++) mbar_init(&full[s], 1);
        mbar_init_fence();
        for (int k = 0; k < 2; k++) {
            const uint32_t t = blockIdx.x + k * gridDim.x;
            if (t < ntiles) {
                mbar_arrive_expect_tx(&full[k], CT::kStageBytes);
                tma_load_2d(in + k * CT::kStageBytes, &tmap, (int32_t)(((ntiles - 1 - t) % ntc) * TC),
                            (int32_t)(((ntiles - 1 - t) / ntc) * CT::TR), &full[k]);
            }
        }
    }
    grid_dependency_wait();
    const float A = tensor_amax_read(a, false);
    const float g = global_scale_of(A);
    build_table(tab, g, tid, blockDim.x);
    const ScaleDiv sd = make_scale_div(g);
    const bool fast = scale_all_fast(g);
    __syncthreads();
    tensor_amax_done(a, A, g);

    const int64_t code_pitch = R >> 1, row_pitch = C >> 1;
    const bool codes16 = (code_pitch & 15) == 0 && (reinterpret_cast<uintptr_t>(a.codes_col) & 15u) == 0;
    const bool words = (reinterpret_cast<uintptr_t>(a.scales_col) & 3u) == 0;
    const bool lin_words = words && (RB & 3u) == 0;
    constexpr int RSB = TC / 16;  // row-scale bytes per row of one TMA tile (4 bf16, 2 fp32)
    const bool rs_vec = (reinterpret_cast<uintptr_t>(a.scales_row) & (RSB - 1)) == 0;
    const bool rs_lin_vec = rs_vec && (CB % RSB) == 0;
    for (uint32_t k = 0;; ++k) {
        const uint32_t t = blockIdx.x + k * gridDim.x;
        if (t >= ntiles) break;
        const uint32_t s = k & 1u;
        if (!mbar_wait(&full[s], (k >> 1) & 1u)) {
            wait_gave_up(a, a.gscale);
        }
        // tiles from the end of the tensor: the amax pass read the tail last, so
        // with a tensor larger than L2 the first tiles here still come from L2
        const uint32_t tr = (ntiles - 1 - t) / ntc, tc = (ntiles - 1 - t) - tr * ntc;
        const uint32_t rb0 = tr * RBT, o0 = tc * TC, rb = rb0 + rbl, ob = o0 + HC * hc;
        const bool valid = rb < RB && ob < C;  // C % 16 == 0: a 16x16 tile is all in or all out
        const uint8_t *stage = in + s * CT::kStageBytes;
        uint8_t *ocs = oc + s * CT::kCodeBytes;
        uint8_t *oss = os + s * CT::kScaleBytes;
        uint2 w[16];
#pragma unroll
        for (int r = 0; r < 16; r++) {
            const int row = rbl * 16 + r;
            w[r] = *reinterpret_cast<const uint2 *>(stage + row * 128 + ((((hc >> 1) ^ (row & 7)) << 4) |
                                                                           ((hc & 1) << 3)));
        }
        // tile amax: unsigned max of magnitude bits (NaN above +inf)
        uint32_t m = 0;
        if (sizeof(T) == 2) {
#pragma unroll
            for (int r = 0; r < 16; r++) {
                uint32_t t2;
                asm("max.u16x2 %0, %1, %2;" : "=r"(t2) : "r"(w[r].x & 0x7FFF7FFFu), "r"(w[r].y & 0x7FFF7FFFu));
                asm("max.u16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(t2));
            }
            m = max(m & 0xFFFFu, m >> 16) << 16;
        } else {
#pragma unroll
            for (int r = 0; r < 16; r++) m = max(m, max(w[r].x & 0x7FFFFFFFu, w[r].y & 0x7FFFFFFFu));
        }
#pragma unroll
        for (int off = 1; off < LPT; off <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
        const uint32_t S = valid ? block_scale(__uint_as_float(m), sd.m6, sd.fast6) : 0u;
        const Divisor D = tab.e[S & 0x7Fu];
        const bool dfast = fast || divisor_fast(D.d);
        const uint32_t keep = S ? 0xFFFFFFFFu : 0u;
        uint2 cw[HC];
#pragma unroll
        for (int h = 0; h < 2; h++) {
            f2 q[8][NP];
#pragma unroll
            for (int r = 0; r < 8; r++)
#pragma unroll
                for (int p = 0; p < NP; p++) {
                    const f2 y = strip_pair<T>(w[8 * h + r], p);
                    q[r][p] = !dfast ? f2{neg_quot_slow(y.x, D.d), neg_quot_slow(y.y, D.d)}
                              : AP ? mul2(y, f2{D.nrh, D.nrh}) : neg_quot2(y, D);
                }
            // column codes: nibble r of column cc = row 8h + r
#pragma unroll
            for (int cc = 0; cc < HC; cc++) {
                const int p = cc >> 1;
                const bool hi = cc & 1;
                const uint32_t word =
                    (e2m1x8(hi ? q[0][p].y : q[0][p].x, hi ? q[1][p].y : q[1][p].x, hi ? q[2][p].y : q[2][p].x,
                            hi ? q[3][p].y : q[3][p].x, hi ? q[4][p].y : q[4][p].x, hi ? q[5][p].y : q[5][p].x,
                            hi ? q[6][p].y : q[6][p].x, hi ? q[7][p].y : q[7][p].x) ^
                     0x88888888u) & keep;
                if (h == 0) cw[cc].x = word; else cw[cc].y = word;
            }
            // row codes: HC nibbles per row, written straight to the row
            if (a.want_row && valid) {
                uint8_t *dst = a.codes_row + (int64_t)(rb * 16 + 8 * h) * row_pitch + (ob >> 1);
                if (HC == 4) {
#pragma unroll
                    for (int r = 0; r < 8; r += 2) {
                        const uint32_t word = (e2m1x8(q[r][0].x, q[r][0].y, q[r][NP - 1].x, q[r][NP - 1].y,
                                                      q[r + 1][0].x, q[r + 1][0].y, q[r + 1][NP - 1].x,
                                                      q[r + 1][NP - 1].y) ^ 0x88888888u) & keep;
                        *reinterpret_cast<uint16_t *>(dst + r * row_pitch) = (uint16_t)word;
                        *reinterpret_cast<uint16_t *>(dst + (r + 1) * row_pitch) = (uint16_t)(word >> 16);
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < 8; r += 4) {
                        const uint32_t word = (e2m1x8(q[r][0].x, q[r][0].y, q[r + 1][0].x, q[r + 1][0].y,
                                                      q[r + 2][0].x, q[r + 2][0].y, q[r + 3][0].x,
                                                      q[r + 3][0].y) ^ 0x88888888u) & keep;
#pragma unroll
                        for (int b = 0; b < 4; b++) dst[(r + b) * row_pitch] = (uint8_t)(word >> (8 * b));
                    }
                }
            }
        }
        // row scales: lane hc of the 16-lane group writes row 16 rb + hc; the
        // group's tiles sit at lanes 0, LPT, 2 LPT, ...
        if (a.want_row) {
            uint32_t rs = 0;
#pragma unroll
            for (int i = 0; i < RSB; i++) rs |= __shfl_sync(0xFFFFFFFFu, S, (lane & 16) + LPT * i) << (8 * i);
            if (rb < RB) {
                const uint32_t r = rb * 16 + hc, cb0 = o0 >> 4;
                if (a.swizzled) {  // cb0 % RSB == 0: the RSB bytes are contiguous; pad columns carry 0
                    uint8_t *dst = a.scales_row + swizzle_offset32(r, cb0, csp_row);
                    if (rs_vec) {
                        if (RSB == 4) *reinterpret_cast<uint32_t *>(dst) = rs;
                        else *reinterpret_cast<uint16_t *>(dst) = (uint16_t)rs;
                    } else {
#pragma unroll
                        for (int i = 0; i < RSB; i++) dst[i] = (uint8_t)(rs >> (8 * i));
                    }
                } else {
                    uint8_t *dst = a.scales_row + (size_t)r * CB + cb0;
                    if (rs_lin_vec && cb0 + RSB <= CB) {
                        if (RSB == 4) *reinterpret_cast<uint32_t *>(dst) = rs;
                        else *reinterpret_cast<uint16_t *>(dst) = (uint16_t)rs;
                    } else {
                        for (int i = 0; i < RSB && cb0 + i < CB; i++) dst[i] = (uint8_t)(rs >> (8 * i));
                    }
                }
            }
        }
        if (a.want_col) {
#pragma unroll
            for (int cc = 0; cc < HC; cc++) {
                const int ol = HC * hc + cc;
                *reinterpret_cast<uint2 *>(ocs + ol * CT::kPitch + ((rbl ^ (hc & (RBT - 1))) << 3)) = cw[cc];
                oss[rbl * TC + ol] = (uint8_t)S;
            }
        }
        __syncthreads();  // output tile complete, stage s consumed
        if (tid == 0) {
            const uint32_t tn = t + 2 * gridDim.x;
            if (tn < ntiles) {
                fence_async_shared();
                mbar_arrive_expect_tx(&full[s], CT::kStageBytes);
                tma_load_2d(in + s * CT::kStageBytes, &tmap, (int32_t)(((ntiles - 1 - tn) % ntc) * TC),
                            (int32_t)(((ntiles - 1 - tn) / ntc) * CT::TR), &full[s]);
            }
        }
        if (a.want_col)
            write_col_tile<T, RBT>(a, ocs, oss, o0, rb0, C, RB, csp, code_pitch, codes16, words, lin_words, tid);
    }
}

// Persistent grid over the tiles (programmatic dependent launch: the first
// tiles are staged while the amax pass finishes).
template <typename CT, typename K>
cudaError_t launch_tiles(K k, const CUtensorMap &map, const QArgs &a, int smem, cudaStream_t s) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, CT::NT, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t tiles = ((a.rows + CT::TR - 1) / CT::TR) * ((a.cols + CT::TC - 1) / CT::TC);
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int grid = (int)(tiles < cap ? tiles : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(CT::NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, map, a);
}

template <int MODE, bool RHT, typename T, bool AP>
cudaError_t run_col(const QArgs &a, cudaStream_t s) {
    auto k = k_quant_col<MODE, RHT, T, AP>;
    constexpr int smem = 2 * ColTile<T, kColRBT>::kStageBytes + 1024;  // input stages only
    static bool configured = false;  // one attribute call per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    CUtensorMap map;
    if (!make_tmap_2d(&map, a.x, (int)sizeof(T), a.rows, a.cols, a.ld, ColTile<T, kColRBT>::TC, ColTile<T, kColRBT>::TR))
        return cudaErrorInvalidValue;
    return launch_tiles<ColTile<T, kColRBT>>(k, map, a, smem, s);
}

template <typename T, bool AP>
cudaError_t run_2d(const QArgs &a, cudaStream_t s) {
    auto k = k_quant_2d<T, AP>;
    constexpr int smem = ColTile<T, kColRBT>::kSmemBytes;
    static bool configured = false;  // one attribute call per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    CUtensorMap map;
    if (!make_tmap_2d(&map, a.x, (int)sizeof(T), a.rows, a.cols, a.ld, ColTile<T, kColRBT>::TC, ColTile<T, kColRBT>::TR))
        return cudaErrorInvalidValue;
    return launch_tiles<ColTile<T, kColRBT>>(k, map, a, ColTile<T, kColRBT>::kSmemBytes, s);
}

template <typename T, bool AP>
cudaError_t dispatch_col(const QArgs &a, int mode, bool rht, cudaStream_t s) {
    if (mode == MODE_RNE) return rht ? run_col<MODE_RNE, true, T, AP>(a, s) : run_col<MODE_RNE, false, T, AP>(a, s);
    if (mode == MODE_SR) return rht ? run_col<MODE_SR, true, T, AP>(a, s) : run_col<MODE_SR, false, T, AP>(a, s);
    if constexpr (!AP) return run_col<MODE_4O6, false, T, false>(a, s);
    return cudaErrorInvalidValue;  // four-over-six has no fast-math form
}

// Columnwise and 2D launches of one quotient kind (AP: fast math).
template <bool AP>
cudaError_t quant_col_launch(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return fp32 ? dispatch_col<float, AP>(a, mode, rht, s) : dispatch_col<bf16_t, AP>(a, mode, rht, s);
}

template <bool AP>
cudaError_t quant_2d_launch(const QArgs &a, bool fp32, cudaStream_t s) {
    return fp32 ? run_2d<float, AP>(a, s) : run_2d<bf16_t, AP>(a, s);
}

}  // namespace
}  // namespace nvfp4
