// nvfp4_quant_col.cu -- columnwise (X^T) 1x16 quantize and 16x16 (2D) tiles.
//
// A thread owns a strip of 16 X rows x one 16-byte chunk of columns (8 bf16 or
// 4 fp32): a warp reads 512 contiguous bytes per row.  Each column of the
// strip is one 16-element block of an X^T row.
#include "nvfp4_encode.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_load.cuh"
#include "nvfp4_tma.cuh"

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

// ------------------------------------------------------------ columnwise
// Tiles of 256 X rows x one 128-byte column span (64 bf16 / 32 fp32 columns)
// arrive by TMA (128-byte swizzle) into one of two stages.  Thread t reads the
// 8-byte half chunk hc = t % 16 of the 16 rows of row block rbl = t / 16 and
// encodes the HC columns in it: each is one 16-element block of an X^T row.
// Codes and scales go to a shared-memory output tile first (16 row blocks x
// 8 bytes per output row, slots XOR-swizzled so the writes do not collide in
// a bank), then out to global memory as 16-byte rows pieces, so every output
// row gets 128 contiguous bytes per tile.
constexpr int kColTileRows = 256;
constexpr int kColStageBytes = kColTileRows * 128;

template <typename T>
struct ColTile {
    static constexpr int TC = 128 / (int)sizeof(T);  // X columns per tile
    static constexpr int HC = 8 / (int)sizeof(T);    // X columns per thread
    static constexpr int kCodeBytes = TC * 128;      // output tile: TC rows x 16 blocks x 8 bytes
    static constexpr int kScaleBytes = TC * 16;
    static constexpr int kSmemBytes = 2 * (kColStageBytes + kCodeBytes + kScaleBytes) + 1024;
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

template <int MODE, bool RHT, typename T>
__global__ void __launch_bounds__(256, 2) k_quant_col(const __grid_constant__ CUtensorMap tmap, const QArgs a) {
    using CT = ColTile<T>;
    constexpr int TC = CT::TC, HC = CT::HC;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ DivTable tab;
    __shared__ RhtMult rm;
    __shared__ __align__(8) uint64_t full[2];
    uint8_t *in = dyn_smem + ((1024u - (smem_addr(dyn_smem) & 1023u)) & 1023u);
    uint8_t *oc = in + 2 * kColStageBytes;
    uint8_t *os = oc + 2 * CT::kCodeBytes;
    const uint32_t R = (uint32_t)a.rows, C = (uint32_t)a.cols, RB = R >> 4, csp = (RB + 3) & ~3u;
    const uint32_t ntc = (C + TC - 1) / TC, ntr = (R + kColTileRows - 1) / kColTileRows;
    const uint32_t ntiles = ntc * ntr;
    const int tid = threadIdx.x, hc = tid & 15, rbl = tid >> 4;
    if (tid == 0) {
        for (int s = 0; s < 2; s++) mbar_init(&full[s], 1);
        mbar_init_fence();
        for (int k = 0; k < 2; k++) {
            const uint32_t t = blockIdx.x + k * gridDim.x;
            if (t < ntiles) {
                mbar_arrive_expect_tx(&full[k], kColStageBytes);
                tma_load_2d(in + k * kColStageBytes, &tmap, (int32_t)((t % ntc) * TC),
                            (int32_t)((t / ntc) * kColTileRows), &full[k]);
            }
        }
    }
    const uint2 signs = RHT ? rht_sign_words(a.sign_mask) : make_uint2(0u, 0u);
    if (RHT) build_rht_mult(rm, a.sign_mask, tid);
    grid_dependency_wait();
    const float g = global_scale_of(a.amax[0]);
    build_table(tab, g, tid, blockDim.x);
    const ScaleDiv sd = make_scale_div(g);
    const bool fast = scale_all_fast(g);
    if (blockIdx.x == 0 && tid == 0) a.gscale[0] = g;
    __syncthreads();

    const int64_t code_pitch = R >> 1;
    const bool codes16 = (code_pitch & 15) == 0 && (reinterpret_cast<uintptr_t>(a.codes_col) & 15u) == 0;
    const bool words = (reinterpret_cast<uintptr_t>(a.scales_col) & 3u) == 0;
    const bool lin_words = words && (RB & 3u) == 0;
    for (uint32_t k = 0;; ++k) {
        const uint32_t t = blockIdx.x + k * gridDim.x;
        if (t >= ntiles) break;
        const uint32_t s = k & 1u;
        if (!mbar_wait(&full[s], (k >> 1) & 1u)) {
            atomicAdd(&g_wait_timeouts, 1u);
            a.gscale[0] = __uint_as_float(0x7FFFFFFFu);
        }
        const uint32_t tr = t / ntc, tc = t - tr * ntc;
        const uint32_t rb0 = tr * 16, o0 = tc * TC, rb = rb0 + rbl;
        const uint8_t *stage = in + s * kColStageBytes;
        uint8_t *ocs = oc + s * CT::kCodeBytes;
        uint8_t *oss = os + s * CT::kScaleBytes;
        uint2 w[16];
#pragma unroll
        for (int r = 0; r < 16; r++) {
            const int row = rbl * 16 + r;
            w[r] = *reinterpret_cast<const uint2 *>(stage + row * 128 + ((((hc >> 1) ^ (row & 7)) << 4) |
                                                                           ((hc & 1) << 3)));
        }
        uint4 rnd[HC];
#pragma unroll
        for (int cc = 0; cc < HC; cc++) {
            rnd[cc] = make_uint4(0u, 0u, 0u, 0u);
            if (MODE == MODE_SR) {
                const uint64_t blk = (uint64_t)(o0 + HC * hc + cc) * RB + rb;
                rnd[cc] = philox4x32_10_keyed((uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)a.offset,
                                              (uint32_t)(a.offset >> 32), a.round_key0, a.round_key1);
            }
        }
#pragma unroll
        for (int cc = 0; cc < HC; cc++) {
            const int ol = HC * hc + cc;
            uint32_t S = 0;
            uint2 c = make_uint2(0u, 0u);
            if (rb < RB && o0 + ol < C) {
                f2 v[8];
                strip_block<T>(w, cc, v);
                if (fast) {
                    c = encode_block_fast<MODE, RHT>(v, sd, tab, signs, rnd[cc], S);
                } else {
                    if (RHT) rht16(v, rm);
                    c = encode_block<MODE>(v, sd, tab, rnd[cc], S);
                }
            }
            // slot rbl of output row ol, XOR-swizzled by ol / HC (= hc)
            *reinterpret_cast<uint2 *>(ocs + ol * 128 + ((rbl ^ hc) << 3)) = c;
            oss[rbl * TC + ol] = (uint8_t)S;
        }
        __syncthreads();  // output tile complete, stage s consumed
        if (tid == 0) {
            const uint32_t tn = t + 2 * gridDim.x;
            if (tn < ntiles) {
                fence_async_shared();
                mbar_arrive_expect_tx(&full[s], kColStageBytes);
                tma_load_2d(in + s * kColStageBytes, &tmap, (int32_t)((tn % ntc) * TC),
                            (int32_t)((tn / ntc) * kColTileRows), &full[s]);
            }
        }
        // codes: output row ol takes 8 pieces of 16 bytes (row blocks 2q, 2q+1)
        for (int i = tid; i < TC * 8; i += 256) {
            const int ol = i >> 3, q = i & 7;
            const uint32_t o = o0 + ol, rba = rb0 + 2 * q;
            if (o >= C || rba >= RB) continue;
            const int f = (ol / HC) & 15;
            uint4 v = *reinterpret_cast<const uint4 *>(ocs + ol * 128 + (((2 * q) ^ (f & 14)) << 3));
            if (f & 1) v = make_uint4(v.z, v.w, v.x, v.y);
            uint8_t *dst = a.codes_col + (int64_t)o * code_pitch + (int64_t)rba * 8;
            if (codes16 && rba + 1 < RB) {
                *reinterpret_cast<uint4 *>(dst) = v;
            } else {
                *reinterpret_cast<uint2 *>(dst) = make_uint2(v.x, v.y);
                if (rba + 1 < RB) *reinterpret_cast<uint2 *>(dst + 8) = make_uint2(v.z, v.w);
            }
        }
        // scales: output row ol takes 4 words (row blocks 4q..4q+3)
        for (int i = tid; i < TC * 4; i += 256) {
            const int ol = i >> 2, q = i & 3;
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
    constexpr int smem = ColTile<T>::kSmemBytes;
    static bool configured = false;  // one attribute call per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    CUtensorMap map;
    if (!make_tmap_2d(&map, a.x, (int)sizeof(T), a.rows, a.cols, a.ld, ColTile<T>::TC, kColTileRows))
        return cudaErrorInvalidValue;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 256, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t tiles = ((a.rows + kColTileRows - 1) / kColTileRows) * ((a.cols + ColTile<T>::TC - 1) / ColTile<T>::TC);
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int grid = (int)(tiles < cap ? tiles : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, map, a);
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
