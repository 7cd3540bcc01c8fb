// nvfp4_quant_row.cuh -- rowwise 1x16 quantize kernels (included by
// nvfp4_quant_row.cu for exact division and nvfp4_quant_row_approx.cu for
// NVFP4_FAST_MATH; AP selects the element quotient, everything else is
// shared).
//
//  k_quant_row               per-tensor global scale (amax from the amax pass
//                            or given by the caller).  TMA brings 128-row
//                            tiles into shared memory; a thread encodes the
//                            four blocks of one tile row.
//  k_quant_row_grouped       the same tiles for row groups, each row encoded
//                            with its group's global scale.
//  k_quant_row_fused         small per-tensor inputs: amax pass, grid barrier
//                            and encode in one cooperative launch.
//  k_quant_rowscaled_staged  one global scale per row, rows of up to 96 KiB:
//                            a CTA stages whole rows in shared memory with
//                            bulk copies, reduces each row's amax, prepares
//                            that row's divisors, then encodes it (single
//                            launch, no separate amax pass).
//  k_quant_rowscaled         the same for longer rows, reading global memory
//                            twice (amax pass, then encode).
#pragma once

#include <algorithm>

#include "nvfp4_encode.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_load.cuh"
#include "nvfp4_tensor_amax.cuh"
#include "nvfp4_tiles.cuh"
#include "nvfp4_tma.cuh"

namespace nvfp4 {
namespace {  // internal linkage: each including unit has its own kernels

// Scale bytes of 4 consecutive blocks of a row go out as one 32-bit store
// (lanes 4m..4m+3 hold blocks j..j+3 with j % 4 == 0); otherwise one byte.
// Scale arrays stay below 4 GiB, so offsets are 32-bit.
__device__ __forceinline__ void store_scale(const QArgs &a, uint8_t *scales, uint32_t S, uint32_t r, uint32_t j,
                                            uint32_t CS, uint32_t csp, bool active, bool words) {
    if (words) {
        const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, S, 1);
        const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, S, 2);
        const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, S, 3);
        if (active && (j & 3u) == 0) {
            const uint32_t off = a.swizzled ? swizzle_offset32(r, j, csp) : r * CS + j;
            *reinterpret_cast<uint32_t *>(scales + off) = S | (s1 << 8) | (s2 << 16) | (s3 << 24);
        }
    } else if (active) {
        scales[a.swizzled ? swizzle_offset32(r, j, csp) : r * CS + j] = (uint8_t)S;
    }
}

// Encode one block from its raw bytes (flat block index i, for the Philox
// counter); returns the codes and writes S.
template <int MODE, bool RHT, typename T, typename Tab>
__device__ __forceinline__ uint2 row_block(const QArgs &a, const ScaleDiv &sd, const Tab &tab, const RhtMult &rm,
                                           const RawBlock<T> &raw, uint32_t i, uint32_t &S) {
    f2 v[8];
    unpack(raw, v);
    if (RHT) rht16(v, rm);
    uint4 rnd = make_uint4(0u, 0u, 0u, 0u);
    if (MODE == MODE_SR) rnd = block_random(a.seed, a.offset, a.blk_base + i);
    return encode_block<MODE>(v, sd, tab, rnd, S);
}

// ---------------------------------------------------------------------
// Per-tensor rowwise quantize, input staged through shared memory by TMA.
//
// The input is cut into tiles of 128 rows x 64 columns (4 blocks per row).
// One thread owns one tile row, i.e. 4 consecutive blocks: its codes are 32
// contiguous bytes and its scales one 32-bit word.  Persistent CTAs walk the
// tiles round-robin; thread 0 keeps RowTile::kStages tiles in flight with TMA copies
// into 128-byte-swizzled buffers, so the 16-byte chunks a warp reads sit in
// distinct bank groups.  Boxes outside the tensor are zero-filled, which also
// yields the zero pad bytes of the swizzled scale layout.
constexpr int kTileRows = 128;  // 64 measured 0.5 us slower on 8192x4096, 256 1.2 us
constexpr int kTileCols = 64;
template <typename T>
struct RowTile {
    // one stage: the other CTAs of the SM cover a tile's copy (two stages, a
    // per-warp release of the stage instead of the CTA barrier, and both
    // together measured the same on 8192x4096)
    static constexpr int kStages = 1;
    static constexpr int kBoxCols = 128 / (int)sizeof(T);  // one 128-byte swizzle span
    static constexpr int kBoxes = kTileCols / kBoxCols;    // 1 (bf16) or 2 (fp32)
    static constexpr int kBoxBytes = kTileRows * 128;
    static constexpr int kStageBytes = kBoxes * kBoxBytes;
    static constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
};

// Raw bytes of block b (0..3) of tile row `row`: chunk c of a 128-byte box
// row is stored at chunk position c ^ (row % 8).
template <typename T>
__device__ __forceinline__ void stage_block(const uint8_t *stage, int row, int b, RawBlock<T> &raw) {
    constexpr int kChunks = (int)sizeof(T);  // 16-byte chunks per block
    constexpr int kPerBoxRow = 8 / kChunks;  // blocks per box row
    const uint8_t *base = stage + (b / kPerBoxRow) * RowTile<T>::kBoxBytes + row * 128;
#pragma unroll
    for (int k = 0; k < kChunks; k++) {
        const int c = (b % kPerBoxRow) * kChunks + k;
        raw.w[k] = *reinterpret_cast<const uint4 *>(base + ((c ^ (row & 7)) << 4));
    }
}

template <typename T>
__device__ __forceinline__ void issue_tile(const CUtensorMap *map, uint8_t *stage, uint64_t *bar, uint32_t tr,
                                           uint32_t tc) {
    mbar_arrive_expect_tx(bar, RowTile<T>::kStageBytes);
#pragma unroll
    for (int b = 0; b < RowTile<T>::kBoxes; b++)
        tma_load_2d(stage + b * RowTile<T>::kBoxBytes, map, (int32_t)(tc * kTileCols + b * RowTile<T>::kBoxCols),
                    (int32_t)(tr * kTileRows), bar);
}

// Group of row r among groups lo..hi: the largest g <= hi with
// group_offsets[g] <= r, else lo (binary search).
__device__ __forceinline__ int64_t group_in(const QArgs &a, int64_t r, int64_t lo, int64_t hi) {
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (__ldg(a.group_offsets + mid) <= r) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int64_t group_of(const QArgs &a, int64_t r) { return group_in(a, r, 0, a.n_groups - 1); }

// The same in 32-bit indices (rows and groups below 2^31).
__device__ __forceinline__ uint32_t group_in32(const QArgs &a, uint32_t r, uint32_t lo, uint32_t hi) {
    while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) >> 1;
        if (__ldg(a.group_offsets + mid) <= (int64_t)r) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// One thread's tile row: its four blocks (j0 .. j0 + 3 of row `row`, staged
// in `stage` as tile row `trow`) encoded with the divisor table `tab` of one
// global scale, then their codes (32 contiguous bytes) and scales (one word)
// stored.  fast: every divisor of that scale is in the fast range (the table
// then carries FastScale::up).
template <int MODE, bool RHT, typename T, bool AP, typename Tab>
__device__ __forceinline__ void encode_tile_row(const QArgs &a, const uint8_t *stage, int trow, uint32_t row,
                                                uint32_t j0, uint32_t C, uint32_t CS, uint32_t csp, const Tab &tab,
                                                const ScaleDiv &sd, const RhtMult &rm, uint2 signs, bool fast,
                                                bool codes16, bool words, bool lin_words) {
    uint32_t S[4] = {0u, 0u, 0u, 0u};
    uint2 c[4];
    if (fast) {
        // the four blocks' random words first: independent integer work
        // the scheduler can interleave with the butterflies and divisions
        uint4 rnd[4];
#pragma unroll
        for (int b = 0; b < 4; b++) {
            rnd[b] = make_uint4(0u, 0u, 0u, 0u);
            if (MODE == MODE_SR) {
                const uint64_t blk = a.blk_base + (uint64_t)(row * CS + j0 + b);
                rnd[b] = philox4x32_10_keyed((uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)a.offset,
                                             (uint32_t)(a.offset >> 32), a.round_key0, a.round_key1);
            }
        }
        // (encoding the zero-filled blocks past the last column instead of
        // branching around them measured 1 us slower per 8192x4096 call)
#pragma unroll
        for (int b = 0; b < 4; b++) {
            if (j0 + b < CS) {
                RawBlock<T> raw;
                stage_block<T>(stage, trow, b, raw);
                f2 v[8];
                if (RHT) unpack_fwht_first(raw, v);
                else unpack(raw, v);
                c[b] = encode_block_fast<MODE, RHT, AP, true, true>(v, sd, tab, signs, rnd[b], S[b]);
            }
        }
    } else {
#pragma unroll
        for (int b = 0; b < 4; b++) {
            if (j0 + b < CS) {
                RawBlock<T> raw;
                stage_block<T>(stage, trow, b, raw);
                c[b] = row_block<MODE, RHT, T>(a, sd, tab, rm, raw, row * CS + j0 + b, S[b]);
            }
        }
    }
    uint8_t *codes = a.codes_row + (int64_t)row * (C >> 1) + j0 * 8;
    if (codes16 && j0 + 3 < CS) {
        reinterpret_cast<uint4 *>(codes)[0] = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
        reinterpret_cast<uint4 *>(codes)[1] = make_uint4(c[2].x, c[2].y, c[3].x, c[3].y);
    } else {
#pragma unroll
        for (int b = 0; b < 4; b++)
            if (j0 + b < CS) reinterpret_cast<uint2 *>(codes)[b] = c[b];
    }
    const uint32_t word = S[0] | (S[1] << 8) | (S[2] << 16) | (S[3] << 24);
    if (a.swizzled) {
        uint8_t *dst = a.scales_row + swizzle_offset32(row, j0, csp);
        if (words) {
            *reinterpret_cast<uint32_t *>(dst) = word;
        } else {
#pragma unroll
            for (int b = 0; b < 4; b++) dst[b] = (uint8_t)S[b];
        }
    } else if (lin_words && j0 + 3 < CS) {
        *reinterpret_cast<uint32_t *>(a.scales_row + row * CS + j0) = word;
    } else {
#pragma unroll
        for (int b = 0; b < 4; b++)
            if (j0 + b < CS) a.scales_row[row * CS + j0 + b] = (uint8_t)S[b];
    }
}

// Zero scale word of a pad row of the swizzled layout (rows R .. Rp - 1).
__device__ __forceinline__ void pad_tile_row(const QArgs &a, uint32_t row, uint32_t j0, uint32_t csp, bool words) {
    uint8_t *dst = a.scales_row + swizzle_offset32(row, j0, csp);
    if (words) {
        *reinterpret_cast<uint32_t *>(dst) = 0u;
    } else {
#pragma unroll
        for (int b = 0; b < 4; b++) dst[b] = 0;
    }
}

template <int MODE, bool RHT, typename T, bool AP>
__global__ void __launch_bounds__(kTileRows) k_quant_row(const __grid_constant__ CUtensorMap tmap, const QArgs a) {
    constexpr int kStages = RowTile<T>::kStages;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ DivTable tab;
    __shared__ RhtMult rm;
    __shared__ __align__(8) uint64_t full[RowTile<T>::kStages];
    uint8_t *stages = dyn_smem + ((1024u - (smem_addr(dyn_smem) & 1023u)) & 1023u);
    const uint32_t R = (uint32_t)a.rows, C = (uint32_t)a.cols, CS = C >> 4, csp = (CS + 3) & ~3u;
    const uint32_t Rp = (R + 127) & ~127u;
    const uint32_t ntc = (C + kTileCols - 1) / kTileCols, ntr = (R + kTileRows - 1) / kTileRows;
    const uint32_t ntiles = ntc * ntr;
    const int tid = threadIdx.x;
    // tile coordinates advance by the grid size per iteration (no division in
    // the loop); a second cursor runs kStages tiles ahead for the copies
    const uint32_t G = gridDim.x, dr = G / ntc, dc = G - dr * ntc;
    uint32_t tr = blockIdx.x / ntc, tc = blockIdx.x - tr * ntc;
    uint32_t ir = tr, ic = tc;
    auto advance = [&](uint32_t &r, uint32_t &c) {
        c += dc;
        r += dr;
        if (c >= ntc) {
            c -= ntc;
            ++r;
        }
    };
    if (tid == 0) {
        for (int s = 0; s < kStages; s++) mbar_init(&full[s], 1);
        mbar_init_fence();
    }
    for (int k = 0; k < kStages; k++) {
        if (tid == 0 && blockIdx.x + k * G < ntiles)
            issue_tile<T>(&tmap, stages + k * RowTile<T>::kStageBytes, &full[k], ntr - 1 - ir, ntc - 1 - ic);
        advance(ir, ic);
    }
    // per-scale state, built while the first copies are in flight; the amax
    // pass may still be running until grid_dependency_wait returns
    const uint2 signs = RHT ? rht_sign_words(a.sign_mask) : make_uint2(0u, 0u);
    if (RHT) build_rht_mult(rm, a.sign_mask, tid);
    grid_dependency_wait();
    const float A = tensor_amax_read(a, RHT);
    const float g = global_scale_of(A);
    const bool fast = scale_all_fast(g);  // uniform: every divisor in the fast range
    // on the fast path the table carries the encoder's power-of-two factor
    build_table(tab, g, tid, blockDim.x, fast ? FastScale<MODE, RHT>::up : 1.0f);
    const ScaleDiv sd = make_scale_div(g);
    __syncthreads();
    tensor_amax_done(a, A, g);

    // vector stores only where every address is aligned for them
    const bool codes16 = (C & 31u) == 0 && (reinterpret_cast<uintptr_t>(a.codes_row) & 15u) == 0;
    const bool words = (reinterpret_cast<uintptr_t>(a.scales_row) & 3u) == 0;
    const bool lin_words = words && (CS & 3u) == 0;
    for (uint32_t k = 0;; ++k) {
        const uint32_t t = blockIdx.x + k * G;
        if (t >= ntiles) break;
        const uint32_t s = k % kStages;
        if (!mbar_wait(&full[s], (k / kStages) & 1u)) {  // a copy never landed: bounded, visible failure
            wait_gave_up(a, a.gscale);
        }
        // tiles from the end of the tensor: the amax pass read the tail last, so
        // with a tensor larger than L2 the first tiles here still come from L2
        // (-0.9 us at 16384x8192; no change when the whole input fits)
        const uint32_t row = (ntr - 1 - tr) * kTileRows + tid, j0 = (ntc - 1 - tc) * 4;
        const uint8_t *stage = stages + s * RowTile<T>::kStageBytes;
        if (row < R) {
            encode_tile_row<MODE, RHT, T, AP>(a, stage, tid, row, j0, C, CS, csp, tab, sd, rm, signs, fast, codes16,
                                              words, lin_words);
        } else if (a.swizzled && row < Rp) {  // pad rows of the swizzled layout
            pad_tile_row(a, row, j0, csp, words);
        }
        advance(tr, tc);
        __syncthreads();  // every thread is done with stage s
        if (tid == 0 && t + kStages * G < ntiles) {
            fence_async_shared();
            issue_tile<T>(&tmap, stages + s * RowTile<T>::kStageBytes, &full[s], ntr - 1 - ir, ntc - 1 - ic);
        }
        advance(ir, ic);
    }
}

// ---------------------------------------------------------------------
// Grouped rowwise quantize on the tiles of k_quant_row.
//
// Row groups [offs[g], offs[g+1]) each have their own global scale, written
// by the finalising kernel before this one reads it.  Tiles are mostly inside
// one group, or across the boundary of two: the CTA holds the divisor tables
// of two groups in shared memory (a two-entry cache that keeps a tile's first
// and last group), so a tile costs a table build only when it needs a group
// the cache does not hold.  Rows of the groups strictly inside a tile (groups
// shorter than a tile) look each divisor up through DivDirect instead, with
// the same bits.  (Building those groups' tables two at a time between CTA
// barriers, and copying the offsets and scales into shared memory, measured
// 2 us slower per 8192x4096 call with 8 groups.)  The tiles cover every byte
// of the swizzled scale layout, pad rows and columns included.
template <int MODE, bool RHT, typename T>
__global__ void __launch_bounds__(kTileRows) k_quant_row_grouped(const __grid_constant__ CUtensorMap tmap,
                                                                 const QArgs a) {
    struct Slot {
        DivTable t;
        ScaleDiv sd;
        int fast;
    };
    extern __shared__ uint8_t dyn_smem[];
    __shared__ Slot slot[2];
    __shared__ RhtMult rm;
    __shared__ __align__(8) uint64_t full;
    uint8_t *stage = dyn_smem + ((1024u - (smem_addr(dyn_smem) & 1023u)) & 1023u);
    const uint32_t R = (uint32_t)a.rows, C = (uint32_t)a.cols, CS = C >> 4, csp = (CS + 3) & ~3u;
    const uint32_t Rp = (R + 127) & ~127u;
    const uint32_t ntc = (C + kTileCols - 1) / kTileCols, ntr = (R + kTileRows - 1) / kTileRows;
    const uint32_t ntiles = ntc * ntr;
    const int tid = threadIdx.x;
    const uint32_t G = gridDim.x, dr = G / ntc, dc = G - dr * ntc;
    uint32_t tr = blockIdx.x / ntc, tc = blockIdx.x - tr * ntc;
    if (tid == 0) {
        mbar_init(&full, 1);
        mbar_init_fence();
        if (blockIdx.x < ntiles) issue_tile<T>(&tmap, stage, &full, tr, tc);
    }
    const uint2 signs = RHT ? rht_sign_words(a.sign_mask) : make_uint2(0u, 0u);
    if (RHT) build_rht_mult(rm, a.sign_mask, tid);
    grid_dependency_wait();  // the group scales are final from here on
    __syncthreads();
    const bool codes16 = (C & 31u) == 0 && (reinterpret_cast<uintptr_t>(a.codes_row) & 15u) == 0;
    const bool words = (reinterpret_cast<uintptr_t>(a.scales_row) & 3u) == 0;
    const bool lin_words = words && (CS & 3u) == 0;
    constexpr float up = FastScale<MODE, RHT>::up;
    const uint32_t ng = (uint32_t)a.n_groups;  // < 2^31
    uint32_t held0 = ~0u, held1 = ~0u;  // the groups whose tables the slots hold (uniform)
    auto build = [&](int q, uint32_t gq) {
        const float g = a.gscale[gq];
        const bool fast = scale_all_fast(g);
        build_table(slot[q].t, g, tid, kTileRows, fast ? up : 1.0f);
        if (tid == 0) {
            slot[q].sd = make_scale_div(g);
            slot[q].fast = fast;
        }
    };
    for (uint32_t k = 0;; ++k) {
        const uint32_t t = blockIdx.x + k * G;
        if (t >= ntiles) break;
        const uint32_t r0 = tr * kTileRows, row = r0 + tid, j0 = tc * 4;
        const uint32_t glo = group_in32(a, r0, 0, ng - 1);
        const uint32_t ghi = group_in32(a, min(R, r0 + kTileRows) - 1, glo, ng - 1);
        // slots for the tile's first and last group, keeping what is held
        uint32_t n0 = held0, n1 = held1;
        if (n0 != glo && n1 != glo) {
            if (n0 == ghi) n1 = glo;
            else n0 = glo;
        }
        if (ghi != glo && n0 != ghi && n1 != ghi) {
            if (n0 == glo) n1 = ghi;
            else n0 = ghi;
        }
        if (n0 != held0 || n1 != held1) {  // the previous tile's barrier freed the slots
            if (n0 != held0) build(0, n0);
            if (n1 != held1) build(1, n1);
            held0 = n0;
            held1 = n1;
            __syncthreads();
        }
        const uint32_t mine = row < R ? group_in32(a, row, glo, ghi) : ~0u;
        if (!mbar_wait(&full, k & 1u)) {  // a copy never landed: bounded, visible failure
            wait_gave_up(a, nullptr);
            if (row < R) *reinterpret_cast<volatile float *>(a.gscale + mine) = __uint_as_float(0x7FFFFFFFu);
        }
        if (row < R) {
            if (mine == held0 || mine == held1) {
                const Slot &sl = slot[mine == held0 ? 0 : 1];
                encode_tile_row<MODE, RHT, T, false>(a, stage, tid, row, j0, C, CS, csp, sl.t, sl.sd, rm, signs,
                                                     sl.fast != 0, codes16, words, lin_words);
            } else {  // a group inside the tile: divisors computed when looked up
                const float g = a.gscale[mine];
                const bool fast = scale_all_fast(g);
                const DivDirect dd{{g, fast ? up : 1.0f}};
                encode_tile_row<MODE, RHT, T, false>(a, stage, tid, row, j0, C, CS, csp, dd, make_scale_div(g), rm,
                                                     signs, fast, codes16, words, lin_words);
            }
        }
        if (row >= R && a.swizzled && row < Rp) pad_tile_row(a, row, j0, csp, words);
        tc += dc;
        tr += dr;
        if (tc >= ntc) {
            tc -= ntc;
            ++tr;
        }
        __syncthreads();  // every thread is done with the stage and the slots
        if (tid == 0 && t + G < ntiles) {
            fence_async_shared();
            issue_tile<T>(&tmap, stage, &full, tr, tc);
        }
    }
}

// ---------------------------------------------------------------------
// Per-tensor rowwise quantize of a small tensor in one cooperative launch.
//
// Below a few million elements the amax pass and the quantize pass each cost
// little more than a launch, so both run in one kernel: pass 1 streams the
// CTA's tiles (TMA, kFusedStages in flight) and reduces its amax, a grid
// barrier makes the tensor amax known to every CTA, and pass 2 streams the
// same tiles again (from L2) and encodes them.  A tile is TR = 128 rows x 64
// columns; thread t takes tile row t % 128 and blocks 2h, 2h+1 (h = t / 128).
// Warps release a stage through an mbarrier (one arrival per warp) instead of
// a CTA barrier, and thread 0 refills it once every warp has released it.
// (Larger tensors run the amax and quantize kernels, whose second launch
// overlaps the first's tail; there the one-kernel form gains nothing.)
constexpr int kFusedThreads = 256;
constexpr int kFusedTileRows = kStreamTileRows;
constexpr int kFusedStages = kStreamStages;
// two threads per tile row, two of its four blocks each
static_assert(kFusedThreads == 2 * kFusedTileRows && kStreamTileCols == 64, "one-kernel thread layout");
// Thread 0 of every CTA: fold the CTA maximum (magnitude bits) into the
// tensor maximum (ws[0]), count the CTA in (ws[1], ordered after the maximum
// by release semantics) and wait until every CTA is in; the maximum is final
// then and is read together with the count in one 64-bit load.  The wait
// gives up after `polls` loads (QArgs::grid_polls; the default bound is about
// a second) and returns false.  grid_amax_depart (at the end of the kernel,
// off the critical path) counts the CTA out either way, so the words return
// to zero even after a give-up.
__device__ __forceinline__ bool grid_amax_barrier(uint32_t *ws, uint32_t m, uint32_t nctas, uint32_t polls,
                                                  uint32_t &total) {
    asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(ws), "r"(m) : "memory");
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ws + 1) : "memory");
    bool ok = false;
    unsigned long long v = 0;
    for (uint32_t i = 0; i < polls; ++i) {
        asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(ws) : "memory");
        if ((uint32_t)(v >> 32) >= nctas) {
            ok = true;
            break;
        }
        if (i >= 4096) __nanosleep(64);  // spin first: the last CTA usually arrives within microseconds
    }
    total = (uint32_t)v;
    return ok;
}

// Thread 0 of every CTA, after its barrier read: a second count (ws[2]) lets
// the last CTA out, when every CTA has read the maximum, clear ws[0..2] for
// the next call.
__device__ __forceinline__ void grid_amax_depart(uint32_t *ws, uint32_t nctas) {
    if (atomicAdd(ws + 2, 1u) == nctas - 1) {
        ws[0] = 0u;
        ws[1] = 0u;
        ws[2] = 0u;
    }
}

template <int MODE, bool RHT, typename T, bool AP>
__global__ void __launch_bounds__(kFusedThreads) k_quant_row_fused(const __grid_constant__ CUtensorMap tmap,
                                                                  const QArgs a) {
    constexpr int NT = kFusedThreads, TR = kFusedTileRows;
    using FT = StreamTile<T>;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ DivTable tab;
    __shared__ RhtMult rm;
    __shared__ __align__(8) uint64_t full[kFusedStages];
    __shared__ __align__(8) uint64_t empty[kFusedStages];
    __shared__ uint32_t red[NT / 32];
    __shared__ float amax_sh;
    uint8_t *stages = dyn_smem + ((1024u - (smem_addr(dyn_smem) & 1023u)) & 1023u);
    const uint32_t R = (uint32_t)a.rows, C = (uint32_t)a.cols, CS = C >> 4, csp = (CS + 3) & ~3u;
    const uint32_t ntc = (C + kTileCols - 1) / kTileCols, ntr = (R + TR - 1) / TR;
    const uint32_t ntiles = ntc * ntr, G = gridDim.x;
    const uint32_t nk = blockIdx.x < ntiles ? (ntiles - blockIdx.x + G - 1) / G : 0;  // my tiles
    const int tid = threadIdx.x, warp = tid >> 5, trow = tid % TR, jb = (tid / TR) * 2;
    // load L (0 <= L < 2 nk) is the CTA's tile L % nk: pass 1, then pass 2
    auto issue = [&](uint32_t L) {
        const uint32_t t = blockIdx.x + (L % nk) * G, s = L % kFusedStages;
        stream_issue<T>(&tmap, stages + s * FT::kStageBytes, &full[s], t / ntc, t % ntc);
    };
    if (tid == 0) {
        for (int s = 0; s < kFusedStages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NT / 32);
        }
        mbar_init_fence();
        for (uint32_t L = 0; L < 2 * nk && L < (uint32_t)kFusedStages; L++) issue(L);
    }
    if (RHT) build_rht_mult(rm, a.sign_mask, tid);
    __syncthreads();
    bool ok = true;

    // ---------------- pass 1: amax
    float m = 0.0f;
    for (uint32_t k = 0; k < nk; ++k) {
        const uint32_t s = k % kFusedStages;
        ok &= mbar_wait(&full[s], (k / kFusedStages) & 1u);
        const uint8_t *stage = stages + s * FT::kStageBytes;
#pragma unroll
        for (int b = 0; b < 2; b++) {
            RawBlock<T> raw;
            stream_block<T>(stage, trow, jb + b, raw);  // past the edge: zeros
            f2 v[8];
            unpack(raw, v);
            if (RHT) fwht16(v);
            m = absmax_nan(m, block_amax(v));
        }
        // pass 2's first loads follow pass 1's last ones without a break
        ok &= stream_release(empty, k, tid, k + kFusedStages < 2 * nk, [&](uint32_t) { issue(k + kFusedStages); });
    }

    // ---------------- grid-wide amax
    {
        uint32_t mb = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m) & 0x7FFFFFFFu);
        if ((tid & 31) == 0) red[warp] = mb;
        __syncthreads();
        if (tid < 32) {
            mb = __reduce_max_sync(0xFFFFFFFFu, tid < NT / 32 ? red[tid] : 0u);
            if (tid == 0) {
                uint32_t bits = 0;
                if (!grid_amax_barrier(a.workspace, mb, G, a.grid_polls, bits)) ok = false;
                float A = __uint_as_float(bits);
                if (RHT) A = __fmul_rn(A, 0.25f);
                amax_sh = A;
                if (blockIdx.x == 0) {
                    a.amax[0] = A;
                    publish_gscale(a, a.gscale, global_scale_of(A));
                }
            }
        }
        __syncthreads();
    }
    const float g = global_scale_of(amax_sh);
    build_table(tab, g, tid, blockDim.x);
    const ScaleDiv sd = make_scale_div(g);
    const bool fast = scale_all_fast(g);
    const uint2 signs = RHT ? rht_sign_words(a.sign_mask) : make_uint2(0u, 0u);
    __syncthreads();

    // ---------------- pass 2: encode
    const bool vec = (reinterpret_cast<uintptr_t>(a.codes_row) & 15u) == 0 && ((C >> 1) & 15u) == 0;
    const bool svec = (reinterpret_cast<uintptr_t>(a.scales_row) & 1u) == 0;
    const bool lin_svec = svec && (CS & 1u) == 0;
    for (uint32_t k = 0; k < nk; ++k) {
        const uint32_t L = nk + k, s = L % kFusedStages;
        const uint32_t t = blockIdx.x + k * G;
        ok &= mbar_wait(&full[s], (L / kFusedStages) & 1u);
        const uint32_t tr = t / ntc, tc = t - tr * ntc;
        const uint32_t row = tr * TR + trow, j0 = tc * 4 + jb;
        const uint8_t *stage = stages + s * FT::kStageBytes;
        if (row < R && j0 < CS) {
            uint4 w[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
            if (MODE == MODE_SR) {
#pragma unroll
                for (int b = 0; b < 2; b++) {
                    const uint64_t blk = a.blk_base + (uint64_t)row * CS + j0 + b;
                    w[b] = philox4x32_10_keyed((uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)a.offset,
                                               (uint32_t)(a.offset >> 32), a.round_key0, a.round_key1);
                }
            }
            uint32_t S[2] = {0u, 0u};
            uint2 c[2];
#pragma unroll
            for (int b = 0; b < 2; b++) {
                RawBlock<T> raw;
                stream_block<T>(stage, trow, jb + b, raw);
                f2 v[8];
                unpack(raw, v);
                if (fast) {
                    c[b] = encode_block_fast<MODE, RHT, AP>(v, sd, tab, signs, w[b], S[b]);
                } else {
                    if (RHT) rht16(v, rm);
                    c[b] = encode_block<MODE>(v, sd, tab, w[b], S[b]);
                }
            }
            // the tile's blocks past the edge (j0 + b >= CS) are not stored;
            // 16-byte stores need C % 32 == 0, so CS is even and j0 + 1 < CS
            uint8_t *codes = a.codes_row + (int64_t)row * (C >> 1) + j0 * 8;
            if (vec) {
                *reinterpret_cast<uint4 *>(codes) = make_uint4(c[0].x, c[0].y, c[1].x, c[1].y);
            } else {
                reinterpret_cast<uint2 *>(codes)[0] = c[0];
                if (j0 + 1 < CS) reinterpret_cast<uint2 *>(codes)[1] = c[1];
            }
            if (a.swizzled) {  // j0 is even: the pair is contiguous in its 4-byte group (pad bytes 0)
                uint8_t *dst = a.scales_row + swizzle_offset32(row, j0, csp);
                if (svec) {
                    *reinterpret_cast<uint16_t *>(dst) = (uint16_t)(S[0] | (S[1] << 8));
                } else {
                    dst[0] = (uint8_t)S[0];
                    dst[1] = (uint8_t)S[1];
                }
            } else {
                uint8_t *dst = a.scales_row + (size_t)row * CS + j0;
                if (lin_svec && j0 + 1 < CS) {
                    *reinterpret_cast<uint16_t *>(dst) = (uint16_t)(S[0] | (S[1] << 8));
                } else {
                    dst[0] = (uint8_t)S[0];
                    if (j0 + 1 < CS) dst[1] = (uint8_t)S[1];
                }
            }
        }
        ok &= stream_release(empty, L, tid, L + kFusedStages < 2 * nk, [&](uint32_t) { issue(L + kFusedStages); });
    }
    if (!ok) wait_gave_up(a, a.gscale);  // a bounded wait gave up in this CTA: the output is not trustworthy
    if (tid == 0) grid_amax_depart(a.workspace, G);
}

template <int MODE, bool RHT, typename T>
__global__ void __launch_bounds__(256) k_quant_rowscaled(const QArgs a) {
    __shared__ DivTable tab;
    __shared__ RhtMult rm;
    __shared__ uint32_t red[32];
    const uint32_t CS = (uint32_t)(a.cols >> 4);
    const uint32_t csp = (CS + 3) & ~3u;
    if (RHT) build_rht_mult(rm, a.sign_mask, threadIdx.x);
    const bool words = (CS & 3u) == 0;
    const T *x = static_cast<const T *>(a.x);
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const T *xr = x + r * a.ld;
        // pass 1: amax of the row (post-RHT magnitudes; the 0.25 is applied to
        // the maximum, which rounds the same way because rounding is monotone)
        float m = 0.0f;
        for (uint32_t j = threadIdx.x; j < CS; j += blockDim.x) {
            RawBlock<T> b;
            load_raw(xr + 16 * j, b);
            f2 v[8];
            unpack(b, v);
            if (RHT) fwht16(v);
            m = absmax_nan(m, block_amax(v));
        }
        float A = __uint_as_float(block_max_u32(__float_as_uint(m), red));
        if (RHT) A = __fmul_rn(A, 0.25f);
        const float g = global_scale_of(A);
        if (threadIdx.x == 0) {
            a.amax[r] = A;
            a.gscale[r] = g;
        }
        build_table(tab, g, threadIdx.x, blockDim.x);
        const ScaleDiv sd = make_scale_div(g);
        __syncthreads();
        // pass 2: encode (warp-uniform trip count for the scale-word shuffles)
        for (uint32_t base = threadIdx.x & ~31u; base < CS; base += blockDim.x) {
            const uint32_t j = base + (threadIdx.x & 31u);
            const bool active = j < CS;
            uint32_t S = 0;
            if (active) {
                RawBlock<T> b;
                load_raw(xr + 16 * j, b);
                f2 v[8];
                unpack(b, v);
                if (RHT) rht16(v, rm);
                uint4 rnd = make_uint4(0u, 0u, 0u, 0u);
                if (MODE == MODE_SR) rnd = block_random(a.seed, a.offset, a.blk_base + (uint64_t)r * CS + j);
                const uint2 c = encode_block<MODE>(v, sd, tab, rnd, S);
                *reinterpret_cast<uint2 *>(a.codes_row + r * (a.cols >> 1) + 8 * j) = c;
            }
            store_scale(a, a.scales_row, S, (uint32_t)r, j, CS, csp, active, words);
        }
        __syncthreads();  // the next row rebuilds the table
    }
}

// ---------------------------------------------------------------------
// Per-row global scale, the row staged in shared memory.  A CTA owns whole
// rows: one bulk copy brings a row in (two buffers, the next-but-one row is
// requested as soon as every thread is past the row that used its buffer),
// pass 1 reduces the row amax from shared memory, the CTA prepares that row's
// 128 element divisors and the two block-scale divisors, and pass 2 encodes
// from shared memory with the same block encoders as the per-tensor kernel.
// Tables and reduction slots alternate between rows, so a row costs two CTA
// barriers.  About four blocks per thread amortise the per-row preparation.
constexpr int kRowBufs = 2;
constexpr uint32_t kMaxStagedRowBytes = 96u * 1024u;  // per buffer

struct RowTables {
    DivTable t;
    Divisor m6, m4;
};

template <typename T>
__device__ __forceinline__ void smem_row_block(const uint8_t *rowp, uint32_t j, RawBlock<T> &b) {
    const uint4 *p = reinterpret_cast<const uint4 *>(rowp + (size_t)j * 16 * sizeof(T));
#pragma unroll
    for (int k = 0; k < (int)sizeof(T); k++) b.w[k] = p[k];
}

// max |x| bits over a staged row without the RHT: any element order will do,
// so threads read consecutive 16-byte words (no bank conflicts) and compare
// magnitude bits as unsigned integers (bf16: two 16-bit lanes per word).
// NaN patterns sort above +inf, so a NaN wins as in the bit-max definition.
template <typename T>
__device__ __forceinline__ uint32_t row_bits_max(const uint8_t *rowp, uint32_t words16, int tid, int nt) {
    const uint4 *p = reinterpret_cast<const uint4 *>(rowp);
    if (sizeof(T) == 2) {
        uint32_t m = 0;
        for (uint32_t i = tid; i < words16; i += nt) {
            const uint4 w = p[i];
            uint32_t t0, t1;
            asm("max.u16x2 %0, %1, %2;" : "=r"(t0) : "r"(w.x & 0x7FFF7FFFu), "r"(w.y & 0x7FFF7FFFu));
            asm("max.u16x2 %0, %1, %2;" : "=r"(t1) : "r"(w.z & 0x7FFF7FFFu), "r"(w.w & 0x7FFF7FFFu));
            asm("max.u16x2 %0, %1, %2;" : "=r"(t0) : "r"(t0), "r"(t1));
            asm("max.u16x2 %0, %1, %2;" : "=r"(m) : "r"(m), "r"(t0));
        }
        return max(m & 0xFFFFu, m >> 16) << 16;
    } else {
        uint32_t m = 0;
        for (uint32_t i = tid; i < words16; i += nt) {
            const uint4 w = p[i];
            m = max(m, max(max(w.x & 0x7FFFFFFFu, w.y & 0x7FFFFFFFu), max(w.z & 0x7FFFFFFFu, w.w & 0x7FFFFFFFu)));
        }
        return m;
    }
}

template <int MODE, bool RHT, typename T, bool AP, bool GROUPED>
__global__ void __launch_bounds__(256) k_quant_rowscaled_staged(const QArgs a, uint32_t buf_bytes) {
    extern __shared__ uint8_t dyn_smem[];
    __shared__ RowTables tabs[2];
    __shared__ RhtMult rm;
    __shared__ uint32_t red[2][8];
    __shared__ float group_amax[2];
    __shared__ __align__(8) uint64_t full[kRowBufs];
    uint8_t *bufs = dyn_smem + ((16u - (smem_addr(dyn_smem) & 15u)) & 15u);
    const uint32_t CS = (uint32_t)(a.cols >> 4);
    const uint32_t csp = (CS + 3) & ~3u;
    const uint32_t row_bytes = (uint32_t)a.cols * sizeof(T);
    const bool words = (CS & 3u) == 0 && (reinterpret_cast<uintptr_t>(a.scales_row) & 3u) == 0;
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const char *x = static_cast<const char *>(a.x);
    if (tid == 0) {
        for (int s = 0; s < kRowBufs; s++) mbar_init(&full[s], 1);
        mbar_init_fence();
        for (int k = 0; k < kRowBufs; k++) {
            const int64_t r = blockIdx.x + (int64_t)k * gridDim.x;
            if (r < a.rows) {
                mbar_arrive_expect_tx(&full[k], row_bytes);
                bulk_load(bufs + k * buf_bytes, x + r * a.ld * (int64_t)sizeof(T), row_bytes, &full[k]);
            }
        }
    }
    if (RHT) build_rht_mult(rm, a.sign_mask, tid);
    const uint2 signs = RHT ? rht_sign_words(a.sign_mask) : make_uint2(0u, 0u);
    __syncthreads();
    for (uint32_t k = 0;; ++k) {
        const int64_t r = blockIdx.x + (int64_t)k * gridDim.x;
        if (r >= a.rows) break;
        const uint32_t s = k % kRowBufs, par = k & 1u;
        const bool arrived = mbar_wait(&full[s], (k / kRowBufs) & 1u);
        if (!arrived) wait_gave_up(a, nullptr);  // the row's scale is poisoned below
        const uint8_t *rowp = bufs + s * buf_bytes;
        // pass 1: amax of the row (post-RHT magnitudes, 0.25 applied to the max);
        // grouped scaling instead reads the final amax of the row's group
        constexpr bool grouped = GROUPED;
        if (grouped && tid == 0) group_amax[par] = a.amax[group_of(a, r)];
        uint32_t mb = 0;
        if (grouped) {
        } else if (RHT) {
            float m = 0.0f;
            for (uint32_t j = tid; j < CS; j += nt) {
                RawBlock<T> raw;
                smem_row_block<T>(rowp, j, raw);
                f2 v[8];
                unpack(raw, v);
                fwht16(v);
                m = absmax_nan(m, block_amax(v));
            }
            mb = __float_as_uint(m) & 0x7FFFFFFFu;
        } else {
            mb = row_bits_max<T>(rowp, row_bytes >> 4, tid, nt);
        }
        mb = __reduce_max_sync(0xFFFFFFFFu, mb);
        if (lane == 0) red[par][warp] = mb;
        __syncthreads();  // (1) reduction slots; every thread is past row k-1
        mb = lane < (nt >> 5) ? red[par][lane] : 0u;
        mb = __reduce_max_sync(0xFFFFFFFFu, mb);
        if (tid == 0) {
            // the buffer of row k-1 is free: request row k+1 into it
            const int64_t rn = r + (int64_t)(kRowBufs - 1) * gridDim.x;
            if (k > 0 && rn < a.rows) {
                const uint32_t sn = (k + kRowBufs - 1) % kRowBufs;
                fence_async_shared();
                mbar_arrive_expect_tx(&full[sn], row_bytes);
                bulk_load(bufs + sn * buf_bytes, x + rn * a.ld * (int64_t)sizeof(T), row_bytes, &full[sn]);
            }
        }
        float A = __uint_as_float(mb);
        if (RHT) A = __fmul_rn(A, 0.25f);
        if (grouped) A = group_amax[par];
        const float g = global_scale_of(A);
        RowTables &tb = tabs[par];
        for (int e = tid; e < 130; e += nt) {
            if (e < 128)
                tb.t.e[e] = make_divisor(__fmul_rn(e4m3_value((uint32_t)e), g));
            else
                (e == 128 ? tb.m6 : tb.m4) = make_divisor(__fmul_rn(e == 128 ? 6.0f : 4.0f, g));
        }
        // a row whose copy never arrived is published with a NaN scale
        const bool lost = __syncthreads_or(!arrived);  // (2) tables ready
        if (tid == 0 && grouped) {
            if (lost) a.gscale[group_of(a, r)] = __uint_as_float(0x7FFFFFFFu);
        } else if (tid == 0) {
            a.amax[r] = A;
            a.gscale[r] = lost ? __uint_as_float(0x7FFFFFFFu) : g;
        }
        ScaleDiv sd;
        sd.m6 = tb.m6;
        sd.m4 = tb.m4;
        sd.fast6 = divisor_fast(sd.m6.d);
        sd.fast4 = divisor_fast(sd.m4.d);
        const bool fast = scale_all_fast(g);
        // pass 2: encode (warp-uniform trip count for the scale-word shuffles)
        for (uint32_t base = tid & ~31u; base < CS; base += nt) {
            const uint32_t j = base + lane;
            const bool active = j < CS;
            uint32_t S = 0;
            if (active) {
                RawBlock<T> raw;
                smem_row_block<T>(rowp, j, raw);
                f2 v[8];
                unpack(raw, v);
                uint4 rnd = make_uint4(0u, 0u, 0u, 0u);
                if (MODE == MODE_SR) {
                    const uint64_t blk = a.blk_base + (uint64_t)r * CS + j;
                    rnd = philox4x32_10_keyed((uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)a.offset,
                                              (uint32_t)(a.offset >> 32), a.round_key0, a.round_key1);
                }
                uint2 c;
                if (fast) {
                    c = encode_block_fast<MODE, RHT, AP>(v, sd, tb.t, signs, rnd, S);
                } else {
                    if (RHT) rht16(v, rm);
                    c = encode_block<MODE>(v, sd, tb.t, rnd, S);
                }
                *reinterpret_cast<uint2 *>(a.codes_row + r * (a.cols >> 1) + 8 * j) = c;
            }
            store_scale(a, a.scales_row, S, (uint32_t)r, j, CS, csp, active, words);
        }
    }
}

template <typename K>
int grid_for(K kernel, int threads, int64_t work_items) {
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0);
    if (per_sm < 1) per_sm = 1;
    const int64_t want = (work_items + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

template <int MODE, bool RHT, typename T, bool AP>
cudaError_t run_row(const QArgs &a, cudaStream_t s) {
    auto k = k_quant_row<MODE, RHT, T, AP>;
    constexpr int smem = RowTile<T>::kSmemBytes;
    static bool configured = false;  // one attribute call per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    CUtensorMap map;
    if (!make_tmap_2d(&map, a.x, (int)sizeof(T), a.rows, a.cols, a.ld, RowTile<T>::kBoxCols, kTileRows))
        return cudaErrorInvalidValue;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kTileRows, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t tiles = ((a.rows + kTileRows - 1) / kTileRows) * ((a.cols + kTileCols - 1) / kTileCols);
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int grid = (int)(tiles < cap ? tiles : cap);
    // programmatic dependent launch: the kernel stages its first tiles while
    // the amax pass finishes, and waits for it before reading the amax
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTileRows);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, map, a);
}

template <int MODE, bool RHT, typename T, bool AP, bool GROUPED>
cudaError_t run_rowscaled_staged(const QArgs &a, cudaStream_t s) {
    auto k = k_quant_rowscaled_staged<MODE, RHT, T, AP, GROUPED>;
    const uint32_t buf = ((uint32_t)(a.cols * sizeof(T)) + 15u) & ~15u;
    const int smem = (int)(kRowBufs * buf + 16);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // about four blocks of a row per thread, 32..256 threads
    const int64_t cs = a.cols >> 4;
    const int threads = (int)std::min<int64_t>(256, std::max<int64_t>(32, ((cs + 3) / 4 + 31) / 32 * 32));
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem);
    const int64_t cap = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
    const int grid = (int)(a.rows < cap ? (a.rows > 0 ? a.rows : 1) : cap);
    k<<<grid, threads, smem, s>>>(a, buf);
    return cudaGetLastError();
}

template <int MODE, bool RHT, typename T, bool AP>
cudaError_t run_rowscaled(const QArgs &a, cudaStream_t s) {
    if ((uint64_t)a.cols * sizeof(T) <= kMaxStagedRowBytes) {
        return run_rowscaled_staged<MODE, RHT, T, AP, false>(a, s);
    }
    auto k = k_quant_rowscaled<MODE, RHT, T>;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 256, 0);
    const int64_t cap = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
    const int grid = (int)(a.rows < cap ? (a.rows > 0 ? a.rows : 1) : cap);
    k<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T, bool AP>
cudaError_t dispatch_row(const QArgs &a, int mode, bool rht, bool scaled_rows, cudaStream_t s) {
    if (scaled_rows) {
        if (mode == MODE_RNE) return rht ? run_rowscaled<MODE_RNE, true, T, AP>(a, s) : run_rowscaled<MODE_RNE, false, T, AP>(a, s);
        if (mode == MODE_SR) return rht ? run_rowscaled<MODE_SR, true, T, AP>(a, s) : run_rowscaled<MODE_SR, false, T, AP>(a, s);
        if constexpr (!AP) return run_rowscaled<MODE_4O6, false, T, false>(a, s);
        return cudaErrorInvalidValue;  // four-over-six has no fast-math form
    }
    if (mode == MODE_RNE) return rht ? run_row<MODE_RNE, true, T, AP>(a, s) : run_row<MODE_RNE, false, T, AP>(a, s);
    if (mode == MODE_SR) return rht ? run_row<MODE_SR, true, T, AP>(a, s) : run_row<MODE_SR, false, T, AP>(a, s);
    if constexpr (!AP) return run_row<MODE_4O6, false, T, false>(a, s);
    return cudaErrorInvalidValue;
}

// Grouped rowwise quantize: the tile kernel, launched while the finalising
// kernel runs (it waits for it before reading the group scales).  If the
// tensor map cannot be made, rows that fit in shared memory take the staged
// per-row kernel instead (*padded = false: the caller zeroes the pad bytes of
// the swizzled layout, which that kernel leaves alone).
template <int MODE, bool RHT, typename T>
cudaError_t run_row_grouped(const QArgs &a, bool *padded, cudaStream_t s) {
    auto k = k_quant_row_grouped<MODE, RHT, T>;
    constexpr int smem = RowTile<T>::kStageBytes + 1024;
    static bool configured = false;  // one attribute call per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    CUtensorMap map;
    if (!make_tmap_2d(&map, a.x, (int)sizeof(T), a.rows, a.cols, a.ld, RowTile<T>::kBoxCols, kTileRows)) {
        *padded = false;
        if ((uint64_t)a.cols * sizeof(T) > kMaxStagedRowBytes) return cudaErrorNotSupported;
        return run_rowscaled_staged<MODE, RHT, T, false, true>(a, s);
    }
    *padded = true;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kTileRows, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t tiles = ((a.rows + kTileRows - 1) / kTileRows) * ((a.cols + kTileCols - 1) / kTileCols);
    const int64_t cap = (int64_t)sm_count() * per_sm;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles < cap ? tiles : cap));
    cfg.blockDim = dim3(kTileRows);
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
cudaError_t dispatch_row_grouped(const QArgs &a, int mode, bool rht, bool *padded, cudaStream_t s) {
    if (mode == MODE_RNE) return run_row_grouped<MODE_RNE, false, T>(a, padded, s);
    if (mode == MODE_SR) return rht ? run_row_grouped<MODE_SR, true, T>(a, padded, s)
                                    : run_row_grouped<MODE_SR, false, T>(a, padded, s);
    return run_row_grouped<MODE_4O6, false, T>(a, padded, s);
}

template <int MODE, bool RHT, typename T, bool AP>
cudaError_t run_row_fused(const QArgs &a, cudaStream_t s) {
    auto k = k_quant_row_fused<MODE, RHT, T, AP>;
    constexpr int smem = StreamTile<T>::kSmemBytes;
    static bool configured = false;  // one attribute call per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kFusedThreads, smem) != cudaSuccess || per_sm < 1)
        return cudaErrorNotSupported;
    CUtensorMap map;
    if (!make_tmap_2d(&map, a.x, (int)sizeof(T), a.rows, a.cols, a.ld, StreamTile<T>::kBoxCols, kFusedTileRows))
        return cudaErrorInvalidValue;
    const int64_t tiles = ((a.rows + kFusedTileRows - 1) / kFusedTileRows) * ((a.cols + kTileCols - 1) / kTileCols);
    const int64_t cap = (int64_t)sm_count() * per_sm;
    const int grid = (int)(tiles < cap ? tiles : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every CTA resident
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, map, a);
}

template <typename T, bool AP>
cudaError_t dispatch_row_fused(const QArgs &a, int mode, bool rht, cudaStream_t s) {
    if (mode == MODE_RNE) return rht ? run_row_fused<MODE_RNE, true, T, AP>(a, s) : run_row_fused<MODE_RNE, false, T, AP>(a, s);
    if (mode == MODE_SR) return rht ? run_row_fused<MODE_SR, true, T, AP>(a, s) : run_row_fused<MODE_SR, false, T, AP>(a, s);
    if constexpr (!AP) return run_row_fused<MODE_4O6, false, T, false>(a, s);
    return cudaErrorInvalidValue;
}

// Per-tensor rowwise quantize with the amax pass folded in (one cooperative
// launch).  Returns an error without enqueuing anything if the launch is not
// possible; the caller then runs the amax and quantize kernels instead.
template <bool AP>
cudaError_t quant_row_fused_launch(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s) {
    return fp32 ? dispatch_row_fused<float, AP>(a, mode, rht, s) : dispatch_row_fused<bf16_t, AP>(a, mode, rht, s);
}

// Rowwise launches of one quotient kind (AP: fast math).
template <bool AP>
cudaError_t quant_row_launch(const QArgs &a, bool fp32, int mode, bool rht, bool scaled_rows, cudaStream_t s) {
    return fp32 ? dispatch_row<float, AP>(a, mode, rht, scaled_rows, s)
                : dispatch_row<bf16_t, AP>(a, mode, rht, scaled_rows, s);
}

}  // namespace
}  // namespace nvfp4
