// nvfp4_amax.cu -- global amax reductions.
//
// Per tensor: rowwise blocks (and the plain maximum of any orientation) are
// streamed through shared memory by TMA; columnwise RHT blocks are read as
// 16-row strips.  Magnitude-bit maximum per thread, warp (redux.sync) and CTA
// trees, then one reduction per CTA into the workspace; the result reaches
// the quantize kernel, or the caller of the standalone entry point, as
// nvfp4_tensor_amax.cuh describes.  No memset, no second launch, no host sync.
//
// With the RHT the maximum is over the post-transform magnitudes.  Signs do
// not change magnitudes and rounding is monotone, so the kernel takes the
// maximum of the raw butterfly outputs and multiplies it by 0.25 once.
#include "nvfp4_encode.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_load.cuh"
#include "nvfp4_tensor_amax.cuh"
#include "nvfp4_tiles.cuh"
#include "nvfp4_tma.cuh"

namespace nvfp4 {

// Unsigned maximum of the magnitude bits of a raw block (bf16: two 16-bit
// lanes per word, compared as integers; NaN patterns sort above +inf).
__device__ __forceinline__ uint32_t block_max_bits(const RawBlock<bf16_t> &b) {
    uint32_t t[2];
#pragma unroll
    for (int k = 0; k < 2; k++) {
        uint32_t u, v;
        asm("max.u16x2 %0, %1, %2;" : "=r"(u) : "r"(b.w[k].x & 0x7FFF7FFFu), "r"(b.w[k].y & 0x7FFF7FFFu));
        asm("max.u16x2 %0, %1, %2;" : "=r"(v) : "r"(b.w[k].z & 0x7FFF7FFFu), "r"(b.w[k].w & 0x7FFF7FFFu));
        asm("max.u16x2 %0, %1, %2;" : "=r"(t[k]) : "r"(u), "r"(v));
    }
    uint32_t m;
    asm("max.u16x2 %0, %1, %2;" : "=r"(m) : "r"(t[0]), "r"(t[1]));
    return max(m & 0xFFFFu, m >> 16) << 16;
}

__device__ __forceinline__ uint32_t block_max_bits(const RawBlock<float> &b) {
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < 4; k++)
        m = max(m, max(max(b.w[k].x & 0x7FFFFFFFu, b.w[k].y & 0x7FFFFFFFu),
                       max(b.w[k].z & 0x7FFFFFFFu, b.w[k].w & 0x7FFFFFFFu)));
    return m;
}

// Rowwise amax (and the plain amax of any orientation) through TMA: tiles of
// 128 rows x 64 columns stream through kStreamStages shared-memory stages per
// CTA, so tens of KB per SM are in flight while the threads transform and
// reduce; thread t takes tile row t % 128 and blocks 2h, 2h+1 (h = t / 128).
// Tiles after the first kStreamStages of each CTA come from a TileQueue:
// from the counter workspace[2] in the standalone pass, round robin in a
// quantize call.  Columns or rows past the edge arrive as zeros, which change no
// maximum (and whose butterfly is zero).
constexpr int kAmaxTmaThreads = 256;
// two threads per tile row, two of its four blocks each
static_assert(kAmaxTmaThreads == 2 * kStreamTileRows && kStreamTileCols == 64, "amax thread layout");

//
// With the RHT, a block is transformed only if it could raise the maximum:
// every stage of the butterfly rounds |a +- b| to at most RN(|a| + |b|)
// (rounding is monotone), so no output of a block exceeds 16 max|v|, and a
// block whose 16 max|v| lies below a maximum some block has already produced
// cannot change the result.  In a quantize call the CTAs fold their running
// maximum into the workspace word once per tile and read it back (one tile
// late), so after the first tiles most blocks cost a bit-max instead of a
// butterfly; the result is the same maximum, bit for bit.  (The standalone
// TMA pass transforms every block: there the shared hint measured 2 us slower
// on 8192x4096, with the tile counter's traffic beside it.)
constexpr bool kAmaxSkip = true;

// A known lower bound of the tensor maximum for the skip test, shared through
// one workspace word: each warp folds its running maximum into a CTA word once
// per tile; thread 0 forwards a larger CTA maximum to the workspace with one
// red.max and publishes, for the next tile, the workspace value it loaded at
// the end of the previous tile (so no thread waits on the load).  Every value
// it ever holds is a maximum some block has produced.
struct MaxHint {
    uint32_t *cta_max, *shared_hint;  // shared words, zeroed before the CTA's first barrier
    uint32_t *word;                   // the workspace word
    uint32_t hint, sent, pending;     // sent, pending: thread 0's

    __device__ __forceinline__ MaxHint(uint32_t *cm, uint32_t *sh, uint32_t *w)
        : cta_max(cm), shared_hint(sh), word(w), hint(0u), sent(0u), pending(0u) {}

    // Blocks whose bound is not above this cannot raise the maximum.
    __device__ __forceinline__ uint32_t threshold(uint32_t m) const { return max(m, hint); }

    __device__ __forceinline__ void fold(uint32_t m) {
        const uint32_t wm = __reduce_max_sync(0xFFFFFFFFu, m);
        if ((threadIdx.x & 31) == 0 && wm > hint) atomicMax(cta_max, wm);
        if (threadIdx.x == 0) {
            const uint32_t cm = *reinterpret_cast<volatile uint32_t *>(cta_max);
            if (cm > sent) {
                asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(word), "r"(cm) : "memory");
                sent = cm;
            }
            *reinterpret_cast<volatile uint32_t *>(shared_hint) = max(cm, pending);
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(pending) : "l"(word) : "memory");
        }
        hint = max(hint, *reinterpret_cast<volatile uint32_t *>(shared_hint));
    }
};

// Bits of a value >= 16 max|v| of a raw 1x16 block: exactly 16 max|v| for
// normal numbers, a little more for subnormals; NaN and Inf stay above every
// finite maximum.  No butterfly output of the block exceeds it.
template <typename T>
__device__ __forceinline__ uint32_t butterfly_bound(const RawBlock<T> &raw) {
    return block_max_bits(raw) + (4u << 23);
}

template <bool RHT, typename T, bool PUBLISH>
__global__ void __launch_bounds__(kAmaxTmaThreads) k_amax_tma(const __grid_constant__ CUtensorMap tmap,
                                                              const QArgs a) {
    using ST = StreamTile<T>;
    constexpr bool SKIP = RHT && !PUBLISH && kAmaxSkip;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t full[kStreamStages];
    __shared__ __align__(8) uint64_t empty[kStreamStages];
    __shared__ uint32_t stage_tile[kStreamStages];  // tile in the stage, or kNoTile: the stream ended
    __shared__ uint32_t warp_max, warps_in;
    __shared__ uint32_t cta_run_max, hint_sh;  // SKIP: the MaxHint words
    uint8_t *stages = dyn_smem + ((1024u - (smem_addr(dyn_smem) & 1023u)) & 1023u);
    const uint32_t ntc = (uint32_t)((a.cols + kStreamTileCols - 1) / kStreamTileCols);
    const uint32_t ntiles = ntc * (uint32_t)((a.rows + kStreamTileRows - 1) / kStreamTileRows);
    const int tid = threadIdx.x, trow = tid % kStreamTileRows, jb = (tid / kStreamTileRows) * 2;
    TileQueue q;  // thread 0's
    // thread 0: put tile t (or the end of the stream) into stage s
    auto fill = [&](uint32_t s, uint32_t t) {
        stage_tile[s] = t;
        if (t == kNoTile) {
            mbar_arrive(&full[s]);
        } else {
            stream_issue<T>(&tmap, stages + s * ST::kStageBytes, &full[s], t / ntc, t % ntc);
        }
    };
    if (tid == 0) {
        for (int s = 0; s < kStreamStages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kAmaxTmaThreads / 32);
        }
        warp_max = 0u;
        warps_in = 0u;
        cta_run_max = 0u;
        hint_sh = 0u;
        mbar_init_fence();
        // dynamic tiles for the standalone pass, whose last CTA publishes (the
        // CTAs then finish together: 1.8 us less on 8192x4096); in a quantize
        // call static tiles measured faster (the quantize kernel's first CTAs
        // start on SMs that finish early)
        q.init(PUBLISH ? a.workspace + 2 : nullptr, ntiles, kStreamStages);
        bool complete = true;
        for (uint32_t k = 0; k < (uint32_t)kStreamStages && complete; k++) {
            const uint32_t t = q.static_tile(k);
            fill(k, t);
            complete = t != kNoTile;
        }
        q.start(complete);
    }
    __syncthreads();
    bool ok = true;
    uint32_t m = 0;
    MaxHint hint(&cta_run_max, &hint_sh, a.workspace);
    for (uint32_t k = 0;; ++k) {
        const uint32_t s = k % kStreamStages;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (k / kStreamStages) & 1u))) {  // warp-uniform exit
            ok = false;
            break;
        }
        if (*reinterpret_cast<volatile uint32_t *>(&stage_tile[s]) == kNoTile) break;
        const uint8_t *stage = stages + s * ST::kStageBytes;
#pragma unroll
        for (int b = 0; b < 2; b++) {
            RawBlock<T> raw;
            stream_block<T>(stage, trow, jb + b, raw);
            if (RHT) {
                if (!SKIP || butterfly_bound(raw) > hint.threshold(m)) {
                    f2 v[8];
                    unpack(raw, v);
                    fwht16(v);
                    m = max(m, __float_as_uint(block_amax(v)) & 0x7FFFFFFFu);
                }
            } else {
                m = max(m, block_max_bits(raw));
            }
        }
        if (SKIP) hint.fold(m);
        ok &= stream_release(empty, k, tid, tid == 0 && !q.done, [&](uint32_t st) { fill(st, q.next()); });
    }
    if (!ok) {  // a bounded wait gave up: record it, and a NaN maximum poisons the scale
        wait_gave_up(a, nullptr);
        m = 0x7FFFFFFFu;
    }
    if (PUBLISH) publish_tensor_amax(a, m, RHT);
    else fold_tensor_amax_warps(a, m, &warp_max, &warps_in);
}

// RHT amax of contiguous bf16 rows (row pitch = row length) for a quantize
// call, with plain 16-byte loads: the tensor is one run of 1x16 blocks, block
// i at element 16 i; each thread keeps kLdgBlocks blocks (128 bytes) in flight
// and a warp's loads of one round cover 1 KiB contiguously.  Same skip test
// and hand-off as k_amax_tma.  The loop that folds the hint runs a
// warp-uniform number of rounds (the tail rounds follow without it).
// PUBLISH (the standalone entry point): the last CTA publishes amax and g;
// only thread 0 of a CTA sends hints to the workspace word, so every hint
// precedes that CTA's ticket and the last ticket's reset follows them all.
constexpr int kLdgBlocks = 4;
constexpr int kAmaxLdgThreads = 256;

template <bool PUBLISH>
__global__ void __launch_bounds__(kAmaxLdgThreads) k_amax_ldg_rht(const QArgs a) {
    constexpr bool SKIP = kAmaxSkip;
    __shared__ uint32_t warp_max, warps_in, hint_words[2];
    if (threadIdx.x == 0) {
        warp_max = 0u;
        warps_in = 0u;
        hint_words[0] = hint_words[1] = 0u;
    }
    __syncthreads();
    const bf16_t *x = static_cast<const bf16_t *>(a.x);
    const uint64_t nblk = (uint64_t)a.rows * (uint64_t)(a.cols >> 4);
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint32_t lane = threadIdx.x & 31;
    uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    MaxHint hint(&hint_words[0], &hint_words[1], a.workspace);
    uint32_t m = 0;
    auto reduce = [&](const RawBlock<bf16_t> &raw) {
        if (!SKIP || butterfly_bound(raw) > hint.threshold(m)) {
            f2 v[8];
            unpack(raw, v);
            fwht16(v);
            m = max(m, __float_as_uint(block_amax(v)) & 0x7FFFFFFFu);
        }
    };
    // full rounds: the warp's last lane still has kLdgBlocks blocks
    for (; i - lane + 31 + (kLdgBlocks - 1) * stride < nblk; i += kLdgBlocks * stride) {
        RawBlock<bf16_t> raw[kLdgBlocks];
#pragma unroll
        for (int u = 0; u < kLdgBlocks; u++) load_raw(x + (i + u * stride) * 16, raw[u]);
#pragma unroll
        for (int u = 0; u < kLdgBlocks; u++) reduce(raw[u]);
        if (SKIP) hint.fold(m);
    }
    for (; i < nblk; i += stride) {
        RawBlock<bf16_t> raw;
        load_raw(x + i * 16, raw);
        reduce(raw);
    }
    if (PUBLISH) publish_tensor_amax(a, m, true);
    else fold_tensor_amax_warps(a, m, &warp_max, &warps_in);
}

// RHT blocks along the columns (16 rows of one column), and optionally the
// row blocks too, from one TMA stream of the bf16 input (the tiles and stages
// of k_amax_tma).  A warp takes a 16-row strip of the tile and each lane two
// adjacent columns of it: sixteen 32-bit reads, one per row, that the 32 lanes
// spread over the row's 128 bytes without bank conflicts.  With ROW, thread t
// also reduces row blocks 2h, 2h+1 of tile row t % 128 (h = t / 128), as
// k_amax_tma does, so both orientations' maxima come from one read of the
// input (the operand of a weight-gradient GEMM needs both).  Both use the
// skip test above.  The column maximum goes to workspace word kColWord (4)
// when ROW is set, else to word 0; the row maximum to word 0.  Consumer calls
// only: the quantize kernels publish.
template <bool ROW>
__global__ void __launch_bounds__(kAmaxTmaThreads) k_amax_tma_cols(const __grid_constant__ CUtensorMap tmap,
                                                                   const QArgs a) {
    using T = bf16_t;
    using ST = StreamTile<T>;
    constexpr uint32_t kColWord = ROW ? 4u : 0u;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t full[kStreamStages];
    __shared__ __align__(8) uint64_t empty[kStreamStages];
    __shared__ uint32_t redr[kAmaxTmaThreads / 32], redc[kAmaxTmaThreads / 32];
    __shared__ uint32_t hint_words[4];  // MaxHint words: rows (0, 1), columns (2, 3)
    uint8_t *stages = dyn_smem + ((1024u - (smem_addr(dyn_smem) & 1023u)) & 1023u);
    const uint32_t ntc = (uint32_t)((a.cols + kStreamTileCols - 1) / kStreamTileCols);
    const uint32_t ntiles = ntc * (uint32_t)((a.rows + kStreamTileRows - 1) / kStreamTileRows), G = gridDim.x;
    const uint32_t nk = blockIdx.x < ntiles ? (ntiles - blockIdx.x + G - 1) / G : 0;  // my tiles
    const int tid = threadIdx.x, trow = tid % kStreamTileRows, jb = (tid / kStreamTileRows) * 2;
    const int strip = tid >> 5, cbyte = (tid & 31) * 4;  // 16-row strip, byte of the lane's column pair
    auto issue = [&](uint32_t k) {
        const uint32_t t = blockIdx.x + k * G, s = k % kStreamStages;
        stream_issue<T>(&tmap, stages + s * ST::kStageBytes, &full[s], t / ntc, t % ntc);
    };
    if (tid == 0) {
        for (int s = 0; s < kStreamStages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kAmaxTmaThreads / 32);
        }
        for (int i = 0; i < 4; i++) hint_words[i] = 0u;
        mbar_init_fence();
        for (uint32_t k = 0; k < nk && k < (uint32_t)kStreamStages; k++) issue(k);
    }
    __syncthreads();
    MaxHint hr(&hint_words[0], &hint_words[1], a.workspace), hc(&hint_words[2], &hint_words[3], a.workspace + kColWord);
    bool ok = true;
    uint32_t mr = 0, mc = 0;
    for (uint32_t k = 0; k < nk; ++k) {
        const uint32_t s = k % kStreamStages;
        ok &= mbar_wait(&full[s], (k / kStreamStages) & 1u);
        const uint8_t *stage = stages + s * ST::kStageBytes;
        if (ROW) {
#pragma unroll
            for (int b = 0; b < 2; b++) {
                RawBlock<T> raw;
                stream_block<T>(stage, trow, jb + b, raw);
                if (!kAmaxSkip || butterfly_bound(raw) > hr.threshold(mr)) {
                    f2 v[8];
                    unpack(raw, v);
                    fwht16(v);
                    mr = max(mr, __float_as_uint(block_amax(v)) & 0x7FFFFFFFu);
                }
            }
        }
        // the strip: word i holds row i of the lane's two columns (low half:
        // the even column); chunk c of a 128-byte row sits at c ^ (row % 8)
        uint32_t w[16];
        uint32_t mx = 0u;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const int r = strip * 16 + i;
            w[i] = *reinterpret_cast<const uint32_t *>(stage + r * 128 + ((((cbyte >> 4) ^ (r & 7)) << 4) | (cbyte & 15)));
            asm("max.u16x2 %0, %1, %2;" : "=r"(mx) : "r"(mx), "r"(w[i] & 0x7FFF7FFFu));
        }
        const uint32_t thr = hc.threshold(mc);
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const uint32_t bound = (h ? (mx & 0xFFFF0000u) : (mx << 16)) + (4u << 23);
            if (!kAmaxSkip || bound > thr) {
                f2 v[8];
#pragma unroll
                for (int p = 0; p < 8; p++)
                    v[p] = h ? f2{bf16_hi(w[2 * p]), bf16_hi(w[2 * p + 1])} : f2{bf16_lo(w[2 * p]), bf16_lo(w[2 * p + 1])};
                fwht16(v);
                mc = max(mc, __float_as_uint(block_amax(v)) & 0x7FFFFFFFu);
            }
        }
        if (kAmaxSkip) {
            if (ROW) hr.fold(mr);
            hc.fold(mc);
        }
        ok &= stream_release(empty, k, tid, k + kStreamStages < nk, [&](uint32_t) { issue(k + kStreamStages); });
    }
    if (!ok) {  // a bounded wait gave up: record it, and NaN maxima poison both scales
        wait_gave_up(a, nullptr);
        mr = mc = 0x7FFFFFFFu;
    }
    allow_dependents();  // the quantize kernel may start staging its tiles
    mr = __reduce_max_sync(0xFFFFFFFFu, mr);
    mc = __reduce_max_sync(0xFFFFFFFFu, mc);
    if ((tid & 31) == 0) {
        redr[tid >> 5] = mr;
        redc[tid >> 5] = mc;
    }
    __syncthreads();
    if (tid < 32) {
        mr = __reduce_max_sync(0xFFFFFFFFu, tid < kAmaxTmaThreads / 32 ? redr[tid] : 0u);
        mc = __reduce_max_sync(0xFFFFFFFFu, tid < kAmaxTmaThreads / 32 ? redc[tid] : 0u);
        if (tid == 0) {
            if (ROW) asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(a.workspace), "r"(mr) : "memory");
            asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(a.workspace + kColWord), "r"(mc)
                         : "memory");
        }
    }
}

// RHT blocks along columns: a thread owns 16 rows x one 16-byte chunk.
template <typename T, bool PUBLISH>
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
    if (PUBLISH) publish_tensor_amax(a, m, true);
    else fold_tensor_amax(a, m);
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

// Per-group amax (grouped quantize): amax[g] = max over the blocks of group g,
// as if each group were a tensor of its own.  A CTA takes a contiguous range
// of rows and, for each group segment in it, reduces the segment's blocks
// (post-RHT magnitudes without the 0.25) and folds the result into amax[g]
// with one atomicMax on its bits (the caller zeroed amax[]; magnitude bits
// order like the floats, NaN above +inf).  Block i of a segment is row
// s0 + i / CS, column i % CS: each thread keeps a (row, column) cursor that
// advances by the CTA's thread count without a division, and has kLdgBlocks
// blocks in flight.  With the RHT, a block whose butterfly bound is not above
// the CTA's running maximum of the segment skips the butterfly (the skip test
// of k_amax_ldg_rht): each warp folds its maximum into a shared word once per
// round and takes the word back as its threshold; the word restarts at 0 for
// every segment, so it only ever holds maxima of the segment's own group.
// (Sharing it through amax[g] across CTAs measured 2 us slower: every CTA of
// a group updates the same word.)
template <bool RHT, typename T>
__global__ void __launch_bounds__(kAmaxLdgThreads) k_amax_groups(const QArgs a) {
    constexpr bool SKIP = RHT && kAmaxSkip;
    __shared__ uint32_t red[32];
    __shared__ uint32_t seg_max;
    const uint32_t CS = (uint32_t)(a.cols >> 4);
    const T *x = static_cast<const T *>(a.x);
    const int64_t per = (a.rows + gridDim.x - 1) / gridDim.x;
    const int64_t r0 = (int64_t)blockIdx.x * per, r1 = min(a.rows, r0 + per);
    if (r0 >= r1) return;
    const uint32_t nt = blockDim.x, dr = nt / CS, dj = nt - dr * CS, lane = threadIdx.x & 31;
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
        const uint32_t nb = (uint32_t)(s1 - s0) * CS;  // < 2^30: the input has < 2^34 elements
        const T *p = x + (s0 + threadIdx.x / CS) * a.ld + 16 * (threadIdx.x % CS);
        uint32_t j = threadIdx.x % CS;
        const int64_t dp = (int64_t)dr * a.ld + 16 * (int64_t)dj, back = 16 * (int64_t)CS - a.ld;
        auto step = [&]() {  // p, j: to the block nt further on
            p += dp;
            j += dj;
            if (j >= CS) {
                j -= CS;
                p -= back;  // one row down, CS blocks back
            }
        };
        if (SKIP) {
            if (threadIdx.x == 0) seg_max = 0u;
            __syncthreads();
        }
        uint32_t m = 0;
        auto reduce = [&](const RawBlock<T> &raw) {
            if (!RHT) {
                m = max(m, block_max_bits(raw));
            } else if (!SKIP || butterfly_bound(raw) > m) {
                f2 v[8];
                unpack(raw, v);
                fwht16(v);
                m = max(m, __float_as_uint(block_amax(v)) & 0x7FFFFFFFu);
            }
        };
        uint32_t i = threadIdx.x;
        // full rounds: the warp's last lane still has kLdgBlocks blocks
        for (; i - lane + 31 + (kLdgBlocks - 1) * nt < nb; i += kLdgBlocks * nt) {
            RawBlock<T> raw[kLdgBlocks];
#pragma unroll
            for (int u = 0; u < kLdgBlocks; u++) {
                load_raw(p, raw[u]);
                step();
            }
#pragma unroll
            for (int u = 0; u < kLdgBlocks; u++) reduce(raw[u]);
            if (SKIP) {
                m = __reduce_max_sync(0xFFFFFFFFu, m);
                if (lane == 0) atomicMax(&seg_max, m);
                m = max(m, *reinterpret_cast<volatile uint32_t *>(&seg_max));
            }
        }
        for (; i < nb; i += nt) {
            RawBlock<T> raw;
            load_raw(p, raw);
            step();
            reduce(raw);
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

template <bool RHT, typename T, bool PUBLISH>
static cudaError_t run_amax_tma(const QArgs &a, cudaStream_t s) {
    auto k = k_amax_tma<RHT, T, PUBLISH>;
    constexpr int smem = StreamTile<T>::kSmemBytes;
    static bool configured = false;  // one attribute call per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    CUtensorMap map;
    if (!make_tmap_2d(&map, a.x, (int)sizeof(T), a.rows, a.cols, a.ld, StreamTile<T>::kBoxCols, kStreamTileRows))
        return cudaErrorInvalidValue;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kAmaxTmaThreads, smem);
    if (per_sm < 1) per_sm = 1;
    const int64_t tiles = ((a.rows + kStreamTileRows - 1) / kStreamTileRows) *
                          ((a.cols + kStreamTileCols - 1) / kStreamTileCols);
    // three CTAs per SM (of four that fit) still keep ~144 KB per SM in flight,
    // and leave room for the quantize kernel's first CTAs to start on every SM
    // while the pass drains (-1.3 us per step on 8192x4096; two per SM: no gain)
    if (per_sm > 3) per_sm = 3;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    k<<<(int)(tiles < cap ? tiles : cap), kAmaxTmaThreads, smem, s>>>(map, a);
    return cudaGetLastError();
}

template <bool ROW>
static cudaError_t run_amax_tma_cols(const QArgs &a, cudaStream_t s) {
    auto k = k_amax_tma_cols<ROW>;
    constexpr int smem = StreamTile<bf16_t>::kSmemBytes;
    static bool configured = false;  // one attribute call per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    CUtensorMap map;
    if (!make_tmap_2d(&map, a.x, 2, a.rows, a.cols, a.ld, StreamTile<bf16_t>::kBoxCols, kStreamTileRows))
        return cudaErrorInvalidValue;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kAmaxTmaThreads, smem);
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 3) per_sm = 3;  // as k_amax_tma: room for the quantize kernel's first CTAs
    const int64_t tiles = ((a.rows + kStreamTileRows - 1) / kStreamTileRows) *
                          ((a.cols + kStreamTileCols - 1) / kStreamTileCols);
    const int64_t cap = (int64_t)sm_count() * per_sm;
    k<<<(int)(tiles < cap ? tiles : cap), kAmaxTmaThreads, smem, s>>>(map, a);
    return cudaGetLastError();
}

// The load-based pass replaces the TMA one for contiguous bf16 rows in a
// quantize call.
constexpr bool kAmaxLdg = true;

template <bool PUBLISH>
static cudaError_t run_amax_ldg_rht(const QArgs &a, cudaStream_t s) {
    auto k = k_amax_ldg_rht<PUBLISH>;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kAmaxLdgThreads, 0);
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 4) per_sm = 4;
    const int64_t nblk = a.rows * (a.cols >> 4);
    const int64_t want = (nblk + kAmaxLdgThreads - 1) / kAmaxLdgThreads;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    k<<<(int)(want < cap ? want : cap), kAmaxLdgThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_amax_cols(const QArgs &a, bool with_rows, cudaStream_t s) {
    return with_rows ? run_amax_tma_cols<true>(a, s) : run_amax_tma_cols<false>(a, s);
}

template <typename T, bool PUBLISH>
static cudaError_t run_amax_tensor(const QArgs &a, bool rht, bool col, cudaStream_t s) {
    constexpr int W = Chunk<T>::W;
    if (kAmaxLdg && rht && !col && sizeof(T) == 2 && a.ld == a.cols) return run_amax_ldg_rht<PUBLISH>(a, s);
    if (!col) return rht ? run_amax_tma<true, T, PUBLISH>(a, s) : run_amax_tma<false, T, PUBLISH>(a, s);
    auto k = k_amax_rht_col<T, PUBLISH>;
    k<<<grid_for(k, (a.rows >> 4) * ((a.cols + W - 1) / W)), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_amax_tensor(const QArgs &a, bool fp32, bool rht, bool col, bool publish, cudaStream_t s) {
    if (publish) return fp32 ? run_amax_tensor<float, true>(a, rht, col, s) : run_amax_tensor<bf16_t, true>(a, rht, col, s);
    return fp32 ? run_amax_tensor<float, false>(a, rht, col, s) : run_amax_tensor<bf16_t, false>(a, rht, col, s);
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
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kAmaxLdgThreads, 0);
    if (per_sm < 1) per_sm = 1;
    if (per_sm > 4) per_sm = 4;  // as k_amax_ldg_rht: more blocks per thread
    const int64_t cap = (int64_t)sm_count() * per_sm;
    k<<<(int)(a.rows < cap ? (a.rows > 0 ? a.rows : 1) : cap), kAmaxLdgThreads, 0, s>>>(a);
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
