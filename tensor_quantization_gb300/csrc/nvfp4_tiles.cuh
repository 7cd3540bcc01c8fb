// nvfp4_tiles.cuh -- row-major input streamed through shared memory in tiles
// of 128 rows x 64 columns (one 128-byte swizzle span for bf16, two for fp32),
// kStreamStages TMA stages per CTA.  Warps release a stage through an mbarrier
// (one arrival per warp) instead of a CTA barrier; thread 0 refills a stage
// once every warp has released it.  Used by the amax pass and by the
// one-kernel path for small tensors.
#pragma once

#include "nvfp4_load.cuh"
#include "nvfp4_tma.cuh"

namespace nvfp4 {

constexpr int kStreamTileRows = 128;
constexpr int kStreamTileCols = 64;
constexpr int kStreamStages = 3;

template <typename T>
struct StreamTile {
    static constexpr int kBoxCols = 128 / (int)sizeof(T);
    static constexpr int kBoxes = kStreamTileCols / kBoxCols;  // column boxes: 1 (bf16) or 2 (fp32)
    static constexpr int kBoxBytes = kStreamTileRows * 128;
    static constexpr int kStageBytes = kBoxes * kBoxBytes;
    static constexpr int kSmemBytes = kStreamStages * kStageBytes + 1024;
};

// Raw bytes of block b (0..3) of tile row `row`: 16-byte chunk c of a box row
// sits at chunk position c ^ (row % 8) (128-byte swizzle).
template <typename T>
__device__ __forceinline__ void stream_block(const uint8_t *stage, int row, int b, RawBlock<T> &raw) {
    constexpr int kChunks = (int)sizeof(T);
    constexpr int kPerBoxRow = 8 / kChunks;
    const uint8_t *base = stage + (b / kPerBoxRow) * StreamTile<T>::kBoxBytes + row * 128;
#pragma unroll
    for (int k = 0; k < kChunks; k++) {
        const int c = (b % kPerBoxRow) * kChunks + k;
        raw.w[k] = *reinterpret_cast<const uint4 *>(base + ((c ^ (row & 7)) << 4));
    }
}

template <typename T>
__device__ __forceinline__ void stream_issue(const CUtensorMap *map, uint8_t *stage, uint64_t *bar, uint32_t tr,
                                             uint32_t tc) {
    using ST = StreamTile<T>;
    mbar_arrive_expect_tx(bar, ST::kStageBytes);
#pragma unroll
    for (int b = 0; b < ST::kBoxes; b++)
        tma_load_2d(stage + b * ST::kBoxBytes, map, (int32_t)(tc * kStreamTileCols + b * ST::kBoxCols),
                    (int32_t)(tr * kStreamTileRows), bar);
}

// Tiles handed to persistent CTAs.  Load k < `stages` of CTA b is the static
// tile b + k * G (G CTAs); every later tile comes from a counter in global
// memory, one atomicAdd per tile, requested one load ahead so that its
// latency hides behind the stage being computed.  A CTA whose data arrives
// late takes fewer tiles, so the CTAs finish together instead of waiting for
// the slowest static share.  Every CTA makes exactly one request that finds
// the tiles exhausted; the request that returns the counter's final value
// (dynamic tiles + G - 1) is the last of the call and zeroes the counter for
// the next one.  Without a counter (a call given no workspace) every tile is
// static.  Used by thread 0 only.
constexpr uint32_t kNoTile = 0xFFFFFFFFu;

struct TileQueue {
    uint32_t *ctr;
    uint32_t ntiles, first_dyn, final_v, pending, k_static;
    bool done;

    __device__ __forceinline__ void init(uint32_t *counter, uint32_t n, uint32_t stages) {
        ctr = counter;
        ntiles = n;
        first_dyn = stages * gridDim.x;
        final_v = (n > first_dyn ? n - first_dyn : 0u) + gridDim.x - 1u;
        pending = 0u;
        k_static = stages;
        done = false;
    }
    // Tile of static load k, or kNoTile.
    __device__ __forceinline__ uint32_t static_tile(uint32_t k) const {
        const uint32_t t = blockIdx.x + k * gridDim.x;
        return t < ntiles ? t : kNoTile;
    }
    __device__ __forceinline__ void request() { pending = atomicAdd(ctr, 1u); }
    // After the first `stages` static loads: request the first dynamic tile,
    // or (if the static loads already ran out) make the CTA's one failing
    // request now.
    __device__ __forceinline__ void start(bool statics_complete) {
        if (!ctr) {
            done = !statics_complete;
            return;
        }
        request();
        if (!statics_complete) finish();
    }
    // The next tile (requesting the one after it), or kNoTile once the tiles
    // are exhausted.
    __device__ __forceinline__ uint32_t next() {
        if (done) return kNoTile;
        if (!ctr) {
            const uint32_t t = static_tile(k_static++);
            done = t == kNoTile;
            return t;
        }
        const uint32_t t = first_dyn + pending;
        if (t < ntiles) {
            request();
            return t;
        }
        finish();
        return kNoTile;
    }
    __device__ __forceinline__ void finish() {
        done = true;
        if (pending == final_v) *reinterpret_cast<volatile uint32_t *>(ctr) = 0u;
    }
};

// One arrival on a stage's release barrier.
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Every warp releases load L (stage L % kStreamStages) after reading it;
// thread 0 then waits for all warps and, if `more`, refills the stage through
// refill(stage index).  Returns false if the wait gave up.
template <typename F>
__device__ __forceinline__ bool stream_release(uint64_t *empty, uint32_t L, int tid, bool more, F &&refill) {
    const uint32_t s = L % kStreamStages;
    __syncwarp();
    if ((tid & 31) == 0) mbar_arrive(&empty[s]);
    bool ok = true;
    if (tid == 0 && more) {
        ok = mbar_wait(&empty[s], (L / kStreamStages) & 1u);
        fence_async_shared();
        refill(s);
    }
    return ok;
}

}  // namespace nvfp4
