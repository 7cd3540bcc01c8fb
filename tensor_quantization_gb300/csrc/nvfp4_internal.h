// nvfp4_internal.h -- launch interface between the C ABI (nvfp4_api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nvfp4 {

// Rounding modes (same values as the Mode enum of the kernels).
enum { MODE_RNE_ID = 0, MODE_SR_ID = 1, MODE_4O6_ID = 2 };

struct QArgs {
    const void *x;
    int64_t rows, cols, ld;  // of X
    uint8_t *codes_row, *scales_row, *codes_col, *scales_col;
    float *amax;          // per tensor: [1] (input to the quantize kernels); per row: [R_out]
    float *gscale;        // written: [1] or [R_out]
    uint32_t *workspace;  // [0] running max bits, [1] CTA count (in), [2] CTA count (out)
    uint32_t sign_mask;
    uint64_t seed, offset;
    // Philox4x32-10 round keys of `seed` (key + round * Weyl constant),
    // precomputed on the host so that kernels read them from the parameter
    // bank instead of recomputing them for every block.
    uint32_t round_key0[10], round_key1[10];
    // global number of this launch's first block (shards of a larger
    // tensor): added to every Philox block counter
    uint64_t blk_base;
    int swizzled;
    int want_row, want_col;
    int fast_math;  // element quotient as y * RN(1/d)
    // the per-tensor amax comes from this call's amax pass through the
    // workspace (the quantize kernel publishes it) instead of amax[0]
    int amax_in_ws;
    // workspace word of that hand-off: the maximum, its CTA count the word
    // after it (0, or 4 for the columnwise half of a both-orientation call)
    uint32_t amax_word;
    // grouped rowwise scaling: n_groups row ranges [offs[g], offs[g+1]), each
    // with its own amax / global scale (amax[g] final before the encode)
    const int64_t *group_offsets;
    int64_t n_groups;
    // bound, in polls, of waits on other CTAs (the one-kernel path's grid
    // barrier); set by nvfp4_set_wait_limit
    uint32_t grid_polls;
};

// Default bound of a wait on other CTAs: 2^24 polls, >= 64 ns each after the
// first 4096, so about a second.
constexpr uint32_t kDefaultGridPolls = 1u << 24;

// Device properties, cached per device.
int sm_count();

// 2-D tensor map over X (row pitch ld elements) with a box of box_cols x
// box_rows elements, 128-byte swizzle, zero fill outside the tensor.
bool make_tmap_2d(CUtensorMap *map, const void *x, int elem_bytes, int64_t rows, int64_t cols, int64_t ld,
                  uint32_t box_cols, uint32_t box_rows);

// ---- launchers (return cudaGetLastError() after the launch) ----
// Per-tensor amax (optionally of RHT blocks along rows (col=0) or columns
// (col=1)).  publish: writes a.amax[0], a.gscale[0] and resets the workspace;
// otherwise leaves the maximum bits in the workspace for the quantize kernel
// launched next with a.amax_in_ws set.
cudaError_t launch_amax_tensor(const QArgs &a, bool fp32, bool rht, bool col, bool publish, cudaStream_t s);
// RHT amax of bf16 column blocks through TMA, for the quantize kernels of a
// consumer call: with_rows also reduces the row blocks in the same read (row
// maximum in workspace word 0, column maximum in word 4); without, the column
// maximum goes to word 0.
cudaError_t launch_amax_cols(const QArgs &a, bool with_rows, cudaStream_t s);
// Per-row amax of the rowwise orientation (one value per X row).
cudaError_t launch_amax_rows(const QArgs &a, bool fp32, bool rht, cudaStream_t s);

// Rowwise 1x16 quantize with a per-tensor scale (a.amax[0], or the workspace).
cudaError_t launch_quant_row(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s);
// Columnwise 1x16 quantize with a per-tensor scale.
cudaError_t launch_quant_col(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s);
// 16x16 tiles, RNE, rowwise and/or columnwise from one read.
cudaError_t launch_quant_2d(const QArgs &a, bool fp32, cudaStream_t s);
// Rowwise with one global scale per row, amax and quantize in one pass.
cudaError_t launch_quant_rowscaled(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s);
// Grouped rowwise scaling: per-group amax (atomic maxima into amax[], which the
// caller has zeroed), then amax[g] / global_scale[g] finalised in place.
cudaError_t launch_amax_groups(const QArgs &a, bool fp32, bool rht, cudaStream_t s);
cudaError_t launch_group_finalize(const QArgs &a, bool rht, bool given, cudaStream_t s);
// Grouped rowwise quantize (after the finalising kernel): each row encoded with
// its group's global scale.  *padded: the launch also wrote the pad bytes of a
// swizzled scale layout (false only on the fallback for inputs the tile kernel
// cannot map; cudaErrorNotSupported when neither applies).
cudaError_t launch_quant_grouped(const QArgs &a, bool fp32, int mode, bool rht, bool *padded, cudaStream_t s);
// Per-tensor rowwise quantize including the amax pass, one cooperative launch
// (an error return means nothing was enqueued).
cudaError_t launch_quant_row_fused(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s);
// The same launches with the fast-math element quotient (defined in their own
// translation units).
cudaError_t launch_quant_row_approx(const QArgs &a, bool fp32, int mode, bool rht, bool scaled_rows,
                                    cudaStream_t s);
cudaError_t launch_quant_col_approx(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s);
cudaError_t launch_quant_2d_approx(const QArgs &a, bool fp32, cudaStream_t s);
cudaError_t launch_quant_row_fused_approx(const QArgs &a, bool fp32, int mode, bool rht, cudaStream_t s);
// Zero the pad bytes of a swizzled scale array.
cudaError_t launch_scale_pad(uint8_t *scales, int64_t rows_out, int64_t cs, cudaStream_t s);

cudaError_t launch_dequant(const uint8_t *codes, const uint8_t *scales, const float *gscale, int64_t rows,
                           int64_t cols, int swizzled, int per_row, void *out, int out_fp32, int rht,
                           uint32_t sign_mask, cudaStream_t s);

}  // namespace nvfp4
