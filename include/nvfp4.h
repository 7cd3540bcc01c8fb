/*
 * nvfp4.h -- C ABI of libnvfp4.so, the GB300 (sm_103a) NVFP4 training quantizer.
 *
 * What the library computes (the CPU oracle under oracle/ is the executable
 * definition, and the GPU output matches it bit for bit):
 *
 *   W      = X (rowwise orientation) or X^T (columnwise orientation); the
 *            output "rows" are the rows of W, blocks are 16 consecutive
 *            elements of a W row.
 *   y      = W widened to fp32 (exact for bf16), optionally passed through the
 *            16-point Random Hadamard Transform of each block:
 *            y = v . H16 / 4 . diag(s), H16[i][j] = (-1)^popcount(i&j), applied
 *            as the butterfly with strides 1, 2, 4, 8; s_j = -1 where bit j of
 *            the sign mask is set.
 *            ("在 RTX 5090 (SM120) 上补全 NVFP4 量化相关 kernel", section
 *            "随机 Hadamard 变换")
 *   A      = max |y| over the tensor (or over each output row), taken as an
 *            unsigned max of the magnitude bits so that NaN propagates.
 *   g      = A / 2688 (2688 = 6 * 448): the fp32 decode ("global") scale.
 *            ("nvfp4-sm120" README, section "Layout": two-level E2M1/E4M3
 *            quantization; section "Results": the scale stays on the device)
 *   S      = e4m3_rn_satfinite(amax_b / (M * g)), M = 6 (four-over-six also
 *            tries M = 4); amax_b over the 16 values of a block, or the 256 of
 *            a 16x16 tile in 2D mode; an all-zero block has S = 0.
 *   q      = y / (Sf * g), correctly rounded fp32 division (Sf = value of S).
 *            ("[nvfp4 training][rl] Add a CuTe DSL fast-path kernel for
 *            four-over-six quantize #4852", PR description: every rounding
 *            step pinned, correctly rounded FP32 division)
 *   code   = E2M1 of q: round-to-nearest-even with saturation to +-6, or
 *            stochastic rounding: between grid neighbours a <= |q| < b, go up
 *            iff (|q|-a)/(b-a) + (r+0.5)/256 >= 1, r = one Philox4x32-10 byte
 *            per element.  NaN encodes as +6; Sf == 0 encodes +0.
 *            ("在 RTX 5090 (SM120) 上补全 NVFP4 量化相关 kernel", sections
 *            "随机舍入" and "随机舍入指令：（半）软件模拟")
 *   four-over-six: encode every block against M = 6 and M = 4 and keep the
 *            candidate whose squared dequantization error (summed by the
 *            clamped shuffle-down tree with offsets 8, 4, 2, 1) is strictly
 *            lower; ties and NaN keep M = 6.  (PR #4852 description)
 *
 * Layouts (all row-major, all device memory):
 *   codes  [R_out, C_out/2] bytes; byte k of a row holds element 2k in its
 *          low nibble and element 2k+1 in its high nibble.
 *   scales linear [R_out, C_out/16] bytes, or SWIZZLE_32_4_4 ("nvfp4-sm120"
 *          README, section "Approach"): padded to ceil(R_out/128)*128 rows and
 *          ceil(C_out/64)*4 scale columns, scale (r, j) at byte
 *          ((r/128)*(Cs_p/4) + j/4)*512 + (r%32)*16 + ((r%128)/32)*4 + j%4;
 *          pad bytes are written as 0.
 *   amax / global_scale: 1 float (per tensor) or R_out floats (per row).
 *
 * Ownership and streams: the caller allocates every buffer.  The library
 * never allocates, never synchronises the host, and enqueues all work on the
 * given stream (a cudaStream_t passed as void*; NULL is the legacy default
 * stream).  Inputs and outputs must stay valid until that work completes.
 *
 * Errors: every argument check runs before anything is enqueued; a failed
 * check returns its status with nothing enqueued.  NVFP4_ERR_CUDA reports a
 * launch failure (cudaGetLastError after the launch).  No exception or abort
 * crosses this ABI.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1, /* null pointer, bad shape, stride or alignment */
    NVFP4_ERR_UNSUPPORTED = 2, /* a valid but unimplemented combination      */
    NVFP4_ERR_CUDA = 3,        /* a CUDA call or launch failed                */
    NVFP4_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up          */
} nvfp4_status;

typedef enum { NVFP4_IN_BF16 = 0, NVFP4_IN_FP32 = 1 } nvfp4_dtype;

/* flags */
enum {
    NVFP4_ROWWISE = 1,       /* emit codes_row/scales_row (blocks along X rows)   */
    NVFP4_COLWISE = 2,       /* emit codes_col/scales_col (blocks along X cols)    */
    NVFP4_BLOCK_2D = 4,      /* one scale per 16x16 tile, replicated to 1x16      */
    NVFP4_SCALE_PER_ROW = 8, /* one global scale per output row                   */
    NVFP4_SWIZZLED = 16,     /* SWIZZLE_32_4_4 scale layout (else linear)         */
    NVFP4_AMAX_GIVEN = 32,   /* out->amax already holds A: skip the amax pass     */
    NVFP4_FAST_MATH = 64     /* q = y * RN(1/d) instead of the exact quotient     */
};

/* NVFP4_FAST_MATH replaces the correctly rounded element quotient q = y / d by
 * the product y * RN(1/d) (one multiply instead of a four-operation exact
 * division).  The product is within 1.5 ulp of the quotient, so an element's
 * code can change only when q lies within that distance of a rounding
 * threshold (RNE) or of a dither threshold (SR): about one element in 10^4
 * on Gaussian data, never by more than one grid step, never its sign.  Global
 * scale, block scales and the Philox stream are unchanged.  ("在 RTX 5090
 * (SM120) 上补全 NVFP4 量化相关 kernel", fast-math note: at most 0.1% of the
 * codes may differ, by at most one step.)  Not available with four-over-six
 * (NVFP4_ERR_UNSUPPORTED): its candidate choice compares exact errors. */

/* The input matrix X: rows x cols elements, row pitch ld elements (ld >= cols).
 * x must be 16-byte aligned and ld * element size a multiple of 16 bytes.
 *
 * row0, col0: where X sits inside the full tensor it was cut from (0, 0 for a
 * whole tensor).  They only number the Philox counters, so that the shards of
 * a tensor quantized separately (one per GPU, say) give exactly the codes of
 * the whole tensor: a rowwise shard is a range of whole rows (col0 = 0; its
 * blocks are numbered (row0 + r) * (cols / 16) + j) and a columnwise shard a
 * range of whole columns (row0 = 0; blocks (col0 + c) * (rows / 16) + b).  A
 * per-tensor amax must then be the whole tensor's (NVFP4_AMAX_GIVEN with the
 * maximum over the shards); per-row scales need nothing.  Stochastic rounding
 * with a nonzero offset along the other dimension returns
 * NVFP4_ERR_UNSUPPORTED; round-to-nearest ignores row0 and col0.  Negative
 * values are NVFP4_ERR_INVALID_ARG. */
typedef struct {
    const void *x;
    int32_t dtype; /* nvfp4_dtype */
    int64_t rows, cols, ld;
    int64_t row0, col0;
} nvfp4_input;

/* Output buffers (device pointers).  The pointers of an orientation that is
 * not requested may be NULL.  For columnwise output R_out = cols and
 * C_out = rows. */
typedef struct {
    uint8_t *codes_row, *scales_row;
    uint8_t *codes_col, *scales_col;
    float *amax;         /* 1 float, R_out floats with NVFP4_SCALE_PER_ROW, or 2
                            with the RHT in both orientations                 */
    float *global_scale; /* same count as amax; written by every call         */
} nvfp4_output;

/* Workspace: per-tensor modes need a small device buffer for the amax
 * reduction (a running maximum and a few counters).  Allocate
 * nvfp4_workspace_bytes() bytes, 8-byte aligned, and zero them once before
 * first use; every call leaves its counters zero again.  Calls that share a
 * workspace must not run concurrently on the GPU.
 *
 * Failure record: word 3 (bytes 12..15) of the workspace records that a
 * bounded device-side wait of a call gave up (a TMA copy that never landed, or
 * the one-kernel path's wait for the other CTAs running past its limit, see
 * nvfp4_set_wait_limit).  That call's global scale is NaN, and the record is
 * sticky: every later per-tensor call on the same workspace also publishes a
 * NaN global scale, until nvfp4_workspace_status reads and clears it.  No
 * wait blocks forever. */
size_t nvfp4_workspace_bytes(void);

/* Reads the failure record of a workspace: enqueues a 4-byte device-to-host
 * copy on `stream` and waits for the stream (the one entry point that
 * synchronises the host).  Returns NVFP4_ERR_TIMEOUT if a bounded wait of an
 * earlier call on this workspace gave up, clearing the record (also on the
 * stream, waited for) so that later calls publish valid scales again;
 * NVFP4_OK if none did; NVFP4_ERR_INVALID_ARG for a NULL or misaligned
 * workspace; NVFP4_ERR_CUDA if a copy failed.  The library has no counterpart
 * on the pages: it is how a caller learns that a device-side wait gave up. */
nvfp4_status nvfp4_workspace_status(void *workspace, void *stream);

/* Bound of the device-side waits on other CTAs (the grid-wide amax barrier of
 * the one-kernel path, taken by per-tensor rowwise calls of at most 2^22
 * elements) in the calls that follow, in polls of the barrier word: a CTA that
 * sees the barrier still open after `polls` loads gives up, encodes with the
 * maximum it has seen, and records the failure (see the workspace above).
 * polls < 0 restores the default of 2^24 polls (about a second: polls after the
 * first 4096 sleep 64 ns); 0 gives up at once.  Process-wide; returns
 * NVFP4_ERR_INVALID_ARG above 2^32 - 1.  Waits on TMA copies keep their own
 * fixed bound.  The pages have no counterpart: this tunes (and lets a test
 * exercise) the failure path. */
nvfp4_status nvfp4_set_wait_limit(int64_t polls);

/* Bytes of one scale array for an [rows_out, cols_out] output (swizzle
 * padding included when flags has NVFP4_SWIZZLED). */
size_t nvfp4_scale_bytes(int64_t rows_out, int64_t cols_out, uint32_t flags);

/* Global amax of the (optionally RHT-transformed) input: writes out->amax and
 * out->global_scale (= amax / 2688).  orientation: NVFP4_ROWWISE or
 * NVFP4_COLWISE (decides along which dimension the RHT blocks run; irrelevant
 * without RHT).  With NVFP4_SCALE_PER_ROW one value per output row is written
 * (rowwise only). */
nvfp4_status nvfp4_amax(const nvfp4_input *in, uint32_t flags, int use_rht, uint16_t sign_mask,
                        nvfp4_output *out, void *workspace, void *stream);

/* Round-to-nearest-even quantization.  flags: any of ROWWISE/COLWISE (at
 * least one), BLOCK_2D (per-tensor only; needs rows % 16 == 0), SCALE_PER_ROW
 * (rowwise only, single orientation), SWIZZLED, AMAX_GIVEN. */
nvfp4_status nvfp4_quantize_rne(const nvfp4_input *in, uint32_t flags, nvfp4_output *out,
                                void *workspace, void *stream);

/* Stochastic rounding driven by Philox4x32-10: key = (seed lo32, seed hi32),
 * counter = (blk lo32, blk hi32, offset lo32, offset hi32), blk the row-major
 * index of the 16-element block in the output orientation; element e of a
 * block uses byte e&3 of output word e>>2.  The caller advances offset
 * between calls.  Not combinable with BLOCK_2D. */
nvfp4_status nvfp4_quantize_sr(const nvfp4_input *in, uint32_t flags, uint64_t seed, uint64_t offset,
                               nvfp4_output *out, void *workspace, void *stream);

/* 16-point RHT (sign_mask bit j = 1 negates output j of each block) followed
 * by stochastic rounding, as nvfp4_quantize_sr.  Either orientation, or both
 * from one call (the operand of a weight-gradient GEMM needs both): the
 * transform then runs along the rows for the rowwise output and along the
 * columns for the columnwise one, the two amaxes differ, and out->amax and
 * out->global_scale hold two floats, [0] rowwise and [1] columnwise (with
 * NVFP4_AMAX_GIVEN both are read). */
nvfp4_status nvfp4_quantize_rht_sr(const nvfp4_input *in, uint32_t flags, uint16_t sign_mask,
                                   uint64_t seed, uint64_t offset, nvfp4_output *out,
                                   void *workspace, void *stream);

/* nvfp4_quantize_rht_sr without a workspace argument.  The pages have no
 * counterpart: this entry point exists for callers that cannot call cudaMalloc,
 * for instance a serving runtime that reserves its whole device-memory budget
 * at start-up and forbids allocation afterwards, or code that must not trigger
 * the implicit device synchronisation an allocation can cause.  It allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine): the amax
 * pass's scratch lives in a 256-byte device array inside the library, which
 * every GPU that loads the library keeps until the process exits.  The passes
 * need at most 24 of those bytes for any input size; the call returns
 * NVFP4_ERR_UNSUPPORTED if the library's workspace need ever exceeds the array.
 * Inputs and outputs are as for nvfp4_quantize_rht_sr, whose checks (sizes
 * included) apply unchanged.
 *
 * The first call on a device looks the array's device address up
 * (cudaGetSymbolAddress) with that device current and caches it for the life
 * of the process; make that first call before any stream capture.  The cached
 * address does not survive cudaDeviceReset (or any other teardown of the
 * device's primary context): do not call this entry point after one.  Every
 * call then clears the scratch
 * on the given stream (it is cleared even when the arguments are rejected; no
 * caller buffer is touched in that case).  All calls share the one array:
 * calls whose work overlaps on the GPU (other streams, other threads) race on
 * it and must be serialised by the caller. */
nvfp4_status nvfp4_quantize_rht_sr_static(const nvfp4_input *in, uint32_t flags, uint16_t sign_mask,
                                          uint64_t seed, uint64_t offset, nvfp4_output *out, void *stream);

/* Four-over-six (RNE candidates for M = 6 and M = 4).  1x16 blocks, per-tensor
 * or per-row global scale; per-row needs exactly one orientation (rowwise). */
nvfp4_status nvfp4_quantize_four_over_six(const nvfp4_input *in, uint32_t flags, nvfp4_output *out,
                                          void *workspace, void *stream);

/* Grouped rowwise quantize: many tensors in one call, e.g. the tokens routed
 * to each expert of a mixture-of-experts layer, stacked as the row ranges of
 * one input ("[nvfp4 training][rl] Add a CuTe DSL fast-path kernel for
 * four-over-six quantize #4852", PR description: grouped / MoE quantization is
 * the named follow-up).  group_offsets is a DEVICE array of n_groups+1
 * non-decreasing row indices, group_offsets[0] = 0 and group_offsets[n_groups]
 * = rows (1 <= n_groups < 2^31; empty groups allowed, so n_groups may exceed
 * rows); group g is rows [group_offsets[g], group_offsets[g+1]) (it may be
 * empty) and is quantized as a tensor of its own: its own amax and global
 * scale (out->amax and out->global_scale hold n_groups floats; an empty group
 * gets amax 0, or the amax given with NVFP4_AMAX_GIVEN, and scale amax / 2688),
 * with the block scales and codes written into the rows of the one output.  Philox blocks keep their numbers in the whole input.  mode: one of
 * NVFP4_MODE_*.  flags: NVFP4_ROWWISE (required), NVFP4_SWIZZLED,
 * NVFP4_AMAX_GIVEN (out->amax holds the n_groups amaxes).  Needs no
 * workspace.  Launches an amax kernel, a tiny finalising kernel and the tiled
 * rowwise quantize kernel, which encodes each row with its group's scale
 * (divisor tables of two groups per CTA; rows of groups shorter than a tile
 * compute their divisors directly, with the same result).  NVFP4_ERR_UNSUPPORTED
 * only if the input's tensor map cannot be made and a row is longer than
 * 96 KiB (the per-row fallback stages whole rows in shared memory). */
enum { NVFP4_MODE_RNE = 0, NVFP4_MODE_SR = 1, NVFP4_MODE_RHT_SR = 2, NVFP4_MODE_FOUR_OVER_SIX = 3 };
nvfp4_status nvfp4_quantize_grouped(const nvfp4_input *in, uint32_t flags, const int64_t *group_offsets,
                                    int64_t n_groups, int32_t mode, uint16_t sign_mask, uint64_t seed,
                                    uint64_t offset, nvfp4_output *out, void *stream);

/* Standard NVFP4 decode: out[r][c] = value(code) * (Sf * g), both products
 * rounded to fp32 (then to bf16 for a bf16 output).  codes [rows, cols/2],
 * scales linear or swizzled per flags (NVFP4_SWIZZLED), global_scale 1 float or
 * one per row (NVFP4_SCALE_PER_ROW).  out is a dense [rows, cols] array of
 * out_dtype (nvfp4_dtype).  cols % 16 == 0. */
nvfp4_status nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales, const float *global_scale,
                              int64_t rows, int64_t cols, uint32_t flags, void *out, int32_t out_dtype,
                              void *stream);

/* Decode of codes produced with the RHT (nvfp4_quantize_rht_sr, rowwise or
 * columnwise output), mapped back to the source basis: the standard decode of
 * each 16-block as nvfp4_dequantize (fp32), then the inverse transform
 * v = ((y . diag(s)) . H16) / 4 (signs on the inputs, the butterfly with
 * strides 1, 2, 4, 8, then x 0.25), then the output rounding.  sign_mask is the
 * one the codes were produced with.  For a columnwise output pass
 * rows = cols of X and cols = rows of X: the result is then X^T.  Arguments
 * and checks as nvfp4_dequantize. */
nvfp4_status nvfp4_dequantize_rht(const uint8_t *codes, const uint8_t *scales, const float *global_scale,
                                  int64_t rows, int64_t cols, uint32_t flags, uint16_t sign_mask, void *out,
                                  int32_t out_dtype, void *stream);

/* Human-readable name of a status. */
const char *nvfp4_status_string(nvfp4_status status);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H */
