// nvfp4_api.cu -- the C ABI of libnvfp4.so (declared in include/nvfp4.h).
//
// Every entry point validates all of its arguments before enqueuing anything,
// then enqueues kernels on the caller's stream and returns without waiting.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4.h"
#include "nvfp4_internal.h"

namespace nvfp4 {

int sm_count() {
    static int cache[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

}  // namespace nvfp4

namespace {

constexpr uint32_t kKnownFlags = NVFP4_ROWWISE | NVFP4_COLWISE | NVFP4_BLOCK_2D | NVFP4_SCALE_PER_ROW |
                                 NVFP4_SWIZZLED | NVFP4_AMAX_GIVEN | NVFP4_FAST_MATH;
constexpr int64_t kMaxDim = (int64_t)1 << 31;
constexpr int64_t kMaxElems = (int64_t)1 << 34;
// Up to this size a per-tensor rowwise call runs as one kernel; above it the
// amax and quantize kernels (the second launched while the first finishes) are
// as fast or faster (measured on GB300 from 2^19 to 2^27 elements).
constexpr int64_t kFusedMaxElems = (int64_t)1 << 22;

// Bound of the device-side waits on other CTAs for the calls that follow
// (nvfp4_set_wait_limit).
std::atomic<uint32_t> g_grid_polls{nvfp4::kDefaultGridPolls};

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t elem_size(int32_t dtype) { return dtype == NVFP4_IN_FP32 ? 4 : 2; }

// The call's Philox4x32-10 seed and offset, and the round keys of the seed
// (key + round * Weyl constant), computed on the host once per call so that
// kernels read them from the parameter bank.
void set_philox(nvfp4::QArgs &a, uint64_t seed, uint64_t offset) {
    a.seed = seed;
    a.offset = offset;
    for (int i = 0; i < 10; i++) {
        a.round_key0[i] = (uint32_t)seed + (uint32_t)i * 0x9E3779B9u;
        a.round_key1[i] = (uint32_t)(seed >> 32) + (uint32_t)i * 0xBB67AE85u;
    }
}

// Shape, stride and pointer checks shared by every entry point that reads X.
nvfp4_status check_input(const nvfp4_input *in) {
    if (!in) return NVFP4_ERR_INVALID_ARG;
    if (in->dtype != NVFP4_IN_BF16 && in->dtype != NVFP4_IN_FP32) return NVFP4_ERR_INVALID_ARG;
    if (in->rows < 0 || in->cols < 0 || in->rows >= kMaxDim || in->cols >= kMaxDim) return NVFP4_ERR_INVALID_ARG;
    if (in->rows * in->cols > kMaxElems) return NVFP4_ERR_INVALID_ARG;
    if (in->row0 < 0 || in->col0 < 0 || in->row0 >= kMaxDim || in->col0 >= kMaxDim) return NVFP4_ERR_INVALID_ARG;
    if (in->rows == 0 || in->cols == 0) return NVFP4_OK;
    if (!in->x || !aligned(in->x, 16)) return NVFP4_ERR_INVALID_ARG;
    if (in->ld < in->cols || (in->ld * elem_size(in->dtype)) % 16 != 0) return NVFP4_ERR_INVALID_ARG;
    return NVFP4_OK;
}

nvfp4_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

nvfp4::QArgs make_args(const nvfp4_input *in, const nvfp4_output *out, void *ws, uint32_t flags) {
    nvfp4::QArgs a{};
    a.x = in->x;
    a.rows = in->rows;
    a.cols = in->cols;
    a.ld = in->ld;
    a.codes_row = out->codes_row;
    a.scales_row = out->scales_row;
    a.codes_col = out->codes_col;
    a.scales_col = out->scales_col;
    a.amax = out->amax;
    a.gscale = out->global_scale;
    a.workspace = static_cast<uint32_t *>(ws);
    a.swizzled = (flags & NVFP4_SWIZZLED) ? 1 : 0;
    a.want_row = (flags & NVFP4_ROWWISE) ? 1 : 0;
    a.want_col = (flags & NVFP4_COLWISE) ? 1 : 0;
    a.grid_polls = g_grid_polls.load(std::memory_order_relaxed);
    return a;
}

nvfp4_status quantize(const nvfp4_input *in, uint32_t flags, int mode, bool rht, uint16_t sign_mask,
                      uint64_t seed, uint64_t offset, nvfp4_output *out, void *ws, void *stream) {
    nvfp4_status st = check_input(in);
    if (st != NVFP4_OK) return st;
    if (!out || (flags & ~kKnownFlags)) return NVFP4_ERR_INVALID_ARG;
    const bool want_row = flags & NVFP4_ROWWISE, want_col = flags & NVFP4_COLWISE;
    const bool block2d = flags & NVFP4_BLOCK_2D, per_row = flags & NVFP4_SCALE_PER_ROW;
    const bool given = flags & NVFP4_AMAX_GIVEN, swz = flags & NVFP4_SWIZZLED;
    if (!want_row && !want_col) return NVFP4_ERR_INVALID_ARG;
    if (block2d && (mode != nvfp4::MODE_RNE_ID || rht || per_row)) return NVFP4_ERR_UNSUPPORTED;
    if (per_row && (want_col || given)) return NVFP4_ERR_UNSUPPORTED;
    if (rht && mode == nvfp4::MODE_4O6_ID) return NVFP4_ERR_UNSUPPORTED;
    if ((flags & NVFP4_FAST_MATH) && mode == nvfp4::MODE_4O6_ID) return NVFP4_ERR_UNSUPPORTED;
    // a stochastic shard is cut along its output rows only
    if (mode == nvfp4::MODE_SR_ID && ((want_row && in->col0 != 0) || (want_col && in->row0 != 0)))
        return NVFP4_ERR_UNSUPPORTED;
    if ((want_row || block2d) && in->cols % 16 != 0) return NVFP4_ERR_INVALID_ARG;
    if ((want_col || block2d) && in->rows % 16 != 0) return NVFP4_ERR_INVALID_ARG;
    const bool empty = in->rows == 0 || in->cols == 0;
    // an empty input has empty code and scale arrays, which may be NULL
    if (!empty && want_row && (!out->codes_row || !out->scales_row || !aligned(out->codes_row, 8)))
        return NVFP4_ERR_INVALID_ARG;
    if (!empty && want_col && (!out->codes_col || !out->scales_col || !aligned(out->codes_col, 8)))
        return NVFP4_ERR_INVALID_ARG;
    // per row: one scale per row; RHT in both orientations: one per orientation
    // (the transform runs along different axes, so the two amaxes differ)
    const bool two_scales = rht && want_row && want_col;
    const int64_t n_scale = per_row ? in->rows : (two_scales ? 2 : 1);
    if (n_scale > 0 && (!out->amax || !out->global_scale)) return NVFP4_ERR_INVALID_ARG;
    if (!per_row && !given && !empty && (!ws || !aligned(ws, 8))) return NVFP4_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (empty) {
        // nothing to encode; an empty tensor (or row) has amax 0 and scale 0
        if (!given && n_scale > 0 && cudaMemsetAsync(out->amax, 0, n_scale * sizeof(float), s) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        if (n_scale > 0 && cudaMemsetAsync(out->global_scale, 0, n_scale * sizeof(float), s) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        return NVFP4_OK;
    }

    nvfp4::QArgs a = make_args(in, out, ws, flags);
    a.sign_mask = sign_mask;
    set_philox(a, seed, offset);
    a.fast_math = (flags & NVFP4_FAST_MATH) ? 1 : 0;
    const bool fp32 = in->dtype == NVFP4_IN_FP32;
    const uint64_t base_row = (uint64_t)in->row0 * (uint64_t)(in->cols / 16);  // rowwise block numbers
    const uint64_t base_col = (uint64_t)in->col0 * (uint64_t)(in->rows / 16);  // columnwise block numbers
    a.blk_base = base_row;
    bool fused = false;
    if (!per_row && !given && !block2d && want_row && !want_col && in->rows * in->cols <= kFusedMaxElems) {
        // a small tensor: amax pass and quantize in one cooperative launch
        // (if the launch is refused, nothing was enqueued: two kernels then)
        fused = nvfp4::launch_quant_row_fused(a, fp32, mode, rht, s) == cudaSuccess;
        if (!fused) (void)cudaGetLastError();
    }
    if (fused) {
    } else if (per_row) {
        st = cuda_status(nvfp4::launch_quant_rowscaled(a, fp32, mode, rht, s));
    } else {
        // bf16 RHT column blocks: one TMA pass, which with both orientations
        // also reduces the row blocks (two maxima from one read)
        const bool tma_cols = rht && want_col && !fp32 && !block2d;
        if (!given) {
            // the next quantize kernel takes the amax from the workspace and
            // publishes it; a second one reads the published amax[0]
            st = cuda_status(tma_cols ? nvfp4::launch_amax_cols(a, want_row, s)
                                      : nvfp4::launch_amax_tensor(a, fp32, rht, rht && want_col && !want_row, false, s));
            if (st != NVFP4_OK) return st;
            a.amax_in_ws = 1;
        }
        if (block2d) {
            st = cuda_status(nvfp4::launch_quant_2d(a, fp32, s));
        } else if (two_scales) {
            // rowwise with amax[0] / global_scale[0], then columnwise with [1]
            nvfp4::QArgs ar = a, ac = a;
            ar.want_col = 0;
            ac.want_row = 0;
            ac.amax = out->amax + 1;
            ac.gscale = out->global_scale + 1;
            ac.blk_base = base_col;
            st = cuda_status(nvfp4::launch_quant_row(ar, fp32, mode, rht, s));
            if (tma_cols) ac.amax_word = 4;  // the column maximum of the one read
            else if (st == NVFP4_OK && !given) st = cuda_status(nvfp4::launch_amax_tensor(ac, fp32, rht, true, false, s));
            if (st == NVFP4_OK) st = cuda_status(nvfp4::launch_quant_col(ac, fp32, mode, rht, s));
        } else {
            if (want_row) {
                st = cuda_status(nvfp4::launch_quant_row(a, fp32, mode, rht, s));
                a.amax_in_ws = 0;
            }
            if (st == NVFP4_OK && want_col) {
                a.blk_base = base_col;
                st = cuda_status(nvfp4::launch_quant_col(a, fp32, mode, rht, s));
            }
        }
    }
    if (st != NVFP4_OK) return st;
    if (swz) {
        if (want_row) st = cuda_status(nvfp4::launch_scale_pad(out->scales_row, in->rows, in->cols / 16, s));
        if (st == NVFP4_OK && want_col) st = cuda_status(nvfp4::launch_scale_pad(out->scales_col, in->cols, in->rows / 16, s));
    }
    return st;
}

}  // namespace

extern "C" {

size_t nvfp4_workspace_bytes(void) { return 256; }

size_t nvfp4_scale_bytes(int64_t rows_out, int64_t cols_out, uint32_t flags) {
    if (rows_out < 0 || cols_out < 0) return 0;
    const int64_t cs = cols_out / 16;
    if (!(flags & NVFP4_SWIZZLED)) return (size_t)(rows_out * cs);
    return (size_t)(((rows_out + 127) / 128 * 128) * ((cs + 3) / 4 * 4));
}

nvfp4_status nvfp4_amax(const nvfp4_input *in, uint32_t flags, int use_rht, uint16_t sign_mask,
                        nvfp4_output *out, void *workspace, void *stream) {
    (void)sign_mask;  // signs do not change magnitudes
    nvfp4_status st = check_input(in);
    if (st != NVFP4_OK) return st;
    if (!out || !out->amax || !out->global_scale) return NVFP4_ERR_INVALID_ARG;
    if (flags & ~(uint32_t)(NVFP4_ROWWISE | NVFP4_COLWISE | NVFP4_SCALE_PER_ROW)) return NVFP4_ERR_INVALID_ARG;
    const bool col = (flags & NVFP4_COLWISE) && !(flags & NVFP4_ROWWISE);
    const bool per_row = flags & NVFP4_SCALE_PER_ROW;
    if (per_row && col) return NVFP4_ERR_UNSUPPORTED;
    if ((per_row || (use_rht && !col)) && in->cols % 16 != 0) return NVFP4_ERR_INVALID_ARG;
    if (use_rht && col && in->rows % 16 != 0) return NVFP4_ERR_INVALID_ARG;
    const bool empty = in->rows == 0 || in->cols == 0;
    if (!per_row && !empty && !workspace) return NVFP4_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (empty) {
        const int64_t n = per_row ? in->rows : 1;
        if (n > 0 && (cudaMemsetAsync(out->amax, 0, n * sizeof(float), s) != cudaSuccess ||
                      cudaMemsetAsync(out->global_scale, 0, n * sizeof(float), s) != cudaSuccess))
            return NVFP4_ERR_CUDA;
        return NVFP4_OK;
    }
    nvfp4::QArgs a = make_args(in, out, workspace, 0);
    const bool fp32 = in->dtype == NVFP4_IN_FP32;
    if (per_row) return cuda_status(nvfp4::launch_amax_rows(a, fp32, use_rht != 0, s));
    return cuda_status(nvfp4::launch_amax_tensor(a, fp32, use_rht != 0, col, true, s));
}

nvfp4_status nvfp4_quantize_rne(const nvfp4_input *in, uint32_t flags, nvfp4_output *out, void *workspace,
                                void *stream) {
    return quantize(in, flags, nvfp4::MODE_RNE_ID, false, 0, 0, 0, out, workspace, stream);
}

nvfp4_status nvfp4_quantize_sr(const nvfp4_input *in, uint32_t flags, uint64_t seed, uint64_t offset,
                               nvfp4_output *out, void *workspace, void *stream) {
    return quantize(in, flags, nvfp4::MODE_SR_ID, false, 0, seed, offset, out, workspace, stream);
}

nvfp4_status nvfp4_quantize_rht_sr(const nvfp4_input *in, uint32_t flags, uint16_t sign_mask, uint64_t seed,
                                   uint64_t offset, nvfp4_output *out, void *workspace, void *stream) {
    return quantize(in, flags, nvfp4::MODE_SR_ID, true, sign_mask, seed, offset, out, workspace, stream);
}

nvfp4_status nvfp4_quantize_four_over_six(const nvfp4_input *in, uint32_t flags, nvfp4_output *out,
                                          void *workspace, void *stream) {
    return quantize(in, flags, nvfp4::MODE_4O6_ID, false, 0, 0, 0, out, workspace, stream);
}

nvfp4_status nvfp4_quantize_grouped(const nvfp4_input *in, uint32_t flags, const int64_t *group_offsets,
                                    int64_t n_groups, int32_t mode, uint16_t sign_mask, uint64_t seed,
                                    uint64_t offset, nvfp4_output *out, void *stream) {
    nvfp4_status st = check_input(in);
    if (st != NVFP4_OK) return st;
    if (!out || (flags & ~(uint32_t)(NVFP4_ROWWISE | NVFP4_SWIZZLED | NVFP4_AMAX_GIVEN | NVFP4_COLWISE |
                                     NVFP4_BLOCK_2D | NVFP4_SCALE_PER_ROW | NVFP4_FAST_MATH)))
        return NVFP4_ERR_INVALID_ARG;
    if (!(flags & NVFP4_ROWWISE)) return NVFP4_ERR_INVALID_ARG;
    if (flags & (NVFP4_COLWISE | NVFP4_BLOCK_2D | NVFP4_SCALE_PER_ROW | NVFP4_FAST_MATH)) return NVFP4_ERR_UNSUPPORTED;
    if (mode < NVFP4_MODE_RNE || mode > NVFP4_MODE_FOUR_OVER_SIX) return NVFP4_ERR_INVALID_ARG;
    // groups may be empty, so there can be more groups than rows (experts without tokens)
    if (n_groups < 1 || n_groups >= kMaxDim || !group_offsets) return NVFP4_ERR_INVALID_ARG;
    if (in->cols % 16 != 0 || in->col0 != 0) return NVFP4_ERR_INVALID_ARG;
    if (!out->amax || !out->global_scale) return NVFP4_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool given = flags & NVFP4_AMAX_GIVEN;
    const bool rht = mode == NVFP4_MODE_RHT_SR;
    nvfp4::QArgs a = make_args(in, out, nullptr, flags);
    a.group_offsets = group_offsets;
    a.n_groups = n_groups;
    if (in->rows == 0 || in->cols == 0) {  // every group empty: amax 0 (or as given), g = amax / 2688
        if (!given && cudaMemsetAsync(out->amax, 0, n_groups * sizeof(float), s) != cudaSuccess) return NVFP4_ERR_CUDA;
        return cuda_status(nvfp4::launch_group_finalize(a, false, given, s));
    }
    if (!out->codes_row || !out->scales_row || !aligned(out->codes_row, 8)) return NVFP4_ERR_INVALID_ARG;

    a.sign_mask = sign_mask;
    set_philox(a, seed, offset);
    a.blk_base = (uint64_t)in->row0 * (uint64_t)(in->cols / 16);
    const bool fp32 = in->dtype == NVFP4_IN_FP32;
    const int kmode = mode == NVFP4_MODE_RNE ? nvfp4::MODE_RNE_ID
                      : mode == NVFP4_MODE_FOUR_OVER_SIX ? nvfp4::MODE_4O6_ID
                                                         : nvfp4::MODE_SR_ID;
    if (!given) {
        if (cudaMemsetAsync(out->amax, 0, n_groups * sizeof(float), s) != cudaSuccess) return NVFP4_ERR_CUDA;
        st = cuda_status(nvfp4::launch_amax_groups(a, fp32, rht, s));
        if (st != NVFP4_OK) return st;
    }
    st = cuda_status(nvfp4::launch_group_finalize(a, rht, given, s));
    if (st != NVFP4_OK) return st;
    bool padded = true;
    const cudaError_t e = nvfp4::launch_quant_grouped(a, fp32, kmode, rht, &padded, s);
    if (e == cudaErrorNotSupported) return NVFP4_ERR_UNSUPPORTED;
    st = cuda_status(e);
    if (st == NVFP4_OK && !padded && (flags & NVFP4_SWIZZLED))
        st = cuda_status(nvfp4::launch_scale_pad(out->scales_row, in->rows, in->cols / 16, s));
    return st;
}

static nvfp4_status dequantize(const uint8_t *codes, const uint8_t *scales, const float *global_scale, int64_t rows,
                               int64_t cols, uint32_t flags, int rht, uint32_t sign_mask, void *out, int32_t out_dtype,
                               void *stream) {
    if (flags & ~(uint32_t)(NVFP4_SWIZZLED | NVFP4_SCALE_PER_ROW)) return NVFP4_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || rows >= kMaxDim || cols >= kMaxDim || rows * cols > kMaxElems || cols % 16 != 0)
        return NVFP4_ERR_INVALID_ARG;
    if (out_dtype != NVFP4_IN_BF16 && out_dtype != NVFP4_IN_FP32) return NVFP4_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return NVFP4_OK;
    if (!codes || !scales || !global_scale || !out || !aligned(codes, 8) || !aligned(out, 16))
        return NVFP4_ERR_INVALID_ARG;
    return cuda_status(nvfp4::launch_dequant(codes, scales, global_scale, rows, cols,
                                             (flags & NVFP4_SWIZZLED) ? 1 : 0, (flags & NVFP4_SCALE_PER_ROW) ? 1 : 0,
                                             out, out_dtype == NVFP4_IN_FP32, rht, sign_mask,
                                             static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales, const float *global_scale,
                              int64_t rows, int64_t cols, uint32_t flags, void *out, int32_t out_dtype,
                              void *stream) {
    return dequantize(codes, scales, global_scale, rows, cols, flags, 0, 0, out, out_dtype, stream);
}

nvfp4_status nvfp4_dequantize_rht(const uint8_t *codes, const uint8_t *scales, const float *global_scale,
                                  int64_t rows, int64_t cols, uint32_t flags, uint16_t sign_mask, void *out,
                                  int32_t out_dtype, void *stream) {
    return dequantize(codes, scales, global_scale, rows, cols, flags, 1, sign_mask, out, out_dtype, stream);
}

nvfp4_status nvfp4_set_wait_limit(int64_t polls) {
    if (polls > (int64_t)UINT32_MAX) return NVFP4_ERR_INVALID_ARG;
    g_grid_polls.store(polls < 0 ? nvfp4::kDefaultGridPolls : (uint32_t)polls, std::memory_order_relaxed);
    return NVFP4_OK;
}

nvfp4_status nvfp4_workspace_status(void *workspace, void *stream) {
    if (!workspace || !aligned(workspace, 8)) return NVFP4_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t *word = static_cast<uint32_t *>(workspace) + 3;  // the give-up record
    uint32_t rec = 0;
    if (cudaMemcpyAsync(&rec, word, sizeof(rec), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (rec == 0) return NVFP4_OK;
    if (cudaMemsetAsync(word, 0, sizeof(rec), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return NVFP4_ERR_TIMEOUT;
}

const char *nvfp4_status_string(nvfp4_status status) {
    switch (status) {
        case NVFP4_OK: return "ok";
        case NVFP4_ERR_INVALID_ARG: return "invalid argument";
        case NVFP4_ERR_UNSUPPORTED: return "unsupported combination";
        case NVFP4_ERR_CUDA: return "CUDA error";
        case NVFP4_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
