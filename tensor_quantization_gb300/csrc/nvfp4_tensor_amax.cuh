// nvfp4_tensor_amax.cuh -- how the per-tensor amax travels from the amax pass
// to the quantize kernel of the same call.
//
// The amax pass folds each CTA's maximum magnitude bits into workspace[0]
// with one red.max and exits: no fence, no ticket, nothing on its critical
// path.  The quantize kernel waits for the pass (grid_dependency_wait), every
// thread reads the bits, and after the CTA's next barrier thread 0 counts the
// CTA in at workspace[1]; the CTA that counts in last returns both words to
// zero for the next call, and CTA 0 publishes amax and g = amax / 2688.
// (Signs do not change magnitudes and rounding is monotone, so with the RHT
// the pass reduces the raw butterfly outputs and the 0.25 is applied once,
// here.)  The standalone amax entry point publishes from the pass itself: the
// CTA that takes the last ticket writes amax and g.  Either way the host never
// waits ("nvfp4-sm120" README, section "Results": the amax host sync was 86%
// of the quantizer's time).
#pragma once

#include "nvfp4_encode.cuh"
#include "nvfp4_internal.h"
#include "nvfp4_load.cuh"
#include "nvfp4_tma.cuh"

namespace nvfp4 {

// ------------------------------------------------------- give-up records
// Workspace word 3 records that a bounded device-side wait gave up.  It is
// sticky: no kernel clears it, so every later call on the same workspace
// publishes a NaN global scale until the host reads and clears the word
// (nvfp4_workspace_status).  A kernel that gives up sets the word, fences,
// then stores NaN into its global scale; the CTA that publishes the global
// scale stores it, fences, then re-reads the word and stores NaN if it is
// set.  With both fences sequentially consistent, either the publisher sees
// the record or its store precedes the NaN: the NaN always wins.
constexpr int kStatusWord = 3;

__device__ __forceinline__ void wait_gave_up(const QArgs &a, float *gs) {
    atomicAdd(&g_wait_timeouts, 1u);
    if (a.workspace) atomicOr(a.workspace + kStatusWord, 1u);
    __threadfence();
    if (gs) *reinterpret_cast<volatile float *>(gs) = __uint_as_float(0x7FFFFFFFu);
}

__device__ __forceinline__ void publish_gscale(const QArgs &a, float *gs, float g) {
    *reinterpret_cast<volatile float *>(gs) = g;
    if (!a.workspace) return;
    __threadfence();
    uint32_t st;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(st) : "l"(a.workspace + kStatusWord) : "memory");
    if (st) *reinterpret_cast<volatile float *>(gs) = __uint_as_float(0x7FFFFFFFu);
}

// End of an amax pass whose consumer is a quantize kernel: one red.max per CTA.
__device__ __forceinline__ void fold_tensor_amax(const QArgs &a, uint32_t m) {
    __shared__ uint32_t red[32];
    allow_dependents();  // the quantize kernel may start staging its tiles
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(a.workspace), "r"(m) : "memory");
}

// The same without a CTA barrier: each warp folds its maximum into a shared
// word (zeroed before the CTA's first barrier) and the last warp to count in
// sends the CTA's maximum, so no warp waits for another.
__device__ __forceinline__ void fold_tensor_amax_warps(const QArgs &a, uint32_t m, uint32_t *cta_max,
                                                       uint32_t *warps_in) {
    allow_dependents();
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0) {
        atomicMax(cta_max, m);
        __threadfence_block();
        if (atomicAdd(warps_in, 1u) == blockDim.x / 32 - 1) {
            __threadfence_block();
            const uint32_t cm = *reinterpret_cast<volatile uint32_t *>(cta_max);
            asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(a.workspace), "r"(cm) : "memory");
        }
    }
}

// End of a standalone amax pass: the last CTA publishes amax and g and zeroes
// the workspace.
__device__ __forceinline__ void publish_tensor_amax(const QArgs &a, uint32_t m, bool rht) {
    __shared__ uint32_t red[32];
    m = block_max_u32(m, red);
    if (threadIdx.x == 0) {
        atomicMax(&a.workspace[0], m);
        __threadfence();
        const uint32_t ticket = atomicAdd(&a.workspace[1], 1u);
        if (ticket == gridDim.x - 1) {
            __threadfence();
            const uint32_t bits = atomicExch(&a.workspace[0], 0u);
            atomicExch(&a.workspace[1], 0u);
            float A = __uint_as_float(bits);
            if (rht) A = __fmul_rn(A, 0.25f);
            a.amax[0] = A;
            publish_gscale(a, a.gscale, global_scale_of(A));
        }
    }
}

// The tensor amax a quantize kernel encodes with (every thread; after
// grid_dependency_wait): from the workspace after this call's amax pass,
// else a.amax[0] (given by the caller, or published by an earlier kernel of
// the call).
__device__ __forceinline__ float tensor_amax_read(const QArgs &a, bool rht) {
    if (!a.amax_in_ws) return a.amax[0];
    uint32_t bits;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(bits) : "l"(a.workspace + a.amax_word) : "memory");
    const float m = __uint_as_float(bits);
    return rht ? __fmul_rn(m, 0.25f) : m;
}

// Thread 0, after a CTA barrier that follows every thread's
// tensor_amax_read: count the CTA in (the last one clears the workspace,
// acquire-ordered after every other CTA's release-ordered count, hence after
// all of their reads) and, in CTA 0, publish amax and g.
__device__ __forceinline__ void tensor_amax_done(const QArgs &a, float A, float g) {
    if (threadIdx.x != 0) return;
    if (a.amax_in_ws) {
        uint32_t n;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(n) : "l"(a.workspace + a.amax_word + 1)
                     : "memory");
        if (n == gridDim.x - 1) {
            a.workspace[a.amax_word] = 0u;
            a.workspace[a.amax_word + 1] = 0u;
        }
        if (blockIdx.x == 0) a.amax[0] = A;
    }
    if (blockIdx.x == 0) publish_gscale(a, a.gscale, g);
}

}  // namespace nvfp4
