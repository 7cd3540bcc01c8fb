// nvfp4_static.cu -- the RHT + stochastic-rounding quantize for callers that
// cannot allocate device memory.
//
// The per-tensor amax pass needs a few words of device scratch (a running
// maximum, a CTA ticket and a status word).  nvfp4_quantize_rht_sr takes that
// scratch from the caller; this variant keeps it in a file-scope device array
// instead, so the caller passes only its inputs and outputs.  The array is part
// of the library image: every GPU that loads the library holds it until the
// process exits.
#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "nvfp4.h"

namespace {

constexpr size_t kStaticScratchBytes = 256;

// Device scratch shared by every call of the entry point below.  Zero at
// module load; each completed amax pass returns it to zero, and every call
// clears it again before its amax pass.
static __device__ __align__(256) uint32_t g_scratch[kStaticScratchBytes / sizeof(uint32_t)];

// In host code g_scratch names a host-side shadow, not device memory, so the
// device address is looked up once per device (with that device current) and
// cached here.
constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

nvfp4_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_UNSUPPORTED;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        p = g_scratch_addr[dev].load(std::memory_order_relaxed);
        if (!p) {
            if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return NVFP4_ERR_CUDA;
            g_scratch_addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = p;
    return NVFP4_OK;
}

}  // namespace

extern "C" nvfp4_status nvfp4_quantize_rht_sr_static(const nvfp4_input *in, uint32_t flags, uint16_t sign_mask,
                                                     uint64_t seed, uint64_t offset, nvfp4_output *out,
                                                     void *stream) {
    if (nvfp4_workspace_bytes() > kStaticScratchBytes) return NVFP4_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const nvfp4_status st = scratch_address(&scratch);
    if (st != NVFP4_OK) return st;
    // the amax pass expects its scratch to start at zero
    if (cudaMemsetAsync(scratch, 0, nvfp4_workspace_bytes(), static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return nvfp4_quantize_rht_sr(in, flags, sign_mask, seed, offset, out, scratch, stream);
}
