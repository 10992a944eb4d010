// mhc_boundary_fused for callers that cannot allocate device memory: the
// per-slice partials live in a fixed array in the library's own device
// memory instead of a caller workspace. Nothing here allocates.
#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "mhc.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;   // 4 MiB per device
constexpr int kMaxDevices = 64;

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the array, looked up per device. In host code the
// symbol itself is only a host-side stand-in, never a device address. Only a
// successful lookup is kept: a lookup that failed (made during a stream
// capture, say, or before the device's context was ready) is retried by the
// next call instead of failing every later call on that device.
struct ScratchSlot {
    std::atomic<void *> ptr{nullptr};
    std::mutex m;
};
ScratchSlot g_slots[kMaxDevices];

mhc_status scratch_of_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MHC_ERR_CUDA;
    ScratchSlot &s = g_slots[dev];
    void *p = s.ptr.load(std::memory_order_acquire);
    if (p == nullptr) {
        std::lock_guard<std::mutex> lock(s.m);
        p = s.ptr.load(std::memory_order_relaxed);
        if (p == nullptr) {
            void *q = nullptr;
            if (cudaGetSymbolAddress(&q, g_noalloc_scratch) != cudaSuccess || q == nullptr) {
                cudaGetLastError();   // clear the error this lookup left behind
                return MHC_ERR_CUDA;
            }
            s.ptr.store(q, std::memory_order_release);
            p = q;
        }
    }
    *out = p;
    return MHC_OK;
}

}  // namespace

extern "C" mhc_status mhc_boundary_fused_noalloc(
    const uint16_t *x, const uint16_t *residual, const float *post, const float *comb,
    const float *pre_lag, const void *weight, const float *scale, const float *base,
    const void *norm_w, mhc_dtype norm_dtype, const mhc_params *params, int64_t tokens,
    int hidden, uint16_t *residual_out, uint16_t *layer_input, float *pre_out, float *post_out,
    float *comb_out, void *stream) {
    if (mhc_workspace_bytes(tokens, hidden) > kScratchBytes) return MHC_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (mhc_status s = scratch_of_current_device(&scratch)) return s;
    return mhc_boundary_fused(x, residual, post, comb, pre_lag, weight, scale, base, norm_w,
                              norm_dtype, params, tokens, hidden, residual_out, layer_input,
                              pre_out, post_out, comb_out, scratch, kScratchBytes, stream);
}
