// mhc_boundary_fused for callers that cannot allocate device memory: the
// per-slice partials live in a fixed array in the library's own device
// memory instead of a caller workspace. Nothing here allocates.
#include <mutex>

#include <cuda_runtime.h>

#include "mhc.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;   // 4 MiB per device
constexpr int kMaxDevices = 64;

// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the array, looked up once per device. In host code the
// symbol itself is only a host-side stand-in, never a device address.
struct ScratchSlot {
    std::once_flag once;
    void *ptr = nullptr;
    cudaError_t err = cudaSuccess;
};
ScratchSlot g_slots[kMaxDevices];

mhc_status scratch_of_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MHC_ERR_CUDA;
    ScratchSlot &s = g_slots[dev];
    std::call_once(s.once, [&] {
        s.err = cudaGetSymbolAddress(&s.ptr, g_noalloc_scratch);
    });
    if (s.err != cudaSuccess || s.ptr == nullptr) return MHC_ERR_CUDA;
    *out = s.ptr;
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
