// noalloc.cu -- moe_expert_forward for callers that must not allocate device
// memory.
//
// moe_expert_forward needs a workspace (routing metadata, the quantized and
// permuted activations, the SwiGLU output and the FC2 rows) that its caller
// allocates.  Some callers cannot: a plugin handed only its input and output
// buffers by a host framework that owns all allocation, or a latency-critical
// step where cudaMalloc/cudaFree would synchronize the device.  For them this
// file keeps one fixed scratch array in device global memory, sized for small
// token counts, and runs the unchanged moe_expert_forward on it.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "../../include/nvfp4moe.h"
#include "kernels.h"

namespace {

// The scratch: every GPU that loads this library holds these 32 MiB until
// the process exits, whether or not the entry point is ever called.
constexpr size_t kScratchBytes = size_t(32) << 20;
__device__ __align__(256) unsigned char g_moe_scratch[kScratchBytes];

// Device address of g_moe_scratch per device.  In host code the array's name
// only stands for the symbol; the device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

int scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nvfp4::set_last_error(NVFP4_ELAUNCH, "moe_expert_forward_noalloc: no usable current CUDA device");
    std::lock_guard<std::mutex> guard(g_lock);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_moe_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char msg[256];
            snprintf(msg, sizeof msg, "moe_expert_forward_noalloc: cudaGetSymbolAddress failed: %s",
                     cudaGetErrorString(e));
            return nvfp4::set_last_error(NVFP4_ELAUNCH, msg);
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return NVFP4_OK;
}

}  // namespace

extern "C" {

NVFP4_API int moe_expert_forward_noalloc(const void* x_bf16, int64_t T, int64_t H, const float* router_logits,
                                         const float* router_bias, int E, int topk, const nvfp4_tensor* w1,
                                         const nvfp4_tensor* w2, int64_t F, const moe_options* opt, void* out_bf16,
                                         void* stream) {
    moe_workspace_layout layout;
    int rc = moe_expert_workspace_layout(T, H, F, E, topk, &layout);  // rejects bad sizes with a message
    if (rc != NVFP4_OK) return rc;
    if (layout.total > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "moe_expert_forward_noalloc: this layer needs %zu bytes of scratch but the built-in array holds "
                 "%zu (fewer tokens, or moe_expert_forward with a caller workspace)",
                 layout.total, kScratchBytes);
        return nvfp4::set_last_error(NVFP4_EWORKSPACE, msg);
    }
    void* ws = nullptr;
    rc = scratch_address(&ws);
    if (rc != NVFP4_OK) return rc;
    // The array keeps the previous call's contents; the device error word must
    // start at zero (every other region is rewritten before it is read).
    cudaError_t e = cudaMemsetAsync(ws, 0, 256, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "moe_expert_forward_noalloc: %s", cudaGetErrorString(e));
        return nvfp4::set_last_error(NVFP4_ELAUNCH, msg);
    }
    return moe_expert_forward(x_bf16, T, H, router_logits, router_bias, E, topk, w1, w2, F, opt, out_bf16,
                              nullptr, ws, kScratchBytes, stream);
}

NVFP4_API int moe_noalloc_error_word(uint32_t** out) {
    if (out == nullptr) return nvfp4::set_last_error(NVFP4_EINVAL, "moe_noalloc_error_word: null out");
    void* ws = nullptr;
    const int rc = scratch_address(&ws);
    if (rc != NVFP4_OK) return rc;
    moe_workspace_layout layout;  // the error word's offset in any layer's workspace (the first field)
    if (moe_expert_workspace_layout(1, 256, 128, 32, 1, &layout) != NVFP4_OK) return NVFP4_ELAUNCH;
    *out = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(ws) + layout.err);
    return NVFP4_OK;
}

}  // extern "C"
