// moe_layer_forward_noalloc: the MoE layer with its scratch in a static device
// array instead of a caller-provided workspace.
//
// Who needs this: callers that cannot allocate device memory at the point where
// they run the layer - for example code running inside a host callback or a
// plugin whose host framework owns every device allocation, or a process whose
// memory budget is fixed before the layer is set up. Such a caller still owns
// x, y and the weights; only the layer's scratch (router logits, top-k lists,
// SwiGLU intermediates, the block start counter) comes from here.
//
// The scratch is one file-scope __device__ array of kNoallocScratchBytes bytes.
// Every GPU that loads this library keeps that much memory reserved until the
// process exits. The host only has a stand-in for the array's name: its device
// address is obtained once per device with cudaGetSymbolAddress, with that
// device current, on the first call made on that device.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = 8u << 20;   // 8 MiB per device (a 64-token call of a
                                                     // 2048-wide, 256-expert, top-8 layer needs 6.0 MB)

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev];
std::atomic<int> g_scratch_ready[kMaxDev];
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (set up once per device).
nvfp4_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return NVFP4_ERR_CUDA;
    if (g_scratch_ready[dev].load(std::memory_order_acquire) == 0) {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        if (g_scratch_ready[dev].load(std::memory_order_relaxed) == 0) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return NVFP4_ERR_CUDA;
            g_scratch_ptr[dev] = p;
            g_scratch_ready[dev].store(1, std::memory_order_release);
        }
    }
    *out = g_scratch_ptr[dev];
    return NVFP4_OK;
}

}  // namespace

extern "C" {

nvfp4_status moe_layer_forward_noalloc(const moe_layer_desc* d, const uint16_t* x, int32_t T, uint16_t* y,
                                       int32_t* topk_ids_out, float* topk_w_out, void* stream) {
    if (!d || T < 0) return NVFP4_ERR_INVALID_ARG;
    if (d->H <= 0 || d->E <= 0 || d->k <= 0 || d->I <= 0 || d->Is < 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    const size_t need = moe_layer_workspace_size(d, T);
    if (need > kNoallocScratchBytes) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    nvfp4_status st = scratch_address(&scratch);
    if (st != NVFP4_OK) return st;
    // The array keeps whatever the previous call left in it; the layer expects a
    // zeroed workspace header and no stale exchange words, so clear the part used.
    if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess) return NVFP4_ERR_CUDA;
    return moe_layer_forward(d, x, T, y, topk_ids_out, topk_w_out, scratch, kNoallocScratchBytes, stream);
}

nvfp4_status nvfp4_noalloc_status(int32_t clear, void* stream) {
    void* scratch = nullptr;
    const nvfp4_status st = scratch_address(&scratch);
    if (st != NVFP4_OK) return st;
    return nvfp4_get_device_status(scratch, clear, stream);   // the array starts with the workspace header
}

}  // extern "C"
