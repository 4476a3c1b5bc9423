// C ABI of the library (declared in include/nvfp4moe.h): host-side argument
// checks, workspace carving and dispatch to the sm_103a kernels. Nothing here
// allocates memory; nothing falls back to another implementation.
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "kernels.cuh"

using namespace nvfp4;

namespace {

std::atomic<uint64_t> g_wait_limit{kDefaultWaitLimit};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::atomic<int> g_dev_ready[kMaxDevices];

nvfp4_status device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    if (g_dev_ready[dev].load(std::memory_order_acquire) == 0) {
        DeviceInfo d{};
        d.device = dev;
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return NVFP4_ERR_CUDA;
        d.num_sms = v;
        if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return NVFP4_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return NVFP4_ERR_CUDA;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return NVFP4_ERR_CUDA;
        d.smem_optin = (size_t)v;
        g_dev[dev] = d;
        g_dev_ready[dev].store(1, std::memory_order_release);
    }
    *out = g_dev[dev];
    if (out->cc_major != 10 || out->cc_minor != 3) return NVFP4_ERR_ARCH;
    return NVFP4_OK;
}

// Scratch bytes of one moe_layer_forward call: the prefill path's for T > 64 with
// E4M3 scales; FP16-scaled layers run T > 64 as 64-token chunks of the decode path.
size_t layer_bytes(const moe_layer_desc& d, int T) {
    if (T > NVFP4_DECODE_MAX_TOKENS)
        return prefill_supported(d, T) ? prefill_ws_bytes(d, T) : layer_ws_bytes(d, NVFP4_DECODE_MAX_TOKENS);
    return layer_ws_bytes(d, T);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool known_kind(int k) {
    return k == NVFP4_SCALE_E4M3 || k == NVFP4_SCALE_FP16 || k == NVFP4_SCALE_FP32 || k == NVFP4_SCALE_UE8M0;
}

nvfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

nvfp4_status check_weight(const nvfp4_weight* W) {
    if (!W || !W->packed || !W->scales || !W->tensor_scale) return NVFP4_ERR_INVALID_ARG;
    if (!known_kind(W->kind)) return NVFP4_ERR_INVALID_ARG;
    if (W->N < 1 || W->K < 32) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (W->K % 32 != 0 || W->K > 8192 || W->N > (1 << 22)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    // the GEMV moves 8-row chunks of scales with 16-byte copies: E8M0 rows of K/32 bytes need K % 64
    if (W->kind == NVFP4_SCALE_UE8M0 && W->K % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(W->packed) || !aligned16(W->scales) || (reinterpret_cast<uintptr_t>(W->tensor_scale) & 3u))
        return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

nvfp4_status check_layer(const moe_layer_desc* d) {
    if (!d) return NVFP4_ERR_INVALID_ARG;
    if (!known_kind(d->kind)) return NVFP4_ERR_INVALID_ARG;
    if (d->H < 32 || d->H % 32 != 0 || d->H > 8192) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (d->I < 32 || d->I % 32 != 0 || d->I > 8192) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (d->Is < 0 || d->Is % 32 != 0 || d->Is > 8192) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (d->E < 1 || d->E > NVFP4_MAX_EXPERTS) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (d->k < 1 || d->k > NVFP4_MAX_TOPK || d->k > d->E) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    const void* req[] = {d->router_w, d->gu_packed, d->gu_scales, d->gu_tscale,
                         d->dn_packed, d->dn_scales, d->dn_tscale};
    for (const void* p : req) {
        if (!p) return NVFP4_ERR_INVALID_ARG;
        if (!aligned16(p)) return NVFP4_ERR_MISALIGNED;
    }
    if (d->Is > 0) {
        const void* sh[] = {d->sh_gu_packed, d->sh_gu_scales, d->sh_gu_tscale, d->sh_dn_packed,
                            d->sh_dn_scales, d->sh_dn_tscale, d->sh_gate_w};
        for (const void* p : sh) {
            if (!p) return NVFP4_ERR_INVALID_ARG;
            if (!aligned16(p)) return NVFP4_ERR_MISALIGNED;
        }
    }
    return NVFP4_OK;
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Scratch of moe_layer_forward_residual: the layer's, then the normalised rows.
size_t residual_bytes(const moe_layer_desc& d, int T) {
    return align256(layer_bytes(d, T)) + align256((size_t)T * d.H * 2);
}

// Run the layer on validated arguments (T >= 1); resid (nullable) is added to every output
// element before its rounding.
nvfp4_status dispatch_layer(const moe_layer_desc& d, const uint16_t* x, int T, uint16_t* y, int32_t* ids_out,
                            float* w_out, void* workspace, const DeviceInfo& dev, cudaStream_t s,
                            const uint16_t* resid) {
    if (T > NVFP4_DECODE_MAX_TOKENS) {
        if (prefill_supported(d, T)) {
            PrefillWs pws = carve_prefill_ws(workspace, d, T);
            return from_cuda(launch_moe_prefill(d, x, T, y, ids_out, w_out, pws, g_wait_limit.load(), s, resid));
        }
        LayerWs cws = carve_layer_ws(workspace, d, NVFP4_DECODE_MAX_TOKENS);
        for (int t0 = 0; t0 < T; t0 += NVFP4_DECODE_MAX_TOKENS) {
            const int tc = T - t0 < NVFP4_DECODE_MAX_TOKENS ? T - t0 : NVFP4_DECODE_MAX_TOKENS;
            const size_t xo = (size_t)t0 * d.H, ko = (size_t)t0 * d.k;
            cudaError_t e = launch_moe_decode(d, x + xo, tc, y + xo, ids_out ? ids_out + ko : nullptr,
                                              w_out ? w_out + ko : nullptr, cws, dev, g_wait_limit.load(), s,
                                              resid ? resid + xo : nullptr);
            if (e != cudaSuccess) return NVFP4_ERR_CUDA;
        }
        return NVFP4_OK;
    }
    LayerWs ws = carve_layer_ws(workspace, d, T);
    if (fused_decode_supported(d, T, dev))
        return from_cuda(launch_moe_decode_fused(d, x, y, ids_out, w_out, ws, dev, g_wait_limit.load(), s,
                                                 nullptr, 0.f, resid));
    return from_cuda(launch_moe_decode(d, x, T, y, ids_out, w_out, ws, dev, g_wait_limit.load(), s, resid));
}

}  // namespace

extern "C" {

size_t nvfp4_pack_workspace_size(void) { return sizeof(WsHeader); }

nvfp4_status nvfp4_pack(const float* w, int32_t N, int32_t K, int32_t kind, uint8_t* packed,
                        void* scales, float* tensor_scale, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if (!w || !packed || !scales || !tensor_scale || !workspace) return NVFP4_ERR_INVALID_ARG;
    if (!known_kind(kind)) return NVFP4_ERR_INVALID_ARG;
    const int blk = kind == NVFP4_SCALE_UE8M0 ? 32 : 16;
    if (N < 1 || K < blk || K % blk != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(w) || !aligned16(packed) || !aligned16(scales) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(tensor_scale) & 3u))
        return NVFP4_ERR_MISALIGNED;
    if (workspace_bytes < nvfp4_pack_workspace_size()) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo dev;
    nvfp4_status st = device_info(&dev);
    if (st != NVFP4_OK) return st;
    return from_cuda(launch_pack(w, N, K, kind, packed, scales, tensor_scale,
                                 static_cast<WsHeader*>(workspace), dev.num_sms,
                                 static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_gemv_w4a16(const nvfp4_weight* W, const uint16_t* x, int32_t T, uint16_t* y,
                              void* workspace, size_t workspace_bytes, void* stream) {
    nvfp4_status st = check_weight(W);
    if (st != NVFP4_OK) return st;
    if (!x || !y) return NVFP4_ERR_INVALID_ARG;
    if (T < 1 || T > NVFP4_MAX_GEMV_TOKENS) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(x) || !aligned16(y) || (workspace && !aligned16(workspace))) return NVFP4_ERR_MISALIGNED;
    if (workspace && workspace_bytes < sizeof(WsHeader)) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != NVFP4_OK) return st;
    return from_cuda(launch_gemv(*W, x, T, y, static_cast<WsHeader*>(workspace), dev, g_wait_limit.load(),
                                 static_cast<cudaStream_t>(stream)));
}

nvfp4_status moe_route_topk(const float* logits, int32_t T, int32_t E, int32_t k,
                            int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                            int32_t* token_list, void* stream) {
    if (!logits || !topk_ids || !topk_w || !expert_offsets || !token_list) return NVFP4_ERR_INVALID_ARG;
    if (T < 1 || T > 65536) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (E < 1 || E > NVFP4_MAX_EXPERTS || k < 1 || k > NVFP4_MAX_TOPK || k > E)
        return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w) ||
        !aligned16(expert_offsets) || !aligned16(token_list))
        return NVFP4_ERR_MISALIGNED;
    DeviceInfo dev;
    nvfp4_status st = device_info(&dev);
    if (st != NVFP4_OK) return st;
    return from_cuda(launch_route(logits, T, E, k, topk_ids, topk_w, expert_offsets, token_list,
                                  static_cast<cudaStream_t>(stream)));
}

size_t moe_layer_workspace_size(const moe_layer_desc* d, int32_t T) {
    if (!d || T < 0 || T > NVFP4_MAX_TOKENS) return 0;
    return layer_bytes(*d, T);
}

nvfp4_status moe_layer_forward(const moe_layer_desc* d, const uint16_t* x, int32_t T, uint16_t* y,
                               int32_t* topk_ids_out, float* topk_w_out, void* workspace,
                               size_t workspace_bytes, void* stream) {
    nvfp4_status st = check_layer(d);
    if (st != NVFP4_OK) return st;
    if (T < 0 || T > NVFP4_MAX_TOKENS) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (T > 0 && (!x || !y)) return NVFP4_ERR_INVALID_ARG;
    if (!workspace) return NVFP4_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (y && !aligned16(y)) || !aligned16(workspace) ||
        (topk_ids_out && !aligned16(topk_ids_out)) || (topk_w_out && !aligned16(topk_w_out)))
        return NVFP4_ERR_MISALIGNED;
    if (workspace_bytes < layer_bytes(*d, T)) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != NVFP4_OK) return st;
    if (T == 0) return NVFP4_OK;
    return dispatch_layer(*d, x, T, y, topk_ids_out, topk_w_out, workspace, dev, static_cast<cudaStream_t>(stream),
                          nullptr);
}

size_t moe_layer_residual_workspace_size(const moe_layer_desc* d, int32_t T) {
    if (!d || T < 0 || T > NVFP4_MAX_TOKENS) return 0;
    return residual_bytes(*d, T);
}

nvfp4_status moe_layer_forward_residual(const moe_layer_desc* d, const uint16_t* norm_w, float eps,
                                        const uint16_t* h, int32_t T, uint16_t* h_out, int32_t* topk_ids_out,
                                        float* topk_w_out, void* workspace, size_t workspace_bytes,
                                        void* stream) {
    nvfp4_status st = check_layer(d);
    if (st != NVFP4_OK) return st;
    if (T < 0 || T > NVFP4_MAX_TOKENS) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!norm_w || !workspace || (T > 0 && (!h || !h_out))) return NVFP4_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !(eps < 1.0e30f)) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(norm_w) || (h && !aligned16(h)) || (h_out && !aligned16(h_out)) || !aligned16(workspace) ||
        (topk_ids_out && !aligned16(topk_ids_out)) || (topk_w_out && !aligned16(topk_w_out)))
        return NVFP4_ERR_MISALIGNED;
    if (workspace_bytes < residual_bytes(*d, T)) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    DeviceInfo dev;
    if ((st = device_info(&dev)) != NVFP4_OK) return st;
    if (T == 0) return NVFP4_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 1) {
        LayerWs ws = carve_layer_ws(workspace, *d, 1);
        if (fused_decode_supported(*d, 1, dev))
            return from_cuda(launch_moe_decode_fused(*d, h, h_out, topk_ids_out, topk_w_out, ws, dev,
                                                     g_wait_limit.load(), s, norm_w, eps, h));
    }
    // the normalised rows live after the layer's scratch
    uint16_t* xn = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + align256(layer_bytes(*d, T)));
    if (cudaError_t e = launch_rmsnorm(h, T, d->H, norm_w, eps, xn, s); e != cudaSuccess) return NVFP4_ERR_CUDA;
    return dispatch_layer(*d, xn, T, h_out, topk_ids_out, topk_w_out, workspace, dev, s, h);
}

nvfp4_status nvfp4_scale_kind_of(int32_t N, int32_t K, size_t scale_count, int32_t scale_elem_bytes,
                                 int32_t* kind_out) {
    if (!kind_out || N < 1 || K < 16 || K % 16 != 0) return NVFP4_ERR_INVALID_ARG;
    const size_t per16 = (size_t)N * (K / 16), per32 = K % 32 == 0 ? (size_t)N * (K / 32) : 0;
    int32_t kind = -1;
    if (scale_count == per16) {
        kind = scale_elem_bytes == 1 ? NVFP4_SCALE_E4M3 : scale_elem_bytes == 2 ? NVFP4_SCALE_FP16
             : scale_elem_bytes == 4 ? NVFP4_SCALE_FP32 : -1;
    } else if (per32 != 0 && scale_count == per32 && scale_elem_bytes == 1) {
        kind = NVFP4_SCALE_UE8M0;
    }
    if (kind < 0) return NVFP4_ERR_INVALID_ARG;
    *kind_out = kind;
    return NVFP4_OK;
}

nvfp4_status nvfp4_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace) return NVFP4_ERR_INVALID_ARG;
    if (workspace_bytes < sizeof(WsHeader)) return NVFP4_ERR_WORKSPACE_TOO_SMALL;
    return from_cuda(cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_get_device_status(void* workspace, int32_t clear, void* stream) {
    if (!workspace) return NVFP4_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t code = 0;
    if (cudaMemcpyAsync(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (clear) {
        if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return NVFP4_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
    }
    return static_cast<nvfp4_status>(code);
}

void nvfp4_set_single_token_form(int32_t form) { set_t1_form(form == 1 || form == 2 ? form : 0); }

int32_t nvfp4_single_token_form_used(const moe_layer_desc* d, int32_t T) {
    if (!d || check_layer(d) != NVFP4_OK) return -1;
    DeviceInfo dev;
    if (device_info(&dev) != NVFP4_OK) return -1;
    return single_token_form_of(*d, T, dev);
}

int32_t nvfp4_single_token_cluster_capacity(const moe_layer_desc* d) {
    if (!d || check_layer(d) != NVFP4_OK) return -1;
    DeviceInfo dev;
    if (device_info(&dev) != NVFP4_OK) return -1;
    return t1c_cluster_capacity(*d, dev);
}

void nvfp4_set_device_wait_limit(uint64_t limit_ns) {
    g_wait_limit.store(limit_ns == 0 ? kDefaultWaitLimit : limit_ns);
}

const char* nvfp4_status_string(nvfp4_status s) {
    switch (s) {
        case NVFP4_OK: return "ok";
        case NVFP4_ERR_INVALID_ARG: return "invalid argument";
        case NVFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case NVFP4_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case NVFP4_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case NVFP4_ERR_CUDA: return "CUDA error";
        case NVFP4_ERR_DEVICE_TIMEOUT: return "bounded device wait ran out";
        case NVFP4_ERR_NONFINITE_INPUT: return "non-finite input";
        case NVFP4_ERR_ARCH: return "device is not sm_103";
    }
    return "unknown status";
}

int32_t nvfp4_version(void) { return NVFP4MOE_VERSION; }

}  // extern "C"
