// Launchers of the sm_103a kernels (internal; the C ABI in api.cu validates
// arguments and calls these).
#pragma once

#include "common.cuh"

namespace nvfp4 {

struct DeviceInfo {
    int device;
    int num_sms;
    int cc_major, cc_minor;
    size_t smem_optin;
};

cudaError_t launch_pack(const float* w, int N, int K, int kind, uint8_t* packed, void* scales,
                        float* tensor_scale, WsHeader* ws, int num_sms, cudaStream_t s);

// hdr (nullable): where a bounded wait that ran out is recorded
cudaError_t launch_gemv(const nvfp4_weight& W, const uint16_t* x, int T, uint16_t* y, WsHeader* hdr,
                        const DeviceInfo& dev, uint64_t wait_limit, cudaStream_t s);

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                              cudaStream_t s);
cudaError_t launch_route_lists(const int32_t* ids, int total, int E, int32_t* offsets,
                               int32_t* token_list, int32_t* active, cudaStream_t s);
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         int32_t* offsets, int32_t* token_list, cudaStream_t s);

// Exchange words of the one-launch single-token kernel: kWordReplicas copies of the E + 1
// logits (8-byte words, each copy padded to 16 words) and of the k*I + Is SwiGLU values
// (4-byte words, each copy padded to 32 words); in 8-byte units.
constexpr int kWordReplicas = 8;
__host__ __device__ inline size_t t1_logit_stride(const moe_layer_desc& d) { return ((size_t)d.E + 1 + 15) & ~size_t(15); }
__host__ __device__ inline size_t t1_h_stride(const moe_layer_desc& d) { return ((size_t)d.k * d.I + d.Is + 31) & ~size_t(31); }
// Exchange area of the cluster form, in 8-byte units: kWordReplicas copies of the Is shared
// values (4-byte tagged words, each copy padded to 32 words), then k * H tagged partial
// outputs (8-byte words).
__host__ __device__ inline size_t t1c_words(const moe_layer_desc& d) {
    return (size_t)kWordReplicas * ((((size_t)d.Is + 31) & ~size_t(31)) / 2) + (size_t)d.k * d.H;
}
__host__ __device__ inline size_t t1_words(const moe_layer_desc& d) {
    const size_t grid = (size_t)kWordReplicas * (t1_logit_stride(d) + t1_h_stride(d) / 2);
    const size_t cl = t1c_words(d);
    return grid > cl ? grid : cl;
}

// Workspace of one layer call (device scratch carved from the caller's buffer).
struct LayerWs {
    WsHeader* hdr;
    float* logits;        // [T, E]
    float* gate_logit;    // [T]        shared-expert sigmoid gate pre-activation
    int32_t* ids;         // [T, k]
    float* w;             // [T, k]
    int32_t* offsets;     // [E + 1]
    int32_t* token_list;  // [T * k]
    int32_t* active;      // [E + 1]    active[0] = A, active[1..A] = expert ids ascending
    float* h;             // [T * k, I] routed SwiGLU intermediates (entry-major)
    float* hs;            // [T, Is]    shared intermediates
    unsigned long long* words;  // [t1_words(d)] (launch tag, value) words of the one-launch kernel
    int32_t* pass_map;    // [E + T*k + 2]  pass_map[0] = P, then (active slot << 8) | pass
    float* part;          // [T*k + T, H]  weighted routed rows, then the shared rows
    uint32_t* amax;       // [T + T*k + T] max |x| of each token, then max |h| of each h row (fp32 bits)
    size_t bytes;
};

LayerWs carve_layer_ws(void* base, const moe_layer_desc& d, int T);
size_t layer_ws_bytes(const moe_layer_desc& d, int T);

// resid (nullable, bf16 [T, H]): added to every output element before its one rounding
cudaError_t launch_moe_decode(const moe_layer_desc& d, const uint16_t* x, int T, uint16_t* y,
                              int32_t* ids_out, float* w_out, const LayerWs& ws,
                              const DeviceInfo& dev, uint64_t wait_limit, cudaStream_t s,
                              const uint16_t* resid = nullptr);

// Multi-token decode on mma.sync (E4M3 scales, H, I, Is multiples of 256, <= 4096).
bool decode_mma_supported(const moe_layer_desc& d, int T);
cudaError_t launch_moe_decode_mma(const moe_layer_desc& d, const uint16_t* x, int T, uint16_t* y,
                                  int32_t* ids_out, float* w_out, const LayerWs& ws, const DeviceInfo& dev,
                                  cudaStream_t s, const uint16_t* resid = nullptr);

// Launch tags of the single-token kernels: every launch adds tag_period(dev) to the
// workspace counter (each of its CTAs adds tag_period / grid size), so the counter is a
// multiple of the period between launches of either form, and a launch's tag is
// counter / period + 1 at any of its CTAs.
unsigned long long t1_tag_period(const DeviceInfo& dev);

// Single-token decode in one launch: the persistent-grid form, or on request the cluster
// form (k clusters of 8 to 16 CTAs) where the shape and the device allow it. form: 0 =
// automatic (the grid form), 1 = grid form, 2 = cluster form (unsupported -> grid form).
void set_t1_form(int form);
bool t1c_supported(const moe_layer_desc& d, int T, const DeviceInfo& dev);
cudaError_t launch_moe_decode_t1c(const moe_layer_desc& d, const uint16_t* x, uint16_t* y, int32_t* ids_out,
                                  float* w_out, const LayerWs& ws, const DeviceInfo& dev, uint64_t wait_limit,
                                  cudaStream_t s, const uint16_t* norm_w, float eps, const uint16_t* resid);
bool fused_decode_supported(const moe_layer_desc& d, int T, const DeviceInfo& dev);
// 2: the cluster form runs this call, 1: the grid form, 0: neither (T != 1 or the shape)
int single_token_form_of(const moe_layer_desc& d, int T, const DeviceInfo& dev);
// resident 16-CTA clusters of the cluster form for this layer (0 when the shape has none)
int t1c_cluster_capacity(const moe_layer_desc& d, const DeviceInfo& dev);
cudaError_t launch_moe_decode_fused(const moe_layer_desc& d, const uint16_t* x, uint16_t* y,
                                    int32_t* ids_out, float* w_out, const LayerWs& ws,
                                    const DeviceInfo& dev, uint64_t wait_limit, cudaStream_t s,
                                    const uint16_t* norm_w = nullptr, float eps = 0.f,
                                    const uint16_t* resid = nullptr);

// Pre-MoE RMSNorm, (1 + w) form: out[t] = bf16(h[t] / sqrt(mean(h[t]^2) + eps) * (1 + w)).
cudaError_t launch_rmsnorm(const uint16_t* h, int T, int H, const uint16_t* w, float eps, uint16_t* out,
                           cudaStream_t s);

// Prefill path (T > 64 tokens, E4M3 scales): grouped tensor-core GEMMs.
constexpr int kTokTile = 256;   // token rows per grouped-GEMM tile

// Everything the two grouped GEMMs read. Slots 0..E-1 are the routed experts
// (rows = their entries in token_list order), slot E the shared expert (rows =
// tokens 0..T-1). tile_prefix[s] is the first kTokTile-row tile of slot s.
struct GroupedParams {
    const uint16_t* x;
    int T, H, E, k, I, Is;
    const uint8_t* gu_packed; const uint8_t* gu_scales; const float* gu_tscale;
    const uint8_t* dn_packed; const uint8_t* dn_scales; const float* dn_tscale;
    const uint8_t* sh_gu_packed; const uint8_t* sh_gu_scales; const float* sh_gu_tscale;
    const uint8_t* sh_dn_packed; const uint8_t* sh_dn_scales; const float* sh_dn_tscale;
    const int32_t* offsets;     // [E + 1]
    const int32_t* token_list;  // [T * k] entries t*k + j grouped by expert
    const int32_t* tile_prefix; // [E + 2]
    const float* w;             // [T, k] routing weights
    const float* gate;          // [T] shared gate pre-activation
    uint16_t* h;                // [T * k, I] bf16, rows in token_list order
    uint16_t* hs;               // [T, Is] bf16
    float* Y;                   // [T, k + 1, H] fp32 scaled expert outputs
};


struct PrefillWs {
    WsHeader* hdr;
    float* logits;        // [T, E]
    float* gate;          // [T]
    int32_t* ids;         // [T, k]
    float* w;             // [T, k]
    int32_t* bcount;      // [ceil(T*k / 1024), E]  per-block counts, then bases
    int32_t* offsets;     // [E + 1]
    int32_t* tile_prefix; // [E + 2]  first kTokTile-row tile of each slot (E = shared)
    int32_t* token_list;  // [T * k]
    uint16_t* h;          // [T * k, I]  bf16 SwiGLU intermediates, token_list order
    uint16_t* hs;         // [T, Is]     bf16 shared intermediates
    float* Y;             // [T, k + 1, H] weighted expert outputs
    size_t bytes;
};

bool prefill_supported(const moe_layer_desc& d, int T);
size_t prefill_ws_bytes(const moe_layer_desc& d, int T);
PrefillWs carve_prefill_ws(void* base, const moe_layer_desc& d, int T);
int prefill_launch_count(const moe_layer_desc& d, int T);
cudaError_t launch_moe_prefill(const moe_layer_desc& d, const uint16_t* x, int T, uint16_t* y,
                               int32_t* ids_out, float* w_out, const PrefillWs& ws, uint64_t wait_limit,
                               cudaStream_t s,
                               const uint16_t* resid = nullptr);
// Grouped tcgen05 GEMM over the token tiles of every slot: mode 0 = gate/up with the
// SwiGLU epilogue (x -> h, hs), mode 1 = down with the weighted epilogue (h, hs -> Y).
cudaError_t launch_grouped_tc(const GroupedParams& P, int mode, int tiles_max, WsHeader* hdr,
                              uint64_t wait_limit, cudaStream_t s);

}  // namespace nvfp4
