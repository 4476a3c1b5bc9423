// Pre-MoE RMSNorm in the (1 + weight) form, for the multi-token and prefill paths of
// moe_layer_forward_residual (the single-token kernel does the same inside its x staging).
//
// lynn-engine tutorials index, row 01 and the Qwen 3.6 config block: RMSNorm =
// (1.0 + weight) x x_norm with x_norm = h / sqrt(mean(h^2) + eps); Lynn Engine write-up,
// "Fused Kernels": the norm is fused with the layer's launches. One CTA per token: the
// squares are summed per thread in a fixed order, per warp by shuffles and over the warps
// in a fixed order (deterministic), r = 1 / sqrt(mean + eps) with IEEE square root and
// division, and each element is rounded once to bf16.
#include "common.cuh"
#include "kernels.cuh"

namespace nvfp4 {

namespace {

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
rmsnorm_kernel(const uint16_t* __restrict__ h, int H, const uint16_t* __restrict__ w, float eps,
               uint16_t* __restrict__ out) {
    __shared__ float s_ss[kNormThreads / 32];
    const int t = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint4* row = reinterpret_cast<const uint4*>(h + (size_t)t * H);
    const int nu = H >> 3;
    float ss = 0.f;
    for (int i = threadIdx.x; i < nu; i += kNormThreads) {
        const uint4 v = row[i];
        const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            ss = fmaf(bf16lo(ww[q]), bf16lo(ww[q]), ss);
            ss = fmaf(bf16hi(ww[q]), bf16hi(ww[q]), ss);
        }
    }
    ss = warp_sum(ss);
    if (lane == 0) s_ss[warp] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int i = 0; i < kNormThreads / 32; ++i) tot += s_ss[i];
    const float r = 1.0f / sqrtf(tot / (float)H + eps);
    uint4* o = reinterpret_cast<uint4*>(out + (size_t)t * H);
    for (int i = threadIdx.x; i < nu; i += kNormThreads) {
        const uint4 v = row[i], wv = reinterpret_cast<const uint4*>(w)[i];
        const uint32_t xx[4] = {v.x, v.y, v.z, v.w}, nw[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t res[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float lo = bf16lo(xx[q]) * r * (1.0f + bf16lo(nw[q]));
            const float hi = bf16hi(xx[q]) * r * (1.0f + bf16hi(nw[q]));
            res[q] = (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
        }
        o[i] = make_uint4(res[0], res[1], res[2], res[3]);
    }
}

}  // namespace

cudaError_t launch_rmsnorm(const uint16_t* h, int T, int H, const uint16_t* w, float eps, uint16_t* out,
                           cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    rmsnorm_kernel<<<T, kNormThreads, 0, s>>>(h, H, w, eps, out);
    return cudaGetLastError();
}

}  // namespace nvfp4
