// Dense NVFP4 W4A16 GEMV for 1..64 tokens: y[t,n] = sum_k W[n,k] x[t,k].
//
// Lynn Engine write-up, "P1 stage": the packed E2M1 + per-16 scale projection is
// computed straight from the packed tensor (no bf16 shadow); lynn-engine README,
// P1-A: batched M > 1 packed projections.
//
// Layout of the work: one warp owns a row at a time (rows are grid-strided over
// all warps). A row of K NVFP4 elements is K/32 segments of 16 bytes (32 codes,
// two scale blocks); lane l takes segments l, l+32, ... so a warp reads each
// row with fully coalesced 128-bit streaming loads. The partial dot products
// are reduced with warp shuffles (split-K inside the warp). Two rows are in
// flight per warp. Activations sit in shared memory as fp32 in a segment-
// interleaved layout (float4 chunk c of segment s at (c * nseg + s)), so the
// 32 lanes of a warp read 32 consecutive 16-byte chunks: no bank conflicts.
#include "common.cuh"
#include "kernels.cuh"

namespace nvfp4 {

namespace {

constexpr int kGemvThreads = 256;
constexpr int kGemvRows = 2;          // rows in flight per warp
constexpr int kGemvMaxSegPerLane = 8; // K <= 8192
constexpr int kGemvMaxTc = 8;         // tokens per pass over the weights

// x[t, :] (bf16, global) -> xs[t][c][s][4] (fp32, shared), c = 0..7, s = 0..nseg-1
__device__ void stage_x_interleaved(float* xs, const uint16_t* __restrict__ x, int t0, int tc,
                                    int K) {
    const int nseg = K >> 5;
    const int n4 = tc * (K >> 2);  // float4 chunks
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const int t = i / (K >> 2);
        const int e4 = i - t * (K >> 2);          // float4 index inside the row
        const int s = e4 >> 3, c = e4 & 7;
        const uint2 raw = *reinterpret_cast<const uint2*>(x + (size_t)(t0 + t) * K + 4 * e4);
        float4 v = make_float4(bf16lo(raw.x), bf16hi(raw.x), bf16lo(raw.y), bf16hi(raw.y));
        reinterpret_cast<float4*>(xs)[(size_t)t * (K >> 2) + c * nseg + s] = v;
    }
}

template <int KIND>
__device__ __forceinline__ void load_scales2(const void* srow, int s, float& s0, float& s1) {
    if constexpr (KIND == NVFP4_SCALE_E4M3) {
        const uint32_t b2 = *reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(srow) + 2 * s);
        s0 = e4m3_to_f32(b2 & 0xFF);
        s1 = e4m3_to_f32(b2 >> 8);
    } else {
        const uint32_t h2 = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(srow) + 2 * s);
        s0 = f16_bits_to_f32(static_cast<uint16_t>(h2 & 0xFFFF));
        s1 = f16_bits_to_f32(static_cast<uint16_t>(h2 >> 16));
    }
}

template <int KIND>
__global__ void __launch_bounds__(kGemvThreads)
gemv_kernel(const uint8_t* __restrict__ packed, const void* __restrict__ scales,
            const float* __restrict__ tscale, int N, int K, const uint16_t* __restrict__ x, int T,
            int tc_max, uint16_t* __restrict__ y) {
    extern __shared__ float4 smem_f4[];
    float* xs = reinterpret_cast<float*>(smem_f4);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nseg = K >> 5;
    const size_t row_bytes = (size_t)K >> 1;
    const size_t srow_elems = (size_t)K >> 4;
    const size_t sbytes = KIND == NVFP4_SCALE_E4M3 ? 1 : 2;
    const float ts = __ldg(tscale);
    const int warps_total = gridDim.x * (kGemvThreads / 32);
    const int gw = blockIdx.x * (kGemvThreads / 32) + warp;

    for (int t0 = 0; t0 < T; t0 += tc_max) {
        const int tc = min(tc_max, T - t0);
        __syncthreads();
        stage_x_interleaved(xs, x, t0, tc, K);
        __syncthreads();
        for (int r0 = gw * kGemvRows; r0 < N; r0 += warps_total * kGemvRows) {
            uint4 wv[kGemvRows][kGemvMaxSegPerLane];
            float sc[kGemvRows][kGemvMaxSegPerLane][2];
#pragma unroll
            for (int rr = 0; rr < kGemvRows; ++rr) {
                const int r = r0 + rr;
#pragma unroll
                for (int i = 0; i < kGemvMaxSegPerLane; ++i) {
                    const int s = lane + 32 * i;
                    if (r < N && s < nseg) {
                        wv[rr][i] = ld_stream_v4(packed + (size_t)r * row_bytes + 16 * (size_t)s);
                        load_scales2<KIND>(static_cast<const uint8_t*>(scales) + (size_t)r * srow_elems * sbytes,
                                           s, sc[rr][i][0], sc[rr][i][1]);
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < kGemvRows; ++rr) {
                const int r = r0 + rr;
                float acc[kGemvMaxTc];
#pragma unroll
                for (int t = 0; t < kGemvMaxTc; ++t) acc[t] = 0.f;
#pragma unroll
                for (int i = 0; i < kGemvMaxSegPerLane; ++i) {
                    const int s = lane + 32 * i;
                    if (r < N && s < nseg) {
                        float q[32];
                        dequant32(wv[rr][i], q);
#pragma unroll
                        for (int t = 0; t < kGemvMaxTc; ++t) {
                            if (t < tc) {
                                const float4* xt = reinterpret_cast<const float4*>(xs) + (size_t)t * (K >> 2);
                                float p0 = 0.f, p1 = 0.f;
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    const float4 a = xt[c * nseg + s];
                                    p0 = fmaf(q[4 * c], a.x, p0);
                                    p0 = fmaf(q[4 * c + 1], a.y, p0);
                                    p0 = fmaf(q[4 * c + 2], a.z, p0);
                                    p0 = fmaf(q[4 * c + 3], a.w, p0);
                                }
#pragma unroll
                                for (int c = 4; c < 8; ++c) {
                                    const float4 a = xt[c * nseg + s];
                                    p1 = fmaf(q[4 * c], a.x, p1);
                                    p1 = fmaf(q[4 * c + 1], a.y, p1);
                                    p1 = fmaf(q[4 * c + 2], a.z, p1);
                                    p1 = fmaf(q[4 * c + 3], a.w, p1);
                                }
                                acc[t] = fmaf(sc[rr][i][0], p0, fmaf(sc[rr][i][1], p1, acc[t]));
                            }
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < kGemvMaxTc; ++t) {
                    if (t < tc) {
                        const float v = warp_sum(acc[t]);
                        if (lane == 0 && r < N) y[(size_t)(t0 + t) * N + r] = f32_to_bf16(v * ts);
                    }
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_gemv(const nvfp4_weight& W, const uint16_t* x, int T, uint16_t* y,
                        const DeviceInfo& dev, cudaStream_t s) {
    const int K = W.K, N = W.N;
    // tokens per pass: as many as fit next to other blocks in shared memory
    int tc = kGemvMaxTc;
    while (tc > 1 && (size_t)tc * K * 4 > 96 * 1024) tc >>= 1;
    if (tc > T) tc = T;
    const size_t smem = (size_t)tc * K * 4;
    const int warps_needed = (N + kGemvRows - 1) / kGemvRows;
    int grid = (warps_needed + (kGemvThreads / 32) - 1) / (kGemvThreads / 32);
    const int max_grid = dev.num_sms * 4;
    if (grid > max_grid) grid = max_grid;
    if (grid < 1) grid = 1;
    cudaError_t err;
    if (W.kind == NVFP4_SCALE_E4M3) {
        err = cudaFuncSetAttribute(gemv_kernel<NVFP4_SCALE_E4M3>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        gemv_kernel<NVFP4_SCALE_E4M3><<<grid, kGemvThreads, smem, s>>>(
            W.packed, W.scales, W.tensor_scale, N, K, x, T, tc, y);
    } else {
        err = cudaFuncSetAttribute(gemv_kernel<NVFP4_SCALE_FP16>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        gemv_kernel<NVFP4_SCALE_FP16><<<grid, kGemvThreads, smem, s>>>(
            W.packed, W.scales, W.tensor_scale, N, K, x, T, tc, y);
    }
    return cudaGetLastError();
}

}  // namespace nvfp4
