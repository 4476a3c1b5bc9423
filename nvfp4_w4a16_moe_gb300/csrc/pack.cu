// NVFP4 packer: fp32 W[N,K] -> E2M1 codes, per-16 block scales, fp32 tensor scale.
//
// Format: Lynn Engine write-up, "1. native NVFP4 support" (4-bit E2M1 weights)
// and "P1 stage" (per-16 FP16 scale); lynn-engine README, P89 note (one scale
// per 16 K elements). Two launches: a max-|w| reduction over the matrix, then
// one thread per 16-element block quantising against the decoded block scale.
// All roundings use the hardware cvt instructions (round to nearest even,
// saturating), every fp32 step is one explicit IEEE op, so the bytes are
// reproducible bit for bit.
#include "common.cuh"
#include "kernels.cuh"

namespace nvfp4 {

// Both halves of the x2 conversion get the same value, so the byte order of the
// packed result does not matter.
__device__ __forceinline__ uint32_t e4m3_rne_satfinite(float v) {
    uint32_t r;
    asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %1;\n cvt.u32.u16 %0, t;\n}"
        : "=r"(r) : "f"(v));
    return r & 0xFFu;
}

__device__ __forceinline__ uint32_t f16_rne_satfinite(float v) {
    uint16_t h;
    asm("cvt.rn.satfinite.f16.f32 %0, %1;" : "=h"(h) : "f"(v));
    return h;
}

// Magnitude code (0..7) of u >= 0 on the E2M1 grid, nearest-even, saturating
// at 6 (both nibbles of the x2 conversion hold the same value).
__device__ __forceinline__ uint32_t e2m1_rne_satfinite(float u) {
    uint32_t r;
    asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %1;\n cvt.u32.u8 %0, t;\n}"
        : "=r"(r) : "f"(u));
    return r & 0x7u;
}

__global__ void pack_amax_kernel(const float4* __restrict__ w, size_t n4, WsHeader* ws) {
    float m = 0.0f;
    bool bad = false;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4;
         i += (size_t)gridDim.x * blockDim.x) {
        float4 v = __ldg(w + i);
        bad |= !isfinite(v.x) || !isfinite(v.y) || !isfinite(v.z) || !isfinite(v.w);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    // non-negative floats order like their bit patterns
    unsigned bits = __float_as_uint(m);
    bits = __reduce_max_sync(0xffffffffu, bits);
    if ((threadIdx.x & 31) == 0) atomicMax(&ws->amax_bits, bits);
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) record_status(ws, NVFP4_ERR_NONFINITE_INPUT);
}

template <int KIND>
__global__ void pack_quant_kernel(const float* __restrict__ w, size_t nblocks,
                                  uint8_t* __restrict__ packed, void* __restrict__ scales,
                                  float* __restrict__ tensor_scale, const WsHeader* ws) {
    const float amax_t = __uint_as_float(ws->amax_bits);
    float s_t = 1.0f;
    if (KIND == NVFP4_SCALE_E4M3 && amax_t > 0.0f) s_t = __fdiv_rn(amax_t, 2688.0f);
    const size_t b = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (b == 0) {
        *tensor_scale = s_t;
        __threadfence();
    }
    if (b >= nblocks) return;
    const float4* src = reinterpret_cast<const float4*>(w + b * 16);
    float v[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float4 t = __ldg(src + i);
        v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
    }
    float amax_b = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax_b = fmaxf(amax_b, fabsf(v[i]));
    const float r = __fdiv_rn(amax_b, 6.0f);
    float dec;
    if (KIND == NVFP4_SCALE_E4M3) {
        const uint32_t e = e4m3_rne_satfinite(__fdiv_rn(r, s_t));
        static_cast<uint8_t*>(scales)[b] = static_cast<uint8_t>(e);
        dec = __fmul_rn(e4m3_to_f32(e), s_t);
    } else if (KIND == NVFP4_SCALE_FP16) {
        const uint32_t e = f16_rne_satfinite(r);
        static_cast<uint16_t*>(scales)[b] = static_cast<uint16_t>(e);
        dec = __fmul_rn(f16_bits_to_f32(static_cast<uint16_t>(e)), s_t);
    } else {   // FP32: the block scale itself
        static_cast<float*>(scales)[b] = r;
        dec = r;
    }
    uint32_t out[2] = {0u, 0u};
    if (dec > 0.0f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float lo = v[2 * j], hi = v[2 * j + 1];
            uint32_t byte = e2m1_rne_satfinite(fabsf(__fdiv_rn(lo, dec))) |
                            (e2m1_rne_satfinite(fabsf(__fdiv_rn(hi, dec))) << 4);
            // the sign of w is kept even when the magnitude rounds to zero
            byte |= (__float_as_uint(lo) >> 31) << 3;
            byte |= (__float_as_uint(hi) >> 31) << 7;
            out[j >> 2] |= byte << (8 * (j & 3));
        }
    }
    *reinterpret_cast<uint2*>(packed + b * 8) = make_uint2(out[0], out[1]);
    // The layer and GEMV kernels launch with programmatic stream serialisation and
    // request their weights before griddepcontrol.wait; a packer that wrote those
    // weights right before them on the same stream has its bytes visible at GPU scope
    // before it completes.
    __threadfence();
}

// UE8M0: one thread per 32-element block; the scale is 2^(floor(log2 amax_b) - 2) (the OCP MX
// rule: E2M1's largest power of two is 2^2), clamped to E8M0's range, 2^0 for a zero block;
// the tensor scale is 1.
__global__ void pack_quant_ue8m0_kernel(const float* __restrict__ w, size_t nblocks, uint8_t* __restrict__ packed,
                                        uint8_t* __restrict__ scales, float* __restrict__ tensor_scale) {
    const size_t b = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    if (b == 0) {
        *tensor_scale = 1.0f;
        __threadfence();
    }
    if (b >= nblocks) return;
    const float4* src = reinterpret_cast<const float4*>(w + b * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 t = __ldg(src + i);
        v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
    }
    float amax_b = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax_b = fmaxf(amax_b, fabsf(v[i]));
    int ex = 0;
    if (amax_b > 0.0f) {
        const int be = (int)((__float_as_uint(amax_b) >> 23) & 0xFFu);   // 0 for subnormal amax
        ex = be == 0 ? -127 : max(-127, min(127, be - 127 - 2));
    }
    scales[b] = static_cast<uint8_t>(ex + 127);
    const float dec = ldexpf(1.0f, ex);
    uint32_t out[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float lo = v[2 * j], hi = v[2 * j + 1];
        uint32_t byte = e2m1_rne_satfinite(fabsf(__fdiv_rn(lo, dec))) |
                        (e2m1_rne_satfinite(fabsf(__fdiv_rn(hi, dec))) << 4);
        byte |= (__float_as_uint(lo) >> 31) << 3;
        byte |= (__float_as_uint(hi) >> 31) << 7;
        out[j >> 2] |= byte << (8 * (j & 3));
    }
    *reinterpret_cast<uint4*>(packed + b * 16) = make_uint4(out[0], out[1], out[2], out[3]);
    __threadfence();
}

cudaError_t launch_pack(const float* w, int N, int K, int kind, uint8_t* packed, void* scales,
                        float* tensor_scale, WsHeader* ws, int num_sms, cudaStream_t s) {
    cudaError_t err = cudaMemsetAsync(&ws->amax_bits, 0, sizeof(unsigned), s);
    if (err != cudaSuccess) return err;
    const size_t n = (size_t)N * K;
    const size_t n4 = n / 4;
    int grid = (int)((n4 + 255) / 256);
    if (grid > num_sms * 8) grid = num_sms * 8;
    if (grid < 1) grid = 1;
    pack_amax_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(w), n4, ws);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if (kind == NVFP4_SCALE_UE8M0) {
        const size_t nb = n / 32;
        pack_quant_ue8m0_kernel<<<(int)((nb + 255) / 256), 256, 0, s>>>(w, nb, packed, static_cast<uint8_t*>(scales),
                                                                         tensor_scale);
        return cudaGetLastError();
    }
    const size_t nb = n / 16;
    const int qgrid = (int)((nb + 255) / 256);
    if (kind == NVFP4_SCALE_E4M3)
        pack_quant_kernel<NVFP4_SCALE_E4M3><<<qgrid, 256, 0, s>>>(w, nb, packed, scales, tensor_scale, ws);
    else if (kind == NVFP4_SCALE_FP16)
        pack_quant_kernel<NVFP4_SCALE_FP16><<<qgrid, 256, 0, s>>>(w, nb, packed, scales, tensor_scale, ws);
    else
        pack_quant_kernel<NVFP4_SCALE_FP32><<<qgrid, 256, 0, s>>>(w, nb, packed, scales, tensor_scale, ws);
    return cudaGetLastError();
}

}  // namespace nvfp4
