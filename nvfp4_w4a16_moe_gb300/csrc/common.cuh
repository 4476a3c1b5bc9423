// Device-side helpers shared by the sm_103a kernels of the NVFP4 W4A16 MoE
// library: number-format conversions done with the Blackwell cvt instructions,
// streaming loads, warp reductions, the workspace header and bounded waits.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/nvfp4moe.h"

namespace nvfp4 {

// ---------------------------------------------------------------- workspace
// Every workspace starts with this header. `status` holds an nvfp4_status the
// device recorded; `barrier` counts grid-barrier arrivals monotonically across
// launches (one 64-bit counter never wraps in practice); `route_tickets` count
// the router blocks of one multi-token call that are done (one counter per token
// block, then one over token blocks) and are reset to 0 by the block that
// finishes last.
constexpr int kRouteTicketBlocks = 8;
struct alignas(256) WsHeader {
    uint32_t status;
    uint32_t pad0;
    unsigned long long barrier;
    unsigned int amax_bits;      // nvfp4_pack: max |w| as fp32 bits
    unsigned int route_tickets[kRouteTicketBlocks + 1];
    unsigned int pad1[50];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Every device-side wait is bounded in time (nanoseconds of %globaltimer).
constexpr uint64_t kDefaultWaitLimit = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void record_status(WsHeader* h, uint32_t code) {
    atomicCAS(&h->status, 0u, code);
}

// ---------------------------------------------------------------- bf16 / f16
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> bf16, round to nearest even (finite inputs; NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
    float f;
    asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
    return f;
}

// Two E2M1 codes (one byte: low nibble = first element) -> two fp32 values.
// cvt.rn.f16x2.e2m1x2 is exact (every E2M1 value is an f16), and so is f16->f32.
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
    uint32_t h2;
    asm("{\n .reg .b8 b;\n cvt.u8.u32 b, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}" : "=r"(h2) : "r"(byte));
    float lo, hi;
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.f32.f16 %0, l;\n cvt.f32.f16 %1, h;\n}"
        : "=f"(lo), "=f"(hi) : "r"(h2));
    return make_float2(lo, hi);
}

// E4M3 byte -> fp32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
    uint32_t h2;
    asm("{\n .reg .b16 b;\n cvt.u16.u32 b, %1;\n cvt.rn.f16x2.e4m3x2 %0, b;\n}" : "=r"(h2) : "r"(byte & 0xFFu));
    return f16_bits_to_f32(static_cast<uint16_t>(h2 & 0xFFFFu));
}

// E8M0 byte -> 2^(b - 127) (exact; 0xFF is NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    b &= 0xFFu;
    if (b == 0xFFu) return __uint_as_float(0x7FC00000u);
    if (b == 0u) return __uint_as_float(0x00400000u);   // 2^-127, an fp32 subnormal
    return __uint_as_float(b << 23);
}

// Bytes of one row of block scales for K elements: E4M3 and FP16 one scale per 16
// elements (1 and 2 bytes), FP32 one per 16 (4 bytes), UE8M0 one per 32 (1 byte).
__host__ __device__ constexpr size_t scale_row_bytes_of(int kind, size_t K) {
    return kind == NVFP4_SCALE_E4M3 ? K / 16 : kind == NVFP4_SCALE_FP16 ? K / 8
         : kind == NVFP4_SCALE_FP32 ? K / 4 : K / 32;
}

// The two block scales of 32-element segment s of a scale row (for UE8M0 the segment is
// one block, so both are the same value).
template <int KIND>
__device__ __forceinline__ void seg_scales(const uint8_t* srow, int s, float& s0, float& s1) {
    if constexpr (KIND == NVFP4_SCALE_E4M3) {
        const uint32_t b = *reinterpret_cast<const uint16_t*>(srow + 2 * s);
        s0 = e4m3_to_f32(b & 0xFFu);
        s1 = e4m3_to_f32(b >> 8);
    } else if constexpr (KIND == NVFP4_SCALE_FP16) {
        const uint32_t h = *reinterpret_cast<const uint32_t*>(srow + 4 * s);
        s0 = f16_bits_to_f32(static_cast<uint16_t>(h & 0xFFFFu));
        s1 = f16_bits_to_f32(static_cast<uint16_t>(h >> 16));
    } else if constexpr (KIND == NVFP4_SCALE_FP32) {
        const float2 f = *reinterpret_cast<const float2*>(srow + 8 * s);
        s0 = f.x;
        s1 = f.y;
    } else {
        s0 = s1 = e8m0_to_f32(srow[s]);
    }
}

// Decoded block scale of block `i` of a scale row (16-element blocks; UE8M0: block i / 2).
template <int KIND>
__device__ __forceinline__ float scale_at(const void* row, int i) {
    if constexpr (KIND == NVFP4_SCALE_E4M3) {
        return e4m3_to_f32(static_cast<const uint8_t*>(row)[i]);
    } else if constexpr (KIND == NVFP4_SCALE_FP16) {
        return f16_bits_to_f32(static_cast<const uint16_t*>(row)[i]);
    } else if constexpr (KIND == NVFP4_SCALE_FP32) {
        return static_cast<const float*>(row)[i];
    } else {
        return e8m0_to_f32(static_cast<const uint8_t*>(row)[i >> 1]);
    }
}

// ---------------------------------------------------------------- loads
// Weights are read exactly once per call: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// Streamed weights with an L2 evict-first policy: they are read once per call,
// so they should not push the code, the routing arrays and the activations out
// of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint4 ld_stream_v4_ef(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ uint32_t ld_stream_u32_ef(const void* p, uint64_t pol) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
    return v;
}

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------- dot kernels
// Sum over 32 consecutive NVFP4 elements (16 bytes = one uint4, two scale
// blocks) against 32 fp32 activations: s0 * sum_{0..15} q x + s1 * sum_{16..31} q x.
// The per-16 partial is multiplied by its scale in fp32 (exact for E4M3 scales
// up to rounding of the partial; FP16 scales are handled the same way).
__device__ __forceinline__ float dot32(const uint4 w, const float* x, float s0, float s1) {
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    float p[2] = {0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            float2 v = e2m1x2_to_f32x2(words[q] >> (8 * b));
            p[q >> 1] = fmaf(v.x, x[8 * q + 2 * b], p[q >> 1]);
            p[q >> 1] = fmaf(v.y, x[8 * q + 2 * b + 1], p[q >> 1]);
        }
    }
    return fmaf(s0, p[0], s1 * p[1]);
}

// Dequantise 32 elements (one uint4) into fp32 q-values (scale not applied).
__device__ __forceinline__ void dequant32(const uint4 w, float* q) {
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            float2 v = e2m1x2_to_f32x2(words[i] >> (8 * b));
            q[i * 8 + 2 * b] = v.x;
            q[i * 8 + 2 * b + 1] = v.y;
        }
    }
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float silu_f32(float z) { return __fdividef(z, 1.0f + __expf(-z)); }
__device__ __forceinline__ float sigmoid_f32(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

__device__ __forceinline__ void nanosleep_ns(unsigned ns) { __nanosleep(ns); }

}  // namespace nvfp4

namespace nvfp4 {

// ---------------------------------------------------------------- TMA bulk copies + mbarriers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

// make mbarrier initialisation visible to the async (TMA) proxy
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// global -> shared bulk copy; dst, src 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// Bring the first floor16(bytes) bytes at p (16-byte aligned) into L2; a prefetch
// never touches memory past the buffer.
__device__ __forceinline__ void prefetch_l2_range(const uint8_t* p, size_t bytes) {
    const size_t n = bytes & ~size_t(15);
    for (size_t o = 0; o < n; o += (1u << 20)) {
        const uint32_t len = (uint32_t)(n - o < (1u << 20) ? n - o : (1u << 20));
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p + o), "r"(len) : "memory");
    }
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier for at most `limit_ns`; false if it ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

}  // namespace nvfp4
