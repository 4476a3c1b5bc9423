// Device helpers of the single-token layer kernels (the grid form and the cluster form):
// tagged exchange words, FP4 segment dot products on f16 activations, warp reductions and
// the order key of the top-k.
#pragma once

#include "common.cuh"

namespace nvfp4 {
namespace {

__device__ __forceinline__ void st_word(unsigned long long* p, uint32_t tag, float v) {
    const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ unsigned long long ld_word(const unsigned long long* p) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

// Read a word until it carries `tag` (bounded); false on timeout.
__device__ __forceinline__ bool poll_word(const unsigned long long* p, uint32_t tag, unsigned long long limit,
                                          float* out) {
    unsigned long long w = ld_word(p);
    if ((uint32_t)(w >> 32) != tag) {
        const unsigned long long t0 = global_timer_ns();
        do {
            if (global_timer_ns() - t0 > limit) return false;
            w = ld_word(p);
        } while ((uint32_t)(w >> 32) != tag);
    }
    *out = __uint_as_float((uint32_t)w);
    return true;
}

// h words: the low 16 bits of the launch tag (never 0) over the bf16 value, single-copy
// atomic as one 32-bit store; readers load four at a time.
__device__ __forceinline__ uint32_t tag16_of(uint32_t tag) { return tag % 65535u + 1u; }
__device__ __forceinline__ void st_hword(uint32_t* p, uint32_t tag16, float v) {
    const uint32_t w = (tag16 << 16) | (uint32_t)f32_to_bf16(v);
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(w) : "memory");
}
// eight words (32 bytes, 32-byte aligned) in one load
__device__ __forceinline__ void ld_hwords8(const uint32_t* p, uint4& a, uint4& b) {
    asm volatile("ld.relaxed.gpu.global.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p) : "memory");
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_addr(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void expand4(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

__device__ __forceinline__ float fma2h(uint32_t q2, uint32_t x2, float acc) {
    asm("{\n .reg .f16 ql, qh, xl, xh;\n mov.b32 {ql, qh}, %1;\n mov.b32 {xl, xh}, %2;\n"
        " fma.rn.f32.f16 %0, ql, xl, %0;\n fma.rn.f32.f16 %0, qh, xh, %0;\n}"
        : "+f"(acc) : "r"(q2), "r"(x2));
    return acc;
}

__device__ __forceinline__ uint32_t to_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// k with m * 2^k in [2^14, 2^15) from the fp32 bits of m >= 0 (0 for m = 0), clamped so
// that 2^k and 2^-k are normal.
__device__ __forceinline__ int pow2_shift(uint32_t fbits) {
    if (fbits == 0u) return 0;
    const int e = (int)(fbits >> 23) - 127;
    return min(126, max(-126, 14 - e));
}
__device__ __forceinline__ float exp2_int(int k) { return __int_as_float((k + 127) << 23); }

template <int KIND>
__device__ __forceinline__ void scales2(const uint8_t* srow, int s, float& s0, float& s1) {
    if constexpr (KIND == NVFP4_SCALE_E4M3) {
        const uint32_t b = *reinterpret_cast<const uint16_t*>(srow + 2 * s);
        s0 = e4m3_to_f32(b & 0xFFu);
        s1 = e4m3_to_f32(b >> 8);
    } else {
        const uint32_t h = *reinterpret_cast<const uint32_t*>(srow + 4 * s);
        s0 = f16_bits_to_f32(static_cast<uint16_t>(h & 0xFFFFu));
        s1 = f16_bits_to_f32(static_cast<uint16_t>(h >> 16));
    }
}

// One 16-byte segment (32 codes, two scale blocks) against its 32 f16 activations (four
// units of eight).
__device__ __forceinline__ float seg_dot_r(const uint4 w, float s0, float s1, const uint4 u0, const uint4 u1,
                                           const uint4 u2, const uint4 u3) {
    uint32_t a[4], b[4], c[4], d[4];
    expand4(w.x, a);
    expand4(w.y, b);
    expand4(w.z, c);
    expand4(w.w, d);
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
    p0 = fma2h(a[0], u0.x, p0); p1 = fma2h(a[1], u0.y, p1); p0 = fma2h(a[2], u0.z, p0); p1 = fma2h(a[3], u0.w, p1);
    p0 = fma2h(b[0], u1.x, p0); p1 = fma2h(b[1], u1.y, p1); p0 = fma2h(b[2], u1.z, p0); p1 = fma2h(b[3], u1.w, p1);
    p2 = fma2h(c[0], u2.x, p2); p3 = fma2h(c[1], u2.y, p3); p2 = fma2h(c[2], u2.z, p2); p3 = fma2h(c[3], u2.w, p3);
    p2 = fma2h(d[0], u3.x, p2); p3 = fma2h(d[1], u3.y, p3); p2 = fma2h(d[2], u3.z, p2); p3 = fma2h(d[3], u3.w, p3);
    return fmaf(s0, p0 + p1, s1 * (p2 + p3));
}

// The same with the activations stored segment-interleaved (unit c of segment s at c * nseg + s).
template <int KIND>
__device__ __forceinline__ float seg_dot(const uint4 w, float s0, float s1, const uint4* xv, int nseg, int s) {
    return seg_dot_r(w, s0, s1, xv[s], xv[nseg + s], xv[2 * nseg + s], xv[3 * nseg + s]);
}

// Sum of each of v[0..7] over the warp, spread over the lanes: lane l ends with the sum of
// v[(l >> 2) & 7] (halving exchanges at distances 16, 8, 4, then the quad; 9 shuffles, a
// fixed order).
__device__ __forceinline__ float warp_sum8(const float (&v)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float w4[4], w2[2];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        w4[j] = (b4 ? v[j + 4] : v[j]) + __shfl_xor_sync(0xffffffffu, b4 ? v[j] : v[j + 4], 16);
#pragma unroll
    for (int j = 0; j < 2; ++j)
        w2[j] = (b3 ? w4[j + 2] : w4[j]) + __shfl_xor_sync(0xffffffffu, b3 ? w4[j] : w4[j + 2], 8);
    float z = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
    z += __shfl_xor_sync(0xffffffffu, z, 2);
    z += __shfl_xor_sync(0xffffffffu, z, 1);
    return z;
}

// (gate . x, up . x) of one pair whose rows sit in shared memory; lanes over segments.
// Lane 0 ends with the gate sum, lane 16 with the up sum.
template <int KIND>
__device__ __noinline__ float pair_dot(const uint8_t* g, const uint8_t* u, const uint8_t* gs, const uint8_t* us,
                                       const uint4* x16, int nseg, int lane) {
    float ga = 0.f, ua = 0.f;
#pragma unroll 2
    for (int s = lane; s < nseg; s += 32) {
        float g0, g1, u0, u1;
        scales2<KIND>(gs, s, g0, g1);
        scales2<KIND>(us, s, u0, u1);
        ga += seg_dot<KIND>(reinterpret_cast<const uint4*>(g)[s], g0, g1, x16, nseg, s);
        ua += seg_dot<KIND>(reinterpret_cast<const uint4*>(u)[s], u0, u1, x16, nseg, s);
    }
    const bool lo = lane < 16;
    float m = lo ? ga : ua;
    m += __shfl_xor_sync(0xffffffffu, lo ? ua : ga, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m += __shfl_xor_sync(0xffffffffu, m, o);
    return m;
}

__device__ __forceinline__ float bf16_dot8(const uint4 w, const uint4 v, float acc) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    const uint32_t xx[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc = fmaf(bf16lo(ww[q]), bf16lo(xx[q]), acc);
        acc = fmaf(bf16hi(ww[q]), bf16hi(xx[q]), acc);
    }
    return acc;
}

// float -> unsigned key with the same order
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint32_t copy_range(uint8_t* dst, const uint8_t* src, uint32_t bytes, uint64_t* bar) {
    if (bytes) bulk_g2s(dst, src, bytes, bar);
    return bytes;
}

}  // namespace
}  // namespace nvfp4
