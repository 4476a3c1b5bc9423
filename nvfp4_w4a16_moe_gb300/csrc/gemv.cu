// Dense NVFP4 W4A16 GEMV for 1..64 tokens: y[t,n] = sum_k W[n,k] x[t,k].
//
// Lynn Engine write-up, "P1 stage": the packed E2M1 + per-16 scale projection is
// computed straight from the packed tensor (no bf16 shadow); lynn-engine README,
// P1-A: batched M > 1 packed projections.
//
// The weight stream is what bounds this call (4.5 bits per weight against 16 bits
// of activation per token), so the kernel is built around keeping HBM busy:
//
//  - A persistent grid of one CTA per SM. The rows are cut into chunks (8 or 32 rows)
//    and CTA c owns the contiguous chunks [ng*c/G, ng*(c+1)/G): every CTA streams one
//    contiguous byte range of the packed codes and one of the block scales.
//  - One producer warp moves each 8-row chunk HBM -> shared memory with two TMA
//    bulk copies (codes, scales) into a ring of slots, each with a "full" mbarrier
//    (transaction bytes) and an "empty" mbarrier (one arrival per row). All slots
//    are requested at once, so a CTA has its whole share (or the ring's worth) of
//    bytes in flight from the first cycle; the copies need nothing the previous
//    kernel on the stream writes, so they are issued before griddepcontrol.wait.
//  - One token and a long row range per CTA (the lm_head): chunks of 32 rows (each SM
//    keeps only a few bulk copies in flight, so the copies are made large: 32 rows cut
//    the lm_head from 97.5 to 75.2 us against 8-row chunks), 4 warps per chunk with 8 rows
//    each; lane l holds the activation units of segments l, l+32, ... in registers and
//    runs them against its warp's 8 rows, so one wait, one activation load and one
//    9-shuffle reduction serve 8 rows. Otherwise chunks of 8 rows: one token with few
//    chunks per CTA, 16 consumer warps, warps 4r .. 4r+3 take row pairs 0-1, 2-3, 4-5,
//    6-7 of the chunks of group r; several tokens, 8 consumer warps and 2 groups; each
//    activation load feeds both rows. Lane l takes the 16-byte segments l, l+32, ... of the rows (32
//    codes, two scale blocks each): cvt.rn.f16x2.e2m1x2 expands two codes
//    into an exact f16 pair, and fma.rn.f32.f16 multiplies each code with its
//    activation (f16) and accumulates in fp32; each 16-element partial is then
//    multiplied by its block scale (E4M3 or FP16, decoded exactly) in fp32. The
//    row's partials are reduced with warp shuffles.
//  - Two CTAs fit on an SM (at most ~100 KB of shared memory each), so under
//    programmatic dependent launch the next call's weight copies overlap this
//    call's arithmetic.
//  - Activations are read once (kept in registers while the row maxima are
//    reduced) and staged in shared memory as f16, token row t multiplied by the
//    power of two 2^k_t that puts max|x_t| in [2^14, 2^15) (exact; no f16
//    overflow, elements down to 2^-31 of the row maximum convert exactly); the
//    output multiplies by ts * 2^-k_t. The layout is segment-interleaved (16-byte
//    unit c of segment s at unit c*nseg + s), so a warp's 32 lanes read 32
//    consecutive 16-byte units.
//  - Up to 8 tokens share one pass over the weights; larger T takes several passes
//    (the producer runs ahead across passes).
//
// Every wait is bounded (%globaltimer). A wait that runs out writes quiet-NaN rows
// and, when the caller passed a workspace, NVFP4_ERR_DEVICE_TIMEOUT to its status
// word; the CTA drains its copies in flight before it returns.
#include <atomic>

#include "common.cuh"
#include "kernels.cuh"

namespace nvfp4 {

namespace {

constexpr int kCRows = 8;                              // rows per chunk (one ring slot)
constexpr int kCRows1 = 8;                             // ... in the one-warp-per-chunk mode
constexpr int kWarpsPerChunk = kCRows / 2;             // two rows per warp (several tokens)
// consumer warps that take one chunk (GemvParams::wpc): 1 for one token when a CTA has at
// least two chunks per consumer warp (that warp does all 8 rows, its activation segment in
// registers across them), else 4 warps of two rows
// consumer warps: 16 at one token (two CTAs of 17 warps fit on an SM at <= 60 registers),
// 8 when several tokens share a pass (more accumulators per thread)
constexpr int consumer_warps(int tc) { return tc == 1 ? 16 : 8; }
constexpr int gemv_threads(int tc) { return (consumer_warps(tc) + 1) * 32; }   // + the producer warp
constexpr int kMaxSlots = 32;
constexpr int kMaxTc = 8;                              // tokens per pass over the weights
constexpr int kKeep = 4;                               // activation units a thread keeps in registers

struct GemvParams {
    const uint8_t* packed;
    const uint8_t* scales;
    const float* tscale;
    const uint16_t* x;
    uint16_t* y;
    WsHeader* hdr;            // nullable: where a timeout is recorded
    unsigned long long wait_limit;
    int N, K, T;
    int ngroups;              // ceil(N / crows)
    int wpc;                  // consumer warps per chunk
    int wide;                 // 1: one token, each warp takes 8 rows of a chunk of 8 * wpc rows
                              // (big copies); 0: chunks of 8 rows, two rows per warp
    int slots;                // ring depth
    uint32_t slot_bytes;      // crows * (K/2 + scale row bytes)
    int crows;                // rows per chunk: kCRows, or kCRows1 with one warp per chunk
    uint32_t off_ring;        // shared-memory offset of the ring (after the x stage)
};

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

// Two codes (one byte; low nibble first) -> f16x2, exact.
__device__ __forceinline__ void expand_word4(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

// acc += q.lo * x.lo + q.hi * x.hi (f16 operands, fp32 accumulation; the products are exact)
__device__ __forceinline__ float fma2_f16(uint32_t q2, uint32_t x2, float acc) {
    asm("{\n .reg .f16 ql, qh, xl, xh;\n mov.b32 {ql, qh}, %1;\n mov.b32 {xl, xh}, %2;\n"
        " fma.rn.f32.f16 %0, ql, xl, %0;\n fma.rn.f32.f16 %0, qh, xh, %0;\n}"
        : "+f"(acc) : "r"(q2), "r"(x2));
    return acc;
}

__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// k with max * 2^k in [2^14, 2^15) from the bf16 bits of max|row| (0 for a zero row),
// clamped so that 2^k and 2^-k are normal fp32 values.
__device__ __forceinline__ int gemv_row_shift(uint32_t bf16_amax) {
    if (bf16_amax == 0u) return 0;
    const int e = (int)(bf16_amax >> 7) - 127;
    return min(126, max(-126, 14 - e));
}
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

// One 16-byte segment (32 codes) of two rows against one token's activations: the
// activation units are loaded once for both rows; eight independent accumulators.
template <int KIND>
__device__ __forceinline__ void seg2(const uint32_t (&qa)[16], const uint32_t (&qb)[16], const uint4* xt,
                                     int nseg, int s, float a0, float a1, float b0, float b1, float& ya,
                                     float& yb) {
    const uint4 u0 = xt[s], u1 = xt[nseg + s], u2 = xt[2 * nseg + s], u3 = xt[3 * nseg + s];
    float pa0 = 0.f, pa1 = 0.f, pa2 = 0.f, pa3 = 0.f, pb0 = 0.f, pb1 = 0.f, pb2 = 0.f, pb3 = 0.f;
    pa0 = fma2_f16(qa[0], u0.x, pa0);   pb0 = fma2_f16(qb[0], u0.x, pb0);
    pa1 = fma2_f16(qa[1], u0.y, pa1);   pb1 = fma2_f16(qb[1], u0.y, pb1);
    pa0 = fma2_f16(qa[2], u0.z, pa0);   pb0 = fma2_f16(qb[2], u0.z, pb0);
    pa1 = fma2_f16(qa[3], u0.w, pa1);   pb1 = fma2_f16(qb[3], u0.w, pb1);
    pa0 = fma2_f16(qa[4], u1.x, pa0);   pb0 = fma2_f16(qb[4], u1.x, pb0);
    pa1 = fma2_f16(qa[5], u1.y, pa1);   pb1 = fma2_f16(qb[5], u1.y, pb1);
    pa0 = fma2_f16(qa[6], u1.z, pa0);   pb0 = fma2_f16(qb[6], u1.z, pb0);
    pa1 = fma2_f16(qa[7], u1.w, pa1);   pb1 = fma2_f16(qb[7], u1.w, pb1);
    pa2 = fma2_f16(qa[8], u2.x, pa2);   pb2 = fma2_f16(qb[8], u2.x, pb2);
    pa3 = fma2_f16(qa[9], u2.y, pa3);   pb3 = fma2_f16(qb[9], u2.y, pb3);
    pa2 = fma2_f16(qa[10], u2.z, pa2);  pb2 = fma2_f16(qb[10], u2.z, pb2);
    pa3 = fma2_f16(qa[11], u2.w, pa3);  pb3 = fma2_f16(qb[11], u2.w, pb3);
    pa2 = fma2_f16(qa[12], u3.x, pa2);  pb2 = fma2_f16(qb[12], u3.x, pb2);
    pa3 = fma2_f16(qa[13], u3.y, pa3);  pb3 = fma2_f16(qb[13], u3.y, pb3);
    pa2 = fma2_f16(qa[14], u3.z, pa2);  pb2 = fma2_f16(qb[14], u3.z, pb2);
    pa3 = fma2_f16(qa[15], u3.w, pa3);  pb3 = fma2_f16(qb[15], u3.w, pb3);
    ya = fmaf(a0, pa0 + pa1, fmaf(a1, pa2 + pa3, ya));
    yb = fmaf(b0, pb0 + pb1, fmaf(b1, pb2 + pb3, yb));
}

// The two block scales of segment s of a scale row in shared memory (ld.shared: a select
// between a shared and a global row would make every read a generic load).
template <int KIND>
__device__ __forceinline__ void seg_scales_sh(uint32_t row, int s, float& s0, float& s1) {
    if constexpr (KIND == NVFP4_SCALE_E4M3) {
        uint16_t b;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(b) : "r"(row + 2u * s));
        s0 = e4m3_to_f32(b & 0xFFu);
        s1 = e4m3_to_f32((uint32_t)b >> 8);
    } else if constexpr (KIND == NVFP4_SCALE_FP16) {
        uint32_t h;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(h) : "r"(row + 4u * s));
        s0 = f16_bits_to_f32(static_cast<uint16_t>(h & 0xFFFFu));
        s1 = f16_bits_to_f32(static_cast<uint16_t>(h >> 16));
    } else if constexpr (KIND == NVFP4_SCALE_FP32) {
        float2 f;
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(f.x), "=f"(f.y) : "r"(row + 8u * s));
        s0 = f.x;
        s1 = f.y;
    } else {
        uint16_t b;
        asm volatile("ld.shared.u8 %0, [%1];" : "=h"(b) : "r"(row + (uint32_t)s));
        s0 = s1 = e8m0_to_f32((uint32_t)b & 0xFFu);
    }
}

// One 16-byte segment (32 codes, two scale blocks) of one row against one token's
// activation units (already in registers); four independent accumulators.
__device__ __forceinline__ float seg1(const uint32_t (&q)[16], const uint4 u0, const uint4 u1, const uint4 u2,
                                      const uint4 u3, float a0, float a1) {
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
    p0 = fma2_f16(q[0], u0.x, p0);   p1 = fma2_f16(q[1], u0.y, p1);
    p0 = fma2_f16(q[2], u0.z, p0);   p1 = fma2_f16(q[3], u0.w, p1);
    p0 = fma2_f16(q[4], u1.x, p0);   p1 = fma2_f16(q[5], u1.y, p1);
    p0 = fma2_f16(q[6], u1.z, p0);   p1 = fma2_f16(q[7], u1.w, p1);
    p2 = fma2_f16(q[8], u2.x, p2);   p3 = fma2_f16(q[9], u2.y, p3);
    p2 = fma2_f16(q[10], u2.z, p2);  p3 = fma2_f16(q[11], u2.w, p3);
    p2 = fma2_f16(q[12], u3.x, p2);  p3 = fma2_f16(q[13], u3.y, p3);
    p2 = fma2_f16(q[14], u3.z, p2);  p3 = fma2_f16(q[15], u3.w, p3);
    return fmaf(a0, p0 + p1, a1 * (p2 + p3));
}

// Warp sums of v[0..7] spread over the lanes: lane l ends with the sum of v[(l >> 2) & 7]
// (halving exchanges at distances 16, 8, 4, then the quad: 9 shuffles, a fixed order).
__device__ __forceinline__ float warp_sum8_lanes(const float (&v)[8], int lane) {
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

__device__ __forceinline__ void expand_seg(const uint4 w, uint32_t (&q)[16]) {
    expand_word4(w.x, *reinterpret_cast<uint32_t(*)[4]>(&q[0]));
    expand_word4(w.y, *reinterpret_cast<uint32_t(*)[4]>(&q[4]));
    expand_word4(w.z, *reinterpret_cast<uint32_t(*)[4]>(&q[8]));
    expand_word4(w.w, *reinterpret_cast<uint32_t(*)[4]>(&q[12]));
}

// Warp sums of two values in five shuffles: lanes 0-15 end with sum(a), 16-31 with sum(b).
__device__ __forceinline__ float warp_sum_pair(float a, float b, int lane) {
    const bool lo = lane < 16;
    float m = lo ? a : b;
    m += __shfl_xor_sync(0xffffffffu, lo ? b : a, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m += __shfl_xor_sync(0xffffffffu, m, o);
    return m;
}

template <int KIND, int TC>
__global__ void __launch_bounds__(gemv_threads(TC), TC <= 2 ? 2 : 1) gemv_kernel(GemvParams p) {
    constexpr int kConsumerWarps = consumer_warps(TC);
    const int wpc = TC == 1 ? p.wpc : kWarpsPerChunk;   // a constant for several tokens
    const bool wide = TC == 1 && p.wide;
    const int kChunkResidues = kConsumerWarps / wpc;
    extern __shared__ __align__(128) uint8_t gsm[];
    __shared__ uint64_t full[kMaxSlots], empty[kMaxSlots];
    __shared__ uint32_t s_amax[kMaxTc];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.N, K = p.K, T = p.T;
    const int G = gridDim.x, c = blockIdx.x;
    const int g0 = (int)((long long)p.ngroups * c / G);
    const int g1 = (int)((long long)p.ngroups * (c + 1) / G);
    const int nc = g1 - g0;                        // chunks per pass
    const int passes = (T + TC - 1) / TC;
    const int nv = nc * passes;                    // chunks streamed by this CTA
    const uint32_t rowB = (uint32_t)K >> 1, srowB = (uint32_t)scale_row_bytes_of(KIND, K);
    const int crows = TC == 1 ? p.crows : kCRows;  // a constant for several tokens
    const uint32_t off_sc = (uint32_t)crows * rowB;   // scale bytes inside a slot
    const int nseg = K >> 5, nunit = K >> 3;
    uint8_t* ring = gsm + p.off_ring;
    uint4* xs = reinterpret_cast<uint4*>(gsm);     // [TC][K/8] f16x8 units, interleaved

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.slots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], TC == 1 ? p.wpc : kWarpsPerChunk);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int v = 0; v < nv; ++v) {
                const int slot = v % p.slots;
                if (v >= p.slots) {
                    if (!mbar_wait_bounded(&empty[slot], (uint32_t)((v / p.slots) - 1) & 1u, p.wait_limit))
                        break;   // the consumers time out on the missing chunks and record it
                    // a consumer that timed out releases its slot without waiting for the copy:
                    // never refill a slot whose previous copy is still in flight
                    if (!mbar_wait_bounded(&full[slot], (uint32_t)((v / p.slots) - 1) & 1u, kDefaultWaitLimit))
                        break;
                }
                const int r0 = (g0 + v % nc) * crows;
                const int nr = min(crows, N - r0);
                const uint32_t pb = (uint32_t)nr * rowB;                 // a multiple of 16
                const uint32_t scb = ((uint32_t)nr * srowB) & ~15u;      // whole 16-byte units
                uint8_t* dst = ring + (size_t)slot * p.slot_bytes;
                mbar_arrive_expect_tx(&full[slot], pb + scb);
                bulk_g2s(dst, p.packed + (size_t)r0 * rowB, pb, &full[slot]);
                if (scb) bulk_g2s(dst + off_sc, p.scales + (size_t)r0 * srowB, scb, &full[slot]);
                issued = v + 1;
            }
            // drain: the last fill of every slot has landed before the CTA may exit (with the
            // library's fixed limit, not the caller's: copies in flight always land)
            for (int v = max(0, issued - p.slots); v < issued; ++v)
                mbar_wait_bounded(&full[v % p.slots], (uint32_t)(v / p.slots) & 1u, kDefaultWaitLimit);
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int res = warp / wpc;                     // chunk residue this warp serves
    const int rp = 2 * (warp % wpc);                // its row pair inside the chunk (wpc 4)
    const int nthr = kConsumerWarps * 32;
    const float ts = __ldg(p.tscale);
    const uint16_t qnan = 0x7FC0u;
    const bool warp_uniform_token = (nunit % 32) == 0;
    bool ok = true;
    for (int pass = 0; pass < passes; ++pass) {
        const int t0 = pass * TC, tc = min(TC, T - t0);
        const int units = tc * nunit;
        named_barrier_sync(1, nthr);   // the previous pass is done with the x stage
        if (threadIdx.x < kMaxTc) s_amax[threadIdx.x] = 0u;
        // one read of x: the first kKeep units of each thread stay in registers
        const uint4* xg = reinterpret_cast<const uint4*>(p.x + (size_t)t0 * K);
        uint4 keep[kKeep];
#pragma unroll
        for (int m = 0; m < kKeep; ++m) {
            const int i = threadIdx.x + m * nthr;
            keep[m] = i < units ? xg[i] : make_uint4(0, 0, 0, 0);
        }
        named_barrier_sync(1, nthr);   // s_amax cleared
        // max |x| per token (bf16 magnitudes order as integers); a warp's 32 units belong
        // to one token when K/8 is a multiple of 32
        auto amax_unit = [&](int i, const uint4 v) {
            const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
            uint32_t mx = 0u;
#pragma unroll
            for (int q = 0; q < 4; ++q) mx = max(mx, max(ww[q] & 0x7FFFu, (ww[q] >> 16) & 0x7FFFu));
            if (warp_uniform_token) {
                mx = __reduce_max_sync(0xffffffffu, mx);
                if (lane == 0) atomicMax(&s_amax[(i - lane) / nunit], mx);
            } else if (i < units) {
                atomicMax(&s_amax[i / nunit], mx);
            }
        };
#pragma unroll
        for (int m = 0; m < kKeep; ++m) {
            const int i = threadIdx.x + m * nthr;
            if (i - lane < units) amax_unit(i, keep[m]);
        }
        for (int i = threadIdx.x + kKeep * nthr; i - lane < units; i += nthr)
            amax_unit(i, i < units ? xg[i] : make_uint4(0, 0, 0, 0));
        named_barrier_sync(1, nthr);
        auto stage_unit = [&](int i, const uint4 v) {
            const int t = i / nunit, u = i - t * nunit;        // unit u = elements 8u .. 8u+7
            const float sc = pow2i(gemv_row_shift(s_amax[t]));
            uint4 o;
            o.x = f16x2_of(bf16lo(v.x) * sc, bf16hi(v.x) * sc);
            o.y = f16x2_of(bf16lo(v.y) * sc, bf16hi(v.y) * sc);
            o.z = f16x2_of(bf16lo(v.z) * sc, bf16hi(v.z) * sc);
            o.w = f16x2_of(bf16lo(v.w) * sc, bf16hi(v.w) * sc);
            xs[(size_t)t * nunit + (u & 3) * nseg + (u >> 2)] = o;
        };
#pragma unroll
        for (int m = 0; m < kKeep; ++m) {
            const int i = threadIdx.x + m * nthr;
            if (i < units) stage_unit(i, keep[m]);
        }
        for (int i = threadIdx.x + kKeep * nthr; i < units; i += nthr) stage_unit(i, xg[i]);
        named_barrier_sync(1, nthr);
        if (pass == 0) asm volatile("griddepcontrol.launch_dependents;");
        float inv[TC];
#pragma unroll
        for (int t = 0; t < TC; ++t) inv[t] = t < tc ? pow2i(-gemv_row_shift(s_amax[t])) : 0.f;

        // group `res` takes the chunks whose sequence number v = pass * nc + ci is res modulo
        // the group count; the slot count is a multiple of it, so every slot is refilled only
        // for the group that consumed it, which takes its fills in order (the parity of a
        // fill's "full" phase is then never mistaken for an older one)
        const int ci0 = ((res - (pass * nc) % kChunkResidues) % kChunkResidues + kChunkResidues) % kChunkResidues;
        if (wide) {
            // one warp per chunk of 8 rows (each warp owns one slot): lane l takes segments l,
            // l + 32, ... of the 8 rows with the activation segment in registers, 8 fp32 sums per
            // lane, then one transpose reduction (warp_sum8_lanes) leaves row (l >> 2) & 7's sum
            // on lane l
            const int rb8 = 8 * (warp % wpc);            // this warp's 8 rows inside the chunk
            for (int ci = ci0; ci < nc; ci += kChunkResidues) {
                const int v = pass * nc + ci, slot = v % p.slots;
                if (ok && !mbar_wait_bounded(&full[slot], (uint32_t)(v / p.slots) & 1u, p.wait_limit)) ok = false;
                const int c0r = (g0 + ci) * crows;                    // the chunk's first row
                const int nrc = min(crows, N - c0r);                  // rows in the chunk
                const int r0 = c0r + rb8, nr = min(kCRows1, nrc - rb8);   // this warp's rows
                if (nr <= 0) {
                } else if (!ok) {
                    if (lane < nr) p.y[r0 + lane] = qnan;
                } else {
                    const uint8_t* slotp = ring + (size_t)slot * p.slot_bytes;
                    const uint32_t slot_sa = smem_addr(slotp);
                    const uint32_t scb = ((uint32_t)nrc * srowB) & ~15u;
                    float acc[kCRows1];
#pragma unroll
                    for (int rr = 0; rr < kCRows1; ++rr) acc[rr] = 0.f;
                    for (int s = lane; s < nseg; s += 32) {
                        const uint4 u0 = xs[s], u1 = xs[nseg + s], u2 = xs[2 * nseg + s], u3 = xs[3 * nseg + s];
#pragma unroll
                        for (int rr = 0; rr < kCRows1; ++rr) {
                            if (rr < nr) {
                                // a row whose scales did not fit the chunk's whole 16-byte units
                                // (only in a ragged last chunk) reads them from global memory
                                float a0, a1;
                                if ((uint32_t)(rb8 + rr + 1) * srowB <= scb)
                                    seg_scales_sh<KIND>(slot_sa + off_sc + (uint32_t)(rb8 + rr) * srowB, s, a0, a1);
                                else
                                    seg_scales<KIND>(p.scales + (size_t)(r0 + rr) * srowB, s, a0, a1);
                                uint32_t q[16];
                                expand_seg(reinterpret_cast<const uint4*>(slotp + (size_t)(rb8 + rr) * rowB)[s], q);
                                acc[rr] += seg1(q, u0, u1, u2, u3, a0, a1);
                            }
                        }
                    }
                    const float z = warp_sum8_lanes(acc, lane);
                    const int rr = (lane >> 2) & 7;
                    if ((lane & 3) == 0 && rr < nr) p.y[r0 + rr] = f32_to_bf16((z * ts) * inv[0]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
            continue;
        }
        for (int ci = ci0; ci < nc; ci += kChunkResidues) {
            const int v = pass * nc + ci, slot = v % p.slots;
            if (ok && !mbar_wait_bounded(&full[slot], (uint32_t)(v / p.slots) & 1u, p.wait_limit)) ok = false;
            const int r0 = (g0 + ci) * crows, ra = r0 + rp;
            if (ra < N) {
                const bool has_b = ra + 1 < N;
                if (!ok) {
                    if (lane < tc) {
                        p.y[(size_t)(t0 + lane) * N + ra] = qnan;
                        if (has_b) p.y[(size_t)(t0 + lane) * N + ra + 1] = qnan;
                    }
                } else {
                    const uint8_t* slotp = ring + (size_t)slot * p.slot_bytes;
                    const uint8_t* rowa = slotp + (size_t)rp * rowB;
                    const uint8_t* rowb = has_b ? rowa + rowB : rowa;
                    const int nr = min(crows, N - r0);
                    const uint32_t scb = ((uint32_t)nr * srowB) & ~15u;
                    // a row whose scales did not fit the chunk's whole 16-byte units (only in a
                    // ragged last chunk) reads them from global memory
                    const int rb = has_b ? ra + 1 : ra;
                    const bool sa_sh = (uint32_t)(rp + 1) * srowB <= scb;
                    const bool sb_sh = (uint32_t)(rp + (has_b ? 2 : 1)) * srowB <= scb;
                    const uint32_t sra_sh = smem_addr(slotp) + off_sc + (uint32_t)rp * srowB;
                    const uint32_t srb_sh = smem_addr(slotp) + off_sc + (uint32_t)(rb - r0) * srowB;
                    const uint8_t* sra = p.scales + (size_t)ra * srowB;
                    const uint8_t* srb = p.scales + (size_t)rb * srowB;
                    float acca[TC], accb[TC];
#pragma unroll
                    for (int t = 0; t < TC; ++t) acca[t] = accb[t] = 0.f;
#pragma unroll 2
                    for (int s = lane; s < nseg; s += 32) {
                        const uint4 wa = reinterpret_cast<const uint4*>(rowa)[s];
                        const uint4 wb = reinterpret_cast<const uint4*>(rowb)[s];
                        float a0, a1, b0, b1;
                        if (sa_sh) seg_scales_sh<KIND>(sra_sh, s, a0, a1);
                        else seg_scales<KIND>(sra, s, a0, a1);
                        if (sb_sh) seg_scales_sh<KIND>(srb_sh, s, b0, b1);
                        else seg_scales<KIND>(srb, s, b0, b1);
                        uint32_t qa[16], qb[16];
                        expand_seg(wa, qa);
                        expand_seg(wb, qb);
#pragma unroll
                        for (int t = 0; t < TC; ++t)
                            if (t < tc) seg2<KIND>(qa, qb, xs + (size_t)t * nunit, nseg, s, a0, a1, b0, b1, acca[t], accb[t]);
                    }
#pragma unroll
                    for (int t = 0; t < TC; ++t) {
                        if (t < tc) {
                            const float v2 = warp_sum_pair(acca[t], accb[t], lane);
                            const float o = (v2 * ts) * inv[t];
                            if (lane == 0) p.y[(size_t)(t0 + t) * N + ra] = f32_to_bf16(o);
                            if (lane == 16 && has_b) p.y[(size_t)(t0 + t) * N + ra + 1] = f32_to_bf16(o);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }
    if (!ok && lane == 0 && p.hdr) record_status(p.hdr, NVFP4_ERR_DEVICE_TIMEOUT);
}

struct GemvPlan {
    int tc, slots, grid, wpc, crows, wide;
    uint32_t slot_bytes, off_ring, smem;
};

GemvPlan plan_gemv(const nvfp4_weight& W, int T, const DeviceInfo& dev) {
    GemvPlan g;
    const int K = W.K, N = W.N;
    const uint32_t srow = (uint32_t)scale_row_bytes_of(W.kind, W.K);
    g.tc = T >= 8 ? 8 : T >= 4 ? 4 : T >= 2 ? 2 : 1;
    if (T == 3) g.tc = 4;
    if (T >= 5 && T < 8) g.tc = 8;
    g.off_ring = (uint32_t)g.tc * (uint32_t)K * 2u;
    const int passes = (T + g.tc - 1) / g.tc;
    // one token and a long row range per CTA: chunks of 32 rows (few, large bulk copies: each
    // SM keeps only a handful of them in flight), 4 warps per chunk with 8 rows each, one ring
    // slot per group of 4 warps (one CTA per SM)
    {
        constexpr int kWideWpc = 4;
        const int cw1 = consumer_warps(1), crows = kCRows1 * kWideWpc, groups = cw1 / kWideWpc;
        const int ngw = (N + crows - 1) / crows;
        const int gridw = ngw < dev.num_sms ? ngw : dev.num_sms;
        const uint32_t sbw = (uint32_t)crows * ((uint32_t)K / 2 + srow);
        if (g.tc == 1 && (ngw + gridw - 1) / gridw >= 2 * groups &&
            g.off_ring + (uint32_t)groups * sbw + 2048u <= (uint32_t)dev.smem_optin) {
            g.wpc = kWideWpc;
            g.wide = 1;
            g.crows = crows;
            g.grid = gridw;
            g.slot_bytes = sbw;
            g.slots = groups;
            g.smem = g.off_ring + (uint32_t)g.slots * g.slot_bytes;
            return g;
        }
    }
    g.wide = 0;
    g.wpc = kWarpsPerChunk;
    g.crows = kCRows;
    const int ngroups = (N + kCRows - 1) / kCRows;
    g.grid = ngroups < dev.num_sms ? ngroups : dev.num_sms;
    const int nc_max = (ngroups + g.grid - 1) / g.grid;
    g.slot_bytes = (uint32_t)kCRows * ((uint32_t)K / 2 + srow);
    const long want = (long)nc_max * passes;
    // two CTAs per SM when the ring and stage fit in ~100 KB (the next launch's
    // weight prologue then overlaps this one under programmatic dependent launch)
    const uint32_t small_cap = 100u * 1024u;
    const uint32_t cap = (g.off_ring + 2u * g.slot_bytes <= small_cap) ? small_cap
                                                                       : (uint32_t)dev.smem_optin - 2048u;
    long fit = ((long)cap - (long)g.off_ring) / (long)g.slot_bytes;
    if (fit > kMaxSlots) fit = kMaxSlots;
    // a multiple of the consumer groups (each group owns the slots of its residue): the
    // chunk count rounded up where that fits, else the largest multiple that fits
    const int groups = consumer_warps(g.tc) / kWarpsPerChunk;
    long slots = (want + groups - 1) / groups * groups;
    if (slots > fit) slots = fit / groups * groups;
    if (slots < groups) slots = groups;
    g.slots = (int)slots;
    g.smem = g.off_ring + (uint32_t)g.slots * g.slot_bytes;
    return g;
}

template <int KIND, int TC>
cudaError_t launch_one(const GemvParams& P, const GemvPlan& g, const DeviceInfo& dev, cudaStream_t s) {
    static std::atomic<uint32_t> set_bytes[64];
    const int dv = dev.device < 64 ? dev.device : 63;
    if (set_bytes[dv].load(std::memory_order_relaxed) < g.smem) {
        cudaError_t err = cudaFuncSetAttribute(gemv_kernel<KIND, TC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)g.smem);
        if (err != cudaSuccess) return err;
        set_bytes[dv].store(g.smem, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.grid);
    cfg.blockDim = dim3(gemv_threads(TC));
    cfg.dynamicSmemBytes = g.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<KIND, TC>, P);
}

template <int KIND>
cudaError_t launch_kind(const GemvParams& P, const GemvPlan& g, const DeviceInfo& dev, cudaStream_t s) {
    switch (g.tc) {
        case 1: return launch_one<KIND, 1>(P, g, dev, s);
        case 2: return launch_one<KIND, 2>(P, g, dev, s);
        case 4: return launch_one<KIND, 4>(P, g, dev, s);
        default: return launch_one<KIND, 8>(P, g, dev, s);
    }
}

}  // namespace

cudaError_t launch_gemv(const nvfp4_weight& W, const uint16_t* x, int T, uint16_t* y, WsHeader* hdr,
                        const DeviceInfo& dev, uint64_t wait_limit, cudaStream_t s) {
    const GemvPlan g = plan_gemv(W, T, dev);
    if (g.smem > dev.smem_optin) return cudaErrorInvalidConfiguration;
    GemvParams P;
    P.packed = W.packed;
    P.scales = static_cast<const uint8_t*>(W.scales);
    P.tscale = W.tensor_scale;
    P.x = x;
    P.y = y;
    P.hdr = hdr;
    P.wait_limit = wait_limit;
    P.N = W.N;
    P.K = W.K;
    P.T = T;
    P.ngroups = (W.N + g.crows - 1) / g.crows;
    P.wpc = g.wpc;
    P.crows = g.crows;
    P.wide = g.wide;
    P.slots = g.slots;
    P.slot_bytes = g.slot_bytes;
    P.off_ring = g.off_ring;
    cudaError_t err;
    switch (W.kind) {
        case NVFP4_SCALE_E4M3: err = launch_kind<NVFP4_SCALE_E4M3>(P, g, dev, s); break;
        case NVFP4_SCALE_FP16: err = launch_kind<NVFP4_SCALE_FP16>(P, g, dev, s); break;
        case NVFP4_SCALE_FP32: err = launch_kind<NVFP4_SCALE_FP32>(P, g, dev, s); break;
        default: err = launch_kind<NVFP4_SCALE_UE8M0>(P, g, dev, s); break;
    }
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace nvfp4
