// MoE layer, multi-token decode (1..64 tokens per call, E4M3 block scales): router
// GEMV with the fused route, grouped gate/up + SwiGLU and grouped down on the
// warp-level tensor cores, then the routing-weighted combine.
//
// Sources (page title, section):
//  - lynn-engine tutorials index, row 06 "MoE router" (softmax over all experts ->
//    top-k -> renormalise; sigmoid-gated shared expert).
//  - lynn-engine README, P28 note (gate/up + SiLU over the active experts only,
//    [top_k, I] intermediate), P29 note (down + weighted sum -> [H]), P46/P48 notes
//    (no float atomics in the combine: every output element is summed by one
//    thread in a fixed order).
//
// Each routed expert with n entries, and the shared expert (whose entries are the T
// tokens), is a small GEMM: weight rows times up to 16 entries per pass. The weight
// rows sit on the M side of mma.sync m16n8k16 (f16 in, fp32 accumulate), the
// entries on its N side (one or two n8 blocks). The NVFP4 codes go from HBM into
// registers and are expanded there into the A fragments: cvt gives the E2M1 codes
// as f16 and one f16x2 multiply applies the E4M3 block scale; the product has at
// most 6 significant bits and lies in [2^-10, 2688], so it is exact. No shared-memory
// round trip, no copy of a weight.
//
// Operand B is the entries' activation rows (x for gate/up, h for down), staged
// once per CTA in shared memory as f16. Each row is first multiplied by 2^k_r, the
// power of two that puts its largest magnitude in [2^14, 2^15): no f16 overflow
// for any finite bf16 or fp32 row, and every element within 2^-28 of the row's largest
// converts exactly (a bf16 has 8 significant bits, f16 11); smaller elements carry
// an absolute error below 2^-39 of the row's largest. The epilogue multiplies the
// fp32 accumulator by 2^-k_r (exact). Row maxima come from the router kernel (x)
// and from the gate/up epilogue (h, an atomicMax over bit patterns of non-negative
// floats: order-independent, so deterministic).
//
// K order. A contraction may visit K in any order as long as both operands use the
// same one. In 256-element chunk j, the lanes of quad position q (lane % 4) own the
// 64 elements [256j + 64q, 256j + 64q + 64): 32 code bytes (two 16-byte loads per
// weight row) and 4 block scales (one 32-bit load). MMA step s (0..15) of the chunk
// takes elements 256j + 64q + 4s + {0, 1} as fragment k positions {2q, 2q+1} and
// + {2, 3} as {2q+8, 2q+9}, in A and in B alike; each lane's four elements of a
// step are one 16-element scale block.
#include "common.cuh"
#include "kernels.cuh"
#include "route_mt.cuh"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPass = 16;          // entries per pass: two n8 MMA blocks
constexpr int kGuPairs = 64;       // gate/up row pairs per CTA item (8 per warp)
constexpr int kDnRows = 128;       // down output rows per CTA item (16 per warp)
constexpr int kRouterTok = 8;      // tokens per router CTA (the last CTA of a block: one warp per token)
constexpr int kMaxDim = 4096;      // H, I, Is bound of this path (shared-memory staging)
static_assert(NVFP4_DECODE_MAX_TOKENS / kRouterTok <= kRouteTicketBlocks, "one ticket counter per token block");

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                 "{%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Row scaling: k with max|row| * 2^k in [2^14, 2^15), from the fp32 bits of max|row|
// (0 for an all-zero row; clamped to [-126, 126] so that 2^k and 2^-k are normal:
// the largest finite row, max|row| < 2^128, still lands below 2^15).
__device__ __forceinline__ int row_shift(uint32_t amax_bits) {
    if (amax_bits == 0u) return 0;
    const int e = (int)(amax_bits >> 23) - 127;
    return min(126, max(-126, 14 - e));
}
__device__ __forceinline__ float exp2i(int k) { return __int_as_float((k + 127) << 23); }

// Two fp32 -> f16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Staged row r, 8-byte unit u (four f16) lives at unit u ^ (((u >> 2) & 12) | (r & 3)).
// In one MMA step the 16 lanes of a half-warp (rows r & 3 = g & 3, quads q) read
// units whose low four bits are s ^ (4q | (g & 3)): 16 distinct bank pairs.
__device__ __forceinline__ uint32_t swz(uint32_t u, uint32_t r) { return u ^ (((u >> 2) & 12u) | (r & 3u)); }

// One weight row's share of a chunk for one lane: 32 code bytes and 4 E4M3 scales.
struct WChunk {
    uint4 lo, hi;
    uint32_t sc;
};

__device__ __forceinline__ WChunk load_chunk(const uint8_t* codes, const uint8_t* scl, int j, uint64_t pol) {
    WChunk c;
    c.lo = ld_stream_v4_ef(codes + 128 * j, pol);
    c.hi = ld_stream_v4_ef(codes + 128 * j + 16, pol);
    c.sc = ld_stream_u32_ef(scl + 16 * j, pol);
    return c;
}

// Four E2M1 code bytes (one 32-bit word: two MMA steps of one weight row) -> four
// f16x2 of code * scale. The word is unpacked into byte registers for cvt.
__device__ __forceinline__ void expand_word(uint32_t w, uint32_t s2, uint32_t (&o)[4]) {
    uint32_t h[4];
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
#pragma unroll
    for (int b = 0; b < 4; ++b) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[b]) : "r"(h[b]), "r"(s2));
}

__device__ __forceinline__ uint32_t word_of(const WChunk& c, int wi) {
    const uint4& v = wi < 4 ? c.lo : c.hi;
    const int w = wi & 3;
    return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

// E4M3 scales of four blocks (one 32-bit word) -> four f16x2 {scale, scale}
// (exact): two cvt of two bytes each, then byte permutes duplicate each half.
__device__ __forceinline__ void scales4(uint32_t sc, uint32_t (&o)[4]) {
    uint32_t lo, hi;
    asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n cvt.rn.f16x2.e4m3x2 %1, b;\n}"
        : "=r"(lo), "=r"(hi) : "r"(sc));
    o[0] = __byte_perm(lo, 0, 0x1010);
    o[1] = __byte_perm(lo, 0, 0x3232);
    o[2] = __byte_perm(hi, 0, 0x1010);
    o[3] = __byte_perm(hi, 0, 0x3232);
}

// The 16 MMA steps of one chunk: A rows (c0: fragment rows 0-7, c1: rows 8-15),
// B from NB staged n8 blocks (row g and g + 8 of the stage). Code word wi holds
// steps 2wi (bytes 0, 1) and 2wi + 1 (bytes 2, 3), both in scale block wi / 2.
template <int NB>
__device__ __forceinline__ void chunk_mma(float (&acc)[2][4], const WChunk& c0, const WChunk& c1,
                                          const uint8_t* brow0, const uint8_t* brow1, uint32_t ubase,
                                          uint32_t xmask) {
    uint32_t s0[4], s1[4];
    scales4(c0.sc, s0);
    scales4(c1.sc, s1);
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
        uint32_t a[4], u[4];
        expand_word(word_of(c0, wi), s0[wi >> 1], a);
        expand_word(word_of(c1, wi), s1[wi >> 1], u);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int s = 2 * wi + h;
            const uint32_t off = 8u * (ubase + ((uint32_t)s ^ xmask));
            const uint2 b0 = *reinterpret_cast<const uint2*>(brow0 + off);
            mma_16816(acc[0], a[2 * h], u[2 * h], a[2 * h + 1], u[2 * h + 1], b0.x, b0.y);
            if (NB == 2) {
                const uint2 b1 = *reinterpret_cast<const uint2*>(brow1 + off);
                mma_16816(acc[1], a[2 * h], u[2 * h], a[2 * h + 1], u[2 * h + 1], b1.x, b1.y);
            }
        }
    }
}

// K loop over nchunk chunks with the next chunk's loads in flight during the MMAs.
template <int NB>
__device__ __forceinline__ void k_loop(float (&acc)[2][4], const uint8_t* codes0, const uint8_t* scl0,
                                       const uint8_t* codes1, const uint8_t* scl1, int nchunk,
                                       const uint8_t* brow0, const uint8_t* brow1, uint32_t q,
                                       uint32_t xmask, WChunk c0, WChunk c1, uint64_t pol) {
    for (int j = 0; j < nchunk; ++j) {
        WChunk n0 = c0, n1 = c1;
        if (j + 1 < nchunk) {
            n0 = load_chunk(codes0, scl0, j + 1, pol);
            n1 = load_chunk(codes1, scl1, j + 1, pol);
        }
        chunk_mma<NB>(acc, c0, c1, brow0, brow1, 64u * j + 16u * q, xmask);
        c0 = n0;
        c1 = n1;
    }
}

// Two 16-row tiles, rows [0, 8) + [8, 16) and the same 128 rows further on, over the
// same K and one n8 block: the K loop runs over the first tile's chunks, then the
// second's, with the next chunk's loads in flight across the boundary.
__device__ __forceinline__ void k_loop_tiles(float (&accA)[2][4], float (&accB)[2][4], const uint8_t* codes0,
                                             const uint8_t* scl0, const uint8_t* codes1, const uint8_t* scl1,
                                             uint32_t tile_codes, uint32_t tile_scl, int nchunk, const uint8_t* brow0,
                                             uint32_t q, uint32_t xmask, WChunk c0, WChunk c1, uint64_t pol) {
    const int n2 = 2 * nchunk;
    for (int v = 0; v < n2; ++v) {
        WChunk n0 = c0, n1 = c1;
        if (v + 1 < n2) {
            const bool tb = v + 1 >= nchunk;
            const int jn = tb ? v + 1 - nchunk : v + 1;
            const uint32_t oc = tb ? tile_codes : 0u, os = tb ? tile_scl : 0u;
            n0 = load_chunk(codes0 + oc, scl0 + os, jn, pol);
            n1 = load_chunk(codes1 + oc, scl1 + os, jn, pol);
        }
        if (v < nchunk) chunk_mma<1>(accA, c0, c1, brow0, brow0, 64u * v + 16u * q, xmask);
        else chunk_mma<1>(accB, c0, c1, brow0, brow0, 64u * (v - nchunk) + 16u * q, xmask);
        c0 = n0;
        c1 = n1;
    }
}

// ------------------------------------------------------------------ router + route
// logits[t, e] = x[t] . Wg[e] (e < E); gate_logit[t] = x[t] . gs (row E). CTA
// (bx, by) = rr rows x the 8 tokens of block by (rr = 2, 4 or 8, the fewest rows that
// keep the grid resident at once): warp w takes row rr bx + w / (8 / rr) and rr of the
// block's tokens, two per pass (at rr = 2 each warp's chain is one row load and one
// pass of two dot products). A lane holds its 16-byte chunks of the row
// as fp32 and reads the tokens' chunks from shared memory (consecutive lanes,
// consecutive 16 bytes: conflict-free). Then a ticket per token block: the CTA that
// finishes last takes the top-k of those tokens, and the token block that finishes
// last builds the lists. Nothing waits: a CTA that is not last simply exits, and the
// last one resets its counter for the next call.
__global__ void __launch_bounds__(kThreads)
router_route_mt_kernel(const uint16_t* __restrict__ wg, const uint16_t* __restrict__ gs,
                       const uint16_t* __restrict__ x, int T, int E, int H, int k, int rr, float* logits,
                       float* gate_logit, int32_t* ids, float* w, int32_t* ids_out, float* w_out,
                       int32_t* offsets, int32_t* token_list, int32_t* active, int32_t* pass_map,
                       uint32_t* amax, WsHeader* hdr) {
    extern __shared__ uint4 xs4[];
    __shared__ ListsSmem S;
    __shared__ int s_last;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = H >> 3;
    const int rows = E + (gs ? 1 : 0);
    const int wpr = kWarps / rr;                          // warps per row
    const int r = blockIdx.x * rr + warp / wpr;
    const int tp = rr * (warp % wpr);                     // the warp's first token in the block
    const int t0 = blockIdx.y * kRouterTok;
    const int tc = min(kRouterTok, T - t0);
    const uint16_t* row = r < E ? wg + (size_t)r * H : gs;
    uint4 wraw[8];   // this lane's chunks of the router row, requested before x is staged
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int c = lane + 32 * i;
        wraw[i] = make_uint4(0, 0, 0, 0);
        if (r < rows && nch <= 256 && c < nch) wraw[i] = *reinterpret_cast<const uint4*>(row + 8 * (size_t)c);
    }
    for (int i = threadIdx.x; i < tc * nch; i += kThreads)
        xs4[i] = *reinterpret_cast<const uint4*>(x + (size_t)t0 * H + 8 * (size_t)i);
    __syncthreads();
    if (blockIdx.x == 0) {
        // max |x| of each token of the block (bf16 magnitudes order as integers),
        // stored as fp32 bits; block (0, 0) also clears the h row maxima that the
        // gate/up kernel accumulates
        for (int t = warp; t < tc; t += kWarps) {
            uint32_t m = 0u;
            for (int c = lane; c < nch; c += 32) {
                const uint4 v = xs4[t * nch + c];
                const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int p = 0; p < 4; ++p) m = max(m, max(ww[p] & 0x7FFFu, (ww[p] >> 16) & 0x7FFFu));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) amax[t0 + t] = m << 16;
        }
        if (blockIdx.y == 0)
            for (int i = threadIdx.x; i < T * k + T; i += kThreads) amax[T + i] = 0u;
    }
    if (r < rows && tp < tc) {
        if (nch <= 256) {
            float wf[8][8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 v = wraw[i];
                const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    wf[i][2 * p] = bf16lo(ww[p]);
                    wf[i][2 * p + 1] = bf16hi(ww[p]);
                }
            }
#pragma unroll 1
            for (int t = tp; t < min(tc, tp + rr); t += 2) {   // two tokens per pass: two independent chains
                const bool two = t + 1 < tc;
                float a = 0.f, b = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = lane + 32 * i;
                    if (c < nch) {
                        const uint4 xv = xs4[t * nch + c];
                        const uint4 yv = two ? xs4[(t + 1) * nch + c] : make_uint4(0, 0, 0, 0);
                        const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
                        const uint32_t yy[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            a = fmaf(wf[i][2 * p], bf16lo(xx[p]), a);
                            a = fmaf(wf[i][2 * p + 1], bf16hi(xx[p]), a);
                            b = fmaf(wf[i][2 * p], bf16lo(yy[p]), b);
                            b = fmaf(wf[i][2 * p + 1], bf16hi(yy[p]), b);
                        }
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    a += __shfl_xor_sync(0xffffffffu, a, o);
                    b += __shfl_xor_sync(0xffffffffu, b, o);
                }
                if (lane == 0) {
                    if (r < E) {
                        logits[(size_t)(t0 + t) * E + r] = a;
                        if (two) logits[(size_t)(t0 + t + 1) * E + r] = b;
                    } else {
                        gate_logit[t0 + t] = a;
                        if (two) gate_logit[t0 + t + 1] = b;
                    }
                }
            }
        } else {
#pragma unroll 1
            for (int t = tp; t < min(tc, tp + rr); ++t) {
                float a = 0.f;
#pragma unroll 1
                for (int c = lane; c < nch; c += 32) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + 8 * (size_t)c));
                    const uint4 xv = xs4[t * nch + c];
                    const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
                    const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        a = fmaf(bf16lo(ww[p]), bf16lo(xx[p]), a);
                        a = fmaf(bf16hi(ww[p]), bf16hi(xx[p]), a);
                    }
                }
                a = warp_sum(a);
                if (lane == 0) {
                    if (r < E) logits[(size_t)(t0 + t) * E + r] = a;
                    else gate_logit[t0 + t] = a;
                }
            }
        }
    }
    // barrier, then one thread fences and takes the ticket (the block's writes are
    // ordered before the fence by the barrier)
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(&hdr->route_tickets[blockIdx.y], 1u) == gridDim.x - 1;
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    // one token block (T <= 8): this CTA is also the last overall, keeps the ids in shared
    // memory for the lists and skips the second ticket
    const bool one_block = gridDim.y == 1;
    for (int t = t0 + warp; t < t0 + tc; t += kWarps) {
        const size_t o = (size_t)t * k;
        topk_warp_mt(logits + (size_t)t * E, E, k, ids + o, w + o, ids_out ? ids_out + o : nullptr,
                     w_out ? w_out + o : nullptr, one_block ? S.ids + o : nullptr);
    }
    __syncthreads();
    if (one_block) {
        if (threadIdx.x == 0) atomicExch(&hdr->route_tickets[0], 0u);
        build_lists_block(S, ids, T * k, E, offsets, token_list, active, pass_map, true);
        return;
    }
    if (threadIdx.x == 0) {
        __threadfence();
        atomicExch(&hdr->route_tickets[blockIdx.y], 0u);
        s_last = atomicAdd(&hdr->route_tickets[kRouteTicketBlocks], 1u) == gridDim.y - 1;
        if (s_last) __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    build_lists_block(S, ids, T * k, E, offsets, token_list, active, pass_map, false);
    if (threadIdx.x == 0) atomicExch(&hdr->route_tickets[kRouteTicketBlocks], 0u);
}

// ------------------------------------------------------------------ gate/up
// Item = (slot pass, block of 64 row pairs); NBMAX n8 entry blocks at most (1 when a
// call has at most 8 tokens, so every pass has at most 8 entries). Routed passes come from the pass map
// (active slot a, entries [16 pi, 16 pi + 16) of expert a's list); the shared
// expert's pass pi is tokens [16 pi, 16 pi + 16). Warp w takes gate rows
// i0 + 8w + g as fragment rows 0-7 and the matching up rows as rows 8-15, so lane
// (g, q) ends with gate and up of row i0 + 8w + g for entries 2q, 2q+1 of each n8
// block: h = silu(ts_g * gate) * (ts_u * up), written in fp32 (entry-major [T*k, I]
// for the routed experts, [T, Is] for the shared one). hmax keeps each h row's
// largest magnitude (routed entry e at e, shared token t at T*k + t).
template <int NBMAX, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
gateup_mt_kernel(moe_layer_desc d, const uint16_t* __restrict__ x, int T,
                 const int32_t* __restrict__ offsets, const int32_t* __restrict__ token_list,
                 const int32_t* __restrict__ active, const int32_t* __restrict__ pass_map,
                 const uint32_t* __restrict__ xmax, uint32_t* __restrict__ hmax, float* __restrict__ h,
                 float* __restrict__ hs) {
    extern __shared__ __align__(16) uint8_t stage[];
    __shared__ uint32_t s_hmax[kPass];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t g = lane >> 2, q = lane & 3;
    const int H = d.H, k = d.k;
    const int rb_r = d.I / kGuPairs, rb_s = d.Is / kGuPairs;
    const int items_r = pass_map[0] * rb_r;
    const int items = items_r + (T + kPass - 1) / kPass * rb_s;
    const int nchunk = H >> 8;
    const uint32_t xmask = 4u * q | (g & 3u);
    const uint64_t pol = l2_evict_first_policy();
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const uint8_t* codes;
        const uint8_t* scl;
        const int32_t* list;   // routed: the pass's entries; shared: none (tokens first + r)
        float tsg, tsu;
        int Irows, i0, n, first;
        float* out;
        if (item < items_r) {
            const int p = item / rb_r;
            const int pm = pass_map[1 + p];
            const int e = active[1 + (pm >> 8)];
            const int beg = offsets[e] + kPass * (pm & 255);
            n = min(kPass, offsets[e + 1] - beg);
            list = token_list + beg;
            first = 0;
            i0 = (item - p * rb_r) * kGuPairs;
            Irows = d.I;
            codes = d.gu_packed + (size_t)e * 2 * d.I * (H / 2);
            scl = static_cast<const uint8_t*>(d.gu_scales) + (size_t)e * 2 * d.I * (H / 16);
            tsg = __ldg(d.gu_tscale + 2 * e);
            tsu = __ldg(d.gu_tscale + 2 * e + 1);
            out = h;
        } else {
            const int it = item - items_r;
            const int pi = it / rb_s;
            first = kPass * pi;
            n = min(kPass, T - first);
            list = nullptr;
            i0 = (it - pi * rb_s) * kGuPairs;
            Irows = d.Is;
            codes = d.sh_gu_packed;
            scl = static_cast<const uint8_t*>(d.sh_gu_scales);
            tsg = __ldg(d.sh_gu_tscale);
            tsu = __ldg(d.sh_gu_tscale + 1);
            out = hs;
        }
        // entry r of the pass: its token, its h row, its slot in hmax
        auto tok = [&](int r) { return list ? list[r] / k : first + r; };
        auto hrow = [&](int r) { return list ? list[r] : first + r; };
        auto hidx = [&](int r) { return list ? list[r] : T * k + first + r; };
        const int i = i0 + 8 * warp + (int)g;
        const uint8_t* cg = codes + (size_t)i * (H / 2) + 32 * q;
        const uint8_t* cu = codes + (size_t)(Irows + i) * (H / 2) + 32 * q;
        const uint8_t* sg = scl + (size_t)i * (H / 16) + 4 * q;
        const uint8_t* su = scl + (size_t)(Irows + i) * (H / 16) + 4 * q;
        const WChunk c0 = load_chunk(cg, sg, 0, pol), c1 = load_chunk(cu, su, 0, pol);
        __syncthreads();   // the previous item is done with the stage and s_hmax
        if (threadIdx.x < kPass) s_hmax[threadIdx.x] = 0u;
        {   // x rows of the entries, times 2^k_t, as f16
            const int per_row = H >> 3;
            for (int idx = threadIdx.x; idx < n * per_row; idx += kThreads) {
                const int r = idx / per_row, v = idx - r * per_row;
                const int t = tok(r);
                const float sc = exp2i(row_shift(__ldg(xmax + t)));
                const uint4 val = *reinterpret_cast<const uint4*>(x + (size_t)t * H + 8 * (size_t)v);
                uint2* dst = reinterpret_cast<uint2*>(stage + (size_t)r * H * 2);
                dst[swz(2 * v, r)] = make_uint2(f16x2_of(bf16lo(val.x) * sc, bf16hi(val.x) * sc),
                                                f16x2_of(bf16lo(val.y) * sc, bf16hi(val.y) * sc));
                dst[swz(2 * v + 1, r)] = make_uint2(f16x2_of(bf16lo(val.z) * sc, bf16hi(val.z) * sc),
                                                    f16x2_of(bf16lo(val.w) * sc, bf16hi(val.w) * sc));
            }
        }
        __syncthreads();
        float acc[2][4] = {};
        const uint8_t* b0 = stage + (size_t)g * H * 2;
        const uint8_t* b1 = stage + (size_t)(g + 8) * H * 2;
        if (NBMAX == 2 && n > 8) k_loop<2>(acc, cg, sg, cu, su, nchunk, b0, b1, q, xmask, c0, c1, pol);
        else k_loop<1>(acc, cg, sg, cu, su, nchunk, b0, b1, q, xmask, c0, c1, pol);
#pragma unroll
        for (int nb = 0; nb < NBMAX; ++nb) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int r = 8 * nb + 2 * (int)q + c;
                uint32_t m = 0u;
                if (r < n) {
                    const float inv = exp2i(-row_shift(__ldg(xmax + tok(r))));
                    const float gv = acc[nb][c] * inv * tsg, uv = acc[nb][2 + c] * inv * tsu;
                    const float hv = silu_f32(gv) * uv;
                    out[(size_t)hrow(r) * Irows + i] = hv;
                    m = __float_as_uint(fabsf(hv));
                }
                // largest |h| of entry r over the warp's eight rows (lanes sharing q)
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
                m = max(m, __shfl_xor_sync(0xffffffffu, m, 16));
                if (g == 0 && r < n) atomicMax(&s_hmax[r], m);
            }
        }
        __syncthreads();
        if (threadIdx.x < n) atomicMax(&hmax[hidx(threadIdx.x)], s_hmax[threadIdx.x]);
    }
}

// ------------------------------------------------------------------ down
// Item = (slot pass, block of 128 TILES output rows). Warp w takes rows
// nr = 128 TILES rb + 16w + g (fragment rows 0-7) and nr + 8 (rows 8-15) over K = I
// (Is for the shared expert), and with TILES = 2 the same rows 128 further on in the
// same K loop; the entries' h rows are staged as f16 times 2^k_h.
// Output rows, fp32, one writer each:
//   P[entry, n] = w_entry * ts_e * (D_e[n] . h_entry)          (routed)
//   Ps[t, n]    = sigmoid(gate_t) * ts_s * (Ds[n] . hs_t)       (shared)
template <int NBMAX, int MINB, int TILES>
__global__ void __launch_bounds__(kThreads, MINB)
down_mt_kernel(moe_layer_desc d, int T, const int32_t* __restrict__ offsets,
               const int32_t* __restrict__ token_list, const int32_t* __restrict__ active,
               const int32_t* __restrict__ pass_map, const float* __restrict__ wts,
               const float* __restrict__ gate_logit, const float* __restrict__ h,
               const float* __restrict__ hs, const uint32_t* __restrict__ hmax, float* __restrict__ P,
               float* __restrict__ Ps) {
    extern __shared__ __align__(16) uint8_t stage[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t g = lane >> 2, q = lane & 3;
    const int H = d.H, k = d.k;
    const int rb_n = H / (TILES * kDnRows);
    const int items_r = pass_map[0] * rb_n;
    const int items = items_r + (d.Is > 0 ? (T + kPass - 1) / kPass * rb_n : 0);
    const uint32_t xmask = 4u * q | (g & 3u);
    const uint64_t pol = l2_evict_first_policy();
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const uint8_t* codes;
        const uint8_t* scl;
        const int32_t* list;
        const float* src;
        float ts;
        int K, n, first, rb;
        if (item < items_r) {
            const int p = item / rb_n;
            const int pm = pass_map[1 + p];
            const int e = active[1 + (pm >> 8)];
            const int beg = offsets[e] + kPass * (pm & 255);
            n = min(kPass, offsets[e + 1] - beg);
            list = token_list + beg;
            first = 0;
            rb = item - p * rb_n;
            K = d.I;
            codes = d.dn_packed + (size_t)e * H * (K / 2);
            scl = static_cast<const uint8_t*>(d.dn_scales) + (size_t)e * H * (K / 16);
            ts = __ldg(d.dn_tscale + e);
            src = h;
        } else {
            const int it = item - items_r;
            const int pi = it / rb_n;
            first = kPass * pi;
            n = min(kPass, T - first);
            list = nullptr;
            rb = it - pi * rb_n;
            K = d.Is;
            codes = d.sh_dn_packed;
            scl = static_cast<const uint8_t*>(d.sh_dn_scales);
            ts = __ldg(d.sh_dn_tscale);
            src = hs;
        }
        auto hrow = [&](int r) { return list ? list[r] : first + r; };
        auto hidx = [&](int r) { return list ? list[r] : T * k + first + r; };
        const int nr = rb * (TILES * kDnRows) + 16 * warp + (int)g;
        const uint8_t* c0p = codes + (size_t)nr * (K / 2) + 32 * q;
        const uint8_t* c1p = codes + (size_t)(nr + 8) * (K / 2) + 32 * q;
        const uint8_t* s0p = scl + (size_t)nr * (K / 16) + 4 * q;
        const uint8_t* s1p = scl + (size_t)(nr + 8) * (K / 16) + 4 * q;
        const WChunk c0 = load_chunk(c0p, s0p, 0, pol), c1 = load_chunk(c1p, s1p, 0, pol);
        __syncthreads();
        {   // h rows of the entries, times 2^k_h, as f16
            const int per_row = K >> 2;
            for (int idx = threadIdx.x; idx < n * per_row; idx += kThreads) {
                const int r = idx / per_row, v = idx - r * per_row;
                const float sc = exp2i(row_shift(__ldg(hmax + hidx(r))));
                const float4 f = *reinterpret_cast<const float4*>(src + (size_t)hrow(r) * K + 4 * (size_t)v);
                reinterpret_cast<uint2*>(stage + (size_t)r * K * 2)[swz(v, r)] =
                    make_uint2(f16x2_of(f.x * sc, f.y * sc), f16x2_of(f.z * sc, f.w * sc));
            }
        }
        __syncthreads();
        float acc[TILES][2][4] = {};
        const uint8_t* b0 = stage + (size_t)g * K * 2;
        const uint8_t* b1 = stage + (size_t)(g + 8) * K * 2;
        if constexpr (TILES == 2) {
            k_loop_tiles(acc[0], acc[1], c0p, s0p, c1p, s1p, (uint32_t)(kDnRows * (K / 2)), (uint32_t)(kDnRows * (K / 16)),
                         K >> 8, b0, q, xmask, c0, c1, pol);
        } else {
            if (NBMAX == 2 && n > 8) k_loop<2>(acc[0], c0p, s0p, c1p, s1p, K >> 8, b0, b1, q, xmask, c0, c1, pol);
            else k_loop<1>(acc[0], c0p, s0p, c1p, s1p, K >> 8, b0, b1, q, xmask, c0, c1, pol);
        }
#pragma unroll
        for (int tt = 0; tt < TILES; ++tt) {
            const int nt = nr + tt * kDnRows;
#pragma unroll
            for (int nb = 0; nb < NBMAX; ++nb) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int r = 8 * nb + 2 * (int)q + c;
                    if (r < n) {
                        const float inv = exp2i(-row_shift(__ldg(hmax + hidx(r))));
                        if (list) {
                            const int en = list[r];
                            const float f = inv * wts[en] * ts;
                            P[(size_t)en * H + nt] = acc[tt][nb][c] * f;
                            P[(size_t)en * H + nt + 8] = acc[tt][nb][2 + c] * f;
                        } else {
                            const int t = first + r;
                            const float f = inv * sigmoid_f32(gate_logit[t]) * ts;
                            Ps[(size_t)t * H + nt] = acc[tt][nb][c] * f;
                            Ps[(size_t)t * H + nt + 8] = acc[tt][nb][2 + c] * f;
                        }
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------------ combine
// y[t, n] = bf16( sum_j P[t*k + j, n]  (j = 0..k-1)  + Ps[t, n] ), that order.
__global__ void __launch_bounds__(kThreads)
combine_mt_kernel(const float* __restrict__ P, const float* __restrict__ Ps, int T, int H, int k,
                  const uint16_t* __restrict__ resid, uint16_t* __restrict__ y) {
    const int q4 = H >> 2;
    const int i = blockIdx.x * kThreads + threadIdx.x;
    if (i >= T * q4) return;
    const int t = i / q4, c = i - t * q4;
    float4 v[NVFP4_MAX_TOPK];   // all k loads in flight before the first add
#pragma unroll
    for (int j = 0; j < NVFP4_MAX_TOPK; ++j)
        if (j < k) v[j] = *reinterpret_cast<const float4*>(P + (size_t)(t * k + j) * H + 4 * c);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NVFP4_MAX_TOPK; ++j) {
        if (j < k) { a.x += v[j].x; a.y += v[j].y; a.z += v[j].z; a.w += v[j].w; }
    }
    if (Ps) {
        const float4 v = *reinterpret_cast<const float4*>(Ps + (size_t)t * H + 4 * c);
        a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
    }
    if (resid) {   // the residual stream, added before the one rounding
        const uint2 r = *reinterpret_cast<const uint2*>(resid + (size_t)t * H + 4 * c);
        a.x += bf16lo(r.x); a.y += bf16hi(r.x); a.z += bf16lo(r.y); a.w += bf16hi(r.y);
    }
    uint2 o;
    o.x = (uint32_t)f32_to_bf16(a.x) | ((uint32_t)f32_to_bf16(a.y) << 16);
    o.y = (uint32_t)f32_to_bf16(a.z) | ((uint32_t)f32_to_bf16(a.w) << 16);
    *reinterpret_cast<uint2*>(y + (size_t)t * H + 4 * c) = o;
}

int resident_ctas(const void* fn, size_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem) != cudaSuccess || n < 1) n = 1;
    return n;
}

}  // namespace

bool decode_mma_supported(const moe_layer_desc& d, int T) {
    return d.kind == NVFP4_SCALE_E4M3 && T >= 1 && T <= NVFP4_DECODE_MAX_TOKENS && d.H % 256 == 0 &&
           d.I % 256 == 0 && d.Is % 256 == 0 && d.H <= kMaxDim && d.I <= kMaxDim && d.Is <= kMaxDim;
}

cudaError_t launch_moe_decode_mma(const moe_layer_desc& d, const uint16_t* x, int T, uint16_t* y,
                                  int32_t* ids_out, float* w_out, const LayerWs& ws, const DeviceInfo& dev,
                                  cudaStream_t s, const uint16_t* resid) {
    cudaError_t err;
    const bool shared = d.Is > 0;
    const int passes_shared = (T + kPass - 1) / kPass;
    const int passes_routed_ub = (d.E < T * d.k ? d.E : T * d.k) + T * d.k / kPass;
    float* h = ws.h;
    float* hs = ws.hs;
    uint32_t* xmax = ws.amax;
    uint32_t* hmax = ws.amax + T;
    float* P = ws.part;
    float* Ps = shared ? ws.part + (size_t)T * d.k * d.H : nullptr;
    // up to 8 tokens: every routed pass has at most 8 entries (a token picks an expert at
    // most once), so the expert kernels take one n8 block, fit 64 registers and run four CTAs
    // per SM; the down kernel's items are 256 rows (two tiles per warp). Then every gate/up
    // and down item of a call is resident at once, with no second wave.
    const bool small = T <= 8;
    {   // 1. router GEMV (+ the shared gate's pre-activation), top-k, lists, pass map
        const int rows = d.E + (shared ? 1 : 0);
        const size_t smem = (size_t)(T < kRouterTok ? T : kRouterTok) * d.H * 2;
        err = cudaFuncSetAttribute(router_route_mt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        const int by = (T + kRouterTok - 1) / kRouterTok;
        const long cap = (long)dev.num_sms * resident_ctas((const void*)router_route_mt_kernel, smem);
        int rr = 2;   // rows per CTA: the fewest that keep the grid resident at once
        while (rr < kWarps && (long)((rows + rr - 1) / rr) * by > cap) rr *= 2;
        const dim3 grid((rows + rr - 1) / rr, by);
        router_route_mt_kernel<<<grid, kThreads, smem, s>>>(
            d.router_w, shared ? d.sh_gate_w : nullptr, x, T, d.E, d.H, d.k, rr, ws.logits, ws.gate_logit, ws.ids,
            ws.w, ids_out, w_out, ws.offsets, ws.token_list, ws.active, ws.pass_map, ws.amax, ws.hdr);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    {   // 3. gate/up + SwiGLU
        const void* fn = small ? (const void*)gateup_mt_kernel<1, 4> : (const void*)gateup_mt_kernel<2, 3>;
        const size_t smem = (size_t)(small ? 8 : kPass) * d.H * 2;
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        const long items_ub = (long)passes_routed_ub * (d.I / kGuPairs) +
                              (shared ? (long)passes_shared * (d.Is / kGuPairs) : 0);
        const long cap = (long)dev.num_sms * resident_ctas(fn, smem);
        const int grid = (int)(items_ub < cap ? items_ub : cap);
        if (small)
            gateup_mt_kernel<1, 4><<<grid, kThreads, smem, s>>>(d, x, T, ws.offsets, ws.token_list, ws.active,
                                                                ws.pass_map, xmax, hmax, h, hs);
        else
            gateup_mt_kernel<2, 3><<<grid, kThreads, smem, s>>>(d, x, T, ws.offsets, ws.token_list, ws.active,
                                                                ws.pass_map, xmax, hmax, h, hs);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    {   // 4. down, weighted rows
        const int K = d.I > d.Is ? d.I : d.Is;
        const void* fn = small ? (const void*)down_mt_kernel<1, 4, 2> : (const void*)down_mt_kernel<2, 3, 1>;
        const size_t smem = (size_t)(small ? 8 : kPass) * K * 2;
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        const int rows_item = (small ? 2 : 1) * kDnRows;
        const long items_ub = (long)(passes_routed_ub + (shared ? passes_shared : 0)) * (d.H / rows_item);
        const long cap = (long)dev.num_sms * resident_ctas(fn, smem);
        const int grid = (int)(items_ub < cap ? items_ub : cap);
        if (small)
            down_mt_kernel<1, 4, 2><<<grid, kThreads, smem, s>>>(d, T, ws.offsets, ws.token_list, ws.active,
                                                                 ws.pass_map, ws.w, ws.gate_logit, h, hs, hmax, P, Ps);
        else
            down_mt_kernel<2, 3, 1><<<grid, kThreads, smem, s>>>(d, T, ws.offsets, ws.token_list, ws.active,
                                                                 ws.pass_map, ws.w, ws.gate_logit, h, hs, hmax, P, Ps);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    {   // 5. combine
        const int n = T * (d.H / 4);
        combine_mt_kernel<<<(n + kThreads - 1) / kThreads, kThreads, 0, s>>>(P, Ps, T, d.H, d.k, resid, y);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace nvfp4
