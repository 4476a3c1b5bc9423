// One-launch decode of the MoE layer for a single token (T = 1).
//
// Sources (page title, section):
//  - lynn-engine README, P45 note: the active-MoE path as one native call
//    (hidden, expert ids, routing weights, gate/up and down weights -> out[H]);
//    P28/P29 notes: gate/up + SiLU -> [top_k, I] intermediate, then down +
//    routing-weighted sum; P46 note: a fused-atomic single kernel was slow and
//    drifted, so the combine here has no atomics: every output row is owned by
//    one block and summed in a fixed order (P48 note: non-atomic row ownership).
//  - lynn-engine tutorials index, row 06: softmax over all experts -> top-k ->
//    renormalise; sigmoid-gated shared expert.
//  - Lynn Engine write-up, "CUDA Graph and scheduling": decode is launch-bound
//    (about 1527 launches per token); here the whole layer is one launch.
//
// Structure: a persistent grid of one block per SM, three phases.
//   phase A  router rows (bf16) and shared-expert (gate, up) row pairs, spread
//            over all blocks -> logits[E], gate pre-activation, hs[Is]
//   phase B  every block takes the top-k of the E logits itself; the k*I routed
//            (gate row, up row) pairs are split into contiguous ranges, one per
//            block -> h[k, I]
//   phase C  block b owns output rows [H*b/G, H*(b+1)/G): y[n] = sum_j w_j
//            ts_j D_j[n].h_j + sigmoid(g) ts_s Ds[n].hs
// Values that cross blocks (logits, gate, hs, h) travel as 64-bit words
// (launch tag, fp32 bits) in the workspace: a block polls the words it needs
// until every one carries this launch's tag, so one L2 read both waits and
// delivers the data; there is no separate grid barrier. The tag is
// floor(n / G) + 1 where n counts block starts in the workspace (one atomic per
// block, overlapped with the activation load). Polls are bounded in time. The
// h words are stored in the order phase C keeps them in shared memory, so the
// reader copies them linearly.
//
// All weights move HBM -> shared memory with TMA bulk copies (cp.async.bulk)
// completing on mbarriers, issued by the lanes of one warp in parallel, so
// every byte a block needs is in flight at once. Phase-A weights and the
// shared-expert down rows depend on nothing, so they are requested before
// griddepcontrol.wait: under programmatic dependent launch they stream in while
// the previous kernel on the stream finishes. Phase-B rows arrive in four
// chunks with one mbarrier each, so the dot products run while later chunks
// are still in flight; the routed down rows are requested at the same time.
//
// The kernel runs each phase once per launch, so its instruction footprint
// decides how much time goes to instruction fetch: the dot products are shared,
// non-inlined device functions and the copy descriptors are computed by small
// loops, keeping the code within the SM instruction cache across launches.
#include <atomic>

#include "common.cuh"
#include "kernels.cuh"

namespace nvfp4 {

namespace {

constexpr int kFThreads = 512;
constexpr int kFWarps = kFThreads / 32;
constexpr int kChunks = 4;            // phase-B copy chunks (one mbarrier each)
constexpr int kMaxPairs = 8;          // h words per thread / 2: k*I + Is <= 2 * kMaxPairs * kFThreads

struct FusedParams {
    moe_layer_desc d;
    const uint16_t* x;
    uint16_t* y;
    int32_t* ids_out;
    float* w_out;
    WsHeader* hdr;
    unsigned long long* words;   // [E + 1] logits and gate, pad to even, [k*I + Is] h and hs
    unsigned long long wait_limit;
    // shared-memory layout (bytes), identical for every block
    uint32_t off_xb, off_lg, off_w, off_d, off_ds, off_part;
    uint32_t dn_stride;   // bytes per expert slot in the packed down region
    uint32_t dns_stride;  // bytes per expert slot in the down-scale region
    // ceil(2^32 / d) for the divisors used on the device (exact for the ranges used)
    unsigned long long mG, mI;
    unsigned long long mG64;   // ceil(2^64 / G)
};

// floor(x / d) given m = ceil(2^32 / d) (a 33-bit value for d = 1); exact whenever x <= 2^32 / d
__device__ __forceinline__ uint32_t fdiv(uint32_t x, unsigned long long m) {
    return (uint32_t)(((unsigned long long)x * m) >> 32);
}

__device__ __forceinline__ void st_word(unsigned long long* p, uint32_t tag, float v) {
    const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ unsigned long long ld_word(const unsigned long long* p) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

__device__ __forceinline__ ulonglong2 ld_word_pair(const unsigned long long* p) {
    ulonglong2 w;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(w.x), "=l"(w.y) : "l"(p) : "memory");
    return w;
}

// Re-read a pair of words until both carry `tag` (bounded); false on timeout.
__device__ __noinline__ bool poll_pair(const unsigned long long* p, uint32_t tag, unsigned long long limit_ns,
                                       ulonglong2* out) {
    const unsigned long long t0 = global_timer_ns();
    ulonglong2 w;
    do {
        w = ld_word_pair(p);
        if ((uint32_t)(w.x >> 32) == tag && (uint32_t)(w.y >> 32) == tag) { *out = w; return true; }
    } while (global_timer_ns() - t0 <= limit_ns);
    *out = w;
    return false;
}

// Position of element e of a K-vector in the segment-interleaved layout used for
// activations in shared memory: float4 chunk c of segment s at float4 index
// c*nseg + s, so the 32 lanes of a warp read 32 consecutive 16-byte words.
__device__ __forceinline__ int il_pos(int e, int nseg) {
    const int e4 = e >> 2;
    return 4 * ((e4 & 7) * nseg + (e4 >> 3)) + (e & 3);
}

template <int KIND>
__device__ __forceinline__ void decode_scale_pair(const uint8_t* srow, int s, float& s0, float& s1) {
    if constexpr (KIND == NVFP4_SCALE_E4M3) {
        const uint32_t raw = *reinterpret_cast<const uint16_t*>(srow + 2 * s);
        s0 = e4m3_to_f32(raw & 0xFF);
        s1 = e4m3_to_f32(raw >> 8);
    } else {
        const uint32_t raw = *reinterpret_cast<const uint32_t*>(srow + 4 * s);
        s0 = f16_bits_to_f32(static_cast<uint16_t>(raw & 0xFFFF));
        s1 = f16_bits_to_f32(static_cast<uint16_t>(raw >> 16));
    }
}

// One 16-byte NVFP4 segment (32 codes, two scale blocks) of a row against 32
// fp32 activations in the interleaved layout: s0 * sum_0..15 + s1 * sum_16..31.
template <int KIND>
__device__ __forceinline__ float seg_dot(const uint8_t* row, const uint8_t* srow, const float4* xv, int nseg,
                                      int s) {
    const uint4 w = reinterpret_cast<const uint4*>(row)[s];
    float s0, s1;
    decode_scale_pair<KIND>(srow, s, s0, s1);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    float p[2] = {0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 a = xv[(2 * q) * nseg + s];
        const float4 b = xv[(2 * q + 1) * nseg + s];
        const float2 v0 = e2m1x2_to_f32x2(words[q]), v1 = e2m1x2_to_f32x2(words[q] >> 8);
        const float2 v2 = e2m1x2_to_f32x2(words[q] >> 16), v3 = e2m1x2_to_f32x2(words[q] >> 24);
        float acc = p[q >> 1];
        acc = fmaf(v0.x, a.x, acc);
        acc = fmaf(v0.y, a.y, acc);
        acc = fmaf(v1.x, a.z, acc);
        acc = fmaf(v1.y, a.w, acc);
        acc = fmaf(v2.x, b.x, acc);
        acc = fmaf(v2.y, b.y, acc);
        acc = fmaf(v3.x, b.z, acc);
        acc = fmaf(v3.y, b.w, acc);
        p[q >> 1] = acc;
    }
    return fmaf(s0, p[0], s1 * p[1]);
}


// Segment s of a gate row and an up row against the same activations (the
// activation loads are shared): (gate, up) partial dot products.
template <int KIND>
__device__ __forceinline__ float2 seg_dot2(const uint8_t* grow, const uint8_t* urow, const uint8_t* gsr,
                                           const uint8_t* usr, const float4* xv, int nseg, int s) {
    const uint4 wg = reinterpret_cast<const uint4*>(grow)[s];
    const uint4 wu = reinterpret_cast<const uint4*>(urow)[s];
    float g0, g1, u0, u1;
    decode_scale_pair<KIND>(gsr, s, g0, g1);
    decode_scale_pair<KIND>(usr, s, u0, u1);
    const uint32_t gw[4] = {wg.x, wg.y, wg.z, wg.w}, uw[4] = {wu.x, wu.y, wu.z, wu.w};
    float pg[2] = {0.f, 0.f}, pu[2] = {0.f, 0.f};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 a = xv[(2 * q) * nseg + s];
        const float4 b = xv[(2 * q + 1) * nseg + s];
        const float xa[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float2 vg = e2m1x2_to_f32x2(gw[q] >> (8 * h)), vu = e2m1x2_to_f32x2(uw[q] >> (8 * h));
            pg[q >> 1] = fmaf(vg.y, xa[2 * h + 1], fmaf(vg.x, xa[2 * h], pg[q >> 1]));
            pu[q >> 1] = fmaf(vu.y, xa[2 * h + 1], fmaf(vu.x, xa[2 * h], pu[q >> 1]));
        }
    }
    return make_float2(fmaf(g0, pg[0], g1 * pg[1]), fmaf(u0, pu[0], u1 * pu[1]));
}

// Warp sums of two values in five shuffles: lane 0 gets sum(a), lane 16 sum(b).
__device__ __forceinline__ float warp_sum2(float a, float b, int lane) {
    const bool lo = lane < 16;
    float m = lo ? a : b;
    m += __shfl_xor_sync(0xffffffffu, lo ? b : a, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m += __shfl_xor_sync(0xffffffffu, m, o);
    return m;
}

// Copy global bytes [begin, end) of `base` (a 16-byte aligned buffer whose length
// is a multiple of 16) into shared memory at dst, widened to 16-byte bounds; the
// data then starts at dst + (begin & 15). Returns the bytes requested.
__device__ __noinline__ uint32_t issue_copy(uint8_t* dst, const uint8_t* base, size_t begin, size_t end,
                                            uint64_t* bar) {
    const size_t b = begin & ~size_t(15), e = (end + 15) & ~size_t(15);
    if (e <= b) return 0;
    bulk_g2s(dst, base + b, (uint32_t)(e - b), bar);
    return (uint32_t)(e - b);
}

__host__ __device__ __forceinline__ uint32_t window_bytes(size_t begin, size_t end) {
    const size_t b = begin & ~size_t(15), e = (end + 15) & ~size_t(15);
    return e > b ? (uint32_t)(e - b) : 0u;
}

__device__ __forceinline__ float bf16_chunk_dot(const uint4 w, const uint4 xv, float acc) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc = fmaf(bf16lo(ww[q]), bf16lo(xx[q]), acc);
        acc = fmaf(bf16hi(ww[q]), bf16hi(xx[q]), acc);
    }
    return acc;
}

// float -> unsigned key with the same order (for the warp max reduction)
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Wait for a copy barrier; on failure record the status.
__device__ __forceinline__ bool copies_done(uint64_t* bar, WsHeader* hdr) {
    const bool ok = mbar_wait_bounded(bar, 0, kDefaultWaitLimit);
    if (!ok) record_status(hdr, NVFP4_ERR_DEVICE_TIMEOUT);
    return ok;
}

template <int KIND>
__global__ void __launch_bounds__(kFThreads, 2) moe_decode_t1_kernel(FusedParams P) {
    extern __shared__ __align__(128) uint8_t fsm[];
    __shared__ uint64_t mbA, mbDS, mbDR, mbB[kChunks];
    __shared__ int s_ids[NVFP4_MAX_TOPK];
    __shared__ float s_coef[NVFP4_MAX_TOPK + 1];   // routing weight x down tensor scale; shared gate
    __shared__ float s_tsg[NVFP4_MAX_TOPK], s_tsu[NVFP4_MAX_TOPK];
    __shared__ uint32_t s_tag;
    __shared__ int s_fail;

    const moe_layer_desc& d = P.d;
    const int H = d.H, E = d.E, k = d.k, I = d.I, Is = d.Is;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int sb = KIND == NVFP4_SCALE_E4M3 ? 1 : 2;
    const int nsegH = H >> 5, nchH = H >> 3, nsegI = I >> 5, nsegS = Is >> 5;
    const int rowH = H / 2, srowH = H / 16 * sb;          // bytes per packed / scale row of K = H
    const int rowI = I / 2, srowI = I / 16 * sb;          // K = I
    const int rowS = Is / 2, srowS = Is / 16 * sb;        // K = Is
    const int total = k * I;
    unsigned long long* w_lg = P.words;                   // E logits, then the gate pre-activation
    unsigned long long* w_h = P.words + ((E + 2) & ~1);   // h (k slots of I) then hs, interleaved order

    float4* xf = reinterpret_cast<float4*>(fsm);                       // [H] fp32, interleaved
    uint4* xb = reinterpret_cast<uint4*>(fsm + P.off_xb);              // [H] bf16
    float* lg = reinterpret_cast<float*>(fsm + P.off_lg);              // [E + 1]
    uint8_t* W = fsm + P.off_w;                                        // phase A / B weights, then h
    uint8_t* D = fsm + P.off_d;                                        // down rows (packed)
    uint8_t* DS = fsm + P.off_ds;                                      // down rows (scale windows)
    float* part = reinterpret_cast<float*>(fsm + P.off_part);          // per-task partial sums

    // ---------------------------------------------------------------- work of this block
    const int nRows = E + (Is > 0 ? 1 : 0);
    const int nR = nRows > c ? (int)fdiv(nRows - 1 - c, P.mG) + 1 : 0;  // router rows c, c+G, ...
    const int cs = G - 1 - c;                                           // shared pairs cs, cs+G, ...
    const int nS = Is > cs ? (int)fdiv(Is - 1 - cs, P.mG) + 1 : 0;
    const int n0 = (int)fdiv(H * c, P.mG), n1 = (int)fdiv(H * (c + 1), P.mG);
    const int nN = n1 - n0;
    // phase-A region: [router rows nR x 2H][pairs: gate row, up row, gate scales, up scales]
    const uint32_t aPair = (uint32_t)nR * 2 * H;
    const uint32_t pairBytes = 2u * (rowH + srowH);
    const uint32_t r_soff = (uint32_t)(((size_t)n0 * srowI) & 15);   // down-scale window offsets
    const uint32_t sh_soff = (uint32_t)(((size_t)n0 * srowS) & 15);

    // ---------------------------------------------------------------- prologue (weights only)
    float sh_tsg = 0.f, sh_tsu = 0.f;
    float sh_tsd = 0.f;
    if (Is > 0) { sh_tsg = __ldg(d.sh_gu_tscale); sh_tsu = __ldg(d.sh_gu_tscale + 1); sh_tsd = __ldg(d.sh_dn_tscale); }
    if (warp == 1 && lane == 0) {
        // the routed tensor scales are read right after the top-k: bring them into L2 now
        prefetch_l2_range(reinterpret_cast<const uint8_t*>(d.gu_tscale), (size_t)E * 8);
        prefetch_l2_range(reinterpret_cast<const uint8_t*>(d.dn_tscale), (size_t)E * 4);
    }
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(&mbA, 1);
            mbar_init(&mbDS, 1);
            mbar_init(&mbDR, 1);
            for (int i = 0; i < kChunks; ++i) mbar_init(&mbB[i], 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(&mbA, (uint32_t)nR * 2 * H + (uint32_t)nS * pairBytes);
            mbar_arrive_expect_tx(&mbDS, Is > 0 && nN > 0 ? (uint32_t)nN * rowS +
                                         window_bytes((size_t)n0 * srowS, (size_t)n1 * srowS) : 0u);
        }
        __syncwarp();
        const uint8_t* gus = static_cast<const uint8_t*>(d.sh_gu_scales);
        for (int i = lane; i < nR + 4 * nS + 2; i += 32) {
            if (i < nR) {
                const int r = c + G * i;
                const uint8_t* row = reinterpret_cast<const uint8_t*>(r < E ? d.router_w + (size_t)r * H : d.sh_gate_w);
                issue_copy(W + (size_t)i * 2 * H, row, 0, 2 * H, &mbA);
            } else if (i < nR + 4 * nS) {
                const int j = (i - nR) >> 2, pt = (i - nR) & 3;
                const size_t row = (size_t)(cs + G * j) + (pt & 1) * Is;     // gate row, or up row
                uint8_t* pr = W + aPair + (size_t)j * pairBytes;     // [gate][up][gate sc][up sc]
                if (pt < 2) issue_copy(pr + (pt & 1) * rowH, d.sh_gu_packed, row * rowH, (row + 1) * rowH, &mbA);
                else issue_copy(pr + 2 * rowH + (pt & 1) * srowH, gus, row * srowH, (row + 1) * srowH, &mbA);
            } else if (Is > 0 && nN > 0) {
                if (i == nR + 4 * nS)
                    issue_copy(D + (size_t)k * P.dn_stride, d.sh_dn_packed, (size_t)n0 * rowS, (size_t)n1 * rowS, &mbDS);
                else
                    issue_copy(DS + (size_t)k * P.dns_stride, static_cast<const uint8_t*>(d.sh_dn_scales),
                               (size_t)n0 * srowS, (size_t)n1 * srowS, &mbDS);
            }
        }
    }
    if (tid == 0) s_fail = 0;

    // everything below may read what the previous kernel on the stream wrote
    asm volatile("griddepcontrol.wait;" ::: "memory");

    unsigned long long nstart = 0;
    if (tid == 0)
        asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], 1;" : "=l"(nstart) : "l"(&P.hdr->barrier) : "memory");
    for (int i = tid; i < nchH; i += kFThreads) {
        const uint4 raw = *reinterpret_cast<const uint4*>(P.x + 8 * (size_t)i);
        xb[i] = raw;
        const int e4 = 2 * i, s = e4 >> 3, cc = e4 & 7;
        xf[cc * nsegH + s] = make_float4(bf16lo(raw.x), bf16hi(raw.x), bf16lo(raw.y), bf16hi(raw.y));
        xf[(cc + 1) * nsegH + s] = make_float4(bf16lo(raw.z), bf16hi(raw.z), bf16lo(raw.w), bf16hi(raw.w));
    }
    if (tid == 0) {
        unsigned long long q = __umul64hi(nstart, P.mG64);          // nstart / G, corrected below
        if ((q + 1) * (unsigned long long)G <= nstart) ++q;
        if (q * (unsigned long long)G > nstart) --q;
        s_tag = (uint32_t)q + 1u;
    }
    __syncthreads();   // also orders the mbarrier initialisation before any wait
    const uint32_t tag = s_tag;

    // ---------------------------------------------------------------- phase A
    // one warp per router row (lanes over its chunks of 8 bf16) and one per shared-expert
    // (gate, up) row pair (lanes over its segments); each is reduced once
    bool alive = copies_done(&mbA, P.hdr);
    if (alive) {
        for (int task = warp; task < nR + nS; task += kFWarps) {
            if (task < nR) {
                const uint4* wr = reinterpret_cast<const uint4*>(W + (size_t)task * 2 * H);
                float acc = 0.f;
#pragma unroll 1
                for (int ch = lane; ch < nchH; ch += 32) acc = bf16_chunk_dot(wr[ch], xb[ch], acc);
                acc = warp_sum(acc);
                if (lane == 0) st_word(w_lg + c + G * task, tag, acc);   // row E: the gate pre-activation
            } else {
                const int j = task - nR, p = cs + G * j;
                const uint8_t* pr = W + aPair + (size_t)j * pairBytes;
                float ga = 0.f, ua = 0.f;
#pragma unroll 1
                for (int sg = lane; sg < nsegH; sg += 32) {
                    const float2 v = seg_dot2<KIND>(pr, pr + rowH, pr + 2 * rowH, pr + 2 * rowH + srowH, xf, nsegH, sg);
                    ga += v.x;
                    ua += v.y;
                }
                const float m = warp_sum2(ga, ua, lane);
                const float gsum = __shfl_sync(0xffffffffu, m, 0), usum = __shfl_sync(0xffffffffu, m, 16);
                if (lane == 0) st_word(w_h + total + il_pos(p, nsegS), tag, silu_f32(gsum * sh_tsg) * (usum * sh_tsu));
            }
        }
    }
    // the next launch on the stream may start its weight-only prologue now
    asm volatile("griddepcontrol.launch_dependents;");

    // ---------------------------------------------------------------- phase B
    bool ok = alive;
    for (int e = tid; e < nRows && ok; e += kFThreads) {
        unsigned long long w = ld_word(w_lg + e);
        const unsigned long long t0 = global_timer_ns();
        while ((uint32_t)(w >> 32) != tag) {
            if (global_timer_ns() - t0 > P.wait_limit) { ok = false; break; }
            w = ld_word(w_lg + e);
        }
        lg[e] = __uint_as_float((uint32_t)w);
    }
    if (!ok) s_fail = 1;
    __syncthreads();
    if (s_fail) {
        if (tid == 0) record_status(P.hdr, NVFP4_ERR_DEVICE_TIMEOUT);
        copies_done(&mbA, P.hdr);
        copies_done(&mbDS, P.hdr);
        return;
    }
    if (warp == 0) {
        // top-k: k rounds of warp arg-max (max-reduction of order-preserving keys), lower id on
        // ties; lane l holds the keys of experts l, l+32, ... in registers and zeroes the ones it
        // gave away
        uint32_t key[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) key[i] = lane + 32 * i < E ? order_key(lg[lane + 32 * i]) : 0u;
        int my_id = -1;
        float ex = 0.f, vmax = 0.f;
#pragma unroll 1
        for (int j = 0; j < k; ++j) {
            uint32_t best = key[0];
            int bi = 0;
#pragma unroll
            for (int i = 1; i < 8; ++i)
                if (key[i] > best) { best = key[i]; bi = i; }   // strict: the lower id wins ties
            const uint32_t wbest = __reduce_max_sync(0xffffffffu, best);
            const uint32_t e = __reduce_min_sync(0xffffffffu, best == wbest ? (uint32_t)(lane + 32 * bi) : 0xffffffffu);
            if ((int)(e & 31) == lane) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i == bi) key[i] = 0u;
            }
            const float v = key_value(wbest);
            if (j == 0) vmax = v;
            if (lane == j) { my_id = (int)e; ex = __expf(v - vmax); }
        }
        const float sum = warp_sum(lane < k ? ex : 0.f);
        if (lane < k) {
            s_ids[lane] = my_id;
            const float wj = __fdividef(ex, sum);
            s_coef[lane] = wj;
            if (c == 0) {
                if (P.ids_out) P.ids_out[lane] = my_id;
                if (P.w_out) P.w_out[lane] = wj;
            }
        }
        if (lane == 0 && Is > 0) s_coef[k] = sigmoid_f32(lg[E]) * sh_tsd;
    }
    __syncthreads();

    const int q0 = (int)fdiv(total * c, P.mG), q1 = (int)fdiv(total * (c + 1), P.mG);
    const int nq = q1 - q0;
    // phase-B region: [gate packed nq][up packed nq][gate scales nq][up scales nq]
    const uint32_t bUP = (uint32_t)nq * rowH, bGS = 2u * nq * rowH, bUS = bGS + (uint32_t)nq * srowH;
    float r_tsg = 0.f, r_tsu = 0.f, r_tsd = 0.f;   // warp 1 lane j: tensor scales of slot j's expert
    if (warp == 0) {
        // chunk ch holds local rows [nq*ch/4, nq*(ch+1)/4), at most two expert slots ("pieces");
        // lane = ch*8 + piece*4 + part issues one contiguous copy of the piece's rows
        if (lane < kChunks)
            mbar_arrive_expect_tx(&mbB[lane], (uint32_t)(nq * (lane + 1) / kChunks - nq * lane / kChunks) * pairBytes);
        __syncwarp();
        const int ch = lane >> 3, piece = (lane >> 2) & 1, pt = lane & 3;
        const int qa = q0 + nq * ch / kChunks, qb = q0 + nq * (ch + 1) / kChunks;
        if (ch < kChunks && qb > qa) {
            const int ja = (int)fdiv(qa, P.mI);
            const int qs = piece == 0 ? qa : (ja + 1) * I;          // first row of this piece
            const int qe = piece == 0 ? min(qb, (ja + 1) * I) : qb;
            if (qe > qs) {
                const int j = (int)fdiv(qs, P.mI), r0 = qs - q0;
                const size_t row = (size_t)s_ids[j] * 2 * I + (qs - j * I) + (pt & 1) * I;   // first gate / up row
                const size_t nr = (size_t)(qe - qs);
                if (pt < 2) issue_copy(W + (pt ? bUP : 0u) + (size_t)r0 * rowH, d.gu_packed, row * rowH, (row + nr) * rowH, &mbB[ch]);
                else issue_copy(W + (pt == 3 ? bUS : bGS) + (size_t)r0 * srowH, static_cast<const uint8_t*>(d.gu_scales),
                                row * srowH, (row + nr) * srowH, &mbB[ch]);
            }
        }
    } else if (warp == 1) {
        // this block's down rows of the k routed experts (read in phase C)
        if (lane == 0)
            mbar_arrive_expect_tx(&mbDR, nN > 0 ? (uint32_t)k * ((uint32_t)nN * rowI +
                                                  window_bytes((size_t)n0 * srowI, (size_t)n1 * srowI)) : 0u);
        __syncwarp();
        if (lane < 2 * k && nN > 0) {
            const int j = lane >> 1;
            const size_t rb = (size_t)s_ids[j] * H;
            if ((lane & 1) == 0)
                issue_copy(D + (size_t)j * P.dn_stride, d.dn_packed, (rb + n0) * rowI, (rb + n1) * rowI, &mbDR);
            else
                issue_copy(DS + (size_t)j * P.dns_stride, static_cast<const uint8_t*>(d.dn_scales),
                           (rb + n0) * srowI, (rb + n1) * srowI, &mbDR);
        }
        if (lane < k) {   // consumed only after the phase-B dot products
            const int e = s_ids[lane];
            r_tsg = __ldg(d.gu_tscale + 2 * e);
            r_tsu = __ldg(d.gu_tscale + 2 * e + 1);
            r_tsd = __ldg(d.dn_tscale + e);
        }
    }

    // one warp per (gate, up) row pair, in chunk order: lane l takes segments l, l + 32,
    // ...; gate and up share the activation loads and are reduced together
    for (int r = warp; r < nq; r += kFWarps) {
        int ch = 0;
        while (ch + 1 < kChunks && r >= nq * (ch + 1) / kChunks) ++ch;
        alive = mbar_wait_bounded(&mbB[ch], 0, kDefaultWaitLimit) && alive;
        float ga = 0.f, ua = 0.f;
#pragma unroll 1
        for (int sg = lane; sg < nsegH; sg += 32) {
            const float2 v = seg_dot2<KIND>(W + (size_t)r * rowH, W + bUP + (size_t)r * rowH, W + bGS + (size_t)r * srowH,
                                            W + bUS + (size_t)r * srowH, xf, nsegH, sg);
            ga += v.x;
            ua += v.y;
        }
        const float m = warp_sum2(ga, ua, lane);
        if ((lane & 15) == 0) part[2 * r + (lane >> 4)] = m;
    }
    if (!alive) s_fail = 1;
    if (warp == 1 && lane < k) {
        s_tsg[lane] = r_tsg;
        s_tsu[lane] = r_tsu;
        s_coef[lane] *= r_tsd;
    }
    __syncthreads();
    if (!s_fail && tid < nq) {
        const float ga = part[2 * tid], ua = part[2 * tid + 1];
        const int q = q0 + tid, j = (int)fdiv(q, P.mI);
        st_word(w_h + j * I + il_pos(q - j * I, nsegI), tag, silu_f32(ga * s_tsg[j]) * (ua * s_tsu[j]));
    }

    // ---------------------------------------------------------------- phase C
    // copy the h words (already in the interleaved order) into shared memory: every
    // read of a thread is in flight before the first tag check
    float* hf = reinterpret_cast<float*>(W);
    {
        const int npair = (total + Is) >> 1;
        ok = !s_fail;
        if (ok) {
            ulonglong2 v[kMaxPairs];
#pragma unroll
            for (int u = 0; u < kMaxPairs; ++u)
                if (tid + u * kFThreads < npair) v[u] = ld_word_pair(w_h + 2 * (tid + u * kFThreads));
#pragma unroll
            for (int u = 0; u < kMaxPairs; ++u) {
                const int pi = tid + u * kFThreads;
                if (pi < npair) {
                    ulonglong2 w = v[u];
                    if ((uint32_t)(w.x >> 32) != tag || (uint32_t)(w.y >> 32) != tag)
                        ok = poll_pair(w_h + 2 * pi, tag, P.wait_limit, &w) && ok;
                    reinterpret_cast<float2*>(hf)[pi] = make_float2(__uint_as_float((uint32_t)w.x), __uint_as_float((uint32_t)w.y));
                }
            }
        }
        if (!ok) s_fail = 1;
    }
    __syncthreads();
    if (s_fail || !copies_done(&mbDS, P.hdr) || !copies_done(&mbDR, P.hdr)) {
        if (tid == 0) record_status(P.hdr, NVFP4_ERR_DEVICE_TIMEOUT);
        for (int i = 0; i < kChunks; ++i) mbar_wait_bounded(&mbB[i], 0, kDefaultWaitLimit);
        mbar_wait_bounded(&mbDS, 0, kDefaultWaitLimit);
        mbar_wait_bounded(&mbDR, 0, kDefaultWaitLimit);
        return;
    }
    {
        // one warp per output row nl: lane l takes the (slot, segment) pairs l, l + 32, ...
        // (slot k is the shared expert), accumulates all their weighted dot products and
        // the warp is reduced once
        const float4* hsm = reinterpret_cast<const float4*>(W);
        const int work = k * nsegI + nsegS;
        for (int nl = warp; nl < nN; nl += kFWarps) {
            float acc = 0.f;
#pragma unroll 1
            for (int p = lane; p < work; p += 32) {
                int j = 0, sg = p;
                while (j < k && sg >= nsegI) { sg -= nsegI; ++j; }
                const bool sh = j == k;
                const uint8_t* row = D + (size_t)j * P.dn_stride + (size_t)nl * (sh ? rowS : rowI);
                const uint8_t* srow = DS + (size_t)j * P.dns_stride + (sh ? sh_soff + (size_t)nl * srowS
                                                                          : r_soff + (size_t)nl * srowI);
                acc = fmaf(s_coef[j], seg_dot<KIND>(row, srow, hsm + j * (I >> 2), sh ? nsegS : nsegI, sg), acc);
            }
            acc = warp_sum(acc);
            if (lane == 0) P.y[n0 + nl] = f32_to_bf16(acc);
        }
    }
}

struct FusedLayout {
    uint32_t off_xb, off_lg, off_w, off_d, off_ds, off_part, total;
    uint32_t dn_stride, dns_stride;
};

uint32_t up16(size_t v) { return (uint32_t)((v + 15) & ~size_t(15)); }

// Shared-memory plan sized for the block with the most work.
FusedLayout fused_layout(const moe_layer_desc& d, int G) {
    const size_t sb = d.kind == NVFP4_SCALE_E4M3 ? 1 : 2;
    const size_t H = d.H, I = d.I, Is = d.Is, k = d.k;
    const size_t nRows = d.E + (Is > 0 ? 1 : 0);
    const size_t nR = (nRows + G - 1) / G, nS = (Is + G - 1) / G;
    const size_t nq = (k * I + G - 1) / G;     // max of q1 - q0 over blocks
    const size_t nN = (H + G - 1) / G;         // max of n1 - n0 over blocks
    const size_t rowH = H / 2, srowH = H / 16 * sb;
    const size_t phaseA = nR * 2 * H + nS * 2 * (rowH + srowH);
    const size_t phaseB = nq * 2 * (rowH + srowH);
    const size_t hbytes = (k * I + Is) * 4;
    size_t w = phaseA > phaseB ? phaseA : phaseB;
    if (hbytes > w) w = hbytes;
    const size_t Im = I > Is ? I : Is;
    FusedLayout L;
    L.dn_stride = up16(nN * (Im / 2));
    L.dns_stride = up16(nN * (Im / 16 * sb) + 32);
    size_t off = up16(H * 4);
    L.off_xb = (uint32_t)off; off += up16(H * 2);
    L.off_lg = (uint32_t)off; off += up16(nRows * 4);
    L.off_w = (uint32_t)off; off += up16(w);
    L.off_d = (uint32_t)off; off += (size_t)L.dn_stride * (k + 1);
    L.off_ds = (uint32_t)off; off += (size_t)L.dns_stride * (k + 1);
    // phase-B (gate, up) sums of the block's row pairs
    const size_t np = 2 * nq;
    L.off_part = (uint32_t)off; off += up16(np * 4);
    L.total = (uint32_t)off;
    return L;
}

}  // namespace

bool fused_decode_supported(const moe_layer_desc& d, int T, const DeviceInfo& dev) {
    return T == 1 && d.H % 256 == 0 && d.H <= 2048 && d.k * d.I + d.Is <= 2 * kMaxPairs * kFThreads &&
           fused_layout(d, dev.num_sms).total <= dev.smem_optin;
}

cudaError_t launch_moe_decode_fused(const moe_layer_desc& d, const uint16_t* x, uint16_t* y,
                                    int32_t* ids_out, float* w_out, const LayerWs& ws,
                                    const DeviceInfo& dev, uint64_t wait_limit, cudaStream_t s) {
    const int G = dev.num_sms;
    const FusedLayout L = fused_layout(d, G);
    if (L.total > dev.smem_optin) return cudaErrorInvalidConfiguration;
    FusedParams P;
    P.d = d;
    P.x = x;
    P.y = y;
    P.ids_out = ids_out;
    P.w_out = w_out;
    P.hdr = ws.hdr;
    P.words = ws.words;
    P.wait_limit = wait_limit;
    P.off_xb = L.off_xb;
    P.off_lg = L.off_lg;
    P.off_w = L.off_w;
    P.off_d = L.off_d;
    P.off_ds = L.off_ds;
    P.off_part = L.off_part;
    P.dn_stride = L.dn_stride;
    P.dns_stride = L.dns_stride;
    auto magic = [](uint32_t dv) { return ((1ull << 32) + dv - 1) / dv; };
    P.mG = magic(G);
    P.mI = magic(d.I);
    P.mG64 = ~0ull / (unsigned long long)G + 1ull;
    auto kern = d.kind == NVFP4_SCALE_E4M3 ? moe_decode_t1_kernel<NVFP4_SCALE_E4M3>
                                           : moe_decode_t1_kernel<NVFP4_SCALE_FP16>;
    // raise the dynamic shared-memory limit once per (device, kernel, size); no
    // runtime calls besides the launch on the steady-state path
    static std::atomic<uint32_t> set_bytes[2][64];
    const int ki = d.kind == NVFP4_SCALE_E4M3 ? 0 : 1;
    const int dv = dev.device < 64 ? dev.device : 63;
    if (set_bytes[ki][dv].load(std::memory_order_relaxed) < L.total) {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
        if (err != cudaSuccess) return err;
        set_bytes[ki][dv].store(L.total, std::memory_order_relaxed);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace nvfp4
