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
//  - Lynn Engine write-up, "CUDA Graph and scheduling": decode is launch-bound;
//    here the whole layer is one launch.
//
// A persistent grid of one CTA per SM: 16 compute warps and one copy warp. Every
// CTA owns contiguous ranges of each weight stream, so each stream is a handful of
// large TMA bulk copies (cp.async.bulk, completing on mbarriers):
//   router rows    [(E+1)c/G, (E+1)(c+1)/G)   (row E = the shared gate vector)
//   shared pairs   [Is c/G, Is (c+1)/G)        (gate row, up row of the shared expert)
//   routed pairs   [kI c/G, kI (c+1)/G)        (pair q = slot q / I, row q % I)
//   output rows    [H c/G, H (c+1)/G)          (the down rows of every slot)
//
// Timeline of a CTA:
//   before griddepcontrol.wait  the router rows, the shared pairs and the shared down
//                               rows are requested (they depend on nothing the previous
//                               kernel writes); under programmatic dependent launch they
//                               stream in while that kernel finishes
//   x                           staged raw (bf16, for the router) and as f16 times the
//                               power of two 2^sx that puts max|x| in [2^14, 2^15)
//   router rows                 bf16 dot products -> logit words (tag, value)
//   shared pairs                hs words, computed while the other CTAs' logits arrive
//   top-k                       every CTA gathers the E logits and takes the top-k itself
//   routed copies               the CTA's routed pairs (2 chunks, one mbarrier each) and
//                               its down rows of the k routed experts
//   routed pairs                one warp per (gate, up) pair as its chunk lands -> h words
//   h                           every CTA gathers the k*I + Is words, scales each slot by
//                               a power of two into f16
//   down                        one warp per output row: sum over the k + 1 slots in a
//                               fixed order, one bf16 rounding
//
// Values that cross CTAs travel as tagged words: logits as 64-bit (tag << 32 | fp32 bits),
// SwiGLU intermediates as 32-bit (16-bit tag << 16 | bf16 bits), read four per 16-byte load
// (every CTA reads all k*I + Is of them, so the L2 request count is what this exchange
// costs). A reader re-reads a word until it carries this launch's tag, so one L2 read both
// waits and delivers the value; there is no separate grid barrier. The tag is floor(n / G)
// + 1 where n counts CTA starts in the workspace header (one atomic per CTA). Every poll
// is bounded in time; a poll that runs out records NVFP4_ERR_DEVICE_TIMEOUT, the CTA
// drains its copies in flight and returns.
//
// Dot products: cvt.rn.f16x2.e2m1x2 expands two codes into an exact f16 pair and
// fma.rn.f32.f16 multiplies each with its f16 activation and accumulates in fp32; each
// 16-element partial is multiplied by its block scale (exact decode) in fp32. The
// activation side is exact for x (bf16 -> f16 after a power-of-two scale); the SwiGLU
// intermediate h is rounded once to bf16 when it is published (relative error 2^-9 per
// element, the activation type and the prefill path's rounding) and then converted exactly
// to f16 after a power-of-two scale per slot for the down pass.
#include <atomic>

#include "common.cuh"
#include "kernels.cuh"
#include "t1_device.cuh"

namespace nvfp4 {

namespace {

constexpr int kW = 16;                    // compute warps
constexpr int kThr = (kW + 1) * 32;       // + the copy warp
constexpr int kCopyWarp = kW;
constexpr int kChunks = 2;                // routed-pair copy chunks (one mbarrier each; 2 measured
                                          // faster than 1 or 4: fewer, larger bulk copies, and the
                                          // first half of the pairs starts while the second lands)
static_assert(kChunks >= 1 && kChunks * 8 <= 32, "the copy warp gives each chunk 8 lanes");
constexpr int kSlots = NVFP4_MAX_TOPK + 1;

struct T1Params {
    moe_layer_desc d;
    const uint16_t* x;
    uint16_t* y;
    int32_t* ids_out;
    float* w_out;
    WsHeader* hdr;
    unsigned long long* words;    // [E + 1] logits and gate, then [k*I + Is] h and hs
    unsigned long long wait_limit;
    const uint16_t* norm_w;       // nullable: x = bf16(RMSNorm_(1+w)(input)) first
    float eps;
    const uint16_t* resid;        // nullable: y = bf16(resid + layer)
    // shared-memory layout (bytes), identical for every CTA
    uint32_t o_xb, o_x16, o_lg, o_rt, o_sg, o_gu, o_dn, o_dns, o_h16;
    uint32_t sg_reg;      // bytes of one region of the shared-pair area (codes)
    uint32_t sg_sreg;     // ... (scales)
    uint32_t gu_reg;      // bytes of one region of the routed-pair area (codes)
    uint32_t gu_sreg;     // ... (scales)
    uint32_t dn_row;      // bytes of one down row over all slots: (k*I + Is) / 2
    uint32_t dn_srow;     // ... of its scales: (k*I + Is) / 16 * scale bytes
    unsigned long long tag_step;   // added by each CTA: tag_period / G
    unsigned long long tag_period;
    unsigned long long mP64;       // ceil(2^64 / tag_period)
};

template <int KIND>
__global__ void __launch_bounds__(kThr, 1) moe_decode_t1_kernel(T1Params P) {
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ uint64_t mbA, mbB[kChunks];
    __shared__ int s_ids[NVFP4_MAX_TOPK];
    __shared__ float s_coef[kSlots];       // slot weight times the down tensor scale
    __shared__ float s_tsg[kSlots], s_tsu[kSlots];
    __shared__ uint32_t s_hm;              // max over slots of |h| |coef| (fp32 bits)
    __shared__ uint32_t s_xmax, s_tag;
    __shared__ int s_fail;
    __shared__ float s_ss[kThr / 32];
    __shared__ float s_red[2][kW][8];       // routed-pair sums of each warp, per batch parity
    __shared__ float s_tg[NVFP4_MAX_EXPERTS * 2], s_td[NVFP4_MAX_EXPERTS];   // every expert's tensor scales

    const moe_layer_desc& d = P.d;
    const int H = d.H, E = d.E, k = d.k, I = d.I, Is = d.Is;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int sb = KIND == NVFP4_SCALE_E4M3 ? 1 : 2;
    const uint32_t rowH = H / 2, srowH = H / 16 * sb;     // bytes of a code / scale row of K = H
    const int nsegH = H >> 5, nunitH = H >> 3;
    const int nR0 = (int)((long long)(E + 1) * c / G), nR1 = (int)((long long)(E + 1) * (c + 1) / G);
    const int s0 = (int)((long long)Is * c / G), s1 = (int)((long long)Is * (c + 1) / G);
    const int q0 = (int)((long long)k * I * c / G), q1 = (int)((long long)k * I * (c + 1) / G);
    const int n0 = (int)((long long)H * c / G), n1 = (int)((long long)H * (c + 1) / G);
    const int nR = nR1 - nR0, nS = s1 - s0, nq = q1 - q0, nN = n1 - n0;
    const int total = k * I;
    // every word is written to kWordReplicas copies and CTA c reads copy c % kWordReplicas:
    // the exchanged lines are read by every CTA, and one L2 line read by all 152 CTAs
    // serialises their requests, so each copy is read by only ~G / kWordReplicas of them
    const size_t lg_stride = t1_logit_stride(d), h_stride = t1_h_stride(d);
    const int rep = c % kWordReplicas;
    unsigned long long* w_lg_all = P.words;
    uint32_t* w_h_all = reinterpret_cast<uint32_t*>(P.words + kWordReplicas * lg_stride);
    const unsigned long long* w_lg = w_lg_all + rep * lg_stride;     // this CTA's copy
    const uint32_t* w_h = w_h_all + rep * h_stride;

    uint16_t* xb = reinterpret_cast<uint16_t*>(sm + P.o_xb);
    uint4* x16 = reinterpret_cast<uint4*>(sm + P.o_x16);
    float* lg = reinterpret_cast<float*>(sm + P.o_lg);
    uint8_t* RT = sm + P.o_rt;
    uint8_t* SG = sm + P.o_sg;                // regions: gate codes, up codes, gate scales, up scales
    uint8_t* GU = sm + P.o_gu;                // same four regions for the routed pairs
    // down rows of the CTA's outputs over all k + 1 slots: row nl holds slot j's codes at
    // j * I/2 (shared slot at k * I/2), its scales likewise in the scale region
    uint8_t* DN = sm + P.o_dn;
    uint8_t* DNs = sm + P.o_dns;
    uint4* h16 = reinterpret_cast<uint4*>(sm + P.o_h16);

    // ------------------------------------------------------------------ prologue
    if (tid == 0) {
        mbar_init(&mbA, 1);
        for (int i = 0; i < kChunks; ++i) mbar_init(&mbB[i], 1);
        fence_mbar_init();
        s_fail = 0;
        s_xmax = 0u;
        s_hm = 0u;
    }
    __syncthreads();
    const uint8_t* sh_gu = d.sh_gu_packed;
    const uint8_t* sh_gus = static_cast<const uint8_t*>(d.sh_gu_scales);
    const uint32_t rowS = Is / 2, srowS = Is / 16 * sb;
    if (warp == kCopyWarp) {
        // weight-only copies: router rows, shared pairs, shared down rows
        if (lane == 0) {
            const uint32_t a = (uint32_t)(min(nR1, E) - min(nR0, E)) * 2u * H + (nR1 > E ? 2u * H : 0u) +
                               (uint32_t)nS * 2u * (rowH + srowH);
            mbar_arrive_expect_tx(&mbA, a);
        }
        __syncwarp();
        const int rE = min(nR1, E) - min(nR0, E);   // router rows of this CTA below E
        if (lane == 0 && rE > 0)
            copy_range(RT, reinterpret_cast<const uint8_t*>(d.router_w + (size_t)nR0 * H), (uint32_t)rE * 2u * H, &mbA);
        if (lane == 1 && nR1 > E)
            copy_range(RT + (size_t)rE * 2 * H, reinterpret_cast<const uint8_t*>(d.sh_gate_w), 2u * H, &mbA);
        if (nS > 0) {
            if (lane == 2) copy_range(SG, sh_gu + (size_t)s0 * rowH, (uint32_t)nS * rowH, &mbA);
            if (lane == 3) copy_range(SG + P.sg_reg, sh_gu + (size_t)(Is + s0) * rowH, (uint32_t)nS * rowH, &mbA);
            if (lane == 4) copy_range(SG + 2 * P.sg_reg, sh_gus + (size_t)s0 * srowH, (uint32_t)nS * srowH, &mbA);
            if (lane == 5)
                copy_range(SG + 2 * P.sg_reg + P.sg_sreg, sh_gus + (size_t)(Is + s0) * srowH, (uint32_t)nS * srowH, &mbA);
        }
    } else if (Is > 0) {
        // the shared expert's down rows of this CTA's outputs, 16 bytes per cp.async, into
        // the shared slot of each row
        const int pr = (int)(rowS >> 4), ps = (int)(srowS >> 4);
        const uint32_t rowI_ = I / 2, srowI_ = I / 16 * sb;
        for (int i = tid; i < nN * (pr + ps); i += kW * 32) {
            if (i < nN * pr) {
                const int nl = i / pr, q = i - nl * pr;
                cp_async16(DN + (size_t)nl * P.dn_row + (size_t)k * rowI_ + 16 * q,
                           d.sh_dn_packed + (size_t)n0 * rowS + 16 * (size_t)i);
            } else {
                const int r = i - nN * pr, nl = r / ps, q = r - nl * ps;
                cp_async16(DNs + (size_t)nl * P.dn_srow + (size_t)k * srowI_ + 16 * q,
                           static_cast<const uint8_t*>(d.sh_dn_scales) + (size_t)n0 * srowS + 16 * (size_t)r);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }

    // every expert's tensor scales (read after the top-k): requested now into registers, written
    // to shared memory after the x staging, so no thread waits for them
    float tsv[3] = {0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const int i = tid + u * kThr;
        if (i < 2 * E) tsv[u] = __ldg(d.gu_tscale + i);
        else if (i < 3 * E) tsv[u] = __ldg(d.dn_tscale + (i - 2 * E));
    }
    float sh_tsg = 0.f, sh_tsu = 0.f, sh_tsd = 0.f;
    if (Is > 0) {
        sh_tsg = __ldg(d.sh_gu_tscale);
        sh_tsu = __ldg(d.sh_gu_tscale + 1);
        sh_tsd = __ldg(d.sh_dn_tscale);
    }

    // this launch's tag. The atomic is issued before griddepcontrol.wait (its latency hides
    // behind the wait and the x load): a dependent launch starts only after every CTA of
    // this one has passed launch_dependents, which comes after this atomic, so the counts
    // of consecutive launches never interleave
    unsigned long long n_start = 0;
    if (tid == 0)
        asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], %2;"
                     : "=l"(n_start) : "l"(&P.hdr->barrier), "l"(P.tag_step) : "memory");

    // everything below may read what the previous kernel on the stream wrote
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // x: raw bf16 for the router, and max |x| for the f16 copy
    uint4 xv = make_uint4(0, 0, 0, 0);
    if (tid < nunitH) xv = reinterpret_cast<const uint4*>(P.x)[tid];
    if (tid == 0) {   // the atomic's result is first used here, after the wait and the x load
        unsigned long long q = __umul64hi(n_start, P.mP64);    // n / period, corrected below
        if ((q + 1) * P.tag_period <= n_start) ++q;
        if (q * P.tag_period > n_start) --q;
        s_tag = (uint32_t)q + 1u;
    }
    if (P.norm_w) {
        // pre-MoE RMSNorm (1 + w) x / sqrt(mean(x^2) + eps): squares summed per thread, per
        // warp by shuffles, then over the warps in a fixed order; rounded once to bf16
        float ss = 0.f;
        {
            const uint32_t ww[4] = {xv.x, xv.y, xv.z, xv.w};
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
        for (int i = 0; i < kThr / 32; ++i) tot += s_ss[i];
        const float r = 1.0f / sqrtf(tot / (float)H + P.eps);
        if (tid < nunitH) {
            const uint4 wv = reinterpret_cast<const uint4*>(P.norm_w)[tid];
            const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w}, nw[4] = {wv.x, wv.y, wv.z, wv.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float lo = bf16lo(xx[q]) * r * (1.0f + bf16lo(nw[q]));
                const float hi = bf16hi(xx[q]) * r * (1.0f + bf16hi(nw[q]));
                o[q] = (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
            }
            xv = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    if (tid < nunitH) {
        reinterpret_cast<uint4*>(xb)[tid] = xv;
        const uint32_t ww[4] = {xv.x, xv.y, xv.z, xv.w};
        uint32_t m = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) m = max(m, max(ww[q] & 0x7FFFu, (ww[q] >> 16) & 0x7FFFu));
        m = __reduce_max_sync(__activemask(), m);
        if (lane == 0) atomicMax(&s_xmax, m << 16);     // as fp32 bits
    }
    __syncthreads();
    const uint32_t tag = s_tag, tag16 = tag16_of(tag);
    const int sx = pow2_shift(s_xmax);
    if (tid < nunitH) {
        const float sc = exp2_int(sx);
        uint4 o;
        o.x = to_f16x2(bf16lo(xv.x) * sc, bf16hi(xv.x) * sc);
        o.y = to_f16x2(bf16lo(xv.y) * sc, bf16hi(xv.y) * sc);
        o.z = to_f16x2(bf16lo(xv.z) * sc, bf16hi(xv.z) * sc);
        o.w = to_f16x2(bf16lo(xv.w) * sc, bf16hi(xv.w) * sc);
        x16[(tid & 3) * nsegH + (tid >> 2)] = o;
    }
    __syncthreads();
    const float inv_x = exp2_int(-sx);

    bool ok = true;
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const int i = tid + u * kThr;
        if (i < 2 * E) s_tg[i] = tsv[u];
        else if (i < 3 * E) s_td[i - 2 * E] = tsv[u];
    }
    if (warp < kW) {
        // router rows (warps 0 .. nR-1) and shared pairs (the other warps)
        ok = mbar_wait_bounded(&mbA, 0, kDefaultWaitLimit);
        if (ok) {
            for (int t = warp; t < nR + nS; t += kW) {
                if (t < nR) {
                    const uint4* wr = reinterpret_cast<const uint4*>(RT + (size_t)t * 2 * H);
                    const uint4* xr = reinterpret_cast<const uint4*>(xb);
                    float acc = 0.f;
#pragma unroll 4
                    for (int ch = lane; ch < nunitH; ch += 32) acc = bf16_dot8(wr[ch], xr[ch], acc);
                    acc = warp_sum(acc);
                    if (lane < kWordReplicas) st_word(w_lg_all + lane * lg_stride + nR0 + t, tag, acc);
                } else {
                    const int j = t - nR;
                    const float m = pair_dot<KIND>(SG + (size_t)j * rowH, SG + P.sg_reg + (size_t)j * rowH,
                                                   SG + 2 * P.sg_reg + (size_t)j * srowH,
                                                   SG + 2 * P.sg_reg + P.sg_sreg + (size_t)j * srowH, x16, nsegH, lane);
                    const float gsum = __shfl_sync(0xffffffffu, m, 0), usum = __shfl_sync(0xffffffffu, m, 16);
                    if (lane < kWordReplicas) {
                        const float hv = silu_f32(gsum * inv_x * sh_tsg) * (usum * inv_x * sh_tsu);
                        st_hword(w_h_all + lane * h_stride + total + s0 + j, tag16, hv);
                    }
                }
            }
        }
        asm volatile("griddepcontrol.launch_dependents;");
        // gather the E logits and the gate pre-activation
        if (ok) {
            for (int e = tid; e <= E; e += kW * 32) {
                float v;
                if (!poll_word(w_lg + e, tag, P.wait_limit, &v)) { ok = false; break; }
                lg[e] = v;
            }
        }
    }
    if (warp == kCopyWarp) asm volatile("griddepcontrol.launch_dependents;");
    if (!ok) s_fail = 1;
    __syncthreads();
    if (s_fail) {
        if (tid == 0) record_status(P.hdr, NVFP4_ERR_DEVICE_TIMEOUT);
        if (tid == 0) mbar_wait_bounded(&mbA, 0, kDefaultWaitLimit);
        if (warp < kW) asm volatile("cp.async.wait_all;" ::: "memory");
        return;
    }

    // ------------------------------------------------------------------ top-k
    if (warp == 0) {
        // lane l holds experts 8l .. 8l+7 as 64-bit keys (order key, then 7 - i so that the
        // lower id wins ties), sorted descending in registers by an odd-even merge network;
        // each round the warp takes the largest head (the lowest lane among equal heads
        // holds the lowest id) and the lane that held it drops it
        unsigned long long kk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = 8 * lane + i;
            kk[i] = e < E ? ((unsigned long long)order_key(lg[e]) << 3) | (unsigned)(7 - i) : 0ull;
        }
#define T1_CX(a, b) { const unsigned long long hi_ = max(kk[a], kk[b]), lo_ = min(kk[a], kk[b]); kk[a] = hi_; kk[b] = lo_; }
        T1_CX(0, 1) T1_CX(2, 3) T1_CX(4, 5) T1_CX(6, 7)
        T1_CX(0, 2) T1_CX(1, 3) T1_CX(4, 6) T1_CX(5, 7)
        T1_CX(1, 2) T1_CX(5, 6)
        T1_CX(0, 4) T1_CX(1, 5) T1_CX(2, 6) T1_CX(3, 7)
        T1_CX(2, 4) T1_CX(3, 5)
        T1_CX(1, 2) T1_CX(3, 4) T1_CX(5, 6)
#undef T1_CX
        int my_id = -1;
        float ex = 0.f, vmax = 0.f;
#pragma unroll 1
        for (int j = 0; j < k; ++j) {
            const uint32_t hk = (uint32_t)(kk[0] >> 3);
            const uint32_t wb = __reduce_max_sync(0xffffffffu, hk);
            const int win = __ffs(__ballot_sync(0xffffffffu, hk == wb)) - 1;
            const int e = __shfl_sync(0xffffffffu, 8 * lane + 7 - (int)((uint32_t)kk[0] & 7u), win);
            if (lane == win) {
#pragma unroll
                for (int i = 0; i < 7; ++i) kk[i] = kk[i + 1];
                kk[7] = 0ull;
            }
            const float v = key_value(wb);
            if (j == 0) vmax = v;
            if (lane == j) { my_id = e; ex = __expf(v - vmax); }
        }
        const float sum = warp_sum(lane < k ? ex : 0.f);
        if (lane < k) {
            const float wj = __fdividef(ex, sum);
            s_ids[lane] = my_id;
            s_coef[lane] = wj * s_td[my_id];
            s_tsg[lane] = s_tg[2 * my_id];
            s_tsu[lane] = s_tg[2 * my_id + 1];
            if (c == 0) {
                if (P.ids_out) P.ids_out[lane] = my_id;
                if (P.w_out) P.w_out[lane] = wj;
            }
        }
        if (lane == 0 && Is > 0) s_coef[k] = sigmoid_f32(lg[E]) * sh_tsd;
    }
    __syncthreads();

    // ------------------------------------------------------------------ routed copies
    const uint8_t* gu_p = d.gu_packed;
    const uint8_t* gu_s = static_cast<const uint8_t*>(d.gu_scales);
    const uint32_t rowI = I / 2, srowI = I / 16 * sb;
    if (warp == kCopyWarp) {
        // chunk ch holds local pairs [nq ch / kChunks, nq (ch+1) / kChunks): at most two slots ("pieces");
        // lane = 8 ch + 4 piece + part issues one contiguous copy (gate codes, up codes,
        // gate scales, up scales) of the piece's pairs
        if (lane < kChunks) {
            const int a = nq * lane / kChunks, b = nq * (lane + 1) / kChunks;
            mbar_arrive_expect_tx(&mbB[lane], (uint32_t)(b - a) * 2u * (rowH + srowH));
        }
        __syncwarp();
        {
            const int ch = lane >> 3, piece = (lane >> 2) & 1, part = lane & 3;
            const int qa = q0 + nq * ch / kChunks, qb = q0 + nq * (ch + 1) / kChunks;
            if (ch < kChunks && qb > qa) {   // lanes of chunks past kChunks issue nothing
                const int ja = qa / I;
                const int qs = piece == 0 ? qa : (ja + 1) * I;
                const int qe = piece == 0 ? min(qb, (ja + 1) * I) : qb;
                if (qe > qs) {
                    const int j = qs / I, i0 = qs - j * I, r0 = qs - q0, nr = qe - qs;
                    const size_t grow = (size_t)s_ids[j] * 2 * I + i0 + (part & 1) * I;   // first gate / up row
                    if (part < 2)
                        copy_range(GU + (part ? P.gu_reg : 0u) + (size_t)r0 * rowH, gu_p + grow * rowH,
                                   (uint32_t)nr * rowH, &mbB[ch]);
                    else
                        copy_range(GU + 2 * P.gu_reg + (part == 3 ? P.gu_sreg : 0u) + (size_t)r0 * srowH,
                                   gu_s + grow * srowH, (uint32_t)nr * srowH, &mbB[ch]);
                }
            }
        }
    } else {
        // the k routed experts' down rows of this CTA's output rows, 16 bytes per cp.async from
        // every compute thread: they are read last, and the SM's TMA unit handles one bulk copy
        // at a time, so these small pieces stay off its queue
        {
            const int pr = (int)(rowI >> 4), ps = (int)(srowI >> 4);   // 16-byte pieces per row
            const int per_slot = nN * (pr + ps);
            for (int i = tid; i < k * per_slot; i += kW * 32) {
                const int j = i / per_slot, r = i - j * per_slot;
                const size_t rb = (size_t)s_ids[j] * H + n0;
                if (r < nN * pr) {
                    const int nl = r / pr, q = r - nl * pr;
                    cp_async16(DN + (size_t)nl * P.dn_row + (size_t)j * rowI + 16 * q,
                               d.dn_packed + rb * rowI + 16 * (size_t)r);
                } else {
                    const int r2 = r - nN * pr, nl = r2 / ps, q = r2 - nl * ps;
                    cp_async16(DNs + (size_t)nl * P.dn_srow + (size_t)j * srowI + 16 * q,
                               static_cast<const uint8_t*>(d.dn_scales) + rb * srowI + 16 * (size_t)r2);
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        // ---------------------------------------------------------------- routed pairs
        // lane group g (warps 2g, 2g + 1) takes local pairs g, g + 8, g + 16, ... in batches of
        // four, its lane i the segments i, i + 64, ... of H. A lane holds its x segment in
        // registers across the batch and keeps a gate and an up sum per pair; each warp reduces
        // its 8 sums (warp_sum8), and the group adds its two warps' sums in a fixed order.
        {
            constexpr int kGroups = kW / 2, kBatch = 4;
            const int g = warp >> 1, gi = tid & 63;
            const int npg = nq > g ? (nq - g + kGroups - 1) / kGroups : 0;   // pairs of group g
            const uint8_t* GUs = GU + 2 * P.gu_reg;
            for (int b = 0; b * kBatch < npg; ++b) {
                float v[2 * kBatch];
#pragma unroll
                for (int i = 0; i < 2 * kBatch; ++i) v[i] = 0.f;
                for (int s = gi; s < nsegH; s += 64) {
                    const uint4 u0 = x16[s], u1 = x16[nsegH + s], u2 = x16[2 * nsegH + s], u3 = x16[3 * nsegH + s];
#pragma unroll
                    for (int m = 0; m < kBatch; ++m) {
                        const int n = b * kBatch + m;
                        if (n < npg) {
                            const int r = g + kGroups * n;
                            int ch = 0;
                            while (ch + 1 < kChunks && r >= nq * (ch + 1) / kChunks) ++ch;
                            if (ok && !mbar_wait_bounded(&mbB[ch], 0, kDefaultWaitLimit)) ok = false;
                            if (ok) {
                                float g0, g1, a0, a1;
                                scales2<KIND>(GUs + (size_t)r * srowH, s, g0, g1);
                                scales2<KIND>(GUs + P.gu_sreg + (size_t)r * srowH, s, a0, a1);
                                v[2 * m] += seg_dot_r(reinterpret_cast<const uint4*>(GU + (size_t)r * rowH)[s],
                                                      g0, g1, u0, u1, u2, u3);
                                v[2 * m + 1] += seg_dot_r(
                                    reinterpret_cast<const uint4*>(GU + P.gu_reg + (size_t)r * rowH)[s], a0, a1,
                                    u0, u1, u2, u3);
                            }
                        }
                    }
                }
                const float z = warp_sum8(v, lane);
                if ((lane & 3) == 0) s_red[b & 1][warp][(lane >> 2) & 7] = z;
                named_sync(2 + g, 64);
                if ((warp & 1) == 0 && ok) {
                    // lane = m * kWordReplicas + copy: pair m of the batch, one replica each
                    for (int i = lane; i < kBatch * kWordReplicas; i += 32) {
                        const int m = i / kWordReplicas, cp = i - m * kWordReplicas, n = b * kBatch + m;
                        if (n < npg) {
                            const int q = q0 + g + kGroups * n, j = q / I;
                            const float gs = s_red[b & 1][warp][2 * m] + s_red[b & 1][warp + 1][2 * m];
                            const float us = s_red[b & 1][warp][2 * m + 1] + s_red[b & 1][warp + 1][2 * m + 1];
                            const float hv = silu_f32(gs * inv_x * s_tsg[j]) * (us * inv_x * s_tsu[j]);
                            st_hword(w_h_all + cp * h_stride + q, tag16, hv);
                        }
                    }
                }
            }
        }
        // ---------------------------------------------------------------- gather h
        // every thread reads 8-word units of the k*I + Is words (one 32-byte load each, all in
        // flight), re-reads the units with an untagged word until all carry this launch's
        // tag (bounded), then stages them for the down pass
        constexpr int kMaxU = 2;    // units per thread: (k*I + Is) <= 16 * 512
        const int nh = total + Is, nu = nh >> 3;
        uint4 wa[kMaxU], wb[kMaxU];
#pragma unroll
        for (int u = 0; u < kMaxU; ++u) {
            const int i = tid + u * kW * 32;
            wa[u] = wb[u] = make_uint4(0, 0, 0, 0);
            if (i < nu) ld_hwords8(w_h + 8 * i, wa[u], wb[u]);
        }
        auto ready4 = [&](const uint4 w) {
            return (w.x >> 16) == tag16 && (w.y >> 16) == tag16 && (w.z >> 16) == tag16 && (w.w >> 16) == tag16;
        };
        {
            unsigned long long t0 = 0;
            for (int round = 0; ok; ++round) {
                bool pending = false;
#pragma unroll
                for (int u = 0; u < kMaxU; ++u)
                    if (tid + u * kW * 32 < nu && !(ready4(wa[u]) && ready4(wb[u]))) pending = true;
                if (!pending) break;
                if (round == 0) t0 = global_timer_ns();
                else if (global_timer_ns() - t0 > P.wait_limit) { ok = false; break; }
#pragma unroll
                for (int u = 0; u < kMaxU; ++u) {
                    const int i = tid + u * kW * 32;
                    if (i < nu && !(ready4(wa[u]) && ready4(wb[u]))) ld_hwords8(w_h + 8 * i, wa[u], wb[u]);
                }
            }
        }
        // max of |h| |coef_j| over all slots (a warp's 256 consecutive words lie in one
        // slot: I % 256 == 0)
#pragma unroll
        for (int u = 0; u < kMaxU; ++u) {
            const int base = 8 * (warp * 32 + u * kW * 32);   // first word of this warp's 256
            if (base < nh) {
                const uint4 a = wa[u], b = wb[u];
                uint32_t m = max(max(a.x & 0x7FFFu, a.y & 0x7FFFu), max(a.z & 0x7FFFu, a.w & 0x7FFFu));
                m = max(m, max(max(b.x & 0x7FFFu, b.y & 0x7FFFu), max(b.z & 0x7FFFu, b.w & 0x7FFFu)));
                m = __reduce_max_sync(0xffffffffu, m);
                if (lane == 0)
                    atomicMax(&s_hm, __float_as_uint(__uint_as_float(m << 16) * fabsf(s_coef[base < total ? base / I : k])));
            }
        }
        named_sync(1, kW * 32);
        // coef_j h as f16 times 2^sh (max in [2^14, 2^15)), the k + 1 slots as one vector of
        // nsegT 32-element segments, segment-interleaved; a unit of eight consecutive
        // elements is one 16-byte store
        const int nsegT = nh >> 5;
        const float s2 = exp2_int(pow2_shift(s_hm));
#pragma unroll
        for (int u = 0; u < kMaxU; ++u) {
            const int i = tid + u * kW * 32;
            if (i < nu && ok) {
                const int e0 = 8 * i;
                const float sc = s_coef[e0 < total ? e0 / I : k] * s2;
                const uint4 a = wa[u], b = wb[u];
                const uint4 o = make_uint4(to_f16x2(bf16lo(a.x) * sc, bf16lo(a.y) * sc),
                                           to_f16x2(bf16lo(a.z) * sc, bf16lo(a.w) * sc),
                                           to_f16x2(bf16lo(b.x) * sc, bf16lo(b.y) * sc),
                                           to_f16x2(bf16lo(b.z) * sc, bf16lo(b.w) * sc));
                h16[((e0 >> 3) & 3) * nsegT + (e0 >> 5)] = o;
            }
        }
    }
    if (warp < kW) asm volatile("cp.async.wait_all;" ::: "memory");   // this thread's down-row pieces
    if (!ok) s_fail = 1;
    __syncthreads();
    if (s_fail) {
        if (tid == 0) {
            record_status(P.hdr, NVFP4_ERR_DEVICE_TIMEOUT);
            for (int i = 0; i < kChunks; ++i) mbar_wait_bounded(&mbB[i], 0, kDefaultWaitLimit);
        }
        return;
    }
    // chunks that no warp waited for (a CTA with fewer pairs than warps waits for all)
    if (tid == 0)
        for (int i = 0; i < kChunks; ++i) mbar_wait_bounded(&mbB[i], 0, kDefaultWaitLimit);

    // ------------------------------------------------------------------ down
    if (warp < kW) {
        const int nsegT = (total + Is) >> 5;
        const float inv_h = exp2_int(-pow2_shift(s_hm));
        for (int nl = warp; nl < nN; nl += kW) {
            // lane l sums segments l, l + 32, ... of the row in that order, then the warp is
            // reduced once: a fixed order, no atomics
            const uint8_t* wr = DN + (size_t)nl * P.dn_row;
            const uint8_t* sr = DNs + (size_t)nl * P.dn_srow;
            float acc = 0.f;
#pragma unroll 1
            for (int S = lane; S < nsegT; S += 32) {
                float sa, sb2;
                scales2<KIND>(sr, S, sa, sb2);
                acc += seg_dot<KIND>(reinterpret_cast<const uint4*>(wr)[S], sa, sb2, h16, nsegT, S);
            }
            acc = warp_sum(acc) * inv_h;
            if (lane == 0) {
                if (P.resid) acc += bf16_to_f32(P.resid[n0 + nl]);   // residual stream, before the rounding
                P.y[n0 + nl] = f32_to_bf16(acc);
            }
        }
    }
}

struct T1Layout {
    uint32_t o_xb, o_x16, o_lg, o_rt, o_sg, o_gu, o_dn, o_dns, o_h16, total;
    uint32_t sg_reg, sg_sreg, gu_reg, gu_sreg, dn_row, dn_srow;
};

uint32_t a16(size_t v) { return (uint32_t)((v + 15) & ~size_t(15)); }

T1Layout t1_layout(const moe_layer_desc& d, int G) {
    const size_t sb = d.kind == NVFP4_SCALE_E4M3 ? 1 : 2;
    const size_t H = d.H, I = d.I, Is = d.Is, k = d.k, E = d.E;
    const size_t nR = (E + 1 + G - 1) / G + 1, nS = (Is + G - 1) / G + 1;
    const size_t nq = (k * I + G - 1) / G + 1, nN = (H + G - 1) / G + 1;
    const size_t KT = k * I + Is;             // the k + 1 slots as one vector
    T1Layout L;
    L.sg_reg = a16(nS * (H / 2));
    L.sg_sreg = a16(nS * (H / 16 * sb));
    L.gu_reg = a16(nq * (H / 2));
    L.gu_sreg = a16(nq * (H / 16 * sb));
    L.dn_row = (uint32_t)(KT / 2);
    L.dn_srow = (uint32_t)(KT / 16 * sb);
    size_t off = 0;
    L.o_xb = (uint32_t)off; off += a16(H * 2);
    L.o_x16 = (uint32_t)off; off += a16(H * 2);
    L.o_lg = (uint32_t)off; off += a16((E + 1) * 4);
    L.o_rt = (uint32_t)off; off += a16(nR * H * 2);
    L.o_sg = (uint32_t)off; off += 2 * (size_t)L.sg_reg + 2 * (size_t)L.sg_sreg;
    L.o_gu = (uint32_t)off; off += 2 * (size_t)L.gu_reg + 2 * (size_t)L.gu_sreg;
    L.o_dn = (uint32_t)off; off += a16(nN * (size_t)L.dn_row);
    L.o_dns = (uint32_t)off; off += a16(nN * (size_t)L.dn_srow);
    L.o_h16 = (uint32_t)off; off += a16(KT * 2);
    L.total = (uint32_t)off;
    return L;
}

}  // namespace

namespace {

bool grid_form_supported(const moe_layer_desc& d, int T, const DeviceInfo& dev) {
    const bool dims = d.H % 256 == 0 && d.I % 256 == 0 && (d.Is == 0 || d.Is % 256 == 0) && d.H <= 4096 &&
                      d.I <= 4096 && d.Is <= 4096;
    // h words per thread: (k*I + Is) <= 16 * 512; output rows per CTA fit the slot area
    const bool kinds = d.kind == NVFP4_SCALE_E4M3 || d.kind == NVFP4_SCALE_FP16;
    return T == 1 && dims && kinds && d.k * d.I + d.Is <= 16 * kW * 32 && (d.Is == 0 || d.Is <= d.I) &&
           t1_layout(d, dev.num_sms).total <= dev.smem_optin;
}

std::atomic<int> g_t1_form{0};

bool use_cluster_form(const moe_layer_desc& d, int T, const DeviceInfo& dev) {
    // automatic: the grid form (measured faster on GB300, where the cluster form runs with
    // 12-CTA clusters on 96 SMs); the cluster form when asked for and supported
    if (g_t1_form.load(std::memory_order_relaxed) != 2) return false;
    return t1c_supported(d, T, dev);
}

cudaError_t launch_grid_form(const moe_layer_desc& d, const uint16_t* x, uint16_t* y,
                             int32_t* ids_out, float* w_out, const LayerWs& ws,
                             const DeviceInfo& dev, uint64_t wait_limit, cudaStream_t s,
                             const uint16_t* norm_w, float eps, const uint16_t* resid);

}  // namespace

void set_t1_form(int form) { g_t1_form.store(form < 0 || form > 2 ? 0 : form); }

unsigned long long t1_tag_period(const DeviceInfo& dev) {
    // lcm of the grid sizes either form launches on this device: G = num_sms, and cs k for
    // the cluster sizes cs in {8, 12, 16} and k <= 8
    auto gcd = [](unsigned long long a, unsigned long long b) {
        while (b) { const unsigned long long t = a % b; a = b; b = t; }
        return a;
    };
    unsigned long long l = (unsigned long long)(dev.num_sms > 0 ? dev.num_sms : 1);
    for (int cs : {8, 12, 16})
        for (int k = 1; k <= NVFP4_MAX_TOPK; ++k) {
            const unsigned long long g = (unsigned long long)cs * k;
            l = l / gcd(l, g) * g;
        }
    return l;
}

bool fused_decode_supported(const moe_layer_desc& d, int T, const DeviceInfo& dev) {
    return use_cluster_form(d, T, dev) || grid_form_supported(d, T, dev);
}

int single_token_form_of(const moe_layer_desc& d, int T, const DeviceInfo& dev) {
    if (use_cluster_form(d, T, dev)) return 2;
    return grid_form_supported(d, T, dev) ? 1 : 0;
}

cudaError_t launch_moe_decode_fused(const moe_layer_desc& d, const uint16_t* x, uint16_t* y,
                                    int32_t* ids_out, float* w_out, const LayerWs& ws,
                                    const DeviceInfo& dev, uint64_t wait_limit, cudaStream_t s,
                                    const uint16_t* norm_w, float eps, const uint16_t* resid) {
    if (use_cluster_form(d, 1, dev))
        return launch_moe_decode_t1c(d, x, y, ids_out, w_out, ws, dev, wait_limit, s, norm_w, eps, resid);
    if (!grid_form_supported(d, 1, dev)) return cudaErrorInvalidConfiguration;
    return launch_grid_form(d, x, y, ids_out, w_out, ws, dev, wait_limit, s, norm_w, eps, resid);
}

namespace {

cudaError_t launch_grid_form(const moe_layer_desc& d, const uint16_t* x, uint16_t* y,
                             int32_t* ids_out, float* w_out, const LayerWs& ws,
                             const DeviceInfo& dev, uint64_t wait_limit, cudaStream_t s,
                             const uint16_t* norm_w, float eps, const uint16_t* resid) {
    const int G = dev.num_sms;
    const T1Layout L = t1_layout(d, G);
    if (L.total > dev.smem_optin) return cudaErrorInvalidConfiguration;
    T1Params P;
    P.d = d;
    P.x = x;
    P.y = y;
    P.ids_out = ids_out;
    P.w_out = w_out;
    P.hdr = ws.hdr;
    P.words = ws.words;
    P.wait_limit = wait_limit;
    P.norm_w = norm_w;
    P.eps = eps;
    P.resid = resid;
    P.o_xb = L.o_xb;
    P.o_x16 = L.o_x16;
    P.o_lg = L.o_lg;
    P.o_rt = L.o_rt;
    P.o_sg = L.o_sg;
    P.o_gu = L.o_gu;
    P.o_dn = L.o_dn;
    P.o_dns = L.o_dns;
    P.o_h16 = L.o_h16;
    P.sg_reg = L.sg_reg;
    P.sg_sreg = L.sg_sreg;
    P.gu_reg = L.gu_reg;
    P.gu_sreg = L.gu_sreg;
    P.dn_row = L.dn_row;
    P.dn_srow = L.dn_srow;
    P.tag_period = t1_tag_period(dev);
    P.tag_step = P.tag_period / (unsigned long long)G;
    P.mP64 = ~0ull / P.tag_period + 1ull;
    auto kern = d.kind == NVFP4_SCALE_E4M3 ? moe_decode_t1_kernel<NVFP4_SCALE_E4M3>
                                           : moe_decode_t1_kernel<NVFP4_SCALE_FP16>;
    // raise the dynamic shared-memory limit once per (device, kind, size)
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
    cfg.blockDim = dim3(kThr);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace

}  // namespace nvfp4
