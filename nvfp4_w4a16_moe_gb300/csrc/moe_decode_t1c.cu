// One-launch decode of the MoE layer for a single token (T = 1), cluster form.
//
// Sources (page title, section): as the grid form in moe_decode_t1.cu
//  - lynn-engine README, P45 note: the active-MoE path as one native call; P28/P29 notes:
//    gate/up + SiLU -> [top_k, I] intermediate, then down + routing-weighted sum; P46/P48
//    notes: no atomics in the combine, every output row summed in a fixed order by one owner.
//  - lynn-engine tutorials index, row 06: softmax over all experts -> top-k -> renormalise;
//    sigmoid-gated shared expert.
//
// Layout of the work: k clusters of cs CTAs (one CTA per SM; cs the largest of 16, 12, 8
// of which the device holds k clusters at once and whose shared-memory layout fits).
// Cluster j owns routed slot j (the j-th selected expert); its CTA of rank r owns
//   router rows      [(E+1) r/cs, (E+1)(r+1)/cs)   every cluster computes all E + 1 logits
//   routed pairs     [I r/cs, I (r+1)/cs)          of the slot's expert (gate row, up row)
//   routed down rows [H r/cs, H (r+1)/cs)          of the slot's expert, K = I
// and, as CTA c of the whole grid (Gt = cs k CTAs),
//   shared pairs     [Is c/Gt, Is (c+1)/Gt)        of the shared expert
//   output rows      [H c/Gt, H (c+1)/Gt)          it finalises (and the shared expert's
//                                                  down rows of them)
// The router rows and the routed pairs share one shared-memory region: the rows are read
// before the top-k, the pairs copied after it.
//
// Exchanges:
//   logits   each CTA writes its logits into the shared memory of every CTA of its cluster
//            (distributed shared memory), then one cluster barrier: no global round trip
//   h_j      the slot's SwiGLU values likewise stay inside the cluster
//   hs       the shared expert's values cross the grid as tagged words (as in the grid
//            form); they are produced before the top-k and read while the routed weights
//            stream in, so their latency is off the critical path
//   y        each CTA publishes coef_j * (down_j . h_j) for its H/cs rows as tagged words; the
//            owner of an output row reads the k partials (one 128-byte line per slot, read by
//            that owner alone) and adds them, then the shared part, in a fixed order
//
// Every global poll is bounded in time; a poll that runs out records NVFP4_ERR_DEVICE_TIMEOUT
// and the CTA carries on with what it has (the call reports the error), so every CTA reaches
// every cluster barrier. No CTA touches a peer's shared memory after the last cluster
// barrier, and each CTA waits (bounded) for its own bulk copies before it exits.
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.cuh"
#include "t1_device.cuh"

namespace nvfp4 {

namespace {

constexpr int kMaxCl = 16;                 // CTAs per cluster, at most
constexpr int kClSizes[3] = {16, 12, 8};   // cluster sizes tried, largest first
constexpr int kCW = 16;                    // compute warps
constexpr int kCThr = (kCW + 1) * 32;      // + the copy warp
constexpr int kCCopy = kCW;
constexpr int kCChunks = 2;                // routed gate/up copy chunks (one mbarrier each)
constexpr int kMaxF = 64;                  // output rows a CTA finalises, at most

struct T1CParams {
    moe_layer_desc d;
    const uint16_t* x;
    uint16_t* y;
    int32_t* ids_out;
    float* w_out;
    WsHeader* hdr;
    uint32_t* hs_words;              // kWordReplicas copies of the Is tagged shared values
    unsigned long long* part;        // [k][H] tagged partial outputs (tag << 32 | fp32 bits)
    unsigned long long wait_limit;
    const uint16_t* norm_w;          // nullable: x = bf16(RMSNorm_(1+w)(input)) first
    float eps;
    const uint16_t* resid;           // nullable: y = bf16(resid + layer)
    // shared-memory layout (bytes), identical for every CTA
    uint32_t o_xb, o_x16, o_lg, o_rt, o_sg, o_sd, o_gu, o_dn, o_hj, o_hj16, o_hs16;
    uint32_t sg_reg, sg_sreg;        // shared-pair regions (codes, scales)
    uint32_t gu_reg, gu_sreg;        // routed-pair regions
    uint32_t sd_sc, dn_sc;           // offset of the scales in the shared / routed down areas
    uint32_t hs_stride;              // 32-bit words per copy of the shared values
    int cs;                          // CTAs per cluster
    unsigned long long tag_step;     // added by each CTA: tag_period / Gt
    unsigned long long tag_period;
    unsigned long long mP64;         // ceil(2^64 / tag_period)
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// address of `p` (this CTA's shared memory) in the shared memory of cluster CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
    return a;
}
__device__ __forceinline__ void st_peer_f32(uint32_t a, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void st_peer_u16(uint32_t a, uint16_t v) {
    asm volatile("st.shared::cluster.u16 [%0], %1;" :: "r"(a), "h"(v) : "memory");
}

// dot products of `rows` down rows (codes at w + row * rb, scales at ws + row * sbr) with
// the f16 vector v (nseg segments, segment-interleaved), nseg in {8, 16, 32}: lane l takes
// row l / nseg, segment l % nseg of each pass; the nseg lanes of a row are reduced by
// shuffles. fn(row, sum) is called on the first lane of each row.
template <int KIND, typename Fn>
__device__ __forceinline__ void rows_dot(const uint8_t* w, uint32_t rb, const uint8_t* ws, uint32_t sbr, int rows,
                                         const uint4* v, int nseg, int warp, int lane, Fn fn) {
    const int rpp = 32 / nseg, rl = lane / nseg, s = lane - rl * nseg;
    for (int n = warp * rpp; n < rows; n += kCW * rpp) {
        const int row = n + rl;
        float acc = 0.f;
        if (row < rows) {
            float a0, a1;
            scales2<KIND>(ws + (size_t)row * sbr, s, a0, a1);
            acc = seg_dot<KIND>(reinterpret_cast<const uint4*>(w + (size_t)row * rb)[s], a0, a1, v, nseg, s);
        }
        for (int o = nseg >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (s == 0 && row < rows) fn(row, acc);
    }
}

// 8 bf16 (one 16-byte unit) times sc as 8 f16
__device__ __forceinline__ uint4 bf16x8_to_f16(const uint4 a, float sc) {
    return make_uint4(to_f16x2(bf16lo(a.x) * sc, bf16hi(a.x) * sc), to_f16x2(bf16lo(a.y) * sc, bf16hi(a.y) * sc),
                      to_f16x2(bf16lo(a.z) * sc, bf16hi(a.z) * sc), to_f16x2(bf16lo(a.w) * sc, bf16hi(a.w) * sc));
}

template <int KIND>
__global__ void __launch_bounds__(kCThr, 1) moe_decode_t1c_kernel(T1CParams P) {
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ uint64_t mbA, mbS, mbD, mbG[kCChunks];
    __shared__ float s_red[2][kCW][8];          // routed-pair sums of each warp, per batch parity
    __shared__ float s_hmx[kMaxCl];             // max |h_j| of each CTA of the cluster (peers write)
    __shared__ float s_ys[kMaxF];               // shared-expert part of each output row
    __shared__ float s_part[NVFP4_MAX_TOPK][kMaxF];
    __shared__ float s_tg[NVFP4_MAX_EXPERTS * 2], s_td[NVFP4_MAX_EXPERTS];
    __shared__ float s_ss[kCThr / 32];
    __shared__ uint32_t s_xmax, s_tag, s_hloc, s_hsm;
    __shared__ float s_coef, s_coef_s, s_tsg, s_tsu;
    __shared__ int s_eid, s_fail;

    const moe_layer_desc& d = P.d;
    const int H = d.H, E = d.E, k = d.k, I = d.I, Is = d.Is;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, Gt = gridDim.x;
    const int cs = P.cs, r = (int)cluster_rank(), j = c / cs;
    const int sb = KIND == NVFP4_SCALE_E4M3 ? 1 : 2;
    const uint32_t rowH = H / 2, srowH = H / 16 * sb;       // code / scale row bytes, K = H
    const uint32_t rowI = I / 2, srowI = I / 16 * sb;       // K = I
    const uint32_t rowS = Is / 2, srowS = Is / 16 * sb;     // K = Is
    const int nsegH = H >> 5, nunitH = H >> 3, nsegI = I >> 5, nsegS = Is >> 5;
    const int Er = Is > 0 ? E + 1 : E;                      // router rows (row E: the shared gate)
    const int rr0 = Er * r / cs, rr1 = Er * (r + 1) / cs;
    const int sp0 = (int)((long long)Is * c / Gt), sp1 = (int)((long long)Is * (c + 1) / Gt);
    const int f0 = (int)((long long)H * c / Gt), f1 = (int)((long long)H * (c + 1) / Gt);
    const int p0 = I * r / cs, p1 = I * (r + 1) / cs;
    const int d0 = H * r / cs, d1 = H * (r + 1) / cs;
    const int nRr = rr1 - rr0, nSp = sp1 - sp0, nF = f1 - f0, nP = p1 - p0, nD = d1 - d0;
    const uint32_t* hs_w = P.hs_words + (size_t)(c % kWordReplicas) * P.hs_stride;   // this CTA's copy

    uint16_t* xb = reinterpret_cast<uint16_t*>(sm + P.o_xb);
    uint4* x16 = reinterpret_cast<uint4*>(sm + P.o_x16);
    float* lg = reinterpret_cast<float*>(sm + P.o_lg);      // written by every CTA of the cluster
    uint8_t* RT = sm + P.o_rt;
    uint8_t* SG = sm + P.o_sg;                // gate codes, up codes, gate scales, up scales
    uint8_t* SD = sm + P.o_sd;                // shared down rows of the output rows: codes, scales
    uint8_t* GU = sm + P.o_gu;                // routed pairs: same four regions as SG
    uint8_t* DN = sm + P.o_dn;                // routed down rows: codes, scales
    uint16_t* hj = reinterpret_cast<uint16_t*>(sm + P.o_hj);    // bf16 h_j, written by the cluster
    uint4* hj16 = reinterpret_cast<uint4*>(sm + P.o_hj16);
    uint4* hs16 = reinterpret_cast<uint4*>(sm + P.o_hs16);

    // no CTA writes into a peer's shared memory before the whole cluster runs
    cluster_arrive_relaxed();

    // ------------------------------------------------------------------ prologue
    if (tid == 0) {
        mbar_init(&mbA, 1);
        mbar_init(&mbS, 1);
        mbar_init(&mbD, 1);
        for (int i = 0; i < kCChunks; ++i) mbar_init(&mbG[i], 1);
        fence_mbar_init();
        s_fail = 0;
        s_xmax = 0u;
        s_hloc = 0u;
        s_hsm = 0u;
    }
    __syncthreads();
    const uint8_t* sh_gu = d.sh_gu_packed;
    const uint8_t* sh_gus = static_cast<const uint8_t*>(d.sh_gu_scales);
    if (warp == kCCopy) {
        // weight-only copies: router rows, shared pairs, shared down rows of the output rows
        const int rE = min(rr1, E) - min(rr0, E);
        if (lane == 0) {
            const uint32_t a = (uint32_t)rE * 2u * H + (rr1 > E ? 2u * H : 0u) + (uint32_t)nSp * 2u * (rowH + srowH);
            mbar_arrive_expect_tx(&mbA, a);
            mbar_arrive_expect_tx(&mbS, Is > 0 ? (uint32_t)nF * (rowS + srowS) : 0u);
        }
        __syncwarp();
        if (lane == 0 && rE > 0)
            copy_range(RT, reinterpret_cast<const uint8_t*>(d.router_w + (size_t)min(rr0, E) * H), (uint32_t)rE * 2u * H,
                       &mbA);
        if (lane == 1 && rr1 > E)
            copy_range(RT + (size_t)rE * 2 * H, reinterpret_cast<const uint8_t*>(d.sh_gate_w), 2u * H, &mbA);
        if (nSp > 0) {
            if (lane == 2) copy_range(SG, sh_gu + (size_t)sp0 * rowH, (uint32_t)nSp * rowH, &mbA);
            if (lane == 3) copy_range(SG + P.sg_reg, sh_gu + (size_t)(Is + sp0) * rowH, (uint32_t)nSp * rowH, &mbA);
            if (lane == 4) copy_range(SG + 2 * P.sg_reg, sh_gus + (size_t)sp0 * srowH, (uint32_t)nSp * srowH, &mbA);
            if (lane == 5)
                copy_range(SG + 2 * P.sg_reg + P.sg_sreg, sh_gus + (size_t)(Is + sp0) * srowH, (uint32_t)nSp * srowH,
                           &mbA);
        }
        if (Is > 0) {
            if (lane == 6) copy_range(SD, d.sh_dn_packed + (size_t)f0 * rowS, (uint32_t)nF * rowS, &mbS);
            if (lane == 7)
                copy_range(SD + P.sd_sc, static_cast<const uint8_t*>(d.sh_dn_scales) + (size_t)f0 * srowS,
                           (uint32_t)nF * srowS, &mbS);
        }
    }
    float tsv[3] = {0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const int i = tid + u * kCThr;
        if (i < 2 * E) tsv[u] = __ldg(d.gu_tscale + i);
        else if (i < 3 * E) tsv[u] = __ldg(d.dn_tscale + (i - 2 * E));
    }
    float sh_tsg = 0.f, sh_tsu = 0.f, sh_tsd = 0.f;
    if (Is > 0) {
        sh_tsg = __ldg(d.sh_gu_tscale);
        sh_tsu = __ldg(d.sh_gu_tscale + 1);
        sh_tsd = __ldg(d.sh_dn_tscale);
    }
    // this launch's tag (see the grid form): the atomic is issued before griddepcontrol.wait,
    // its result first used after the x load
    unsigned long long n_start = 0;
    if (tid == 0)
        asm volatile("atom.relaxed.gpu.global.add.u64 %0, [%1], %2;"
                     : "=l"(n_start) : "l"(&P.hdr->barrier), "l"(P.tag_step) : "memory");

    // everything below may read what the previous kernel on the stream wrote
    asm volatile("griddepcontrol.wait;" ::: "memory");

    uint4 xv = make_uint4(0, 0, 0, 0);
    if (tid < nunitH) xv = reinterpret_cast<const uint4*>(P.x)[tid];
    if (tid == 0) {
        unsigned long long q = __umul64hi(n_start, P.mP64);    // n / period, corrected below
        if ((q + 1) * P.tag_period <= n_start) ++q;
        if (q * P.tag_period > n_start) --q;
        s_tag = (uint32_t)q + 1u;
    }
    if (P.norm_w) {
        // pre-MoE RMSNorm (1 + w) x / sqrt(mean(x^2) + eps), as in the grid form
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
        for (int i = 0; i < kCThr / 32; ++i) tot += s_ss[i];
        const float rn = 1.0f / sqrtf(tot / (float)H + P.eps);
        if (tid < nunitH) {
            const uint4 wv = reinterpret_cast<const uint4*>(P.norm_w)[tid];
            const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w}, nw[4] = {wv.x, wv.y, wv.z, wv.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float lo = bf16lo(xx[q]) * rn * (1.0f + bf16lo(nw[q]));
                const float hi = bf16hi(xx[q]) * rn * (1.0f + bf16hi(nw[q]));
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
        if (lane == 0) atomicMax(&s_xmax, m << 16);
    }
    __syncthreads();
    const uint32_t tag = s_tag, tag16 = tag16_of(tag);
    const int sx = pow2_shift(s_xmax);
    if (tid < nunitH) {
        const float sc = exp2_int(sx);
        x16[(tid & 3) * nsegH + (tid >> 2)] = make_uint4(
            to_f16x2(bf16lo(xv.x) * sc, bf16hi(xv.x) * sc), to_f16x2(bf16lo(xv.y) * sc, bf16hi(xv.y) * sc),
            to_f16x2(bf16lo(xv.z) * sc, bf16hi(xv.z) * sc), to_f16x2(bf16lo(xv.w) * sc, bf16hi(xv.w) * sc));
    }
#pragma unroll
    for (int u = 0; u < 3; ++u) {
        const int i = tid + u * kCThr;
        if (i < 2 * E) s_tg[i] = tsv[u];
        else if (i < 3 * E) s_td[i - 2 * E] = tsv[u];
    }
    __syncthreads();
    const float inv_x = exp2_int(-sx);
    bool ok = true;

    // ------------------------------------------------------------------ router rows, shared pairs
    cluster_wait();   // the cluster runs: peers' shared memory may be written from here on
    if (warp < kCW) {
        ok = mbar_wait_bounded(&mbA, 0, kDefaultWaitLimit);
        for (int t = warp; t < nRr + nSp; t += kCW) {
            if (t < nRr) {
                const uint4* wr = reinterpret_cast<const uint4*>(RT + (size_t)t * 2 * H);
                const uint4* xr = reinterpret_cast<const uint4*>(xb);
                float acc = 0.f;
#pragma unroll 4
                for (int ch = lane; ch < nunitH; ch += 32) acc = bf16_dot8(wr[ch], xr[ch], acc);
                acc = warp_sum(acc);
                if (lane < cs) st_peer_f32(peer_addr(&lg[rr0 + t], lane), acc);
            } else {
                const int i = t - nRr;
                const float m = pair_dot<KIND>(SG + (size_t)i * rowH, SG + P.sg_reg + (size_t)i * rowH,
                                               SG + 2 * P.sg_reg + (size_t)i * srowH,
                                               SG + 2 * P.sg_reg + P.sg_sreg + (size_t)i * srowH, x16, nsegH, lane);
                const float gsum = __shfl_sync(0xffffffffu, m, 0), usum = __shfl_sync(0xffffffffu, m, 16);
                if (lane < kWordReplicas) {
                    const float hv = silu_f32(gsum * inv_x * sh_tsg) * (usum * inv_x * sh_tsu);
                    st_hword(P.hs_words + (size_t)lane * P.hs_stride + sp0 + i, tag16, hv);
                }
            }
        }
    }
    asm volatile("griddepcontrol.launch_dependents;");
    cluster_arrive();
    cluster_wait();   // all E + 1 logits are in this CTA's shared memory

    // ------------------------------------------------------------------ top-k
    if (warp == 0) {
        // as the grid form: per-lane sorted 64-bit keys, the lower id wins ties
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
        for (int jj = 0; jj < k; ++jj) {
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
            if (jj == 0) vmax = v;
            if (lane == jj) { my_id = e; ex = __expf(v - vmax); }
        }
        const float sum = warp_sum(lane < k ? ex : 0.f);
        if (lane < k) {
            const float wj = __fdividef(ex, sum);
            if (lane == j) {
                s_eid = my_id;
                s_coef = wj * s_td[my_id];
                s_tsg = s_tg[2 * my_id];
                s_tsu = s_tg[2 * my_id + 1];
            }
            if (c == 0) {
                if (P.ids_out) P.ids_out[lane] = my_id;
                if (P.w_out) P.w_out[lane] = wj;
            }
        }
        if (lane == 0) s_coef_s = Is > 0 ? sigmoid_f32(lg[E]) * sh_tsd : 0.f;
    }
    __syncthreads();

    // ------------------------------------------------------------------ routed copies, hs
    const int e = s_eid;
    uint4 hsv = make_uint4(0, 0, 0, 0);   // 8 shared values (bf16) of unit tid
    if (warp == kCCopy) {
        // the routed pairs land where the router rows were read (generic loads, finished
        // before the barrier above): order those reads before the bulk copies' writes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // chunk ch: pairs [nP ch / 2, nP (ch+1) / 2) of the slot's expert, lane 4 ch + part
        // copies gate codes, up codes, gate scales or up scales; lanes 8, 9 the down rows
        if (lane < kCChunks) {
            const int a = nP * lane / kCChunks, b = nP * (lane + 1) / kCChunks;
            mbar_arrive_expect_tx(&mbG[lane], (uint32_t)(b - a) * 2u * (rowH + srowH));
        }
        if (lane == kCChunks) mbar_arrive_expect_tx(&mbD, (uint32_t)nD * (rowI + srowI));
        __syncwarp();
        if (lane < 4 * kCChunks) {
            const int ch = lane >> 2, part = lane & 3;
            const int a = nP * ch / kCChunks, b = nP * (ch + 1) / kCChunks;
            if (b > a) {
                const size_t grow = (size_t)e * 2 * I + p0 + a + (part & 1) * I;   // first gate / up row
                if (part < 2)
                    copy_range(GU + (part ? P.gu_reg : 0u) + (size_t)a * rowH, d.gu_packed + grow * rowH,
                               (uint32_t)(b - a) * rowH, &mbG[ch]);
                else
                    copy_range(GU + 2 * P.gu_reg + (part == 3 ? P.gu_sreg : 0u) + (size_t)a * srowH,
                               static_cast<const uint8_t*>(d.gu_scales) + grow * srowH, (uint32_t)(b - a) * srowH,
                               &mbG[ch]);
            }
        } else if (lane == 8) {
            copy_range(DN, d.dn_packed + ((size_t)e * H + d0) * rowI, (uint32_t)nD * rowI, &mbD);
        } else if (lane == 9) {
            copy_range(DN + P.dn_sc, static_cast<const uint8_t*>(d.dn_scales) + ((size_t)e * H + d0) * srowI,
                       (uint32_t)nD * srowI, &mbD);
        }
    } else if (Is > 0 && tid < (Is >> 3)) {
        // the Is shared values, 8 tagged words per 32-byte load, re-read until tagged (bounded)
        uint4 wa, wb;
        auto ready = [&](const uint4 w) {
            return (w.x >> 16) == tag16 && (w.y >> 16) == tag16 && (w.z >> 16) == tag16 && (w.w >> 16) == tag16;
        };
        ld_hwords8(hs_w + 8 * tid, wa, wb);
        if (!(ready(wa) && ready(wb))) {
            const unsigned long long t0 = global_timer_ns();
            do {
                if (global_timer_ns() - t0 > P.wait_limit) { ok = false; break; }
                ld_hwords8(hs_w + 8 * tid, wa, wb);
            } while (!(ready(wa) && ready(wb)));
        }
        // the bf16 halves (low 16 bits of each word), two per 32-bit lane
        hsv = make_uint4((wa.x & 0xFFFFu) | (wa.y << 16), (wa.z & 0xFFFFu) | (wa.w << 16),
                         (wb.x & 0xFFFFu) | (wb.y << 16), (wb.z & 0xFFFFu) | (wb.w << 16));
        uint32_t m = max(max(hsv.x & 0x7FFFu, (hsv.x >> 16) & 0x7FFFu), max(hsv.y & 0x7FFFu, (hsv.y >> 16) & 0x7FFFu));
        m = max(m, max(max(hsv.z & 0x7FFFu, (hsv.z >> 16) & 0x7FFFu), max(hsv.w & 0x7FFFu, (hsv.w >> 16) & 0x7FFFu)));
        atomicMax(&s_hsm, m << 16);
    }
    __syncthreads();
    // the shared values as f16 times 2^sh_s (max in [2^14, 2^15)), segment-interleaved
    const int sh_s = pow2_shift(s_hsm);
    if (warp < kCW && tid < (Is >> 3)) {
        const int e0 = 8 * tid;
        hs16[((e0 >> 3) & 3) * nsegS + (e0 >> 5)] = bf16x8_to_f16(hsv, exp2_int(sh_s));
    }
    __syncthreads();
    // the shared expert's down rows of the output rows (K = Is), while the routed weights
    // stream in
    if (warp < kCW && Is > 0) {
        if (!mbar_wait_bounded(&mbS, 0, kDefaultWaitLimit)) ok = false;
        const float cs = s_coef_s * exp2_int(-sh_s);
        rows_dot<KIND>(SD, rowS, SD + P.sd_sc, srowS, nF, hs16, nsegS, warp, lane,
                       [&](int row, float acc) { s_ys[row] = acc * cs; });
    }

    // ------------------------------------------------------------------ routed pairs
    // lane group g (warps 2g, 2g + 1) takes local pairs g, g + 8, g + 16, ... in batches of
    // four, its lane i the segments i, i + 64, ... of H (x segment in registers across the
    // batch); each warp reduces its 8 sums (warp_sum8) and, after a barrier, the even warp of
    // the group adds the two warps' sums in a fixed order and writes bf16(h) into every CTA
    // of the cluster. Every warp runs the batch loop (the barrier is the CTA's).
    {
        constexpr int kGroups = kCW / 2, kBatch = 4;
        const int g = warp >> 1, gi = tid & 63;
        const int nb = (nP + kGroups * kBatch - 1) / (kGroups * kBatch);
        const uint8_t* GUs = GU + 2 * P.gu_reg;
        const float cg = inv_x * s_tsg, cu = inv_x * s_tsu;
        for (int b = 0; b < nb; ++b) {
            if (warp < kCW) {
                float v[2 * kBatch];
#pragma unroll
                for (int i = 0; i < 2 * kBatch; ++i) v[i] = 0.f;
                for (int s = gi; s < nsegH; s += 64) {
                    const uint4 u0 = x16[s], u1 = x16[nsegH + s], u2 = x16[2 * nsegH + s], u3 = x16[3 * nsegH + s];
#pragma unroll
                    for (int m = 0; m < kBatch; ++m) {
                        const int rl = g + kGroups * (b * kBatch + m);
                        if (rl < nP) {
                            const int ch = rl < nP / kCChunks ? 0 : kCChunks - 1;
                            if (ok && !mbar_wait_bounded(&mbG[ch], 0, kDefaultWaitLimit)) ok = false;
                            float g0, g1, a0, a1;
                            scales2<KIND>(GUs + (size_t)rl * srowH, s, g0, g1);
                            scales2<KIND>(GUs + P.gu_sreg + (size_t)rl * srowH, s, a0, a1);
                            v[2 * m] += seg_dot_r(reinterpret_cast<const uint4*>(GU + (size_t)rl * rowH)[s], g0, g1,
                                                  u0, u1, u2, u3);
                            v[2 * m + 1] += seg_dot_r(
                                reinterpret_cast<const uint4*>(GU + P.gu_reg + (size_t)rl * rowH)[s], a0, a1, u0,
                                u1, u2, u3);
                        }
                    }
                }
                const float z = warp_sum8(v, lane);
                if ((lane & 3) == 0) s_red[b & 1][warp][(lane >> 2) & 7] = z;
            }
            __syncthreads();
            if (warp < kCW && (warp & 1) == 0) {
                // i = m * 16 + peer: pair m of the batch into cluster CTA `peer`
                for (int i = lane; i < kBatch * cs; i += 32) {
                    const int m = i / cs, peer = i - m * cs, rl = g + kGroups * (b * kBatch + m);
                    if (rl < nP) {
                        const float gs = s_red[b & 1][warp][2 * m] + s_red[b & 1][warp + 1][2 * m];
                        const float us = s_red[b & 1][warp][2 * m + 1] + s_red[b & 1][warp + 1][2 * m + 1];
                        const uint16_t hb16 = f32_to_bf16(silu_f32(gs * cg) * (us * cu));
                        st_peer_u16(peer_addr(&hj[p0 + rl], (uint32_t)peer), hb16);
                        if (peer == 0) atomicMax(&s_hloc, (uint32_t)(hb16 & 0x7FFFu));
                    }
                }
            }
        }
    }
    __syncthreads();
    if (warp == 0 && lane < cs) st_peer_f32(peer_addr(&s_hmx[r], (uint32_t)lane), __uint_as_float(s_hloc << 16));
    cluster_arrive();
    cluster_wait();   // h_j (I values) and the 16 maxima are in this CTA's shared memory;
                      // no CTA writes into a peer's shared memory after this point

    // ------------------------------------------------------------------ down
    // h_j as f16 times 2^sh (max over the cluster in [2^14, 2^15)), segment-interleaved
    uint32_t hm = 0u;
#pragma unroll
    for (int i = 0; i < kMaxCl; ++i)
        if (i < cs) hm = max(hm, __float_as_uint(s_hmx[i]));
    const int sh = pow2_shift(hm);
    for (int u = tid; u < (I >> 3); u += kCThr) {
        const int e0 = 8 * u;
        hj16[((e0 >> 3) & 3) * nsegI + (e0 >> 5)] =
            bf16x8_to_f16(reinterpret_cast<const uint4*>(hj)[u], exp2_int(sh));
    }
    __syncthreads();
    if (warp < kCW) {
        if (!mbar_wait_bounded(&mbD, 0, kDefaultWaitLimit)) ok = false;
        const float cj = s_coef * exp2_int(-sh);
        unsigned long long* part = P.part + (size_t)j * H + d0;
        rows_dot<KIND>(DN, rowI, DN + P.dn_sc, srowI, nD, hj16, nsegI, warp, lane,
                       [&](int row, float acc) { st_word(part + row, tag, acc * cj); });
    }

    // ------------------------------------------------------------------ combine
    // the k partials of the output rows [f0, f1), then the shared part, in a fixed order
    if (tid < k * nF) {
        const int jj = tid / nF, i = tid - jj * nF;
        float v = 0.f;
        if (!poll_word(P.part + (size_t)jj * H + f0 + i, tag, P.wait_limit, &v)) ok = false;
        s_part[jj][i] = v;
    }
    if (!ok) s_fail = 1;
    __syncthreads();
    if (tid < nF) {
        float acc = 0.f;
        for (int jj = 0; jj < k; ++jj) acc += s_part[jj][tid];
        if (Is > 0) acc += s_ys[tid];
        if (P.resid) acc += bf16_to_f32(P.resid[f0 + tid]);   // residual stream, before the rounding
        P.y[f0 + tid] = f32_to_bf16(acc);
    }
    if (tid == 0) {
        if (s_fail) record_status(P.hdr, NVFP4_ERR_DEVICE_TIMEOUT);
        // no bulk copy of this CTA is still in flight when it exits
        mbar_wait_bounded(&mbA, 0, kDefaultWaitLimit);
        mbar_wait_bounded(&mbS, 0, kDefaultWaitLimit);
        mbar_wait_bounded(&mbD, 0, kDefaultWaitLimit);
        for (int i = 0; i < kCChunks; ++i) mbar_wait_bounded(&mbG[i], 0, kDefaultWaitLimit);
    }
}

struct T1CLayout {
    uint32_t o_xb, o_x16, o_lg, o_rt, o_sg, o_sd, o_gu, o_dn, o_hj, o_hj16, o_hs16, total;
    uint32_t sg_reg, sg_sreg, gu_reg, gu_sreg, sd_sc, dn_sc;
};

uint32_t c16(size_t v) { return (uint32_t)((v + 15) & ~size_t(15)); }

T1CLayout t1c_layout(const moe_layer_desc& d, int cs) {
    const size_t sb = d.kind == NVFP4_SCALE_E4M3 ? 1 : 2;
    const size_t H = d.H, I = d.I, Is = d.Is, k = d.k, E = d.E;
    const size_t Gt = (size_t)cs * k;
    const size_t nR = (E + 1 + cs - 1) / cs, nS = (Is + Gt - 1) / Gt, nF = (H + Gt - 1) / Gt;
    const size_t nP = (I + cs - 1) / cs, nD = (H + cs - 1) / cs;
    T1CLayout L;
    L.sg_reg = c16(nS * (H / 2));
    L.sg_sreg = c16(nS * (H / 16 * sb));
    L.gu_reg = c16(nP * (H / 2));
    L.gu_sreg = c16(nP * (H / 16 * sb));
    L.sd_sc = c16(nF * (Is / 2));
    L.dn_sc = c16(nD * (I / 2));
    const size_t rt = c16(nR * H * 2), gu = 2 * (size_t)L.gu_reg + 2 * (size_t)L.gu_sreg;
    size_t off = 0;
    L.o_xb = (uint32_t)off; off += c16(H * 2);
    L.o_x16 = (uint32_t)off; off += c16(H * 2);
    L.o_lg = (uint32_t)off; off += c16((E + 1) * 4);
    // the router rows (read before the top-k) and the routed pairs (copied after it)
    // share one region
    L.o_rt = L.o_gu = (uint32_t)off; off += rt > gu ? rt : gu;
    L.o_sg = (uint32_t)off; off += 2 * (size_t)L.sg_reg + 2 * (size_t)L.sg_sreg;
    L.o_sd = (uint32_t)off; off += (size_t)L.sd_sc + c16(nF * (Is / 16 * sb));
    L.o_dn = (uint32_t)off; off += (size_t)L.dn_sc + c16(nD * (I / 16 * sb));
    L.o_hj = (uint32_t)off; off += c16(I * 2);
    L.o_hj16 = (uint32_t)off; off += c16(I * 2);
    L.o_hs16 = (uint32_t)off; off += c16(Is * 2 + 16);
    L.total = (uint32_t)off;
    return L;
}

// the largest dynamic shared memory any launch asked for, per device and kind
std::atomic<uint32_t> g_t1c_smem_set[64][2];

template <int KIND>
cudaError_t prepare_t1c(int dev_index, uint32_t smem) {
    const int dv = dev_index < 64 ? dev_index : 63, ki = KIND == NVFP4_SCALE_E4M3 ? 0 : 1;
    if (g_t1c_smem_set[dv][ki].load(std::memory_order_relaxed) < smem) {
        cudaError_t err = cudaFuncSetAttribute(moe_decode_t1c_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(moe_decode_t1c_kernel<KIND>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (err != cudaSuccess) return err;
        g_t1c_smem_set[dv][ki].store(smem, std::memory_order_relaxed);
    }
    return cudaSuccess;
}

// How many clusters of `cs` CTAs of this kernel with `smem` bytes of dynamic shared memory
// can be resident at once (0 on any error); cached per (device, kind, cs, smem).
struct CapEntry {
    int dev, kind, cs;
    uint32_t smem;
    int n;
};
std::mutex g_cap_mu;
std::vector<CapEntry> g_cap;

template <int KIND>
int t1c_max_clusters(const DeviceInfo& dev, uint32_t smem, int cs) {
    {
        std::lock_guard<std::mutex> lk(g_cap_mu);
        for (const CapEntry& e : g_cap)
            if (e.dev == dev.device && e.kind == KIND && e.cs == cs && e.smem == smem) return e.n;
    }
    int n = 0;
    if (prepare_t1c<KIND>(dev.device, smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs * NVFP4_MAX_TOPK);
        cfg.blockDim = dim3(kCThr);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, moe_decode_t1c_kernel<KIND>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
    }
    std::lock_guard<std::mutex> lk(g_cap_mu);
    if (g_cap.size() < 256) g_cap.push_back(CapEntry{dev.device, KIND, cs, smem, n});
    return n;
}

bool t1c_shape_ok(const moe_layer_desc& d) {
    const bool kinds = d.kind == NVFP4_SCALE_E4M3 || d.kind == NVFP4_SCALE_FP16;
    const bool seg = (d.I == 256 || d.I == 512 || d.I == 1024) &&
                     (d.Is == 0 || d.Is == 256 || d.Is == 512 || d.Is == 1024);
    return kinds && seg && d.H % 256 == 0 && d.H <= 4096;
}

bool t1c_fits(const moe_layer_desc& d, const DeviceInfo& dev, int cs) {
    const int Gt = cs * d.k;
    // dynamic plus this kernel's static shared memory (under 8 KB) within the opt-in limit
    return Gt <= dev.num_sms && (d.H + Gt - 1) / Gt <= kMaxF &&
           (size_t)t1c_layout(d, cs).total + 8192 <= dev.smem_optin;
}

int t1c_capacity(const moe_layer_desc& d, const DeviceInfo& dev, int cs) {
    const uint32_t smem = t1c_layout(d, cs).total;
    return d.kind == NVFP4_SCALE_E4M3 ? t1c_max_clusters<NVFP4_SCALE_E4M3>(dev, smem, cs)
                                      : t1c_max_clusters<NVFP4_SCALE_FP16>(dev, smem, cs);
}

// cluster size for this layer on this device: the largest tried size whose layout fits
// and of which the device holds k clusters at once; 0 if none
int t1c_cluster_size(const moe_layer_desc& d, const DeviceInfo& dev) {
    if (!t1c_shape_ok(d)) return 0;
    for (int cs : kClSizes)
        if (t1c_fits(d, dev, cs) && t1c_capacity(d, dev, cs) >= d.k) return cs;
    return 0;
}

}  // namespace

bool t1c_supported(const moe_layer_desc& d, int T, const DeviceInfo& dev) {
    return T == 1 && t1c_cluster_size(d, dev) > 0;
}

int t1c_cluster_capacity(const moe_layer_desc& d, const DeviceInfo& dev) {
    const int cs = t1c_cluster_size(d, dev);
    return cs ? cs * 100 + t1c_capacity(d, dev, cs) : 0;
}

cudaError_t launch_moe_decode_t1c(const moe_layer_desc& d, const uint16_t* x, uint16_t* y, int32_t* ids_out,
                                  float* w_out, const LayerWs& ws, const DeviceInfo& dev, uint64_t wait_limit,
                                  cudaStream_t s, const uint16_t* norm_w, float eps, const uint16_t* resid) {
    const int cs = t1c_cluster_size(d, dev);
    if (cs == 0) return cudaErrorInvalidConfiguration;
    const T1CLayout L = t1c_layout(d, cs);
    const int Gt = cs * d.k;
    T1CParams P;
    P.d = d;
    P.x = x;
    P.y = y;
    P.ids_out = ids_out;
    P.w_out = w_out;
    P.hdr = ws.hdr;
    P.hs_stride = (uint32_t)(((size_t)d.Is + 31) & ~size_t(31));
    P.cs = cs;
    P.hs_words = reinterpret_cast<uint32_t*>(ws.words);
    P.part = ws.words + (size_t)kWordReplicas * P.hs_stride / 2;
    P.wait_limit = wait_limit;
    P.norm_w = norm_w;
    P.eps = eps;
    P.resid = resid;
    P.o_xb = L.o_xb;
    P.o_x16 = L.o_x16;
    P.o_lg = L.o_lg;
    P.o_rt = L.o_rt;
    P.o_sg = L.o_sg;
    P.o_sd = L.o_sd;
    P.o_gu = L.o_gu;
    P.o_dn = L.o_dn;
    P.o_hj = L.o_hj;
    P.o_hj16 = L.o_hj16;
    P.o_hs16 = L.o_hs16;
    P.sg_reg = L.sg_reg;
    P.sg_sreg = L.sg_sreg;
    P.gu_reg = L.gu_reg;
    P.gu_sreg = L.gu_sreg;
    P.sd_sc = L.sd_sc;
    P.dn_sc = L.dn_sc;
    P.tag_period = t1_tag_period(dev);
    P.tag_step = P.tag_period / (unsigned long long)Gt;
    P.mP64 = ~0ull / P.tag_period + 1ull;
    const bool e4 = d.kind == NVFP4_SCALE_E4M3;
    cudaError_t err = e4 ? prepare_t1c<NVFP4_SCALE_E4M3>(dev.device, L.total)
                         : prepare_t1c<NVFP4_SCALE_FP16>(dev.device, L.total);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(Gt);
    cfg.blockDim = dim3(kCThr);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return e4 ? cudaLaunchKernelEx(&cfg, moe_decode_t1c_kernel<NVFP4_SCALE_E4M3>, P)
              : cudaLaunchKernelEx(&cfg, moe_decode_t1c_kernel<NVFP4_SCALE_FP16>, P);
}

}  // namespace nvfp4
