// MoE layer, multi-token decode path on fp32 FMA (T <= 64) for the layers the
// tensor-core path in decode_mma.cu does not take (FP16 block scales, or H / I /
// Is off the multiple-of-256 grid): router GEMV, route, grouped gate/up + SiLU,
// down + routing-weighted combine + sigmoid-gated shared expert. This file also
// owns the workspace layout of every T <= 64 call.
//
// Sources (page title, section):
//  - lynn-engine tutorials index, row 06 "MoE router" (softmax-all -> top-k ->
//    renormalise, sigmoid-gated shared expert).
//  - lynn-engine README, P28 note (gate/up + SiLU over the active experts only,
//    [top_k, I] intermediate), P29 note (down + weighted sum -> [H]), P21 note
//    (shared gate/up rows fused into one pass), P46/P48 notes (no float
//    atomics in the combine: every output row is owned by one warp and summed
//    in a fixed order).
//
// The routed and the shared experts go through the same grouped kernels: the
// shared expert is one more "slot" whose token list is every token.
#include "common.cuh"
#include "kernels.cuh"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// ------------------------------------------------------------------ router
// logits[t, e] = x[t] . Wg[e] for e < E; gate_logit[t] = x[t] . gs (row E).
// Warp per row, lane l reads 16-byte chunks l, l+32, ... of the bf16 row; x
// chunk staged in shared memory as raw bf16 (conflict-free 16-byte reads).
constexpr int kRouterTc = 16;

__global__ void __launch_bounds__(kThreads)
router_kernel(const uint16_t* __restrict__ wg, const uint16_t* __restrict__ gs,
              const uint16_t* __restrict__ x, int T, int E, int H,
              float* __restrict__ logits, float* __restrict__ gate_logit) {
    extern __shared__ uint4 xs4[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = H >> 3;                  // 16-byte chunks per row
    const int rows = E + (gs ? 1 : 0);
    const int warps_total = gridDim.x * kWarps;
    for (int t0 = 0; t0 < T; t0 += kRouterTc) {
        const int tc = min(kRouterTc, T - t0);
        __syncthreads();
        for (int i = threadIdx.x; i < tc * nch; i += kThreads)
            xs4[i] = *reinterpret_cast<const uint4*>(x + (size_t)t0 * H + 8 * (size_t)i);
        __syncthreads();
        for (int r = blockIdx.x * kWarps + warp; r < rows; r += warps_total) {
            const uint16_t* row = r < E ? wg + (size_t)r * H : gs;
            float acc[kRouterTc];
#pragma unroll
            for (int t = 0; t < kRouterTc; ++t) acc[t] = 0.f;
            for (int c = lane; c < nch; c += 32) {
                const uint4 wv = *reinterpret_cast<const uint4*>(row + 8 * (size_t)c);
                const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                for (int t = 0; t < kRouterTc; ++t) {
                    if (t < tc) {
                        const uint4 xv = xs4[t * nch + c];
                        const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
                        float a = acc[t];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            a = fmaf(bf16lo(ww[q]), bf16lo(xx[q]), a);
                            a = fmaf(bf16hi(ww[q]), bf16hi(xx[q]), a);
                        }
                        acc[t] = a;
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kRouterTc; ++t) {
                if (t < tc) {
                    const float v = warp_sum(acc[t]);
                    if (lane == 0) {
                        if (r < E) logits[(size_t)(t0 + t) * E + r] = v;
                        else gate_logit[t0 + t] = v;
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------------ gate/up
// Work item = (slot, block of kPairRows intermediate rows). Slots 0..A-1 are the
// active routed experts in ascending id, slot A the shared expert (if any).
// For every token of the slot and every row i: h = silu(ts_g * G[i].x) * (ts_u * U[i].x).
constexpr int kPairRows = 32;   // pair-rows (gate row i + up row i) per item
constexpr int kGuTc = 8;        // tokens per staged chunk
constexpr int kMaxSegH = 8;     // H <= 8192 (H/32 segments, <= 8 per lane)

struct SlotInfo {
    const uint8_t* packed;  // [2*Irows, H/2]
    const uint8_t* scales;  // [2*Irows, H/16 * sbytes]
    float ts_g, ts_u;
    int Irows;
    int ntok;
    const int32_t* list;    // routed: entries (t*k + j); shared: nullptr (tokens 0..T-1)
    float* hout;            // routed: h (entry-major), shared: hs (token-major)
};

template <int KIND>
__device__ __forceinline__ void scales2(const uint8_t* srow, int s, float& s0, float& s1) {
    seg_scales<KIND>(srow, s, s0, s1);
}

// x[t] (bf16) for the chunk's tokens -> xs[tt][c][s][4] fp32 (segment-interleaved)
__device__ void stage_tokens(float* xs, const uint16_t* __restrict__ x, const int* tok, int tc,
                             int H) {
    const int nseg = H >> 5, q4 = H >> 2;
    for (int i = threadIdx.x; i < tc * q4; i += blockDim.x) {
        const int tt = i / q4, e4 = i - tt * q4;
        const int s = e4 >> 3, c = e4 & 7;
        const uint2 raw = *reinterpret_cast<const uint2*>(x + (size_t)tok[tt] * H + 4 * e4);
        reinterpret_cast<float4*>(xs)[(size_t)tt * q4 + c * nseg + s] =
            make_float4(bf16lo(raw.x), bf16hi(raw.x), bf16lo(raw.y), bf16hi(raw.y));
    }
}

// sum over one 32-element segment against staged activations of token tt
__device__ __forceinline__ float seg_dot(const float* q, const float4* xt, int nseg, int s,
                                         float s0, float s1) {
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
    return fmaf(s0, p0, s1 * p1);
}

template <int KIND>
__global__ void __launch_bounds__(kThreads)
gateup_kernel(moe_layer_desc d, const uint16_t* __restrict__ x, int T, const int32_t* offsets,
              const int32_t* token_list, const int32_t* active, float* h, float* hs) {
    extern __shared__ float4 gsm[];
    float* xs = reinterpret_cast<float*>(gsm);
    __shared__ int tok[kGuTc];
    __shared__ int ent[kGuTc];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = d.H, nseg = H >> 5;
    constexpr int kind = KIND;
    const int A = active[0];
    const int ib_r = (d.I + kPairRows - 1) / kPairRows;
    const int ib_s = d.Is > 0 ? (d.Is + kPairRows - 1) / kPairRows : 0;
    const int n_items = A * ib_r + ib_s;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        SlotInfo si;
        int rb;
        if (item < A * ib_r) {
            const int slot = item / ib_r;
            rb = item - slot * ib_r;
            const int e = active[1 + slot];
            si.Irows = d.I;
            si.packed = d.gu_packed + (size_t)e * 2 * d.I * (H / 2);
            si.scales = static_cast<const uint8_t*>(d.gu_scales) + (size_t)e * 2 * d.I * scale_row_bytes_of(kind, H);
            si.ts_g = __ldg(d.gu_tscale + 2 * e);
            si.ts_u = __ldg(d.gu_tscale + 2 * e + 1);
            si.list = token_list + offsets[e];
            si.ntok = offsets[e + 1] - offsets[e];
            si.hout = h;
        } else {
            rb = item - A * ib_r;
            si.Irows = d.Is;
            si.packed = d.sh_gu_packed;
            si.scales = static_cast<const uint8_t*>(d.sh_gu_scales);
            si.ts_g = __ldg(d.sh_gu_tscale);
            si.ts_u = __ldg(d.sh_gu_tscale + 1);
            si.list = nullptr;
            si.ntok = T;
            si.hout = hs;
        }
        const int Ir = si.Irows;
        for (int c0 = 0; c0 < si.ntok; c0 += kGuTc) {
            const int tc = min(kGuTc, si.ntok - c0);
            __syncthreads();
            if (threadIdx.x < tc) {
                const int en = si.list ? si.list[c0 + threadIdx.x] : c0 + threadIdx.x;
                ent[threadIdx.x] = en;
                tok[threadIdx.x] = si.list ? en / d.k : en;
            }
            __syncthreads();
            stage_tokens(xs, x, tok, tc, H);
            __syncthreads();
            for (int pr = warp; pr < kPairRows; pr += kWarps) {
                const int i = rb * kPairRows + pr;
                if (i >= Ir) break;
                const uint8_t* grow = si.packed + (size_t)i * (H / 2);
                const uint8_t* urow = si.packed + (size_t)(Ir + i) * (H / 2);
                const uint8_t* gsc = si.scales + (size_t)i * scale_row_bytes_of(kind, H);
                const uint8_t* usc = si.scales + (size_t)(Ir + i) * scale_row_bytes_of(kind, H);
                float ga[kGuTc], ua[kGuTc];
#pragma unroll
                for (int t = 0; t < kGuTc; ++t) { ga[t] = 0.f; ua[t] = 0.f; }
#pragma unroll
                for (int m = 0; m < kMaxSegH; ++m) {
                    const int s = lane + 32 * m;
                    if (s < nseg) {
                        const uint4 gw = *reinterpret_cast<const uint4*>(grow + 16 * (size_t)s);
                        const uint4 uw = *reinterpret_cast<const uint4*>(urow + 16 * (size_t)s);
                        float g0, g1, u0, u1;
                        scales2<KIND>(gsc, s, g0, g1);
                        scales2<KIND>(usc, s, u0, u1);
                        float qg[32], qu[32];
                        dequant32(gw, qg);
                        dequant32(uw, qu);
#pragma unroll
                        for (int t = 0; t < kGuTc; ++t) {
                            if (t < tc) {
                                const float4* xt = reinterpret_cast<const float4*>(xs) + (size_t)t * (H >> 2);
                                ga[t] += seg_dot(qg, xt, nseg, s, g0, g1);
                                ua[t] += seg_dot(qu, xt, nseg, s, u0, u1);
                            }
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < kGuTc; ++t) {
                    if (t < tc) {
                        const float g = warp_sum(ga[t]) * si.ts_g;
                        const float u = warp_sum(ua[t]) * si.ts_u;
                        if (lane == 0) si.hout[(size_t)ent[t] * Ir + i] = silu_f32(g) * u;
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------------------ down + combine
// Warp per (output row n, token t). Lane work: the (entry j, segment s) pairs of
// the routed experts then the shared expert's segments, in a fixed mapping, so
// the reduction order never changes. y[t,n] = sum_j w_j ts_j D_j[n].h_j + sig_t ts_s Ds[n].hs
constexpr int kMaxSegI = 16;    // I, Is <= 512 per 32-lane pass is covered by the loop

template <int KIND>
__global__ void __launch_bounds__(kThreads)
down_kernel(moe_layer_desc d, int T, const int32_t* __restrict__ ids, const float* __restrict__ wts,
            const float* __restrict__ gate_logit, const float* __restrict__ h,
            const float* __restrict__ hs, const uint16_t* __restrict__ resid, uint16_t* __restrict__ y) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = d.H, I = d.I, Is = d.Is, k = d.k;
    constexpr int kind = KIND;
    const int nseg_r = I >> 5, nseg_s = Is >> 5;
    const int work_r = k * nseg_r;
    const int work = work_r + nseg_s;
    const long total = (long)H * T;
    for (long item = (long)blockIdx.x * kWarps + warp; item < total; item += (long)gridDim.x * kWarps) {
        const int t = (int)(item / H);
        const int n = (int)(item - (long)t * H);
        float acc_r = 0.f, acc_s = 0.f;
        for (int p = lane; p < work; p += 32) {
            if (p < work_r) {
                const int j = p / nseg_r, s = p - j * nseg_r;
                const int e = ids[t * k + j];
                const uint8_t* row = d.dn_packed + ((size_t)e * H + n) * (I / 2);
                const uint8_t* srow = static_cast<const uint8_t*>(d.dn_scales) + ((size_t)e * H + n) * scale_row_bytes_of(kind, I);
                const uint4 wv = *reinterpret_cast<const uint4*>(row + 16 * (size_t)s);
                float s0, s1;
                scales2<KIND>(srow, s, s0, s1);
                float q[32];
                dequant32(wv, q);
                const float4* hv = reinterpret_cast<const float4*>(h + (size_t)(t * k + j) * I + 32 * s);
                float p0 = 0.f, p1 = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4 a = hv[c];
                    p0 = fmaf(q[4 * c], a.x, p0); p0 = fmaf(q[4 * c + 1], a.y, p0);
                    p0 = fmaf(q[4 * c + 2], a.z, p0); p0 = fmaf(q[4 * c + 3], a.w, p0);
                }
#pragma unroll
                for (int c = 4; c < 8; ++c) {
                    const float4 a = hv[c];
                    p1 = fmaf(q[4 * c], a.x, p1); p1 = fmaf(q[4 * c + 1], a.y, p1);
                    p1 = fmaf(q[4 * c + 2], a.z, p1); p1 = fmaf(q[4 * c + 3], a.w, p1);
                }
                acc_r = fmaf(wts[t * k + j] * __ldg(d.dn_tscale + e), fmaf(s0, p0, s1 * p1), acc_r);
            } else {
                const int s = p - work_r;
                const uint8_t* row = d.sh_dn_packed + (size_t)n * (Is / 2);
                const uint8_t* srow = static_cast<const uint8_t*>(d.sh_dn_scales) + (size_t)n * scale_row_bytes_of(kind, Is);
                const uint4 wv = *reinterpret_cast<const uint4*>(row + 16 * (size_t)s);
                float s0, s1;
                scales2<KIND>(srow, s, s0, s1);
                float q[32];
                dequant32(wv, q);
                const float4* hv = reinterpret_cast<const float4*>(hs + (size_t)t * Is + 32 * s);
                float p0 = 0.f, p1 = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4 a = hv[c];
                    p0 = fmaf(q[4 * c], a.x, p0); p0 = fmaf(q[4 * c + 1], a.y, p0);
                    p0 = fmaf(q[4 * c + 2], a.z, p0); p0 = fmaf(q[4 * c + 3], a.w, p0);
                }
#pragma unroll
                for (int c = 4; c < 8; ++c) {
                    const float4 a = hv[c];
                    p1 = fmaf(q[4 * c], a.x, p1); p1 = fmaf(q[4 * c + 1], a.y, p1);
                    p1 = fmaf(q[4 * c + 2], a.z, p1); p1 = fmaf(q[4 * c + 3], a.w, p1);
                }
                acc_s += fmaf(s0, p0, s1 * p1);
            }
        }
        acc_r = warp_sum(acc_r);
        acc_s = warp_sum(acc_s);
        if (lane == 0) {
            float v = acc_r;
            if (Is > 0) v = fmaf(sigmoid_f32(gate_logit[t]) * __ldg(d.sh_dn_tscale), acc_s, v);
            if (resid) v += bf16_to_f32(resid[(size_t)t * H + n]);   // residual stream, before the rounding
            y[(size_t)t * H + n] = f32_to_bf16(v);
        }
    }
}

__global__ void write_route_outputs(const int32_t* ids, const float* w, int n, int32_t* ids_out,
                                    float* w_out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        if (ids_out) ids_out[i] = ids[i];
        if (w_out) w_out[i] = w[i];
    }
}

}  // namespace

size_t layer_ws_bytes(const moe_layer_desc& d, int T) {
    const size_t Tk = (size_t)T * d.k;
    size_t b = sizeof(WsHeader);
    b += align256(sizeof(float) * (size_t)T * d.E);
    b += align256(sizeof(float) * (size_t)T);
    b += align256(sizeof(int32_t) * Tk);
    b += align256(sizeof(float) * Tk);
    b += align256(sizeof(int32_t) * (size_t)(d.E + 1));
    b += align256(sizeof(int32_t) * Tk);
    b += align256(sizeof(int32_t) * (size_t)(d.E + 1));
    b += align256(sizeof(float) * Tk * d.I);
    b += align256(sizeof(float) * (size_t)T * d.Is);
    b += align256(sizeof(unsigned long long) * t1_words(d));
    b += align256(sizeof(int32_t) * (Tk + d.E + 2));
    b += align256(sizeof(float) * (Tk + T) * d.H);
    b += align256(sizeof(uint32_t) * (Tk + 2 * (size_t)T));
    return b;
}

LayerWs carve_layer_ws(void* base, const moe_layer_desc& d, int T) {
    LayerWs w;
    const size_t Tk = (size_t)T * d.k;
    char* p = static_cast<char*>(base);
    w.hdr = reinterpret_cast<WsHeader*>(p); p += sizeof(WsHeader);
    w.logits = reinterpret_cast<float*>(p); p += align256(sizeof(float) * (size_t)T * d.E);
    w.gate_logit = reinterpret_cast<float*>(p); p += align256(sizeof(float) * (size_t)T);
    w.ids = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * Tk);
    w.w = reinterpret_cast<float*>(p); p += align256(sizeof(float) * Tk);
    w.offsets = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * (size_t)(d.E + 1));
    w.token_list = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * Tk);
    w.active = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * (size_t)(d.E + 1));
    w.h = reinterpret_cast<float*>(p); p += align256(sizeof(float) * Tk * d.I);
    w.hs = reinterpret_cast<float*>(p); p += align256(sizeof(float) * (size_t)T * d.Is);
    w.words = reinterpret_cast<unsigned long long*>(p);
    p += align256(sizeof(unsigned long long) * t1_words(d));
    w.pass_map = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * (Tk + d.E + 2));
    w.part = reinterpret_cast<float*>(p); p += align256(sizeof(float) * (Tk + T) * d.H);
    w.amax = reinterpret_cast<uint32_t*>(p); p += align256(sizeof(uint32_t) * (Tk + 2 * (size_t)T));
    w.bytes = (size_t)(p - static_cast<char*>(base));
    return w;
}

template <int KIND>
static cudaError_t decode_impl(const moe_layer_desc& d, const uint16_t* x, int T, uint16_t* y,
                               int32_t* ids_out, float* w_out, const LayerWs& ws,
                               const DeviceInfo& dev, cudaStream_t s, const uint16_t* resid) {
    cudaError_t err;
    // 1. router GEMV (+ shared gate pre-activation)
    {
        const int rows = d.E + (d.Is > 0 ? 1 : 0);
        int grid = (rows + kWarps - 1) / kWarps;
        if (grid > dev.num_sms * 2) grid = dev.num_sms * 2;
        const size_t smem = (size_t)min(T, kRouterTc) * d.H * 2;
        err = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        router_kernel<<<grid, kThreads, smem, s>>>(d.router_w, d.Is > 0 ? d.sh_gate_w : nullptr, x, T,
                                                   d.E, d.H, ws.logits, ws.gate_logit);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    // 2. route: top-k + renormalise, then per-expert lists and the active-expert list
    if ((err = launch_route_topk(ws.logits, T, d.E, d.k, ws.ids, ws.w, s)) != cudaSuccess) return err;
    if ((err = launch_route_lists(ws.ids, T * d.k, d.E, ws.offsets, ws.token_list, ws.active, s)) != cudaSuccess)
        return err;
    // 3. grouped gate/up + SiLU*up over the active experts and the shared expert
    {
        const int maxI = d.I > d.Is ? d.I : d.Is;
        const int slots = (d.E < T * d.k ? d.E : T * d.k) + (d.Is > 0 ? 1 : 0);
        int grid = slots * ((maxI + kPairRows - 1) / kPairRows);
        if (grid > dev.num_sms * 2) grid = dev.num_sms * 2;
        const size_t smem = (size_t)min(T, kGuTc) * d.H * 4;
        err = cudaFuncSetAttribute(gateup_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        gateup_kernel<KIND><<<grid, kThreads, smem, s>>>(d, x, T, ws.offsets, ws.token_list, ws.active,
                                                         ws.h, ws.hs);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    // 4. down + combine, row-owned
    {
        const long items = (long)d.H * T;
        long grid = (items + kWarps - 1) / kWarps;
        if (grid > dev.num_sms * 4) grid = dev.num_sms * 4;
        down_kernel<KIND><<<(int)grid, kThreads, 0, s>>>(d, T, ws.ids, ws.w, ws.gate_logit, ws.h, ws.hs, resid, y);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if (ids_out || w_out) {
        const int n = T * d.k;
        write_route_outputs<<<(n + 255) / 256, 256, 0, s>>>(ws.ids, ws.w, n, ids_out, w_out);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    return cudaSuccess;
}

cudaError_t launch_moe_decode(const moe_layer_desc& d, const uint16_t* x, int T, uint16_t* y,
                              int32_t* ids_out, float* w_out, const LayerWs& ws,
                              const DeviceInfo& dev, uint64_t wait_limit, cudaStream_t s,
                              const uint16_t* resid) {
    (void)wait_limit;
    if (decode_mma_supported(d, T)) return launch_moe_decode_mma(d, x, T, y, ids_out, w_out, ws, dev, s, resid);
    switch (d.kind) {
        case NVFP4_SCALE_E4M3: return decode_impl<NVFP4_SCALE_E4M3>(d, x, T, y, ids_out, w_out, ws, dev, s, resid);
        case NVFP4_SCALE_FP16: return decode_impl<NVFP4_SCALE_FP16>(d, x, T, y, ids_out, w_out, ws, dev, s, resid);
        case NVFP4_SCALE_FP32: return decode_impl<NVFP4_SCALE_FP32>(d, x, T, y, ids_out, w_out, ws, dev, s, resid);
        default: return decode_impl<NVFP4_SCALE_UE8M0>(d, x, T, y, ids_out, w_out, ws, dev, s, resid);
    }
}

}  // namespace nvfp4
