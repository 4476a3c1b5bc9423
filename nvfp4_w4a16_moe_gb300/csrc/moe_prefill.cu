// MoE layer for prefill-sized batches (T > 64 tokens): the same layer as the
// decode kernels, reorganised as grouped GEMMs because at this size every
// projection is a dense contraction.
//
// Sources (page title, section):
//  - lynn-engine README, P2/P3-A notes (grouped MoE prefill: the routed active
//    path run as batched projections), P28/P29 notes (gate/up + SiLU -> [top_k, I]
//    intermediate, then down + routing-weighted sum), P46/P48 notes (no float
//    atomics in the combine); README "next steps" (CUTLASS-style grouped GEMM).
//  - lynn-engine tutorials index, row 06 (softmax over all experts -> top-k ->
//    renormalise; sigmoid-gated shared expert).
//
// Pipeline (one stream, deterministic):
//   1. router GEMM      logits[T, E] and the gate pre-activation = x [T,H] . [Wg; gs]^T
//   2. top-k            per token (route_topk_kernel)
//   3. expert lists     stable counting sort of the T*k entries by expert (three
//                       grid-wide passes: per-block histograms, one scan, placement)
//   4. gate/up GEMM     per active expert and for the shared expert: [n_e, H] x
//                       [2I, H]^T with the SiLU(gate) * up epilogue -> h (bf16,
//                       rows in expert-sorted order)
//   5. down GEMM        h [n_e, I] x D_e [H, I]^T -> one fp32 row per (token, slot)
//   6. combine          y[t] = sum_j w_tj ts_j Y[t, j] + sigmoid(g_t) ts_s Ys[t], fixed order
//
// The GEMMs run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
// accumulate). NVFP4 weight tiles are dequantised into shared memory as bf16:
// an E2M1 value (at most 2 significant bits) times an E4M3 block scale (at most
// 4) has at most 6 significant bits and
// lies in [2^-10, 2688], so it is exact in bf16; the fp32 tensor scale is applied
// in the epilogue. Activations stay bf16.
#include "common.cuh"
#include "kernels.cuh"

namespace nvfp4 {

namespace {

// ------------------------------------------------------------------ GEMM core
// Block tile 128 (rows of A: tokens) x 128 (rows of B: weight rows), K step 32,
// 8 warps as 2 (M) x 4 (N), warp tile 64 x 32, two shared-memory stages.
constexpr int kBM = 128, kBN = 128, kBK = 32;
constexpr int kGThreads = 256;
constexpr int kLds = kBK + 8;   // shared row stride in bf16 elements (80 bytes: ldmatrix rows hit distinct banks)

__device__ __forceinline__ uint32_t cvta_shared(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(cvta_shared(p)));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16-byte global -> shared copy; src_bytes = 0 fills the destination with zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(cvta_shared(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Sixteen E2M1 codes (8 bytes) times one E4M3 block scale -> sixteen bf16 (exact).
__device__ __forceinline__ uint4 dequant16_bf16(uint2 codes, float scale, uint4* hi) {
    uint32_t out[8];
    const uint32_t w[2] = {codes.x, codes.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float2 v = e2m1x2_to_f32x2(w[i] >> (8 * b));
            uint32_t p;
            asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(p) : "f"(v.y * scale), "f"(v.x * scale));
            out[4 * i + b] = p;
        }
    }
    *hi = make_uint4(out[4], out[5], out[6], out[7]);
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// Per-thread sources of one 128 x 128 tile. Thread `tid` stages A rows tid/4 and
// tid/4 + 64 (16-byte part tid%4 of each 64-byte K step); for a bf16 B it stages B
// rows tid/4 and tid/4 + 64 the same way, for an NVFP4 B the 16-element half tid%2
// of B row tid/2.
struct TileSrc {
    const uint16_t* a[2];    // bf16 A rows (K elements), nullptr: zero row
    const uint16_t* bh[2];   // bf16 B rows (K elements), nullptr: zero row
    const uint8_t* bq;       // NVFP4 B row: K/2 bytes of codes, nullptr: zero row
    const uint8_t* bs;       // its K/16 E4M3 block scales
    const void* dummy;       // a valid global address, source of zero-filled copies
};

// acc += A_tile . B_tile^T over K (K % 32 == 0); the caller owns the epilogue.
template <bool kNvfp4>
__device__ __forceinline__ void gemm_tile(const TileSrc& S, int K, float (&acc)[4][4][4], uint16_t* As,
                                          uint16_t* Bs) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp >> 2, wn = warp & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.f;

    const int nk = K / kBK;
    const int lr = tid >> 2, part = tid & 3;
    auto load_A = [&](int kt, int st) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint16_t* src = S.a[c];
            cp_async16(As + ((size_t)st * kBM + lr + 64 * c) * kLds + part * 8,
                       src ? (const void*)(src + kt * kBK + part * 8) : S.dummy, src ? 16u : 0u);
        }
    };
    auto load_Bh = [&](int kt, int st) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint16_t* src = S.bh[c];
            cp_async16(Bs + ((size_t)st * kBN + lr + 64 * c) * kLds + part * 8,
                       src ? (const void*)(src + kt * kBK + part * 8) : S.dummy, src ? 16u : 0u);
        }
    };
    const int bn = tid >> 1, bh = tid & 1;
    uint2 braw = make_uint2(0, 0);
    uint32_t bsc = 0;
    auto fetch_Bq = [&](int kt) {
        if (S.bq) {
            braw = __ldg(reinterpret_cast<const uint2*>(S.bq + kt * (kBK / 2) + bh * 8));
            bsc = __ldg(S.bs + kt * (kBK / 16) + bh);
        }
    };
    auto store_Bq = [&](int st) {
        uint4 hi;
        const uint4 lo = dequant16_bf16(braw, e4m3_to_f32(bsc), &hi);
        uint4* dst = reinterpret_cast<uint4*>(Bs + ((size_t)st * kBN + bn) * kLds + bh * 16);
        dst[0] = lo;
        dst[1] = hi;
    };

    load_A(0, 0);
    if (kNvfp4) { fetch_Bq(0); store_Bq(0); } else load_Bh(0, 0);
    cp_async_commit();
    for (int kt = 0; kt < nk; ++kt) {
        const int st = kt & 1;
        cp_async_wait_all();
        __syncthreads();
        if (kt + 1 < nk) {
            load_A(kt + 1, st ^ 1);
            if (kNvfp4) fetch_Bq(kt + 1); else load_Bh(kt + 1, st ^ 1);
            cp_async_commit();
        }
#pragma unroll
        for (int kk = 0; kk < kBK; kk += 16) {
            uint32_t af[4][4], bfr[2][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = wm * 64 + i * 16 + (lane & 15);
                ldsm_x4(af[i], As + ((size_t)st * kBM + r) * kLds + kk + (lane >> 4) * 8);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int n = wn * 32 + j * 16 + ((lane >> 4) << 3) + (lane & 7);
                ldsm_x4(bfr[j], Bs + ((size_t)st * kBN + n) * kLds + kk + ((lane >> 3) & 1) * 8);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_bf16(acc[i][j], af[i], bfr[j >> 1][(j & 1) * 2], bfr[j >> 1][(j & 1) * 2 + 1]);
        }
        if (kNvfp4 && kt + 1 < nk) store_Bq(st ^ 1);
    }
    __syncthreads();
}

// Accumulator element (i, j, q) of this thread sits at tile row / column:
__device__ __forceinline__ int acc_row(int i, int q) {
    return ((threadIdx.x >> 5) >> 2) * 64 + i * 16 + ((threadIdx.x & 31) >> 2) + (q >> 1) * 8;
}
__device__ __forceinline__ int acc_col(int j, int q) {
    return ((threadIdx.x >> 5) & 3) * 32 + j * 8 + (threadIdx.x & 3) * 2 + (q & 1);
}

// ------------------------------------------------------------------ kernels
// 1. router: logits[t, e] = x[t] . Wg[e] as one bf16 GEMM, K split in blockIdx.z parts
//    of kc elements (each writes its own partial slice; router_sum_kernel adds them in a
//    fixed order); grid = (ceil(T/128), ceil(E/128), splits).
__global__ void __launch_bounds__(kGThreads) router_gemm_kernel(const uint16_t* __restrict__ x, int T, int H,
                                                              const uint16_t* __restrict__ wg, int E, int kc,
                                                              float* __restrict__ logits) {
    extern __shared__ __align__(128) uint16_t gsm[];
    uint16_t* As = gsm;
    uint16_t* Bs = gsm + 2 * kBM * kLds;
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN, k0 = blockIdx.z * kc;
    const int tid = threadIdx.x;
    logits += (size_t)blockIdx.z * T * E;
    TileSrc S{};
    S.dummy = x;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int r = (tid >> 2) + 64 * c;
        S.a[c] = m0 + r < T ? x + (size_t)(m0 + r) * H + k0 : nullptr;
        S.bh[c] = n0 + r < E ? wg + (size_t)(n0 + r) * H + k0 : nullptr;
    }
    float acc[4][4][4];
    gemm_tile<false>(S, kc, acc, As, Bs);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int r = acc_row(i, q), c = acc_col(j, q);
                if (m0 + r < T && n0 + c < E) logits[(size_t)(m0 + r) * E + n0 + c] = acc[i][j][q];
            }
}

// logits = sum of the router's K-split partial slices, in split order (in place in slice 0).
__global__ void router_sum_kernel(float* __restrict__ logits, int n4, int splits, size_t slice4) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    float4* p = reinterpret_cast<float4*>(logits);
    float4 a = p[i];
    for (int sp = 1; sp < splits; ++sp) {
        const float4 v = p[i + sp * slice4];
        a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
    }
    p[i] = a;
}

// The gate pre-activation sigma_t = x_t . gs for every token (one warp per token).
__global__ void gate_dot_kernel(const uint16_t* __restrict__ x, int T, int H, const uint16_t* __restrict__ gs,
                                float* __restrict__ gate) {
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= T) return;
    float acc = 0.f;
    for (int c = lane; c < H / 8; c += 32) {
        const uint4 a = *reinterpret_cast<const uint4*>(x + (size_t)t * H + 8 * c);
        const uint4 b = *reinterpret_cast<const uint4*>(gs + 8 * c);
        const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc = fmaf(bf16lo(aa[q]), bf16lo(bb[q]), acc);
            acc = fmaf(bf16hi(aa[q]), bf16hi(bb[q]), acc);
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) gate[t] = acc;
}

// 3. expert lists for large T: stable counting sort of the T*k entries by expert.
//    pass 1: histogram of each block of 1024 entries -> bcount[block][E]
constexpr int kLB = 1024;
__global__ void __launch_bounds__(kLB) lists_hist_kernel(const int32_t* __restrict__ ids, int total, int E,
                                                        int32_t* __restrict__ bcount) {
    __shared__ int cnt[NVFP4_MAX_EXPERTS];
    for (int e = threadIdx.x; e < E; e += kLB) cnt[e] = 0;
    __syncthreads();
    const int i = blockIdx.x * kLB + threadIdx.x;
    if (i < total) atomicAdd(&cnt[ids[i]], 1);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kLB) bcount[(size_t)blockIdx.x * E + e] = cnt[e];
}

//    pass 2 (one block): bases of every (expert, block) in expert-major order, the
//    per-expert offsets, and the prefix of kTokTile-row tiles per slot (E experts, then
//    the shared expert with T rows) used to schedule the grouped GEMMs
__global__ void __launch_bounds__(NVFP4_MAX_EXPERTS) lists_scan_kernel(int32_t* __restrict__ bcount, int nblocks,
                                                                      int E, int shared_rows,
                                                                      int32_t* __restrict__ offsets,
                                                                      int32_t* __restrict__ tile_prefix) {
    __shared__ int tot[NVFP4_MAX_EXPERTS];
    const int e = threadIdx.x;
    int s = 0;
    if (e < E) {
        for (int b = 0; b < nblocks; ++b) {   // exclusive prefix inside expert e, over blocks
            const int c = bcount[(size_t)b * E + e];
            bcount[(size_t)b * E + e] = s;
            s += c;
        }
        tot[e] = s;
    }
    __syncthreads();
    if (e == 0) {
        int run = 0, mt = 0;
        for (int x = 0; x < E; ++x) {
            offsets[x] = run;
            tile_prefix[x] = mt;
            run += tot[x];
            mt += (tot[x] + kTokTile - 1) / kTokTile;
        }
        offsets[E] = run;
        tile_prefix[E] = mt;
        tile_prefix[E + 1] = mt + (shared_rows + kTokTile - 1) / kTokTile;   // the shared expert: every token
    }
    __syncthreads();
    if (e < E) {
        const int base = offsets[e];
        for (int b = 0; b < nblocks; ++b) bcount[(size_t)b * E + e] += base;
    }
}

//    pass 3: place every entry at bcount[block][e] + (its rank among the block's
//    entries of expert e)
__global__ void __launch_bounds__(kLB) lists_place_kernel(const int32_t* __restrict__ ids, int total, int E,
                                                         const int32_t* __restrict__ bbase,
                                                         int32_t* __restrict__ token_list) {
    __shared__ int wcnt[kLB / 32][NVFP4_MAX_EXPERTS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < (kLB / 32) * E; i += kLB) wcnt[i / E][i % E] = 0;
    __syncthreads();
    const int idx = blockIdx.x * kLB + tid;
    const int e = idx < total ? ids[idx] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank_w = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && rank_w == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    for (int ee = tid; ee < E; ee += kLB) {
        int pre = 0;
        for (int w = 0; w < kLB / 32; ++w) {
            const int c = wcnt[w][ee];
            wcnt[w][ee] = pre;
            pre += c;
        }
    }
    __syncthreads();
    if (e >= 0) {
        const int pos = bbase[(size_t)blockIdx.x * E + e] + wcnt[warp][e] + rank_w;
        token_list[pos] = idx;
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 6. combine: y[t] = sum over the token's k routed rows, then the shared row, in
//    that fixed order; one thread per 4 output features.
__global__ void combine_kernel(const float* __restrict__ Y, int T, int H, int k, int n_slots,
                               const uint16_t* __restrict__ resid, uint16_t* __restrict__ y) {
    const size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int q = H / 4;
    if (g >= (size_t)T * q) return;
    const int t = (int)(g / q), c = (int)(g - (size_t)t * q) * 4;
    const float* src = Y + (size_t)t * (k + 1) * H + c;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < n_slots; ++j) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(src + (size_t)j * H));
        a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
    }
    if (resid) {   // the residual stream, added before the one rounding
        const uint2 r = *reinterpret_cast<const uint2*>(resid + (size_t)t * H + c);
        a.x += bf16lo(r.x); a.y += bf16hi(r.x); a.z += bf16lo(r.y); a.w += bf16hi(r.y);
    }
    uint2 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    *reinterpret_cast<uint2*>(y + (size_t)t * H + c) = o;
}

size_t align256p(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

// The grouped tcgen05 GEMMs read the weights through TMA tensor maps whose row
// strides (K/16 bytes for the scales) must be multiples of 16: H, I and Is
// multiples of 256, E4M3 scales (their products with E2M1 values are exact in bf16).
// K splits of the router GEMM (so that its grid covers the SMs at 4096 tokens); each split
// is a multiple of the 32-element K step, and the partial slices must stay 16-byte
// aligned for the float4 sum (T*E a multiple of 4).
int router_splits(int H, int T, int E) {
    if (((size_t)T * E) % 4 != 0) return 1;
    return (H / 32) % 4 == 0 ? 4 : ((H / 32) % 2 == 0 ? 2 : 1);
}

bool prefill_supported(const moe_layer_desc& d, int T) {
    return T > NVFP4_DECODE_MAX_TOKENS && d.kind == NVFP4_SCALE_E4M3 && d.H % 256 == 0 && d.I % 256 == 0 &&
           d.Is % 256 == 0;
}

size_t prefill_ws_bytes(const moe_layer_desc& d, int T) {
    const size_t Tk = (size_t)T * d.k;
    const size_t nb = (Tk + kLB - 1) / kLB;
    size_t b = sizeof(WsHeader);
    b += align256p(sizeof(float) * (size_t)T * d.E * router_splits(d.H, T, d.E));   // logits (split partials)
    b += align256p(sizeof(float) * (size_t)T);                  // gate
    b += align256p(sizeof(int32_t) * Tk);                       // ids
    b += align256p(sizeof(float) * Tk);                         // w
    b += align256p(sizeof(int32_t) * nb * d.E);                 // bcount
    b += align256p(sizeof(int32_t) * (size_t)(d.E + 1));        // offsets
    b += align256p(sizeof(int32_t) * (size_t)(d.E + 2));        // tile_prefix
    b += align256p(sizeof(int32_t) * Tk);                       // token_list
    b += align256p(sizeof(uint16_t) * Tk * d.I);                // h
    b += align256p(sizeof(uint16_t) * (size_t)T * d.Is);        // hs
    b += align256p(sizeof(float) * (size_t)T * (d.k + 1) * d.H); // Y
    return b;
}

PrefillWs carve_prefill_ws(void* base, const moe_layer_desc& d, int T) {
    PrefillWs w;
    const size_t Tk = (size_t)T * d.k;
    const size_t nb = (Tk + kLB - 1) / kLB;
    char* p = static_cast<char*>(base);
    auto take = [&](size_t bytes) { char* r = p; p += align256p(bytes); return r; };
    w.hdr = reinterpret_cast<WsHeader*>(p); p += sizeof(WsHeader);
    w.logits = reinterpret_cast<float*>(take(sizeof(float) * (size_t)T * d.E * router_splits(d.H, T, d.E)));
    w.gate = reinterpret_cast<float*>(take(sizeof(float) * (size_t)T));
    w.ids = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * Tk));
    w.w = reinterpret_cast<float*>(take(sizeof(float) * Tk));
    w.bcount = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * nb * d.E));
    w.offsets = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (size_t)(d.E + 1)));
    w.tile_prefix = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (size_t)(d.E + 2)));
    w.token_list = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * Tk));
    w.h = reinterpret_cast<uint16_t*>(take(sizeof(uint16_t) * Tk * d.I));
    w.hs = reinterpret_cast<uint16_t*>(take(sizeof(uint16_t) * (size_t)T * d.Is));
    w.Y = reinterpret_cast<float*>(take(sizeof(float) * (size_t)T * (d.k + 1) * d.H));
    w.bytes = (size_t)(p - static_cast<char*>(base));
    return w;
}

int prefill_launch_count(const moe_layer_desc& d, int T) {
    return (d.Is > 0 ? 9 : 8) + (router_splits(d.H, T, d.E) > 1 ? 1 : 0);
}

cudaError_t launch_moe_prefill(const moe_layer_desc& d, const uint16_t* x, int T, uint16_t* y,
                               int32_t* ids_out, float* w_out, const PrefillWs& ws, uint64_t wait_limit,
                               cudaStream_t s, const uint16_t* resid) {
    const int E = d.E, k = d.k, H = d.H;
    const int total = T * k;
    int32_t* ids = ids_out ? ids_out : ws.ids;
    float* w = w_out ? w_out : ws.w;
    cudaError_t err;
    // 1. router logits (+ the shared gate pre-activation)
    {
        const dim3 grid((T + kBM - 1) / kBM, (E + kBN - 1) / kBN);
        const int splits = router_splits(H, T, E);
        const dim3 gridk(grid.x, grid.y, splits);
        router_gemm_kernel<<<gridk, kGThreads, 4 * kBM * kLds * sizeof(uint16_t), s>>>(x, T, H, d.router_w, E,
                                                                                       H / splits, ws.logits);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
        if (splits > 1) {
            const int n4 = T * E / 4;
            router_sum_kernel<<<(n4 + 255) / 256, 256, 0, s>>>(ws.logits, n4, splits, (size_t)T * E / 4);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
        }
        if (d.Is > 0) {
            gate_dot_kernel<<<(T + 7) / 8, 256, 0, s>>>(x, T, H, d.sh_gate_w, ws.gate);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
        }
    }
    // 2. softmax, top-k, renormalise
    if ((err = launch_route_topk(ws.logits, T, E, k, ids, w, s)) != cudaSuccess) return err;
    // 3. stable per-expert lists and the tile prefix
    const int nb = (total + kLB - 1) / kLB;
    lists_hist_kernel<<<nb, kLB, 0, s>>>(ids, total, E, ws.bcount);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    lists_scan_kernel<<<1, NVFP4_MAX_EXPERTS, 0, s>>>(ws.bcount, nb, E, d.Is > 0 ? T : 0, ws.offsets,
                                                       ws.tile_prefix);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    lists_place_kernel<<<nb, kLB, 0, s>>>(ids, total, E, ws.bcount, ws.token_list);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;

    GroupedParams P{};
    P.x = x; P.T = T; P.H = H; P.E = E; P.k = k; P.I = d.I; P.Is = d.Is;
    P.gu_packed = d.gu_packed; P.gu_scales = static_cast<const uint8_t*>(d.gu_scales); P.gu_tscale = d.gu_tscale;
    P.dn_packed = d.dn_packed; P.dn_scales = static_cast<const uint8_t*>(d.dn_scales); P.dn_tscale = d.dn_tscale;
    P.sh_gu_packed = d.sh_gu_packed; P.sh_gu_scales = static_cast<const uint8_t*>(d.sh_gu_scales);
    P.sh_gu_tscale = d.sh_gu_tscale;
    P.sh_dn_packed = d.sh_dn_packed; P.sh_dn_scales = static_cast<const uint8_t*>(d.sh_dn_scales);
    P.sh_dn_tscale = d.sh_dn_tscale;
    P.offsets = ws.offsets; P.token_list = ws.token_list; P.tile_prefix = ws.tile_prefix;
    P.w = w; P.gate = ws.gate; P.h = ws.h; P.hs = ws.hs; P.Y = ws.Y;
    // upper bound on the number of token tiles: every non-empty expert adds at most
    // one partial tile
    const int nonempty = min(E, total);
    const long long tiles_max = ((long long)total + (long long)(kTokTile - 1) * nonempty) / kTokTile +
                                (d.Is > 0 ? (T + kTokTile - 1) / kTokTile : 0);
    // 4. gate/up + SwiGLU, 5. down scaled into Y
    if ((err = launch_grouped_tc(P, 0, (int)tiles_max, ws.hdr, wait_limit, s)) != cudaSuccess) return err;
    if ((err = launch_grouped_tc(P, 1, (int)tiles_max, ws.hdr, wait_limit, s)) != cudaSuccess) return err;
    // 6. combine
    {
        const size_t n = (size_t)T * (H / 4);
        combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(ws.Y, T, H, k, k + (d.Is > 0 ? 1 : 0), resid, y);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace nvfp4
