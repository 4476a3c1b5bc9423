// Grouped expert GEMMs of the prefill path on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory).
//
// Sources (page title, section):
//  - lynn-engine README, P2/P3-A notes (grouped MoE prefill: the routed active path
//    run as batched projections over each expert's tokens), P28/P29 notes (gate/up
//    + SiLU -> intermediate, then down + routing-weighted sum), README "next steps"
//    (grouped GEMM instead of per-expert launches).
//  - Lynn Engine write-up (zingnex.cn), "1. native NVFP4 support": the weights stay
//    packed in memory; they are expanded only on chip, here tile by tile in shared
//    memory, never as a bf16 copy in global memory.
//
// One CTA computes one tile D[128 weight rows x N tokens] (N <= 256, a multiple
// of 16) of one slot (a routed expert or the shared expert):
//   gate/up (mode 0): two accumulators, gate rows and up rows of 128 intermediate
//     indices, K = H; epilogue h = silu(ts_g G) * (ts_u U) -> bf16 rows of h / hs.
//   down (mode 1): one accumulator, 128 output features, K = I (or Is); epilogue
//     scales by w * ts_d (or sigmoid(gate) * ts_s) and writes fp32 rows of Y.
// Weights are the MMA's A operand (M = 128), tokens its B operand (N = tokens), so
// small experts waste no MMA work on padding and each weight tile is expanded once
// for up to 256 tokens.
//
// Pipeline per CTA (288 threads): warps 0-7 stage the operands of K step kt + S - 1
// with cp.async (token rows into the 128-byte-swizzled B tile, raw NVFP4 bytes into
// a staging area), expand the NVFP4 bytes of step kt to bf16 in the swizzled A tile,
// and arrive on full[kt % S]; warp 8 (one lane) waits on full, issues the MMAs and
// commits them to empty[kt % S]; after the last step it commits to the accumulator
// barrier, and warps 0-7 read TMEM, run the epilogue through shared memory and store
// coalesced rows. Every wait is bounded; a wait that runs out records
// NVFP4_ERR_DEVICE_TIMEOUT and makes every later wait of the CTA give up at once.
//
// NVFP4 -> bf16 expansion (exact): cvt.rn.f16x2.e2m1x2 gives the E2M1 values as
// f16; shifting an f16 bit pattern right by 3 (sign kept in place) reads it as a
// bf16 of the same value times 2^-112; one bf16x2 multiply by (block scale * 2^112)
// restores the scale. Every product has at most 6 significant bits and lies in
// [2^-10, 2688], so no step rounds.
#include "common.cuh"
#include "kernels.cuh"

namespace nvfp4 {

namespace {

constexpr int kM = 128;           // weight rows per accumulator (MMA M)
constexpr int kKS = 64;           // K elements per stage: one 128-byte row of the swizzle atom
constexpr int kProd = 256;        // operand / epilogue threads (warps 0-7)
constexpr int kTcThreads = kProd + 32;

template <int kParts>
struct TcLayout {
    static constexpr int kStages = kParts == 2 ? 3 : 4;
    static constexpr int kA = kParts * kM * 128;               // A tile bytes per stage
    static constexpr int kB = kTokTile * 128;                  // B tile bytes per stage
    static constexpr int kStage = kA + kB;
    static constexpr int kCodeT = kParts == 2 ? 32 : 16;       // raw code bytes per thread per stage
    static constexpr int kRawCodes = kProd * kCodeT;
    static constexpr int kRawStage = kRawCodes + kProd * 4;    // + 4 scale bytes per thread
    static constexpr int kOffRaw = kStages * kStage;
    static constexpr int kOffCols = kOffRaw + kStages * kRawStage;  // per token column: (Y row, scale)
    static constexpr int kOffBar = kOffCols + kTokTile * 8;
    static constexpr int kBytes = kOffBar + (2 * kStages + 1) * 8 + 16;
    static constexpr int kTmemCols = kParts == 2 ? 512 : 256;
    static constexpr int kAccStride = 256;                     // TMEM column offset of the up accumulator
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// generic-proxy writes to shared memory -> visible to the tensor cores' async proxy
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(su32(bar)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// TMEM allocation (one full warp); the allocated base address is written to *slot.
template <int kCols>
__device__ __forceinline__ void tmem_alloc(uint32_t* slot) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(su32(slot)), "n"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <int kCols>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "n"(kCols) : "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle layout
// (8-row x 128-byte atoms, 1024 bytes apart); start address in 16-byte units.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu)      // start address
           | ((uint64_t)1 << 16)                    // leading byte offset (unused for swizzled K-major)
           | ((uint64_t)(1024 >> 4) << 32)          // stride byte offset: next 8-row group
           | ((uint64_t)1 << 46)                    // descriptor version
           | ((uint64_t)2 << 61);                   // swizzle mode: 128-byte
}

// Instruction descriptor of kind::f16: bf16 A and B (both K-major), fp32 D, M x N.
__device__ __forceinline__ uint32_t f16_idesc(int M, int N) {
    return (1u << 4)                                // D format: f32
           | (1u << 7)                              // A format: bf16
           | (1u << 10)                             // B format: bf16
           | ((uint32_t)(N >> 3) << 17)             // N / 8
           | ((uint32_t)(M >> 4) << 24);            // M / 16
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(su32(bar))
                 : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- NVFP4 -> bf16
// Two E4M3 block scales (low 16 bits of `two`) -> two bf16x2 words, each holding
// (scale * 2^112) in both halves.
__device__ __forceinline__ void scale_pair_bf16(uint32_t two, uint32_t& s0, uint32_t& s1) {
    uint32_t h;
    asm("{\n .reg .b16 b;\n cvt.u16.u32 b, %1;\n cvt.rn.f16x2.e4m3x2 %0, b;\n}" : "=r"(h) : "r"(two & 0xFFFFu));
    // scales are non-negative and have 3 mantissa bits, so the shift moves nothing
    // across the halves; +224 in the exponent turns 2^-112 into 2^+112
    const uint32_t t = (h >> 3) + 0x70007000u;
    s0 = __byte_perm(t, 0, 0x1010);
    s1 = __byte_perm(t, 0, 0x3232);
}

// Eight E2M1 codes (one word, element 0 in the low nibble) times a block scale
// prepared by scale_pair_bf16 -> four bf16x2 words (elements 0..7).
__device__ __forceinline__ void expand8(uint32_t w, uint32_t s2, uint32_t (&o)[4]) {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        uint32_t x;
        asm("{\n .reg .b8 c;\n cvt.u8.u32 c, %1;\n cvt.rn.f16x2.e2m1x2 %0, c;\n}" : "=r"(x) : "r"(w >> (8 * b)));
        const uint32_t y = ((x & 0x7FFF7FFFu) >> 3) | (x & 0x80008000u);
        uint32_t r;
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(y), "r"(s2));
        o[b] = r;
    }
}

// ---------------------------------------------------------------- tiles
struct TcTile {
    int slot;     // routed expert, or E for the shared expert
    int p0;       // first row of the tile in the slot's row space
    int n_rows;   // rows (tokens) of the tile, 1..kTokTile
};

// Token tile tt -> slot (binary search over the tile prefix) and its rows.
__device__ __forceinline__ bool locate_tc_tile(const GroupedParams& P, int tt, TcTile* tr) {
    const int nslots = P.E + 1;
    if (tt >= __ldg(P.tile_prefix + nslots)) return false;
    int lo = 0, hi = nslots;   // tile_prefix[0] = 0 <= tt < tile_prefix[nslots]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(P.tile_prefix + mid) <= tt) lo = mid; else hi = mid;
    }
    const int lt = tt - __ldg(P.tile_prefix + lo);
    tr->slot = lo;
    if (lo < P.E) {
        tr->p0 = __ldg(P.offsets + lo) + lt * kTokTile;
        tr->n_rows = min(kTokTile, __ldg(P.offsets + lo + 1) - tr->p0);
    } else {
        tr->p0 = lt * kTokTile;
        tr->n_rows = min(kTokTile, P.T - tr->p0);
    }
    return true;
}

// Bounded wait on an mbarrier phase. A wait that runs out records the timeout and
// raises the CTA's abort flag; once raised, every wait returns at once.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              WsHeader* hdr, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            record_status(hdr, NVFP4_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
    return true;
}

constexpr int kHS = kM + 8;   // bf16 staging row stride of the gate/up epilogue
constexpr int kYS = kM + 4;   // fp32 staging row stride of the down epilogue

// ---------------------------------------------------------------- kernel
template <int kParts>
__global__ void __launch_bounds__(kTcThreads, 1)
grouped_tc_kernel(const GroupedParams P, int n_ft, WsHeader* hdr, unsigned long long wait_limit) {
    using L = TcLayout<kParts>;
    constexpr int S = L::kStages;
    extern __shared__ uint8_t tc_smem_raw[];
    // the swizzle pattern follows shared-memory address bits: align the base to 1024
    uint8_t* sm = tc_smem_raw + ((1024u - (su32(tc_smem_raw) & 1023u)) & 1023u);

    const int ft = blockIdx.x % n_ft, tt = blockIdx.x / n_ft;
    TcTile tr;
    if (!locate_tc_tile(P, tt, &tr)) return;
    const bool shared = tr.slot == P.E;
    const int Fvalid = kParts == 2 ? (shared ? P.Is : P.I) : P.H;   // output features of this GEMM
    const int feat0 = ft * kM;
    if (feat0 >= Fvalid) return;
    const int Kd = kParts == 2 ? P.H : (shared ? P.Is : P.I);
    const int nk = Kd / kKS;
    const int N = (tr.n_rows + 15) & ~15;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::kOffBar);
    uint64_t* empty = full + S;
    uint64_t* accb = empty + S;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int2* cols = reinterpret_cast<int2*>(sm + L::kOffCols);

    if (warp == kProd / 32) {
        if (lane == 0) {
            for (int i = 0; i < S; ++i) {
                mbar_init(&full[i], kProd);
                mbar_init(&empty[i], 1);
            }
            mbar_init(accb, 1);
            *abort_flag = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc<L::kTmemCols>(tmem_slot);
    }
    if (kParts == 1) {
        // per token column of the tile: its row of Y and the epilogue scale
        for (int c = tid; c < tr.n_rows; c += kTcThreads) {
            int t, j;
            float sc;
            if (shared) {
                t = tr.p0 + c;
                j = P.k;
                sc = sigmoid_f32(__ldg(P.gate + t)) * __ldg(P.sh_dn_tscale);
            } else {
                const int idx = __ldg(P.token_list + tr.p0 + c);
                t = idx / P.k;
                j = idx - t * P.k;
                sc = __ldg(P.w + idx) * __ldg(P.dn_tscale + tr.slot);
            }
            cols[c] = make_int2(t * (P.k + 1) + j, __float_as_int(sc));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sm_base = su32(sm);

    if (warp < kProd / 32) {
        // ---------------- operand producers
        const uint8_t* a_codes = nullptr;   // this thread's weight bytes at K step 0
        const uint8_t* a_scales = nullptr;
        if (kParts == 2) {
            const int part = tid >> 7, f = feat0 + (tid & 127);
            if (f < Fvalid) {
                const size_t wrow = (size_t)(part == 0 ? f : Fvalid + f);   // gate rows, then up rows
                const uint8_t* pk = shared ? P.sh_gu_packed : P.gu_packed + (size_t)tr.slot * 2 * P.I * (P.H / 2);
                const uint8_t* sc = shared ? P.sh_gu_scales : P.gu_scales + (size_t)tr.slot * 2 * P.I * (P.H / 16);
                a_codes = pk + wrow * (P.H / 2);
                a_scales = sc + wrow * (P.H / 16);
            }
        } else {
            const int f = feat0 + (tid >> 1);
            if (f < P.H) {
                const uint8_t* pk = shared ? P.sh_dn_packed : P.dn_packed + (size_t)tr.slot * P.H * (P.I / 2);
                const uint8_t* sc = shared ? P.sh_dn_scales : P.dn_scales + (size_t)tr.slot * P.H * (P.I / 16);
                a_codes = pk + (size_t)f * (Kd / 2) + (tid & 1) * 16;
                a_scales = sc + (size_t)f * (Kd / 16);
            }
        }
        // token rows: 16-byte chunk (tid & 7) of rows (tid >> 3) + 32 j
        const uint16_t* brow[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int row = (tid >> 3) + 32 * j;
            brow[j] = nullptr;
            if (row < tr.n_rows) {
                if (kParts == 2) {
                    const int tok = shared ? tr.p0 + row : __ldg(P.token_list + tr.p0 + row) / P.k;
                    brow[j] = P.x + (size_t)tok * P.H;
                } else {
                    brow[j] = (shared ? P.hs : P.h) + (size_t)(tr.p0 + row) * Kd;
                }
            }
        }
        const int bc = tid & 7;

        auto issue = [&](int s) {
            const int st = s % S;
            const uint32_t bt = sm_base + st * L::kStage + L::kA;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int row = (tid >> 3) + 32 * j;
                if (row < N) {
                    const uint32_t dst = bt + row * 128 + ((bc ^ (row & 7)) << 4);
                    if (brow[j]) cp_async16_zfill(dst, brow[j] + s * kKS + bc * 8, 16u);
                    else cp_async16_zfill(dst, P.x, 0u);
                }
            }
            if (a_codes) {
                const uint32_t raw = sm_base + L::kOffRaw + st * L::kRawStage;
                const uint32_t cd = raw + tid * L::kCodeT;
                cp_async16_zfill(cd, a_codes + s * 32, 16u);
                if (kParts == 2) cp_async16_zfill(cd + 16, a_codes + s * 32 + 16, 16u);
                cp_async4(raw + L::kRawCodes + tid * 4, a_scales + s * 4);
            }
            cp_async_commit_group();
        };

        auto expand = [&](int kt) {
            const int st = kt % S;
            uint8_t* stage = sm + st * L::kStage;
            const uint8_t* raw = sm + L::kOffRaw + st * L::kRawStage;
            if (kParts == 2) {
                const int r = tid & 127;
                uint8_t* arow = stage + (tid >> 7) * (kM * 128) + r * 128;
                if (a_codes) {
                    const uint4 c0 = *reinterpret_cast<const uint4*>(raw + tid * 32);
                    const uint4 c1 = *reinterpret_cast<const uint4*>(raw + tid * 32 + 16);
                    const uint32_t sw = *reinterpret_cast<const uint32_t*>(raw + L::kRawCodes + tid * 4);
                    uint32_t sc[4];
                    scale_pair_bf16(sw, sc[0], sc[1]);
                    scale_pair_bf16(sw >> 16, sc[2], sc[3]);
                    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                    for (int c = 0; c < 8; ++c) {   // chunk c = elements 8c..8c+7 of the step, block c/2
                        uint32_t o[4];
                        expand8(words[c], sc[c >> 1], o);
                        *reinterpret_cast<uint4*>(arow + ((c ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(arow + (c << 4)) = make_uint4(0, 0, 0, 0);
                }
            } else {
                const int r = tid >> 1, half = tid & 1;
                uint8_t* arow = stage + r * 128;
                if (a_codes) {
                    const uint4 c0 = *reinterpret_cast<const uint4*>(raw + tid * 16);
                    const uint32_t sw = *reinterpret_cast<const uint32_t*>(raw + L::kRawCodes + tid * 4);
                    uint32_t s0, s1;
                    scale_pair_bf16(sw >> (16 * half), s0, s1);
                    const uint32_t words[4] = {c0.x, c0.y, c0.z, c0.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {   // chunk 4 half + c, block 2 half + c/2
                        uint32_t o[4];
                        expand8(words[c], c < 2 ? s0 : s1, o);
                        const int ch = 4 * half + c;
                        *reinterpret_cast<uint4*>(arow + ((ch ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(arow + ((4 * half + c) << 4)) = make_uint4(0, 0, 0, 0);
                }
            }
        };

#pragma unroll 1
        for (int s = 0; s < S - 1; ++s) {
            if (s < nk) issue(s);
            else cp_async_commit_group();
        }
#pragma unroll 1
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt + S - 1;
            if (s < nk) {
                if (s >= S) wait_or_abort(&empty[s % S], ((s / S) - 1) & 1, abort_flag, hdr, wait_limit);
                issue(s);
            } else {
                cp_async_commit_group();
            }
            cp_async_wait_group<S - 1>();
            expand(kt);
            fence_proxy_async_smem();
            mbar_arrive(&full[kt % S]);
        }

        // ---------------- epilogue: TMEM -> registers -> shared staging -> global
        wait_or_abort(accb, 0, abort_flag, hdr, wait_limit);
        tc_fence_after();
        const int q = warp & 3, c_begin = (warp >> 2) * (kTokTile / 2);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const int f = 32 * q + lane;
        if (kParts == 2) {
            uint16_t* stg = reinterpret_cast<uint16_t*>(sm);
            const float* tsp = shared ? P.sh_gu_tscale : P.gu_tscale + 2 * tr.slot;
            const float tsg = __ldg(tsp), tsu = __ldg(tsp + 1);
#pragma unroll 1
            for (int c0 = c_begin; c0 < c_begin + kTokTile / 2 && c0 < N; c0 += 16) {
                float g[16], u[16];
                tmem_ld16(lane_base + c0, g);
                tmem_ld16(lane_base + L::kAccStride + c0, u);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    stg[(c0 + j) * kHS + f] = f32_to_bf16(silu_f32(g[j] * tsg) * (u[j] * tsu));
            }
        } else {
            float* stg = reinterpret_cast<float*>(sm);
#pragma unroll 1
            for (int c0 = c_begin; c0 < c_begin + kTokTile / 2 && c0 < N; c0 += 16) {
                float a[16];
                tmem_ld16(lane_base + c0, a);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) stg[(c0 + j) * kYS + f] = a[j];
            }
        }
        tc_fence_before();
        named_bar_sync(1, kProd);
        if (kParts == 2) {
            const uint16_t* stg = reinterpret_cast<const uint16_t*>(sm);
            uint16_t* out = shared ? P.hs : P.h;
            const int ch = tid & 15;
            if (feat0 + 8 * ch < Fvalid) {
#pragma unroll 4
                for (int c = tid >> 4; c < tr.n_rows; c += kProd / 16)
                    *reinterpret_cast<uint4*>(out + (size_t)(tr.p0 + c) * Fvalid + feat0 + 8 * ch) =
                        *reinterpret_cast<const uint4*>(stg + c * kHS + 8 * ch);
            }
        } else {
            const float* stg = reinterpret_cast<const float*>(sm);
            const int ch = tid & 31;
            if (feat0 + 4 * ch < P.H) {
#pragma unroll 4
                for (int c = tid >> 5; c < tr.n_rows; c += kProd / 32) {
                    const int2 ci = cols[c];
                    const float sc = __int_as_float(ci.y);
                    float4 v = *reinterpret_cast<const float4*>(stg + c * kYS + 4 * ch);
                    v.x *= sc; v.y *= sc; v.z *= sc; v.w *= sc;
                    *reinterpret_cast<float4*>(P.Y + (size_t)ci.x * P.H + feat0 + 4 * ch) = v;
                }
            }
        }
    } else if (lane == 0) {
        // ---------------- MMA issuer (one thread)
        const uint32_t idesc = f16_idesc(kM, N);
#pragma unroll 1
        for (int kt = 0; kt < nk; ++kt) {
            const int st = kt % S;
            if (!wait_or_abort(&full[st], (kt / S) & 1, abort_flag, hdr, wait_limit)) break;
            tc_fence_after();
            const uint32_t stage = sm_base + st * L::kStage;
#pragma unroll
            for (int j = 0; j < kKS / 16; ++j) {
                const uint64_t bd = sw128_desc(stage + L::kA + j * 32);
#pragma unroll
                for (int p = 0; p < kParts; ++p)
                    tc_mma(tmem + p * L::kAccStride, sw128_desc(stage + p * (kM * 128) + j * 32), bd, idesc,
                           (kt | j) != 0);
            }
            tc_commit(&empty[st]);
        }
        tc_commit(accb);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kProd / 32) {
        tc_fence_after();
        tmem_dealloc<L::kTmemCols>(tmem);
    }
}

}  // namespace

cudaError_t launch_grouped_tc(const GroupedParams& P, int mode, int tiles_max, WsHeader* hdr,
                              uint64_t wait_limit, cudaStream_t s) {
    if (tiles_max <= 0) return cudaSuccess;
    if (mode == 0) {
        using L = TcLayout<2>;
        static bool attr_set = false;
        if (!attr_set) {
            cudaError_t e = cudaFuncSetAttribute(grouped_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 L::kBytes + 1024);
            if (e != cudaSuccess) return e;
            attr_set = true;
        }
        const int n_ft = (max(P.I, P.Is) + kM - 1) / kM;
        grouped_tc_kernel<2><<<(unsigned)tiles_max * n_ft, kTcThreads, L::kBytes + 1024, s>>>(P, n_ft, hdr, wait_limit);
    } else {
        using L = TcLayout<1>;
        static bool attr_set = false;
        if (!attr_set) {
            cudaError_t e = cudaFuncSetAttribute(grouped_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 L::kBytes + 1024);
            if (e != cudaSuccess) return e;
            attr_set = true;
        }
        const int n_ft = (P.H + kM - 1) / kM;
        grouped_tc_kernel<1><<<(unsigned)tiles_max * n_ft, kTcThreads, L::kBytes + 1024, s>>>(P, n_ft, hdr, wait_limit);
    }
    return cudaGetLastError();
}

}  // namespace nvfp4
