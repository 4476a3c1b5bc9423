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
// Warp roles per CTA (704 threads) and three rings that move at their own pace:
//   warp 16, one lane (raw stream): for step s, wait until the expanders have read
//     the raw slot of step s - R, then TMA the step's NVFP4 codes and block scales of
//     the 256 weight rows into it (R = 5..8 slots: the HBM-latency stream runs far
//     ahead);
//   warps 17-20 (token stream): for step s, wait until the MMAs of step s - SB are
//     done, then bring the tile's token rows into the 128-byte-swizzled B slot
//     (gate/up: gathered rows of x by cp.async, whose completion arrives on the slot's
//     barrier; down: contiguous rows of h / hs by TMA);
//   warps 0-15 (expanders): wait for the raw slot, read it, release it, wait for a
//     free A slot (two), expand the NVFP4 bytes into the swizzled bf16 A tile, fence
//     to the async proxy and arrive;
//   warp 21, one lane: wait for the A and B slots of step s, issue the MMAs and
//     commit them to both slots' empty barriers; after the last step, commit to the
//     accumulator barrier;
//   warps 0-15 then read TMEM, run the epilogue through shared memory and store
//     coalesced rows.
// Every wait is bounded; a wait that runs out records NVFP4_ERR_DEVICE_TIMEOUT and
// makes every later wait of the CTA give up at once.
//
// NVFP4 -> bf16 expansion (exact): cvt.rn.f16x2.e2m1x2 gives the E2M1 values as
// f16; shifting an f16 bit pattern right by 3 (sign kept in place) reads it as a
// bf16 of the same value times 2^-112; one bf16x2 multiply by (block scale * 2^112)
// restores the scale. Every product has at most 6 significant bits and lies in
// [2^-10, 2688], so no step rounds.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace nvfp4 {

namespace {

constexpr int kM = 128;           // weight rows per accumulator (MMA M)
constexpr int kKS = 64;           // K elements per stage: one 128-byte row of the swizzle atom
constexpr int kRows = 2 * kM;     // weight rows per CTA: two accumulators share the token tile
constexpr int kExp = 512;         // expander / epilogue threads (warps 0-15): half a weight row each
constexpr int kRawWarp = kExp / 32;           // warp 16, lane 0: weight codes and scales (TMA)
constexpr int kBWarp0 = kRawWarp + 1;         // warps 17-20: token rows (cp.async; the down GEMM: TMA by lane 0)
constexpr int kBThreads = 128;
constexpr int kMmaWarp = kBWarp0 + kBThreads / 32;   // warp 21: TMEM owner and MMA issuer
constexpr int kTcThreads = (kMmaWarp + 1) * 32;
constexpr int kMaxRaw = 8;        // raw weight ring depth (at most)
constexpr int kMaxB = 4;          // token-row ring depth (at most)

// Dynamic shared memory: [1024-byte alignment slack][rings][fixed tables]. Three rings
// move at their own pace: the raw NVFP4 bytes of the A rows (TMA boxes from HBM, the
// longest latency: the deepest ring), the bf16 token rows (N x 64, 128-byte swizzled;
// N = the tile's token count rounded up to 16), and the expanded bf16 A tile (two
// slots: one being expanded while the MMAs read the other).
constexpr int kA = kRows * 128;
constexpr int kRawScales = kRows * 32;      // raw: codes [kRows][32 B], then scales [kRows][16 B]
constexpr int kRawStage = kRows * 48;       // (the 16 scale bytes hold 4 K steps; step s uses bytes 4(s%4)..)
constexpr int kRing = 220 * 1024;
constexpr int kOffTok = kRing;                          // per token row: source row (-1: none)
constexpr int kOffCols = kOffTok + kTokTile * 4;        // per token column: (Y row, scale)
constexpr int kOffBar = kOffCols + kTokTile * 8;
constexpr int kNumBars = 2 * kMaxRaw + 2 * kMaxB + 4 + 1;
constexpr int kSmemBytes = 1024 + kOffBar + kNumBars * 8 + 16;
constexpr int kTmemCols = 512;
constexpr int kAccStride = 256;   // TMEM column offset of the second accumulator

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Arrive on `bar` when every cp.async issued so far by this thread has landed (the
// arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(su32(bar)) : "memory");
}

// 2D tensor copy global -> shared (TMA), completing on `bar`'s transaction count.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar)) : "memory");
}

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

// ---------------------------------------------------------------- tensor maps
// The grouped GEMMs read the NVFP4 weights through TMA: for each matrix group, the
// codes as a 2D byte tensor [rows, K/2] (box 32 bytes x 128 rows = one K step of
// 128 weight rows) and the block scales as [rows, K/16] (box 16 bytes x 128 rows =
// four K steps); the down GEMM also reads its token rows h / hs as bf16 [rows, K]
// with the 128-byte swizzle (box 64 x 16 rows).
struct TcMaps {
    CUtensorMap gu_codes, gu_scales, dn_codes, dn_scales;
    CUtensorMap sh_gu_codes, sh_gu_scales, sh_dn_codes, sh_dn_scales;
    CUtensorMap h, hs;
};
constexpr int kBoxRowsB = 16;   // token rows per B box of the down GEMM

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

// Bounded wait that ignores the abort flag: after an abort, a thread that issued bulk copies
// or MMAs waits (with the library's fixed limit) until they have landed, so that the CTA
// never exits with its own asynchronous operations in flight.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    mbar_wait_bounded(bar, parity, kDefaultWaitLimit);
}

constexpr int kHS = kM + 8;   // bf16 staging row stride of the gate/up epilogue
constexpr int kYS = kM + 4;   // fp32 staging row stride of the down epilogue

// ---------------------------------------------------------------- kernel
// kMode 0: gate/up (A rows 0-127 = gate rows, 128-255 = the matching up rows of 128
// intermediate indices), kMode 1: down (A rows = 256 consecutive output features).
template <int kMode>
__global__ void __launch_bounds__(kTcThreads, 1)
grouped_tc_kernel(const GroupedParams P, const __grid_constant__ TcMaps maps, int n_ft, WsHeader* hdr,
                  unsigned long long wait_limit) {
    extern __shared__ uint8_t tc_smem_raw[];
    // the swizzle pattern follows shared-memory address bits: align the base to 1024
    uint8_t* sm = tc_smem_raw + ((1024u - (su32(tc_smem_raw) & 1023u)) & 1023u);

    const int ft = blockIdx.x % n_ft, tt = blockIdx.x / n_ft;
    TcTile tr;
    if (!locate_tc_tile(P, tt, &tr)) return;
    const bool shared = tr.slot == P.E;
    const int Fvalid = kMode == 0 ? (shared ? P.Is : P.I) : P.H;   // output features of this GEMM
    const int feat0 = ft * (kMode == 0 ? kM : kRows);
    if (feat0 >= Fvalid) return;
    const int Kd = kMode == 0 ? P.H : (shared ? P.Is : P.I);
    const int nk = Kd / kKS;
    const int N = (tr.n_rows + 15) & ~15;
    const int bbytes = N * 128;                                      // one token-row stage (multiple of 2048)
    const int SB = N > 128 ? 3 : kMaxB;                              // token-row ring depth
    const int R = min(kMaxRaw, (kRing - 2 * kA - SB * bbytes) / kRawStage);   // raw weight ring depth
    const uint32_t offB = 2 * kA, offRaw = offB + SB * bbytes;       // ring offsets (multiples of 1024)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    uint64_t* raw_full = reinterpret_cast<uint64_t*>(sm + kOffBar);   // raw weight bytes landed (TMA)
    uint64_t* raw_empty = raw_full + kMaxRaw;                          // raw slot read by the expanders
    uint64_t* b_full = raw_empty + kMaxRaw;                            // token rows landed
    uint64_t* b_empty = b_full + kMaxB;                                // MMAs done with the token rows
    uint64_t* a_full = b_empty + kMaxB;                                // [2] A tile expanded
    uint64_t* a_empty = a_full + 2;                                    // [2] MMAs done with the A tile
    uint64_t* accb = a_empty + 2;                                      // all MMAs done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* tok = reinterpret_cast<int*>(sm + kOffTok);
    int2* cols = reinterpret_cast<int2*>(sm + kOffCols);

    if (warp == kMmaWarp) {
        if (lane == 0) {
            for (int i = 0; i < R; ++i) {
                mbar_init(&raw_full[i], 1);
                mbar_init(&raw_empty[i], kExp);
            }
            for (int i = 0; i < SB; ++i) {
                mbar_init(&b_full[i], kMode == 0 ? kBThreads : 1);
                mbar_init(&b_empty[i], 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(&a_full[i], kExp);
                mbar_init(&a_empty[i], 1);
            }
            mbar_init(accb, 1);
            *abort_flag = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc<kTmemCols>(tmem_slot);
    }
    // per token row: the row of x (gate/up) or of h / hs (down) it reads; -1 past the tile
    for (int c = tid; c < kTokTile; c += kTcThreads) {
        int src = -1;
        if (c < tr.n_rows) {
            if (kMode == 0 && !shared) src = __ldg(P.token_list + tr.p0 + c) / P.k;
            else src = tr.p0 + c;
        }
        tok[c] = src;
        if (kMode == 1 && c < tr.n_rows) {
            // the row of Y this column feeds and the epilogue scale
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

    // weight row r (0 .. kRows-1) of the tile: its packed codes and E4M3 scales
    auto weight_row = [&](int r, const uint8_t** codes, const uint8_t** scales) {
        *codes = nullptr;
        *scales = nullptr;
        if (kMode == 0) {
            const int f = feat0 + (r & (kM - 1));
            if (f >= Fvalid) return;
            const size_t wrow = (size_t)(r < kM ? f : Fvalid + f);   // gate rows, then up rows
            const uint8_t* pk = shared ? P.sh_gu_packed : P.gu_packed + (size_t)tr.slot * 2 * P.I * (P.H / 2);
            const uint8_t* sc = shared ? P.sh_gu_scales : P.gu_scales + (size_t)tr.slot * 2 * P.I * (P.H / 16);
            *codes = pk + wrow * (P.H / 2);
            *scales = sc + wrow * (P.H / 16);
        } else {
            const int f = feat0 + r;
            if (f >= P.H) return;
            const uint8_t* pk = shared ? P.sh_dn_packed : P.dn_packed + (size_t)tr.slot * P.H * (P.I / 2);
            const uint8_t* sc = shared ? P.sh_dn_scales : P.dn_scales + (size_t)tr.slot * P.H * (P.I / 16);
            *codes = pk + (size_t)f * (Kd / 2);
            *scales = sc + (size_t)f * (Kd / 16);
        }
    };

    if (warp == kRawWarp) {
        // ---------------- raw weight stream (one thread): codes and scales of the A rows,
        // up to R steps ahead of the expanders
        if (lane == 0) {
            const CUtensorMap* mc = kMode == 0 ? (shared ? &maps.sh_gu_codes : &maps.gu_codes)
                                               : (shared ? &maps.sh_dn_codes : &maps.dn_codes);
            const CUtensorMap* ms = kMode == 0 ? (shared ? &maps.sh_gu_scales : &maps.gu_scales)
                                               : (shared ? &maps.sh_dn_scales : &maps.dn_scales);
            int y0, y1;   // first weight row of A rows 0-127 and 128-255
            if (kMode == 0) {
                const int base = shared ? 0 : tr.slot * 2 * P.I;
                y0 = base + feat0;
                y1 = base + Fvalid + feat0;
            } else {
                y0 = (shared ? 0 : tr.slot * P.H) + feat0;
                y1 = y0 + kM;
            }
            int issued = 0;
#pragma unroll 1
            for (int s = 0; s < nk; ++s) {
                const int r = s % R, u = s / R;
                if (u > 0 && !wait_or_abort(&raw_empty[r], (u - 1) & 1, abort_flag, hdr, wait_limit)) break;
                if (*abort_flag) break;
                const uint32_t raw = sm_base + offRaw + r * kRawStage;
                mbar_arrive_expect_tx(&raw_full[r], 2 * (32 * kM) + 2 * (16 * kM));
                tma_load_2d(raw, mc, s * 32, y0, &raw_full[r]);
                tma_load_2d(raw + kM * 32, mc, s * 32, y1, &raw_full[r]);
                tma_load_2d(raw + kRawScales, ms, (s >> 2) * 16, y0, &raw_full[r]);
                tma_load_2d(raw + kRawScales + kM * 16, ms, (s >> 2) * 16, y1, &raw_full[r]);
                issued = s + 1;
            }
            // every issued copy has landed before the CTA may exit (the last fill of each slot)
            for (int s = max(0, issued - R); s < issued; ++s) drain_wait(&raw_full[s % R], (s / R) & 1);
        }
    } else if (warp >= kBWarp0 && warp < kMmaWarp) {
        // ---------------- token-row stream, up to SB steps ahead of the MMAs (gate/up:
        // gathered rows of x by cp.async from 128 threads; down: the tile's contiguous
        // rows of h / hs by TMA from one thread)
        const int bt = tid - kBWarp0 * 32;
        if (kMode == 0) {
            const int bc = bt & 7;
            int boff[16];   // element offset of this thread's chunk in row (bt >> 3) + 16 j, or -1
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int src = tok[(bt >> 3) + 16 * j];
                boff[j] = src < 0 ? -1 : src * P.H + bc * 8;
            }
#pragma unroll 1
            for (int s = 0; s < nk; ++s) {
                const int b = s % SB, u = s / SB;
                if (u > 0 && !wait_or_abort(&b_empty[b], (u - 1) & 1, abort_flag, hdr, wait_limit)) break;
                if (*abort_flag) break;
                const uint32_t bb = sm_base + offB + b * bbytes;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int row = (bt >> 3) + 16 * j;
                    if (row < N) {
                        const uint32_t dst = bb + row * 128 + ((bc ^ (row & 7)) << 4);
                        if (boff[j] >= 0) cp_async16_zfill(dst, P.x + boff[j] + s * kKS, 16u);
                        else cp_async16_zfill(dst, P.x, 0u);
                    }
                }
                cp_async_arrive_noinc(&b_full[b]);
            }
            asm volatile("cp.async.wait_all;" ::: "memory");   // this thread's copies have landed
        } else if (bt == 0) {
            const CUtensorMap* mb = shared ? &maps.hs : &maps.h;
            int issued = 0;
#pragma unroll 1
            for (int s = 0; s < nk; ++s) {
                const int b = s % SB, u = s / SB;
                if (u > 0 && !wait_or_abort(&b_empty[b], (u - 1) & 1, abort_flag, hdr, wait_limit)) break;
                if (*abort_flag) break;
                const uint32_t bb = sm_base + offB + b * bbytes;
                mbar_arrive_expect_tx(&b_full[b], (uint32_t)bbytes);
                for (int i = 0; i < N / kBoxRowsB; ++i)
                    tma_load_2d(bb + i * (kBoxRowsB * 128), mb, s * kKS, tr.p0 + i * kBoxRowsB, &b_full[b]);
                issued = s + 1;
            }
            for (int s = max(0, issued - SB); s < issued; ++s) drain_wait(&b_full[s % SB], (s / SB) & 1);
        }
    } else if (warp < kExp / 32) {
        // ---------------- expanders: raw NVFP4 bytes -> bf16 A tile (half a row each)
        const uint8_t* rcode;
        const uint8_t* rscale;
        const int r = tid >> 1, half = tid & 1;
        weight_row(r, &rcode, &rscale);
        const bool valid = rcode != nullptr;
        const int rl = r & 7;   // swizzle phase of the row
        const int a_off = (r >> 7) * (kM * 128) + (r & (kM - 1)) * 128;
#pragma unroll 1
        for (int kt = 0; kt < nk; ++kt) {
            const int rr = kt % R, a = kt & 1;
            wait_or_abort(&raw_full[rr], (kt / R) & 1, abort_flag, hdr, wait_limit);
            const uint8_t* raw = sm + offRaw + rr * kRawStage;
            uint4 c0 = make_uint4(0, 0, 0, 0);
            uint32_t sw = 0;
            if (valid) {
                c0 = *reinterpret_cast<const uint4*>(raw + r * 32 + half * 16);
                sw = *reinterpret_cast<const uint32_t*>(raw + kRawScales + r * 16 + (kt & 3) * 4);
            }
            mbar_arrive(&raw_empty[rr]);   // the raw slot may be refilled
            if (kt >= 2) wait_or_abort(&a_empty[a], ((kt >> 1) - 1) & 1, abort_flag, hdr, wait_limit);
            uint8_t* arow = sm + a * kA + a_off;
            if (valid) {
                uint32_t s0, s1;
                scale_pair_bf16(sw >> (16 * half), s0, s1);
                const uint32_t words[4] = {c0.x, c0.y, c0.z, c0.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {   // chunk 4 half + c = elements 8(4 half + c) .., block 2 half + c/2
                    uint32_t o[4];
                    expand8(words[c], c < 2 ? s0 : s1, o);
                    *reinterpret_cast<uint4*>(arow + (((4 * half + c) ^ rl) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4*>(arow + ((4 * half + c) << 4)) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            mbar_arrive(&a_full[a]);
        }

        // ---------------- epilogue: TMEM -> registers -> shared staging -> global
        // (after an abort: still wait, with the fixed limit, until the MMAs the issuer committed
        // are done, so that no read of tensor memory races them; the outputs are then garbage
        // and the call reports the timeout)
        if (!wait_or_abort(accb, 0, abort_flag, hdr, wait_limit)) drain_wait(accb, 0);
        tc_fence_after();
        const int q = warp & 3, c_begin = (warp >> 2) * (kTokTile / 4);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const int f = 32 * q + lane;
        if (kMode == 0) {
            uint16_t* stg = reinterpret_cast<uint16_t*>(sm);
            const float* tsp = shared ? P.sh_gu_tscale : P.gu_tscale + 2 * tr.slot;
            const float tsg = __ldg(tsp), tsu = __ldg(tsp + 1);
#pragma unroll 1
            for (int c0 = c_begin; c0 < c_begin + kTokTile / 4 && c0 < N; c0 += 16) {
                float g[16], u[16];
                tmem_ld16(lane_base + c0, g);
                tmem_ld16(lane_base + kAccStride + c0, u);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    stg[(c0 + j) * kHS + f] = f32_to_bf16(silu_f32(g[j] * tsg) * (u[j] * tsu));
            }
            tc_fence_before();
            named_bar_sync(1, kExp);
            uint16_t* out = shared ? P.hs : P.h;
            const int ch = tid & 15;
            if (feat0 + 8 * ch < Fvalid) {
#pragma unroll 4
                for (int c = tid >> 4; c < tr.n_rows; c += kExp / 16)
                    *reinterpret_cast<uint4*>(out + (size_t)(tr.p0 + c) * Fvalid + feat0 + 8 * ch) =
                        *reinterpret_cast<const uint4*>(stg + c * kHS + 8 * ch);
            }
        } else {
            float* stg = reinterpret_cast<float*>(sm);
#pragma unroll 1
            for (int p = 0; p < 2; ++p) {
                const int fp0 = feat0 + p * kM;
                if (fp0 >= P.H) break;
#pragma unroll 1
                for (int c0 = c_begin; c0 < c_begin + kTokTile / 4 && c0 < N; c0 += 16) {
                    float a[16];
                    tmem_ld16(lane_base + p * kAccStride + c0, a);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) stg[(c0 + j) * kYS + f] = a[j];
                }
                named_bar_sync(1, kExp);
                const int ch = tid & 31;
                if (fp0 + 4 * ch < P.H) {
#pragma unroll 4
                    for (int c = tid >> 5; c < tr.n_rows; c += kExp / 32) {
                        const int2 ci = cols[c];
                        const float sc = __int_as_float(ci.y);
                        float4 v = *reinterpret_cast<const float4*>(stg + c * kYS + 4 * ch);
                        v.x *= sc; v.y *= sc; v.z *= sc; v.w *= sc;
                        *reinterpret_cast<float4*>(P.Y + (size_t)ci.x * P.H + fp0 + 4 * ch) = v;
                    }
                }
                named_bar_sync(1, kExp);   // staging is reused by the next part
            }
            tc_fence_before();
        }
    } else if (warp == kMmaWarp && lane == 0) {
        // ---------------- MMA issuer (one thread)
        const uint32_t idesc = f16_idesc(kM, N);
#pragma unroll 1
        for (int kt = 0; kt < nk; ++kt) {
            const int a = kt & 1, b = kt % SB;
            if (!wait_or_abort(&a_full[a], (kt >> 1) & 1, abort_flag, hdr, wait_limit)) break;
            if (!wait_or_abort(&b_full[b], (kt / SB) & 1, abort_flag, hdr, wait_limit)) break;
            // the token rows may have been written by cp.async (generic proxy): order them
            // before the tensor cores' reads
            fence_proxy_async_smem();
            tc_fence_after();
            const uint32_t abase = sm_base + a * kA, bbase = sm_base + offB + b * bbytes;
#pragma unroll
            for (int j = 0; j < kKS / 16; ++j) {
                const uint64_t bd = sw128_desc(bbase + j * 32);
#pragma unroll
                for (int p = 0; p < 2; ++p)
                    tc_mma(tmem + p * kAccStride, sw128_desc(abase + p * (kM * 128) + j * 32), bd, idesc,
                           (kt | j) != 0);
            }
            tc_commit(&a_empty[a]);
            tc_commit(&b_empty[b]);
        }
        tc_commit(accb);
        // after an abort the epilogue does not wait for the MMAs: wait here (fixed limit) so that
        // none is still writing tensor memory when it is freed
        if (*abort_flag) drain_wait(accb, 0);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc<kTmemCols>(tmem);
    }
}

}  // namespace

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Byte matrix [rows, inner] read in boxes of box_inner bytes x 128 rows.
bool encode_u8(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* m, const void* base, uint64_t inner,
               uint64_t rows, uint32_t box_inner) {
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner};
    const cuuint32_t box[2] = {box_inner, (cuuint32_t)kM};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 matrix [rows, cols] read in boxes of 64 x kBoxRowsB, 128-byte swizzled in shared memory.
bool encode_bf16_sw128(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* m, const void* base, uint64_t cols,
                       uint64_t rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kKS, (cuuint32_t)kBoxRowsB};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_maps(const GroupedParams& P, TcMaps* m) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
    if (!fn) return false;
    memset(m, 0, sizeof(*m));
    const uint64_t E = (uint64_t)P.E, H = (uint64_t)P.H, I = (uint64_t)P.I, Is = (uint64_t)P.Is;
    bool ok = encode_u8(fn, &m->gu_codes, P.gu_packed, H / 2, E * 2 * I, 32) &&
              encode_u8(fn, &m->gu_scales, P.gu_scales, H / 16, E * 2 * I, 16) &&
              encode_u8(fn, &m->dn_codes, P.dn_packed, I / 2, E * H, 32) &&
              encode_u8(fn, &m->dn_scales, P.dn_scales, I / 16, E * H, 16) &&
              encode_bf16_sw128(fn, &m->h, P.h, I, (uint64_t)P.T * P.k);
    if (ok && Is > 0)
        ok = encode_u8(fn, &m->sh_gu_codes, P.sh_gu_packed, H / 2, 2 * Is, 32) &&
             encode_u8(fn, &m->sh_gu_scales, P.sh_gu_scales, H / 16, 2 * Is, 16) &&
             encode_u8(fn, &m->sh_dn_codes, P.sh_dn_packed, Is / 2, H, 32) &&
             encode_u8(fn, &m->sh_dn_scales, P.sh_dn_scales, Is / 16, H, 16) &&
             encode_bf16_sw128(fn, &m->hs, P.hs, Is, (uint64_t)P.T);
    return ok;
}

}  // namespace

cudaError_t launch_grouped_tc(const GroupedParams& P, int mode, int tiles_max, WsHeader* hdr,
                              uint64_t wait_limit, cudaStream_t s) {
    if (tiles_max <= 0) return cudaSuccess;
    static bool attr_set[2] = {false, false};
    if (!attr_set[mode]) {
        cudaError_t e = cudaFuncSetAttribute(mode == 0 ? grouped_tc_kernel<0> : grouped_tc_kernel<1>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[mode] = true;
    }
    TcMaps maps;
    if (!encode_maps(P, &maps)) return cudaErrorInvalidValue;
    if (mode == 0) {
        const int n_ft = (max(P.I, P.Is) + kM - 1) / kM;
        grouped_tc_kernel<0><<<(unsigned)tiles_max * n_ft, kTcThreads, kSmemBytes, s>>>(P, maps, n_ft, hdr,
                                                                                       wait_limit);
    } else {
        const int n_ft = (P.H + kRows - 1) / kRows;
        grouped_tc_kernel<1><<<(unsigned)tiles_max * n_ft, kTcThreads, kSmemBytes, s>>>(P, maps, n_ft, hdr,
                                                                                       wait_limit);
    }
    return cudaGetLastError();
}

}  // namespace nvfp4
