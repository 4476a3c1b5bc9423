// Routing helpers of the multi-token decode path (T <= 64 tokens, E <= 256,
// k <= 8): a warp top-k and the block-level construction of the per-expert lists,
// the active-expert list and the pass map.
//
// lynn-engine tutorials index, row 06 (MoE router): softmax over all experts,
// top-k, renormalise, which equals a softmax over the k selected logits. The k
// largest logits are taken in the order (larger logit first, lower expert id
// first among equal logits: the sorted-router order of the lynn-engine README,
// P35 note); weights are exp(l_j - l_max) / sum_j' exp(l_j' - l_max).
#pragma once

#include <cfloat>

#include "common.cuh"

namespace nvfp4 {

constexpr int kMtPass = 16;          // entries per pass of the multi-token expert kernels
constexpr int kMtMaxEntries = 512;   // T * k <= 64 * 8

// Order-preserving 32-bit key of a logit (a larger logit gives a larger key); -0 is
// taken as +0 first, so equal logits give equal keys.
__device__ __forceinline__ uint32_t route_key(float f) {
    const uint32_t b = __float_as_uint(__fadd_rn(f, 0.0f));
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float route_key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Top-k of one token's E logits (E <= 256), by one warp. Lane l holds experts 8l .. 8l+7
// as 64-bit keys (route_key, then 7 - i so that the lower id ranks first among equal
// logits) and sorts them descending in registers (a 19-exchange merge network). Each of
// the k rounds takes the largest head over the warp (among equal heads the lowest lane,
// which holds the lowest ids) and the lane that held it drops it. The result is the
// routing order: larger logit first, lower expert id first among equal logits. Lane
// j < k writes ids[j] and w[j] (and sids[j] when sids is not null). Logits are read
// through L2 (`ld.cg`) because other blocks wrote them.
__device__ __forceinline__ void topk_warp_mt(const float* lg, int E, int k, int32_t* ids, float* w,
                                             int32_t* ids_out, float* w_out, int* sids) {
    const int lane = threadIdx.x & 31;
    unsigned long long kk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = 8 * lane + i;
        kk[i] = e < E ? ((unsigned long long)route_key(__ldcg(lg + e)) << 3) | (unsigned)(7 - i) : 0ull;
    }
#define MT_CX(a, b) { const unsigned long long hi_ = max(kk[a], kk[b]), lo_ = min(kk[a], kk[b]); kk[a] = hi_; kk[b] = lo_; }
    MT_CX(0, 1) MT_CX(2, 3) MT_CX(4, 5) MT_CX(6, 7)
    MT_CX(0, 2) MT_CX(1, 3) MT_CX(4, 6) MT_CX(5, 7)
    MT_CX(1, 2) MT_CX(5, 6)
    MT_CX(0, 4) MT_CX(1, 5) MT_CX(2, 6) MT_CX(3, 7)
    MT_CX(2, 4) MT_CX(3, 5)
    MT_CX(1, 2) MT_CX(3, 4) MT_CX(5, 6)
#undef MT_CX
    int my_e = 0;
    float my_v = 0.f, vmax = 0.f;
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
        const float v = route_key_value(wb);
        if (j == 0) vmax = v;
        if (lane == j) { my_e = e; my_v = v; }
    }
    // w_j = exp(l_j - l_max) / sum_{j' < k} exp(l_j' - l_max), summed in rank order
    const float ex = lane < k ? expf(my_v - vmax) : 0.f;
    float sum = 0.f;
#pragma unroll 1
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
        const float wj = ex / sum;
        ids[lane] = my_e;
        w[lane] = wj;
        if (sids) sids[lane] = my_e;
        if (ids_out) ids_out[lane] = my_e;
        if (w_out) w_out[lane] = wj;
    }
}

// Shared memory of build_lists_block.
struct ListsSmem {
    uint32_t mask[NVFP4_MAX_EXPERTS][kMtMaxEntries / 32];   // entries of each expert, as bits
    int ids[kMtMaxEntries];
    int off[NVFP4_MAX_EXPERTS];
    int wsum[3][NVFP4_MAX_EXPERTS / 32];
};

// Per-expert lists of the total = T*k entries, by one block of exactly 256 threads;
// the ids are read through L2, or are already in S.ids (ids_in_smem: written by this
// block before a barrier). Entry i of expert e goes to offsets[e] + (number of
// entries i' < i of expert e): a stable counting sort. active[0] = A, active[1+a]
// = the a-th expert with entries (ascending); pass_map[0] = P, pass_map[1+p] =
// (active slot << 8) | pass, a pass being up to kMtPass consecutive entries of
// one expert's list.
__device__ __forceinline__ void build_lists_block(ListsSmem& S, const int32_t* ids, int total, int E,
                                                  int32_t* offsets, int32_t* token_list, int32_t* active,
                                                  int32_t* pass_map, bool ids_in_smem) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = (total + 31) >> 5;
    for (int i = tid; i < NVFP4_MAX_EXPERTS * nw; i += 256) S.mask[i / nw][i - (i / nw) * nw] = 0u;
    __syncthreads();
    for (int i = tid; i < total; i += 256) {
        int e;
        if (ids_in_smem) {
            e = S.ids[i];
        } else {
            e = __ldcg(ids + i);
            S.ids[i] = e;
        }
        atomicOr(&S.mask[e][i >> 5], 1u << (i & 31));
    }
    __syncthreads();
    int c = 0;
    if (tid < E)
        for (int q = 0; q < nw; ++q) c += __popc(S.mask[tid][q]);
    const int v0 = c, v1 = c > 0 ? 1 : 0, v2 = (c + kMtPass - 1) / kMtPass;
    int i0 = v0, i1 = v1, i2 = v2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n0 = __shfl_up_sync(0xffffffffu, i0, o);
        const int n1 = __shfl_up_sync(0xffffffffu, i1, o);
        const int n2 = __shfl_up_sync(0xffffffffu, i2, o);
        if (lane >= o) { i0 += n0; i1 += n1; i2 += n2; }
    }
    if (lane == 31) {
        S.wsum[0][warp] = i0;
        S.wsum[1][warp] = i1;
        S.wsum[2][warp] = i2;
    }
    __syncthreads();
    if (tid < E) {
        int b0 = 0, b1 = 0, b2 = 0;
        for (int ww = 0; ww < warp; ++ww) { b0 += S.wsum[0][ww]; b1 += S.wsum[1][ww]; b2 += S.wsum[2][ww]; }
        const int off = b0 + i0 - v0, slot = b1 + i1 - v1, pass0 = b2 + i2 - v2;
        S.off[tid] = off;
        offsets[tid] = off;
        if (c > 0) {
            active[1 + slot] = tid;
            for (int pi = 0; pi < v2; ++pi) pass_map[1 + pass0 + pi] = (slot << 8) | pi;
        }
        if (tid == E - 1) {
            offsets[E] = off + c;
            active[0] = slot + v1;
            pass_map[0] = pass0 + v2;
        }
    }
    __syncthreads();
    for (int i = tid; i < total; i += 256) {
        const int e = S.ids[i], qw = i >> 5;
        int r = __popc(S.mask[e][qw] & ((1u << (i & 31)) - 1u));
        for (int q = 0; q < qw; ++q) r += __popc(S.mask[e][q]);
        token_list[S.off[e] + r] = i;
    }
}

}  // namespace nvfp4
