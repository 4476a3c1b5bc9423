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

// (v, e) comes before (v2, e2) in routing order.
__device__ __forceinline__ bool route_before(float v, int e, float v2, int e2) {
    return v > v2 || (v == v2 && e < e2);
}

// Order (va, ea), (vb, eb) so the first comes first; selects, no branch.
__device__ __forceinline__ void route_cas(float& va, int& ea, float& vb, int& eb) {
    const bool sw = route_before(vb, eb, va, ea);
    const float v0 = sw ? vb : va, v1 = sw ? va : vb;
    const int e0 = sw ? eb : ea, e1 = sw ? ea : eb;
    va = v0; vb = v1; ea = e0; eb = e1;
}

// Top-k of one token's E logits (lane l holds experts l, l+32, ..., l+224): each
// lane sorts its eight (bitonic network), then five butterfly rounds each merge a
// lane's sorted eight with its partner's and keep the first eight: element-wise the
// better of one list and the other reversed is a bitonic sequence holding the top
// eight, and three compare-exchange stages sort it. Every lane ends with the same
// sorted top eight. The chain of dependent steps is short (about 45 compare-
// exchange or select levels) and branch-free; the butterfly loop stays rolled to
// keep the code small. Lane j < k writes ids[j] and w[j]. Logits are read through
// L2 (`ld.cg`) because other blocks wrote them.
__device__ __forceinline__ void topk_warp_mt(const float* lg, int E, int k, int32_t* ids, float* w,
                                             int32_t* ids_out, float* w_out) {
    const int lane = threadIdx.x & 31;
    float v[8];
    int e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        e[i] = lane + 32 * i;
        v[i] = e[i] < E ? __ldcg(lg + e[i]) : -INFINITY;
        if (e[i] >= E) e[i] = 0x7fffffff;
    }
#pragma unroll
    for (int size = 2; size <= 8; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    if ((i & size) == 0 || size == 8) route_cas(v[i], e[i], v[j], e[j]);
                    else route_cas(v[j], e[j], v[i], e[i]);
                }
            }
        }
    }
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
        float pv[8];
        int pe[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            pv[i] = __shfl_xor_sync(0xffffffffu, v[i], o);
            pe[i] = __shfl_xor_sync(0xffffffffu, e[i], o);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const bool mine = route_before(v[i], e[i], pv[7 - i], pe[7 - i]);
            v[i] = mine ? v[i] : pv[7 - i];
            e[i] = mine ? e[i] : pe[7 - i];
        }
#pragma unroll
        for (int stride = 4; stride > 0; stride >>= 1) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = i ^ stride;
                if (j > i) route_cas(v[i], e[i], v[j], e[j]);
            }
        }
    }
    // w_j = exp(l_j - l_max) / sum_{j' < k} exp(l_j' - l_max), summed in rank order;
    // lane j takes element j of the (identical) lists
    float my_v = v[0];
    int my_e = e[0];
#pragma unroll
    for (int j = 1; j < 8; ++j) {
        if (lane == j) { my_v = v[j]; my_e = e[j]; }
    }
    const float ex = lane < k ? expf(my_v - v[0]) : 0.f;
    float sum = 0.f;
#pragma unroll 1
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
        const float wj = ex / sum;
        ids[lane] = my_e;
        w[lane] = wj;
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

// Per-expert lists of the total = T*k entries (ids read through L2), by one block
// of exactly 256 threads. Entry i of expert e goes to offsets[e] + (number of
// entries i' < i of expert e): a stable counting sort. active[0] = A, active[1+a]
// = the a-th expert with entries (ascending); pass_map[0] = P, pass_map[1+p] =
// (active slot << 8) | pass, a pass being up to kMtPass consecutive entries of
// one expert's list.
__device__ __forceinline__ void build_lists_block(ListsSmem& S, const int32_t* ids, int total, int E,
                                                  int32_t* offsets, int32_t* token_list, int32_t* active,
                                                  int32_t* pass_map) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = (total + 31) >> 5;
    for (int i = tid; i < NVFP4_MAX_EXPERTS * (kMtMaxEntries / 32); i += 256) (&S.mask[0][0])[i] = 0u;
    __syncthreads();
    for (int i = tid; i < total; i += 256) {
        const int e = __ldcg(ids + i);
        S.ids[i] = e;
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
