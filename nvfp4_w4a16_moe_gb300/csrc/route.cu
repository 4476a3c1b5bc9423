// Router tail: softmax over all experts -> top-k -> renormalise, then the
// per-expert token lists for the grouped expert kernels.
//
// lynn-engine tutorials index, row 06 (MoE router): Qwen routes with softmax over
// all experts, then top-k, then renormalisation, which equals a softmax over the
// k selected logits. That identity is what the kernel evaluates: the k largest
// logits are found with warp arg-max rounds (ties go to the lower expert id,
// the sorted-router order of the lynn-engine README, P35 note) and the weights
// are exp(l_j - l_max) / sum_j' exp(l_j' - l_max). Expert ids are int32 once,
// right after the router (README, P23 note).
#include <cfloat>

#include "common.cuh"
#include "kernels.cuh"

namespace nvfp4 {

namespace {

// One warp per token. E <= 256: lane l holds logits l, l+32, ..., l+224.
__device__ __forceinline__ void topk_warp(const float* __restrict__ lg, int E, int k,
                                          int32_t* __restrict__ ids_out, float* __restrict__ w_out) {
    const int lane = threadIdx.x & 31;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? lg[e] : -FLT_MAX;
    }
    unsigned taken = 0;
    float sel_v[NVFP4_MAX_TOPK];
    int sel_e[NVFP4_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < NVFP4_MAX_TOPK; ++j) {
        if (j >= k) break;
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u)) {
                if (v[i] > bv || (v[i] == bv && e < be) || be == 0x7fffffff) { bv = v[i]; be = e; }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) { bv = ov; be = oe; }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        sel_v[j] = bv;
        sel_e[j] = be;
    }
    float ex[NVFP4_MAX_TOPK];
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NVFP4_MAX_TOPK; ++j) {
        if (j < k) { ex[j] = expf(sel_v[j] - sel_v[0]); sum += ex[j]; }
    }
#pragma unroll
    for (int j = 0; j < NVFP4_MAX_TOPK; ++j) {
        if (j < k && lane == j) { ids_out[j] = sel_e[j]; w_out[j] = ex[j] / sum; }
    }
}

__global__ void route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                  int32_t* __restrict__ ids, float* __restrict__ w) {
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    topk_warp(logits + (size_t)t * E, E, k, ids + (size_t)t * k, w + (size_t)t * k);
}

// Stable counting sort of the T*k entries by expert id, one block of 1024
// threads, chunks of 1024 entries. Inside a chunk, the rank of an entry among
// the entries of the same expert is: entries of that expert in earlier warps
// (prefix over per-warp counts) + entries in earlier lanes of its warp
// (__match_any_sync). Fully deterministic (no order-dependent atomics).
constexpr int kListThreads = 1024;

__global__ void __launch_bounds__(kListThreads)
route_lists_kernel(const int32_t* __restrict__ ids, int total, int E,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ token_list,
                   int32_t* __restrict__ active) {
    __shared__ int cnt[NVFP4_MAX_EXPERTS];
    __shared__ int cursor[NVFP4_MAX_EXPERTS];
    __shared__ int wcnt[kListThreads / 32][NVFP4_MAX_EXPERTS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += kListThreads) cnt[e] = 0;
    __syncthreads();
    for (int i = tid; i < total; i += kListThreads) atomicAdd(&cnt[ids[i]], 1);
    __syncthreads();
    if (tid == 0) {
        int run = 0, na = 0;
        for (int e = 0; e < E; ++e) {
            offsets[e] = run;
            cursor[e] = run;
            if (cnt[e] > 0 && active) active[1 + na++] = e;
            run += cnt[e];
        }
        offsets[E] = run;
        if (active) active[0] = na;
    }
    __syncthreads();
    for (int base = 0; base < total; base += kListThreads) {
        for (int i = tid; i < (kListThreads / 32) * E; i += kListThreads) wcnt[i / E][i % E] = 0;
        __syncthreads();
        const int idx = base + tid;
        const int e = idx < total ? ids[idx] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank_w = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank_w == 0) wcnt[warp][e] = __popc(peers);
        __syncthreads();
        for (int ee = tid; ee < E; ee += kListThreads) {
            int pre = 0;
            for (int w = 0; w < kListThreads / 32; ++w) {
                const int c = wcnt[w][ee];
                wcnt[w][ee] = pre;
                pre += c;
            }
            cnt[ee] = pre;   // entries of expert ee in this chunk
        }
        __syncthreads();
        if (e >= 0) token_list[cursor[e] + wcnt[warp][e] + rank_w] = idx;
        __syncthreads();
        for (int ee = tid; ee < E; ee += kListThreads) cursor[ee] += cnt[ee];
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_route_lists(const int32_t* ids, int total, int E, int32_t* offsets,
                               int32_t* token_list, int32_t* active, cudaStream_t s) {
    route_lists_kernel<<<1, kListThreads, 0, s>>>(ids, total, E, offsets, token_list, active);
    return cudaGetLastError();
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                              cudaStream_t s) {
    const int warps = 8;
    const int grid = (T + warps - 1) / warps;
    route_topk_kernel<<<grid, warps * 32, 0, s>>>(logits, T, E, k, ids, w);
    return cudaGetLastError();
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         int32_t* offsets, int32_t* token_list, cudaStream_t s) {
    if (T == 0) {
        return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
    }
    cudaError_t err = launch_route_topk(logits, T, E, k, ids, w, s);
    if (err != cudaSuccess) return err;
    return launch_route_lists(ids, T * k, E, offsets, token_list, nullptr, s);
}

}  // namespace nvfp4
