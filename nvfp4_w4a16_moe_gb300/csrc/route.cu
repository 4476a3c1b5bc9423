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

// Fused route for up to 64 tokens (T*k <= 512 entries, E <= 256): top-k per
// token, then the per-expert lists, the active-expert list and the pass map of
// the multi-token decode kernels, in one block. Entry i = t*k + j goes to
// offsets[e] + (number of entries i' < i of expert e), read off a per-expert bit
// mask of entries: the same stable order as the counting sort above. Pass map:
// pass_map[0] = number of passes P; pass_map[1 + p] = (active slot << 8) | pass,
// a pass being up to kMtPass consecutive entries of one expert's list.
constexpr int kMtRouteThreads = 512;
constexpr int kMtMaxEntries = 512;
constexpr int kMtPass = 16;

__global__ void __launch_bounds__(kMtRouteThreads)
route_mt_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids,
                float* __restrict__ w, int32_t* __restrict__ ids_out, float* __restrict__ w_out,
                int32_t* __restrict__ offsets, int32_t* __restrict__ token_list,
                int32_t* __restrict__ active, int32_t* __restrict__ pass_map) {
    __shared__ uint32_t mask[NVFP4_MAX_EXPERTS][kMtMaxEntries / 32];
    __shared__ int s_ids[kMtMaxEntries];
    __shared__ int s_off[NVFP4_MAX_EXPERTS];
    __shared__ int wsum[3][NVFP4_MAX_EXPERTS / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total = T * k;
    const int nw = (total + 31) >> 5;
    for (int i = tid; i < NVFP4_MAX_EXPERTS * (kMtMaxEntries / 32); i += kMtRouteThreads)
        (&mask[0][0])[i] = 0u;
    for (int t = warp; t < T; t += kMtRouteThreads / 32)
        topk_warp(logits + (size_t)t * E, E, k, ids + (size_t)t * k, w + (size_t)t * k);
    __syncthreads();
    if (tid < total) {
        const int e = ids[tid];
        s_ids[tid] = e;
        atomicOr(&mask[e][tid >> 5], 1u << (tid & 31));
        if (ids_out) ids_out[tid] = e;
        if (w_out) w_out[tid] = w[tid];
    }
    __syncthreads();
    // per-expert count c, then exclusive scans over experts (threads 0..255) of
    // c (list offset), [c > 0] (active slot) and ceil(c / kMtPass) (first pass)
    int c = 0;
    if (tid < E)
        for (int qq = 0; qq < nw; ++qq) c += __popc(mask[tid][qq]);
    const int v0 = c, v1 = c > 0 ? 1 : 0, v2 = (c + kMtPass - 1) / kMtPass;
    int i0 = v0, i1 = v1, i2 = v2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n0 = __shfl_up_sync(0xffffffffu, i0, o);
        const int n1 = __shfl_up_sync(0xffffffffu, i1, o);
        const int n2 = __shfl_up_sync(0xffffffffu, i2, o);
        if (lane >= o) { i0 += n0; i1 += n1; i2 += n2; }
    }
    if (warp < NVFP4_MAX_EXPERTS / 32 && lane == 31) {
        wsum[0][warp] = i0;
        wsum[1][warp] = i1;
        wsum[2][warp] = i2;
    }
    __syncthreads();
    if (tid < E) {
        int b0 = 0, b1 = 0, b2 = 0;
        for (int ww = 0; ww < warp; ++ww) { b0 += wsum[0][ww]; b1 += wsum[1][ww]; b2 += wsum[2][ww]; }
        const int off = b0 + i0 - v0, slot = b1 + i1 - v1, pass0 = b2 + i2 - v2;
        s_off[tid] = off;
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
    if (tid < total) {
        const int e = s_ids[tid], qw = tid >> 5;
        int r = __popc(mask[e][qw] & ((1u << (tid & 31)) - 1u));
        for (int qq = 0; qq < qw; ++qq) r += __popc(mask[e][qq]);
        token_list[s_off[e] + r] = tid;
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

cudaError_t launch_route_mt(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                            int32_t* ids_out, float* w_out, int32_t* offsets, int32_t* token_list,
                            int32_t* active, int32_t* pass_map, cudaStream_t s) {
    if (T < 1 || T * k > kMtMaxEntries || E > NVFP4_MAX_EXPERTS) return cudaErrorInvalidValue;
    route_mt_kernel<<<1, kMtRouteThreads, 0, s>>>(logits, T, E, k, ids, w, ids_out, w_out, offsets,
                                                  token_list, active, pass_map);
    return cudaGetLastError();
}

}  // namespace nvfp4
